"""The layer-chaining step of the multi-layer workloads (moe_residual_rmsnorm): bf16 RMSNorm
of x + y with unit weight, computed in fp32 on the device, against the oracle's fp64
statement.  Both round the same real value to bf16, so they agree to one bf16 ulp (the fp32
sum of squares moves the scale by a few fp32 ulps, which can cross a bf16 rounding
boundary); in-place output (x_next aliasing x) gives the same bits."""
import numpy as np
import pytest
import torch

import fp4_routed_expert_gb300 as moe
import oracle
from synth import tensors as syn

from workloads import bits_to_torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,d", [(1, 5120), (16, 5120), (37, 512), (3, 96)])
def test_residual_rmsnorm_matches_oracle(T, d):
    xb = syn.activations(21, 0, T, d, stream=1)
    yb = syn.activations(21, 1, T, d, stream=2)
    x, y = bits_to_torch(xb, "cuda"), bits_to_torch(yb, "cuda")
    out = torch.empty_like(x)
    moe.moe_residual_rmsnorm(T, d, x, y, 1e-6, out)
    inplace = x.clone()
    moe.moe_residual_rmsnorm(T, d, inplace, y, 1e-6, inplace)
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(inplace.view(torch.int16).cpu().numpy().view(np.uint16), got)
    ref = oracle.residual_rmsnorm(xb, syn.bf16_bits_to_f32(yb).astype(np.float64), 1e-6)
    g = syn.bf16_bits_to_f32(got).astype(np.float64)
    r = syn.bf16_bits_to_f32(ref).astype(np.float64)
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(r), 1e-30))[1] - 8)   # bf16 spacing at |r|
    assert (np.abs(g - r) <= ulp).all()
    assert (got != ref).mean() < 0.01


def test_residual_rmsnorm_rejects_bad_arguments():
    x = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        moe.moe_residual_rmsnorm(2, 64, x, x, float("nan"), x)
    with pytest.raises(RuntimeError):
        moe.moe_residual_rmsnorm(2, 0, x, x, 1e-6, x)
    moe.moe_residual_rmsnorm(0, 64, None, None, 1e-6, None)   # T = 0: nothing to do
