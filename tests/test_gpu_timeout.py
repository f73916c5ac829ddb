"""Bounded waits: a dependency wait that runs out sets MOE_STATUS_TIMEOUT, the kernel drains
its own copies and returns, and a workspace re-initialised afterwards serves a normal call.

The wait is made to run out without any fault: moe_workspace_set_wait_limit makes every wait
of the expert kernels (the tensor-core kernel in decode and in prefill, the CUDA-core
streaming decode kernel) on another CTA's progress (x encoded, a key's or a token tile's h
rows complete) give up after one poll, and in a small call the CTAs that take down units
check their h count long before any gate/up tile has finished.  Waits on a CTA's own copies and MMAs keep their default limit, so
every copy that was issued lands, and every MMA completes, before its CTA exits."""
import numpy as np
import pytest
import torch

import fp4_routed_expert_gb300 as moe
from fp4_routed_expert_gb300.layer import MoeLayer
from synth import tensors as syn

from test_gpu_parity import oracle_with_routing
from workloads import bits_to_torch, make_workload, row_rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tiny():
    return make_workload(512, 256, 16, 2, seed=0, scale=(-8, -4))


@pytest.mark.parametrize("cuda_cores", [False, True], ids=["tensor_cores", "cuda_cores"])
def test_decode_dependency_wait_times_out_then_workspace_recovers(tiny, cuda_cores):
    T = 3
    layer = MoeLayer(tiny.d, tiny.f, tiny.E, tiny.k, T, tiny.arena)
    x_bits = syn.activations(0, 60, T, tiny.d)
    x = bits_to_torch(x_bits, DEV)
    wr = bits_to_torch(tiny.wr, DEV)
    tab = torch.from_numpy(tiny.table).to(DEV)
    layer.route(x, wr, tab)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    moe.moe_workspace_set_wait_limit(layer.dims, layer.ws, 1)
    layer.experts(x, cuda_cores=cuda_cores)
    torch.cuda.synchronize()                      # the call returned
    assert int(layer.status.item()) & moe.MOE_STATUS_TIMEOUT
    # recovery: re-initialise the workspace (default limit again), route and run normally
    moe.moe_workspace_init(layer.dims, layer.ws)
    layer.status.zero_()
    layer.route(x, wr, tab)
    y = layer.experts(x, cuda_cores=cuda_cores)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    r = dict(ids=layer.ids[:T].cpu().numpy(), slots=layer.slots[:T].cpu().numpy(), weights=layer.w[:T].cpu().numpy())
    ref = oracle_with_routing(tiny, x_bits, r)
    err = row_rel_err(y[:T].float().cpu().numpy(), ref)
    assert err.max() <= 1e-2, err


def test_single_request_decode_wait_times_out_then_workspace_recovers(tiny):
    """The same through moe_layer_decode_fp4, whose expert kernel also waits for the router's
    key records (one poll of the router's counter, then the key hand-offs): the call returns
    with MOE_STATUS_TIMEOUT, and after moe_workspace_init the next single request equals the
    oracle."""
    T = 3
    layer = MoeLayer(tiny.d, tiny.f, tiny.E, tiny.k, T, tiny.arena)
    x_bits = syn.activations(0, 62, T, tiny.d)
    x = bits_to_torch(x_bits, DEV)
    wr = bits_to_torch(tiny.wr, DEV)
    tab = torch.from_numpy(tiny.table).to(DEV)
    moe.moe_workspace_set_wait_limit(layer.dims, layer.ws, 1)
    layer.decode(x, wr, tab)
    torch.cuda.synchronize()                      # the call returned
    assert int(layer.status.item()) & moe.MOE_STATUS_TIMEOUT
    moe.moe_workspace_init(layer.dims, layer.ws)
    layer.status.zero_()
    y = layer.decode(x, wr, tab)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    r = dict(ids=layer.ids[:T].cpu().numpy(), slots=layer.slots[:T].cpu().numpy(), weights=layer.w[:T].cpu().numpy())
    ref = oracle_with_routing(tiny, x_bits, r)
    err = row_rel_err(y[:T].float().cpu().numpy(), ref)
    assert err.max() <= 1e-2, err


def test_prefill_dependency_wait_times_out_then_workspace_recovers(tiny):
    """The same on the tensor-core prefill path (T = 40 > 16: permuted rows in token tiles; a
    down unit waits for every gate/up unit of its tile)."""
    T = 40
    layer = MoeLayer(tiny.d, tiny.f, tiny.E, tiny.k, T, tiny.arena)
    x_bits = syn.activations(0, 61, T, tiny.d)
    x = bits_to_torch(x_bits, DEV)
    wr = bits_to_torch(tiny.wr, DEV)
    tab = torch.from_numpy(tiny.table).to(DEV)
    layer.route(x, wr, tab)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    moe.moe_workspace_set_wait_limit(layer.dims, layer.ws, 1)
    layer.experts(x, fused_prefill=True)
    torch.cuda.synchronize()
    assert int(layer.status.item()) & moe.MOE_STATUS_TIMEOUT
    moe.moe_workspace_init(layer.dims, layer.ws)
    layer.status.zero_()
    layer.route(x, wr, tab)
    y = layer.experts(x, fused_prefill=True)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    r = dict(ids=layer.ids[:T].cpu().numpy(), slots=layer.slots[:T].cpu().numpy(), weights=layer.w[:T].cpu().numpy())
    ref = oracle_with_routing(tiny, x_bits, r)
    err = row_rel_err(y[:T].float().cpu().numpy(), ref)
    assert err.max() <= 1e-2, err
