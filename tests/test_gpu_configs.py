"""The 40-layer workloads at full size, checked layer by layer on sampled tokens.

Keep-set arena: 40 layers x 154 resident experts of 384 (6,160 slots, 115.8 GB of FP4 experts)
behind per-layer expert->slot tables drawn from a Zipf(1.1) popularity; routing masks the
non-resident experts.  Decode (T = 1) and DSpark verify (T = 16) run one step through all 40
layers; long prefill runs 8,192-token chunks through all 40 layers with a fresh Zipf(1.1)
score bias per layer.  Each layer's input is the previous layer's input plus its output after
RMSNorm (eps 1e-6, unit weight), rounded to bf16 -- formed here by the oracle's routine from
the GPU's output, so every layer is checked on exactly the input the GPU used."""
import numpy as np
import pytest
import torch

import fp4_routed_expert_gb300 as moe
from fp4_routed_expert_gb300.layer import Arena, MoeLayer
import oracle
from synth import tensors as syn
from synth.keepset import D, E, F, K, KEEP, LAYERS, SCALE, KeepSetArena

from workloads import bits_to_torch, elem_rel_err, row_rel_err

pytestmark = pytest.mark.gpu

TOL = 1e-2
DEV = "cuda"


class KeepSet(KeepSetArena):
    def __init__(self):
        torch.cuda.empty_cache()
        super().__init__(DEV)

    def oracle_layer(self, l, x_bits, tokens, bias=None):
        """Oracle routing (all given tokens) and outputs of the sampled tokens."""
        r = oracle.route_topk(x_bits[tokens], self.wr_bits[l], bias, self.tabs[l], K)
        ys = []
        cache = {}
        for n, t in enumerate(tokens):
            z = np.zeros((K, D), np.float32)
            for j in range(K):
                e = int(r["ids"][n, j])
                if e < 0:
                    continue
                if e not in cache:
                    cache[e] = syn.expert_tensors(0, l, e, D, F, *SCALE)
                _, z[j] = oracle.expert_ffn_f32(x_bits[t], cache[e])
            ys.append(oracle.combine_f32(z, r["weights"][n]))
        return r, np.stack(ys)


@pytest.fixture(scope="module")
def keepset():
    ks = KeepSet()
    yield ks
    del ks.arena
    torch.cuda.empty_cache()


def run_layer(ks, l, x_bits, layer, bias=None):
    x = bits_to_torch(x_bits, DEV)
    T = x_bits.shape[0]
    b = None if bias is None else torch.from_numpy(bias).to(DEV)
    layer.route(x, ks.wr[l], ks.tab_dev[l], b, T=T)
    y = layer.experts(x, T=T, fused_prefill=True)
    torch.cuda.synchronize()
    return dict(ids=layer.ids[:T].cpu().numpy(), slots=layer.slots[:T].cpu().numpy(),
                w=layer.w[:T].cpu().numpy(), status=int(layer.status.item()), y=y[:T].float().cpu().numpy())


def check_layer(ks, l, x_bits, got, tokens, bias=None):
    r, y = ks.oracle_layer(l, x_bits, tokens, bias)
    np.testing.assert_array_equal(got["ids"][tokens], r["ids"], err_msg="layer %d" % l)
    np.testing.assert_array_equal(got["slots"][tokens], r["slots"], err_msg="layer %d" % l)
    np.testing.assert_allclose(got["w"][tokens], r["weights"], rtol=2e-5, atol=1e-7)
    assert (got["slots"][tokens] >= 0).all()                      # 154 resident >= k: never short
    err = row_rel_err(got["y"][tokens], y)
    assert err.max() <= TOL, (l, err)
    check_layer.elem = max(getattr(check_layer, "elem", 0.0), float(elem_rel_err(got["y"][tokens], y).max()))
    return err.max()


@pytest.mark.parametrize("T", [1, 16], ids=["decode_T1", "verify_T16"])
def test_keepset_decode_40_layers(keepset, T):
    """One decode (T = 1) or DSpark-verify (T = 16) step through the 40 keep-set layers: every
    layer's ids and slots against the oracle for all tokens at every 8th layer (for T = 1 at
    every layer), outputs of sampled tokens against the oracle layer, and the resident mask
    holding (every chosen slot is a resident one)."""
    ks = keepset
    x = syn.activations(0, 0, T, D, stream=11)
    layer = MoeLayer(D, F, E, K, T, ks.arena)
    worst = 0.0
    for l in range(LAYERS):
        got = run_layer(ks, l, x, layer)
        assert got["status"] == 0
        resident = ks.tabs[l][got["ids"]]
        assert (resident == got["slots"]).all() and (got["slots"] >= 0).all()
        if T == 1 or l % 8 == 0 or l == LAYERS - 1:
            tokens = [0] if T == 1 else [0, T - 1]
            if T > 1:   # ids of every token of the step
                r = oracle.route_topk(x, ks.wr_bits[l], None, ks.tabs[l], K)
                np.testing.assert_array_equal(got["ids"], r["ids"], err_msg="layer %d" % l)
            worst = max(worst, check_layer(ks, l, x, got, tokens))
        x = oracle.residual_rmsnorm(x, got["y"].astype(np.float64))
    print("max row error over the checked layers %.3e (elementwise, 1e-3 floor: %.3e)" % (worst, check_layer.elem))


def test_keepset_long_prefill_40_layers(keepset):
    """8,192-token chunks (the first and the last of a 32,768-token sequence) through the 40
    keep-set layers, fresh Zipf(1.1) bias per layer: sampled tokens' ids, slots and outputs
    against the oracle at every 5th layer, the whole chunk's permutation against the oracle's
    at every 10th, the resident mask at every layer."""
    ks = keepset
    T = 8192
    layer = MoeLayer(D, F, E, K, T, ks.arena)
    worst = 0.0
    for chunk in (0, 3):
        x = syn.activations(0, 0, T, D, start_token=chunk * T, stream=13)
        for l in range(LAYERS):
            bias = syn.zipf_score_bias(0, l, E, 1.1, 0.04)
            got = run_layer(ks, l, x, layer, bias=bias)
            assert got["status"] == 0
            assert (ks.tabs[l][got["ids"]] == got["slots"]).all() and (got["slots"] >= 0).all()
            if l % 5 == 0 or l == LAYERS - 1:
                worst = max(worst, check_layer(ks, l, x, got, [0, 4095, T - 1], bias=bias))
            if l % 10 == 0:
                perm = oracle.permute(got["ids"], E)
                n = perm["rows"]
                np.testing.assert_array_equal(layer.offsets.cpu().numpy(), perm["offsets"])
                np.testing.assert_array_equal(layer.row_src[:n].cpu().numpy(), perm["row_src"])
            x = oracle.residual_rmsnorm(x, got["y"].astype(np.float64))
    print("max row error over the checked layers %.3e (elementwise, 1e-3 floor: %.3e)" % (worst, check_layer.elem))
