"""The seeded input generator: Philox4x32-10 against its published known-answer vectors,
and the shape/range contracts of the synthetic tensors."""
import os

import numpy as np

from synth import philox
from synth import tensors as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        v = [int(t, 16) for t in line.split()]
        out = philox.philox4x32_10(*[np.array([c], np.uint64) for c in v[:4]], v[4], v[5])
        assert [int(o[0]) for o in out] == v[6:]


def test_stream_windows_agree():
    a = philox.words(7, 99, 50)
    b = philox.words(7, 99, 37, start=13)
    assert np.array_equal(a[13:50], b)


def test_expert_tensors_ranges_and_determinism():
    ex = syn.expert_tensors(0, 3, 17, 64, 32, -10, -6)
    for n, shp in syn.expert_tensor_shapes(64, 32).items():
        assert ex[n].shape == shp and ex[n].dtype == np.uint8
    for n in ("gate_s", "up_s", "down_s"):
        assert ex[n].min() >= 117 and ex[n].max() <= 121
    ex2 = syn.expert_tensors(0, 3, 17, 64, 32, -10, -6)
    assert all(np.array_equal(ex[n], ex2[n]) for n in ex)
    ex3 = syn.expert_tensors(0, 3, 18, 64, 32, -10, -6)
    assert not np.array_equal(ex["gate_q"], ex3["gate_q"])


def test_bf16_rounding_ties_to_even():
    v = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20], np.float32)
    b = syn.f32_to_bf16_bits(v)
    assert syn.bf16_bits_to_f32(b).tolist() == [1.0, 1 + 2 ** -6, 1 + 2 ** -7]


def test_activation_statistics():
    x = syn.bf16_bits_to_f32(syn.activations(0, 0, 64, 512)).astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02


def test_keepset_tables():
    tab = syn.keepset_slot_tables(0, 3, 384, 154, 1.1)
    assert tab.shape == (3, 384)
    assert all((tab[l] >= 0).sum() == 154 for l in range(3))
    used = np.sort(tab[tab >= 0])
    assert np.array_equal(used, np.arange(3 * 154))


def test_bias_is_centered_and_skewed():
    b = syn.zipf_score_bias(0, 0, 384, 1.2, 0.04)
    assert abs(float(b.mean())) < 1e-6 and b.max() > 0.1
