"""The seeded input generator, pinned to its published definitions."""
import numpy as np
import pytest
import torch

import synth


def test_splitmix64_published_vector():
    # SplitMix64 started at state 0: the first outputs of the reference
    # implementation (Vigna's splitmix64.c) are these three words.
    got = [int(v) for v in synth.splitmix64_raw(0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_bf16_rounding_matches_torch():
    # torch converts float32 -> bfloat16 by round to nearest even.
    vals = np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 1.0078125, 3.14159, -2.71828,
                     65504.0, 1e-30, -1e30, 0.1, 1 / 3, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9],
                    dtype=np.float32)
    rng = np.random.default_rng(0)
    vals = np.concatenate([vals, rng.standard_normal(2000).astype(np.float32) * 10])
    ours = synth.f32_to_bf16_bits(vals)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_normal_moments_and_shape():
    a = synth.bf16_bits_to_f32(synth.normal_bf16(0, 0, (1 << 20,))).astype(np.float64)
    assert abs(a.mean()) < 5e-3
    assert abs(a.std() - 1.0) < 5e-3
    # fourth moment of a normal is 3
    assert abs((a ** 4).mean() - 3.0) < 0.05
    w = synth.bf16_bits_to_f32(synth.normal_bf16(0, 1, (1 << 18,), std=0.02)).astype(np.float64)
    assert abs(w.std() - 0.02) < 2e-4


def test_normal_matches_scipy_cdf():
    scipy_stats = pytest.importorskip("scipy.stats")
    z = synth.normal_f64(3, 2, (200000,))
    assert scipy_stats.kstest(z, "norm").pvalue > 1e-3


def test_counter_based_slices_and_determinism():
    full = synth.normal_bf16(7, 4, (10000,))
    part = synth.normal_bf16(7, 4, (1000,), start=4321)
    assert np.array_equal(full[4321:5321], part)
    assert np.array_equal(full, synth.normal_bf16(7, 4, (10000,)))
    assert not np.array_equal(full, synth.normal_bf16(7, 5, (10000,)))
    assert not np.array_equal(full, synth.normal_bf16(8, 4, (10000,)))


def test_expert_slice_matches_whole_tensor():
    wl = synth.workload("tiny", T=4)
    inp = synth.make_inputs(wl)
    for name in ("w_gate", "w_up", "w_down"):
        assert np.array_equal(synth.expert_slice(wl, name, 5), inp[name][5])


def test_random_topk_distinct_and_skewed():
    idx = synth.random_topk(0, 2000, 64, 4, alpha=2.0)
    assert idx.shape == (2000, 4)
    assert all(len(set(r)) == 4 for r in idx.tolist())
    counts = np.bincount(idx.ravel(), minlength=64)
    assert counts[0] > 1900 and counts[0] == counts.max()  # rank-1 expert dominates under alpha=2
    u = synth.random_topk(0, 2000, 64, 4, alpha=0.0)
    assert np.bincount(u.ravel(), minlength=64).max() < 250


def test_zipf_bias():
    b = synth.zipf_logit_bias(0, 64, 0.0).astype(np.float64)
    assert np.allclose(b, -np.log(64.0))
    b2 = synth.zipf_logit_bias(0, 64, 2.0).astype(np.float64)
    p = np.exp(b2)
    assert abs(p.sum() - 1.0) < 1e-5
    assert np.allclose(np.sort(p)[::-1] / p.max(), np.arange(1, 65) ** -2.0, rtol=1e-5)
