"""Stage-by-stage parity of the CUDA path with the oracle, through the C ABI.

Each stage is driven by inputs from the seeded generator (not by another
stage's GPU output), at sizes that span several tiles and ragged tails.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_06_gb300 as moe
import oracle
import synth
from synth.workloads import Workload

from gpu_util import (check_routing, dev_bf16, dev_f16, dev_f32, dev_i32, device_inputs, host_bits, host_f64,
                      make_cfg)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load_library()


# ----------------------------------------------------------------------------- router

ROUTER_CASES = [
    ("tiny", 128, {}), ("tiny", 1, {}), ("tiny", 200, {}),
    ("mixtral", 300, {}),
    ("qwen2", 256, {}),
    ("skew", 256, {"alpha": 0.0}), ("skew", 512, {"alpha": 1.0}), ("skew", 512, {"alpha": 2.0}),
    ("deepseek", 512, {}),
    # unpaired batches of 10+ token tiles, whose K split stops at clusters of 4
    # (the grid would pass half the SMs with clusters of 8)
    ("deepseek", 2048, {}), ("mixtral", 2000, {}),
    # group-limited variants: 8 groups of 8 (groups inside a 32-column block),
    # top-3 / top-1 per group, 16 groups of 16
    ("deepseek", 256, {"E": 64}), ("deepseek", 256, {"group_topn": 3}), ("deepseek", 256, {"group_topn": 1}),
    ("deepseek", 256, {"n_group": 16, "topk_group": 6}),
    # batches that run the router as CTA pairs (256 tokens per MMA, half of
    # W_r on each CTA): a ragged last pair tile, and 144 experts (72 W_r rows
    # per CTA) without groups
    ("deepseek", 4100, {}), ("deepseek", 4096, {"E": 144, "n_group": 1, "topk_group": 1, "group_topn": 0}),
]


@pytest.mark.parametrize("name,T,kw", ROUTER_CASES, ids=[f"{c[0]}-T{c[1]}-{c[2]}" for c in ROUTER_CASES])
def test_route(name, T, kw):
    wl = synth.workload(name, T=T, **kw)
    inp = synth.make_inputs(wl, with_experts=False)
    d = device_inputs(inp)
    cfg = make_cfg(wl, d)
    idx, w, ss = moe.moe_route(d["x"], d["w_router"], wl.k, cfg)
    st, raw = moe.moe_device_error()
    assert st == 0, raw
    r = oracle.Routing.of(wl)
    logits = oracle.router_logits(inp["x"], inp["w_router"], inp.get("logit_bias"))
    scores = oracle.router_scores(logits, r.score)
    o_idx = oracle.select_experts(scores, wl.k, r)
    orc = {"idx": o_idx, "scores": scores, "w": oracle.routing_weights(scores, o_idx, r),
           "margin": oracle.selection_margin(scores, wl.k, r)}
    same = check_routing(wl, idx.cpu().numpy(), w.cpu().numpy(), orc)
    assert same.mean() > 0.95
    if wl.shared_gate:
        xf = oracle.widen(inp["x"])
        want = 1.0 / (1.0 + np.exp(-(xf @ oracle.widen(inp["w_shared_gate"]))))
        np.testing.assert_allclose(ss.cpu().numpy(), want, rtol=1e-5, atol=1e-6)


def test_route_equal_logits_and_one_hot_bias():
    wl = Workload("t", T=70, H=256, F=128, E=16, k=4)
    x = synth.normal_bf16(0, 0, (70, 256))
    wr = np.zeros((16, 256), dtype=np.uint16)
    idx, w, _ = moe.moe_route(dev_bf16(x), dev_bf16(wr), 4)
    assert np.all(idx.cpu().numpy() == np.arange(4)[None, :])  # ties -> lowest ids
    np.testing.assert_allclose(w.cpu().numpy(), 0.25, rtol=1e-6)
    bias = np.zeros(16, dtype=np.float32)
    bias[11] = 30.0
    cfg = moe.MoeConfig.make(logit_bias=dev_f32(bias))
    idx, w, _ = moe.moe_route(dev_bf16(x), dev_bf16(wr), 1, cfg)
    assert np.all(idx.cpu().numpy() == 11)
    np.testing.assert_allclose(w.cpu().numpy(), 1.0)


# ----------------------------------------------------------------------------- permute

PERMUTE_CASES = [(1, 8, 2, 0.0, 512), (37, 8, 2, 0.0, 512), (1000, 64, 4, 0.0, 256), (1000, 64, 4, 2.0, 128),
                 (4096, 8, 2, 1.0, 128), (3000, 256, 8, 0.0, 256), (8192, 256, 8, 1.5, 128), (33, 3, 3, 0.0, 128)]


@pytest.mark.parametrize("T,E,k,alpha,H", PERMUTE_CASES)
def test_permute(T, E, k, alpha, H):
    idx = synth.random_topk(3, T, E, k, alpha=alpha)
    x = synth.normal_bf16(3, 50, (T, H))
    counts, offsets, perm, inv, x_perm = moe.moe_permute(dev_i32(idx), dev_bf16(x), E)
    st, raw = moe.moe_device_error()
    assert st == 0, raw
    c, o, p, i = oracle.permute(idx, E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(perm.cpu().numpy(), p)
    assert np.array_equal(inv.cpu().numpy(), i)
    assert np.array_equal(host_bits(x_perm), x[p // k])


def test_permute_rejects_out_of_range_expert_on_device():
    idx = synth.random_topk(3, 100, 8, 2)
    idx[17, 1] = 999
    idx[40, 0] = -3
    counts, offsets, perm, inv, _ = moe.moe_permute(dev_i32(idx), dev_bf16(synth.normal_bf16(3, 1, (100, 128))), 8)
    st, raw = moe.moe_device_error()
    assert st == 6 and raw & 2
    assert counts.cpu().numpy().sum() == 198
    iv = inv.cpu().numpy()
    assert iv[17 * 2 + 1] == -1 and iv[40 * 2] == -1
    assert moe.moe_device_error()[0] == 0  # cleared


# ----------------------------------------------------------------------------- expert FFN

def _ffn_case(rows_per_group, H, F, seed=9):
    """Grouped rows with the given per-group counts; weights ~ N(0, 0.02)."""
    E = len(rows_per_group)
    counts = np.array(rows_per_group, dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    R = int(offsets[-1])
    xp = synth.normal_bf16(seed, 60, (R, H))
    wg = synth.normal_bf16(seed, 61, (E, F, H), std=0.02)
    wu = synth.normal_bf16(seed, 62, (E, F, H), std=0.02)
    wd = synth.normal_bf16(seed, 63, (E, H, F), std=0.02)
    return xp, offsets, wg, wu, wd


def _oracle_ffn(xp, offsets, wg, wu, wd, activation="silu"):
    xf = oracle.widen(xp)
    E = wg.shape[0]
    h = np.zeros((xf.shape[0], wg.shape[1]))
    y = np.zeros((xf.shape[0], wd.shape[1]))
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            g = xf[a:b] @ oracle.widen(wg[e]).T
            u = xf[a:b] @ oracle.widen(wu[e]).T
            h[a:b] = oracle.activate(g, activation) * u
            y[a:b] = oracle.swiglu_expert(xf[a:b], wg[e], wu[e], wd[e], activation)
    return h, y


FFN_CASES = [
    ("ragged_small", [5, 0, 17, 1, 30, 0, 0, 11], 512, 1024),
    ("bn16", [3, 9, 14, 16, 7, 1, 12, 2], 256, 384),
    ("bn32", [31, 20, 33, 25], 384, 256),
    ("bn64", [64, 70, 1, 55, 60, 66, 0, 80], 512, 512),
    ("bn128", [128, 100, 129, 150], 256, 640),
    ("bn256", [300, 257, 200, 255], 512, 512),
    ("one_expert_all_rows", [0, 0, 333, 0, 0, 0, 0, 0], 512, 1024),
    ("single_row", [0, 1, 0, 0], 128, 128),
]


@pytest.mark.parametrize("name,counts,H,F", FFN_CASES, ids=[c[0] for c in FFN_CASES])
def test_expert_ffn(name, counts, H, F):
    xp, offsets, wg, wu, wd = _ffn_case(counts, H, F)
    h, y = moe.moe_expert_ffn(dev_bf16(xp), dev_i32(offsets), dev_bf16(wg), dev_bf16(wu), dev_bf16(wd))
    st, raw = moe.moe_device_error()
    assert st == 0, raw
    h_or, y_or = _oracle_ffn(xp, offsets, wg, wu, wd)
    h_gpu = host_f64(h)
    # h: one bf16 rounding of an fp32-accumulated value
    assert np.all(np.abs(h_gpu - h_or) <= 2.0 ** -8 * np.abs(h_or) + 1e-4)
    y_gpu = host_f64(y)
    rel = np.linalg.norm(y_gpu - y_or) / np.linalg.norm(y_or)
    assert rel < 4e-3, rel
    assert np.abs(y_gpu - y_or).max() <= 1e-2 * np.abs(y_or).max()


@pytest.mark.parametrize("counts,H,F", [([5, 17, 1, 30, 0, 64], 256, 384), ([130, 100, 129, 120], 256, 640),
                                        ([300, 257, 200, 255], 512, 512)],
                         ids=["bn16", "bn128", "pair_tiles"])
def test_expert_ffn_geglu(counts, H, F):
    """GELU in place of SiLU in the same fused epilogue (GEGLU experts)."""
    xp, offsets, wg, wu, wd = _ffn_case(counts, H, F)
    h, y = moe.moe_expert_ffn(dev_bf16(xp), dev_i32(offsets), dev_bf16(wg), dev_bf16(wu), dev_bf16(wd),
                              activation="gelu")
    assert moe.moe_device_error()[0] == 0
    h_or, y_or = _oracle_ffn(xp, offsets, wg, wu, wd, "gelu")
    h_gpu, y_gpu = host_f64(h), host_f64(y)
    assert np.all(np.abs(h_gpu - h_or) <= 2.0 ** -8 * np.abs(h_or) + 1e-4)
    assert np.linalg.norm(y_gpu - y_or) / np.linalg.norm(y_or) < 4e-3
    # and it is not the SwiGLU result
    h_silu, _ = _oracle_ffn(xp, offsets, wg, wu, wd, "silu")
    assert np.abs(h_gpu - h_silu).max() > 1e-2


@pytest.mark.parametrize("counts,H,F", [([5, 17, 1, 30], 256, 384), ([300, 257, 200, 255], 512, 512)],
                         ids=["small_tiles", "pair_tiles"])
def test_expert_ffn_weight_placement(counts, H, F):
    """The gate+up GEMM loads 64 gate rows and the 64 up rows of the same
    features as one tile, through a view whose extra dimension steps from one
    weight tensor to the other.  The result must not depend on where the two
    tensors lie: gate below up, up below gate, or one tensor passed as both
    (the view cannot be formed; two loads per tile)."""
    xp, offsets, wg, wu, wd = _ffn_case(counts, H, F)
    n = wg.size
    x_d, off_d, wd_d = dev_bf16(xp), dev_i32(offsets), dev_bf16(wd)
    gate_low = dev_bf16(np.concatenate([wg.reshape(-1), wu.reshape(-1)]))
    up_low = dev_bf16(np.concatenate([wu.reshape(-1), wg.reshape(-1)]))
    runs = {
        "gate_below_up": (gate_low[:n].view(wg.shape), gate_low[n:].view(wu.shape)),
        "up_below_gate": (up_low[n:].view(wg.shape), up_low[:n].view(wu.shape)),
    }
    outs = {}
    for name, (g_d, u_d) in runs.items():
        assert (g_d.data_ptr() < u_d.data_ptr()) == (name == "gate_below_up")
        outs[name] = moe.moe_expert_ffn(x_d, off_d, g_d, u_d, wd_d)
        assert moe.moe_device_error()[0] == 0
    h_or, y_or = _oracle_ffn(xp, offsets, wg, wu, wd)
    for name, (h, y) in outs.items():
        h_gpu, y_gpu = host_f64(h), host_f64(y)
        assert np.all(np.abs(h_gpu - h_or) <= 2.0 ** -8 * np.abs(h_or) + 1e-4), name
        assert np.linalg.norm(y_gpu - y_or) / np.linalg.norm(y_or) < 4e-3, name
    # the same dot products in the same order: bitwise equal
    assert torch.equal(outs["gate_below_up"][0], outs["up_below_gate"][0])
    assert torch.equal(outs["gate_below_up"][1], outs["up_below_gate"][1])
    # one tensor as gate and up: h = SiLU(g) * g
    g_d = gate_low[:n].view(wg.shape)
    h, y = moe.moe_expert_ffn(x_d, off_d, g_d, g_d, wd_d)
    assert moe.moe_device_error()[0] == 0
    h_or, y_or = _oracle_ffn(xp, offsets, wg, wg, wd)
    h_gpu, y_gpu = host_f64(h), host_f64(y)
    assert np.all(np.abs(h_gpu - h_or) <= 2.0 ** -8 * np.abs(h_or) + 1e-4)
    assert np.linalg.norm(y_gpu - y_or) / np.linalg.norm(y_or) < 4e-3


@pytest.mark.parametrize("counts,H,F,act", [([5, 17, 1, 30, 0, 64], 256, 384, "silu"),
                                            ([300, 257, 200, 255], 512, 512, "silu"),
                                            ([130, 100, 129, 120], 256, 640, "gelu")],
                         ids=["bn16", "pair_tiles", "bn128-gelu"])
def test_expert_ffn_unfused_ablation(counts, H, F, act):
    """The fusion ablation: g and u as two GEMMs with bf16 outputs, the
    activation element-wise.  g and u are each one bf16 rounding of the
    projections; h is act(g) * u of those rounded values, rounded once."""
    xp, offsets, wg, wu, wd = _ffn_case(counts, H, F)
    h, y, g, u = moe.moe_expert_ffn_unfused(dev_bf16(xp), dev_i32(offsets), dev_bf16(wg), dev_bf16(wu),
                                            dev_bf16(wd), activation=act)
    assert moe.moe_device_error()[0] == 0
    xf = oracle.widen(xp)
    g_or = np.zeros((xf.shape[0], F))
    u_or = np.zeros_like(g_or)
    for e in range(len(counts)):
        a, b = offsets[e], offsets[e + 1]
        g_or[a:b] = xf[a:b] @ oracle.widen(wg[e]).T
        u_or[a:b] = xf[a:b] @ oracle.widen(wu[e]).T
    g_gpu, u_gpu = host_f64(g), host_f64(u)
    assert np.all(np.abs(g_gpu - g_or) <= 2.0 ** -8 * np.abs(g_or) + 1e-4)
    assert np.all(np.abs(u_gpu - u_or) <= 2.0 ** -8 * np.abs(u_or) + 1e-4)
    # h from the GPU's own rounded g, u: one more rounding
    h_want = oracle.activate(g_gpu, act) * u_gpu
    assert np.all(np.abs(host_f64(h) - h_want) <= 2.0 ** -8 * np.abs(h_want) + 1e-4)
    _, y_or = _oracle_ffn(xp, offsets, wg, wu, wd, act)
    y_gpu = host_f64(y)
    assert np.linalg.norm(y_gpu - y_or) / np.linalg.norm(y_or) < 4e-3


@pytest.mark.parametrize("counts,H,F,block_m", [([5, 17, 1, 30, 0, 64], 256, 384, 16),
                                                ([130, 100, 129, 120, 300, 1], 256, 640, 64),
                                                ([300, 257, 200, 255], 512, 512, 128)],
                         ids=["bm16", "bm64", "bm128"])
def test_expert_ffn_static_schedule_ablation(counts, H, F, block_m):
    """The pages' schedule (host-read counts, fixed tiles, one CTA per tile)
    computes the same dot products in the same order: bit-equal to the
    persistent kernel's result."""
    xp, offsets, wg, wu, wd = _ffn_case(counts, H, F)
    args = (dev_bf16(xp), dev_i32(offsets), dev_bf16(wg), dev_bf16(wu), dev_bf16(wd))
    h_s, y_s = moe.moe_expert_ffn_static(*args, block_m=block_m)
    h, y = moe.moe_expert_ffn(*args)
    assert moe.moe_device_error()[0] == 0
    assert torch.equal(h_s.view(torch.int16), h.view(torch.int16))
    assert torch.equal(y_s, y)
    _, y_or = _oracle_ffn(xp, offsets, wg, wu, wd)
    assert np.linalg.norm(host_f64(y_s) - y_or) / np.linalg.norm(y_or) < 4e-3


def test_dense_ffn_matches_plain_swiglu():
    xp, _, wg, wu, wd = _ffn_case([200], 512, 768)
    h, y = moe.moe_expert_ffn(dev_bf16(xp), None, dev_bf16(wg[0]), dev_bf16(wu[0]), dev_bf16(wd[0]))
    assert moe.moe_device_error()[0] == 0
    y_or = oracle.swiglu_expert(oracle.widen(xp), wg[0], wu[0], wd[0])
    y_gpu = host_f64(y)
    assert np.linalg.norm(y_gpu - y_or) / np.linalg.norm(y_or) < 4e-3


# ----------------------------------------------------------------------------- combine

@pytest.mark.parametrize("T,k,H,shared", [(1, 2, 128, False), (129, 2, 512, False), (300, 8, 384, True),
                                          (64, 4, 2048, True), (4100, 8, 256, True)])
def test_combine(T, k, H, shared):
    """Inputs are fp16 expert outputs (as moe_expert_ffn writes them)."""
    E = 16
    idx = synth.random_topk(5, T, E, k)
    _, _, perm, inv = oracle.permute(idx, E)
    y_perm = synth.normal_f64(5, 70, (T * k, H)).astype(np.float16)
    w = synth.uniform01(5, 71, T * k).reshape(T, k).astype(np.float32)
    ys = synth.normal_f64(5, 72, (T, H)).astype(np.float16) if shared else None
    sc = synth.uniform01(5, 73, T).astype(np.float32) if shared else None

    def run():
        return moe.moe_combine(dev_f16(y_perm), dev_i32(inv), dev_f32(w), dev_f16(ys) if shared else None,
                               dev_f32(sc) if shared else None)

    out = run()
    Y = y_perm.astype(np.float64)[inv.reshape(T, k)]
    want = oracle.combine(Y, w.astype(np.float64))
    if shared:
        want = want + sc.astype(np.float64)[:, None] * ys.astype(np.float64)
    got = host_f64(out)
    # fp32 sum of k+1 terms rounded once to bf16
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-5)
    # deterministic: a second call gives identical bits
    assert torch.equal(out.view(torch.int16), run().view(torch.int16))


# ----------------------------------------------------------------------------- failure path

def test_bounded_wait_gives_up_and_context_survives():
    moe.moe_selftest_wait_timeout(2000)  # a wait nothing releases, 2 ms limit
    st, raw = moe.moe_device_error()
    assert st == 5 and (raw & 1) and (raw >> 17) & 1
    assert moe.moe_device_error()[0] == 0  # the word was cleared
    # the context is still usable: a full stage runs and is right
    idx = synth.random_topk(6, 64, 8, 2)
    x = synth.normal_bf16(6, 1, (64, 128))
    counts, offsets, perm, inv, x_perm = moe.moe_permute(dev_i32(idx), dev_bf16(x), 8)
    assert np.array_equal(perm.cpu().numpy(), oracle.permute(idx, 8)[2])
