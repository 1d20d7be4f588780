"""The CPU oracle, pinned to things other than itself.

Each check would fail on a plausible slip in the oracle: a hand-worked
closed form (dropped SiLU, swapped gate/up, transposed weight, wrong softmax
axis), brute-force enumeration of the selection (ascending instead of
descending, wrong tie rule, wrong group score), sorting-free permutation,
the identical-experts invariant, and an independently written dense
run-every-expert-then-mask forward.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth
from synth.workloads import Workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "handworked_two_experts.json")


def _bits(a):
    """Exact bf16 bits of values that are representable in bf16."""
    f = np.asarray(a, dtype=np.float32)
    b = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    assert np.array_equal(oracle.widen(b), f.astype(np.float64))
    return b


def _ev(expr):
    return eval(expr, {"__builtins__": {}}, {"exp": math.exp})


# ----------------------------------------------------------------------------- golden

@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_handworked_golden(case):
    g = json.load(open(GOLDEN))["inputs"]
    inp = {k: _bits(v) for k, v in g.items()}
    wl = Workload("hand", T=2, H=2, F=1, E=2, k=case["k"], score=case["score"],
                  renormalize=case["renormalize"], route_scale=case["route_scale"])
    r = oracle.forward(inp, wl)
    assert r["idx"].tolist() == case["idx"]
    want_w = np.array([[_ev(e) for e in row] for row in case["w"]])
    np.testing.assert_allclose(r["w"], want_w, rtol=1e-14, atol=1e-15)
    want = np.array([[_ev(e) for e in row] for row in case["out"]])
    np.testing.assert_allclose(r["out"], want, rtol=1e-13, atol=1e-15)
    assert r["counts"].tolist() == case["counts"]
    assert r["perm"].tolist() == case["perm"]
    assert r["inv"].tolist() == case["inv"]


# ----------------------------------------------------------------------------- selection

def _brute_topk(s, k):
    """Best k-subset by total score (unique for distinct scores), sorted by score."""
    best = max(itertools.combinations(range(len(s)), k), key=lambda c: sum(s[i] for i in c))
    return sorted(best, key=lambda i: (-s[i], i))


@pytest.mark.parametrize("k", [1, 2, 3, 8])
def test_topk_bruteforce(k):
    s = synth.normal_f64(1, 100 + k, (64, 8))
    idx = oracle.select_experts(s, k, oracle.Routing())
    for t in range(64):
        assert idx[t].tolist() == _brute_topk(s[t], k)


def test_topk_ties_lower_index_wins():
    s = np.array([[0.5, 0.7, 0.7, 0.1, 0.7]])
    assert oracle.select_experts(s, 2, oracle.Routing()).tolist() == [[1, 2]]
    assert oracle.select_experts(np.zeros((1, 6)), 3, oracle.Routing()).tolist() == [[0, 1, 2]]


def _brute_group_limited(s, k, n_group, topk_group, group_topn):
    E = len(s)
    size = E // n_group
    gsc = [sum(sorted(s[g * size:(g + 1) * size], reverse=True)[:group_topn]) for g in range(n_group)]
    keep = max(itertools.combinations(range(n_group), topk_group), key=lambda c: sum(gsc[g] for g in c))
    cand = [e for g in keep for e in range(g * size, (g + 1) * size)]
    return sorted(cand, key=lambda e: (-s[e], e))[:k]


def test_group_limited_bruteforce_small():
    r = oracle.Routing(score="sigmoid", n_group=4, topk_group=2, group_topn=2)
    s = 1 / (1 + np.exp(-synth.normal_f64(2, 7, (50, 16))))
    idx = oracle.select_experts(s, 3, r)
    for t in range(50):
        want = _brute_group_limited(s[t], 3, 4, 2, 2)
        # the chosen subset must also be the best-sum 3-subset among kept experts
        assert idx[t].tolist() == want


def test_group_limited_bruteforce_deepseek_shape():
    r = oracle.Routing(score="sigmoid", renormalize=True, route_scale=2.5,
                       n_group=8, topk_group=4, group_topn=2)
    s = 1 / (1 + np.exp(-synth.normal_f64(2, 8, (12, 256))))
    idx = oracle.select_experts(s, 8, r)
    for t in range(12):
        assert idx[t].tolist() == _brute_group_limited(s[t], 8, 8, 4, 2)
    # the group limit matters: plain top-8 differs for some token
    plain = oracle.select_experts(s, 8, oracle.Routing(score="sigmoid"))
    assert any(set(plain[t]) != set(idx[t]) for t in range(12))


def test_selection_margin():
    s = np.array([[0.40, 0.30, 0.2999, 0.0001], [0.5, 0.5, 0.0, 0.0]])
    m = oracle.selection_margin(s, 2, oracle.Routing())
    np.testing.assert_allclose(m, [0.0001, 0.5], rtol=1e-9)
    assert oracle.selection_margin(s, 4, oracle.Routing())[0] == np.inf


# ----------------------------------------------------------------------------- weights

def test_softmax_renorm_equals_softmax_over_selected_logits():
    logits = synth.normal_f64(3, 1, (40, 8), std=2.0)
    sc = oracle.router_scores(logits, "softmax")
    idx = oracle.select_experts(sc, 2, oracle.Routing())
    w = oracle.routing_weights(sc, idx, oracle.Routing())
    sel = np.take_along_axis(logits, idx, axis=1)
    want = np.exp(sel) / np.exp(sel).sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w, want, rtol=1e-12)


def test_softmax_is_normalised_exponential():
    logits = synth.normal_f64(3, 2, (5, 6))
    sc = oracle.router_scores(logits, "softmax")
    for t in range(5):
        z = [math.exp(v) for v in logits[t]]
        np.testing.assert_allclose(sc[t], [v / sum(z) for v in z], rtol=1e-13)
    sg = oracle.router_scores(logits, "sigmoid")
    np.testing.assert_allclose(sg, [[1 / (1 + math.exp(-v)) for v in row] for row in logits], rtol=1e-13)


@pytest.mark.parametrize("name,total", [("mixtral", 1.0), ("skew", 1.0), ("deepseek", 2.5)])
def test_weight_sums(name, total):
    wl = synth.workload(name, T=64)
    inp = synth.make_inputs(wl, with_experts=False)
    r = oracle.Routing.of(wl)
    sc = oracle.router_scores(oracle.router_logits(inp["x"], inp["w_router"], inp.get("logit_bias")), r.score)
    w = oracle.routing_weights(sc, oracle.select_experts(sc, wl.k, r), r)
    np.testing.assert_allclose(w.sum(axis=1), total, rtol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)  # slots in descending score


def test_qwen2_weights_are_raw_softmax():
    wl = synth.workload("qwen2", T=32)
    inp = synth.make_inputs(wl, with_experts=False)
    r = oracle.Routing.of(wl)
    sc = oracle.router_scores(oracle.router_logits(inp["x"], inp["w_router"]), r.score)
    idx = oracle.select_experts(sc, wl.k, r)
    w = oracle.routing_weights(sc, idx, r)
    assert np.all(w.sum(axis=1) < 1.0)
    np.testing.assert_array_equal(w, np.take_along_axis(sc, idx, axis=1))


# ----------------------------------------------------------------------------- permute

def test_permute_against_tuple_sort():
    idx = synth.random_topk(4, 300, 16, 3, alpha=1.0)
    counts, offsets, perm, inv = oracle.permute(idx, 16)
    rows = sorted(((int(idx[t, j]), t, t * 3 + j) for t in range(300) for j in range(3)))
    assert perm.tolist() == [q for (_, _, q) in rows]
    assert counts.tolist() == [sum(1 for (e, _, _) in rows if e == x) for x in range(16)]
    assert offsets[0] == 0 and offsets[-1] == 900
    assert np.array_equal(inv[perm], np.arange(900))
    assert np.array_equal(perm[inv], np.arange(900))


def test_permute_empty_and_one_hot():
    c, o, p, i = oracle.permute(np.zeros((0, 2), dtype=np.int64), 4)
    assert c.tolist() == [0, 0, 0, 0] and o.tolist() == [0] * 5 and p.size == 0
    c, o, p, i = oracle.permute(np.full((7, 1), 2), 4)
    assert c.tolist() == [0, 0, 7, 0] and p.tolist() == list(range(7))


# ----------------------------------------------------------------------------- experts

def _loop_swiglu(xr, wg, wu, wd):
    """Pure-Python SwiGLU on one row: y_i = sum_f Wd[i,f] * silu(g_f) * u_f."""
    F, H = len(wg), len(xr)
    h = []
    for f in range(F):
        g = sum(wg[f][c] * xr[c] for c in range(H))
        u = sum(wu[f][c] * xr[c] for c in range(H))
        h.append(g / (1 + math.exp(-g)) * u)
    return [sum(wd[i][f] * h[f] for f in range(F)) for i in range(len(wd))]


def _loop_geglu(xr, wg, wu, wd):
    """Pure-Python GEGLU on one row: y_i = sum_f Wd[i,f] * gelu(g_f) * u_f,
    gelu(g) = g * Phi(g) with Phi from math.erf."""
    F, H = len(wg), len(xr)
    h = []
    for f in range(F):
        g = sum(wg[f][c] * xr[c] for c in range(H))
        u = sum(wu[f][c] * xr[c] for c in range(H))
        h.append(g * 0.5 * (1 + math.erf(g / math.sqrt(2))) * u)
    return [sum(wd[i][f] * h[f] for f in range(F)) for i in range(len(wd))]


# Standard normal CDF at a few points (printed tables of the normal distribution).
_PHI = {0.0: 0.5, 1.0: 0.8413447460685429, -1.0: 0.15865525393145707, 2.0: 0.9772498680518208,
        -3.0: 0.0013498980316300946}


def _gelu_table_ok(mod) -> bool:
    x = np.array(list(_PHI))
    want = x * np.array(list(_PHI.values()))
    return bool(np.allclose(mod.activate(x, "gelu"), want, rtol=1e-13, atol=0.0))


def test_gelu_matches_normal_cdf_table():
    import oracle.moe_oracle as mo
    assert _gelu_table_ok(mo)
    x = np.array(list(_PHI))
    np.testing.assert_allclose(mo.activate(x, "silu"), [v / (1 + math.exp(-v)) for v in x], rtol=1e-15)
    with pytest.raises(ValueError):
        mo.activate(x, "relu")


def test_single_expert_is_plain_geglu_mlp():
    wl, inp = _small(T=3, H=8, F=4, E=1, k=1, activation="gelu")
    r = oracle.forward(inp, wl)
    X = oracle.widen(inp["x"]).tolist()
    wg, wu, wd = (oracle.widen(inp[n][0]).tolist() for n in ("w_gate", "w_up", "w_down"))
    for t in range(3):
        np.testing.assert_allclose(r["out"][t], _loop_geglu(X[t], wg, wu, wd), rtol=1e-12, atol=1e-14)


def _small(T, H, F, E, k, seed=5, **kw):
    wl = Workload("small", T=T, H=H, F=F, E=E, k=k, seed=seed, **kw)
    s = seed
    inp = {"x": synth.normal_bf16(s, 0, (T, H)),
           "w_router": synth.normal_bf16(s, 1, (E, H), std=0.3),
           "w_gate": synth.normal_bf16(s, 2, (E, F, H), std=0.3),
           "w_up": synth.normal_bf16(s, 3, (E, F, H), std=0.3),
           "w_down": synth.normal_bf16(s, 4, (E, H, F), std=0.3)}
    if wl.F_shared:
        inp["ws_gate"] = synth.normal_bf16(s, 5, (wl.F_shared, H), std=0.3)
        inp["ws_up"] = synth.normal_bf16(s, 6, (wl.F_shared, H), std=0.3)
        inp["ws_down"] = synth.normal_bf16(s, 7, (H, wl.F_shared), std=0.3)
    if wl.shared_gate:
        inp["w_shared_gate"] = synth.normal_bf16(s, 8, (H,), std=0.3)
    if wl.alpha is not None:
        inp["logit_bias"] = synth.zipf_logit_bias(s, E, wl.alpha)
    return wl, inp


def test_single_expert_is_plain_swiglu_mlp():
    wl, inp = _small(T=3, H=8, F=4, E=1, k=1)
    r = oracle.forward(inp, wl)
    X = oracle.widen(inp["x"]).tolist()
    wg, wu, wd = (oracle.widen(inp[n][0]).tolist() for n in ("w_gate", "w_up", "w_down"))
    for t in range(3):
        np.testing.assert_allclose(r["out"][t], _loop_swiglu(X[t], wg, wu, wd), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["w"], 1.0)


def test_shared_expert_closed_form():
    wl, inp = _small(T=3, H=8, F=4, E=4, k=2, F_shared=6, shared_gate=True, renormalize=False)
    inp["w_down"] = np.zeros_like(inp["w_down"])
    r = oracle.forward(inp, wl)
    X = oracle.widen(inp["x"]).tolist()
    ws = oracle.widen(inp["w_shared_gate"]).tolist()
    wg, wu, wd = (oracle.widen(inp[n]).tolist() for n in ("ws_gate", "ws_up", "ws_down"))
    for t in range(3):
        scale = 1 / (1 + math.exp(-sum(a * b for a, b in zip(X[t], ws))))
        want = [scale * v for v in _loop_swiglu(X[t], wg, wu, wd)]
        np.testing.assert_allclose(r["out"][t], want, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("variant", ["mixtral", "deepseek"])
def test_identical_experts_make_routing_irrelevant(variant):
    if variant == "mixtral":
        wl, inp = _small(T=20, H=16, F=8, E=8, k=2)
        scale = 1.0
    else:
        wl, inp = _small(T=20, H=16, F=8, E=16, k=4, score="sigmoid", route_scale=2.5,
                         n_group=4, topk_group=2, group_topn=2)
        scale = 2.5
    for n in ("w_gate", "w_up", "w_down"):
        inp[n] = np.repeat(inp[n][:1], wl.E, axis=0)
    r = oracle.forward(inp, wl)
    X = oracle.widen(inp["x"]).tolist()
    wg, wu, wd = (oracle.widen(inp[n][0]).tolist() for n in ("w_gate", "w_up", "w_down"))
    for t in range(20):
        np.testing.assert_allclose(r["out"][t], [scale * v for v in _loop_swiglu(X[t], wg, wu, wd)],
                                   rtol=1e-11, atol=1e-13)


def test_zero_down_projection_gives_zero():
    wl, inp = _small(T=10, H=16, F=8, E=4, k=2)
    inp["w_down"] = np.zeros_like(inp["w_down"])
    assert np.all(oracle.forward(inp, wl)["out"] == 0.0)


def test_one_hot_bias_routes_everything_to_one_expert():
    wl, inp = _small(T=37, H=16, F=8, E=8, k=1, alpha=0.0)
    bias = np.zeros(8, dtype=np.float32)
    bias[3] = 30.0
    inp["logit_bias"] = bias
    r = oracle.forward(inp, wl)
    assert r["counts"].tolist() == [0, 0, 0, 37, 0, 0, 0, 0]
    assert r["perm"].tolist() == list(range(37))
    np.testing.assert_allclose(r["w"], 1.0)


def test_equal_logits_pick_first_experts():
    wl, inp = _small(T=5, H=16, F=8, E=8, k=3)
    inp["w_router"] = np.zeros_like(inp["w_router"])
    r = oracle.forward(inp, wl)
    assert r["idx"].tolist() == [[0, 1, 2]] * 5
    np.testing.assert_allclose(r["w"], 1 / 3)


def test_k_equals_E_is_dense_softmax_mixture():
    wl, inp = _small(T=6, H=16, F=8, E=4, k=4)
    r = oracle.forward(inp, wl)
    X = oracle.widen(inp["x"])
    p = np.exp(X @ oracle.widen(inp["w_router"]).T)
    p /= p.sum(axis=1, keepdims=True)
    Xl = X.tolist()
    for t in range(6):
        want = np.zeros(16)
        for e in range(4):
            wg, wu, wd = (oracle.widen(inp[n][e]).tolist() for n in ("w_gate", "w_up", "w_down"))
            want += p[t, e] * np.array(_loop_swiglu(Xl[t], wg, wu, wd))
        np.testing.assert_allclose(r["out"][t], want, rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------------------- dense

@pytest.mark.parametrize("shape", ["tiny", "qwen2_like", "deepseek_like", "skew_like", "geglu_deepseek_like"])
def test_dense_masked_matches_forward(shape):
    if shape == "tiny":
        wl = synth.workload("tiny")
        inp = synth.make_inputs(wl)
    elif shape == "qwen2_like":
        wl, inp = _small(T=40, H=64, F=32, E=16, k=4, renormalize=False, F_shared=48, shared_gate=True)
    elif shape == "deepseek_like":
        wl, inp = _small(T=40, H=64, F=32, E=32, k=4, score="sigmoid", route_scale=2.5,
                         n_group=8, topk_group=4, group_topn=2, F_shared=32)
    elif shape == "skew_like":
        wl, inp = _small(T=40, H=64, F=32, E=16, k=4, alpha=2.0)
    else:
        wl, inp = _small(T=40, H=64, F=32, E=32, k=4, score="sigmoid", route_scale=2.5,
                         n_group=8, topk_group=4, group_topn=2, F_shared=32, activation="gelu")
    r = oracle.forward(inp, wl)
    dense = oracle.dense_masked_forward(inp, wl)
    scale = np.abs(r["out"]).max()
    np.testing.assert_allclose(r["out"], dense, rtol=1e-10, atol=1e-12 * scale)


def test_forward_tokens_matches_forward():
    wl = synth.workload("skew", T=96, alpha=1.0)
    inp = synth.make_inputs(wl)
    full = oracle.forward(inp, wl)
    toks = [0, 5, 17, 95, 40]
    part = oracle.forward_tokens(inp, wl, toks)
    np.testing.assert_array_equal(part["idx"], full["idx"][toks])
    np.testing.assert_allclose(part["out"], full["out"][toks], rtol=1e-12, atol=1e-14)
    gen = oracle.forward_tokens(inp, wl, toks, expert_weights=lambda n, e: synth.expert_slice(wl, n, e))
    np.testing.assert_array_equal(gen["out"], part["out"])


def test_invariants_on_real_workloads():
    for name in ("tiny", "skew", "qwen2"):
        wl = synth.workload(name, T=64)
        inp = synth.make_inputs(wl, with_experts=False)
        r = oracle.Routing.of(wl)
        sc = oracle.router_scores(oracle.router_logits(inp["x"], inp["w_router"], inp.get("logit_bias")), r.score)
        idx = oracle.select_experts(sc, wl.k, r)
        assert all(len(set(row)) == wl.k for row in idx.tolist())
        c, o, p, i = oracle.permute(idx, wl.E)
        assert c.sum() == 64 * wl.k
        assert np.array_equal(np.sort(p), np.arange(64 * wl.k))


class _CountingMemory:
    """A global memory that counts the bytes of every 16-bit tensor moved
    through it, stored rounded to bf16-like width (2 bytes per element)."""

    def __init__(self):
        self.arrays, self.read, self.written = {}, 0, 0

    def store(self, name, a):
        self.arrays[name] = np.array(a, dtype=np.float64)
        self.written += 2 * a.size

    def load(self, name):
        a = self.arrays[name]
        self.read += 2 * a.size
        return a

    @property
    def total(self):
        return self.read + self.written


def _run_unfused(x, wg, wu):
    """Gate projection, up projection and activation as three passes through
    global memory; returns (bytes before the activation's h write, bytes
    with it, h)."""
    m = _CountingMemory()
    m.arrays["x"] = x  # already resident: the input itself is not an intermediate
    m.store("g", m.load("x") @ wg.T)          # gate projection kernel
    m.store("u", m.load("x") @ wu.T)          # up projection kernel
    g, u = m.load("g"), m.load("u")           # activation kernel
    h = g / (1.0 + np.exp(-g)) * u
    before_h = m.total
    m.store("h", h)
    return before_h, m.total, h


def _run_fused(x, wg, wu):
    m = _CountingMemory()
    m.arrays["x"] = x
    xt = m.load("x")                          # one shared load of the input rows
    g, u = xt @ wg.T, xt @ wu.T               # both projections from it, in registers
    h = g / (1.0 + np.exp(-g)) * u
    m.store("h", h)
    return m.total, h


@pytest.mark.parametrize("T,F,d", [(3, 5, 7), (16, 40, 12), (1, 9, 2), (11, 4, 30)])
def test_traffic_model_against_executed_sequences(T, F, d):
    """The byte model equals the bytes that executed fused and unfused SwiGLU
    passes move through a counting memory (distinct T, F, d, so a dropped
    term, a swapped dimension or a wrong coefficient fails)."""
    rng = np.random.default_rng(T * 100 + F)
    x, wg, wu = rng.normal(size=(T, d)), rng.normal(size=(F, d)), rng.normal(size=(F, d))
    before_h, with_h, h_unf = _run_unfused(x, wg, wu)
    fused, h_f = _run_fused(x, wg, wu)
    np.testing.assert_allclose(h_unf, h_f, rtol=1e-12)  # both sequences compute the same h
    np.testing.assert_allclose(h_f, oracle.activate(x @ wg.T) * (x @ wu.T), rtol=1e-12)
    m = oracle.traffic_model_bytes(T=T, F=F, d=d)
    assert m["unfused"] == before_h
    assert m["unfused_with_h"] == with_h
    assert m["fused"] == fused
    assert m["saving"] == pytest.approx(1 - fused / before_h)
    assert m["saving_with_h"] == pytest.approx(1 - fused / with_h)


def test_traffic_model_saving_is_not_the_quoted_35_percent():
    m = oracle.traffic_model_bytes(T=512, F=14336, d=4096)  # Mixtral-8x7B expert widths
    assert 0.70 < m["saving"] < 0.73 and 0.76 < m["saving_with_h"] < 0.79


# ----------------------------------------------------------------------------- teacher forcing

def test_teacher_forced_choice_reweights_from_oracle_scores():
    """A forced expert set is run with the oracle's own scores of those
    experts: forcing the oracle's own choice changes nothing, and forcing
    another set equals the brute-force mixture of those experts."""
    wl, inp = _small(T=6, H=32, F=16, E=8, k=2)
    free = oracle.forward(inp, wl)
    same = oracle.forward(inp, wl, forced_idx=free["idx"])
    np.testing.assert_array_equal(same["out"], free["out"])
    forced = np.array([[7, 0], [1, 2], [3, 4], [5, 6], [0, 1], [2, 7]])
    r = oracle.forward(inp, wl, forced_idx=forced)
    xf = oracle.widen(inp["x"])
    s = free["scores"]
    for t in range(6):
        w = s[t, forced[t]] / s[t, forced[t]].sum()
        want = sum(w[j] * oracle.swiglu_expert(xf[t:t + 1], inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e])[0]
                   for j, e in enumerate(forced[t]))
        np.testing.assert_allclose(r["out"][t], want, rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(r["margin"], free["margin"])  # the margin stays the oracle's own
    part = oracle.forward_tokens(inp, wl, [4, 1], forced_idx=forced[[4, 1]])
    np.testing.assert_allclose(part["out"], r["out"][[4, 1]], rtol=1e-12, atol=1e-15)


# ----------------------------------------------------------------------------- planted mistakes

def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant typical slips in the oracle (CPU only) and check a pin fails."""
    import oracle.moe_oracle as mo
    case = json.load(open(GOLDEN))["cases"][1]

    def golden_ok():
        try:
            test_handworked_golden(case)
            return True
        except AssertionError:
            return False

    assert golden_ok()
    orig = mo.swiglu_expert
    monkeypatch.setattr(mo, "swiglu_expert",
                        lambda x, g, u, d, act="silu": (x @ mo.widen(g).T * (x @ mo.widen(u).T)) @ mo.widen(d).T)
    assert not golden_ok()  # SiLU dropped
    monkeypatch.setattr(mo, "swiglu_expert", lambda x, g, u, d, act="silu": orig(x, u, g, d, act))
    assert not golden_ok()  # gate and up swapped
    monkeypatch.setattr(mo, "swiglu_expert", orig)
    orig_act = mo.activate

    def gelu_tanh(g, act="silu"):
        if act != "gelu":
            return orig_act(g, act)
        return 0.5 * g * (1 + np.tanh(np.sqrt(2 / np.pi) * (g + 0.044715 * g ** 3)))

    monkeypatch.setattr(mo, "activate", gelu_tanh)
    assert not _gelu_table_ok(mo)  # tanh approximation instead of the exact GELU
    monkeypatch.setattr(mo, "activate", lambda g, act="silu": orig_act(g, "silu"))
    assert not _gelu_table_ok(mo)  # activation ignored
    monkeypatch.setattr(mo, "activate", orig_act)
    monkeypatch.setattr(mo, "_descending", lambda v: np.argsort(v, kind="stable"))
    assert not golden_ok()  # ascending selection
