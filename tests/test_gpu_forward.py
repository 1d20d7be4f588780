"""End-to-end parity of moe_forward / moe_forward_ex with the oracle on the five
layer shapes, through the C ABI.

Small token counts are compared on every output element; the full-size
token counts (the ones the benchmark times, in the same launch
configuration) are compared on sampled tokens the oracle computes one by
one.  Tokens whose oracle selection margin is below 1e-4 may legitimately
pick another expert set: their choice is validated and their outputs are
left out of the element comparison.
"""
import functools

import numpy as np
import pytest
import torch

import mixture_experts_layer_06_gb300 as moe
import oracle
import synth
from synth.workloads import Workload

from gpu_util import (check_grouping, check_routing, compare_outputs, device_inputs, host_f64, make_cfg)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load_library()


# Largest token count each workload is run at here; smaller T use a prefix of
# the same x (the generator indexes x by flat position) and the same weights.
TMAX = {"tiny": 250, "mixtral": 4096, "qwen2": 512, "skew": 512, "deepseek": 8192, "mixtral22b": 4096}


@functools.lru_cache(maxsize=1)
def _full(name, alpha):
    kw = {} if alpha is None else {"alpha": alpha}
    wl = synth.workload(name, T=TMAX[name], **kw)
    inp = synth.make_inputs(wl)
    return wl, inp, device_inputs(inp)


def _inputs(name, T, alpha):
    wl, inp, d = _full(name, alpha)
    inp, d = dict(inp), dict(d)
    inp["x"] = inp["x"][:T]
    d["x"] = d["x"][:T]
    return wl.with_T(T), inp, d


def _run(wl, d):
    cfg = make_cfg(wl, d)
    out = moe.moe_forward_ex(d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k, cfg)
    st, raw = moe.moe_device_error()
    assert st == 0, f"device error word {raw:#x}"
    return out, cfg


def _sampled_tokens(T, n, seed=11):
    if T <= n:
        return np.arange(T)
    pick = np.sort(np.unique((synth.uniform01(seed, 90, 4 * n) * T).astype(np.int64)))[:n - 2]
    return np.unique(np.concatenate([[0, T - 1], pick]))


FULL_CASES = [("tiny", 128, None), ("mixtral", 1, None), ("mixtral", 32, None), ("qwen2", 128, None),
              ("skew", 128, 0.0), ("skew", 256, 1.0), ("skew", 256, 2.0)]


@pytest.mark.parametrize("name,T,alpha", FULL_CASES, ids=[f"{c[0]}-T{c[1]}-a{c[2]}" for c in FULL_CASES])
def test_forward_all_tokens(name, T, alpha):
    wl, inp, d = _inputs(name, T, alpha)
    out, cfg = _run(wl, d)
    orc = oracle.forward(inp, wl)
    gidx, gw, _ = moe.moe_route(d["x"], d["w_router"], wl.k, cfg)
    same = check_routing(wl, gidx.cpu().numpy(), gw.cpu().numpy(), orc)
    rel, mx = compare_outputs(host_f64(out)[same], orc["out"][same])
    print(f"{wl.label}: rel-L2 {rel:.2e} max-abs {mx:.2e} near-tie flips {int((~same).sum())}")
    # grouping of the GPU's own routing, and equality with the oracle's when no token flipped
    counts, offsets, perm, inv, _ = moe.moe_permute(gidx, d["x"], wl.E)
    c, o, p, i = (t.cpu().numpy() for t in (counts, offsets, perm, inv))
    check_grouping(gidx.cpu().numpy(), wl.E, c, o, p, i)
    if same.all():
        assert np.array_equal(c, orc["counts"]) and np.array_equal(p, orc["perm"])


@pytest.mark.parametrize("name,T,kw", [("tiny", 128, {}), ("qwen2", 96, {}), ("deepseek", 256, {"E": 32})],
                         ids=["tiny", "qwen2", "deepseek-E32"])
def test_forward_geglu(name, T, kw):
    """GEGLU experts (routed and shared) through the whole layer."""
    wl = synth.workload(name, T=T, activation="gelu", **kw)
    inp = synth.make_inputs(wl)
    d = device_inputs(inp)
    out, cfg = _run(wl, d)
    if name == "deepseek":
        tokens = _sampled_tokens(T, 24)
        orc = oracle.forward_tokens(inp, wl, tokens)
        gidx, gw, _ = moe.moe_route(d["x"], d["w_router"], wl.k, cfg)
        same = check_routing(wl, gidx.cpu().numpy()[tokens], gw.cpu().numpy()[tokens], orc)
        compare_outputs(host_f64(out)[tokens][same], orc["out"][same])
        return
    orc = oracle.forward(inp, wl)
    gidx, gw, _ = moe.moe_route(d["x"], d["w_router"], wl.k, cfg)
    same = check_routing(wl, gidx.cpu().numpy(), gw.cpu().numpy(), orc)
    rel, mx = compare_outputs(host_f64(out)[same], orc["out"][same])
    print(f"{wl.label}: rel-L2 {rel:.2e} max-abs {mx:.2e}")


@pytest.mark.parametrize("E,T", [(16, 96), (64, 128), (128, 200)])
def test_forward_expert_count_sweep(E, T):
    """The expert-count sweep's shapes: E experts of width 8 * 14336 / E."""
    from synth.workloads import expert_sweep
    wl = expert_sweep(E, T)
    inp = synth.make_inputs(wl)
    d = device_inputs(inp)
    out, cfg = _run(wl, d)
    orc = oracle.forward(inp, wl)
    gidx, gw, _ = moe.moe_route(d["x"], d["w_router"], wl.k, cfg)
    same = check_routing(wl, gidx.cpu().numpy(), gw.cpu().numpy(), orc)
    rel, mx = compare_outputs(host_f64(out)[same], orc["out"][same])
    print(f"{wl.label}: rel-L2 {rel:.2e} max-abs {mx:.2e}")


@functools.lru_cache(maxsize=1)
def _deepseek32():
    wl = synth.workload("deepseek", T=40, E=32)
    inp = synth.make_inputs(wl)
    return wl, inp, device_inputs(inp)


@pytest.mark.parametrize("T", [1, 3, 40])
def test_forward_deepseek_shape_decode_sizes(T):
    """DeepSeek-V3-shaped experts (32 of them, same H, F, k, group routing and
    shared expert) at decode-sized batches: K-split down projection, the
    few-warp combine, one-row tiles.  Smaller T use a prefix of the same x."""
    wl_full, inp_full, d_full = _deepseek32()
    wl = wl_full.with_T(T)
    inp, d = dict(inp_full), dict(d_full)
    inp["x"], d["x"] = inp_full["x"][:T], d_full["x"][:T]
    out, cfg = _run(wl, d)
    orc = oracle.forward(inp, wl)
    gidx, gw, _ = moe.moe_route(d["x"], d["w_router"], wl.k, cfg)
    same = check_routing(wl, gidx.cpu().numpy(), gw.cpu().numpy(), orc)
    rel, mx = compare_outputs(host_f64(out)[same], orc["out"][same])
    print(f"{wl.label}: rel-L2 {rel:.2e} max-abs {mx:.2e}")


@pytest.mark.parametrize("shape", ["k16_of_32", "one_expert", "k_equals_E"])
def test_forward_limits_and_degenerate_routing(shape):
    """The largest top-k the kernels take (16), a layer with a single expert
    (every token's one weight is 1), and k = E (every expert on every token)."""
    kw = {"k16_of_32": dict(E=32, k=16), "one_expert": dict(E=1, k=1), "k_equals_E": dict(E=8, k=8)}[shape]
    wl = Workload(shape, T=77, H=256, F=384, **kw)
    inp = synth.make_inputs(wl)
    d = device_inputs(inp)
    out, cfg = _run(wl, d)
    orc = oracle.forward(inp, wl)
    gidx, gw, _ = moe.moe_route(d["x"], d["w_router"], wl.k, cfg)
    same = check_routing(wl, gidx.cpu().numpy(), gw.cpu().numpy(), orc)
    compare_outputs(host_f64(out)[same], orc["out"][same])
    if wl.k == wl.E:  # every token picks every expert: the grouping is the identity per expert
        counts, _, _, _, _ = moe.moe_permute(gidx, d["x"], wl.E)
        assert np.all(counts.cpu().numpy() == wl.T)


def test_forward_default_entry_point_matches_ex():
    wl, inp, d = _inputs("tiny", 128, None)
    a = moe.moe_forward(d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k)
    b = moe.moe_forward_ex(d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k)
    assert moe.moe_device_error()[0] == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c = moe.moe_forward(d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k)
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))  # bitwise deterministic


@pytest.mark.parametrize("name,T", [("tiny", 64), ("qwen2", 8)])
def test_forward_replays_in_a_cuda_graph(name, T):
    """The forward issues no host synchronisation and no allocation with caller
    workspace, so it can be captured once and replayed: the replay must write
    the eager call's bits, and must follow new contents of the input buffer."""
    wl, inp, d = _inputs(name, 2 * T, None)
    cfg = make_cfg(wl, d)
    x = d["x"][:T].clone()
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(moe.moe_workspace_bytes(cfg, T, wl.H, wl.F, wl.E, wl.k), dtype=torch.uint8, device="cuda")

    def fwd():
        moe.moe_forward_ex(x, d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k, cfg, out=out, workspace=ws)

    fwd()
    torch.cuda.synchronize()
    eager = out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fwd()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fwd()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert moe.moe_device_error()[0] == 0
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    # new tokens in the captured input buffer
    x.copy_(d["x"][T:2 * T])
    g.replay()
    torch.cuda.synchronize()
    replayed = out.clone()
    fwd()
    torch.cuda.synchronize()
    assert torch.equal(replayed.view(torch.int16), out.view(torch.int16))
    assert not torch.equal(replayed.view(torch.int16), eager.view(torch.int16))


def test_forward_ragged_token_counts():
    for T in (3, 127, 129, 250):
        wl, inp, d = _inputs("tiny", T, None)
        out, cfg = _run(wl, d)
        orc = oracle.forward(inp, wl)
        gidx, gw, _ = moe.moe_route(d["x"], d["w_router"], wl.k, cfg)
        same = check_routing(wl, gidx.cpu().numpy(), gw.cpu().numpy(), orc)
        compare_outputs(host_f64(out)[same], orc["out"][same])


# Full-size token counts: the shapes and launch configuration the benchmark times.
SAMPLED_CASES = [("mixtral", 4096, None, 48), ("mixtral", 512, None, 32), ("mixtral22b", 4096, None, 24),
                 ("mixtral22b", 32, None, 32), ("qwen2", 512, None, 32),
                 ("skew", 512, 2.0, 48), ("skew", 512, 0.0, 48), ("deepseek", 512, None, 24),
                 ("deepseek", 8192, None, 24)]


@pytest.mark.parametrize("name,T,alpha,n", SAMPLED_CASES, ids=[f"{c[0]}-T{c[1]}-a{c[2]}" for c in SAMPLED_CASES])
def test_forward_full_size_sampled(name, T, alpha, n):
    wl, inp, d = _inputs(name, T, alpha)
    out, cfg = _run(wl, d)
    tokens = _sampled_tokens(T, n)
    orc = oracle.forward_tokens(inp, wl, tokens)
    gidx, gw, _ = moe.moe_route(d["x"], d["w_router"], wl.k, cfg)
    gi, gwn = gidx.cpu().numpy(), gw.cpu().numpy()
    same = check_routing(wl, gi[tokens], gwn[tokens], orc)
    rel, mx = compare_outputs(host_f64(out)[tokens][same], orc["out"][same])
    print(f"{wl.label}: {tokens.size} sampled tokens, rel-L2 {rel:.2e} max-abs {mx:.2e}")
    # properties that hold at any size: a valid stable grouping of the GPU's routing
    counts, offsets, perm, inv, _ = moe.moe_permute(gidx, d["x"], wl.E)
    check_grouping(gi, wl.E, *(t.cpu().numpy() for t in (counts, offsets, perm, inv)))
    o = host_f64(out)
    assert np.all(np.isfinite(o))
