"""End-to-end parity of moe_forward / moe_forward_ex with the oracle, through
the C ABI, at every (layer, T, alpha) point the layer is built for.

Every point checks the routing of all tokens (exact expert sets outside the
1e-4 near-tie margin), the grouping bit-exact against the oracle's, and the
output rows against the oracle run teacher-forced on the GPU's expert set for
the few near-tie tokens whose set differs, so no output row is exempt.  Where
the oracle finishes the whole batch in seconds every row is compared; at the
largest token counts (the shapes and launch configuration the benchmark
times) the compared rows are those on every token-tile seam and expert
segment end of the GPU's grouping, plus seeded random ones.
"""
import functools

import numpy as np
import pytest
import torch

import mixture_experts_layer_06_gb300 as moe
import oracle
import synth
from synth.workloads import SKEW_ALPHAS, T_SWEEP, Workload

from gpu_util import check_forward, device_inputs, make_cfg, tile_targeted_tokens

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


# Every (layer, T, alpha) point of the five layer shapes.  "all": every output
# row; "tiles": tile-seam and segment-end rows (the oracle cannot run the whole
# batch in seconds).
def _points():
    pts = [("tiny", 128, None, "all")]
    pts += [("mixtral", T, None, "tiles" if T > 512 else "all") for T in T_SWEEP["mixtral"]]
    pts += [("qwen2", T, None, "all") for T in T_SWEEP["qwen2"]]
    pts += [("skew", T, a, "all") for a in SKEW_ALPHAS for T in T_SWEEP["skew"]]
    pts += [("deepseek", T, None, "tiles" if T > 512 else "all") for T in T_SWEEP["deepseek"]]
    return pts


POINTS = _points()


@pytest.mark.parametrize("name,T,alpha,mode", POINTS, ids=[f"{p[0]}-T{p[1]}" + (f"-a{p[2]:g}" if p[2] is not None
                                                                                  else "") for p in POINTS])
def test_forward_config_point(name, T, alpha, mode):
    wl, inp, d = _inputs(name, T, alpha)
    out, cfg = _run(wl, d)
    if mode == "all":
        tokens = None
    else:
        # at most 6 rows per expert segment on the 256-expert layer
        cap = 6 if wl.E > 64 else None
        tokens = lambda c, p: tile_targeted_tokens(c, p, wl.k, T, n_random=16, cap_per_expert=cap)  # noqa: E731
    r = check_forward(wl, inp, d, out, cfg, tokens=tokens)
    print(f"{wl.label}: {r['rows_compared']} rows, rel-L2 {r['rel_l2']:.2e} max-abs {r['max_abs']:.2e} "
          f"(max |out| {r['max_abs_out']:.1f}), near-tie flips {r['flipped']}, routing identical to the "
          f"oracle's: {r['identical_routing']}")


# The Mixtral-8x22B shape (second Mixtral layer of the review's tables).  Its
# outputs reach |out| >= 16, where the bf16 output's rounding alone exceeds
# 5e-2: the element-wise bound scales with the value (compare_outputs).
@pytest.mark.parametrize("T", [32, 4096])
def test_forward_mixtral22b(T):
    wl, inp, d = _inputs("mixtral22b", T, None)
    out, cfg = _run(wl, d)
    tokens = None if T <= 32 else (lambda c, p: tile_targeted_tokens(c, p, wl.k, T, n_random=16))
    r = check_forward(wl, inp, d, out, cfg, tokens=tokens, scaled=True)
    print(f"{wl.label}: {r['rows_compared']} rows, rel-L2 {r['rel_l2']:.2e} max-abs {r['max_abs']:.2e} "
          f"(max |out| {r['max_abs_out']:.1f})")


@pytest.mark.parametrize("name,T,kw", [("tiny", 128, {}), ("qwen2", 96, {}), ("deepseek", 256, {"E": 32})],
                         ids=["tiny", "qwen2", "deepseek-E32"])
def test_forward_geglu(name, T, kw):
    """GEGLU experts (routed and shared) through the whole layer."""
    wl = synth.workload(name, T=T, activation="gelu", **kw)
    inp = synth.make_inputs(wl)
    d = device_inputs(inp)
    out, cfg = _run(wl, d)
    r = check_forward(wl, inp, d, out, cfg)
    print(f"{wl.label}: rel-L2 {r['rel_l2']:.2e} max-abs {r['max_abs']:.2e}")


@pytest.mark.parametrize("E,T", [(16, 96), (64, 128), (128, 200)])
def test_forward_expert_count_sweep(E, T):
    """The expert-count sweep's shapes: E experts of width 8 * 14336 / E."""
    from synth.workloads import expert_sweep
    wl = expert_sweep(E, T)
    inp = synth.make_inputs(wl)
    d = device_inputs(inp)
    out, cfg = _run(wl, d)
    r = check_forward(wl, inp, d, out, cfg)
    print(f"{wl.label}: rel-L2 {r['rel_l2']:.2e} max-abs {r['max_abs']:.2e}")


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
    r = check_forward(wl, inp, d, out, cfg)
    print(f"{wl.label}: rel-L2 {r['rel_l2']:.2e} max-abs {r['max_abs']:.2e}")


@pytest.mark.parametrize("shape", ["k16_of_32", "one_expert", "k_equals_E"])
def test_forward_limits_and_degenerate_routing(shape):
    """The largest top-k the kernels take (16), a layer with a single expert
    (every token's one weight is 1), and k = E (every expert on every token)."""
    kw = {"k16_of_32": dict(E=32, k=16), "one_expert": dict(E=1, k=1), "k_equals_E": dict(E=8, k=8)}[shape]
    wl = Workload(shape, T=77, H=256, F=384, **kw)
    inp = synth.make_inputs(wl)
    d = device_inputs(inp)
    out, cfg = _run(wl, d)
    r = check_forward(wl, inp, d, out, cfg)
    if wl.k == wl.E:  # every token picks every expert: every expert gets every token
        assert np.all(r["counts"] == wl.T)


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


@pytest.mark.parametrize("T", [3, 127, 129, 250])
def test_forward_ragged_token_counts(T):
    wl, inp, d = _inputs("tiny", T, None)
    out, cfg = _run(wl, d)
    check_forward(wl, inp, d, out, cfg)


def test_forward_workspace_grows_safely_across_streams():
    """moe_forward's one library workspace, grown by calls queued on two
    streams in turn without a host synchronisation in between: each call must
    still see a workspace of its own (the library orders the calls), so every
    output equals moe_forward_ex's with a private workspace."""
    wl, inp, d = _inputs("tiny", 250, None)
    streams = (torch.cuda.Stream(), torch.cuda.Stream())
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = []
    for i, T in enumerate((8, 40, 96, 250, 33)):
        s = streams[i % 2]
        o = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
        s.wait_stream(torch.cuda.current_stream())  # o's allocation
        moe.moe_forward(d["x"][:T], d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k, out=o, stream=s)
        outs.append((T, o))
    torch.cuda.synchronize()
    assert moe.moe_device_error()[0] == 0
    for T, o in outs:
        ref = moe.moe_forward_ex(d["x"][:T], d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16)), T


@pytest.mark.parametrize("name,T,kw", [("tiny", 128, {}), ("qwen2", 64, {}), ("deepseek", 40, {"E": 32}),
                                       ("mixtral", 1, {})], ids=["tiny", "qwen2", "deepseek-E32", "mixtral-T1"])
def test_forward_launch_count_matches_the_query(name, T, kw):
    """The number of kernels the library launches for one forward (counted as
    they are launched) equals what moe_forward_launches reports for it."""
    if name == "mixtral":
        wl, inp, d = _inputs(name, T, None)
    else:
        wl = synth.workload(name, T=T, **kw)
        d = device_inputs(synth.make_inputs(wl))
    cfg = make_cfg(wl, d)
    want = moe.moe_forward_launches(cfg, T, wl.H, wl.F, wl.E, wl.k)
    before = moe.moe_launches_issued()
    moe.moe_forward_ex(d["x"][:T], d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k, cfg)
    assert moe.moe_launches_issued() - before == want > 0
    assert moe.moe_device_error()[0] == 0


@pytest.mark.parametrize("name,T,alpha", [("skew", 1, 2.0), ("skew", 5, 2.0), ("skew", 8, 0.0), ("mixtral", 8, None),
                                          ("tiny", 7, None)], ids=["skew-T1-a2", "skew-T5-a2", "skew-T8-a0",
                                                                   "mixtral-T8", "tiny-T7"])
def test_forward_decode_sizes_one_launch_routing(name, T, alpha):
    """Decode-sized batches whose router weights are small route and group the
    tokens in one launch (logits on the CUDA cores, the logit bias included):
    routing, grouping and outputs against the oracle, and the launch count."""
    wl, inp, d = _inputs(name, T, alpha)
    cfg = make_cfg(wl, d)
    before = moe.moe_launches_issued()
    out = moe.moe_forward_ex(d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k, cfg)
    assert moe.moe_launches_issued() - before == moe.moe_forward_launches(cfg, T, wl.H, wl.F, wl.E, wl.k) == 4
    assert moe.moe_device_error()[0] == 0
    r = check_forward(wl, inp, d, out, cfg)
    print(f"{wl.label}: rel-L2 {r['rel_l2']:.2e} max-abs {r['max_abs']:.2e}")
