"""Helpers shared by the GPU parity tests: moving generator bits to the device,
building the library config, and comparing against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import mixture_experts_layer_06_gb300 as moe
import oracle

NEAR_TIE = 1e-4  # oracle k-th/(k+1)-th score gap below which either choice is correct
REL_L2_TOL = 1e-2
MAX_ABS_TOL = 5e-2


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    """bf16 bit patterns (uint16) -> CUDA bfloat16 tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to("cuda").view(torch.bfloat16)


def dev_f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda")


def dev_f16(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to("cuda")


def dev_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to("cuda")


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return oracle.widen(host_bits(t))
    return t.double().cpu().numpy()


def device_inputs(inp: dict) -> dict:
    d = {}
    for k, v in inp.items():
        d[k] = dev_f32(v) if k == "logit_bias" else dev_bf16(v)
    return d


def make_cfg(wl, d: dict) -> moe.MoeConfig:
    return moe.MoeConfig.make(score=wl.score, renormalize=wl.renormalize, route_scale=wl.route_scale,
                              n_group=wl.n_group, topk_group=wl.topk_group, group_topn=wl.group_topn,
                              logit_bias=d.get("logit_bias"), ws_gate=d.get("ws_gate"), ws_up=d.get("ws_up"),
                              ws_down=d.get("ws_down"), w_shared_gate=d.get("w_shared_gate"),
                              activation=wl.activation)


def candidate_kth(scores_row: np.ndarray, wl) -> float:
    """The oracle's k-th best candidate score of one token."""
    r = oracle.Routing.of(wl)
    idx = oracle.select_experts(scores_row[None, :], wl.k, r)[0]
    return float(scores_row[idx[-1]])


def check_routing(wl, gpu_idx: np.ndarray, gpu_w: np.ndarray, orc: dict) -> np.ndarray:
    """Compare the GPU's selection with the oracle's.

    Tokens whose selection margin exceeds NEAR_TIE must pick exactly the
    oracle's experts; the slot order must be descending in oracle score.
    Near-tie tokens may pick another valid set: every chosen expert must be
    within NEAR_TIE of the oracle's k-th score and the k ids distinct.
    Weights are compared per expert where the sets agree.  Returns the mask
    of tokens whose sets agree.
    """
    k = wl.k
    o_idx, sc, margin = orc["idx"], orc["scores"], orc["margin"]
    same = np.all(np.sort(gpu_idx, axis=1) == np.sort(o_idx, axis=1), axis=1)
    sure = margin > NEAR_TIE
    bad = np.nonzero(sure & ~same)[0]
    assert bad.size == 0, f"{bad.size} tokens with a clear margin picked other experts, e.g. token {bad[:5]}"
    for t in np.nonzero(~same)[0]:
        assert len(set(gpu_idx[t].tolist())) == k
        kth = candidate_kth(sc[t], wl)
        assert np.all(sc[t, gpu_idx[t]] >= kth - NEAR_TIE), f"token {t}: invalid near-tie choice"
    # slot order: descending oracle score (ties within 1e-6 may swap)
    s_sel = np.take_along_axis(sc, gpu_idx.astype(np.int64), axis=1)
    assert np.all(np.diff(s_sel, axis=1) <= 1e-6)
    # weights, matched by expert id
    rows = np.nonzero(same)[0]
    if rows.size:
        go = np.argsort(gpu_idx[rows], axis=1)
        oo = np.argsort(o_idx[rows], axis=1)
        gw = np.take_along_axis(gpu_w[rows], go, axis=1)
        ow = np.take_along_axis(orc["w"][rows], oo, axis=1)
        np.testing.assert_allclose(gw, ow, rtol=2e-5, atol=2e-6)
    return same


def compare_outputs(gpu_out: np.ndarray, orc_out: np.ndarray, what: str = "out", scaled: bool = False):
    """rel-L2 and max-abs over all compared elements (both in float64).

    The five layer shapes use the fixed bounds (rel-L2 1e-2, max-abs 5e-2).
    ``scaled`` (the other shapes, whose outputs reach |out| >= 16, where the
    bf16 output's own rounding alone can cost 2^-8 |out| > 5e-2): element by
    element |gpu - oracle| <= max(5e-2, 2^-8 |oracle| + 2e-2), i.e. half a bf16
    ulp of the value plus the computation's own error budget.
    """
    diff = gpu_out - orc_out
    rel = np.linalg.norm(diff) / max(np.linalg.norm(orc_out), 1e-300)
    mx = float(np.abs(diff).max()) if diff.size else 0.0
    assert rel <= REL_L2_TOL, f"{what}: rel-L2 {rel:.3e} > {REL_L2_TOL}"
    if scaled:
        bound = np.maximum(MAX_ABS_TOL, 2.0 ** -8 * np.abs(orc_out) + 2e-2)
        worst = np.unravel_index(np.argmax(np.abs(diff) - bound), diff.shape) if diff.size else None
        assert np.all(np.abs(diff) <= bound), \
            f"{what}: |diff| {abs(diff[worst]):.3e} > {bound[worst]:.3e} at |oracle| {abs(orc_out[worst]):.3f}"
    else:
        assert mx <= MAX_ABS_TOL, f"{what}: max-abs {mx:.3e} > {MAX_ABS_TOL} (max |oracle| " \
                                  f"{float(np.abs(orc_out).max()):.2f})"
    return rel, mx


def seam_rows(counts, boxes=(512, 256, 128, 64), cap_per_expert=None) -> np.ndarray:
    """Grouped rows where a token-tile bug would show: the first and last row
    of every expert segment, and the rows on both sides of every boundary of
    the balanced token tiles (ceil(r / box) tiles of equal rows rounded up to
    16) an expert with r rows gets under each token box in ``boxes``.  With a
    cap, an expert keeps its first rows in that order (ends, then the seams
    of the larger boxes first)."""
    rows = []
    off = 0
    for r in np.asarray(counts, dtype=np.int64).tolist():
        if r > 0:
            mine = [off, off + r - 1]
            for bn in boxes:
                ntb = -(-r // bn)
                if ntb < 2:
                    continue
                tr = -(-(-(-r // ntb)) // 16) * 16
                for b in range(tr, r, tr):
                    mine += [off + b, off + b - 1]
            mine = list(dict.fromkeys(mine))
            if cap_per_expert is not None:
                mine = mine[:cap_per_expert]
            rows.extend(mine)
        off += r
    return np.unique(np.asarray(rows, dtype=np.int64))


def tile_targeted_tokens(counts, perm, k, T, n_random=16, boxes=(512, 256, 128, 64), cap_per_expert=None,
                         seed=11) -> np.ndarray:
    """Tokens whose grouped rows sit on tile seams and segment ends (from the
    GPU's own grouping: which rows are checked, not what they should hold),
    plus the first and last token and n_random seeded random ones."""
    rows = seam_rows(counts, boxes, cap_per_expert)
    toks = np.asarray(perm)[rows] // k
    import synth
    rnd = (synth.uniform01(seed, 90, n_random) * T).astype(np.int64)
    return np.unique(np.concatenate([toks, rnd, [0, T - 1]]).astype(np.int64))


def check_forward(wl, inp: dict, d: dict, out: torch.Tensor, cfg, tokens=None, orc_route=None,
                  scaled=False) -> dict:
    """Parity of one layer forward with the oracle.

    1. Routing of every token (check_routing).
    2. Grouping: counts / offsets / perm / inv of the GPU's routing bit-exact
       against the oracle's grouping of the GPU's indices, and against the
       oracle's own grouping when every token picked the oracle's experts in
       the oracle's slot order.
    3. Output rows of ``tokens`` (every token when None; a callable is given
       the GPU's counts and perm and returns the tokens) against the oracle
       teacher-forced on the GPU's expert set for the tokens whose set
       differs (near ties): their weights are the oracle's own scores of the
       GPU's experts.  No row is left out.
    Returns the statistics.
    """
    if tokens is not None and not callable(tokens) and len(tokens) == 0:
        raise ValueError("no tokens to compare")
    gidx_t, gw_t, _ = moe.moe_route(d["x"], d["w_router"], wl.k, cfg)
    gidx, gw = gidx_t.cpu().numpy().astype(np.int64), gw_t.cpu().numpy()
    orc = orc_route if orc_route is not None else oracle.route(inp, wl)
    same = check_routing(wl, gidx, gw, orc)
    counts, offsets, perm, inv, _ = moe.moe_permute(gidx_t, d["x"], wl.E)
    c, o, p, i = (t.cpu().numpy().astype(np.int64) for t in (counts, offsets, perm, inv))
    check_grouping(gidx, wl.E, c, o, p, i)
    for got, want in zip((c, o, p, i), oracle.permute(gidx, wl.E)):
        assert np.array_equal(got, want)
    identical = np.array_equal(gidx, orc["idx"])
    if identical:
        for got, want in zip((c, o, p, i), oracle.permute(orc["idx"], wl.E)):
            assert np.array_equal(got, want)
    forced = np.where(same[:, None], orc["idx"], gidx)
    if callable(tokens):
        tokens = tokens(c, p)
    if tokens is None:
        ref = oracle.forward(inp, wl, forced_idx=forced)["out"]
        got_out = host_f64(out)
    else:
        tokens = np.asarray(tokens, dtype=np.int64)
        ref = oracle.forward_tokens(inp, wl, tokens, forced_idx=forced[tokens])["out"]
        got_out = host_f64(out)[tokens]
    assert np.all(np.isfinite(got_out))
    rel, mx = compare_outputs(got_out, ref, scaled=scaled)
    return {"rel_l2": rel, "max_abs": mx, "max_abs_out": float(np.abs(ref).max()), "flipped": int((~same).sum()), "identical_routing": identical,
            "rows_compared": int(got_out.shape[0]), "counts": c, "perm": p}


def check_grouping(gpu_idx: np.ndarray, E: int, counts, offsets, perm, inv):
    """Properties of a correct stable grouping of the GPU's own routing."""
    T, k = gpu_idx.shape
    flat = gpu_idx.reshape(-1).astype(np.int64)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(np.sort(perm), np.arange(T * k))
    assert np.array_equal(inv[perm], np.arange(T * k))
    e_of_row = flat[perm]
    assert np.all(np.diff(e_of_row) >= 0)
    same_e = np.diff(e_of_row) == 0
    assert np.all(np.diff(perm // k)[same_e] > 0)  # token order inside an expert
