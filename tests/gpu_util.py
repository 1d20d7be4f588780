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


def compare_outputs(gpu_out: np.ndarray, orc_out: np.ndarray, what: str = "out"):
    """rel-L2 and max-abs over all compared elements (both in float64)."""
    diff = gpu_out - orc_out
    rel = np.linalg.norm(diff) / max(np.linalg.norm(orc_out), 1e-300)
    mx = float(np.abs(diff).max()) if diff.size else 0.0
    assert rel <= REL_L2_TOL, f"{what}: rel-L2 {rel:.3e} > {REL_L2_TOL}"
    assert mx <= MAX_ABS_TOL, f"{what}: max-abs {mx:.3e} > {MAX_ABS_TOL}"
    return rel, mx


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
