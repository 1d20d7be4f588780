"""Seeded synthetic inputs for the MoE layer forward (oracle side and GPU side).

This module holds no arithmetic of the MoE method.  It turns a workload
description (shapes, routing variant, seed) into the bf16 bit patterns that
both the CPU oracle and the CUDA path read, so that the two see identical
inputs.  The generator itself is plain C (``synth.c``: SplitMix64 counter form
+ Box-Muller, rounded to bf16 by round-to-nearest-even), compiled with gcc on
first use.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .workloads import Workload, WORKLOADS, workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# Stream numbers: one independent counter-based stream per tensor.
STREAM_X, STREAM_WR, STREAM_WG, STREAM_WU, STREAM_WD = 0, 1, 2, 3, 4
STREAM_WSG, STREAM_WSU, STREAM_WSD, STREAM_WSGATE = 5, 6, 7, 8
STREAM_SKEW_PERM = 9
STREAM_TOPK = 10
STREAM_MISC = 11


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so (gcc, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, p = ctypes.c_uint64, ctypes.c_void_p
            lib.synth_mix64.restype = u64
            lib.synth_mix64.argtypes = [u64]
            lib.synth_stream_key.restype = u64
            lib.synth_stream_key.argtypes = [u64, u64]
            lib.synth_f32_to_bf16.restype = ctypes.c_uint16
            lib.synth_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.synth_normal_bf16.restype = None
            lib.synth_normal_bf16.argtypes = [u64, u64, u64, u64, ctypes.c_double, ctypes.c_double, p]
            lib.synth_normal_f64.restype = None
            lib.synth_normal_f64.argtypes = [u64, u64, u64, u64, ctypes.c_double, ctypes.c_double, p]
            lib.synth_u64.restype = None
            lib.synth_u64.argtypes = [u64, u64, u64, u64, p]
            lib.synth_splitmix64_raw.restype = None
            lib.synth_splitmix64_raw.argtypes = [u64, u64, p]
            _lib = lib
    return _lib


def normal_bf16(seed: int, stream: int, shape, std: float = 1.0, mean: float = 0.0,
                start: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of mean + std * N(0,1), element i = index start+i."""
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.size == n and out.flags.c_contiguous
    if n:
        _load().synth_normal_bf16(seed, stream, start, n, mean, std, out.ctypes.data)
    return out


def normal_f64(seed: int, stream: int, shape, std: float = 1.0, mean: float = 0.0,
               start: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(shape, dtype=np.float64)
    if n:
        _load().synth_normal_f64(seed, stream, start, n, mean, std, out.ctypes.data)
    return out


def u64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    if n:
        _load().synth_u64(seed, stream, start, n, out.ctypes.data)
    return out


def uniform01(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """Doubles in [0, 1): top 53 bits of each 64-bit output times 2^-53."""
    return (u64(seed, stream, n, start) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def splitmix64_raw(state: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_splitmix64_raw(state, n, out.ctypes.data)
    return out


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even) with the generator's routine."""
    lib = _load()
    flat = np.ascontiguousarray(f, dtype=np.float32).ravel()
    return np.array([lib.synth_f32_to_bf16(float(v)) for v in flat], dtype=np.uint16).reshape(np.shape(f))


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------------------
# Routing-side inputs that are not tensors of the layer itself.


def random_permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of range(n) driven by the counter-based stream."""
    r = u64(seed, stream, n)
    perm = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(r[i] % np.uint64(i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return perm


def zipf_logit_bias(seed: int, E: int, alpha: float) -> np.ndarray:
    """Per-expert router bias log(p_e), p_e proportional to rank^-alpha.

    Ranks 1..E are dealt to the experts by a seeded random permutation drawn
    from seed+1.  Returned as float32 (the value both sides read).
    """
    perm = random_permutation(seed + 1, STREAM_SKEW_PERM, E)
    rank = np.empty(E, dtype=np.float64)
    rank[perm] = np.arange(1, E + 1, dtype=np.float64)
    p = rank ** (-float(alpha))
    p /= p.sum()
    return np.log(p).astype(np.float32)


def random_topk(seed: int, T: int, E: int, k: int, alpha: float = 0.0,
                stream: int = STREAM_TOPK) -> np.ndarray:
    """[T,k] int32 expert ids, k distinct per token (Gumbel-top-k, Zipf weights).

    Used to drive the permute / expert-FFN / combine stages on their own.
    """
    if T == 0:
        return np.zeros((0, k), dtype=np.int32)
    p = np.arange(1, E + 1, dtype=np.float64) ** (-float(alpha))
    u = uniform01(seed, stream, T * E).reshape(T, E)
    u = np.clip(u, 1e-300, 1.0 - 2.0 ** -53)
    key = np.log(p)[None, :] - np.log(-np.log(u))
    order = np.argsort(-key, axis=1, kind="stable")[:, :k]
    return order.astype(np.int32)


def make_inputs(wl: Workload, with_experts: bool = True, with_shared: bool = False) -> dict:
    """All tensors of one workload as numpy arrays (bf16 as uint16 bit patterns).

    x ~ N(0,1); every weight ~ N(0, 0.02); router bias (skew only) fp32.
    The tensor for stream s holds element i = index i of stream s of wl.seed,
    so an expert's slice e of a [E, rows, cols] weight is elements
    e*rows*cols ... of that stream.  with_experts=False leaves out the routed
    experts' weights (and, unless with_shared, the shared expert's).
    """
    s = wl.seed
    d = {"x": normal_bf16(s, STREAM_X, (wl.T, wl.H)),
         "w_router": normal_bf16(s, STREAM_WR, (wl.E, wl.H), std=0.02)}
    if with_experts:
        d["w_gate"] = normal_bf16(s, STREAM_WG, (wl.E, wl.F, wl.H), std=0.02)
        d["w_up"] = normal_bf16(s, STREAM_WU, (wl.E, wl.F, wl.H), std=0.02)
        d["w_down"] = normal_bf16(s, STREAM_WD, (wl.E, wl.H, wl.F), std=0.02)
    if wl.F_shared and (with_experts or with_shared):
        d["ws_gate"] = normal_bf16(s, STREAM_WSG, (wl.F_shared, wl.H), std=0.02)
        d["ws_up"] = normal_bf16(s, STREAM_WSU, (wl.F_shared, wl.H), std=0.02)
        d["ws_down"] = normal_bf16(s, STREAM_WSD, (wl.H, wl.F_shared), std=0.02)
    if wl.shared_gate:
        d["w_shared_gate"] = normal_bf16(s, STREAM_WSGATE, (wl.H,), std=0.02)
    if wl.alpha is not None:
        d["logit_bias"] = zipf_logit_bias(s, wl.E, wl.alpha)
    return d


def expert_slice(wl: Workload, name: str, e: int) -> np.ndarray:
    """One expert's weight matrix, generated on its own (same bits as make_inputs)."""
    if name == "w_gate":
        return normal_bf16(wl.seed, STREAM_WG, (wl.F, wl.H), std=0.02, start=e * wl.F * wl.H)
    if name == "w_up":
        return normal_bf16(wl.seed, STREAM_WU, (wl.F, wl.H), std=0.02, start=e * wl.F * wl.H)
    if name == "w_down":
        return normal_bf16(wl.seed, STREAM_WD, (wl.H, wl.F), std=0.02, start=e * wl.H * wl.F)
    raise KeyError(name)
