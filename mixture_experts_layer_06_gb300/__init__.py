"""GB300-native single-GPU Mixture-of-Experts layer forward.

Thin Python binding over the C ABI of ``libmoe_gb300.so`` (declared in
include/moe.h).  Every function here only marshals arguments: it checks
dtypes and shapes, allocates output tensors with torch when the caller did
not pass them, and calls the library entry point of the same name on the
current CUDA stream.  All computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing or cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MoeConfig", "MoeError", "load_library", "library_path", "moe_route", "moe_route_scratch_bytes", "moe_permute",
    "moe_permute_scratch_bytes", "moe_permute_noalloc", "moe_expert_ffn", "moe_expert_ffn_unfused",
    "moe_expert_ffn_static", "moe_combine", "moe_workspace_bytes", "moe_forward_ex",
    "moe_forward", "moe_device_error", "moe_set_trace_events", "moe_selftest_wait_timeout", "moe_status_string",
    "moe_forward_launches", "moe_launches_issued", "EXPORTED_SYMBOLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")
_lib = None

# Entry points declared in include/moe.h.
EXPORTED_SYMBOLS = (
    "moe_config_default", "moe_route", "moe_route_scratch_bytes", "moe_permute_scratch_bytes", "moe_permute", "moe_expert_ffn",
    "moe_combine", "moe_workspace_bytes", "moe_forward_ex", "moe_forward", "moe_status_string",
    "moe_device_error", "moe_set_trace_events", "moe_selftest_wait_timeout", "moe_abi_version",
    "moe_permute_noalloc", "moe_expert_ffn_ex", "moe_expert_ffn_unfused", "moe_expert_ffn_static",
    "moe_forward_launches", "moe_launches_issued",
)

ACTIVATIONS = {"silu": 0, "gelu": 1}  # moe_activation_t

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_VALUE", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT", 6: "MOE_ERR_DEVICE_BOUNDS"}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class MoeConfig(ctypes.Structure):
    """Mirror of moe_config_t (include/moe.h)."""
    _fields_ = [
        ("score", ctypes.c_int),
        ("renormalize", ctypes.c_int),
        ("route_scale", ctypes.c_float),
        ("n_group", ctypes.c_int),
        ("topk_group", ctypes.c_int),
        ("group_topn", ctypes.c_int),
        ("logit_bias", ctypes.c_void_p),
        ("F_shared", ctypes.c_int),
        ("ws_gate", ctypes.c_void_p),
        ("ws_up", ctypes.c_void_p),
        ("ws_down", ctypes.c_void_p),
        ("w_shared_gate", ctypes.c_void_p),
        ("activation", ctypes.c_int),
    ]

    @classmethod
    def make(cls, score="softmax", renormalize=True, route_scale=1.0, n_group=1, topk_group=1, group_topn=0,
             logit_bias=None, ws_gate=None, ws_up=None, ws_down=None, w_shared_gate=None,
             activation="silu") -> "MoeConfig":
        c = cls()
        c.score = {"softmax": 0, "sigmoid": 1}[score]
        c.renormalize = int(bool(renormalize))
        c.route_scale = float(route_scale)
        c.n_group, c.topk_group, c.group_topn = int(n_group), int(topk_group), int(group_topn)
        c.logit_bias = _ptr(logit_bias, torch.float32)
        c.F_shared = 0 if ws_gate is None else int(ws_gate.shape[0])
        c.ws_gate = _ptr(ws_gate)
        c.ws_up = _ptr(ws_up)
        c.ws_down = _ptr(ws_down)
        c.w_shared_gate = _ptr(w_shared_gate)
        c.activation = ACTIVATIONS[activation]
        c._keep = (logit_bias, ws_gate, ws_up, ws_down, w_shared_gate)  # keep tensors alive
        return c


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libmoe_gb300.so (build it first with __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: the CUDA library has not been built")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, S, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint32
    sig = {
        "moe_config_default": (None, [P]),
        "moe_route": (I, [P, P, P, I, I, I, I, P, P, P, P, S, P]),
        "moe_route_scratch_bytes": (S, [P, I, I, I]),
        "moe_permute_scratch_bytes": (S, [I, I]),
        "moe_permute": (I, [P, P, I, I, I, I, P, P, P, P, P, P, S, P]),
        "moe_permute_noalloc": (I, [P, P, I, I, I, I, P, P, P, P, P, P]),
        "moe_expert_ffn": (I, [P, P, I, I, I, I, P, P, P, P, P, P]),
        "moe_expert_ffn_ex": (I, [P, P, I, I, I, I, P, P, P, I, P, P, P]),
        "moe_expert_ffn_unfused": (I, [P, P, I, I, I, I, P, P, P, I, P, P, P, P, P]),
        "moe_expert_ffn_static": (I, [P, P, I, I, I, I, P, P, P, I, P, P, P]),
        "moe_combine": (I, [P, P, P, P, P, I, I, I, P, P]),
        "moe_workspace_bytes": (S, [P, I, I, I, I, I]),
        "moe_forward_ex": (I, [P, P, P, P, P, P, I, I, I, I, I, P, P, S, P]),
        "moe_forward": (I, [P, P, P, P, P, I, I, I, I, I, P, P]),
        "moe_status_string": (ctypes.c_char_p, [I]),
        "moe_device_error": (I, [P, ctypes.POINTER(U)]),
        "moe_set_trace_events": (I, [P, I]),
        "moe_selftest_wait_timeout": (I, [U, P]),
        "moe_abi_version": (I, []),
        "moe_forward_launches": (I, [P, I, I, I, I, I]),
        "moe_launches_issued": (ctypes.c_ulonglong, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


# ----------------------------------------------------------------------------- helpers

def _ptr(t, dtype=torch.bfloat16):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, where: str):
    if status != 0:
        raise MoeError(status, where)


def _out(t, shape, dtype, device):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"output must be {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")
    return t


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


# ----------------------------------------------------------------------------- entry points

def moe_route_scratch_bytes(cfg: MoeConfig | None, T: int, H: int, E: int) -> int:
    return int(load_library().moe_route_scratch_bytes(ctypes.byref(cfg) if cfg is not None else None, T, H, E))


def moe_route(x, w_router, k, cfg: MoeConfig | None = None, topk_idx=None, topk_w=None, shared_scale=None,
              scratch=None, stream=None):
    """Router scoring + top-k.  Returns (topk_idx int32 [T,k], topk_w fp32 [T,k], shared_scale or None)."""
    lib = load_library()
    T, H = x.shape
    E = w_router.shape[0]
    topk_idx = _out(topk_idx, (T, k), torch.int32, x.device)
    topk_w = _out(topk_w, (T, k), torch.float32, x.device)
    if cfg is not None and cfg.w_shared_gate:
        shared_scale = _out(shared_scale, (T,), torch.float32, x.device)
    if scratch is None:
        scratch = torch.empty(max(moe_route_scratch_bytes(cfg, T, H, E), 16), dtype=torch.uint8, device=x.device)
    st = lib.moe_route(ctypes.byref(cfg) if cfg is not None else None, _ptr(x), _ptr(w_router), T, H, E, k,
                       _ptr(topk_idx, torch.int32), _ptr(topk_w, torch.float32),
                       _ptr(shared_scale, torch.float32), _ptr(scratch, torch.uint8), scratch.numel(),
                       _stream(stream))
    _check(st, "moe_route")
    return topk_idx, topk_w, shared_scale


def moe_permute_scratch_bytes(T: int, E: int) -> int:
    return int(load_library().moe_permute_scratch_bytes(T, E))


def moe_permute(topk_idx, x, E, counts=None, offsets=None, perm=None, inv=None, x_perm=None, scratch=None,
                stream=None):
    """Group token copies by expert.  Returns (counts, offsets, perm, inv, x_perm)."""
    lib = load_library()
    T, k = topk_idx.shape
    H = x.shape[1]
    dev = x.device
    counts = _out(counts, (E,), torch.int32, dev)
    offsets = _out(offsets, (E + 1,), torch.int32, dev)
    perm = _out(perm, (T * k,), torch.int32, dev)
    inv = _out(inv, (T * k,), torch.int32, dev)
    x_perm = _out(x_perm, (T * k, H), torch.bfloat16, dev)
    nbytes = moe_permute_scratch_bytes(T, E)
    if scratch is None:
        scratch = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    st = lib.moe_permute(_ptr(topk_idx, torch.int32), _ptr(x), T, H, E, k, _ptr(counts, torch.int32),
                         _ptr(offsets, torch.int32), _ptr(perm, torch.int32), _ptr(inv, torch.int32),
                         _ptr(x_perm), _ptr(scratch, torch.uint8), scratch.numel(), _stream(stream))
    _check(st, "moe_permute")
    return counts, offsets, perm, inv, x_perm


def moe_permute_noalloc(topk_idx, x, E, counts=None, offsets=None, perm=None, inv=None, x_perm=None,
                        stream=None):
    """moe_permute with the library's built-in scratch, for callers that cannot allocate device
    memory (pass every output tensor to allocate nothing here either).
    Returns (counts, offsets, perm, inv, x_perm)."""
    lib = load_library()
    T, k = topk_idx.shape
    H = x.shape[1]
    dev = x.device
    counts = _out(counts, (E,), torch.int32, dev)
    offsets = _out(offsets, (E + 1,), torch.int32, dev)
    perm = _out(perm, (T * k,), torch.int32, dev)
    inv = _out(inv, (T * k,), torch.int32, dev)
    x_perm = _out(x_perm, (T * k, H), torch.bfloat16, dev)
    st = lib.moe_permute_noalloc(_ptr(topk_idx, torch.int32), _ptr(x), T, H, E, k, _ptr(counts, torch.int32),
                                 _ptr(offsets, torch.int32), _ptr(perm, torch.int32), _ptr(inv, torch.int32),
                                 _ptr(x_perm), _stream(stream))
    _check(st, "moe_permute_noalloc")
    return counts, offsets, perm, inv, x_perm


def moe_expert_ffn(x_perm, offsets, w_gate, w_up, w_down, h=None, y=None, stream=None, activation="silu"):
    """Grouped gated FFN (SwiGLU, or GEGLU with activation="gelu").  offsets None =
    one dense group (w_* given as [1,...] or 2-D).  Returns (h bf16 [rows,F], y fp16 [rows,H])."""
    lib = load_library()
    rows, H = x_perm.shape
    if w_gate.dim() == 2:
        E, F = 1, w_gate.shape[0]
    else:
        E, F = w_gate.shape[0], w_gate.shape[1]
    h = _out(h, (rows, F), torch.bfloat16, x_perm.device)
    y = _out(y, (rows, H), torch.float16, x_perm.device)
    if activation == "silu":
        st = lib.moe_expert_ffn(_ptr(x_perm), _ptr(offsets, torch.int32), rows, H, F, E, _ptr(w_gate), _ptr(w_up),
                                _ptr(w_down), _ptr(h), _ptr(y, torch.float16), _stream(stream))
    else:
        st = lib.moe_expert_ffn_ex(_ptr(x_perm), _ptr(offsets, torch.int32), rows, H, F, E, _ptr(w_gate),
                                   _ptr(w_up), _ptr(w_down), ACTIVATIONS[activation], _ptr(h),
                                   _ptr(y, torch.float16), _stream(stream))
    _check(st, "moe_expert_ffn")
    return h, y


def moe_expert_ffn_unfused(x_perm, offsets, w_gate, w_up, w_down, activation="silu", stream=None):
    """Fusion ablation: gate and up as two GEMMs into bf16 g, u, then the
    element-wise activation, then the down projection.  Returns (h, y, g, u)."""
    lib = load_library()
    rows, H = x_perm.shape
    if w_gate.dim() == 2:
        E, F = 1, w_gate.shape[0]
    else:
        E, F = w_gate.shape[0], w_gate.shape[1]
    g = torch.empty((rows, F), dtype=torch.bfloat16, device=x_perm.device)
    u = torch.empty_like(g)
    h = torch.empty_like(g)
    y = torch.empty((rows, H), dtype=torch.float16, device=x_perm.device)
    st = lib.moe_expert_ffn_unfused(_ptr(x_perm), _ptr(offsets, torch.int32), rows, H, F, E, _ptr(w_gate),
                                    _ptr(w_up), _ptr(w_down), ACTIVATIONS[activation], _ptr(g), _ptr(u), _ptr(h),
                                    _ptr(y, torch.float16), _stream(stream))
    _check(st, "moe_expert_ffn_unfused")
    return h, y, g, u


def moe_expert_ffn_static(x_perm, offsets, w_gate, w_up, w_down, block_m=64, stream=None):
    """Schedule ablation: offsets read back to the host (a sync), fixed block_m
    token tiles, one CTA per tile.  Returns (h bf16 [rows,F], y fp16 [rows,H])."""
    lib = load_library()
    rows, H = x_perm.shape
    E, F = w_gate.shape[0], w_gate.shape[1]
    h = torch.empty((rows, F), dtype=torch.bfloat16, device=x_perm.device)
    y = torch.empty((rows, H), dtype=torch.float16, device=x_perm.device)
    st = lib.moe_expert_ffn_static(_ptr(x_perm), _ptr(offsets, torch.int32), rows, H, F, E, _ptr(w_gate),
                                   _ptr(w_up), _ptr(w_down), int(block_m), _ptr(h), _ptr(y, torch.float16),
                                   _stream(stream))
    _check(st, "moe_expert_ffn_static")
    return h, y


def moe_combine(y_perm, inv, topk_w, y_shared=None, shared_scale=None, out=None, stream=None):
    """Deterministic weighted scatter-back of fp16 expert outputs.  Returns out bf16 [T,H]."""
    lib = load_library()
    T, k = topk_w.shape
    H = y_perm.shape[1]
    out = _out(out, (T, H), torch.bfloat16, y_perm.device)
    st = lib.moe_combine(_ptr(y_perm, torch.float16), _ptr(inv, torch.int32), _ptr(topk_w, torch.float32),
                         _ptr(y_shared, torch.float16), _ptr(shared_scale, torch.float32), T, H, k, _ptr(out),
                         _stream(stream))
    _check(st, "moe_combine")
    return out


def moe_workspace_bytes(cfg: MoeConfig | None, T, H, F, E, k) -> int:
    return int(load_library().moe_workspace_bytes(ctypes.byref(cfg) if cfg is not None else None, T, H, F, E, k))


def moe_forward_ex(x, w_router, w_gate, w_up, w_down, k, cfg: MoeConfig | None = None, out=None, workspace=None,
                   stream=None):
    """The whole layer with caller workspace (allocated here if not given)."""
    lib = load_library()
    T, H = x.shape
    E, F = w_gate.shape[0], w_gate.shape[1]
    out = _out(out, (T, H), torch.bfloat16, x.device)
    need = moe_workspace_bytes(cfg, T, H, F, E, k)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    st = lib.moe_forward_ex(ctypes.byref(cfg) if cfg is not None else None, _ptr(x), _ptr(w_router), _ptr(w_gate),
                            _ptr(w_up), _ptr(w_down), T, H, F, E, k, _ptr(out), _ptr(workspace, torch.uint8),
                            workspace.numel(), _stream(stream))
    _check(st, "moe_forward_ex")
    return out


def moe_forward(x, w_router, w_gate, w_up, w_down, k, out=None, stream=None):
    """The whole layer, Mixtral routing, library-owned workspace."""
    lib = load_library()
    T, H = x.shape
    E, F = w_gate.shape[0], w_gate.shape[1]
    out = _out(out, (T, H), torch.bfloat16, x.device)
    st = lib.moe_forward(_ptr(x), _ptr(w_router), _ptr(w_gate), _ptr(w_up), _ptr(w_down), T, H, F, E, k, _ptr(out),
                         _stream(stream))
    _check(st, "moe_forward")
    return out


def moe_forward_launches(cfg: MoeConfig | None, T, H, F, E, k) -> int:
    """Kernels one moe_forward_ex call launches for these shapes (-1: rejected arguments)."""
    return int(load_library().moe_forward_launches(ctypes.byref(cfg) if cfg is not None else None, T, H, F, E, k))


def moe_launches_issued() -> int:
    """Kernels the library has launched since it was loaded."""
    return int(load_library().moe_launches_issued())


def moe_set_trace_events(events):
    """Record the given 6 torch.cuda.Event objects (None entries: no event at that
    boundary) around the stages of later forwards; None turns it off."""
    lib = load_library()
    if events is None:
        _check(lib.moe_set_trace_events(None, 0), "moe_set_trace_events")
        return
    for e in events:
        if e is not None and not e.cuda_event:  # torch creates the CUDA event on first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event if e is not None else None for e in events])
    _check(lib.moe_set_trace_events(arr, len(events)), "moe_set_trace_events")


def moe_selftest_wait_timeout(limit_us: int, stream=None):
    """Launch the failure-path self-test (a wait nothing releases); see include/moe.h."""
    _check(load_library().moe_selftest_wait_timeout(limit_us, _stream(stream)), "moe_selftest_wait_timeout")


def moe_device_error(stream=None):
    """Synchronise, read and clear the device error word.  Returns (status, raw)."""
    raw = ctypes.c_uint32(0)
    st = load_library().moe_device_error(_stream(stream), ctypes.byref(raw))
    return st, raw.value
