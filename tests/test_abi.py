"""The C-ABI library: it builds, loads without a GPU, exports every entry point
include/moe.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_06_gb300 as moe
from mixture_experts_layer_06_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", src))


def test_header_and_binding_agree():
    assert _declared() == set(moe.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.moe_abi_version() == 102
    assert moe.moe_status_string(0) == "MOE_OK"
    assert moe.moe_status_string(6) == "MOE_ERR_DEVICE_BOUNDS"
    assert moe.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def test_config_default(lib):
    c = moe.MoeConfig()
    c.score = 7
    lib.moe_config_default(ctypes.byref(c))
    assert (c.score, c.renormalize, c.route_scale, c.n_group, c.F_shared) == (0, 1, 1.0, 1, 0)
    assert c.logit_bias is None and c.ws_gate is None


def test_workspace_sizes(lib):
    assert lib.moe_workspace_bytes(None, 128, 512, 1024, 8, 2) > 128 * 2 * (512 * 2 + 1024 * 2 + 512 * 2)
    assert lib.moe_workspace_bytes(None, 128, 500, 1024, 8, 2) == 0  # H not a multiple of 128
    assert lib.moe_permute_scratch_bytes(8192, 256) >= 2 * 256 * 256 * 4
    shared = moe.MoeConfig()
    lib.moe_config_default(ctypes.byref(shared))
    shared.F_shared = 1024
    assert lib.moe_workspace_bytes(ctypes.byref(shared), 64, 512, 1024, 8, 2) > \
        lib.moe_workspace_bytes(None, 64, 512, 1024, 8, 2)


@pytest.mark.parametrize("T,H,E,k,status", [
    (4, 512, 8, 9, 2),     # k > E
    (4, 512, 300, 2, 2),   # E > 256
    (4, 500, 8, 2, 2),     # H not a multiple of 128
    (-1, 512, 8, 2, 1),    # negative T
    (4, 512, 8, 0, 1),     # k == 0
    (4, 512, 8, 17, 2),    # k > 16
])
def test_route_rejects_bad_shapes_without_a_launch(lib, T, H, E, k, status):
    assert lib.moe_route(None, None, None, T, H, E, k, None, None, None, None, 0, None) == status


def test_null_and_misaligned_pointers_rejected(lib):
    assert lib.moe_route(None, None, None, 4, 512, 8, 2, None, None, None, None, 0, None) == 1
    assert lib.moe_route(None, 0x1008, 0x2000, 4, 512, 8, 2, 0x3000, 0x4000, None, 0x5000, 1 << 20, None) == 1  # misaligned x
    assert lib.moe_forward_ex(None, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 4, 512, 1024, 8, 2, 0x6000,
                              0x7000, 16, None) == 3  # workspace too small
    assert lib.moe_combine(None, None, None, None, None, 4, 512, 2, None, None) == 1
    assert lib.moe_expert_ffn(0x1000, None, 16, 512, 1024, 8, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, None) == 1
    assert lib.moe_expert_ffn_unfused(0x1000, 0x7000, 16, 512, 1024, 8, 0x2000, 0x3000, 0x4000, 0, None, 0x8000,
                                      0x5000, 0x6000, None) == 1  # no g buffer
    assert lib.moe_expert_ffn_static(0x1000, 0x7000, 16, 512, 1024, 8, 0x2000, 0x3000, 0x4000, 48, 0x5000, 0x6000,
                                     None) == 1  # block_m not a supported tile
    assert lib.moe_expert_ffn_static(0x1000, None, 16, 512, 1024, 8, 0x2000, 0x3000, 0x4000, 64, 0x5000, 0x6000,
                                     None) == 1  # offsets required
    # unknown activation
    assert lib.moe_expert_ffn_ex(0x1000, 0x7000, 16, 512, 1024, 8, 0x2000, 0x3000, 0x4000, 7, 0x5000, 0x6000,
                                 None) == 1


def test_bad_group_config_rejected(lib):
    c = moe.MoeConfig()
    lib.moe_config_default(ctypes.byref(c))
    c.n_group, c.topk_group, c.group_topn = 8, 9, 2  # keeps more groups than exist
    assert lib.moe_route(ctypes.byref(c), 0x1000, 0x2000, 4, 512, 256, 8, 0x3000, 0x4000, None, 0x5000, 1 << 20, None) == 1
    c.n_group, c.topk_group, c.group_topn = 7, 4, 2  # 256 experts do not split into 7 groups
    assert lib.moe_route(ctypes.byref(c), 0x1000, 0x2000, 4, 512, 256, 8, 0x3000, 0x4000, None, 0x5000, 1 << 20, None) == 2
    c.n_group, c.topk_group, c.group_topn = 8, 1, 2  # k=8 > one group of 4 experts
    assert lib.moe_route(ctypes.byref(c), 0x1000, 0x2000, 4, 512, 32, 8, 0x3000, 0x4000, None, 0x5000, 1 << 20,
                         None) == 1


def test_bad_activation_rejected(lib):
    c = moe.MoeConfig()
    lib.moe_config_default(ctypes.byref(c))
    assert c.activation == 0  # SiLU by default
    c.activation = 3
    assert lib.moe_route(ctypes.byref(c), 0x1000, 0x2000, 4, 512, 8, 2, 0x3000, 0x4000, None, 0x5000, 1 << 20,
                         None) == 1


def test_zero_tokens_is_a_noop(lib):
    assert lib.moe_route(None, 0x1000, 0x2000, 0, 512, 8, 2, 0x3000, 0x4000, None, None, 0, None) == 0
    assert lib.moe_forward_ex(None, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0, 512, 1024, 8, 2, 0x6000,
                              0x7000, 0, None) == 0
    assert lib.moe_combine(None, None, None, None, None, 0, 512, 2, None, None) == 0


def test_trace_event_argument_check(lib):
    assert lib.moe_set_trace_events(None, 0) == 0
    arr = (ctypes.c_void_p * 3)(1, 2, 3)
    assert lib.moe_set_trace_events(arr, 3) == 1  # six boundaries, not three
    none = (ctypes.c_void_p * 6)()
    assert lib.moe_set_trace_events(none, 6) == 1  # at least one event
    assert lib.moe_set_trace_events(None, 0) == 0


def test_package_has_no_cpu_fallback():
    import inspect
    src = inspect.getsource(moe)
    assert "oracle" not in src and "numpy" not in src


def test_selftest_limit_checked_on_host(lib):
    assert lib.moe_selftest_wait_timeout(0, None) == 1
    assert lib.moe_selftest_wait_timeout(2000000, None) == 1


def test_route_needs_no_scratch(lib):
    """The router reduces its K-split partial logits on chip: no scratch, and a
    NULL scratch pointer is accepted; the shape checks still come first."""
    assert lib.moe_route_scratch_bytes(None, 4, 512, 8) == 0
    assert lib.moe_route_scratch_bytes(None, 8192, 7168, 256) == 0
    assert lib.moe_route_scratch_bytes(None, 4, 500, 8) == 0  # rejected shape
    assert lib.moe_route(None, 0x1000, 0x2000, 4, 500, 8, 2, 0x3000, 0x4000, None, None, 0, None) == 2


def test_forward_launch_query_on_the_host(lib):
    # tiny layer: router GEMM + top-k, three permute launches, two GEMMs, combine
    n = moe.moe_forward_launches(None, 128, 512, 1024, 8, 2)
    assert 4 <= n <= 12
    assert moe.moe_forward_launches(None, 0, 512, 1024, 8, 2) == 0  # T = 0 launches nothing
    assert moe.moe_forward_launches(None, 128, 500, 1024, 8, 2) == -1  # rejected shape
    assert moe.moe_launches_issued() >= 0
