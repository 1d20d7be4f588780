"""moe_permute_noalloc: the permute for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc at all (a serving engine that plans all
device memory at start-up, a plugin inside an application that owns the CUDA
allocator, latency-bound code that cannot take cudaMalloc's implicit
synchronisation).  For them the library offers a permute whose scratch lives
in a fixed array inside the library's device image.  This file checks, through
the C ABI, that it gives the same results as moe_permute on two calls in a
row (the second call must not see anything left over from the first), and
that calls too large for the built-in array are refused.  It runs last so
that a failure here does not hide the results of the other GPU tests.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_06_gb300 as moe
import synth

pytestmark = pytest.mark.gpu


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to("cuda").view(torch.bfloat16)


def _dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to("cuda")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load_library()


def test_noalloc_permute_matches_permute_on_two_calls_in_a_row():
    # Two different routings back to back: a dense one, then a skewed one with
    # fewer tokens, so stale scratch from the first call would show up.
    cases = [(8192, 256, 8, 0.0, 256), (3000, 64, 4, 2.0, 384)]
    for i, (T, E, k, alpha, H) in enumerate(cases):
        idx = _dev_i32(synth.random_topk(20 + i, T, E, k, alpha=alpha))
        x = _dev_bf16(synth.normal_bf16(20 + i, 1, (T, H)))
        want = moe.moe_permute(idx, x, E)
        # every output preallocated: the call itself allocates nothing
        got = tuple(torch.full_like(t, -7) for t in want)
        moe.moe_permute_noalloc(idx, x, E, *got)
        st, raw = moe.moe_device_error()
        assert st == 0, f"device error word {raw:#x}"
        for name, a, b in zip(("counts", "offsets", "perm", "inv", "x_perm"), want, got):
            assert torch.equal(a.view(torch.int32) if a.dtype != torch.bfloat16 else a.view(torch.int16),
                               b.view(torch.int32) if b.dtype != torch.bfloat16 else b.view(torch.int16)), name


def test_noalloc_permute_refuses_calls_beyond_its_scratch():
    E, k, T = 256, 8, 8193  # ceil(8193/32) * 256 = 65792 words > 65536
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    x = torch.zeros((T, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_permute_noalloc(idx, x, E)
    assert ei.value.status == 3  # MOE_ERR_WORKSPACE, nothing launched
