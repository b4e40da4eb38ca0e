"""moe_permute_noalloc against moe_permute, through the C ABI (needs a B300).

moe_permute_noalloc serves callers that cannot give the library a workspace. It keeps
its scratch in a fixed array inside the library's device image. These checks compare it
with the workspace-based moe_permute on the same inputs, on two calls in a row (the
second call reuses the array the first one left behind), and check that an oversized
problem is refused. This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import moe_synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import sparse_mixture_experts_57_b300 as moe
    L = moe.lib()
    moe.get_device_status()
    return L


def _buffers(T, H, E, k):
    d = "cuda"
    return {"counts": torch.empty(E, dtype=torch.int32, device=d),
            "offsets": torch.empty(E + 1, dtype=torch.int32, device=d),
            "row_token": torch.empty(T * k, dtype=torch.int32, device=d),
            "slot_row": torch.empty(T * k, dtype=torch.int32, device=d),
            "x_perm": torch.empty((T * k, H), dtype=torch.bfloat16, device=d)}


def _call_with_workspace(L, idx, x, T, H, E, k, stream):
    out = _buffers(T, H, E, k)
    ws = torch.empty(L.moe_permute_workspace_size(T, E, k), dtype=torch.uint8, device="cuda")
    rc = L.moe_permute(idx.data_ptr(), x.data_ptr(), T, H, E, k, out["counts"].data_ptr(),
                       out["offsets"].data_ptr(), out["row_token"].data_ptr(),
                       out["slot_row"].data_ptr(), out["x_perm"].data_ptr(), ws.data_ptr(),
                       ws.numel(), stream)
    assert rc == 0
    return out


def _call_no_alloc(L, idx, x, T, H, E, k, stream):
    out = _buffers(T, H, E, k)
    rc = L.moe_permute_noalloc(idx.data_ptr(), x.data_ptr(), T, H, E, k,
                               out["counts"].data_ptr(), out["offsets"].data_ptr(),
                               out["row_token"].data_ptr(), out["slot_row"].data_ptr(),
                               out["x_perm"].data_ptr(), stream)
    assert rc == 0
    return out


def test_no_alloc_permute_matches_workspace_permute_twice(lib):
    stream = torch.cuda.current_stream().cuda_stream
    # Two different problems in a row: the second runs on the scratch the first left behind.
    cases = [(1000, 128, 6, 1.2, 11), (4099, 512, 24, 0.5, 12)]
    for T, E, k, skew, seed in cases:
        H = 128
        idx = moe_synth.to_torch(moe_synth.random_topk(seed, T, E, k, skew), "cuda")
        x = moe_synth.to_torch(moe_synth.normal_bf16(seed, 50, (T, H), 1.0), "cuda")
        ref = _call_with_workspace(lib, idx, x, T, H, E, k, stream)
        got = _call_no_alloc(lib, idx, x, T, H, E, k, stream)
        torch.cuda.synchronize()
        # integer and byte results: bit-exact
        for key in ("counts", "offsets", "row_token", "slot_row"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["x_perm"].view(torch.int16), ref["x_perm"].view(torch.int16))
    status = ctypes.c_int(-1)
    assert lib.moe_get_device_status(stream, ctypes.byref(status)) == 0
    assert status.value == 0


def test_no_alloc_permute_at_capacity_and_empty(lib):
    """The largest problem the array holds (ceil(T/32) * E * 8 bytes = exactly 2 MiB:
    T = 16384 tokens, E = 512 experts) is accepted and matches moe_permute bit for bit; a
    call with T = 0 writes all-zero counts and offsets."""
    stream = torch.cuda.current_stream().cuda_stream
    T, E, k, H = 16384, 512, 2, 64
    assert (T + 31) // 32 * E * 8 == lib.moe_permute_noalloc_max_scratch_bytes()
    idx = moe_synth.to_torch(moe_synth.random_topk(13, T, E, k, 0.7), "cuda")
    x = moe_synth.to_torch(moe_synth.normal_bf16(13, 50, (T, H), 1.0), "cuda")
    ref = _call_with_workspace(lib, idx, x, T, H, E, k, stream)
    got = _call_no_alloc(lib, idx, x, T, H, E, k, stream)
    torch.cuda.synchronize()
    for key in ("counts", "offsets", "row_token", "slot_row"):
        assert torch.equal(got[key], ref[key]), key
    assert torch.equal(got["x_perm"].view(torch.int16), ref["x_perm"].view(torch.int16))
    # T = 0: counts and offsets are written (zeros), nothing else is touched
    out = _buffers(0, H, E, k)
    out["counts"].fill_(-7)
    out["offsets"].fill_(-7)
    rc = lib.moe_permute_noalloc(idx.data_ptr(), x.data_ptr(), 0, H, E, k,
                                 out["counts"].data_ptr(), out["offsets"].data_ptr(),
                                 out["row_token"].data_ptr(), out["slot_row"].data_ptr(),
                                 out["x_perm"].data_ptr(), stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(out["counts"].abs().sum()) == 0 and int(out["offsets"].abs().sum()) == 0
    status = ctypes.c_int(-1)
    assert lib.moe_get_device_status(stream, ctypes.byref(status)) == 0
    assert status.value == 0


def test_no_alloc_permute_refuses_oversized_problems(lib):
    cap = lib.moe_permute_noalloc_max_scratch_bytes()
    assert cap == 2 << 20
    T, E, k, H = 32768, 512, 2, 64     # ceil(T/32) * E * 8 bytes = 4 MiB > 2 MiB
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    out = _buffers(T, H, E, k)
    rc = lib.moe_permute_noalloc(idx.data_ptr(), x.data_ptr(), T, H, E, k,
                                 out["counts"].data_ptr(), out["offsets"].data_ptr(),
                                 out["row_token"].data_ptr(), out["slot_row"].data_ptr(),
                                 out["x_perm"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 2   # MOE_ERR_UNSUPPORTED
