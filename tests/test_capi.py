"""The C ABI library builds, loads and exports every symbol that include/moe.h declares.

CPU only: no compute call is made (there is no GPU here). Argument checks that return
before any CUDA call are exercised too.
"""
import ctypes
import os
import re

import pytest

import sparse_mixture_experts_57_b300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n.startswith(("moe_", "latent_"))))


def test_header_declares_the_calls():
    names = declared_functions()
    for want in ["moe_route", "moe_permute", "moe_grouped_ffn", "moe_combine", "moe_forward",
                 "latent_moe", "moe_linear", "moe_get_device_status", "moe_status_string"]:
        assert want in names


def test_library_exports_every_declared_symbol():
    L = moe.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in moe.SIGNATURES, f"binding lacks {name}"


def test_status_strings():
    assert moe.status_string(0) == "ok"
    assert "timed out" in moe.status_string(5)
    assert moe.status_string(99) == "unknown status"


def test_workspace_sizes_are_monotone():
    L = moe.lib()
    a = L.moe_forward_workspace_size(64, 2688, 128, 6, 1856)
    b = L.moe_forward_workspace_size(16384, 2688, 128, 6, 1856)
    assert 0 < a < b
    # x_perm + h + y_perm dominate: rows * (2H + F) * 2 bytes
    assert b >= 16384 * 6 * (2 * 2688 + 1856) * 2
    assert L.moe_forward_workspace_size(-1, 64, 4, 2, 64) == 0
    # the fused combine drops y_perm (rows * H * 2 bytes) and adds the int64 sums (T * H * 8)
    T, H, E, k, F = 16384, 2688, 128, 6, 1856
    fused = L.moe_forward_fused_combine_workspace_size(T, H, E, k, F)
    plain = L.moe_forward_workspace_size(T, H, E, k, F)
    assert abs((plain - fused) - (T * k * H * 2 - T * H * 8)) <= 1024
    assert L.moe_forward_fused_combine_workspace_size(-1, 64, 4, 2, 64) == 0
    assert L.latent_moe_workspace_size(8192, 4096, 1024, 512, 24, 1024, 1) > \
        L.latent_moe_workspace_size(8192, 4096, 1024, 512, 24, 1024, 0)


@pytest.mark.parametrize("args", [
    (0, 0, 0, 4, 64, 8, 2, 0, 0, 0, 0, 0, 0),        # null pointers with T > 0
    (1, 1, 1, 4, 64, 2000, 2, 1, 1, 1, 1, 1, 0),     # E > 1024
    (1, 1, 1, 4, 64, 8, 9, 1, 1, 1, 1, 1, 0),        # k > E
    (1, 1, 1, -3, 64, 8, 2, 1, 1, 1, 1, 1, 0),       # negative T
])
def test_route_rejects_bad_arguments_before_any_cuda_call(args):
    L = moe.lib()
    assert L.moe_route(*args) == 1   # MOE_ERR_INVALID_ARG


def test_unaligned_sizes_are_unsupported():
    L = moe.lib()
    # H not a multiple of 64 (pointers are fake but never dereferenced)
    r = L.moe_forward(16, 16, 16, 16, 16, 4, 100, 8, 2, 64, 16, None, None, 16, 1 << 20, None)
    assert r == 2
    r = L.moe_forward_fused_combine(16, 16, 16, 16, 16, 4, 100, 8, 2, 64, 16, None, None, 16,
                                    1 << 20, None)
    assert r == 2
    # null weights with T > 0, and k > E: rejected before any CUDA call
    assert L.moe_forward_fused_combine(16, 16, 16, 0, 16, 4, 128, 8, 2, 64, 16, None, None, 16,
                                       1 << 20, None) == 1
    assert L.moe_forward_fused_combine(16, 16, 16, 16, 16, 4, 128, 8, 9, 64, 16, None, None, 16,
                                       1 << 20, None) == 1
    r = L.moe_linear(16, 16, 4, 96, 64, 16, None)
    assert r == 2


@pytest.mark.parametrize("call,dims,size_fn", [
    ("moe_forward_nvfp4_view", (300, 256, 64, 4, 192), "moe_forward_nvfp4_workspace_size"),
    ("moe_grouped_ffn_nvfp4_view", (1200, 256, 192, 64), "moe_grouped_ffn_nvfp4_workspace_size"),
    ("moe_forward_fp8_view", (300, 256, 64, 4, 192), "moe_forward_fp8_workspace_size"),
    ("moe_grouped_ffn_fp8_view", (1200, 256, 192, 64), "moe_grouped_ffn_fp8_workspace_size"),
])
def test_quant_views_are_disjoint_slices_of_the_workspace(call, dims, size_fn):
    """The views only compute addresses (no CUDA call): every buffer lies inside the
    workspace the matching size query asks for, 256-byte aligned, and no two overlap."""
    from sparse_mixture_experts_57_b300._binding import QuantView
    L = moe.lib()
    size = getattr(L, size_fn)(*dims)
    base = 1 << 40                     # a fake device address: never dereferenced
    v = QuantView()
    assert getattr(L, call)(*dims, base, size, ctypes.byref(v)) == 0
    nvfp4 = "nvfp4" in call
    fwd = "forward" in call
    if fwd:
        T, H, E, k, F = dims
        rows = T * k
    else:
        rows, H, F, E = dims
    P = v.buffer_rows
    if nvfp4:
        assert P >= rows + 127 * E and P % 128 == 0
        sf = lambda K: (P + 127) // 128 * (K // 64) * 512  # noqa: E731
    else:
        assert P == rows
    # code rows (NVFP4: two codes per byte) are padded to 128-byte pitches
    c = 2 if nvfp4 else 1
    assert (v.x_codes_ld, v.h_codes_ld) == (-(-H // c // 128) * 128, -(-F // c // 128) * 128)
    ext = {"amax": 8, "x_codes": P * v.x_codes_ld, "h": P * F * 2, "h_codes": P * v.h_codes_ld}
    if nvfp4:
        ext.update(padded_offsets=(E + 1) * 4, x_scales=sf(H), h_scales=sf(F))
    if fwd:
        ext.update(offsets=(E + 1) * 4, row_token=rows * 4)
    spans = []
    for name, _ in QuantView._fields_:
        if name in ("buffer_rows", "x_codes_ld", "h_codes_ld"):
            continue
        p = getattr(v, name)
        if name not in ext:
            assert p is None, name
            continue
        off = p - base
        assert off % 256 == 0 and 0 <= off and off + ext[name] <= size, name
        spans.append((off, off + ext[name], name))
    spans.sort()
    for a, b in zip(spans, spans[1:]):
        assert a[1] <= b[0], (a, b)
    # a workspace one byte short of what the call needs, and sizes the call rejects
    assert getattr(L, call)(*dims, base, spans[-1][1] - 1, ctypes.byref(v)) == 3
    bad = (dims[0], -1) + tuple(dims[2:])
    assert getattr(L, call)(*bad, base, size, ctypes.byref(v)) == 1
    assert getattr(L, call)(*dims, base, size, None) == 1
