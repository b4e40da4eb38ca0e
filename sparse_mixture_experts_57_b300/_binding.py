"""ctypes binding of libmoe's C ABI (argument marshalling only).

Every function here checks tensor dtypes, devices and shapes, allocates outputs and
workspaces with torch (device memory only), and calls the C entry point of the same
name on the current CUDA stream. All arithmetic happens in the library's CUDA kernels.
There is no CPU fallback: without the built library or a CUDA device, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_LIB = None

_VP, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t



class QuantView(ctypes.Structure):
    """struct moe_quant_view of include/moe.h."""
    _fields_ = [("offsets", _VP), ("row_token", _VP), ("padded_offsets", _VP), ("amax", _VP),
                ("x_codes", _VP), ("x_scales", _VP), ("h", _VP), ("h_codes", _VP),
                ("h_scales", _VP), ("buffer_rows", ctypes.c_longlong),
                ("x_codes_ld", ctypes.c_longlong), ("h_codes_ld", ctypes.c_longlong)]


_QV = ctypes.POINTER(QuantView)

# name -> (restype, argtypes); mirrors include/moe.h
SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_get_device_status": (_I, [_VP, ctypes.POINTER(_I)]),
    "moe_route_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "moe_route": (_I, [_VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "moe_route_dispatch_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "moe_route_dispatch": (_I, [_VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                _VP, _VP, _SZ, _VP]),
    "moe_permute_workspace_size": (_SZ, [_I, _I, _I]),
    "moe_permute": (_I, [_VP, _VP, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "moe_permute_noalloc_max_scratch_bytes": (_SZ, []),
    "moe_permute_noalloc": (_I, [_VP, _VP, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP]),
    "moe_grouped_ffn_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "moe_grouped_ffn": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _SZ, _VP]),
    "moe_combine": (_I, [_VP, _I, _VP, _VP, _I, _I, _I, _VP, _VP]),
    "moe_linear": (_I, [_VP, _VP, _I, _I, _I, _VP, _VP]),
    "moe_forward_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_forward_gathered": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP, _VP,
                                  _VP, _SZ, _VP]),
    "moe_forward": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _SZ,
                         _VP]),
    "moe_forward_fused_combine_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_fixed_to_bf16": (_I, [_VP, ctypes.c_longlong, _VP, _I, _VP]),
    "moe_set_profile_events": (_I, [_VP, _I]),
    "moe_fp8_codes_bytes": (_SZ, [_I, _I, _I]),
    "moe_route_cluster_refusal": (_I, []),
    "moe_forward_fused_combine": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP,
                                       _VP, _VP, _SZ, _VP]),
    "moe_nvfp4_codes_bytes": (_SZ, [_I, _I, _I]),
    "moe_nvfp4_scales_bytes": (_SZ, [_I, _I, _I]),
    "moe_quantize_nvfp4_weights": (_I, [_VP, _I, _I, _I, _VP, _VP, _VP, _VP]),
    "moe_quantize_nvfp4_weights_2d": (_I, [_VP, _I, _I, _I, _VP, _VP, _VP, _VP]),
    "moe_grouped_ffn_nvfp4_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "moe_grouped_ffn_nvfp4": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP,
                                   _VP, _SZ, _VP]),
    "moe_forward_nvfp4_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_forward_nvfp4": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I,
                               _VP, _VP, _VP, _VP, _SZ, _VP]),
    "moe_quantize_fp8_weights": (_I, [_VP, _I, _I, _I, _VP, _VP, _VP]),
    "moe_grouped_ffn_fp8_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "moe_grouped_ffn_fp8": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _SZ,
                                 _VP]),
    "moe_forward_fp8_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_forward_fp8": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP,
                             _VP, _VP, _SZ, _VP]),
    "moe_grouped_ffn_nvfp4_view": (_I, [_I, _I, _I, _I, _VP, _SZ, _QV]),
    "moe_forward_nvfp4_view": (_I, [_I, _I, _I, _I, _I, _VP, _SZ, _QV]),
    "moe_grouped_ffn_fp8_view": (_I, [_I, _I, _I, _I, _VP, _SZ, _QV]),
    "moe_forward_fp8_view": (_I, [_I, _I, _I, _I, _I, _VP, _SZ, _QV]),
    "moe_selftest_wait_timeout": (_I, [_VP, _I, _I, _VP, _VP]),
    "moe_debug_build": (_I, []),
    "moe_debug_guard_selftest": (_I, [_VP, _SZ, _VP]),
    "moe_forward_shared_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_forward_shared": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _VP,
                                _VP, _VP, _VP, _SZ, _VP]),
    "latent_moe_shared_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "latent_moe_shared": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _VP, _VP, _VP, _VP, _I, _I, _I, _I,
                               _I, _I, _I, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "latent_moe_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "latent_moe": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _VP, _VP, _I, _I, _I, _I, _I, _I, _VP, _VP,
                        _VP, _VP, _SZ, _VP]),
}


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the in-tree libmoe.so, or libmoe_debug.so (the
    MOE_DEBUG build: workspace guards and extra device checks) when the environment variable
    MOE_DEBUG is 1 at the first call."""
    global _LIB
    with _lock:
        if _LIB is None:
            path = _build.ensure_built(debug=os.environ.get("MOE_DEBUG") == "1")
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _LIB = L
    return _LIB


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _check(code: int, where: str):
    if code != 0:
        raise MoeError(code, where)


def _cuda_tensor(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (this library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    return t


def _workspace(nbytes: int, device, ws=None):
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError("workspace too small")
        return ws
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def get_device_status(stream=None) -> int:
    out = ctypes.c_int(0)
    _check(lib().moe_get_device_status(_stream(stream), ctypes.byref(out)),
           "moe_get_device_status")
    return out.value


# ------------------------------------------------------------------------------ calls ----

def moe_route(x, w_router, bias, k: int, *, workspace=None, stream=None):
    bf = torch.bfloat16
    _cuda_tensor(x, bf, "x", 2)
    _cuda_tensor(w_router, bf, "w_router", 2)
    _cuda_tensor(bias, torch.float32, "bias", 1)
    T, D = x.shape
    E = w_router.shape[0]
    idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
    gates = torch.empty((T, k), dtype=torch.float32, device=x.device)
    tie = torch.empty((T,), dtype=torch.uint8, device=x.device)
    L = lib()
    ws = _workspace(L.moe_route_workspace_size(T, D, E, k), x.device, workspace)
    _check(L.moe_route(_ptr(x), _ptr(w_router), _ptr(bias), T, D, E, k, _ptr(idx), _ptr(gates),
                       _ptr(tie), _ptr(ws), ws.numel(), _stream(stream)), "moe_route")
    return idx, gates, tie


def moe_route_dispatch(x, w_router, bias, k: int, *, workspace=None, stream=None):
    """moe_route then moe_permute in one call; returns (idx, gates, tie, permutation dict)."""
    bf = torch.bfloat16
    _cuda_tensor(x, bf, "x", 2)
    _cuda_tensor(w_router, bf, "w_router", 2)
    _cuda_tensor(bias, torch.float32, "bias", 1)
    T, D = x.shape
    E = w_router.shape[0]
    dev = x.device
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gates = torch.empty((T, k), dtype=torch.float32, device=dev)
    tie = torch.empty((T,), dtype=torch.uint8, device=dev)
    p = {"counts": torch.empty((E,), dtype=torch.int32, device=dev),
         "offsets": torch.empty((E + 1,), dtype=torch.int32, device=dev),
         "row_token": torch.empty((T * k,), dtype=torch.int32, device=dev),
         "slot_row": torch.empty((T * k,), dtype=torch.int32, device=dev),
         "x_perm": torch.empty((T * k, D), dtype=bf, device=dev)}
    L = lib()
    ws = _workspace(L.moe_route_dispatch_workspace_size(T, D, E, k), dev, workspace)
    _check(L.moe_route_dispatch(_ptr(x), _ptr(w_router), _ptr(bias), T, D, E, k, _ptr(idx),
                                _ptr(gates), _ptr(tie), _ptr(p["counts"]), _ptr(p["offsets"]),
                                _ptr(p["row_token"]), _ptr(p["slot_row"]), _ptr(p["x_perm"]),
                                _ptr(ws), ws.numel(), _stream(stream)), "moe_route_dispatch")
    return idx, gates, tie, p


def moe_permute(topk_idx, x, E: int, *, workspace=None, stream=None):
    _cuda_tensor(topk_idx, torch.int32, "topk_idx", 2)
    _cuda_tensor(x, torch.bfloat16, "x", 2)
    T, k = topk_idx.shape
    H = x.shape[1]
    dev = x.device
    counts = torch.empty((E,), dtype=torch.int32, device=dev)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=dev)
    row_token = torch.empty((T * k,), dtype=torch.int32, device=dev)
    slot_row = torch.empty((T * k,), dtype=torch.int32, device=dev)
    x_perm = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
    L = lib()
    ws = _workspace(L.moe_permute_workspace_size(T, E, k), dev, workspace)
    _check(L.moe_permute(_ptr(topk_idx), _ptr(x), T, H, E, k, _ptr(counts), _ptr(offsets),
                         _ptr(row_token), _ptr(slot_row), _ptr(x_perm), _ptr(ws), ws.numel(),
                         _stream(stream)), "moe_permute")
    return {"counts": counts, "offsets": offsets, "row_token": row_token, "slot_row": slot_row,
            "x_perm": x_perm}


def moe_grouped_ffn(x_perm, offsets, w_up, w_down, *, out=None, workspace=None, stream=None):
    bf = torch.bfloat16
    _cuda_tensor(x_perm, bf, "x_perm", 2)
    _cuda_tensor(offsets, torch.int32, "offsets", 1)
    _cuda_tensor(w_up, bf, "w_up", 3)
    _cuda_tensor(w_down, bf, "w_down", 3)
    rows, H = x_perm.shape
    E, F, _ = w_up.shape
    y = out if out is not None else torch.empty((rows, H), dtype=bf, device=x_perm.device)
    L = lib()
    ws = _workspace(L.moe_grouped_ffn_workspace_size(rows, H, F, E), x_perm.device, workspace)
    _check(L.moe_grouped_ffn(_ptr(x_perm), _ptr(offsets), _ptr(w_up), _ptr(w_down), rows, H, F,
                             E, _ptr(y), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_grouped_ffn")
    return y


def moe_combine(y_perm, slot_row, gates, T: int, k: int, *, out=None, stream=None):
    _cuda_tensor(y_perm, torch.bfloat16, "y_perm", 2)
    _cuda_tensor(slot_row, torch.int32, "slot_row")
    _cuda_tensor(gates, torch.float32, "gates")
    rows, H = y_perm.shape
    y = out if out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=y_perm.device)
    _check(lib().moe_combine(_ptr(y_perm), rows, _ptr(slot_row), _ptr(gates), T, H, k, _ptr(y),
                             _stream(stream)), "moe_combine")
    return y


def moe_linear(x, w, *, out=None, stream=None):
    _cuda_tensor(x, torch.bfloat16, "x", 2)
    _cuda_tensor(w, torch.bfloat16, "w", 2)
    T, K = x.shape
    N = w.shape[0]
    y = out if out is not None else torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    _check(lib().moe_linear(_ptr(x), _ptr(w), T, K, N, _ptr(y), _stream(stream)), "moe_linear")
    return y


def moe_forward_workspace_size(T, H, E, k, F) -> int:
    return int(lib().moe_forward_workspace_size(T, H, E, k, F))


def moe_forward_fused_combine_workspace_size(T, H, E, k, F) -> int:
    return int(lib().moe_forward_fused_combine_workspace_size(T, H, E, k, F))


def moe_forward(x, w_router, bias, w_up, w_down, k: int, *, out=None, topk_idx_out=None,
                gates_out=None, workspace=None, stream=None, gathered: bool = False,
                fused_combine: bool = False):
    """gathered=True calls moe_forward_gathered (token rows gathered by the up-projection);
    fused_combine=True calls moe_forward_fused_combine (combine in the down-projection's
    epilogue, fixed-point sums)."""
    if gathered and fused_combine:
        raise ValueError("gathered and fused_combine select different entry points")
    bf = torch.bfloat16
    _cuda_tensor(x, bf, "x", 2)
    _cuda_tensor(w_router, bf, "w_router", 2)
    _cuda_tensor(bias, torch.float32, "bias", 1)
    _cuda_tensor(w_up, bf, "w_up", 3)
    _cuda_tensor(w_down, bf, "w_down", 3)
    T, H = x.shape
    E, F, _ = w_up.shape
    y = out if out is not None else torch.empty((T, H), dtype=bf, device=x.device)
    L = lib()
    if fused_combine:
        ws = _workspace(L.moe_forward_fused_combine_workspace_size(T, H, E, k, F), x.device,
                        workspace)
        fn = L.moe_forward_fused_combine
    else:
        ws = _workspace(L.moe_forward_workspace_size(T, H, E, k, F), x.device, workspace)
        fn = L.moe_forward_gathered if gathered else L.moe_forward
    _check(fn(_ptr(x), _ptr(w_router), _ptr(bias), _ptr(w_up), _ptr(w_down), T, H, E,
              k, F, _ptr(y), _ptr(topk_idx_out), _ptr(gates_out), _ptr(ws),
              ws.numel(), _stream(stream)), "moe_forward")
    return y


def latent_moe_workspace_size(T, H, L_, Ep, kp, F, router_on_latent=True) -> int:
    return int(lib().latent_moe_workspace_size(T, H, L_, Ep, kp, F, int(router_on_latent)))


def latent_moe(x, w_in, w_out, w_router, bias, w_up, w_down, kp: int, *,
               router_on_latent: bool = True, out=None, topk_idx_out=None, gates_out=None,
               workspace=None, stream=None):
    bf = torch.bfloat16
    for t, n, d in ((x, "x", 2), (w_in, "w_in", 2), (w_out, "w_out", 2),
                    (w_router, "w_router", 2), (w_up, "w_up", 3), (w_down, "w_down", 3)):
        _cuda_tensor(t, bf, n, d)
    _cuda_tensor(bias, torch.float32, "bias", 1)
    T, H = x.shape
    Lat = w_in.shape[0]
    Ep, F, _ = w_up.shape
    y = out if out is not None else torch.empty((T, H), dtype=bf, device=x.device)
    L = lib()
    ws = _workspace(L.latent_moe_workspace_size(T, H, Lat, Ep, kp, F, int(router_on_latent)),
                    x.device, workspace)
    _check(L.latent_moe(_ptr(x), _ptr(w_in), _ptr(w_out), _ptr(w_router), _ptr(bias),
                        int(router_on_latent), _ptr(w_up), _ptr(w_down), T, H, Lat, Ep, kp, F,
                        _ptr(y), _ptr(topk_idx_out), _ptr(gates_out), _ptr(ws), ws.numel(),
                        _stream(stream)), "latent_moe")
    return y


# ------------------------------------------------------------------------------ NVFP4 ----

class Nvfp4Weights:
    """G expert matrices [N, K] quantised to NVFP4 on the device (formats of include/moe.h):
    codes [G, N, K/2] uint8, scales (tile-ordered E4M3 atoms) uint8, gscale [G] fp32."""

    def __init__(self, codes, scales, gscale, G, N, K):
        self.codes, self.scales, self.gscale = codes, scales, gscale
        self.G, self.N, self.K = G, N, K

    def ptrs(self):
        return _ptr(self.codes), _ptr(self.scales), _ptr(self.gscale)


def moe_quantize_nvfp4_weights(w, *, blocks: str = "1d", stream=None) -> Nvfp4Weights:
    """blocks="1d": one scale per 16 K elements of a row; "2d": per 16 rows x 16 K."""
    if blocks not in ("1d", "2d"):
        raise ValueError("blocks must be '1d' or '2d'")
    _cuda_tensor(w, torch.bfloat16, "w", 3)
    G, N, K = w.shape
    L = lib()
    nc, ns = int(L.moe_nvfp4_codes_bytes(G, N, K)), int(L.moe_nvfp4_scales_bytes(G, N, K))
    if nc == 0 or ns == 0:
        raise MoeError(1, "moe_quantize_nvfp4_weights")
    codes = torch.empty((G, N, K // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((ns,), dtype=torch.uint8, device=w.device)
    gscale = torch.empty((G,), dtype=torch.float32, device=w.device)
    fn = L.moe_quantize_nvfp4_weights if blocks == "1d" else L.moe_quantize_nvfp4_weights_2d
    _check(fn(_ptr(w), G, N, K, _ptr(codes), _ptr(scales), _ptr(gscale), _stream(stream)),
           "moe_quantize_nvfp4_weights")
    return Nvfp4Weights(codes, scales, gscale, G, N, K)


def moe_grouped_ffn_nvfp4(x_perm, offsets, w_up: Nvfp4Weights, w_down: Nvfp4Weights, *,
                          out=None, workspace=None, stream=None):
    _cuda_tensor(x_perm, torch.bfloat16, "x_perm", 2)
    _cuda_tensor(offsets, torch.int32, "offsets", 1)
    rows, H = x_perm.shape
    E, F = w_up.G, w_up.N
    if (w_up.K, w_down.G, w_down.N, w_down.K) != (H, E, H, F):
        raise ValueError("NVFP4 weight shapes do not match x_perm")
    y = out if out is not None else torch.empty((rows, H), dtype=torch.bfloat16,
                                                device=x_perm.device)
    L = lib()
    ws = _workspace(L.moe_grouped_ffn_nvfp4_workspace_size(rows, H, F, E), x_perm.device,
                    workspace)
    _check(L.moe_grouped_ffn_nvfp4(_ptr(x_perm), _ptr(offsets), *w_up.ptrs(), *w_down.ptrs(),
                                   rows, H, F, E, _ptr(y), _ptr(ws), ws.numel(),
                                   _stream(stream)), "moe_grouped_ffn_nvfp4")
    return y


def moe_forward_nvfp4_workspace_size(T, H, E, k, F) -> int:
    return int(lib().moe_forward_nvfp4_workspace_size(T, H, E, k, F))


def moe_forward_nvfp4(x, w_router, bias, w_up: Nvfp4Weights, w_down: Nvfp4Weights, k: int, *,
                      out=None, topk_idx_out=None, gates_out=None, workspace=None, stream=None):
    bf = torch.bfloat16
    _cuda_tensor(x, bf, "x", 2)
    _cuda_tensor(w_router, bf, "w_router", 2)
    _cuda_tensor(bias, torch.float32, "bias", 1)
    T, H = x.shape
    E, F = w_up.G, w_up.N
    if (w_up.K, w_down.G, w_down.N, w_down.K) != (H, E, H, F):
        raise ValueError("NVFP4 weight shapes do not match x")
    y = out if out is not None else torch.empty((T, H), dtype=bf, device=x.device)
    L = lib()
    ws = _workspace(L.moe_forward_nvfp4_workspace_size(T, H, E, k, F), x.device, workspace)
    _check(L.moe_forward_nvfp4(_ptr(x), _ptr(w_router), _ptr(bias), *w_up.ptrs(),
                               *w_down.ptrs(), T, H, E, k, F, _ptr(y), _ptr(topk_idx_out),
                               _ptr(gates_out), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_forward_nvfp4")
    return y


# -------------------------------------------------------------------------------- FP8 ----

class Fp8Weights:
    """G expert matrices [N, K] quantised to per-tensor E4M3 on the device:
    codes [G, N, ldk] uint8 (ldk = K rounded up to 128; columns past K are padding) and
    scale [G] fp32 (include/moe.h)."""

    def __init__(self, codes, scale, G, N, K):
        self.codes, self.scale = codes, scale
        self.G, self.N, self.K = G, N, K

    def ptrs(self):
        return _ptr(self.codes), _ptr(self.scale)


def moe_quantize_fp8_weights(w, *, stream=None) -> Fp8Weights:
    _cuda_tensor(w, torch.bfloat16, "w", 3)
    G, N, K = w.shape
    ldk = int(lib().moe_fp8_codes_bytes(G, N, K)) // (G * N)
    codes = torch.zeros((G, N, ldk), dtype=torch.uint8, device=w.device)
    scale = torch.empty((G,), dtype=torch.float32, device=w.device)
    _check(lib().moe_quantize_fp8_weights(_ptr(w), G, N, K, _ptr(codes), _ptr(scale),
                                          _stream(stream)), "moe_quantize_fp8_weights")
    return Fp8Weights(codes, scale, G, N, K)


def moe_grouped_ffn_fp8(x_perm, offsets, w_up: Fp8Weights, w_down: Fp8Weights, *, out=None,
                        workspace=None, stream=None):
    _cuda_tensor(x_perm, torch.bfloat16, "x_perm", 2)
    _cuda_tensor(offsets, torch.int32, "offsets", 1)
    rows, H = x_perm.shape
    E, F = w_up.G, w_up.N
    if (w_up.K, w_down.G, w_down.N, w_down.K) != (H, E, H, F):
        raise ValueError("FP8 weight shapes do not match x_perm")
    y = out if out is not None else torch.empty((rows, H), dtype=torch.bfloat16,
                                                device=x_perm.device)
    L = lib()
    ws = _workspace(L.moe_grouped_ffn_fp8_workspace_size(rows, H, F, E), x_perm.device,
                    workspace)
    _check(L.moe_grouped_ffn_fp8(_ptr(x_perm), _ptr(offsets), *w_up.ptrs(), *w_down.ptrs(),
                                 rows, H, F, E, _ptr(y), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_grouped_ffn_fp8")
    return y


def moe_forward_fp8_workspace_size(T, H, E, k, F) -> int:
    return int(lib().moe_forward_fp8_workspace_size(T, H, E, k, F))


def moe_forward_fp8(x, w_router, bias, w_up: Fp8Weights, w_down: Fp8Weights, k: int, *,
                    out=None, topk_idx_out=None, gates_out=None, workspace=None, stream=None):
    bf = torch.bfloat16
    _cuda_tensor(x, bf, "x", 2)
    _cuda_tensor(w_router, bf, "w_router", 2)
    _cuda_tensor(bias, torch.float32, "bias", 1)
    T, H = x.shape
    E, F = w_up.G, w_up.N
    if (w_up.K, w_down.G, w_down.N, w_down.K) != (H, E, H, F):
        raise ValueError("FP8 weight shapes do not match x")
    y = out if out is not None else torch.empty((T, H), dtype=bf, device=x.device)
    L = lib()
    ws = _workspace(L.moe_forward_fp8_workspace_size(T, H, E, k, F), x.device, workspace)
    _check(L.moe_forward_fp8(_ptr(x), _ptr(w_router), _ptr(bias), *w_up.ptrs(), *w_down.ptrs(),
                             T, H, E, k, F, _ptr(y), _ptr(topk_idx_out), _ptr(gates_out),
                             _ptr(ws), ws.numel(), _stream(stream)), "moe_forward_fp8")
    return y


# ------------------------------------------------------------ quantised activation views ----

_VIEW_CALLS = {"grouped_ffn_nvfp4": "moe_grouped_ffn_nvfp4_view",
               "forward_nvfp4": "moe_forward_nvfp4_view",
               "grouped_ffn_fp8": "moe_grouped_ffn_fp8_view",
               "forward_fp8": "moe_forward_fp8_view"}


def quant_view(call: str, dims, workspace) -> dict:
    """Where the quantised activations of `call` sit inside `workspace` (a uint8 CUDA tensor
    used by that call with the same sizes). dims: (rows, H, F, E) for the grouped-FFN calls,
    (T, H, E, k, F) for the forward calls. Returns byte offsets into the workspace (None where
    the call has no such buffer) and "buffer_rows"."""
    _cuda_tensor(workspace, torch.uint8, "workspace")
    v = QuantView()
    _check(getattr(lib(), _VIEW_CALLS[call])(*[int(d) for d in dims], _ptr(workspace),
                                             workspace.numel(), ctypes.byref(v)),
           _VIEW_CALLS[call])
    base = workspace.data_ptr()
    sizes = ("buffer_rows", "x_codes_ld", "h_codes_ld")
    out = {name: (None if getattr(v, name) is None else getattr(v, name) - base)
           for name, _ in QuantView._fields_ if name not in sizes}
    for name in sizes:
        out[name] = int(getattr(v, name))
    return out


# ---------------------------------------------------------------------- shared expert ----

def moe_forward_shared(x, w_router, bias, w_up, w_down, w_up_shared, w_down_shared, k: int, *,
                       out=None, topk_idx_out=None, gates_out=None, workspace=None, stream=None):
    bf = torch.bfloat16
    for t, n, d in ((x, "x", 2), (w_router, "w_router", 2), (w_up, "w_up", 3),
                    (w_down, "w_down", 3), (w_up_shared, "w_up_shared", 2),
                    (w_down_shared, "w_down_shared", 2)):
        _cuda_tensor(t, bf, n, d)
    _cuda_tensor(bias, torch.float32, "bias", 1)
    T, H = x.shape
    E, F, _ = w_up.shape
    Fs = w_up_shared.shape[0]
    y = out if out is not None else torch.empty((T, H), dtype=bf, device=x.device)
    L = lib()
    ws = _workspace(L.moe_forward_shared_workspace_size(T, H, E, k, F, Fs), x.device, workspace)
    _check(L.moe_forward_shared(_ptr(x), _ptr(w_router), _ptr(bias), _ptr(w_up), _ptr(w_down),
                                _ptr(w_up_shared), _ptr(w_down_shared), T, H, E, k, F, Fs,
                                _ptr(y), _ptr(topk_idx_out), _ptr(gates_out), _ptr(ws),
                                ws.numel(), _stream(stream)), "moe_forward_shared")
    return y


def latent_moe_shared(x, w_in, w_out, w_router, bias, w_up, w_down, w_up_shared, w_down_shared,
                      kp: int, *, router_on_latent: bool = True, out=None, topk_idx_out=None,
                      gates_out=None, workspace=None, stream=None):
    bf = torch.bfloat16
    for t, n, d in ((x, "x", 2), (w_in, "w_in", 2), (w_out, "w_out", 2),
                    (w_router, "w_router", 2), (w_up, "w_up", 3), (w_down, "w_down", 3),
                    (w_up_shared, "w_up_shared", 2), (w_down_shared, "w_down_shared", 2)):
        _cuda_tensor(t, bf, n, d)
    _cuda_tensor(bias, torch.float32, "bias", 1)
    T, H = x.shape
    Lat = w_in.shape[0]
    Ep, F, _ = w_up.shape
    Fs = w_up_shared.shape[0]
    y = out if out is not None else torch.empty((T, H), dtype=bf, device=x.device)
    L = lib()
    ws = _workspace(L.latent_moe_shared_workspace_size(T, H, Lat, Ep, kp, F, Fs,
                                                       int(router_on_latent)), x.device,
                    workspace)
    _check(L.latent_moe_shared(_ptr(x), _ptr(w_in), _ptr(w_out), _ptr(w_router), _ptr(bias),
                               int(router_on_latent), _ptr(w_up), _ptr(w_down), _ptr(w_up_shared),
                               _ptr(w_down_shared), T, H, Lat, Ep, kp, F, Fs, _ptr(y),
                               _ptr(topk_idx_out), _ptr(gates_out), _ptr(ws), ws.numel(),
                               _stream(stream)), "latent_moe_shared")
    return y
