"""Every call stays inside the workspace and the output it is given (needs a B300).

Each workspace is carved out of the middle of a larger buffer whose 64 KiB on either side
hold a fixed byte pattern (canaries); the layer output is placed the same way. After the
call completes, the canaries must be intact: a slice carved past the size the workspace
query reported, or a kernel indexing before or after its buffer, would overwrite them.
The calls run on small configurations that still take every code path of the big ones
(ragged tiles, empty experts, both GEMM operand orders, the CTA-pair GEMM, the fused
small-batch routing and the multi-kernel routing).
"""
import numpy as np
import pytest

import moe_synth
from helpers import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PAD = 64 << 10
PATTERN = 0xA5


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import sparse_mixture_experts_57_b300 as m
    m.lib()
    m.get_device_status()
    return m


class Guarded:
    """nbytes of device memory with PAD canary bytes on each side."""

    def __init__(self, nbytes):
        self.n = int(nbytes)
        self.buf = torch.full((self.n + 2 * PAD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.inner = self.buf[PAD:PAD + self.n]

    def as_bf16(self, shape):
        return self.inner.view(torch.bfloat16).view(shape)

    def intact(self):
        b = self.buf.cpu().numpy()
        return bool((b[:PAD] == PATTERN).all() and (b[PAD + self.n:] == PATTERN).all())


def _layer_inputs(T, H, E, k, F, seed, **kw):
    w = moe_synth.Workload("ws", T=T, H=H, E=E, k=k, F=F, seed=seed, **kw)
    inp = moe_synth.layer_inputs(w)
    return w, {n: to_dev(v) for n, v in inp.items()}


def _run_guarded(moe, call, ws_bytes, out_shape, *args, **kw):
    ws = Guarded(ws_bytes)
    out = Guarded(int(np.prod(out_shape)) * 2)
    call(*args, out=out.as_bf16(out_shape), workspace=ws.inner, **kw)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    assert ws.intact(), f"{call.__name__}: write outside the workspace"
    assert out.intact(), f"{call.__name__}: write outside the output"


# (T, H, E, k, F): fused small-batch routing, weights-as-M FFN / multi-kernel routing,
# rows-as-M FFN / CTA-pair FFN
SHAPES = [(64, 256, 16, 2, 128), (300, 320, 24, 3, 192), (2048, 256, 8, 2, 128)]


@pytest.mark.parametrize("T,H,E,k,F", SHAPES)
def test_moe_forward_stays_in_bounds(moe, T, H, E, k, F):
    w, d = _layer_inputs(T, H, E, k, F, seed=T)
    L = moe.lib()
    n = L.moe_forward_workspace_size(T, H, E, k, F)
    for gathered in (False, True):
        _run_guarded(moe, moe.moe_forward, n, (T, H), d["x"], d["w_router"], d["bias"],
                     d["w_up"], d["w_down"], k, gathered=gathered)
    n = L.moe_forward_fused_combine_workspace_size(T, H, E, k, F)
    _run_guarded(moe, moe.moe_forward, n, (T, H), d["x"], d["w_router"], d["bias"],
                 d["w_up"], d["w_down"], k, fused_combine=True)


@pytest.mark.parametrize("T,H,E,k,F", SHAPES)
def test_moe_forward_shared_stays_in_bounds(moe, T, H, E, k, F):
    w, d = _layer_inputs(T, H, E, k, F, seed=T + 1)
    s = {n: to_dev(v) for n, v in moe_synth.shared_expert_inputs(w, 192).items()}
    L = moe.lib()
    n = L.moe_forward_shared_workspace_size(T, H, E, k, F, 192)
    _run_guarded(moe, moe.moe_forward_shared, n, (T, H), d["x"], d["w_router"], d["bias"],
                 d["w_up"], d["w_down"], s["w_up_shared"], s["w_down_shared"], k)


@pytest.mark.parametrize("T", [200, 1100])
def test_latent_moe_stays_in_bounds(moe, T):
    H, Lat, E, k, F = 512, 128, 32, 8, 128
    for rol in (True, False):
        w, d = _layer_inputs(T, H, E, k, F, seed=T + 2, latent=Lat, router_on_latent=rol)
        L = moe.lib()
        n = L.latent_moe_workspace_size(T, H, Lat, E, k, F, int(rol))
        _run_guarded(moe, moe.latent_moe, n, (T, H), d["x"], d["w_in"], d["w_out"],
                     d["w_router"], d["bias"], d["w_up"], d["w_down"], k, router_on_latent=rol)
        s = {nm: to_dev(v) for nm, v in moe_synth.shared_expert_inputs(w, 128).items()}
        n = L.latent_moe_shared_workspace_size(T, H, Lat, E, k, F, 128, int(rol))
        _run_guarded(moe, moe.latent_moe_shared, n, (T, H), d["x"], d["w_in"], d["w_out"],
                     d["w_router"], d["bias"], d["w_up"], d["w_down"], s["w_up_shared"],
                     s["w_down_shared"], k, router_on_latent=rol)


@pytest.mark.parametrize("T,H,E,k,F", SHAPES)
def test_quantised_layers_stay_in_bounds(moe, T, H, E, k, F):
    w, d = _layer_inputs(T, H, E, k, F, seed=T + 3)
    L = moe.lib()
    nu = moe.moe_quantize_nvfp4_weights(d["w_up"])
    nd = moe.moe_quantize_nvfp4_weights(d["w_down"])
    n = L.moe_forward_nvfp4_workspace_size(T, H, E, k, F)
    _run_guarded(moe, moe.moe_forward_nvfp4, n, (T, H), d["x"], d["w_router"], d["bias"], nu,
                 nd, k)
    fu = moe.moe_quantize_fp8_weights(d["w_up"])
    fd = moe.moe_quantize_fp8_weights(d["w_down"])
    n = L.moe_forward_fp8_workspace_size(T, H, E, k, F)
    _run_guarded(moe, moe.moe_forward_fp8, n, (T, H), d["x"], d["w_router"], d["bias"], fu, fd,
                 k)


@pytest.mark.parametrize("T,H,E,k,F", SHAPES)
def test_pieces_stay_in_bounds(moe, T, H, E, k, F):
    """The separate calls: routing, permutation and the grouped FFNs (bf16, NVFP4, FP8)."""
    w, d = _layer_inputs(T, H, E, k, F, seed=T + 4)
    L = moe.lib()
    ws = Guarded(L.moe_route_workspace_size(T, H, E, k))
    idx, gates, tie = moe.moe_route(d["x"], d["w_router"], d["bias"], k, workspace=ws.inner)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0 and ws.intact(), "moe_route"
    ws = Guarded(L.moe_route_dispatch_workspace_size(T, H, E, k))
    moe.moe_route_dispatch(d["x"], d["w_router"], d["bias"], k, workspace=ws.inner)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0 and ws.intact(), "moe_route_dispatch"
    ws = Guarded(L.moe_permute_workspace_size(T, E, k))
    p = moe.moe_permute(idx, d["x"], E, workspace=ws.inner)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0 and ws.intact(), "moe_permute"
    rows = T * k
    n = L.moe_grouped_ffn_workspace_size(rows, H, F, E)
    _run_guarded(moe, moe.moe_grouped_ffn, n, (rows, H), p["x_perm"], p["offsets"], d["w_up"],
                 d["w_down"])
    nu = moe.moe_quantize_nvfp4_weights(d["w_up"])
    nd = moe.moe_quantize_nvfp4_weights(d["w_down"])
    n = L.moe_grouped_ffn_nvfp4_workspace_size(rows, H, F, E)
    _run_guarded(moe, moe.moe_grouped_ffn_nvfp4, n, (rows, H), p["x_perm"], p["offsets"], nu, nd)
    fu = moe.moe_quantize_fp8_weights(d["w_up"])
    fd = moe.moe_quantize_fp8_weights(d["w_down"])
    n = L.moe_grouped_ffn_fp8_workspace_size(rows, H, F, E)
    _run_guarded(moe, moe.moe_grouped_ffn_fp8, n, (rows, H), p["x_perm"], p["offsets"], fu, fd)
