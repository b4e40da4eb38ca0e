"""Byte-exact parity of the activation quantisers inside the NVFP4 and FP8 layer calls.

The NVFP4 and FP8 FFN calls quantise two activation tensors on the device: the routed
tokens entering the up-projection (gathered from x by the permutation in the layer calls,
read from x_perm in the grouped-FFN calls) and the hidden activations h entering the
down-projection. After a call, the library's workspace views (moe_*_view) say where those
buffers sit, and these tests read them back and compare every byte with the fp64 oracle's
quantiser ("NVIDIA Nemotron 3" notes §2.4 for NVFP4: E2M1 elements, an E4M3 scale per
16-element block, one fp32 scale per tensor; per-tensor E4M3 for FP8):
  * every E2M1 / E4M3 code value and every E4M3 block scale of every real row;
  * the zero codes and zero scales of the padding rows that round each NVFP4 expert segment
    up to whole 128-row tiles, and the padded segment offsets themselves;
  * the two amax words (fp32 bit patterns) that set the per-tensor scales.
For h the oracle is fed the GPU's own stored bf16 h, so the comparison is of the quantiser
alone: the library stores h in bf16 before quantising it, the oracle's layer functions
quantise the exact h. h itself is compared with the oracle's product of the dequantised
operands within bf16 rounding.

Cases: an empty expert, a one-row expert, segments one short of, equal to and one past a
128-row tile, tokens repeated across experts (each token is routed to k experts), values
exactly on E2M1 / E4M3 rounding boundaries and one bf16 step to either side, all-zero
blocks, and rows spread over many binades (E4M3 subnormal block scales).
"""
import numpy as np
import pytest

import moe_synth
from oracle import moe_oracle as O
from helpers import (decode_codes, decode_e4m3, decode_e4m3_scale, scale_rows, tie_matrix,
                     tie_matrix_e4m3, to_dev)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import sparse_mixture_experts_57_b300 as m
    m.lib()
    m.get_device_status()
    return m


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def _slice(ws, off, n, dtype=np.uint8):
    """n elements of `dtype` at byte offset off of the workspace, as numpy."""
    nbytes = n * np.dtype(dtype).itemsize
    return ws[off:off + nbytes].cpu().numpy().view(dtype)


def _activations(rows, K, seed, amax_tie):
    """bf16 rows [rows, K]: random rows spread over 20 binades, all-zero blocks, and (when
    amax_tie) the first rows taken from a rounding-boundary matrix whose amax then sets the
    tensor's scale."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((rows, K)).astype(np.float32)
    a *= np.exp2(-(np.arange(rows) % 20))[:, None].astype(np.float32)
    a[5::7, 16:48] = 0.0
    tie = amax_tie(min(rows, 40), K)
    a[:tie.shape[0]] = tie
    bits = moe_synth.bf16_bits(a)
    assert (O.widen_bf16(bits[:tie.shape[0]]) == tie).all()
    return bits


def _f32_bits(v) -> int:
    return int(np.float32(v).view(np.uint32))


def _amax_bits(bits) -> int:
    return _f32_bits(np.max(np.abs(O.widen_bf16(bits)))) if bits.size else 0


# --------------------------------------------------------------------------- NVFP4 ----

def _check_nvfp4_rows(codes_buf, ld, sf_buf, P, K, poff, counts, src_rows, g_ref, what):
    """Every real row of the padded buffers equals the oracle's quantisation of its source
    row with the tensor's global scale; padding rows hold zero codes and scales. Code rows
    are ld bytes apart (K/2 rounded up to 128)."""
    assert ld % 128 == 0 and K // 2 <= ld < K // 2 + 128
    codes = codes_buf.reshape(P, ld)[:, :K // 2]
    sf = scale_rows(sf_buf, P, K)
    live = np.zeros(P, bool)
    for e, c in enumerate(counts):
        live[poff[e]:poff[e] + c] = True
    q_ref = O.nvfp4_quantize(src_rows, g_ref)
    assert np.float32(q_ref["g"]).tobytes() == np.float32(g_ref).tobytes()
    rows_live = np.nonzero(live)[0]
    np.testing.assert_array_equal(decode_codes(codes[rows_live]), q_ref["q"],
                                  err_msg=f"{what}: E2M1 codes")
    np.testing.assert_array_equal(decode_e4m3_scale(sf[rows_live]), q_ref["sb"],
                                  err_msg=f"{what}: E4M3 block scales")
    pad = np.nonzero(~live[:int(poff[-1])])[0]
    assert (codes[pad] == 0).all(), f"{what}: padding rows must hold zero codes"
    assert (sf[pad] == 0).all(), f"{what}: padding rows must hold zero scales"
    return rows_live


def _check_nvfp4_view(view, ws, counts, H, F, src_rows, x_amax_src, wu):
    """Compare the x and h quantisation recorded in the workspace with the oracle."""
    E = len(counts)
    P = view["buffer_rows"]
    poff = _slice(ws, view["padded_offsets"], E + 1, np.int32)
    want = _offsets([(c + 127) // 128 * 128 for c in counts])
    np.testing.assert_array_equal(poff, want, err_msg="padded segment offsets")
    assert poff[-1] <= P
    amax = _slice(ws, view["amax"], 2, np.uint32)
    # routed tokens
    assert int(amax[0]) == _amax_bits(x_amax_src), "amax of the token tensor"
    gx = O.nvfp4_global_scale(np.max(np.abs(O.widen_bf16(x_amax_src))))
    ldx, ldh = view["x_codes_ld"], view["h_codes_ld"]
    live = _check_nvfp4_rows(_slice(ws, view["x_codes"], P * ldx), ldx,
                             _slice(ws, view["x_scales"], moe_nvfp4_sf_bytes(P, H)), P, H, poff,
                             counts, src_rows, gx, "routed tokens")
    # hidden activations: the stored bf16 h, its amax and its quantisation
    h = _slice(ws, view["h"], P * F, np.uint16).reshape(P, F)
    pad = np.setdiff1d(np.arange(int(poff[-1])), live)
    assert (h[pad] == 0).all(), "padding rows of h must be zero"
    h_live = h[live]
    assert int(amax[1]) == _amax_bits(h_live), "amax of h"
    gh = O.nvfp4_global_scale(np.max(np.abs(O.widen_bf16(h_live))))
    _check_nvfp4_rows(_slice(ws, view["h_codes"], P * ldh), ldh,
                      _slice(ws, view["h_scales"], moe_nvfp4_sf_bytes(P, F)), P, F, poff,
                      counts, h_live, gh, "hidden activations")
    # h itself: squared ReLU of the product of the dequantised operands (bf16 rounding)
    xq = O.nvfp4_quantize(src_rows, gx)["deq"]
    off = _offsets(counts)
    ref = np.zeros((len(h_live), F))
    for e, c in enumerate(counts):
        if c:
            ref[off[e]:off[e + 1]] = np.maximum(
                xq[off[e]:off[e + 1]] @ O.nvfp4_dequantize(wu[e]).T, 0.0) ** 2
    got = O.widen_bf16(h_live)
    err = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= 1e-2, f"h: relative Frobenius error {err:.3e}"


def moe_nvfp4_sf_bytes(rows, K):
    """Bytes of the scale atoms of a [rows, K] NVFP4 matrix (include/moe.h)."""
    return (rows + 127) // 128 * (K // 64) * 512


@pytest.mark.parametrize("counts,H,F", [
    ([300, 0, 1, 127, 128, 129, 57, 3], 320, 192),
    ([0, 1, 0, 256, 2], 256, 128),
    ([300, 0, 1, 600, 257], 256, 192),         # several row tiles per group
])
def test_grouped_ffn_nvfp4_activation_bytes(moe, counts, H, F):
    E = len(counts)
    off = _offsets(counts)
    rows = int(off[-1])
    xp = _activations(rows, H, rows + H, tie_matrix)
    wu = moe_synth.expert_stack(rows, moe_synth.TAG_UP, E, F, H)
    wd = moe_synth.expert_stack(rows, moe_synth.TAG_DOWN, E, H, F)
    nu = moe.moe_quantize_nvfp4_weights(to_dev(wu))
    nd = moe.moe_quantize_nvfp4_weights(to_dev(wd))
    L = moe.lib()
    ws = torch.empty(L.moe_grouped_ffn_nvfp4_workspace_size(rows, H, F, E), dtype=torch.uint8,
                     device="cuda")
    moe.moe_grouped_ffn_nvfp4(to_dev(xp), to_dev(off), nu, nd, workspace=ws)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    view = moe.quant_view("grouped_ffn_nvfp4", (rows, H, F, E), ws)
    assert view["offsets"] is None and view["row_token"] is None
    _check_nvfp4_view(view, ws, counts, H, F, xp, xp, wu)


def _layer(seed, T=300, E=64, k=4, H=256, F=192, **kw):
    # seed 43 (with the first 40 token rows replaced by a rounding-boundary matrix): the
    # expert loads include empty experts, a one-row expert and segments of more than one
    # 128-row tile that are not tile multiples (Zipf-skewed bias), and no near-ties
    return moe_synth.Workload("quant_act", T=T, H=H, E=E, k=k, F=F, seed=seed, bias="zipf", **kw)


def _dispatch_from_view(ws, view, w, idx):
    offsets = _slice(ws, view["offsets"], w.E + 1, np.int32)
    row_token = _slice(ws, view["row_token"], w.T * w.k, np.int32)
    p = O.permute(idx, w.E)
    np.testing.assert_array_equal(offsets, p["offsets"])
    np.testing.assert_array_equal(row_token, p["row_token"])
    counts = np.diff(offsets)
    assert (counts == 0).any() and (counts == 1).any()
    assert ((counts > 128) & (counts % 128 != 0)).any()
    return offsets, row_token, counts


def test_forward_nvfp4_gathered_activation_bytes(moe):
    """moe_forward_nvfp4 gathers each routed row from x by row_token and quantises it into
    the padded expert order in one pass: every token appears k times, in k experts."""
    w = _layer(43, nvfp4=True)
    inp = moe_synth.layer_inputs(w)
    x = inp["x"].copy()
    x[:40] = moe_synth.bf16_bits(tie_matrix(40, w.H))     # rounding boundaries; sets amax
    nu = moe.moe_quantize_nvfp4_weights(to_dev(inp["w_up"]))
    nd = moe.moe_quantize_nvfp4_weights(to_dev(inp["w_down"]))
    L = moe.lib()
    ws = torch.empty(L.moe_forward_nvfp4_workspace_size(w.T, w.H, w.E, w.k, w.F),
                     dtype=torch.uint8, device="cuda")
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    moe.moe_forward_nvfp4(to_dev(x), to_dev(inp["w_router"]), to_dev(inp["bias"]), nu, nd, w.k,
                          topk_idx_out=idx, workspace=ws)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    view = moe.quant_view("forward_nvfp4", (w.T, w.H, w.E, w.k, w.F), ws)
    _, row_token, counts = _dispatch_from_view(ws, view, w, idx.cpu().numpy())
    _check_nvfp4_view(view, ws, counts, w.H, w.F, x[row_token], x, inp["w_up"])


# ----------------------------------------------------------------------------- FP8 ----

def _check_fp8_view(ws, view, rows, H, F, src_rows, x_amax_src, wu, off):
    amax = _slice(ws, view["amax"], 2, np.uint32)
    assert view["buffer_rows"] == rows
    assert int(amax[0]) == _amax_bits(x_amax_src), "amax of the token tensor"
    sx = O.fp8_scale(np.max(np.abs(O.widen_bf16(x_amax_src))))
    ldx, ldh = view["x_codes_ld"], view["h_codes_ld"]
    assert ldx % 128 == 0 and ldh % 128 == 0 and ldx >= H and ldh >= F
    xq = _slice(ws, view["x_codes"], rows * ldx).reshape(rows, ldx)[:, :H]
    ref = O.fp8_quantize(src_rows, sx)
    np.testing.assert_array_equal(decode_e4m3(xq), ref["q"], err_msg="routed tokens: E4M3")
    h = _slice(ws, view["h"], rows * F, np.uint16).reshape(rows, F)
    assert int(amax[1]) == _amax_bits(h), "amax of h"
    sh = O.fp8_scale(np.max(np.abs(O.widen_bf16(h))))
    hq = _slice(ws, view["h_codes"], rows * ldh).reshape(rows, ldh)[:, :F]
    np.testing.assert_array_equal(decode_e4m3(hq), O.fp8_quantize(h, sh)["q"],
                                  err_msg="hidden activations: E4M3")
    href = np.zeros((rows, F))
    for e in range(len(off) - 1):
        if off[e + 1] > off[e]:
            href[off[e]:off[e + 1]] = np.maximum(
                ref["deq"][off[e]:off[e + 1]] @ O.fp8_dequantize(wu[e]).T, 0.0) ** 2
    got = O.widen_bf16(h)
    err = np.linalg.norm(got - href) / max(np.linalg.norm(href), 1e-30)
    assert err <= 1e-2, f"h: relative Frobenius error {err:.3e}"


def test_grouped_ffn_fp8_activation_bytes(moe):
    counts, H, F = [300, 0, 1, 127, 129, 57], 320, 192
    E = len(counts)
    off = _offsets(counts)
    rows = int(off[-1])
    xp = _activations(rows, H, rows + 7, tie_matrix_e4m3)
    wu = moe_synth.expert_stack(rows, moe_synth.TAG_UP, E, F, H)
    wd = moe_synth.expert_stack(rows, moe_synth.TAG_DOWN, E, H, F)
    fu = moe.moe_quantize_fp8_weights(to_dev(wu))
    fd = moe.moe_quantize_fp8_weights(to_dev(wd))
    L = moe.lib()
    ws = torch.empty(L.moe_grouped_ffn_fp8_workspace_size(rows, H, F, E), dtype=torch.uint8,
                     device="cuda")
    moe.moe_grouped_ffn_fp8(to_dev(xp), to_dev(off), fu, fd, workspace=ws)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    view = moe.quant_view("grouped_ffn_fp8", (rows, H, F, E), ws)
    assert view["padded_offsets"] is None and view["x_scales"] is None
    _check_fp8_view(ws, view, rows, H, F, xp, xp, wu, off)


def test_forward_fp8_gathered_activation_bytes(moe):
    w = _layer(43, fp8=True)
    inp = moe_synth.layer_inputs(w)
    x = inp["x"].copy()
    x[:40] = moe_synth.bf16_bits(tie_matrix_e4m3(40, w.H))
    fu = moe.moe_quantize_fp8_weights(to_dev(inp["w_up"]))
    fd = moe.moe_quantize_fp8_weights(to_dev(inp["w_down"]))
    L = moe.lib()
    ws = torch.empty(L.moe_forward_fp8_workspace_size(w.T, w.H, w.E, w.k, w.F),
                     dtype=torch.uint8, device="cuda")
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    moe.moe_forward_fp8(to_dev(x), to_dev(inp["w_router"]), to_dev(inp["bias"]), fu, fd, w.k,
                        topk_idx_out=idx, workspace=ws)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    view = moe.quant_view("forward_fp8", (w.T, w.H, w.E, w.k, w.F), ws)
    offsets, row_token, _ = _dispatch_from_view(ws, view, w, idx.cpu().numpy())
    _check_fp8_view(ws, view, w.T * w.k, w.H, w.F, x[row_token], x, inp["w_up"], offsets)
