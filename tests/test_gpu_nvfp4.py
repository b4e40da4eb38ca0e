"""NVFP4 GPU path vs the fp64 oracle on seeded inputs (needs a B300).

The quantiser is compared bit for bit: every E2M1 code value, every E4M3 block scale and
every fp32 global scale. The block-scaled expert FFNs and the NVFP4 layer are compared on
outputs: relative Frobenius error <= 8e-2 over the whole output, and <= 0.15 for every row,
since a wrong block scale spoils a few rows (by 50% or more) rather than all of them.

Where the per-row bound comes from: the library stores the hidden activations h in bf16
before quantising them, while the oracle quantises the exact h. The bf16 rounding (about
2^-9 relative) moves some h values across an E2M1 rounding boundary, which changes them by a
whole E2M1 step. Evaluating the oracle with h rounded to bf16 shows the size of this effect
on these cases: about 2e-2 relative Frobenius over the output and up to 0.10 for single rows
when F is small (12 blocks per row), less for wider rows.
"""
import numpy as np
import pytest

import moe_synth
from oracle import moe_oracle as O
from helpers import (REL_FROB_NVFP4, bf16_out, check_selection, decode_codes, sample_tokens,
                     decode_e4m3_scale as decode_e4m3, scale_rows, tie_matrix, to_dev)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROW_REL_NVFP4 = 0.15


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import sparse_mixture_experts_57_b300 as m
    m.lib()
    m.get_device_status()
    return m


def _status_ok(moe):
    assert moe.get_device_status() == 0


def _rel_checks(got, ref, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), what
    rf = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    print(f"{what}: relative Frobenius error {rf:.3e}")
    assert rf <= REL_FROB_NVFP4, f"{what}: relative Frobenius error {rf:.3e}"
    rn = np.linalg.norm(ref, axis=1)
    live = rn > 1e-6 * max(rn.max(), 1e-30)
    per_row = np.linalg.norm(got - ref, axis=1)[live] / rn[live]
    worst = per_row.max() if per_row.size else 0.0
    assert worst <= ROW_REL_NVFP4, f"{what}: worst row relative error {worst:.3e}"
    return rf, worst


# --------------------------------------------------------------------- quantiser ----

def test_quantize_weights_bit_exact(moe):
    G, N, K = 5, 200, 320                  # ragged last 128-row block, 5 K steps
    rng = np.random.default_rng(31)
    w = rng.standard_normal((G, N, K)).astype(np.float32) / np.sqrt(K)
    # matrix 1: rows spanning 24 binades, so small blocks get subnormal E4M3 scales
    w[1] *= np.exp2(-(np.arange(N) % 24))[:, None].astype(np.float32)
    w[2] = 0.0                             # all-zero matrix: g = 0, every scale 0
    w[3, :, :16] = 0.0                     # all-zero blocks inside a live matrix
    w[4] = tie_matrix(N, K)               # rounding ties and their neighbours
    wb = moe_synth.bf16_bits(w)
    assert (O.widen_bf16(wb[4]) == w[4]).all()     # the tie values are exact in bf16
    nv = moe.moe_quantize_nvfp4_weights(to_dev(wb))
    torch.cuda.synchronize()
    _status_ok(moe)
    codes = nv.codes.cpu().numpy()
    sf = nv.scales.cpu().numpy().reshape(G, -1)
    gs = nv.gscale.cpu().numpy()
    for g in range(G):
        ref = O.nvfp4_quantize(wb[g])
        assert np.float32(gs[g]).tobytes() == np.float32(ref["g"]).tobytes(), g
        np.testing.assert_array_equal(decode_codes(codes[g]), ref["q"], err_msg=f"codes {g}")
        rows = scale_rows(sf[g], N, K)
        np.testing.assert_array_equal(decode_e4m3(rows[:N]), ref["sb"], err_msg=f"scales {g}")
        assert (rows[N:] == 0).all(), "scales of rows past N must be zero"


def test_quantize_weights_2d_bit_exact(moe):
    """2-D (16 rows x 16 K) weight blocks: every code value and every block scale (read per
    row from the tile-ordered atoms) equal the oracle's, including the ragged last row block."""
    G, N, K = 3, 200, 320
    rng = np.random.default_rng(32)
    w = rng.standard_normal((G, N, K)).astype(np.float32) / np.sqrt(K)
    w[1] *= np.exp2(-(np.arange(N) % 24))[:, None].astype(np.float32)
    w[2, :, :32] = 0.0
    wb = moe_synth.bf16_bits(w)
    nv = moe.moe_quantize_nvfp4_weights(to_dev(wb), blocks="2d")
    torch.cuda.synchronize()
    _status_ok(moe)
    codes = nv.codes.cpu().numpy()
    sf = nv.scales.cpu().numpy().reshape(G, -1)
    gs = nv.gscale.cpu().numpy()
    for g in range(G):
        ref = O.nvfp4_quantize_2d(wb[g])
        assert np.float32(gs[g]).tobytes() == np.float32(ref["g"]).tobytes(), g
        np.testing.assert_array_equal(decode_codes(codes[g]), ref["q"], err_msg=f"codes {g}")
        rows = scale_rows(sf[g], N, K)
        np.testing.assert_array_equal(decode_e4m3(rows[:N]), ref["sb"], err_msg=f"scales {g}")
        assert (rows[N:] == 0).all()


def test_grouped_ffn_nvfp4_2d_weights(moe):
    counts, H, F = [300, 0, 1, 129, 57, 200], 320, 192
    E = len(counts)
    off = _offsets(counts)
    rows = int(off[-1])
    seed = rows + H + 5
    xp = moe_synth.normal_bf16(seed, 50, (rows, H), 1.0)
    wu = moe_synth.expert_stack(seed, moe_synth.TAG_UP, E, F, H)
    wd = moe_synth.expert_stack(seed, moe_synth.TAG_DOWN, E, H, F)
    nu = moe.moe_quantize_nvfp4_weights(to_dev(wu), blocks="2d")
    nd = moe.moe_quantize_nvfp4_weights(to_dev(wd), blocks="2d")
    y = moe.moe_grouped_ffn_nvfp4(to_dev(xp), to_dev(off), nu, nd)
    torch.cuda.synchronize()
    _status_ok(moe)
    ref = O.grouped_ffn_nvfp4(xp, off, wu, wd, weight_blocks="2d")
    _rel_checks(bf16_out(y), ref, "nvfp4 grouped ffn, 2-D weight blocks")


# ------------------------------------------------------------------- grouped FFN ----

def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


@pytest.mark.parametrize("counts,H,F", [
    ([300, 0, 1, 129, 57, 200], 320, 192),     # empty, single-row, ragged and multi-tile groups
    ([128, 256, 127, 3], 256, 128),            # exact tile multiples and near misses
    ([40] * 30 + [700, 0], 512, 448),          # many small groups, one large, ragged N tiles
    ([90, 410, 5, 260], 2688, 1856),           # Nano widths: K tails of 2 and 1 MMA steps
    # many rows per expert: several row tiles per group with a partial last one, a ragged
    # single column tile (N = 192) and a K tail of one MMA step in a partial stage (K = 320)
    ([300, 0, 1, 129, 1000, 600], 320, 192),
    ([90, 410, 5, 700, 300], 2688, 1856),      # Nano widths, many row tiles per group
    # several row tiles per group, odd 128-row block counts (a half-filled last 256-row
    # tile), a single-row and an empty group. With 192-column tiles, N = 448 gives tiles
    # of 192, 192 and 64 columns: the second starts half way into a 128-row weight scale
    # block, the last has no second block (its scale box reads zeros past the tensor);
    # N = 320 gives 192 and 128, the second block partly past N
    ([600, 520, 130, 900], 320, 448),
    ([1200, 1, 800, 900, 0], 256, 448),
    ([385, 640, 1], 256, 576),                 # N = 576: three full 192-column tiles
    ([700, 900, 520, 1300], 2688, 1856),
])
def test_grouped_ffn_nvfp4(moe, counts, H, F):
    E = len(counts)
    off = _offsets(counts)
    rows = int(off[-1])
    seed = rows + H
    xp = moe_synth.normal_bf16(seed, 50, (rows, H), 1.0)
    wu = moe_synth.expert_stack(seed, moe_synth.TAG_UP, E, F, H)
    wd = moe_synth.expert_stack(seed, moe_synth.TAG_DOWN, E, H, F)
    nu = moe.moe_quantize_nvfp4_weights(to_dev(wu))
    nd = moe.moe_quantize_nvfp4_weights(to_dev(wd))
    y = moe.moe_grouped_ffn_nvfp4(to_dev(xp), to_dev(off), nu, nd)
    torch.cuda.synchronize()
    _status_ok(moe)
    ref = O.grouped_ffn_nvfp4(xp, off, wu, wd)
    _rel_checks(bf16_out(y), ref, f"nvfp4 grouped ffn {counts[:4]} H={H} F={F}")


# -------------------------------------------------------------------- whole layer ----

def _layer_nvfp4(moe, w):
    inp = moe_synth.layer_inputs(w)
    dev = {k: to_dev(v) for k, v in inp.items()}
    nu = moe.moe_quantize_nvfp4_weights(dev["w_up"])
    nd = moe.moe_quantize_nvfp4_weights(dev["w_down"])
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    y = moe.moe_forward_nvfp4(dev["x"], dev["w_router"], dev["bias"], nu, nd, w.k,
                              topk_idx_out=idx)
    torch.cuda.synchronize()
    _status_ok(moe)
    return inp, idx.cpu().numpy(), bf16_out(y)


@pytest.mark.parametrize("T,H,E,k,F", [(256, 256, 16, 2, 128), (700, 320, 10, 3, 192),
                                       (1, 64, 4, 1, 64), (2048, 256, 8, 2, 192)])
def test_layer_nvfp4(moe, T, H, E, k, F):
    w = moe_synth.Workload("nvfp4_small", T=T, H=H, E=E, k=k, F=F, seed=T + H, nvfp4=True)
    inp, gi, got = _layer_nvfp4(moe, w)
    ref = O.moe_layer_nvfp4(inp["x"], inp["w_router"], inp["bias"], inp["w_up"], inp["w_down"],
                            k)
    same = check_selection(gi, ref, inp["bias"], k)
    _rel_checks(got[same], ref["y"][same], f"nvfp4 layer T={T}")


@pytest.mark.slow
def test_layer_nvfp4_prefill_sampled(moe):
    """The full NVFP4 prefill workload: every token's routing, and sampled token outputs
    against the oracle, which needs the tensor-wide amax of the hidden activations."""
    w = moe_synth.WORKLOADS["nvfp4_prefill"]
    inp, gi, got = _layer_nvfp4(moe, w)
    ref = O.route(inp["x"], inp["w_router"], inp["bias"], w.k)
    same = check_selection(gi, ref, inp["bias"], w.k)
    h_amax = O.nvfp4_hidden_amax(inp["x"], ref["idx"], inp["w_up"])
    toks = sample_tokens(w.T, ref["idx"], same, 100, w.seed)
    ref_y = O.moe_tokens_nvfp4(inp["x"], inp["x"][toks], ref["idx"][toks], ref["gates"][toks],
                               inp["w_up"], inp["w_down"], h_amax=h_amax)
    _rel_checks(got[toks], ref_y, "nvfp4 prefill sampled tokens")
