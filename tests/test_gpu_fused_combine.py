"""moe_forward_fused_combine against the fp64 oracle (needs a B300).

The combine runs in the down-projection's epilogue: every routed row adds gate * output to
its token's 64-bit fixed-point sum, and a last pass writes y = bf16(sum * 2^-32). The shapes
reach the three epilogues that do this: weights on the MMA's M side (at most 48 rows per
expert), one-CTA rows-as-M tiles, and CTA-pair tiles (256 or more rows per expert).
"""
import numpy as np
import pytest

import moe_synth
from oracle import moe_oracle as O
from helpers import assert_close, bf16_out, check_selection, sample_tokens, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MOE_ERR_UNSUPPORTED = 2


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import sparse_mixture_experts_57_b300 as m
    m.lib()
    m.get_device_status()   # clears the status word
    return m


def _run(moe, inp, k, fused=True):
    dev = {key: to_dev(v) for key, v in inp.items()}
    T = inp["x"].shape[0]
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    y = moe.moe_forward(dev["x"], dev["w_router"], dev["bias"], dev["w_up"], dev["w_down"], k,
                        topk_idx_out=idx, gates_out=gates, fused_combine=fused)
    torch.cuda.synchronize()
    return y, idx.cpu().numpy()


# rows per expert: 1 and 33 (weights on M), 64 (one-CTA rows-as-M), 262 and 512 (CTA pairs,
# the first with a ragged last pair tile), plus the decode workload's shape
@pytest.mark.parametrize("T,H,E,k,F", [(1, 64, 4, 1, 64), (33, 128, 8, 8, 64),
                                       (64, 2688, 128, 6, 1856), (513, 256, 32, 4, 192),
                                       (700, 512, 8, 3, 448), (1024, 256, 4, 2, 192)])
def test_fused_combine_layer(moe, T, H, E, k, F):
    w = moe_synth.Workload("fused", T=T, H=H, E=E, k=k, F=F, seed=T + H + 11)
    inp = moe_synth.layer_inputs(w)
    y, gi = _run(moe, inp, k)
    assert moe.get_device_status() == 0
    ref = O.moe_layer(inp["x"], inp["w_router"], inp["bias"], inp["w_up"], inp["w_down"], k)
    same = check_selection(gi, ref, inp["bias"], k)
    assert_close(bf16_out(y)[same], ref["y"][same], f"fused combine T={T}")


@pytest.mark.parametrize("T,H,E,k,F", [(64, 2688, 128, 6, 1856), (1024, 256, 4, 2, 192)])
def test_fused_combine_is_deterministic(moe, T, H, E, k, F):
    """Integer sums do not depend on the order in which the tiles add their terms."""
    w = moe_synth.Workload("fused_det", T=T, H=H, E=E, k=k, F=F, seed=T + 5)
    inp = moe_synth.layer_inputs(w)
    y1, _ = _run(moe, inp, k)
    y2, _ = _run(moe, inp, k)
    assert moe.get_device_status() == 0
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("T,H,E,k,F", [(64, 2688, 128, 6, 1856), (700, 512, 8, 3, 448)])
def test_fused_combine_skips_a_rounding(moe, T, H, E, k, F):
    """The fused path sums the unrounded expert outputs, where moe_forward first rounds them
    to bf16 (y_perm): against the fp64 oracle its error is no larger."""
    w = moe_synth.Workload("fused_err", T=T, H=H, E=E, k=k, F=F, seed=T + 9)
    inp = moe_synth.layer_inputs(w)
    yf, gf = _run(moe, inp, k, fused=True)
    yu, gu = _run(moe, inp, k, fused=False)
    assert moe.get_device_status() == 0
    assert (gf == gu).all()
    ref = O.moe_layer(inp["x"], inp["w_router"], inp["bias"], inp["w_up"], inp["w_down"], k)
    same = check_selection(gf, ref, inp["bias"], k)
    rf_fused, _ = assert_close(bf16_out(yf)[same], ref["y"][same], "fused")
    rf_plain, _ = assert_close(bf16_out(yu)[same], ref["y"][same], "unfused")
    assert rf_fused <= rf_plain * 1.02, (rf_fused, rf_plain)


def test_fused_combine_reports_out_of_range_terms(moe):
    """A term |gate * output| >= 2^26 is not added and leaves MOE_ERR_UNSUPPORTED on the
    device status word; the call itself returns normally."""
    w = moe_synth.Workload("fused_range", T=40, H=128, E=8, k=2, F=64, seed=77)
    inp = moe_synth.layer_inputs(w)
    big = dict(inp)
    # bf16 weights times 2^40 (exact): the outputs far exceed the fixed-point sum's range
    big["w_down"] = _scale_bf16_bits(inp["w_down"], 40)
    _run(moe, big, w.k)
    assert moe.get_device_status() == MOE_ERR_UNSUPPORTED
    assert moe.get_device_status() == 0   # reading cleared it
    _run(moe, inp, w.k)
    assert moe.get_device_status() == 0


def _scale_bf16_bits(bits, e):
    """bf16 bit patterns times 2^e (exponent field shifted; zeros stay zero)."""
    b = bits.astype(np.uint32)
    exp = (b >> 7) & 0xFF
    nz = exp != 0
    assert (exp[nz] + e < 255).all()
    b = np.where(nz, b + (np.uint32(e) << 7), b)
    return b.astype(np.uint16)


@pytest.mark.slow
def test_fused_combine_nano_prefill_sampled(moe):
    """The prefill workload (16384 tokens, 128 experts, top-6, Zipf-biased routing) on the
    CTA-pair epilogue: routing on every token, outputs on sampled tokens."""
    w = moe_synth.WORKLOADS["nano_prefill"]
    inp = moe_synth.layer_inputs(w)
    y, gi = _run(moe, inp, w.k)
    assert moe.get_device_status() == 0
    ref = O.route(inp["x"], inp["w_router"], inp["bias"], w.k)
    same = check_selection(gi, ref, inp["bias"], w.k)
    toks = sample_tokens(w.T, ref["idx"], same, 200, w.seed)
    ref_y = O.moe_tokens(inp["x"][toks], ref["idx"][toks], ref["gates"][toks], inp["w_up"],
                         inp["w_down"])
    assert_close(bf16_out(y)[toks], ref_y, "fused combine, prefill sampled tokens")


def test_conversion_kernel_matches_host_rounding(moe):
    """The conversion kernel and the host path share one rounding function; on random 64-bit
    sums (every magnitude) the kernel's bf16 bits equal the host's, and on sums exact in
    float32 they equal torch's round-to-nearest-even."""
    import ctypes
    rng = np.random.default_rng(3)
    n = 1 << 20
    q = rng.integers(-(1 << 63), (1 << 63) - 1, size=n, dtype=np.int64, endpoint=True)
    q >>= rng.integers(0, 63, size=n, dtype=np.int64)      # spread the magnitudes
    host = np.zeros(n, dtype=np.uint16)
    L = moe.lib()
    assert L.moe_fixed_to_bf16(q.ctypes.data_as(ctypes.c_void_p), n,
                               host.ctypes.data_as(ctypes.c_void_p), 0, None) == 0
    qd = torch.from_numpy(q).cuda()
    out = torch.empty(n, dtype=torch.int16, device="cuda")
    assert L.moe_fixed_to_bf16(qd.data_ptr(), n, out.data_ptr(), 1, None) == 0
    torch.cuda.synchronize()
    assert (out.cpu().numpy().view(np.uint16) == host).all()
    small = q[np.abs(q) < (1 << 24)]
    want = torch.from_numpy(small.astype(np.float64) * 2.0 ** -32).to(torch.float32) \
        .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (host[np.abs(q) < (1 << 24)] == want).all()
