"""Shared test helpers: tolerances, near-tie handling, device transfer."""
from __future__ import annotations

import numpy as np

import moe_synth
from oracle import moe_oracle as O

# Output tolerances for bf16 results: relative Frobenius error <= 1e-2 and
# max |err| <= 3e-2 * rms(oracle). NVFP4 results: relative Frobenius error <= 8e-2.
REL_FROB_BF16 = 1e-2
MAXABS_RMS_BF16 = 3e-2
REL_FROB_NVFP4 = 8e-2
# Tokens whose k-th and (k+1)-th biased scores differ by less than this are near-ties.
TIE_GAP = 1e-5


def f64(a) -> np.ndarray:
    return O.widen_bf16(a) if np.asarray(a).dtype == np.uint16 else np.asarray(a, np.float64)


def bf16_out(t) -> np.ndarray:
    """Device bf16 tensor -> float64 numpy."""
    return O.widen_bf16(moe_synth.from_torch_bf16(t))


def assert_close(got, ref, what="", rel_frob=REL_FROB_BF16, maxabs_rms=MAXABS_RMS_BF16):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = got - ref
    nref = np.linalg.norm(ref)
    rf = np.linalg.norm(err) / (nref if nref > 0 else 1.0)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    ma = np.abs(err).max() if err.size else 0.0
    assert rf <= rel_frob, f"{what}: relative Frobenius error {rf:.3e} > {rel_frob}"
    if maxabs_rms is not None:
        assert ma <= maxabs_rms * max(rms, 1e-30), \
            f"{what}: max abs error {ma:.3e} > {maxabs_rms} * rms {rms:.3e}"
    return rf, ma / max(rms, 1e-30)


def check_selection(gpu_idx: np.ndarray, ref: dict, bias: np.ndarray, k: int):
    """Selection parity with the near-tie rule.

    What is unique is compared exactly; what is not unique is checked for validity.
      * Tokens whose oracle gap u_(k) - u_(k+1) is at least TIE_GAP must select exactly the
        oracle's set of experts.
      * Inside the selected set, the order is by descending u. Two chosen experts whose u
        differ by less than TIE_GAP may appear in either order, so the GPU's order must be
        non-increasing in the oracle's u up to TIE_GAP.
      * Near-tie tokens may pick a different set, but it must still be a valid top-k within
        TIE_GAP: k distinct experts, each with u >= u_(k) - TIE_GAP.
    Returns the boolean mask of tokens whose expert set equals the oracle's.
    """
    gpu_idx = np.asarray(gpu_idx)
    o_idx = ref["idx"]
    gap = ref["gap"]
    u = ref["scores"] + np.asarray(bias, np.float64)[None, :]
    same = (np.sort(gpu_idx, axis=1) == np.sort(o_idx, axis=1)).all(axis=1)
    strict = gap >= TIE_GAP
    bad = np.nonzero(strict & ~same)[0]
    assert bad.size == 0, f"{bad.size} non-tie tokens select other experts, e.g. token {bad[:5]}"
    ug = np.take_along_axis(u, gpu_idx.astype(np.int64), axis=1)
    order_bad = np.nonzero((np.diff(ug, axis=1) > TIE_GAP).any(axis=1))[0]
    assert order_bad.size == 0, f"tokens {order_bad[:5]}: slots not in descending score order"
    for t in np.nonzero(~same)[0]:
        row = gpu_idx[t]
        assert len(set(row.tolist())) == k
        uk = u[t, o_idx[t, k - 1]]
        assert (u[t, row] >= uk - TIE_GAP).all(), f"token {t}: invalid near-tie choice"
    return same


def gates_by_expert(idx: np.ndarray, gates: np.ndarray) -> np.ndarray:
    """Reorder each token's gates by ascending expert index (slot order is not unique)."""
    order = np.argsort(idx, axis=1, kind="stable")
    return np.take_along_axis(np.asarray(gates, np.float64), order, axis=1)


def to_dev(a, device="cuda"):
    return moe_synth.to_torch(a, device)


# ------------------------------------------------------------------ format decoding ----
# Plain decoders of the library's documented NVFP4 and FP8 storage formats (include/moe.h).

E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def decode_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] -> E2M1 values [..., K]; element 2i in the low nibble."""
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(*codes.shape[:-1], -1)
    mag = E2M1_MAG[nib & 7]
    return np.where(nib & 8, -mag, mag)


def decode_e4m3_scale(b: np.ndarray) -> np.ndarray:
    """Non-negative E4M3 scale bytes (exponent bias 7, 3 mantissa bits) -> values."""
    b = b.astype(np.int64)
    e, m = (b >> 3) & 15, b & 7
    return np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * np.exp2(e - 7.0))


def scale_rows(buf: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Scale atoms of one matrix -> E4M3 bytes [ceil(rows/128)*128, K/16] in row order."""
    nb, ks = (rows + 127) // 128, K // 64
    a = buf.reshape(nb, ks, 32, 4, 4)          # block, K step, r0, r1, kb
    return a.transpose(0, 3, 2, 1, 4).reshape(nb * 128, ks * 4)


def decode_e4m3(b: np.ndarray) -> np.ndarray:
    """E4M3 bytes (sign bit 7, exponent bias 7, 3 mantissa bits) -> values."""
    b = np.asarray(b).astype(np.int64)
    mag = decode_e4m3_scale(b & 0x7F)
    return np.where(b & 0x80, -mag, mag)


def tie_matrix(N, K):
    """Values exactly on every E2M1 rounding boundary of their block, and one bf16 step to
    either side. The matrix amax is 168 = 2688 / 16, so g = 1/16 exactly; every other block
    has amax 6 g s for a block scale s with few mantissa bits, so its divisor is s g exactly
    and the boundaries t s g are exact bf16 values."""
    g = 1.0 / 16
    scales = [1.0, 1.25, 1.5, 1.75, 0.5625, 3.0, 0.75, 2.5]
    bounds = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    w = np.zeros((N, K), np.float32)
    for r in range(N):
        for b in range(K // 16):
            sc = scales[(r + b) % len(scales)]
            d = sc * g
            blk = [6 * g * sc]
            for i in range(15):
                t = bounds[(r * 3 + b + i) % len(bounds)]
                v = np.float32(t * d)
                side = (i + r) % 3                  # on, below, above the boundary
                if side:
                    bits = moe_synth.bf16_bits(np.array([v], np.float32)).astype(np.int32)
                    bits += 1 if side == 2 else -1
                    v = O.widen_bf16(bits.astype(np.uint16))[0]
                blk.append(v if (i + b) % 2 else -v)
            w[r, 16 * b:16 * b + 16] = blk
    w[0, 0] = 2688 * g                             # the matrix amax
    return w


def tie_matrix_e4m3(N, K):
    """Values exactly halfway between neighbouring E4M3 values (times s = 2^-4), and one bf16
    step to either side. amax = 448 / 16, so s = 1/16 exactly."""
    s = 1.0 / 16
    rng = np.random.default_rng(7)
    w = np.zeros((N, K), np.float32)
    for r in range(N):
        for c in range(K):
            ex = int(rng.integers(-6, 8))                # binade of the E4M3 value
            m = int(rng.integers(0, 7))
            lo = (1 + m / 8) * 2.0 ** ex
            v = np.float32((lo + 2.0 ** (ex - 3) / 2) * s)   # midpoint to the next value
            side = (r + c) % 3
            if side:
                bits = moe_synth.bf16_bits(np.array([v], np.float32)).astype(np.int32)
                bits += 1 if side == 2 else -1
                v = O.widen_bf16(bits.astype(np.uint16))[0]
            w[r, c] = v if (r + c) % 2 else -v
    w[0, 0] = 448 * s
    return w


def sample_tokens(T: int, idx: np.ndarray, same: np.ndarray, n: int, seed: int) -> np.ndarray:
    """Tokens for sampled full-size parity: the first and last token, n random ones, and for
    every expert that receives tokens the first token routed to it (so every touched
    expert's FFN is evaluated), restricted to tokens whose selection equals the oracle's."""
    rng = np.random.default_rng(seed)
    idx = np.asarray(idx)
    firsts = [int(np.nonzero((idx == e).any(axis=1))[0][0]) for e in np.unique(idx)]
    toks = np.unique(np.concatenate([[0, T - 1], rng.choice(T, min(n, T), replace=False),
                                     firsts]))
    return toks[same[toks]]
