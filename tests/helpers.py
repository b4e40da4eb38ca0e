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
