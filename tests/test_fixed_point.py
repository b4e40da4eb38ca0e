"""The fused combine's conversion of 64-bit fixed-point sums to bf16 (CPU, host path).

moe_fixed_to_bf16 with on_device = 0 runs the same rounding function the conversion kernel
uses. It must return the bf16 nearest to q * 2^-32, ties to even. The expected values come
from torch's float32 -> bfloat16 conversion (round to nearest even) of inputs whose value
q * 2^-32 is exact in float32 (at most 24 significant bits), and from cases built around
exact ties, where the correct bf16 is known from the construction.
"""
import ctypes

import numpy as np
import pytest
import torch

import sparse_mixture_experts_57_b300 as moe


def _host_convert(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int64)
    out = np.zeros(q.shape, dtype=np.uint16)
    r = moe.lib().moe_fixed_to_bf16(q.ctypes.data_as(ctypes.c_void_p), q.size,
                                    out.ctypes.data_as(ctypes.c_void_p), 0, None)
    assert r == 0
    return out


def _torch_bf16_bits(q: np.ndarray) -> np.ndarray:
    """bf16 bits of q * 2^-32 for q whose magnitude has at most 24 significant bits."""
    v = torch.from_numpy(q.astype(np.float64) * 2.0 ** -32).to(torch.float32)
    assert (v.to(torch.float64).numpy() == q.astype(np.float64) * 2.0 ** -32).all()
    return v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _with_24_bits(rng, n):
    m = rng.integers(1, 1 << 24, size=n, dtype=np.int64)
    s = rng.integers(0, 40, size=n, dtype=np.int64)        # q < 2^63
    sign = np.where(rng.random(n) < 0.5, -1, 1)
    return sign * (m << s)


def test_matches_round_to_nearest_even():
    rng = np.random.default_rng(7)
    q = _with_24_bits(rng, 200_000)
    assert (_host_convert(q) == _torch_bf16_bits(q)).all()


def test_exact_ties_and_sticky_bits():
    rng = np.random.default_rng(8)
    b = rng.integers(0x80, 0x100, size=5000, dtype=np.int64)   # 8-bit significands 1xxxxxxx
    s = rng.integers(8, 30, size=5000, dtype=np.int64)
    tie = ((b << 1) | 1) << s            # exactly halfway between b and b + 1 (scaled)
    got_tie = _host_convert(tie)
    want_tie = _torch_bf16_bits(tie)     # 9 significant bits: exact in float32
    assert (got_tie == want_tie).all()
    # ties go to the even significand
    even = np.where(b % 2 == 0, b, b + 1)
    assert (_host_convert(even << (s + 1)) == want_tie).all()
    # one unit above or below the tie decides it, however far below the kept bits it sits
    assert (_host_convert(tie + 1) == _host_convert((b + 1) << (s + 1))).all()
    assert (_host_convert(tie - 1) == _host_convert(b << (s + 1))).all()


def test_special_values():
    q = np.array([0, 1, -1, (1 << 63) - 1, -(1 << 63), 1 << 32, -(3 << 31)], dtype=np.int64)
    got = _host_convert(q)
    assert got[0] == 0x0000
    assert got[1] == 0x2F80 and got[2] == 0xAF80         # +-2^-32
    assert got[3] == 0x4F00 and got[4] == 0xCF00         # +-2^31 (the first rounds up)
    assert got[5] == 0x3F80                              # 1.0
    assert got[6] == 0xBFC0                              # -1.5


def test_rejects_bad_arguments():
    L = moe.lib()
    assert L.moe_fixed_to_bf16(None, 4, None, 0, None) == 1
    assert L.moe_fixed_to_bf16(None, -1, None, 0, None) == 1
    assert L.moe_fixed_to_bf16(None, 0, None, 0, None) == 0
