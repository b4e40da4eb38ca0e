"""Seeded synthetic inputs for the routed MoE layer.

This module is shared by the fp64 oracle's tests and by the CUDA path's tests and
benchmark. It holds workload shapes and random-number recipes only, and none of the
layer's arithmetic (no routing, no FFN, no combine).

Every tensor comes from its own stream. The stream is keyed by (seed, tensor tag,
expert index), so one expert's weights can be regenerated alone: the oracle only
rebuilds the experts that sampled tokens touch. Values are drawn in float32 and
rounded to bfloat16 with round-to-nearest-even. They are returned as the raw uint16
bit patterns, and both sides read exactly those bits.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import math
import os

import numpy as np

# ----------------------------------------------------------------------------------------
# Workloads. Shapes follow the layer described in "NVIDIA Nemotron 3: Efficient and Open
# Intelligence" (papercache notes) §2.1-§2.2 (128 routable experts, 6 active in Nano; the
# LatentMoE ablation with H=4096, l=1024, E'=E*H/l, k'=k*H/l), and the news piece "NVIDIA AI
# 发布了Nemotron 3" (混合Mamba Transformer MoE架构: a learned router picks 6 of 128).
# ----------------------------------------------------------------------------------------

TAG_X, TAG_ROUTER, TAG_BIAS, TAG_UP, TAG_DOWN, TAG_WIN, TAG_WOUT, TAG_UP_S, TAG_DOWN_S = \
    range(1, 10)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens
    H: int            # model hidden size
    E: int            # routable experts (E' for the latent layer)
    k: int            # active experts per token (k' for the latent layer)
    F: int            # expert FFN intermediate size
    seed: int
    bias: str = "uniform"   # "uniform": U[-0.1, 0.1]; "zipf": -0.4*ln(e+1) + U[-0.05, 0.05]
    latent: int = 0         # l > 0 marks a LatentMoE layer (experts live in R^l)
    router_on_latent: bool = True
    nvfp4: bool = False
    fp8: bool = False       # per-tensor E4M3 experts

    @property
    def D(self) -> int:
        """Width of the expert input rows (l for the latent layer, H otherwise)."""
        return self.latent if self.latent else self.H

    @property
    def rows(self) -> int:
        return self.T * self.k


def latent_scaled(E: int, k: int, H: int, latent: int) -> tuple[int, int]:
    """E' = E*H/l and k' = k*H/l, the LatentMoE expert-count scaling (Nemotron 3 notes §2.2)."""
    if H % latent:
        raise ValueError("H must be a multiple of the latent size")
    r = H // latent
    return E * r, k * r


_EP, _KP = latent_scaled(128, 6, 4096, 1024)

WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", T=256, H=256, E=16, k=2, F=128, seed=0),
    "nano_decode": Workload("nano_decode", T=64, H=2688, E=128, k=6, F=1856, seed=1),
    "nano_prefill": Workload("nano_prefill", T=16384, H=2688, E=128, k=6, F=1856, seed=2,
                             bias="zipf"),
    "latent": Workload("latent", T=8192, H=4096, E=_EP, k=_KP, F=1024, seed=3, latent=1024),
    "nvfp4_prefill": Workload("nvfp4_prefill", T=16384, H=2688, E=128, k=6, F=1856, seed=4,
                              bias="zipf", nvfp4=True),
    # the decode and prefill layers with FP8 experts (same inputs as their bf16 versions)
    "nano_decode_fp8": Workload("nano_decode_fp8", T=64, H=2688, E=128, k=6, F=1856, seed=1,
                                fp8=True),
    "nano_prefill_fp8": Workload("nano_prefill_fp8", T=16384, H=2688, E=128, k=6, F=1856,
                                 seed=2, bias="zipf", fp8=True),
}


# ----------------------------------------------------------------------------------------
# bfloat16 bit handling (data format only)
# ----------------------------------------------------------------------------------------

def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen uint16 bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------------------
# Streams
# ----------------------------------------------------------------------------------------

def _rng(seed: int, tag: int, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, sub])))


def normal_bf16(seed: int, tag: int, shape, std: float, sub: int = 0) -> np.ndarray:
    g = _rng(seed, tag, sub)
    a = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return bf16_bits(a)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def expert_matrix(seed: int, tag: int, e: int, N: int, K: int) -> np.ndarray:
    """One expert's [N, K] weight matrix, N(0, 1/K), as bfloat16 bits."""
    return normal_bf16(seed, tag, (N, K), 1.0 / math.sqrt(K), sub=e)


def expert_stack(seed: int, tag: int, E: int, N: int, K: int,
                 experts=None) -> np.ndarray:
    """[E, N, K] stack of expert matrices (all, or only the listed experts; others zero)."""
    out = np.zeros((E, N, K), dtype=np.uint16)
    which = range(E) if experts is None else sorted(set(int(e) for e in experts))

    def fill(e):
        out[e] = expert_matrix(seed, tag, e, N, K)

    with _cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, which))
    return out


def router_bias(w: Workload) -> np.ndarray:
    """Per-expert selection bias (float32)."""
    g = _rng(w.seed, TAG_BIAS)
    if w.bias == "uniform":
        return g.uniform(-0.1, 0.1, size=w.E).astype(np.float32)
    if w.bias == "zipf":
        e = np.arange(w.E, dtype=np.float64)
        base = 0.5 * np.log(1.0 / (e + 1.0) ** 0.8)
        return (base + g.uniform(-0.05, 0.05, size=w.E)).astype(np.float32)
    raise ValueError(w.bias)


def layer_inputs(w: Workload, experts=None, with_experts: bool = True) -> dict:
    """All inputs of one layer as numpy arrays (bfloat16 as uint16 bits, bias float32).

    Keys: x [T,H]; w_router [E,D_r]; bias [E]; w_up [E,F,D]; w_down [E,D,F];
    and for the latent layer w_in [l,H], w_out [H,l].
    `experts` restricts which expert matrices are materialised (the rest are zero).
    """
    D = w.D
    d_router = D if (not w.latent or w.router_on_latent) else w.H
    out = {
        "x": normal_bf16(w.seed, TAG_X, (w.T, w.H), 1.0),
        "w_router": normal_bf16(w.seed, TAG_ROUTER, (w.E, d_router), 1.0 / math.sqrt(d_router)),
        "bias": router_bias(w),
    }
    if w.latent:
        out["w_in"] = normal_bf16(w.seed, TAG_WIN, (w.latent, w.H), 1.0 / math.sqrt(w.H))
        out["w_out"] = normal_bf16(w.seed, TAG_WOUT, (w.H, w.latent), 1.0 / math.sqrt(w.latent))
    if with_experts:
        out["w_up"] = expert_stack(w.seed, TAG_UP, w.E, w.F, D, experts)
        out["w_down"] = expert_stack(w.seed, TAG_DOWN, w.E, D, w.F, experts)
    return out


def shared_expert_inputs(w: Workload, Fs: int) -> dict:
    """Weights of one shared expert in H: w_up_shared [Fs, H] ~ N(0, 1/H) and
    w_down_shared [H, Fs] ~ N(0, 1/Fs), bfloat16 bits."""
    return {"w_up_shared": normal_bf16(w.seed, TAG_UP_S, (Fs, w.H), 1.0 / math.sqrt(w.H)),
            "w_down_shared": normal_bf16(w.seed, TAG_DOWN_S, (w.H, Fs), 1.0 / math.sqrt(Fs))}


def random_topk(seed: int, T: int, E: int, k: int, skew: float = 0.0) -> np.ndarray:
    """Seeded [T,k] int32 expert choices with k distinct experts per token.

    skew > 0 draws experts with probability proportional to (e+1)^-skew, which gives
    Zipf-like load imbalance. Used to test the permutation in isolation.
    """
    g = _rng(seed, 99)
    p = None
    if skew > 0:
        p = (np.arange(E, dtype=np.float64) + 1.0) ** (-skew)
        p /= p.sum()
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        out[t] = g.choice(E, size=k, replace=False, p=p)
    return out


def random_gates(seed: int, T: int, k: int) -> np.ndarray:
    """Seeded positive [T,k] float32 weights that sum to one per row."""
    g = _rng(seed, 98)
    a = g.uniform(0.05, 1.0, size=(T, k))
    return (a / a.sum(axis=1, keepdims=True)).astype(np.float32)


def to_torch(a: np.ndarray, device=None):
    """numpy array -> torch tensor (uint16 bit patterns become torch.bfloat16)."""
    import torch
    if a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device) if device is not None else t


def from_torch_bf16(t) -> np.ndarray:
    """torch.bfloat16 tensor -> numpy uint16 bit patterns."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
