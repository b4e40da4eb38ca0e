"""fp64 CPU oracle for the routed MoE / LatentMoE layer forward pass.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check of the package entry and the
benchmark's CPU-baseline leg may import this module. The CUDA path never calls it, and it
shares no code with the CUDA path. Inputs are the exact bfloat16 bit patterns widened to
float64, and every step is carried out in float64, except where noted for NVFP4.

Sources, by page and section:
  [N3]   "NVIDIA Nemotron 3: Efficient and Open Intelligence" (papercache notes):
         §2.1 hybrid MoE, §2.2 LatentMoE with Fig. 3b and the E' = E*H/l, k' = k*H/l
         formula, §2.4 NVFP4 training (format and latent projections kept in BF16).
  [NANO] "Nemotron 3 Nano" summary (papers.lianghsun.dev), §2.2: DeepSeek's
         aux-loss-free load balancing.
  [SHD]  "Nemotron 3 Nano" summary (shd-paper.top), 方法详解 / 技术框架: a routing
         network picks the experts, the experts run in parallel, and a combination
         layer forms the weighted combination of their outputs.
  [NEWS] "NVIDIA AI发布了Nemotron 3" (MarkTechPost translation), section
         混合Mamba Transformer MoE架构: a learned router picks 6 of 128 routable
         experts per token; MoE layers replace the FFN layers.

Readings where the pages are silent:
  * Scores are sigmoid(logits). The per-expert bias is added for SELECTION only (the
    aux-loss-free scheme [NANO]). Gates are the unbiased scores of the chosen experts,
    renormalised to sum to one, with no extra scale factor.
  * Top-k order: descending biased score, and the lower expert index wins exact ties.
  * Expert FFN: up-projection, squared ReLU max(0, .)^2, down-projection, no gating branch.
  * Rows inside an expert segment are in ascending token order.
  * LatentMoE applies W_out once, after the combine. W_out is linear, so this equals
    applying it per expert.

Parity status: the bf16 widening, routing, permutation, FFN, combine, per-token and
LatentMoE functions are pinned by the CPU tests in tests/test_oracle_pins.py (brute force,
closed forms, invariants, special cases, a full table of bf16 bit patterns). The NVFP4 and FP8 functions are pinned by exhaustive format tables, error
bounds and brute force.
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------------------
# data widening
# ----------------------------------------------------------------------------------------


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return widen_bf16(a)
    return a.astype(np.float64)


# ----------------------------------------------------------------------------------------
# Router ([NEWS] learned router, top-k of E routable experts; [NANO] aux-loss-free bias)
# ----------------------------------------------------------------------------------------


def router_logits(x, w_router) -> np.ndarray:
    """z[t, e] = sum_h x[t, h] * Wr[e, h] (fp64 matrix product)."""
    return _f64(x) @ _f64(w_router).T


def sigmoid(z: np.ndarray) -> np.ndarray:
    """s = 1 / (1 + exp(-z)), evaluated without overflow for large |z|."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = ez / (1.0 + ez)
    return out


def select_topk(scores: np.ndarray, bias: np.ndarray, k: int):
    """Pick the k experts with the largest biased score u = s + b for every token.

    Returns (idx [T,k] int32, gap [T] float64). idx is ordered by descending u, and the
    lower expert index wins on equal u. gap = u_(k) - u_(k+1) is +inf when k == E.
    """
    s = np.asarray(scores, dtype=np.float64)
    T, E = s.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    u = s + np.asarray(bias, dtype=np.float64)[None, :]
    idx = np.empty((T, k), dtype=np.int32)
    gap = np.full(T, np.inf)
    experts = np.arange(E)
    for t in range(T):
        order = np.lexsort((experts, -u[t]))     # primary: -u ascending, then e ascending
        idx[t] = order[:k]
        if k < E:
            gap[t] = u[t, order[k - 1]] - u[t, order[k]]
    return idx, gap


def gates_from_scores(scores: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """g[t, j] = s[t, idx[t, j]] / sum_j' s[t, idx[t, j']] (unbiased, renormalised)."""
    sel = np.take_along_axis(np.asarray(scores, dtype=np.float64), idx.astype(np.int64), axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def route_from_logits(z: np.ndarray, bias, k: int) -> dict:
    s = sigmoid(z)
    idx, gap = select_topk(s, bias, k)
    return {"idx": idx, "gates": gates_from_scores(s, idx), "scores": s, "gap": gap,
            "logits": np.asarray(z, dtype=np.float64)}


def route(x, w_router, bias, k: int) -> dict:
    """The full router: logits, sigmoid scores, biased top-k, renormalised gates."""
    return route_from_logits(router_logits(x, w_router), bias, k)


# ----------------------------------------------------------------------------------------
# Dispatch ([SHD] experts process their tokens in parallel): group (token, slot) pairs
# by expert.
# ----------------------------------------------------------------------------------------


def permute(idx: np.ndarray, E: int) -> dict:
    """Counting sort of the routed (token, slot) pairs by expert.

    counts[e]   number of rows routed to e;
    offsets[e]  exclusive prefix sum of counts (offsets[E] = T*k);
    row_token   token of each permuted row (ascending token order inside a segment);
    slot_row    permuted row of each (token, slot), flattened as t*k + j.
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    if idx.size and (idx.min() < 0 or idx.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:-1].copy()
    row_token = np.empty(T * k, dtype=np.int64)
    slot_row = np.empty(T * k, dtype=np.int64)
    for t in range(T):                  # visiting tokens in order keeps segments sorted
        for j in range(k):
            e = idx[t, j]
            r = fill[e]
            fill[e] += 1
            row_token[r] = t
            slot_row[t * k + j] = r
    return {"counts": counts.astype(np.int32), "offsets": offsets.astype(np.int32),
            "row_token": row_token.astype(np.int32), "slot_row": slot_row.astype(np.int32)}


def gather_rows(x, row_token) -> np.ndarray:
    return np.asarray(x)[np.asarray(row_token, dtype=np.int64)]


# ----------------------------------------------------------------------------------------
# Expert FFN ([N3] §2.2: each expert matrix is H x C; activation: squared ReLU)
# ----------------------------------------------------------------------------------------


def expert_ffn(rows, w_up_e, w_down_e) -> np.ndarray:
    """o = max(0, rows @ W_up^T)^2 @ W_down^T, with W_up [F, D] and W_down [D, F]."""
    a = _f64(rows) @ _f64(w_up_e).T
    h = np.maximum(a, 0.0) ** 2
    return h @ _f64(w_down_e).T


def grouped_ffn(x_perm, offsets, w_up, w_down) -> np.ndarray:
    """Apply every expert's FFN to its contiguous segment of permuted rows."""
    xp = _f64(x_perm)
    E = len(offsets) - 1
    D = np.asarray(w_down).shape[1]
    out = np.zeros((xp.shape[0], D))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            out[a:b] = expert_ffn(xp[a:b], w_up[e], w_down[e])
    return out


# ----------------------------------------------------------------------------------------
# Combination layer ([SHD] weighted combination of the chosen experts' outputs)
# ----------------------------------------------------------------------------------------


def combine(y_perm, slot_row, gates, T: int, k: int) -> np.ndarray:
    """y[t] = sum_j g[t, j] * y_perm[slot_row[t*k + j]]."""
    yp = _f64(y_perm)
    g = np.asarray(gates, dtype=np.float64).reshape(T, k)
    sr = np.asarray(slot_row, dtype=np.int64).reshape(T, k)
    y = np.zeros((T, yp.shape[1]))
    for j in range(k):
        y += g[:, j:j + 1] * yp[sr[:, j]]
    return y


# ----------------------------------------------------------------------------------------
# Whole layer
# ----------------------------------------------------------------------------------------


def moe_layer(x, w_router, bias, w_up, w_down, k: int) -> dict:
    """Route, permute, expert FFNs, combine: the standard routed MoE layer forward."""
    r = route(x, w_router, bias, k)
    E = np.asarray(w_router).shape[0]
    p = permute(r["idx"], E)
    x_perm = gather_rows(_f64(x), p["row_token"])
    y_perm = grouped_ffn(x_perm, p["offsets"], w_up, w_down)
    T = np.asarray(x).shape[0]
    y = combine(y_perm, p["slot_row"], r["gates"], T, k)
    return {"y": y, **r, **p}


def moe_tokens(x_rows, idx_rows, gates_rows, w_up, w_down) -> np.ndarray:
    """Layer output for a subset of tokens, given their routing (per-token evaluation).

    Used for sampled parity at full size: y[t] = sum_j g[t,j] * FFN_{idx[t,j]}(x[t]).
    """
    xr = _f64(x_rows)
    n, k = np.asarray(idx_rows).shape
    out = np.zeros((n, np.asarray(w_down).shape[1]))
    by_expert: dict[int, list[tuple[int, int]]] = {}
    for i in range(n):
        for j in range(k):
            by_expert.setdefault(int(idx_rows[i][j]), []).append((i, j))
    for e, pairs in by_expert.items():
        ii = np.array([p[0] for p in pairs])
        jj = np.array([p[1] for p in pairs])
        o = expert_ffn(xr[ii], w_up[e], w_down[e])
        np.add.at(out, ii, np.asarray(gates_rows, dtype=np.float64)[ii, jj][:, None] * o)
    return out


def latent_project_in(x, w_in) -> np.ndarray:
    """x_lat = x @ W_in^T : H -> l ([N3] §2.2, Fig. 3b)."""
    return _f64(x) @ _f64(w_in).T


def latent_moe(x, w_in, w_out, w_router, bias, w_up, w_down, kp: int,
               router_on_latent: bool = True) -> dict:
    """LatentMoE ([N3] §2.2, Fig. 3b): project H -> l, route to E' experts with k' active,
    run the experts in l, combine in l, project l -> H.

    router_on_latent selects the router input: the latent vector (as in the seeded
    latent workload), or the hidden-size token (the §2.2 remark that the routing gate
    stays in H). w_router is [E', l] or [E', H] accordingly.
    """
    x_lat = latent_project_in(x, w_in)
    r = route(x_lat if router_on_latent else x, w_router, bias, kp)
    E = np.asarray(w_router).shape[0]
    p = permute(r["idx"], E)
    y_perm = grouped_ffn(gather_rows(x_lat, p["row_token"]), p["offsets"], w_up, w_down)
    T = x_lat.shape[0]
    y_lat = combine(y_perm, p["slot_row"], r["gates"], T, kp)
    y = y_lat @ _f64(w_out).T
    return {"y": y, "y_lat": y_lat, "x_lat": x_lat, **r, **p}


# ----------------------------------------------------------------------------------------
# Shared expert ([N3] §2.2: the shared-expert computation, like the routing gate, stays in
# the hidden size H). Reading: an FFN of the routed experts' form (up, squared ReLU, down)
# applied to every token with weight 1 and added to the routed output. Several shared
# experts of width F_s sum to one FFN whose intermediate width is their total.
# ----------------------------------------------------------------------------------------


def shared_ffn(x, w_up_s, w_down_s) -> np.ndarray:
    """max(0, x @ W_up_s^T)^2 @ W_down_s^T for every token (W_up_s [F_s, H], W_down_s [H, F_s])."""
    return expert_ffn(x, w_up_s, w_down_s)


def moe_layer_shared(x, w_router, bias, w_up, w_down, w_up_s, w_down_s, k: int) -> dict:
    """Routed MoE layer plus the shared expert: y = routed(x) + shared(x)."""
    out = moe_layer(x, w_router, bias, w_up, w_down, k)
    out["y_routed"] = out["y"]
    out["y"] = out["y"] + shared_ffn(x, w_up_s, w_down_s)
    return out


def latent_moe_shared(x, w_in, w_out, w_router, bias, w_up, w_down, w_up_s, w_down_s, kp: int,
                      router_on_latent: bool = True) -> dict:
    """LatentMoE plus a shared expert in H: y = W_out(latent routed(x)) + shared(x)."""
    out = latent_moe(x, w_in, w_out, w_router, bias, w_up, w_down, kp, router_on_latent)
    out["y"] = out["y"] + shared_ffn(x, w_up_s, w_down_s)
    return out


# ----------------------------------------------------------------------------------------
# NVFP4 ([N3] §2.4): E2M1 elements, one E4M3 scale per 16-element micro-block, and a
# second-level FP32 per-tensor scale. Blocks run along the contraction (K) axis.
# Scale and code decisions are made in float32, the precision the pages give to the
# second-level scale; dequantised values are exact in float64.
# ----------------------------------------------------------------------------------------

E2M1_MAX = 6.0
E4M3_MAX = 448.0
NVFP4_BLOCK = 16


def e2m1_round(v) -> np.ndarray:
    """Round to the nearest E2M1 value (ties to the even code), saturating at +-6.

    E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit. Magnitudes 0, 0.5, 1, 1.5, 2, 3,
    4, 6: spacing 0.5 below 2, 1 in [2, 4), 2 in [4, 6].
    """
    v = np.asarray(v, dtype=np.float64)
    m = np.abs(v)
    q = np.where(m < 2.0, 0.5, np.where(m < 4.0, 1.0, 2.0))
    r = np.rint(m / q) * q                      # rint: round half to even
    r = np.minimum(r, E2M1_MAX)
    return np.copysign(r, v)


def e4m3_round(v) -> np.ndarray:
    """Round to the nearest E4M3 (OCP FP8 "fn") value, ties to even, saturating at +-448.

    E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; smallest normal 2^-6, subnormal
    spacing 2^-9, largest finite 448 = 1.75 * 2^8, no infinities.
    """
    v = np.asarray(v, dtype=np.float64)
    m = np.abs(v)
    _, ex = np.frexp(m)                          # m = f * 2^ex with f in [0.5, 1)
    e = np.maximum(ex - 1, -6)                   # binade exponent, subnormals share -6
    quantum = np.ldexp(1.0, e - 3)
    r = np.rint(m / quantum) * quantum
    r = np.where(m == 0, 0.0, r)
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, v)


def nvfp4_global_scale(amax) -> np.float32:
    """Per-tensor FP32 scale g = amax / (6 * 448), so the largest block scale is 448."""
    return np.float32(np.float32(amax) / np.float32(E2M1_MAX * E4M3_MAX))


def nvfp4_quantize(mat, g: np.float32 | None = None) -> dict:
    """Quantise a [rows, K] matrix into NVFP4 with 16-element blocks along K.

    Block scale sb = E4M3(amax(block) / (6 g)); element code q = E2M1(v / (sb g)).
    A block whose scale rounds to zero gets zero codes. The decisions use float32, as
    a kernel holding an FP32 global scale would. Returns the E2M1 values q [rows, K],
    the block scales sb [rows, K/16] (values), g, and the dequantised matrix q*sb*g.
    """
    a32 = np.asarray(_f64(mat), dtype=np.float32)
    rows, K = a32.shape
    if K % NVFP4_BLOCK:
        raise ValueError("K must be a multiple of 16")
    if g is None:
        g = nvfp4_global_scale(np.max(np.abs(a32)) if a32.size else 0.0)
    g = np.float32(g)
    blocks = a32.reshape(rows, K // NVFP4_BLOCK, NVFP4_BLOCK)
    bmax = np.max(np.abs(blocks), axis=2)
    if g > 0:
        ratio = bmax / (np.float32(E2M1_MAX) * g)                  # float32 arithmetic
        sb = e4m3_round(ratio.astype(np.float64)).astype(np.float32)
    else:
        sb = np.zeros_like(bmax)
    denom = (sb * g).astype(np.float32)                              # float32 product
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = np.where(denom[:, :, None] > 0, blocks / denom[:, :, None], np.float32(0))
    q = e2m1_round(scaled.astype(np.float64))
    deq = q * denom.astype(np.float64)[:, :, None]
    return {"q": q.reshape(rows, K), "sb": sb.astype(np.float64), "g": g,
            "deq": deq.reshape(rows, K)}


def nvfp4_dequantize(mat, g: np.float32 | None = None) -> np.ndarray:
    return nvfp4_quantize(mat, g)["deq"]


def nvfp4_quantize_2d(mat, g: np.float32 | None = None) -> dict:
    """NVFP4 with 2-D weight blocks ([N3] §2.4: 2-D block scaling for weights): one E4M3
    scale per 16 rows x 16 K elements (a last block of fewer rows when rows % 16 != 0).

    sb = E4M3(amax(16x16 block) / (6 g)); every element of the block is coded as in
    nvfp4_quantize with that scale. Returns q [rows, K], sb [rows, K/16] (each row's
    scale, repeated over the block's rows), g and deq.
    """
    a32 = np.asarray(_f64(mat), dtype=np.float32)
    rows, K = a32.shape
    if K % NVFP4_BLOCK:
        raise ValueError("K must be a multiple of 16")
    if g is None:
        g = nvfp4_global_scale(np.max(np.abs(a32)) if a32.size else 0.0)
    g = np.float32(g)
    nb = K // NVFP4_BLOCK
    sb = np.zeros((rows, nb), dtype=np.float32)
    for r0 in range(0, rows, NVFP4_BLOCK):
        blk = a32[r0:r0 + NVFP4_BLOCK].reshape(-1, nb, NVFP4_BLOCK)
        bmax = np.max(np.abs(blk), axis=(0, 2))                      # per 16x16 block
        if g > 0:
            ratio = bmax / (np.float32(E2M1_MAX) * g)                    # float32 arithmetic
            sb[r0:r0 + NVFP4_BLOCK] = e4m3_round(ratio.astype(np.float64)).astype(np.float32)
    denom = (sb * g).astype(np.float32)
    blocks = a32.reshape(rows, nb, NVFP4_BLOCK)
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = np.where(denom[:, :, None] > 0, blocks / denom[:, :, None], np.float32(0))
    q = e2m1_round(scaled.astype(np.float64))
    deq = q * denom.astype(np.float64)[:, :, None]
    return {"q": q.reshape(rows, K), "sb": sb.astype(np.float64), "g": g,
            "deq": deq.reshape(rows, K)}


def nvfp4_weight_dequantize(w, weight_blocks: str = "1d") -> np.ndarray:
    """Dequantised NVFP4 weight matrix with 1-D (16 along K) or 2-D (16x16) block scales."""
    if weight_blocks == "2d":
        return nvfp4_quantize_2d(w)["deq"]
    if weight_blocks != "1d":
        raise ValueError(weight_blocks)
    return nvfp4_dequantize(w)


def moe_tokens_nvfp4(x_all, x_rows, idx_rows, gates_rows, w_up, w_down, h_amax=None,
                     weight_blocks: str = "1d"):
    """NVFP4 layer output for a subset of tokens.

    Expert weights are quantised per expert matrix. The routed activations use one
    global scale over the whole permuted input (equal to that of x, since every token
    is routed). The hidden activations h use one global scale over the whole h tensor;
    h_amax supplies that tensor-wide amax when only a sample of rows is evaluated.
    """
    gx = nvfp4_global_scale(np.max(np.abs(_f64(x_all).astype(np.float32))))
    xr = nvfp4_dequantize(x_rows, gx)
    n, k = np.asarray(idx_rows).shape
    out = np.zeros((n, np.asarray(w_down).shape[1]))
    hs = []
    wu_cache: dict[int, np.ndarray] = {}
    for i in range(n):
        for j in range(k):
            e = int(idx_rows[i][j])
            if e not in wu_cache:
                wu_cache[e] = nvfp4_weight_dequantize(w_up[e], weight_blocks)
            a = xr[i:i + 1] @ wu_cache[e].T
            hs.append((i, j, e, np.maximum(a, 0.0) ** 2))
    if h_amax is None:
        h_amax = max(float(np.max(np.abs(h[3]))) for h in hs) if hs else 0.0
    gh = nvfp4_global_scale(np.float32(h_amax))
    wd_cache: dict[int, np.ndarray] = {}
    for i, j, e, h in hs:
        if e not in wd_cache:
            wd_cache[e] = nvfp4_weight_dequantize(w_down[e], weight_blocks)
        hq = nvfp4_dequantize(h.astype(np.float32), gh)
        out[i] += float(gates_rows[i][j]) * (hq @ wd_cache[e].T)[0]
    return out


def nvfp4_hidden_amax(x, idx, w_up, weight_blocks: str = "1d") -> float:
    """amax of the hidden activations h over every routed (token, expert) pair, with the
    tokens and the up-projection weights in NVFP4 as in grouped_ffn_nvfp4. This is the
    tensor-wide amax that sets the global scale of h; moe_tokens_nvfp4 takes it as h_amax
    when only a sample of tokens is evaluated."""
    xq = nvfp4_dequantize(_f64(x).astype(np.float32))
    idx = np.asarray(idx)
    amax = 0.0
    for e in np.unique(idx):
        toks = np.nonzero((idx == e).any(axis=1))[0]
        a = xq[toks] @ nvfp4_weight_dequantize(w_up[int(e)], weight_blocks).T
        amax = max(amax, float(np.max(np.maximum(a, 0.0) ** 2)))
    return amax


def grouped_ffn_nvfp4(x_perm, offsets, w_up, w_down, weight_blocks: str = "1d") -> np.ndarray:
    """The expert FFNs with NVFP4 operands ([N3] §2.4).

    Each expert matrix is quantised with its own global scale. The permuted activations are
    quantised with one global scale over the whole x_perm tensor, and the hidden activations
    with one over the whole h tensor (all experts). Products and sums are exact in fp64 on
    the dequantised values.
    """
    xp = _f64(x_perm).astype(np.float32)
    E = len(offsets) - 1
    xq = nvfp4_dequantize(xp)
    hs = {}
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            hs[e] = np.maximum(xq[a:b] @ nvfp4_weight_dequantize(w_up[e], weight_blocks).T,
                               0.0) ** 2
    h_amax = max((float(np.max(np.abs(h))) for h in hs.values()), default=0.0)
    gh = nvfp4_global_scale(np.float32(h_amax))
    out = np.zeros((xp.shape[0], np.asarray(w_down).shape[1]))
    for e, h in hs.items():
        a, b = int(offsets[e]), int(offsets[e + 1])
        out[a:b] = (nvfp4_dequantize(h.astype(np.float32), gh)
                    @ nvfp4_weight_dequantize(w_down[e], weight_blocks).T)
    return out


def moe_layer_nvfp4(x, w_router, bias, w_up, w_down, k: int, weight_blocks: str = "1d") -> dict:
    """Routed MoE layer with NVFP4 experts: bf16 routing, NVFP4 expert FFNs, fp64 combine."""
    r = route(x, w_router, bias, k)
    E = np.asarray(w_router).shape[0]
    p = permute(r["idx"], E)
    y_perm = grouped_ffn_nvfp4(gather_rows(x, p["row_token"]), p["offsets"], w_up, w_down,
                               weight_blocks)
    T = np.asarray(x).shape[0]
    return {"y": combine(y_perm, p["slot_row"], r["gates"], T, k), **r, **p}


# ----------------------------------------------------------------------------------------
# FP8 experts ("Nemotron 3 Nano" summary, §4: FP8 post-training quantisation with selective
# precision; BF16 and FP8 weights are released). The pages give no scaling granularity;
# the reading here is per-tensor E4M3: one FP32 scale s = amax / 448 per expert matrix, one
# over the whole routed-token tensor and one over the whole h. Elements q = E4M3(v / s),
# nearest with ties to even, saturating at +-448; value q * s. Decisions in float32.
# ----------------------------------------------------------------------------------------


def fp8_scale(amax) -> np.float32:
    """Per-tensor FP32 scale s = amax / 448, so the largest magnitude maps to E4M3's max."""
    return np.float32(np.float32(amax) / np.float32(E4M3_MAX))


def fp8_quantize(mat, s: np.float32 | None = None) -> dict:
    """Quantise a matrix to E4M3 with one FP32 scale. Returns the E4M3 values q, s and the
    dequantised matrix q*s. A zero scale gives zero codes."""
    a32 = np.asarray(_f64(mat), dtype=np.float32)
    if s is None:
        s = fp8_scale(np.max(np.abs(a32)) if a32.size else 0.0)
    s = np.float32(s)
    if s > 0:
        with np.errstate(over="ignore"):
            q = e4m3_round((a32 / s).astype(np.float64))     # float32 division, then rounding
    else:
        q = np.zeros(a32.shape)
    return {"q": q, "s": s, "deq": q * np.float64(s)}


def fp8_dequantize(mat, s: np.float32 | None = None) -> np.ndarray:
    return fp8_quantize(mat, s)["deq"]


def grouped_ffn_fp8(x_perm, offsets, w_up, w_down) -> np.ndarray:
    """The expert FFNs with FP8 operands: per-tensor scales for every expert matrix, for the
    whole x_perm and for the whole h (all experts); fp64 products of the dequantised values."""
    xp = _f64(x_perm).astype(np.float32)
    E = len(offsets) - 1
    xq = fp8_dequantize(xp)
    hs = {}
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            hs[e] = np.maximum(xq[a:b] @ fp8_dequantize(w_up[e]).T, 0.0) ** 2
    h_amax = max((float(np.max(h)) for h in hs.values()), default=0.0)
    sh = fp8_scale(np.float32(h_amax))
    out = np.zeros((xp.shape[0], np.asarray(w_down).shape[1]))
    for e, h in hs.items():
        a, b = int(offsets[e]), int(offsets[e + 1])
        out[a:b] = fp8_dequantize(h.astype(np.float32), sh) @ fp8_dequantize(w_down[e]).T
    return out


def moe_layer_fp8(x, w_router, bias, w_up, w_down, k: int) -> dict:
    """Routed MoE layer with FP8 experts: bf16 routing, FP8 expert FFNs, fp64 combine."""
    r = route(x, w_router, bias, k)
    E = np.asarray(w_router).shape[0]
    p = permute(r["idx"], E)
    y_perm = grouped_ffn_fp8(gather_rows(x, p["row_token"]), p["offsets"], w_up, w_down)
    T = np.asarray(x).shape[0]
    return {"y": combine(y_perm, p["slot_row"], r["gates"], T, k), **r, **p}


def fp8_hidden_amax(x, idx, w_up) -> float:
    """amax of h over every routed (token, expert) pair with FP8 tokens and weights."""
    xq = fp8_dequantize(_f64(x).astype(np.float32))
    idx = np.asarray(idx)
    amax = 0.0
    for e in np.unique(idx):
        toks = np.nonzero((idx == e).any(axis=1))[0]
        a = xq[toks] @ fp8_dequantize(w_up[int(e)]).T
        amax = max(amax, float(np.max(np.maximum(a, 0.0) ** 2)))
    return amax


def moe_tokens_fp8(x_all, x_rows, idx_rows, gates_rows, w_up, w_down, h_amax):
    """FP8 layer output for a subset of tokens, given the tensor-wide amax of h."""
    sx = fp8_scale(np.max(np.abs(_f64(x_all).astype(np.float32))))
    xr = fp8_dequantize(_f64(x_rows).astype(np.float32), sx)
    sh = fp8_scale(np.float32(h_amax))
    n, k = np.asarray(idx_rows).shape
    out = np.zeros((n, np.asarray(w_down).shape[1]))
    cache: dict[tuple[int, int], np.ndarray] = {}

    def wq(tag, e, w):
        if (tag, e) not in cache:
            cache[(tag, e)] = fp8_dequantize(w[e])
        return cache[(tag, e)]

    for i in range(n):
        for j in range(k):
            e = int(idx_rows[i][j])
            h = np.maximum(xr[i:i + 1] @ wq(0, e, w_up).T, 0.0) ** 2
            hq = fp8_dequantize(h.astype(np.float32), sh)
            out[i] += float(gates_rows[i][j]) * (hq @ wq(1, e, w_down).T)[0]
    return out
