"""Pins of the fp64 oracle against things other than itself (CPU only).

Each check takes the oracle module as an argument. The mutation tests at the bottom
plant plausible mistakes in a copy of the oracle and show that some pin then fails.
"""
import copy
import itertools
import json
import math
import os
import types

import numpy as np
import pytest

import moe_synth
from oracle import moe_oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


_LOGIT = {"ln3": math.log(3.0), "0": 0.0, "-ln3": -math.log(3.0), "ln9": math.log(9.0),
          "-ln9": -math.log(9.0)}


# ---------------------------------------------------------------------------- checks ----

def check_route_closed_form(o):
    g = _load("route_closed_form.json")
    bias = np.array(g["bias"])
    for c in g["cases"]:
        z = np.array([[_LOGIT[v] for v in c["logits"]]])
        r = o.route_from_logits(z, bias, c["k"])
        np.testing.assert_allclose(r["scores"][0], c["scores"], rtol=0, atol=1e-14)
        assert r["idx"][0].tolist() == c["idx"], (r["idx"][0], c)
        np.testing.assert_allclose(r["gates"][0], c["gates"], rtol=0, atol=1e-14)
        np.testing.assert_allclose(r["gap"][0], c["gap"], rtol=0, atol=1e-14)


def _brute_topk(u_row, k):
    """Best k-subset by sum of u; among equal sums the lexicographically smallest index
    set wins. Ordered by descending u, lower index first on equal u."""
    E = len(u_row)
    best, best_set = None, None
    for comb in itertools.combinations(range(E), k):
        s = math.fsum(u_row[list(comb)])
        if best is None or s > best + 0.0:
            best, best_set = s, comb
    return sorted(best_set, key=lambda e: (-u_row[e], e))


def check_topk_brute_force(o):
    rng = np.random.default_rng(11)
    for E, k in [(5, 1), (5, 2), (6, 3), (8, 4), (8, 8), (7, 6)]:
        s = rng.uniform(0.01, 0.99, size=(40, E))
        b = rng.uniform(-0.1, 0.1, size=E)
        idx, gap = o.select_topk(s, b, k)
        u = s + b
        for t in range(40):
            assert idx[t].tolist() == _brute_topk(u[t], k), (E, k, t)
            rest = sorted(set(range(E)) - set(idx[t].tolist()))
            if rest:
                assert gap[t] == pytest.approx(u[t, idx[t, -1]] - max(u[t, rest]), abs=1e-15)


def _brute_moe(x, wr, b, wu, wd, k):
    """Whole layer by scalar loops on tiny sizes (no matrix library calls)."""
    T, H = x.shape
    E, F = wu.shape[0], wu.shape[1]
    y = np.zeros((T, H))
    for t in range(T):
        s = []
        for e in range(E):
            z = math.fsum(x[t, i] * wr[e, i] for i in range(H))
            s.append(1.0 / (1.0 + math.exp(-z)))
        s = np.array(s)
        chosen = _brute_topk(s + b, k)
        tot = math.fsum(s[e] for e in chosen)
        for e in chosen:
            hid = []
            for f in range(F):
                a = math.fsum(x[t, i] * wu[e, f, i] for i in range(H))
                hid.append(max(a, 0.0) ** 2)
            for i in range(H):
                y[t, i] += (s[e] / tot) * math.fsum(wd[e, i, f] * hid[f] for f in range(F))
    return y


def _tiny_layer(seed, T=5, H=4, E=6, k=2, F=3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) / 2
    b = rng.uniform(-0.1, 0.1, E)
    wu = rng.standard_normal((E, F, H))
    wd = rng.standard_normal((E, H, F))
    return x, wr, b, wu, wd, k


def check_layer_brute_force(o):
    for seed in range(4):
        x, wr, b, wu, wd, k = _tiny_layer(seed)
        got = o.moe_layer(x, wr, b, wu, wd, k)["y"]
        np.testing.assert_allclose(got, _brute_moe(x, wr, b, wu, wd, k), rtol=1e-11, atol=1e-11)


def check_ffn_closed_form(o):
    g = _load("ffn_closed_form.json")
    out = o.expert_ffn(np.array([g["x"]]), np.array(g["w_up"]), np.array(g["w_down"]))
    np.testing.assert_array_equal(out[0], g["o"])


def check_single_expert_is_dense_ffn(o):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 5))
    wr = rng.standard_normal((1, 5))
    wu = rng.standard_normal((1, 4, 5))
    wd = rng.standard_normal((1, 5, 4))
    got = o.moe_layer(x, wr, np.zeros(1), wu, wd, 1)["y"]
    ref = np.zeros((7, 5))
    for t in range(7):
        hid = [max(math.fsum(x[t, i] * wu[0, f, i] for i in range(5)), 0.0) ** 2 for f in range(4)]
        ref[t] = [math.fsum(wd[0, i, f] * hid[f] for f in range(4)) for i in range(5)]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def check_identical_experts(o):
    """With every expert equal, any renormalised routing gives the dense FFN."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((9, 6))
    wr = rng.standard_normal((5, 6))
    wu1, wd1 = rng.standard_normal((4, 6)), rng.standard_normal((6, 4))
    wu = np.stack([wu1] * 5)
    wd = np.stack([wd1] * 5)
    got = o.moe_layer(x, wr, rng.uniform(-0.1, 0.1, 5), wu, wd, 3)["y"]
    np.testing.assert_allclose(got, o.expert_ffn(x, wu1, wd1), rtol=1e-12, atol=1e-12)
    # and that dense FFN is the closed-form one
    ref = np.maximum(x @ wu1.T, 0) ** 2 @ wd1.T
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def check_k_equals_E(o):
    rng = np.random.default_rng(6)
    x, wr, b, wu, wd, _ = _tiny_layer(6, T=4, H=3, E=4, F=2)
    r = o.moe_layer(x, wr, b, wu, wd, 4)
    assert all(sorted(row) == [0, 1, 2, 3] for row in r["idx"].tolist())
    np.testing.assert_allclose(r["y"], _brute_moe(x, wr, b, wu, wd, 4), rtol=1e-11, atol=1e-11)
    del rng


def check_forced_expert(o):
    rng = np.random.default_rng(8)
    s = rng.uniform(0, 1, (50, 10))
    b = np.zeros(10)
    b[7] = 10.0
    idx, _ = o.select_topk(s, b, 3)
    assert (idx[:, 0] == 7).all()


def check_gate_and_count_invariants(o):
    w = moe_synth.WORKLOADS["tiny"]
    inp = moe_synth.layer_inputs(w, with_experts=False)
    r = o.route(inp["x"], inp["w_router"], inp["bias"], w.k)
    np.testing.assert_allclose(r["gates"].sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert (r["gates"] > 0).all()
    p = o.permute(r["idx"], w.E)
    assert int(p["counts"].sum()) == w.T * w.k == int(p["offsets"][-1])
    assert p["offsets"][0] == 0 and (np.diff(p["offsets"]) == p["counts"]).all()
    # permute o unpermute is the identity
    xp = o.gather_rows(inp["x"], p["row_token"])
    for t in range(w.T):
        for j in range(w.k):
            assert (xp[p["slot_row"][t * w.k + j]] == inp["x"][t]).all()
    # each token at most once per segment, in ascending order
    for e in range(w.E):
        seg = p["row_token"][p["offsets"][e]:p["offsets"][e + 1]]
        assert (np.diff(seg) > 0).all()
        for t in seg:
            assert e in r["idx"][t]
    assert sorted(p["slot_row"].tolist()) == list(range(w.T * w.k))


def check_latent_identity(o):
    """l = H with W_in = W_out = I reduces LatentMoE to the standard layer."""
    x, wr, b, wu, wd, k = _tiny_layer(9, T=6, H=4, E=5, F=3)
    eye = np.eye(4)
    lat = o.latent_moe(x, eye, eye, wr, b, wu, wd, k, router_on_latent=True)
    std = o.moe_layer(x, wr, b, wu, wd, k)
    np.testing.assert_allclose(lat["y"], std["y"], rtol=1e-13, atol=1e-13)
    lat_h = o.latent_moe(x, eye, eye, wr, b, wu, wd, k, router_on_latent=False)
    np.testing.assert_allclose(lat_h["y"], std["y"], rtol=1e-13, atol=1e-13)


def check_latent_brute_force(o):
    """A non-trivial projection: brute-force layer on x W_in^T, then W_out."""
    rng = np.random.default_rng(12)
    T, H, L, E, k, F = 4, 6, 3, 5, 2, 2
    x = rng.standard_normal((T, H))
    w_in = rng.standard_normal((L, H))
    w_out = rng.standard_normal((H, L))
    wr = rng.standard_normal((E, L))
    b = rng.uniform(-0.1, 0.1, E)
    wu = rng.standard_normal((E, F, L))
    wd = rng.standard_normal((E, L, F))
    got = o.latent_moe(x, w_in, w_out, wr, b, wu, wd, k)["y"]
    xl = np.array([[math.fsum(x[t, i] * w_in[l, i] for i in range(H)) for l in range(L)]
                   for t in range(T)])
    yl = _brute_moe(xl, wr, b, wu, wd, k)
    ref = np.array([[math.fsum(yl[t, l] * w_out[h, l] for l in range(L)) for h in range(H)]
                    for t in range(T)])
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-10)


def check_combine_weights(o):
    yp = np.arange(12.0).reshape(6, 2)
    slot_row = np.array([5, 0, 2, 3, 1, 4])
    gates = np.array([0.25, 0.75, 0.5, 0.5, 1.0, 0.0])
    y = o.combine(yp, slot_row, gates, 3, 2)
    # token 0: 0.25*yp[5] + 0.75*yp[0]; token 1: 0.5*yp[2] + 0.5*yp[3]; token 2: yp[1]
    np.testing.assert_array_equal(y, [[2.5, 3.5], [5.0, 6.0], [2.0, 3.0]])


def check_e2m1_table(o):
    """Exhaustive E2M1: decode all 16 codes from the bit fields, then check nearest/even."""
    table = []
    for code in range(16):
        s, ex, m = code >> 3, (code >> 1) & 3, code & 1
        mag = (m * 0.5) if ex == 0 else (1 + m * 0.5) * 2.0 ** (ex - 1)
        table.append((-1.0 if s else 1.0) * mag)
    pos = sorted(set(abs(v) for v in table))
    assert pos == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    probes = np.concatenate([np.array(pos), (np.array(pos[1:]) + np.array(pos[:-1])) / 2,
                             np.random.default_rng(1).uniform(0, 8, 500)])
    for v in probes:
        got = float(o.e2m1_round(v))
        d = [abs(v - p) for p in pos]
        best = min(d)
        cands = [i for i, di in enumerate(d) if di == best]
        want = pos[cands[0]] if len(cands) == 1 else pos[[c for c in cands if c % 2 == 0][0]]
        if v > 6:
            want = 6.0
        assert got == want, (v, got, want)
        assert float(o.e2m1_round(-v)) == -want


def check_e4m3_table(o):
    """Exhaustive E4M3: decode the 254 finite codes from the bit fields (S.1111.111 is
    NaN), then check that rounding picks the nearest value, ties to the even code."""
    vals = {}
    for code in range(128):
        ex, m = (code >> 3) & 15, code & 7
        if ex == 15 and m == 7:
            continue
        v = m * 2.0 ** -9 if ex == 0 else (1 + m / 8) * 2.0 ** (ex - 7)
        vals[code] = v
    assert max(vals.values()) == 448.0 and min(v for v in vals.values() if v) == 2.0 ** -9
    codes = sorted(vals, key=lambda c: vals[c])
    mags = [vals[c] for c in codes]
    probes = list(mags) + [(a + b) / 2 for a, b in zip(mags, mags[1:])]
    probes += list(np.random.default_rng(2).uniform(0, 460, 400))
    probes += list(np.exp(np.random.default_rng(3).uniform(-8, 6, 400)))
    for v in probes:
        got = float(o.e4m3_round(v))
        if v >= 448:
            assert got == 448.0
            continue
        d = [abs(v - p) for p in mags]
        best = min(d)
        cands = [i for i, di in enumerate(d) if di == best]
        if len(cands) == 1:
            want = mags[cands[0]]
        else:
            want = [mags[i] for i in cands if codes[i] % 2 == 0][0]
        assert got == want, (v, got, want)


def check_nvfp4_block(o):
    g = _load("nvfp4_block.json")
    q = o.nvfp4_quantize(np.array([g["values"]], dtype=np.float32), np.float32(g["g"]))
    assert q["sb"].tolist() == [[g["block_scale"]]]
    np.testing.assert_array_equal(q["q"][0], g["codes_value"])
    np.testing.assert_array_equal(q["deq"][0], g["codes_value"])


def check_nvfp4_bounds(o):
    rng = np.random.default_rng(4)
    a = (rng.standard_normal((64, 128)) * np.exp(rng.uniform(-4, 4, (64, 1)))).astype(np.float32)
    a[3, 16:32] = 0.0                                     # an all-zero block
    q = o.nvfp4_quantize(a)
    g = float(q["g"])
    assert g == pytest.approx(float(np.abs(a).max()) / 2688.0, rel=1e-6)
    assert q["sb"].max() <= 448.0
    assert (q["q"][3, 16:32] == 0).all() and q["sb"][3, 1] == 0
    assert np.isin(np.abs(q["q"]), [0, 0.5, 1, 1.5, 2, 3, 4, 6]).all()
    blocks = a.reshape(64, 8, 16).astype(np.float64)
    deq = q["deq"].reshape(64, 8, 16)
    step = np.where(np.abs(blocks) < 2 * q["sb"][:, :, None] * g, 0.5, 2.0)   # coarsest spacing
    scale = (q["sb"] * g)[:, :, None]
    inside = np.abs(blocks) <= 6 * scale
    err = np.abs(deq - blocks)
    assert (err[inside] <= (0.5 * step * scale)[inside] * (1 + 1e-6) + 1e-30).all()
    # values on the scaled grid survive exactly
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -6, -4, -3, -2, -1.5, -1, -0.5, 0], np.float32)
    blk = (grid * np.float32(2.0 ** -3)).reshape(1, 16)
    q2 = o.nvfp4_quantize(blk, np.float32(2.0 ** -3))
    np.testing.assert_array_equal(q2["deq"], blk.astype(np.float64))


def _nearest_even(v, table_vals, table_codes):
    """Brute-force round-to-nearest over a decoded value table, ties to the even code."""
    d = np.abs(np.asarray(table_vals) - v)
    best = d.min()
    cands = [i for i in range(len(d)) if d[i] == best]
    if len(cands) > 1:
        cands = [i for i in cands if table_codes[i] % 2 == 0]
    return table_vals[cands[0]]


def _brute_nvfp4(mat, g):
    """NVFP4 quantise-dequantise by table search (no rint-based rounding)."""
    e2 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    e4_vals, e4_codes = [], []
    for code in range(127):            # non-negative finite E4M3 values (0x7F is NaN)
        ex, m = code >> 3, code & 7
        e4_vals.append(m * 2.0 ** -9 if ex == 0 else (1 + m / 8) * 2.0 ** (ex - 7))
        e4_codes.append(code)
    a = np.asarray(mat, np.float32)
    out = np.zeros(a.shape)
    g = np.float32(g)
    for r in range(a.shape[0]):
        for b in range(a.shape[1] // 16):
            blk = a[r, 16 * b:16 * b + 16]
            ratio = np.float32(np.max(np.abs(blk)) / np.float32(np.float32(6) * g))
            sb = min(_nearest_even(float(ratio), e4_vals, e4_codes), 448.0) if g > 0 else 0.0
            den = np.float32(np.float32(sb) * g)
            for i in range(16):
                if den > 0:
                    s = float(np.float32(blk[i] / den))
                    q = 6.0 if abs(s) > 6 else _nearest_even(abs(s), e2, list(range(8)))
                    out[r, 16 * b + i] = np.copysign(q, s) * float(den)
    return out


def check_nvfp4_brute_force(o):
    rng = np.random.default_rng(21)
    a = (rng.standard_normal((5, 64)) * np.exp(rng.uniform(-6, 3, (5, 1)))).astype(np.float32)
    g = o.nvfp4_global_scale(np.max(np.abs(a)))
    np.testing.assert_array_equal(o.nvfp4_quantize(a)["deq"], _brute_nvfp4(a, g))


def check_grouped_ffn_nvfp4(o):
    """NVFP4 expert FFNs by brute force: table-search quantiser, scalar-loop products."""
    rng = np.random.default_rng(22)
    E, D, F = 2, 32, 16
    x = rng.standard_normal((5, D)).astype(np.float32)
    offsets = np.array([0, 2, 5])
    wu = rng.standard_normal((E, F, D)).astype(np.float32)
    wd = rng.standard_normal((E, D, F)).astype(np.float32)
    got = o.grouped_ffn_nvfp4(x, offsets, wu, wd)
    xq = _brute_nvfp4(x, o.nvfp4_global_scale(np.max(np.abs(x))))
    hs = []
    for e in range(E):
        wq = _brute_nvfp4(wu[e], o.nvfp4_global_scale(np.max(np.abs(wu[e]))))
        for r in range(offsets[e], offsets[e + 1]):
            hs.append([max(math.fsum(xq[r, i] * wq[f, i] for i in range(D)), 0.0) ** 2
                       for f in range(F)])
    hs = np.array(hs)
    hq = _brute_nvfp4(hs, o.nvfp4_global_scale(np.float32(np.max(np.abs(hs)))))
    ref = np.zeros((5, D))
    for e in range(E):
        wq = _brute_nvfp4(wd[e], o.nvfp4_global_scale(np.max(np.abs(wd[e]))))
        for r in range(offsets[e], offsets[e + 1]):
            ref[r] = [math.fsum(hq[r, f] * wq[i, f] for f in range(F)) for i in range(D)]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def check_nvfp4_layer_paths(o):
    """The NVFP4 layer, the tensor-wide hidden amax and the sampled per-token evaluation
    against brute force: table-search quantiser, scalar-loop products, explicit combine."""
    rng = np.random.default_rng(23)
    T, D, F, E, k = 6, 32, 16, 3, 2
    x = moe_synth.bf16_bits(rng.standard_normal((T, D)).astype(np.float32))
    wr = moe_synth.bf16_bits(rng.standard_normal((E, D)).astype(np.float32))
    bias = np.zeros(E, np.float32)
    wu = moe_synth.bf16_bits(rng.standard_normal((E, F, D)).astype(np.float32))
    wd = moe_synth.bf16_bits(rng.standard_normal((E, D, F)).astype(np.float32))
    r = o.route(x, wr, bias, k)
    xf = o.widen_bf16(x).astype(np.float32)
    xq = _brute_nvfp4(xf, o.nvfp4_global_scale(np.max(np.abs(xf))))
    wuq = [_brute_nvfp4(o.widen_bf16(wu[e]), o.nvfp4_global_scale(np.max(np.abs(
        o.widen_bf16(wu[e]).astype(np.float32))))) for e in range(E)]
    wdq = [_brute_nvfp4(o.widen_bf16(wd[e]), o.nvfp4_global_scale(np.max(np.abs(
        o.widen_bf16(wd[e]).astype(np.float32))))) for e in range(E)]
    pairs = [(t, j, int(r["idx"][t, j])) for t in range(T) for j in range(k)]
    hs = np.array([[max(math.fsum(xq[t, i] * wuq[e][f, i] for i in range(D)), 0.0) ** 2
                    for f in range(F)] for t, j, e in pairs])
    h_amax = float(np.max(hs))
    assert o.nvfp4_hidden_amax(x, r["idx"], wu) == pytest.approx(h_amax, rel=1e-12)
    hq = _brute_nvfp4(hs.astype(np.float32), o.nvfp4_global_scale(np.float32(h_amax)))
    ref = np.zeros((T, D))
    for n, (t, j, e) in enumerate(pairs):
        ref[t] += r["gates"][t, j] * np.array(
            [math.fsum(hq[n, f] * wdq[e][i, f] for f in range(F)) for i in range(D)])
    got = o.moe_layer_nvfp4(x, wr, bias, wu, wd, k)["y"]
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-10)
    toks = np.array([1, 4])
    sampled = o.moe_tokens_nvfp4(x, x[toks], r["idx"][toks], r["gates"][toks], wu, wd,
                                 h_amax=h_amax)
    np.testing.assert_allclose(sampled, ref[toks], rtol=1e-10, atol=1e-10)


def _brute_fp8(mat, s):
    """Per-tensor E4M3 quantise-dequantise by table search."""
    e4_vals = [(m * 2.0 ** -9 if ex == 0 else (1 + m / 8) * 2.0 ** (ex - 7))
               for code in range(127) for ex, m in [(code >> 3, code & 7)]]
    a = np.asarray(mat, np.float32)
    out = np.zeros(a.shape)
    s = np.float32(s)
    for idx in np.ndindex(a.shape):
        if s > 0:
            v = float(np.float32(a[idx] / s))
            q = 448.0 if abs(v) > 448 else _nearest_even(abs(v), e4_vals, list(range(127)))
            out[idx] = np.copysign(q, v) * float(s)
    return out


def check_fp8_quantize(o):
    rng = np.random.default_rng(24)
    a = (rng.standard_normal((6, 48)) * np.exp(rng.uniform(-9, 4, (6, 1)))).astype(np.float32)
    s = o.fp8_scale(np.max(np.abs(a)))
    assert float(s) == pytest.approx(float(np.abs(a).max()) / 448.0, rel=1e-6)
    q = o.fp8_quantize(a)
    np.testing.assert_array_equal(q["deq"], _brute_fp8(a, s))
    assert np.max(np.abs(q["q"])) == 448.0                # the amax maps to E4M3's maximum
    # error bound: half an E4M3 step (2^(e-3) in binade e, 2^-9 subnormal spacing) times s
    v = np.abs(a.astype(np.float64) / float(s))
    step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(v, 2.0 ** -9))), -6) - 3)
    assert (np.abs(q["deq"] - a) <= 0.5 * step * float(s) * (1 + 1e-6) + 1e-30).all()
    assert (o.fp8_quantize(np.zeros((2, 16), np.float32))["deq"] == 0).all()


def check_fp8_layer_paths(o):
    """FP8 grouped FFN, layer, hidden amax and sampled tokens against brute force."""
    rng = np.random.default_rng(25)
    T, D, F, E, k = 6, 32, 16, 3, 2
    x = moe_synth.bf16_bits(rng.standard_normal((T, D)).astype(np.float32))
    wr = moe_synth.bf16_bits(rng.standard_normal((E, D)).astype(np.float32))
    bias = np.zeros(E, np.float32)
    wu = moe_synth.bf16_bits(rng.standard_normal((E, F, D)).astype(np.float32))
    wd = moe_synth.bf16_bits(rng.standard_normal((E, D, F)).astype(np.float32))
    r = o.route(x, wr, bias, k)
    xf = o.widen_bf16(x).astype(np.float32)
    xq = _brute_fp8(xf, o.fp8_scale(np.max(np.abs(xf))))
    def wq(w):
        wf = o.widen_bf16(w).astype(np.float32)
        return _brute_fp8(wf, o.fp8_scale(np.max(np.abs(wf))))
    wuq = [wq(wu[e]) for e in range(E)]
    wdq = [wq(wd[e]) for e in range(E)]
    pairs = [(t, j, int(r["idx"][t, j])) for t in range(T) for j in range(k)]
    hs = np.array([[max(math.fsum(xq[t, i] * wuq[e][f, i] for i in range(D)), 0.0) ** 2
                    for f in range(F)] for t, j, e in pairs])
    h_amax = float(np.max(hs))
    assert o.fp8_hidden_amax(x, r["idx"], wu) == pytest.approx(h_amax, rel=1e-12)
    hq = _brute_fp8(hs.astype(np.float32), o.fp8_scale(np.float32(h_amax)))
    ref = np.zeros((T, D))
    for n, (t, j, e) in enumerate(pairs):
        ref[t] += r["gates"][t, j] * np.array(
            [math.fsum(hq[n, f] * wdq[e][i, f] for f in range(F)) for i in range(D)])
    np.testing.assert_allclose(o.moe_layer_fp8(x, wr, bias, wu, wd, k)["y"], ref,
                               rtol=1e-10, atol=1e-10)
    toks = np.array([0, 5])
    got = o.moe_tokens_fp8(x, x[toks], r["idx"][toks], r["gates"][toks], wu, wd, h_amax)
    np.testing.assert_allclose(got, ref[toks], rtol=1e-10, atol=1e-10)


def check_shared_expert(o):
    """Shared expert: brute force, a zero shared expert changes nothing, and with one routed
    expert (k = 1) equal to the shared one the layer is twice the dense FFN."""
    rng = np.random.default_rng(26)
    T, H, E, k, F, Fs = 5, 16, 3, 2, 8, 12
    x = moe_synth.bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = moe_synth.bf16_bits(rng.standard_normal((E, H)).astype(np.float32))
    bias = np.zeros(E, np.float32)
    wu = moe_synth.bf16_bits(rng.standard_normal((E, F, H)).astype(np.float32) * 0.3)
    wd = moe_synth.bf16_bits(rng.standard_normal((E, H, F)).astype(np.float32) * 0.3)
    wus = moe_synth.bf16_bits(rng.standard_normal((Fs, H)).astype(np.float32) * 0.3)
    wds = moe_synth.bf16_bits(rng.standard_normal((H, Fs)).astype(np.float32) * 0.3)
    xf, wusf, wdsf = o.widen_bf16(x), o.widen_bf16(wus), o.widen_bf16(wds)
    sh = np.array([[math.fsum(max(math.fsum(xf[t, i] * wusf[f, i] for i in range(H)), 0.0) ** 2
                              * wdsf[j, f] for f in range(Fs)) for j in range(H)]
                   for t in range(T)])
    np.testing.assert_allclose(o.shared_ffn(x, wus, wds), sh, rtol=1e-12, atol=1e-12)
    base = o.moe_layer(x, wr, bias, wu, wd, k)["y"]
    got = o.moe_layer_shared(x, wr, bias, wu, wd, wus, wds, k)["y"]
    np.testing.assert_allclose(got, base + sh, rtol=1e-12, atol=1e-12)
    z = np.zeros_like(wus)
    np.testing.assert_array_equal(o.moe_layer_shared(x, wr, bias, wu, wd, z, z.T.copy(), k)["y"],
                                  base)
    one = o.moe_layer_shared(x, wr[:1], bias[:1], wus[None], wds[None], wus, wds, 1)["y"]
    np.testing.assert_allclose(one, 2 * sh, rtol=1e-12, atol=1e-12)
    # LatentMoE: the shared expert is added in H, after the projection back
    L = 8
    w_in = moe_synth.bf16_bits(rng.standard_normal((L, H)).astype(np.float32) * 0.3)
    w_out = moe_synth.bf16_bits(rng.standard_normal((H, L)).astype(np.float32) * 0.3)
    wrl = moe_synth.bf16_bits(rng.standard_normal((E, L)).astype(np.float32))
    wul = moe_synth.bf16_bits(rng.standard_normal((E, F, L)).astype(np.float32) * 0.3)
    wdl = moe_synth.bf16_bits(rng.standard_normal((E, L, F)).astype(np.float32) * 0.3)
    lat = o.latent_moe(x, w_in, w_out, wrl, bias, wul, wdl, k)["y"]
    np.testing.assert_allclose(
        o.latent_moe_shared(x, w_in, w_out, wrl, bias, wul, wdl, wus, wds, k)["y"], lat + sh,
        rtol=1e-12, atol=1e-12)


def _brute_nvfp4_2d(mat, g):
    """2-D NVFP4 by table search: one scale per 16x16 block, then every element as in 1-D."""
    e2 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    e4_vals = [(m * 2.0 ** -9 if ex == 0 else (1 + m / 8) * 2.0 ** (ex - 7))
               for code in range(127) for ex, m in [(code >> 3, code & 7)]]
    a = np.asarray(mat, np.float32)
    out = np.zeros(a.shape)
    g = np.float32(g)
    for r0 in range(0, a.shape[0], 16):
        for b in range(a.shape[1] // 16):
            blk = a[r0:r0 + 16, 16 * b:16 * b + 16]
            ratio = np.float32(np.max(np.abs(blk)) / np.float32(np.float32(6) * g))
            sb = min(_nearest_even(float(ratio), e4_vals, list(range(127))), 448.0) if g > 0 else 0.0
            den = np.float32(np.float32(sb) * g)
            for r in range(blk.shape[0]):
                for i in range(16):
                    if den > 0:
                        s = float(np.float32(blk[r, i] / den))
                        q = 6.0 if abs(s) > 6 else _nearest_even(abs(s), e2, list(range(8)))
                        out[r0 + r, 16 * b + i] = np.copysign(q, s) * float(den)
    return out


def check_nvfp4_2d(o):
    """2-D weight blocks: brute force on a matrix with a ragged last row block; a matrix whose
    16-row groups repeat one row equals the 1-D quantisation; the 2-D grouped FFN matches a
    brute-force evaluation."""
    rng = np.random.default_rng(27)
    a = (rng.standard_normal((37, 48)) * np.exp(rng.uniform(-5, 3, (37, 1)))).astype(np.float32)
    g = o.nvfp4_global_scale(np.max(np.abs(a)))
    np.testing.assert_array_equal(o.nvfp4_quantize_2d(a)["deq"], _brute_nvfp4_2d(a, g))
    rep = np.repeat(a[:3], 16, axis=0)
    np.testing.assert_array_equal(o.nvfp4_quantize_2d(rep)["deq"], o.nvfp4_quantize(rep)["deq"])
    E, D, F = 2, 32, 16
    x = rng.standard_normal((5, D)).astype(np.float32)
    offsets = np.array([0, 2, 5])
    wu = rng.standard_normal((E, F, D)).astype(np.float32)
    wd = rng.standard_normal((E, D, F)).astype(np.float32)
    got = o.grouped_ffn_nvfp4(x, offsets, wu, wd, weight_blocks="2d")
    xq = _brute_nvfp4(x, o.nvfp4_global_scale(np.max(np.abs(x))))
    hs = []
    for e in range(E):
        wq = _brute_nvfp4_2d(wu[e], o.nvfp4_global_scale(np.max(np.abs(wu[e]))))
        for r in range(offsets[e], offsets[e + 1]):
            hs.append([max(math.fsum(xq[r, i] * wq[f, i] for i in range(D)), 0.0) ** 2
                       for f in range(F)])
    hs = np.array(hs)
    hq = _brute_nvfp4(hs, o.nvfp4_global_scale(np.float32(np.max(hs))))
    ref = np.zeros((5, D))
    for e in range(E):
        wq = _brute_nvfp4_2d(wd[e], o.nvfp4_global_scale(np.max(np.abs(wd[e]))))
        for r in range(offsets[e], offsets[e + 1]):
            ref[r] = [math.fsum(hq[r, f] * wq[i, f] for f in range(F)) for i in range(D)]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def _brute_tokens(x, idx, gates, wu, wd):
    """y[t] = sum_j gates[t, j] * FFN_{idx[t, j]}(x[t]) by scalar loops (given routing)."""
    n, H = x.shape
    F = wu.shape[1]
    y = np.zeros((n, wd.shape[1]))
    for t in range(n):
        for j in range(idx.shape[1]):
            e = int(idx[t, j])
            hid = [max(math.fsum(x[t, i] * wu[e, f, i] for i in range(H)), 0.0) ** 2
                   for f in range(F)]
            for i in range(wd.shape[1]):
                y[t, i] += gates[t, j] * math.fsum(wd[e, i, f] * hid[f] for f in range(F))
    return y


def _brute_route(x, wr, b, k):
    """Routing by scalar loops: sigmoid scores, brute-force top-k, renormalised gates."""
    T, H = x.shape
    E = wr.shape[0]
    idx = np.zeros((T, k), dtype=np.int64)
    gates = np.zeros((T, k))
    for t in range(T):
        s = np.array([1.0 / (1.0 + math.exp(-math.fsum(x[t, i] * wr[e, i] for i in range(H))))
                      for e in range(E)])
        chosen = _brute_topk(s + b, k)
        tot = math.fsum(s[e] for e in chosen)
        idx[t] = chosen
        gates[t] = [s[e] / tot for e in chosen]
    return idx, gates


def check_moe_tokens(o):
    """The per-token evaluator used for sampled parity at full size equals the scalar-loop
    layer on every token (k = 1, 1 < k < E and k = E), and weights each (token, slot)
    by that slot's own gate when the gates are arbitrary and a sample is out of order."""
    for seed, (T, H, E, k, F) in enumerate([(6, 4, 5, 1, 3), (7, 5, 6, 3, 2), (5, 3, 4, 4, 2)]):
        x, wr, b, wu, wd, _ = _tiny_layer(20 + seed, T=T, H=H, E=E, k=k, F=F)
        idx, gates = _brute_route(x, wr, b, k)
        got = o.moe_tokens(x, idx, gates, wu, wd)
        np.testing.assert_allclose(got, _brute_moe(x, wr, b, wu, wd, k), rtol=1e-11,
                                   atol=1e-11)
        # the full layer's output on every token is the per-token evaluation
        np.testing.assert_allclose(got, o.moe_layer(x, wr, b, wu, wd, k)["y"], rtol=1e-11,
                                   atol=1e-11)
    rng = np.random.default_rng(31)
    x, _, _, wu, wd, _ = _tiny_layer(31, T=6, H=4, E=5, F=3)
    # a sample in no particular order; slot order not sorted by expert; distinct gates that
    # do not sum to one, so a gate taken from the wrong slot or token changes the result
    sample = np.array([4, 0, 5, 2])
    idx = np.array([[3, 0, 4], [1, 4, 2], [0, 2, 1], [4, 3, 0]])
    gates = rng.uniform(0.1, 2.0, size=idx.shape)
    got = o.moe_tokens(x[sample], idx, gates, wu, wd)
    np.testing.assert_allclose(got, _brute_tokens(x[sample], idx, gates, wu, wd), rtol=1e-11,
                               atol=1e-11)


def check_widen_bf16(o):
    """bfloat16 is the upper half of an IEEE binary32 word: decode hand-picked patterns from
    the bit fields, then every one of the 65536 patterns through struct's binary32 reader."""
    import struct
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x0001: 2.0 ** -133, 0x0080: 2.0 ** -126,
             0x7F7F: (2.0 - 2.0 ** -7) * 2.0 ** 127, 0x3EAB: 0.333984375, 0x4049: 3.140625,
             0x7F80: math.inf, 0xFF80: -math.inf}
    got = o.widen_bf16(np.array(list(cases), dtype=np.uint16))
    assert got.dtype == np.float64
    assert got.tolist() == list(cases.values())
    z = o.widen_bf16(np.array([0x0000, 0x8000], dtype=np.uint16))
    assert z.tolist() == [0.0, 0.0] and not math.copysign(1, z[0]) < 0 \
        and math.copysign(1, z[1]) < 0
    assert math.isnan(o.widen_bf16(np.array([0x7FC0], dtype=np.uint16))[0])
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):          # signalling NaN patterns widen to NaN
        w = o.widen_bf16(allbits)
    ref = np.array([struct.unpack(">f", int(b).to_bytes(2, "big") + b"\0\0")[0]
                    for b in range(1 << 16)])
    nan = np.isnan(ref)
    assert (np.isnan(w) == nan).all()
    assert (w[~nan] == ref[~nan]).all()
    assert (np.signbit(w[~nan]) == np.signbit(ref[~nan])).all()
    # shape is kept
    assert o.widen_bf16(allbits[:12].reshape(3, 4)).shape == (3, 4)


ALL_CHECKS = [check_route_closed_form, check_topk_brute_force, check_layer_brute_force,
              check_ffn_closed_form, check_single_expert_is_dense_ffn, check_identical_experts,
              check_k_equals_E, check_forced_expert, check_gate_and_count_invariants,
              check_latent_identity, check_latent_brute_force, check_combine_weights,
              check_e2m1_table, check_e4m3_table, check_nvfp4_block, check_nvfp4_bounds,
              check_nvfp4_brute_force, check_grouped_ffn_nvfp4, check_nvfp4_layer_paths,
              check_fp8_quantize, check_fp8_layer_paths, check_shared_expert, check_nvfp4_2d,
              check_moe_tokens, check_widen_bf16]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(moe_oracle)


def test_latent_expert_scaling_formula():
    # E' = E*H/l and k' = k*H/l (Nemotron 3 notes §2.2): 128 experts, top-6, H/l = 4
    assert moe_synth.latent_scaled(128, 6, 4096, 1024) == (512, 24)
    w = moe_synth.WORKLOADS["latent"]
    assert (w.E, w.k, w.latent, w.H) == (512, 24, 1024, 4096)


# ------------------------------------------------------------------ planted mistakes ----

def _mutant(**overrides):
    m = types.ModuleType("mutant")
    m.__dict__.update({k: v for k, v in vars(moe_oracle).items() if not k.startswith("__")})
    for name, fn in overrides.items():
        m.__dict__[name] = fn
    # re-bind functions so internal calls see the mutated globals
    for k, v in list(m.__dict__.items()):
        if isinstance(v, types.FunctionType):
            m.__dict__[k] = types.FunctionType(v.__code__, m.__dict__, v.__name__,
                                               v.__defaults__, v.__closure__)
    for name, fn in overrides.items():
        m.__dict__[name] = types.FunctionType(fn.__code__, m.__dict__, fn.__name__,
                                              fn.__defaults__, fn.__closure__)
    return m


def _gates_biased(scores, idx):          # mistake: bias leaks into the gates
    sel = np.take_along_axis(np.asarray(scores) + 0.1, idx.astype(np.int64), axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def _ffn_plain_relu(rows, w_up_e, w_down_e):  # mistake: ReLU instead of squared ReLU
    return np.maximum(_f64(rows) @ _f64(w_up_e).T, 0.0) @ _f64(w_down_e).T


def _grouped_wrong_expert(x_perm, offsets, w_up, w_down):  # mistake: off-by-one expert
    xp = _f64(x_perm)
    E = len(offsets) - 1
    out = np.zeros((xp.shape[0], np.asarray(w_down).shape[1]))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            out[a:b] = expert_ffn(xp[a:b], w_up[e], w_down[(e + 1) % E])
    return out


def _select_high_index_wins(scores, bias, k):  # mistake: higher index wins exact ties
    s = np.asarray(scores, dtype=np.float64)
    u = s + np.asarray(bias)[None, :]
    T, E = s.shape
    idx = np.empty((T, k), dtype=np.int32)
    gap = np.full(T, np.inf)
    for t in range(T):
        order = np.lexsort((-np.arange(E), -u[t]))
        idx[t] = order[:k]
        if k < E:
            gap[t] = u[t, order[k - 1]] - u[t, order[k]]
    return idx, gap


def _combine_no_gates(y_perm, slot_row, gates, T, k):   # mistake: unweighted mean
    yp = _f64(y_perm)
    sr = np.asarray(slot_row, dtype=np.int64).reshape(T, k)
    return sum(yp[sr[:, j]] for j in range(k)) / k


def _sigmoid_sign(z):                     # mistake: sign error in the sigmoid
    return 1.0 / (1.0 + np.exp(np.asarray(z, dtype=np.float64)))


def _e2m1_ties_away(v):                   # mistake: ties rounded away from zero
    v = np.asarray(v, dtype=np.float64)
    m = np.abs(v)
    q = np.where(m < 2.0, 0.5, np.where(m < 4.0, 1.0, 2.0))
    return np.copysign(np.minimum(np.floor(m / q + 0.5) * q, 6.0), v)


def _fp8_scale_e2m1_max(amax):            # mistake: NVFP4's element maximum in the FP8 scale
    return np.float32(np.float32(amax) / np.float32(6.0))


def _tokens_first_slot_gate(x_rows, idx_rows, gates_rows, w_up, w_down):
    # mistake: every (token, slot) takes the token's first gate
    xr = _f64(x_rows)
    n, k = np.asarray(idx_rows).shape
    out = np.zeros((n, np.asarray(w_down).shape[1]))
    g = np.asarray(gates_rows, dtype=np.float64)
    for i in range(n):
        for j in range(k):
            e = int(idx_rows[i][j])
            out[i] += g[i, 0] * expert_ffn(xr[i:i + 1], w_up[e], w_down[e])[0]
    return out


def _tokens_overwrite(x_rows, idx_rows, gates_rows, w_up, w_down):
    # mistake: a later expert's output replaces the earlier ones instead of adding to them
    xr = _f64(x_rows)
    n, k = np.asarray(idx_rows).shape
    out = np.zeros((n, np.asarray(w_down).shape[1]))
    g = np.asarray(gates_rows, dtype=np.float64)
    for e in sorted({int(v) for v in np.asarray(idx_rows).reshape(-1)}):
        ii, jj = np.nonzero(np.asarray(idx_rows) == e)
        out[ii] = g[ii, jj][:, None] * expert_ffn(xr[ii], w_up[e], w_down[e])
    return out


def _tokens_gate_by_position(x_rows, idx_rows, gates_rows, w_up, w_down):
    # mistake: gates read by the row's position inside its expert group, not by (token, slot)
    xr = _f64(x_rows)
    n, k = np.asarray(idx_rows).shape
    out = np.zeros((n, np.asarray(w_down).shape[1]))
    g = np.asarray(gates_rows, dtype=np.float64)
    for e in sorted({int(v) for v in np.asarray(idx_rows).reshape(-1)}):
        ii, jj = np.nonzero(np.asarray(idx_rows) == e)
        o_e = expert_ffn(xr[ii], w_up[e], w_down[e])
        np.add.at(out, ii, g.reshape(-1)[np.arange(len(ii))][:, None] * o_e)
    return out


def _widen_as_fp16(bits):                 # mistake: the 16 bits read as IEEE half precision
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _widen_shift_15(bits):                # mistake: off-by-one shift into the binary32 word
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(15)
    return u.view(np.float32).astype(np.float64)


_f64 = moe_oracle._f64

MUTANTS = {
    "gates_use_bias": ({"gates_from_scores": _gates_biased}, check_route_closed_form),
    "plain_relu": ({"expert_ffn": _ffn_plain_relu}, check_ffn_closed_form),
    "plain_relu_layer": ({"expert_ffn": _ffn_plain_relu}, check_layer_brute_force),
    "wrong_expert_index": ({"grouped_ffn": _grouped_wrong_expert}, check_layer_brute_force),
    "tie_high_index": ({"select_topk": _select_high_index_wins}, check_route_closed_form),
    "combine_unweighted": ({"combine": _combine_no_gates}, check_combine_weights),
    "combine_unweighted_layer": ({"combine": _combine_no_gates}, check_layer_brute_force),
    "sigmoid_sign": ({"sigmoid": _sigmoid_sign}, check_route_closed_form),
    "e2m1_ties_away": ({"e2m1_round": _e2m1_ties_away}, check_e2m1_table),
    "fp8_scale_wrong_max": ({"fp8_scale": _fp8_scale_e2m1_max}, check_fp8_quantize),
    "tokens_first_slot_gate": ({"moe_tokens": _tokens_first_slot_gate}, check_moe_tokens),
    "tokens_overwrite": ({"moe_tokens": _tokens_overwrite}, check_moe_tokens),
    "tokens_gate_by_position": ({"moe_tokens": _tokens_gate_by_position}, check_moe_tokens),
    "widen_as_fp16": ({"widen_bf16": _widen_as_fp16}, check_widen_bf16),
    "widen_shift_15": ({"widen_bf16": _widen_shift_15}, check_widen_bf16),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    overrides, check = MUTANTS[name]
    m = _mutant(**copy.copy(overrides))
    with pytest.raises(AssertionError):
        check(m)
