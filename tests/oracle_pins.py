"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` function takes a loaded oracle library (the real one, or a
mutant built by ``test_oracle_mutants.py``) and raises AssertionError when the
oracle disagrees with:

* exact rational arithmetic on tiny inputs (``fractions.Fraction``),
* a numpy dense matmul over a matrix decoded here with numpy bit operations,
* closed forms (all-equal nibbles, hand-derived fixtures in ``tests/golden``),
* invariants (linearity in scales and in x, additivity over groups, a
  stable full sort for top-k, the sum of routing weights),
* special cases that reduce to textbook routines (gs = K is a per-row scale,
  k = 1 with weight 1 is one SwiGLU feed-forward block).
"""
from __future__ import annotations

import itertools
import json
import os
from fractions import Fraction

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
RNG_SEED = 1234


def _rng(offset=0):
    return np.random.default_rng(RNG_SEED + offset)


def np_unpack(wq: np.ndarray) -> np.ndarray:
    """Independent numpy decode: low nibble first, value = nibble - 8."""
    lo = (wq & 0x0F).astype(np.int64) - 8
    hi = (wq >> 4).astype(np.int64) - 8
    return np.stack([lo, hi], axis=-1).reshape(wq.shape[:-1] + (wq.shape[-1] * 2,))


def np_dequant(wq, s, gs=64):
    vals = np_unpack(wq).astype(np.float64)
    return vals * np.repeat(s.astype(np.float64), gs, axis=-1)


def rand_int4(rng, N, K, gs=64):
    wq = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = (np.abs(rng.normal(0, 0.02, size=(N, K // gs))) + 1e-4).astype(np.float32)
    return wq, s


# ----------------------------------------------------------------- a1 decode

def pin_pack_roundtrip(lib):
    b = np.arange(256, dtype=np.uint8)
    v = oracle.unpack_int4(b, lib=lib)
    assert v.min() >= -8 and v.max() <= 7
    assert np.array_equal(v, np_unpack(b)), "decode disagrees with numpy bit decode"
    assert np.array_equal(oracle.pack_int4(v, lib=lib), b), "pack(unpack(b)) != b"
    assert np.array_equal(oracle.unpack_int4(np.array([0x88], np.uint8), lib=lib), [0, 0])
    vals = _rng(1).integers(-8, 8, size=1000).astype(np.int8)
    assert np.array_equal(oracle.unpack_int4(oracle.pack_int4(vals, lib=lib), lib=lib), vals)


def pin_golden_nibble_order(lib):
    d = json.load(open(os.path.join(GOLDEN, "int4_gs64_nibble_order.json")))
    N, K, gs = d["N"], d["K"], d["gs"]
    wq = np.repeat(np.array(d["row_byte"], np.uint8)[:, None], K // 2, axis=1)
    s = np.array(d["scales"], np.float32)
    x = np.where(np.arange(K) % 2 == 0, d["x_even"], d["x_odd"]).astype(np.float32)[None]
    y = oracle.qmv_int4_gs(wq, s, x, gs, lib=lib)[0]
    assert np.array_equal(y, np.array(d["expected_y"])), (y, d["expected_y"])


# ----------------------------------------------------------------- a2 GEMV

def pin_int4_exact_bruteforce(lib):
    """Exact rational y on tiny shapes; the oracle must be within double rounding."""
    rng = _rng(2)
    for (N, K, S) in [(1, 64, 1), (3, 64, 2), (8, 128, 3), (5, 192, 1)]:
        wq, s = rand_int4(rng, N, K)
        x = rng.normal(size=(S, K)).astype(np.float32)
        y = oracle.qmv_int4_gs(wq, s, x, 64, lib=lib)
        vals = np_unpack(wq)
        for t in range(S):
            for i in range(N):
                exact = Fraction(0)
                mag = Fraction(0)
                for k in range(K):
                    term = int(vals[i, k]) * Fraction(float(s[i, k // 64])) * Fraction(float(x[t, k]))
                    exact += term
                    mag += abs(term)
                err = abs(Fraction(float(y[t, i])) - exact)
                assert err <= mag * Fraction(1, 2 ** 45), (N, K, t, i, float(err), float(mag))


def pin_int4_library_identity(lib):
    """Form (i) == numpy W @ x over a numpy-decoded W; oracle form (ii) agrees too."""
    rng = _rng(3)
    for (N, K, S) in [(16, 256, 2), (33, 1024, 3)]:
        wq, s = rand_int4(rng, N, K)
        x = rng.normal(size=(S, K)).astype(np.float32)
        W = np_dequant(wq, s)
        ref = x.astype(np.float64) @ W.T
        den = np.abs(x.astype(np.float64)) @ np.abs(W).T
        y1 = oracle.qmv_int4_gs(wq, s, x, 64, lib=lib)
        assert np.all(np.abs(y1 - ref) <= 1e-13 * den), np.max(np.abs(y1 - ref) / den)
        Wo = oracle.dequant_int4(wq, s, 64, lib=lib)
        assert np.array_equal(Wo, W), "explicit dequantization differs from numpy decode"
        y2 = oracle.matvec_f64(Wo, x, lib=lib)
        assert np.all(np.abs(y2 - ref) <= 1e-13 * den)
        _, d = oracle.qmv_int4_gs(wq, s, x, 64, with_den=True, lib=lib)
        assert np.allclose(d, den, rtol=1e-13, atol=0)


def pin_int4_linearity(lib):
    rng = _rng(4)
    N, K, S = 12, 512, 2
    wq, s = rand_int4(rng, N, K)
    x = rng.normal(size=(S, K)).astype(np.float32)
    y = oracle.qmv_int4_gs(wq, s, x, 64, lib=lib)
    # power-of-two scaling of the scales is exact
    for a in (0.25, 2.0, 1024.0):
        ya = oracle.qmv_int4_gs(wq, (s * np.float32(a)).astype(np.float32), x, 64, lib=lib)
        assert np.array_equal(ya, a * y)
    # additivity across groups
    G = K // 64
    acc = np.zeros_like(y)
    for g in range(G):
        sg = np.zeros_like(s)
        sg[:, g] = s[:, g]
        acc += oracle.qmv_int4_gs(wq, sg, x, 64, lib=lib)
    _, den = oracle.qmv_int4_gs(wq, s, x, 64, with_den=True, lib=lib)
    assert np.all(np.abs(acc - y) <= 1e-13 * den)
    # linearity in x (small integer x: every sum is exact in fp32)
    x1 = rng.integers(-50, 50, size=(S, K)).astype(np.float32)
    x2 = rng.integers(-50, 50, size=(S, K)).astype(np.float32)
    y12 = oracle.qmv_int4_gs(wq, s, x1 + x2, 64, lib=lib)
    y1 = oracle.qmv_int4_gs(wq, s, x1, 64, lib=lib)
    y2 = oracle.qmv_int4_gs(wq, s, x2, 64, lib=lib)
    _, d12 = oracle.qmv_int4_gs(wq, s, np.abs(x1) + np.abs(x2), 64, with_den=True, lib=lib)
    assert np.all(np.abs(y12 - (y1 + y2)) <= 1e-13 * d12)


def pin_int4_all_equal_closed_form(lib):
    """nibble == c everywhere: y_i = (c-8) * sum_g s_ig * sum_{k in g} x_k (exact for
    dyadic s and small-integer x)."""
    rng = _rng(5)
    N, K, S = 7, 320, 2
    x = rng.integers(-20, 21, size=(S, K)).astype(np.float32)
    s = (2.0 ** rng.integers(-8, 2, size=(N, K // 64))).astype(np.float32)
    for c in range(16):
        wq = np.full((N, K // 2), c | (c << 4), np.uint8)
        y = oracle.qmv_int4_gs(wq, s, x, 64, lib=lib)
        gsum = x.reshape(S, K // 64, 64).sum(-1).astype(np.float64)  # [S][G]
        ref = (c - 8) * (gsum @ s.astype(np.float64).T)
        assert np.array_equal(y, ref), c
        if c == 8:
            assert not np.any(y)


def pin_gs_equals_k_is_row_scale(lib):
    """One group spanning the row is a per-row scale: equals the int8 per-row path."""
    rng = _rng(6)
    N, K = 9, 256
    wq = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    r = (np.abs(rng.normal(0, 0.02, size=(N, 1))) + 1e-4).astype(np.float32)
    x = rng.normal(size=(2, K)).astype(np.float32)
    y4 = oracle.qmv_int4_gs(wq, r, x, K, lib=lib)
    y8, _ = oracle.qmv_int8_row(np_unpack(wq).astype(np.int8), r[:, 0], x, lib=lib)
    assert np.array_equal(y4, y8)


# ----------------------------------------------------------------- a3 int8

def pin_int8_exact(lib):
    rng = _rng(7)
    N, K = 6, 96
    w = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    r = np.abs(rng.normal(0, 0.01, size=N)).astype(np.float32)
    x = rng.normal(size=(2, K)).astype(np.float32)
    y, den = oracle.qmv_int8_row(w, r, x, lib=lib)
    for t in range(2):
        for i in range(N):
            exact = Fraction(float(r[i])) * sum(int(w[i, k]) * Fraction(float(x[t, k])) for k in range(K))
            mag = Fraction(float(r[i])) * sum(abs(int(w[i, k]) * Fraction(float(x[t, k]))) for k in range(K))
            assert abs(Fraction(float(y[t, i])) - exact) <= mag * Fraction(1, 2 ** 45)
            assert abs(Fraction(float(den[t, i])) - mag) <= mag * Fraction(1, 2 ** 45)
    # -128 decodes as -128
    w2 = np.full((1, 64), -128, np.int8)
    y2, _ = oracle.qmv_int8_row(w2, np.ones(1, np.float32), np.ones((1, 64), np.float32), lib=lib)
    assert y2[0, 0] == -128 * 64


# ----------------------------------------------------------------- a4 routing

def _softmax64(l):
    l = l.astype(np.float64)
    e = np.exp(l - l.max())
    return e / e.sum()


def pin_route_stable_sort(lib):
    rng = _rng(8)
    for (T, E, k) in [(5, 6, 1), (7, 6, 3), (4, 16, 8), (3, 160, 8), (2, 256, 8)]:
        logits = rng.normal(size=(T, E)).astype(np.float32)
        # crafted ties: copy some logits onto other experts
        if E >= 6:
            logits[:, 3] = logits[:, 1]
            logits[:, 5] = logits[:, 1]
        ids, w = oracle.route_topk(logits, k, lib=lib)
        for t in range(T):
            order = np.argsort(-logits[t], kind="stable")[:k]
            assert np.array_equal(ids[t], order), (ids[t], order)
            p = _softmax64(logits[t])
            ref = p[order] / p[order].sum()
            assert np.allclose(w[t], ref, rtol=1e-14, atol=0)
            assert abs(w[t].sum() - 1.0) < 1e-14


def pin_route_exhaustive(lib):
    """Tiny E: the selected set is the unique best k-subset when logits are distinct."""
    rng = _rng(9)
    for E in range(1, 7):
        for k in range(1, min(E, 3) + 1):
            logits = rng.permutation(E).astype(np.float32)[None] * np.float32(0.5)
            ids, _ = oracle.route_topk(logits, k, lib=lib)
            best = max(itertools.combinations(range(E), k), key=lambda c: sum(logits[0, list(c)]))
            assert set(ids[0].tolist()) == set(best)


def pin_golden_route(lib):
    d = json.load(open(os.path.join(GOLDEN, "route_top3_tie.json")))
    ids, w = oracle.route_topk(np.array([d["logits"]], np.float32), d["k"], lib=lib)
    assert ids[0].tolist() == d["expected_ids"]
    assert np.allclose(w[0], d["expected_w"], rtol=1e-15, atol=0)


def pin_golden_route_nan(lib):
    """NaN logits count as -inf (never ahead of a finite logit, weight 0); a
    token whose logits are all -inf or NaN takes the k lowest indices at 1/k;
    -0 ties with +0. Hand-derived fixture."""
    d = json.load(open(os.path.join(GOLDEN, "route_nan_as_minus_inf.json")))
    logits = np.array([[float(v) for v in row] for row in d["logits"]], np.float32)
    ids, w = oracle.route_topk(logits, d["k"], lib=lib)
    assert ids.tolist() == d["expected_ids"], ids
    assert np.all(np.isfinite(w))
    assert np.allclose(w, d["expected_w"], rtol=1e-15, atol=0), w


# ----------------------------------------------------------------- a5 grouping

def pin_group_bruteforce(lib):
    rng = _rng(10)
    for (T, k, E) in [(1, 8, 256), (8, 8, 160), (5, 3, 6), (33, 2, 7)]:
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        off, lst, used = oracle.group(ids, E, lib=lib)
        flat = ids.reshape(-1)
        expect_list = [p for e in range(E) for p in range(T * k) if flat[p] == e]
        assert lst.tolist() == expect_list
        counts = np.bincount(flat, minlength=E)
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(counts)]))
        assert used.tolist() == [e for e in range(E) if counts[e] > 0]


# ----------------------------------------------------------------- a6 / a7 FFN

def _rand_experts(rng, n, H, I):
    return dict(
        gu_q=rng.integers(0, 256, size=(n, 2 * I, H // 2), dtype=np.uint8),
        gu_s=(np.abs(rng.normal(0, 0.02, size=(n, 2 * I, H // 64))) + 1e-4).astype(np.float32),
        dn_q=rng.integers(0, 256, size=(n, H, I // 2), dtype=np.uint8),
        dn_s=(np.abs(rng.normal(0, 0.02, size=(n, H, I // 64))) + 1e-4).astype(np.float32),
    )


def _np_ffn(wts, e, x, I):
    Wg = np_dequant(wts["gu_q"][e, :I], wts["gu_s"][e, :I])
    Wu = np_dequant(wts["gu_q"][e, I:], wts["gu_s"][e, I:])
    Wd = np_dequant(wts["dn_q"][e], wts["dn_s"][e])
    g, u = Wg @ x, Wu @ x
    h = g / (1.0 + np.exp(-g)) * u
    return Wd @ h, h, np.abs(Wd) @ np.abs(h)


def pin_ffn_textbook_swiglu(lib):
    """k = 1, w = 1 is one SwiGLU block; k > 1 is the weighted sum of such blocks."""
    rng = _rng(11)
    H, I, n, T = 128, 192, 4, 3
    wts = _rand_experts(rng, n, H, I)
    x = rng.normal(size=(T, H))
    x = x.astype(np.float32).astype(np.float64)
    for k in (1, 3):
        ids = np.stack([rng.choice(n, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        w = np.ones((T, k), np.float32) if k == 1 else rng.random((T, k)).astype(np.float32)
        res = oracle.moe_ffn(wts, x, ids, w, want_h=True, lib=lib)
        for t in range(T):
            ref = np.zeros(H)
            den = np.zeros(H)
            for j in range(k):
                y, h, d = _np_ffn(wts, ids[t, j], x[t], I)
                ref += float(w[t, j]) * y
                den += abs(float(w[t, j])) * d
                assert np.allclose(res["h"][t * k + j], h, rtol=1e-12, atol=1e-300)
            assert np.all(np.abs(res["out"][t] - ref) <= 1e-12 * den)
            # the tolerance denominator sum_j |w_j| sum_c |D_ij h_c|, from numpy
            assert np.allclose(res["den"][t], den, rtol=1e-12, atol=0)


def pin_ffn_zero_gate(lib):
    """All gate nibbles equal 8: g = 0, SiLU(0) = 0, so out is exactly 0."""
    rng = _rng(12)
    H, I = 64, 128
    wts = _rand_experts(rng, 2, H, I)
    wts["gu_q"][:, :I] = 0x88
    x = rng.normal(size=(2, H)).astype(np.float32).astype(np.float64)
    res = oracle.moe_ffn(wts, x, np.array([[0, 1], [1, 0]], np.int32),
                         np.full((2, 2), 0.5, np.float32), lib=lib)
    assert not np.any(res["out"])


def pin_golden_swiglu(lib):
    d = json.load(open(os.path.join(GOLDEN, "swiglu_expert_closed_form.json")))
    H, I = d["H"], d["I"]
    wts = dict(
        gu_q=np.concatenate([np.full((1, I, H // 2), d["gate_byte"], np.uint8),
                             np.full((1, I, H // 2), d["up_byte"], np.uint8)], axis=1),
        gu_s=np.concatenate([np.full((1, I, H // 64), d["gate_scale"], np.float32),
                             np.full((1, I, H // 64), d["up_scale"], np.float32)], axis=1),
        dn_q=np.full((1, H, I // 2), d["down_byte"], np.uint8),
        dn_s=np.full((1, H, I // 64), d["down_scale"], np.float32),
    )
    x = np.full((1, H), d["x_value"], np.float64)
    res = oracle.moe_ffn(wts, x, np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), lib=lib)
    assert np.allclose(res["out"], d["expected_out"], rtol=1e-15, atol=0)


def pin_ffn_hidden_bound(lib):
    """hden bounds the first-order change of h when the gate and up dot products each move
    by a relative eps of their |.| sums, for every sign combination."""
    rng = _rng(13)
    H, I = 128, 64
    wts = _rand_experts(rng, 1, H, I)
    x = rng.normal(size=(1, H)).astype(np.float32).astype(np.float64)
    res = oracle.moe_ffn(wts, x, np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32),
                         want_h=True, lib=lib)
    Wg = np_dequant(wts["gu_q"][0, :I], wts["gu_s"][0, :I])
    Wu = np_dequant(wts["gu_q"][0, I:], wts["gu_s"][0, I:])
    g, u = Wg @ x[0], Wu @ x[0]
    ag, au = np.abs(Wg) @ np.abs(x[0]), np.abs(Wu) @ np.abs(x[0])
    eps = 1e-7
    h0 = g / (1 + np.exp(-g)) * u
    worst = np.zeros(I)
    for sg, su in itertools.product((-1, 1), repeat=2):
        g1, u1 = g + sg * eps * ag, u + su * eps * au
        worst = np.maximum(worst, np.abs(g1 / (1 + np.exp(-g1)) * u1 - h0))
    assert np.all(worst <= eps * res["hden"][0] * (1 + 1e-4) + 1e-300)
    # and the bound is attained by some sign pattern (not vacuous)
    assert np.all(worst >= eps * res["hden"][0] * (1 - 1e-4))


# ----------------------------------------------------------------- f2 int3-g64

def np_unpack3(wq3: np.ndarray, K: int) -> np.ndarray:
    """Reading R6 by explicit bit slicing: [N][K/64*24] bytes -> [N][K] values."""
    N = wq3.shape[0]
    g = wq3.reshape(N, K // 64, 24)
    low = np.unpackbits(g[:, :, :16], axis=2, bitorder="little").reshape(N, K // 64, 64, 2)
    lo = low[..., 0].astype(np.int16) + 2 * low[..., 1].astype(np.int16)
    hi = np.unpackbits(g[:, :, 16:], axis=2, bitorder="little").astype(np.int16)
    return (lo + 4 * hi - 4).reshape(N, K)


def pin_int3_pack_roundtrip(lib):
    rng = _rng(20)
    vals = rng.integers(-4, 4, size=64 * 20).astype(np.int8)
    b = oracle.pack_int3(vals, lib=lib)
    assert b.size == 20 * 24
    assert np.array_equal(oracle.unpack_int3(b, vals.size, lib=lib), vals)
    assert np.array_equal(np_unpack3(b[None], vals.size)[0], vals), "oracle != numpy bit slicing"
    raw = rng.integers(0, 256, size=24 * 7, dtype=np.uint8)  # every byte pattern decodes
    v = oracle.unpack_int3(raw, 7 * 64, lib=lib)
    assert v.min() >= -4 and v.max() <= 3
    assert np.array_equal(oracle.pack_int3(v, lib=lib), raw)


def pin_int3_as_int4(lib):
    """An int3 matrix re-encoded as int4 nibbles (value + 8) gives the same y,
    bit for bit: both forms sum the same products in the same order."""
    rng = _rng(21)
    for (N, K, S) in [(5, 64, 1), (9, 256, 3), (17, 1024, 2)]:
        vals = rng.integers(-4, 4, size=(N, K)).astype(np.int8)
        wq3 = np.stack([oracle.pack_int3(vals[i], lib=lib) for i in range(N)])
        wq4 = np.stack([oracle.pack_int4(vals[i], lib=lib) for i in range(N)])
        s = (np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4).astype(np.float32)
        x = rng.normal(size=(S, K)).astype(np.float32)
        y3, d3 = oracle.qmv_int3_gs(wq3, s, x, lib=lib)
        y4 = oracle.qmv_int4_gs(wq4, s, x, 64, lib=lib)
        assert np.array_equal(y3, y4)
        assert np.all(d3 >= np.abs(y3) * (1 - 1e-12))


def pin_int3_exact_bruteforce(lib):
    rng = _rng(22)
    for (N, K, S) in [(2, 64, 1), (3, 128, 2)]:
        vals = rng.integers(-4, 4, size=(N, K)).astype(np.int8)
        wq3 = np.stack([oracle.pack_int3(vals[i], lib=lib) for i in range(N)])
        s = (np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4).astype(np.float32)
        x = rng.normal(size=(S, K)).astype(np.float32)
        y, _ = oracle.qmv_int3_gs(wq3, s, x, lib=lib)
        for t in range(S):
            for i in range(N):
                exact = sum(int(vals[i, k]) * Fraction(float(s[i, k // 64])) * Fraction(float(x[t, k]))
                            for k in range(K))
                mag = sum(abs(int(vals[i, k]) * Fraction(float(s[i, k // 64])) * Fraction(float(x[t, k])))
                          for k in range(K))
                assert abs(Fraction(float(y[t, i])) - exact) <= mag * Fraction(1, 2 ** 45)


def pin_int3_den(lib):
    """den = |W3| @ |x| over a numpy bit-sliced matrix times its group scales."""
    rng = _rng(23)
    for (N, K, S) in [(7, 128, 2), (12, 512, 3)]:
        vals = rng.integers(-4, 4, size=(N, K)).astype(np.int8)
        wq3 = np.stack([oracle.pack_int3(vals[i], lib=lib) for i in range(N)])
        s = (np.abs(rng.normal(0, 0.02, size=(N, K // 64))) + 1e-4).astype(np.float32)
        x = rng.normal(size=(S, K)).astype(np.float32)
        W3 = np_unpack3(wq3, K).astype(np.float64) * np.repeat(s.astype(np.float64), 64, axis=-1)
        y, den = oracle.qmv_int3_gs(wq3, s, x, lib=lib)
        ref_den = np.abs(x.astype(np.float64)) @ np.abs(W3).T
        assert np.allclose(den, ref_den, rtol=1e-12, atol=0)
        assert np.all(np.abs(y - x.astype(np.float64) @ W3.T) <= 1e-13 * ref_den)


def pin_golden_int3_planes(lib):
    d = json.load(open(os.path.join(GOLDEN, "int3_g64_two_plane.json")))
    row = np.array([d["low_byte"]] * 16 + [d["high_byte"]] * 8, np.uint8)
    v = oracle.unpack_int3(row, 64, lib=lib)
    assert v[:8].tolist() == d["expected_values_first8"]
    x = np.where(np.arange(64) % 4 == 3, 3.0, 1.0).astype(np.float32)[None]
    y, _ = oracle.qmv_int3_gs(row[None], np.array([[d["scale"]]], np.float32), x, lib=lib)
    assert y[0, 0] == d["expected_y"]


ALL_PINS = [
    pin_pack_roundtrip, pin_golden_nibble_order, pin_int4_exact_bruteforce,
    pin_int4_library_identity, pin_int4_linearity, pin_int4_all_equal_closed_form,
    pin_gs_equals_k_is_row_scale, pin_int8_exact, pin_route_stable_sort, pin_route_exhaustive,
    pin_golden_route, pin_golden_route_nan, pin_group_bruteforce, pin_ffn_textbook_swiglu, pin_ffn_zero_gate,
    pin_golden_swiglu, pin_ffn_hidden_bound, pin_int3_pack_roundtrip, pin_int3_as_int4,
    pin_int3_exact_bruteforce, pin_int3_den, pin_golden_int3_planes,
]
