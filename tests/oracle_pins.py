"""Pins for the CPU oracle: facts fixed by the pages and by the mathematics.

Each pin takes an oracle object (``sdpa``/``mha`` methods) and raises
AssertionError when the oracle disagrees.  They are collected into ``PINS`` so
the same checks run against the real oracle and against deliberately broken
copies of it (every broken copy must fail at least one pin).

Sources of the fixed values:
  - worked example with key dimension 1 (Arquitectura Transformer, section
    "Como hacerlo"), stored in golden/worked_example_dk1.json;
  - toy rows of Fig. 1 and Fig. 2 (Self-Attention explainer), stored in
    golden/toy_rows_fig2.json;
  - Eq. (1) and its footnote on the 1/sqrt(d_k) scale ("Attention Is All You
    Need", section 3.2.1), the causal mask of section 3.2.3 and the multi-head
    definition of section 3.2.2, through closed forms and invariants;
  - a brute-force evaluation in 50-digit decimal arithmetic, written
    independently (explicit score matrix, softmax without the max shift).
"""
from __future__ import annotations

import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np

MASK_NONE, MASK_CAUSAL, MASK_PADDING = 0, 1, 2
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _t(x):
    """Lift a 2-D [n, d] array to BHSD [1, 1, n, d]."""
    return np.asarray(x, dtype=np.float64)[None, None]


def _parse_key(s):
    return math.log(3.0) if s == "ln3" else float(s)


# --------------------------------------------------------------------------
def pin_worked_example(o):
    g = _golden("worked_example_dk1.json")
    q = _t([g["q"]])
    k = _t([[_parse_key(s)] for s in g["keys"]])
    v = _t([[x] for x in g["values"]])
    out = o.sdpa(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32))
    # float32 storage of ln(3) limits agreement to ~1e-7
    assert abs(out[0, 0, 0, 0] - g["output"]) < 1e-6, out
    # weights: with V = identity the output row is the weight row
    eye = _t(np.eye(2))
    w = o.sdpa(q.astype(np.float32), k.astype(np.float32), eye.astype(np.float32))
    assert np.allclose(w[0, 0, 0], g["weights"], atol=1e-6), w
    # second key forbidden: key padding with length 1
    lens = np.array([1], dtype=np.int32)
    out_m = o.sdpa(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32),
                   MASK_PADDING, lens)
    assert out_m[0, 0, 0, 0] == g["masked_second_key"]["output"], out_m
    w_m = o.sdpa(q.astype(np.float32), k.astype(np.float32), eye.astype(np.float32),
                 MASK_PADDING, lens)
    assert np.array_equal(w_m[0, 0, 0], g["masked_second_key"]["weights"]), w_m


def pin_worked_example_causal(o):
    """Same numbers as a two-position decoder: row 0 may not see key 1."""
    g = _golden("worked_example_dk1.json")
    q = _t([g["q"], g["q"]]).astype(np.float32)
    k = _t([[_parse_key(s)] for s in g["keys"]]).astype(np.float32)
    v = _t([[x] for x in g["values"]]).astype(np.float32)
    out = o.sdpa(q, k, v, MASK_CAUSAL)
    assert out[0, 0, 0, 0] == g["masked_second_key"]["output"], out
    assert abs(out[0, 0, 1, 0] - g["output"]) < 1e-6, out


def pin_toy_rows(o):
    g = _golden("toy_rows_fig2.json")
    vals = _t([[x] for x in g["values"]]).astype(np.float32)
    n = len(g["values"])
    for row in g["rows"]:
        # logits log(w) at temperature 1 reproduce the table weights
        k = _t([[math.log(w)] for w in row["weights"]]).astype(np.float32)
        q = _t([[1.0]]).astype(np.float32)
        out = o.sdpa(q, k, vals, scale=1.0)
        assert abs(out[0, 0, 0, 0] - row["output"]) < 1e-5, (row, out)
        w = o.sdpa(q, k, _t(np.eye(n)).astype(np.float32), scale=1.0)
        assert np.allclose(w[0, 0, 0], row["weights"], atol=1e-7), w
    # causal: the first position keeps everything on itself
    k = _t([[math.log(w)] for w in g["rows"][0]["weights"]]).astype(np.float32)
    q = np.ones((1, 1, n, 1), dtype=np.float32)
    out = o.sdpa(q, k, vals, MASK_CAUSAL, scale=1.0)
    assert out[0, 0, 0, 0] == g["causal_first_row"]["output"], out


def pin_scale_is_inverse_sqrt_dk(o):
    """Footnote to Eq. (1): dot products are divided by sqrt(d_k).

    With q = ones(d) and key 1 = (ln3 / sqrt(d)) * ones(d), q.k1 / sqrt(d) = ln 3
    and key 2 = 0, so the worked example's weights 3/4, 1/4 and output 3 return
    for every d; any other power of d breaks it for d > 1.
    """
    for d in (4, 9, 64):
        q = np.ones((1, 1, 1, d), dtype=np.float64)
        k = np.zeros((1, 1, 2, d), dtype=np.float64)
        k[0, 0, 0, :] = math.log(3.0) / math.sqrt(d)
        v = np.zeros((1, 1, 2, 1))
        v[0, 0, :, 0] = [2.0, 6.0]
        out = o.sdpa(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32))
        assert abs(out[0, 0, 0, 0] - 3.0) < 1e-5, (d, out)


def pin_rows_sum_to_one(o):
    rng = np.random.default_rng(7)
    for mask in (MASK_NONE, MASK_CAUSAL, MASK_PADDING, MASK_CAUSAL | MASK_PADDING):
        q = rng.standard_normal((2, 3, 9, 5)).astype(np.float32)
        k = rng.standard_normal((2, 3, 9, 5)).astype(np.float32)
        v = np.ones((2, 3, 9, 4), dtype=np.float32)
        lens = np.array([9, 4], dtype=np.int32)
        out = o.sdpa(q, k, v, mask, lens if mask & MASK_PADDING else None)
        assert np.allclose(out, 1.0, atol=1e-13), (mask, out)


def pin_equal_scores_give_mean(o):
    """Equal keys give equal scores; the softmax then splits evenly (the
    explainer's [100,100,100] vs [0,0,0] remark), so the output is the mean of
    the visible value rows."""
    rng = np.random.default_rng(8)
    n, d = 7, 6
    q = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    key = rng.standard_normal(d).astype(np.float32)
    k = np.broadcast_to(key, (1, 1, n, d)).copy()
    v = rng.standard_normal((1, 1, n, 3)).astype(np.float32)
    out = o.sdpa(q, k, v)
    assert np.allclose(out[0, 0], v[0, 0].astype(np.float64).mean(0), atol=1e-12)
    out_c = o.sdpa(q, k, v, MASK_CAUSAL)
    for i in range(n):
        assert np.allclose(out_c[0, 0, i], v[0, 0, : i + 1].astype(np.float64).mean(0), atol=1e-12)
    lens = np.array([3], dtype=np.int32)
    out_p = o.sdpa(q, k, v, MASK_PADDING, lens)
    assert np.allclose(out_p[0, 0], v[0, 0, :3].astype(np.float64).mean(0), atol=1e-12)


def pin_high_temperature_is_uniform(o):
    """As the temperature grows (scale -> 0) the weights tend to 1/n."""
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 2, 5, 4)).astype(np.float32)
    k = rng.standard_normal((1, 2, 6, 4)).astype(np.float32)
    v = rng.standard_normal((1, 2, 6, 3)).astype(np.float32)
    out = o.sdpa(q, k, v, scale=1e-12)
    mean = v.astype(np.float64).mean(2, keepdims=True)
    assert np.allclose(out, np.broadcast_to(mean, out.shape), atol=1e-9)


def pin_shift_invariance(o):
    """Adding one constant to every score of a row changes nothing."""
    g = _golden("worked_example_dk1.json")
    base = [_parse_key(s) for s in g["keys"]]
    v = _t([[x] for x in g["values"]]).astype(np.float32)
    q = _t([[1.0]]).astype(np.float32)
    for c in (-50.0, 25.0, 750.0):  # exp(750) overflows fp64 without the max shift
        k = _t([[x + c] for x in base]).astype(np.float32)
        out = o.sdpa(q, k, v)
        assert abs(out[0, 0, 0, 0] - g["output"]) < 1e-3, (c, out)


def pin_causal_ignores_future(o):
    rng = np.random.default_rng(10)
    n, d = 11, 4
    q = rng.standard_normal((2, 2, n, d)).astype(np.float32)
    k = rng.standard_normal((2, 2, n, d)).astype(np.float32)
    v = rng.standard_normal((2, 2, n, d)).astype(np.float32)
    ref = o.sdpa(q, k, v, MASK_CAUSAL)
    for i in (0, 3, n - 2):
        k2, v2 = k.copy(), v.copy()
        k2[:, :, i + 1:] = rng.standard_normal(k2[:, :, i + 1:].shape) * 5
        v2[:, :, i + 1:] = rng.standard_normal(v2[:, :, i + 1:].shape) * 5
        out = o.sdpa(q, k2, v2, MASK_CAUSAL)
        assert np.array_equal(out[:, :, : i + 1], ref[:, :, : i + 1]), i
        assert not np.allclose(out[:, :, i + 1:], ref[:, :, i + 1:])
    # the first position sees only itself
    assert np.allclose(ref[:, :, 0], v[:, :, 0], atol=0)


def pin_padding_ignores_masked_keys(o):
    rng = np.random.default_rng(11)
    b, n, d = 3, 9, 5
    q = rng.standard_normal((b, 2, n, d)).astype(np.float32)
    k = rng.standard_normal((b, 2, n, d)).astype(np.float32)
    v = rng.standard_normal((b, 2, n, d)).astype(np.float32)
    lens = np.array([5, 1, 0], dtype=np.int32)
    ref = o.sdpa(q, k, v, MASK_PADDING, lens)
    k2, v2 = k.copy(), v.copy()
    for bi, L in enumerate(lens):
        k2[bi, :, L:] = rng.standard_normal(k2[bi, :, L:].shape) * 5
        v2[bi, :, L:] = rng.standard_normal(v2[bi, :, L:].shape) * 5
    out = o.sdpa(q, k2, v2, MASK_PADDING, lens)
    assert np.array_equal(out, ref)
    # length 1: every query returns value row 0
    assert np.allclose(ref[1], np.broadcast_to(v[1, :, :1], ref[1].shape), atol=0)
    # length 0: no visible key, the row is 0 by convention
    assert np.array_equal(ref[2], np.zeros_like(ref[2]))
    # lengths clamp into [0, n_k]
    big = o.sdpa(q, k, v, MASK_PADDING, np.array([n + 7, -3, n], dtype=np.int32))
    assert np.array_equal(big[0], o.sdpa(q, k, v)[0])
    assert np.array_equal(big[1], np.zeros_like(big[1]))


def pin_permutation_equivariance(o):
    """Without masks or positions, attention treats keys as a set and maps each
    query independently."""
    rng = np.random.default_rng(12)
    q = rng.standard_normal((1, 2, 6, 4)).astype(np.float32)
    k = rng.standard_normal((1, 2, 8, 4)).astype(np.float32)
    v = rng.standard_normal((1, 2, 8, 3)).astype(np.float32)
    ref = o.sdpa(q, k, v)
    pk = rng.permutation(8)
    out = o.sdpa(q, k[:, :, pk], v[:, :, pk])
    assert np.allclose(out, ref, atol=1e-14)
    pq = rng.permutation(6)
    out_q = o.sdpa(q[:, :, pq], k, v)
    assert np.allclose(out_q, ref[:, :, pq], atol=0)


def _decimal_attention(q, k, v, mask, lens, scale, window=None):
    """Independent brute force: explicit score matrix, softmax as
    exp(s)/sum(exp(s)) without a max shift, all in 50-digit decimals.
    ``window`` = r keeps keys i - (r-1)//2 .. i + r//2 (restricted attention)."""
    getcontext().prec = 50
    b, h, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    out = np.zeros((b, h, n_q, d_v))
    sc = Decimal(scale) if scale > 0 else Decimal(1) / Decimal(d_k).sqrt()
    for bi in range(b):
        L = n_k if not (mask & MASK_PADDING) else max(0, min(n_k, int(lens[bi])))
        for hi in range(h):
            S = [[None] * n_k for _ in range(n_q)]
            for i in range(n_q):
                for j in range(n_k):
                    if j >= L or ((mask & MASK_CAUSAL) and j > i):
                        continue
                    if window is not None and not (i - (window - 1) // 2 <= j <= i + window // 2):
                        continue
                    S[i][j] = sc * sum(Decimal(float(q[bi, hi, i, c])) * Decimal(float(k[bi, hi, j, c]))
                                       for c in range(d_k))
            for i in range(n_q):
                e = [s.exp() if s is not None else Decimal(0) for s in S[i]]
                tot = sum(e)
                if tot == 0:
                    continue
                for c in range(d_v):
                    acc = sum(e[j] / tot * Decimal(float(v[bi, hi, j, c])) for j in range(n_k))
                    out[bi, hi, i, c] = float(acc)
    return out


def pin_brute_force(o):
    rng = np.random.default_rng(13)
    cases = [(1, 1, 1, 1, 1, 1), (2, 2, 5, 5, 3, 2), (1, 3, 4, 7, 4, 3), (2, 1, 6, 6, 2, 4)]
    for (b, h, n_q, n_k, d_k, d_v) in cases:
        q = (rng.standard_normal((b, h, n_q, d_k)) * 2).astype(np.float32)
        k = (rng.standard_normal((b, h, n_k, d_k)) * 2).astype(np.float32)
        v = rng.standard_normal((b, h, n_k, d_v)).astype(np.float32)
        lens = rng.integers(0, n_k + 1, size=b).astype(np.int32)
        masks = [MASK_NONE, MASK_PADDING] + ([MASK_CAUSAL, MASK_CAUSAL | MASK_PADDING] if n_q == n_k else [])
        for mask in masks:
            for scale in (0.0, 0.7):
                ref = _decimal_attention(q, k, v, mask, lens, scale)
                out = o.sdpa(q, k, v, mask, lens if mask & MASK_PADDING else None, scale)
                assert np.allclose(out, ref, rtol=0, atol=1e-13), (b, h, n_q, n_k, mask, scale)


def pin_rows_selection(o):
    """The sampled-rows mode returns exactly the rows of the full evaluation."""
    rng = np.random.default_rng(14)
    q = rng.standard_normal((2, 3, 7, 4)).astype(np.float32)
    k = rng.standard_normal((2, 3, 7, 4)).astype(np.float32)
    v = rng.standard_normal((2, 3, 7, 5)).astype(np.float32)
    full = o.sdpa(q, k, v, MASK_CAUSAL)
    rows = np.array([0, 41, 13, 6, 20], dtype=np.int64)
    part = o.sdpa(q, k, v, MASK_CAUSAL, rows=rows)
    assert np.array_equal(part, full.reshape(-1, 5)[rows])


# ---------------------------------------------------------------- multi-head
def pin_mha_single_head_identity(o):
    """h = 1 with identity projections reduces MultiHead to Eq. (1)."""
    rng = np.random.default_rng(20)
    b, n_q, n_k, dm = 2, 5, 7, 4
    xq = rng.standard_normal((b, n_q, dm)).astype(np.float32)
    xkv = rng.standard_normal((b, n_k, dm)).astype(np.float32)
    eye = np.eye(dm, dtype=np.float32)
    lens = np.array([7, 3], dtype=np.int32)
    y = o.mha(xq, xkv, eye, eye, eye, eye, 1, dm, dm, MASK_PADDING, lens)
    ref = o.sdpa(xq[:, None], xkv[:, None], xkv[:, None], MASK_PADDING, lens)[:, 0]
    assert np.allclose(y, ref, atol=1e-14)


def _np_mha(xq, xkv, wq, wk, wv, wo, h, d_k, d_v, mask, lens):
    """Second formulation with numpy matmuls over whole matrices."""
    xq, xkv, wq, wk, wv, wo = (a.astype(np.float64) for a in (xq, xkv, wq, wk, wv, wo))
    b, n_q, _ = xq.shape
    n_k = xkv.shape[1]
    Q = (xq @ wq).reshape(b, n_q, h, d_k).transpose(0, 2, 1, 3)
    K = (xkv @ wk).reshape(b, n_k, h, d_k).transpose(0, 2, 1, 3)
    V = (xkv @ wv).reshape(b, n_k, h, d_v).transpose(0, 2, 1, 3)
    S = Q @ K.transpose(0, 1, 3, 2) / math.sqrt(d_k)
    vis = np.ones((b, 1, n_q, n_k), dtype=bool)
    if mask & MASK_CAUSAL:
        vis &= np.tril(np.ones((n_q, n_k), dtype=bool))[None, None]
    if mask & MASK_PADDING:
        vis &= (np.arange(n_k)[None, :] < lens[:, None])[:, None, None, :]
    E = np.where(vis, np.exp(np.where(vis, S, 0.0)), 0.0)
    P = E / E.sum(-1, keepdims=True)
    heads = P @ V
    concat = heads.transpose(0, 2, 1, 3).reshape(b, n_q, h * d_v)
    return concat @ wo


def pin_mha_matches_matrix_form(o):
    rng = np.random.default_rng(21)
    for (b, n_q, n_k, dm, h, d_k, d_v, mask) in [(2, 6, 6, 8, 2, 3, 4, MASK_CAUSAL),
                                                 (3, 4, 7, 6, 3, 2, 2, MASK_PADDING),
                                                 (1, 5, 5, 10, 2, 5, 5, MASK_NONE)]:
        xq = rng.standard_normal((b, n_q, dm)).astype(np.float32)
        xkv = xq if n_q == n_k and mask != MASK_PADDING else rng.standard_normal((b, n_k, dm)).astype(np.float32)
        wq = rng.standard_normal((dm, h * d_k)).astype(np.float32) / 2
        wk = rng.standard_normal((dm, h * d_k)).astype(np.float32) / 2
        wv = rng.standard_normal((dm, h * d_v)).astype(np.float32) / 2
        wo = rng.standard_normal((h * d_v, dm)).astype(np.float32) / 2
        lens = rng.integers(1, n_k + 1, size=b).astype(np.int32)
        y = o.mha(xq, xkv, wq, wk, wv, wo, h, d_k, d_v, mask, lens)
        ref = _np_mha(xq, xkv, wq, wk, wv, wo, h, d_k, d_v, mask, lens)
        assert np.allclose(y, ref, atol=1e-12), (b, n_q, n_k, mask)


def pin_mha_concat_not_average(o):
    """Heads are concatenated (section 3.2.2): with W^O selecting head 2's
    block, the output is exactly head 2's attention, not a mix of heads."""
    rng = np.random.default_rng(22)
    b, n, dm, h, d = 1, 5, 6, 3, 2
    x = rng.standard_normal((b, n, dm)).astype(np.float32)
    wq = rng.standard_normal((dm, h * d)).astype(np.float32)
    wk = rng.standard_normal((dm, h * d)).astype(np.float32)
    wv = rng.standard_normal((dm, h * d)).astype(np.float32)
    sel = 2
    wo = np.zeros((h * d, dm), dtype=np.float32)
    wo[sel * d:(sel + 1) * d, :d] = np.eye(d)
    y = o.mha(x, x, wq, wk, wv, wo, h, d, d)
    xq64 = x.astype(np.float64)[0]
    Q = xq64 @ wq[:, sel * d:(sel + 1) * d]
    K = xq64 @ wk[:, sel * d:(sel + 1) * d]
    V = xq64 @ wv[:, sel * d:(sel + 1) * d]
    head = o.sdpa(Q[None, None].astype(np.float32), K[None, None].astype(np.float32),
                  V[None, None].astype(np.float32))[0, 0]
    assert np.allclose(y[0, :, :d], head, atol=1e-6)
    assert np.array_equal(y[0, :, d:], np.zeros((n, dm - d)))


def pin_mha_rows_selection(o):
    rng = np.random.default_rng(23)
    b, n_q, n_k, dm, h, d = 3, 4, 6, 8, 2, 4
    xq = rng.standard_normal((b, n_q, dm)).astype(np.float32)
    xkv = rng.standard_normal((b, n_k, dm)).astype(np.float32)
    ws = [rng.standard_normal(s).astype(np.float32) for s in [(dm, h * d)] * 3 + [(h * d, dm)]]
    lens = np.array([6, 2, 4], dtype=np.int32)
    full = o.mha(xq, xkv, *ws, h, d, d, MASK_PADDING, lens)
    rows = np.array([11, 0, 5, 7], dtype=np.int64)
    part = o.mha(xq, xkv, *ws, h, d, d, MASK_PADDING, lens, rows=rows)
    assert np.array_equal(part, full.reshape(-1, dm)[rows])


# ------------------------------------------------------ restricted attention
def pin_restricted_worked_example(o):
    """Section 4's neighbourhood of size r around position i, on the worked
    example's numbers: with r = 2 position 0 sees keys 0 and 1 (weights 3/4,
    1/4, output 3); with r = 3 and the causal mask position 1 sees keys 0 and
    1 (output 3) and position 0 sees only itself (output 2)."""
    g = _golden("worked_example_dk1.json")
    keys = [_parse_key(s) for s in g["keys"]] + [5.0]
    vals = g["values"] + [10.0]
    q = np.ones((1, 1, 3, 1), np.float32)
    k = _t([[x] for x in keys]).astype(np.float32)
    v = _t([[x] for x in vals]).astype(np.float32)
    out = o.sdpa(q, k, v, window=2)
    assert abs(out[0, 0, 0, 0] - g["output"]) < 1e-6, out
    w = o.sdpa(q, k, _t(np.eye(3)).astype(np.float32), window=2)
    assert np.allclose(w[0, 0, 0], g["weights"] + [0.0], atol=1e-6), w
    outc = o.sdpa(q, k, v, MASK_CAUSAL, window=3)
    assert outc[0, 0, 0, 0] == g["masked_second_key"]["output"], outc
    assert abs(outc[0, 0, 1, 0] - g["output"]) < 1e-6, outc
    e = math.exp(5.0)
    assert abs(outc[0, 0, 2, 0] - (6.0 + 10.0 * e) / (1.0 + e)) < 1e-5, outc


def pin_restricted_extremes(o):
    """r = 1 keeps only position i (output = V[i]); r covering the whole
    sequence changes nothing."""
    rng = np.random.default_rng(30)
    n = 13
    q = rng.standard_normal((2, 2, n, 4)).astype(np.float32)
    k = rng.standard_normal((2, 2, n, 4)).astype(np.float32)
    v = rng.standard_normal((2, 2, n, 3)).astype(np.float32)
    one = o.sdpa(q, k, v, window=1)
    assert np.array_equal(one, v.astype(np.float64))
    lens = np.array([n, 6], np.int32)
    for mask in (MASK_NONE, MASK_CAUSAL, MASK_PADDING, MASK_CAUSAL | MASK_PADDING):
        ln = lens if mask & MASK_PADDING else None
        assert np.array_equal(o.sdpa(q, k, v, mask, ln, window=2 * n + 1), o.sdpa(q, k, v, mask, ln))


def pin_restricted_brute_force(o):
    rng = np.random.default_rng(31)
    for (n_q, n_k, d) in [(6, 6, 3), (5, 8, 2)]:
        q = rng.standard_normal((2, 1, n_q, d)).astype(np.float32)
        k = rng.standard_normal((2, 1, n_k, d)).astype(np.float32)
        v = rng.standard_normal((2, 1, n_k, 2)).astype(np.float32)
        lens = np.array([n_k, 3], np.int32)
        masks = [MASK_NONE, MASK_PADDING] + ([MASK_CAUSAL, MASK_CAUSAL | MASK_PADDING] if n_q == n_k else [])
        for mask in masks:
            for r in (1, 2, 3, 4, 7):
                ref = _decimal_attention(q, k, v, mask, lens, 0.0, window=r)
                out = o.sdpa(q, k, v, mask, lens if mask & MASK_PADDING else None, window=r)
                assert np.allclose(out, ref, rtol=0, atol=1e-13), (n_q, n_k, mask, r)


# ---------------------------------------------------------------- decoding
def pin_decode_matches_causal_rows(o):
    """A decoding step of n_q queries over a cache of length n equals the last
    n_q rows of causal self-attention over the full sequence; one query over
    the whole cache equals unmasked attention of that query."""
    rng = np.random.default_rng(40)
    n, d = 11, 4
    q = rng.standard_normal((2, 2, n, d)).astype(np.float32)
    k = rng.standard_normal((2, 2, n, d)).astype(np.float32)
    v = rng.standard_normal((2, 2, n, 3)).astype(np.float32)
    full = o.sdpa(q, k, v, MASK_CAUSAL)
    for n_q in (1, 3, n):
        dec = o.decode(q[:, :, n - n_q:], k, v)
        assert np.array_equal(dec, full[:, :, n - n_q:]), n_q
    one = o.decode(q[:, :, 4:5], k, v)
    assert np.array_equal(one, o.sdpa(q[:, :, 4:5], k, v))


def pin_decode_cache_lengths(o):
    """Per-sequence cache lengths: keys past len_b are ignored; a query placed
    before the cache start sees nothing (zeros); the worked example as a
    one-query step over a two-entry cache gives 3."""
    rng = np.random.default_rng(41)
    n, d = 9, 3
    q = rng.standard_normal((3, 1, 2, d)).astype(np.float32)
    k = rng.standard_normal((3, 1, n, d)).astype(np.float32)
    v = rng.standard_normal((3, 1, n, 2)).astype(np.float32)
    lens = np.array([5, 1, 0], np.int32)
    dec = o.decode(q, k, v, lens)
    ref0 = o.sdpa(q[:1], k[:1, :, :5], v[:1, :, :5], MASK_NONE)    # both queries see keys < 5 ...
    ref0c = o.decode(q[:1], k[:1, :, :5], v[:1, :, :5])            # ... with the causal shift
    assert np.array_equal(dec[0], ref0c[0])
    assert np.array_equal(dec[0, :, 1], ref0[0, :, 1])             # last query sees the whole cache
    assert np.array_equal(dec[1, :, 0], np.zeros((1, 2)))          # position -1: nothing
    assert np.allclose(dec[1, :, 1], v[1, :, 0], atol=0)           # position 0: key 0 only
    assert np.array_equal(dec[2], np.zeros_like(dec[2]))
    g = _golden("worked_example_dk1.json")
    kk = _t([[_parse_key(x)] for x in g["keys"]]).astype(np.float32)
    vv = _t([[x] for x in g["values"]]).astype(np.float32)
    w = o.decode(_t([g["q"]]).astype(np.float32), kk, vv)
    assert abs(w[0, 0, 0, 0] - g["output"]) < 1e-6


# ---------------------------------------------------------------- gradients
def pin_backward_finite_differences(o):
    """The gradients are those of L = sum(dO * Attention(Q, K, V)): central
    differences of the oracle's own forward along random directions agree."""
    rng = np.random.default_rng(50)
    cases = [(2, 2, 5, 5, 3, 2, MASK_CAUSAL, None), (1, 2, 4, 7, 4, 3, MASK_PADDING, None),
             (2, 1, 6, 6, 2, 2, MASK_NONE, 3), (1, 1, 6, 6, 3, 3, MASK_CAUSAL | MASK_PADDING, 4)]
    for (b, h, n_q, n_k, d_k, d_v, mask, r) in cases:
        q = rng.standard_normal((b, h, n_q, d_k))
        k = rng.standard_normal((b, h, n_k, d_k))
        v = rng.standard_normal((b, h, n_k, d_v))
        do = rng.standard_normal((b, h, n_q, d_v))
        lens = np.array([n_k, max(1, n_k // 2)][:b], np.int32) if mask & MASK_PADDING else None
        # float32 storage: keep the inputs exactly representable
        q, k, v, do = (x.astype(np.float32).astype(np.float64) for x in (q, k, v, do))
        dq, dk, dv = o.backward(q, k, v, do, mask, lens, window=r)

        def loss(qq, kk, vv):
            return float(np.sum(do * o.sdpa(qq, kk, vv, mask, lens, window=r)))
        eps = 1e-3
        for (x, g, which) in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
            direction = rng.standard_normal(x.shape)
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which] = x + eps * direction
            args_m[which] = x - eps * direction
            # the oracle reads float32: central differences on float64 copies
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - float(np.sum(g * direction))) < 2e-4 * (1 + abs(fd)), (which, mask, fd)


def pin_backward_closed_forms(o):
    """Identical keys give dQ = 0 (softmax rows sum to one, so the rows of dS
    sum to zero); the dV rows sum to the dO rows; keys hidden by padding get
    zero gradient."""
    rng = np.random.default_rng(51)
    n, d = 6, 3
    q = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    key = rng.standard_normal(d).astype(np.float32)
    k = np.broadcast_to(key, (1, 1, n, d)).copy()
    v = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    do = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    dq, dk, dv = o.backward(q, k, v, do)
    assert np.allclose(dq, 0.0, atol=1e-12)
    assert np.allclose(dv.sum(2), do.astype(np.float64).sum(2), atol=1e-12)
    k2 = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    lens = np.array([4], np.int32)
    dq, dk, dv = o.backward(q, k2, v, do, MASK_PADDING, lens)
    assert np.array_equal(dk[0, 0, 4:], np.zeros((2, d))) and np.array_equal(dv[0, 0, 4:], np.zeros((2, d)))
    assert np.allclose(dv.sum(2), do.astype(np.float64).sum(2), atol=1e-12)


def pin_backward_given_output(o):
    """The forward output handed to the backward enters only through
    D_i = dO_i . O_i.  Handing in the exact output (rounded to float32)
    changes the gradients by that rounding alone.  Moving row i of it so that
    D_i moves by c_i leaves dV unchanged, moves dQ_i by -scale c_i sum_j P_ij k_j
    (the attention output of row i with the keys as values), and moves the sum
    of dK over keys by -scale sum_i c_i q_i over the rows that see a key."""
    rng = np.random.default_rng(53)
    b, h, n, d_k, d_v = 2, 2, 7, 3, 4
    q = rng.standard_normal((b, h, n, d_k)).astype(np.float32)
    k = rng.standard_normal((b, h, n, d_k)).astype(np.float32)
    v = rng.standard_normal((b, h, n, d_v)).astype(np.float32)
    do = rng.standard_normal((b, h, n, d_v)).astype(np.float32)
    lens = np.array([n, 4], np.int32)
    scale = 1.0 / np.sqrt(d_k)
    for mask, r in ((MASK_NONE, None), (MASK_CAUSAL | MASK_PADDING, None), (MASK_PADDING, 3)):
        exact = o.backward(q, k, v, do, mask, lens, window=r)
        out32 = o.sdpa(q, k, v, mask, lens, window=r).astype(np.float32)
        given = o.backward(q, k, v, do, mask, lens, window=r, out=out32)
        assert np.array_equal(given[2], exact[2])
        for g, e in zip(given[:2], exact[:2]):
            assert np.allclose(g, e, rtol=0, atol=1e-6), mask
        moved = (out32 + rng.standard_normal(out32.shape).astype(np.float32)).astype(np.float32)
        c = (np.einsum("bhic,bhic->bhi", do.astype(np.float64), moved.astype(np.float64))
             - np.einsum("bhic,bhic->bhi", do.astype(np.float64), out32.astype(np.float64)))
        dq, dk, dv = o.backward(q, k, v, do, mask, lens, window=r, out=moved)
        assert np.array_equal(dv, given[2])
        kbar = o.sdpa(q, k, k, mask, lens, window=r)
        assert np.allclose(dq, given[0] - scale * c[..., None] * kbar, rtol=0, atol=1e-10), mask
        seen = np.isfinite(o.lse(q, k, mask, lens, window=r))
        want = given[1].sum(2) - scale * np.einsum("bhi,bhic->bhc", np.where(seen, c, 0.0),
                                                   q.astype(np.float64))
        assert np.allclose(dk.sum(2), want, rtol=0, atol=1e-10), mask


def pin_lse_closed_forms(o):
    """The per-row log-sum-exp: zero keys give ln(number of visible keys)
    under every mask; a row that sees nothing gives -inf; one query 1 against
    keys 0 and t (d_k = 1, scale 1) gives ln(1 + e^t)."""
    n, d = 9, 4
    zeros_q = np.ones((2, 1, n, d), np.float32)
    zeros_k = np.zeros((2, 1, n, d), np.float32)
    lens = np.array([n, 3], np.int32)
    lse = o.lse(zeros_q, zeros_k, MASK_CAUSAL | MASK_PADDING, lens, window=5)
    for bi in range(2):
        for i in range(n):
            # visible: j <= i, j < len, i - 2 <= j <= i + 2
            count = sum(1 for j in range(n) if j <= i and j < lens[bi] and i - 2 <= j <= i + 2)
            want = np.log(count) if count else -np.inf
            assert lse[bi, 0, i] == want or abs(lse[bi, 0, i] - want) < 1e-12, (bi, i)
    assert np.all(np.isneginf(o.lse(zeros_q[:1], zeros_k[:1], MASK_PADDING,
                                    np.array([0], np.int32))))
    t = np.float32(1.0986123)
    q = np.ones((1, 1, 1, 1), np.float32)
    k = np.array([0.0, t], np.float32).reshape(1, 1, 2, 1)
    got = o.lse(q, k, scale=1.0)[0, 0, 0]
    assert abs(got - np.log1p(np.exp(np.float64(t)))) < 1e-12


def pin_lse_rebuilds_softmax(o):
    """exp(scale q_i.k_j - lse_i) are the softmax weights: with V the identity
    (one value row per key) the attention output is exactly those weights."""
    rng = np.random.default_rng(52)
    b, h, n, d = 2, 2, 11, 5
    q = (rng.standard_normal((b, h, n, d)) * 2).astype(np.float32)
    k = rng.standard_normal((b, h, n, d)).astype(np.float32)
    v = np.broadcast_to(np.eye(n, dtype=np.float32), (b, h, n, n)).copy()
    lens = np.array([n, 6], np.int32)
    for mask, r in ((MASK_NONE, None), (MASK_CAUSAL | MASK_PADDING, None), (MASK_PADDING, 4)):
        weights = o.sdpa(q, k, v, mask, lens, window=r)
        lse = o.lse(q, k, mask, lens, window=r)
        s = np.einsum("bhid,bhjd->bhij", q.astype(np.float64), k.astype(np.float64)) / np.sqrt(d)
        rebuilt = np.where(weights > 0, np.exp(s - lse[..., None]), 0.0)
        assert np.allclose(rebuilt, weights, rtol=1e-12, atol=1e-15), mask


PINS = [pin_worked_example, pin_worked_example_causal, pin_toy_rows, pin_scale_is_inverse_sqrt_dk,
        pin_rows_sum_to_one, pin_equal_scores_give_mean, pin_high_temperature_is_uniform,
        pin_shift_invariance, pin_causal_ignores_future, pin_padding_ignores_masked_keys,
        pin_permutation_equivariance, pin_brute_force, pin_rows_selection,
        pin_mha_single_head_identity, pin_mha_matches_matrix_form, pin_mha_concat_not_average,
        pin_mha_rows_selection, pin_restricted_worked_example, pin_restricted_extremes,
        pin_restricted_brute_force, pin_decode_matches_causal_rows, pin_decode_cache_lengths,
        pin_backward_finite_differences, pin_backward_closed_forms, pin_backward_given_output,
        pin_lse_closed_forms, pin_lse_rebuilds_softmax]
