"""Gradients of attention (training by back-propagation through Eq. (1)) on
the tensor cores against the oracle's fp64 gradients.

Each case runs three comparisons:
  1. The forward that feeds the backward: its output under both measures of
     gpu_util (whole tensor and every row, 2e-2), its per-row log-sum-exp to
     1e-3 absolute (a log of a sum of fp32 exponentials of exact bf16
     products).
  2. The backward on its own.  It is handed the oracle's output rounded to
     bf16 and the oracle's log-sum-exp in fp32, and compared with the
     oracle's gradients for that same output (the output enters only through
     D_i = dO_i . O_i).  Every row of dQ and every key row of dK and dV is held
     to 2e-2 of its own scale, and each tensor to 2e-2 of its scale.  The
     arithmetic behind that bar: P and dS enter the tensor cores rounded to
     bf16 (relative 2^-9 each), the results are rounded to bf16 once, and all
     accumulation is fp32.
  3. The backward chained from the GPU forward, against the exact gradients,
     whole tensor only.  Here D_i uses the forward's bf16 output while the
     exact gradients use the exact one; a row whose dS nearly cancels (a short
     causal or windowed row) then carries that rounding, relative to D_i, in a
     row that is small, so only the whole-tensor bar applies to this chain.
"""
import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_BF16, dev, dev_int, host, parity_err, rel_err

pytestmark = pytest.mark.gpu

LSE_TOL = 1e-3


def _rand(rng, shape, std=1.0):
    return synthetic.round_to_bf16(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def _inputs(seed, b, h, n_q, n_k, d, std=1.0):
    rng = np.random.default_rng(seed)
    return (_rand(rng, (b, h, n_q, d), std), _rand(rng, (b, h, n_k, d)), _rand(rng, (b, h, n_k, d)),
            _rand(rng, (b, h, n_q, d)))


def _gpu_forward_backward(q, k, v, do, mask, lens, r=0, scale=0.0):
    lens_d = None if lens is None else dev_int(lens)
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    out, lse = sd.attention_with_lse(qd, kd, vd, mask, lens_d, r, scale)
    dq, dk, dv = sd.attention_backward(qd, kd, vd, out, lse, dod, mask, lens_d, r, scale)
    sd.sdpa_device_check()
    return host(out), lse.double().cpu().numpy(), host(dq), host(dk), host(dv)


def _gpu_backward_given(q, k, v, do, out, lse, mask, lens, r=0, scale=0.0):
    """The backward alone, handed out (bf16 values) and lse (fp32) from the caller."""
    t = __import__("torch")
    lens_d = None if lens is None else dev_int(lens)
    lse_d = t.from_numpy(np.ascontiguousarray(lse, dtype=np.float32)).cuda()
    dq, dk, dv = sd.attention_backward(dev(q), dev(k), dev(v), dev(out), lse_d, dev(do), mask,
                                       lens_d, r, scale)
    sd.sdpa_device_check()
    return host(dq), host(dk), host(dv)


def _check(q, k, v, do, mask, lens, r=0, scale=0.0):
    out, lse, dq, dk, dv = _gpu_forward_backward(q, k, v, do, mask, lens, r, scale)
    window = r or None
    ref_out = oracle.sdpa(q, k, v, mask, lens, scale=scale, window=window)
    ref_lse = oracle.lse(q, k, mask, lens, scale=scale, window=window)
    assert parity_err(out, ref_out) <= TOL_BF16
    hidden = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), hidden)
    if (~hidden).any():
        assert np.abs(lse[~hidden] - ref_lse[~hidden]).max() <= LSE_TOL

    # 2. the backward alone, on the oracle's output and log-sum-exp
    out_in = synthetic.round_to_bf16(ref_out.astype(np.float32))
    gq, gk, gv = _gpu_backward_given(q, k, v, do, out_in, ref_lse, mask, lens, r, scale)
    rq, rk, rv = oracle.backward(q, k, v, do, mask, lens, scale=scale, window=window, out=out_in)
    errs = {"dq": parity_err(gq, rq), "dk": parity_err(gk, rk), "dv": parity_err(gv, rv)}
    assert max(errs.values()) <= TOL_BF16, errs

    # 3. chained from the GPU forward, against the exact gradients
    eq, ek, ev = oracle.backward(q, k, v, do, mask, lens, scale=scale, window=window)
    chained = {"dq": rel_err(dq, eq), "dk": rel_err(dk, ek), "dv": rel_err(dv, ev)}
    assert max(chained.values()) <= TOL_BF16, chained
    return errs


@pytest.mark.parametrize("d", [16, 32, 64, 128, 256, 512])
@pytest.mark.parametrize("mask", [0, 1, 2, 3])
def test_backward_shapes(d, mask):
    b, h, n = 2, 3, 300
    n_k = n if mask & 1 else 650
    q, k, v, do = _inputs(9000 + d + mask, b, h, n, n_k, d)
    lens = np.array([n_k, 171], np.int32) if mask & 2 else None
    _check(q, k, v, do, mask, lens)


@pytest.mark.parametrize("d", [128, 256, 512])
@pytest.mark.parametrize("n", [1, 17, 63, 64, 65, 127, 128, 129, 256, 383])
def test_backward_ragged_lengths(d, n):
    q, k, v, do = _inputs(9100 + n + d, 1, 2, n, n, d)
    _check(q, k, v, do, 1, None)


@pytest.mark.parametrize("r", [1, 2, 64, 127, 129, 300])
@pytest.mark.parametrize("mask", [0, 1, 3])
def test_backward_restricted(r, mask):
    b, h, n = 2, 2, 520
    q, k, v, do = _inputs(9200 + r + mask, b, h, n, n, 64)
    lens = np.array([n, 290], np.int32) if mask & 2 else None
    _check(q, k, v, do, mask, lens, r=r)


def test_backward_unscaled_and_sharp():
    """scale 1 (the unscaled dot-product attention of section 3.2.1) with
    larger queries: peaked softmax rows."""
    q, k, v, do = _inputs(9300, 1, 2, 256, 256, 64, std=0.25)
    _check(q, k, v, do, 0, None, scale=1.0)
    q, k, v, do = _inputs(9301, 1, 2, 256, 256, 128, std=3.0)
    _check(q, k, v, do, 1, None)


def test_backward_empty_rows_and_sequences():
    """A batch whose every key is hidden gives zero gradients (and lse
    -inf); n_q = 0 gives dK = dV = 0; n_k = 0 gives dQ = 0."""
    q, k, v, do = _inputs(9400, 2, 2, 200, 200, 64)
    lens = np.array([0, 77], np.int32)
    out, lse, dq, dk, dv = _gpu_forward_backward(q, k, v, do, 2, lens)
    assert np.all(np.isneginf(lse[0])) and not np.isneginf(lse[1]).any()
    assert not dq[0].any() and not dk[0].any() and not dv[0].any()
    assert not dk[1, :, 77:].any() and not dv[1, :, 77:].any()
    _check(q, k, v, do, 2, lens)

    # n_q = 0 and n_k = 0 with valid one-row buffers the sizes leave unread
    t = __import__("torch")
    d = 64
    one = dev(np.ones((1, 2, 1, d), np.float32))
    lse1 = t.zeros((1, 2, 1), dtype=t.float32, device="cuda")
    kd = dev(_rand(np.random.default_rng(1), (1, 2, 50, d)))
    vd = dev(_rand(np.random.default_rng(2), (1, 2, 50, d)))
    dk = t.full((1, 2, 50, d), 5.0, dtype=t.bfloat16, device="cuda")
    dv = t.full((1, 2, 50, d), 5.0, dtype=t.bfloat16, device="cuda")
    ws = t.empty(max(16, sd.sdpa_backward_workspace_size(1, 2, 0, d)), dtype=t.uint8, device="cuda")
    sd.sdpa_backward(one, kd, vd, one, one, lse1, one.clone(), dk, dv, ws, ws.numel(), 1, 2, 0, 50,
                     d, d)
    sd.sdpa_device_check()
    assert not dk.any().item() and not dv.any().item()

    qd = dev(_rand(np.random.default_rng(3), (1, 2, 40, d)))
    dod = dev(_rand(np.random.default_rng(4), (1, 2, 40, d)))
    out = t.full((1, 2, 40, d), 5.0, dtype=t.bfloat16, device="cuda")
    lse = t.zeros((1, 2, 40), dtype=t.float32, device="cuda")
    sd.sdpa_forward_lse(qd, one, one, out, lse, 1, 2, 40, 0, d, d)
    dq = t.full((1, 2, 40, d), 5.0, dtype=t.bfloat16, device="cuda")
    ws = t.empty(sd.sdpa_backward_workspace_size(1, 2, 40, d), dtype=t.uint8, device="cuda")
    sd.sdpa_backward(qd, one, one, out, dod, lse, dq, one.clone(), one.clone(), ws, ws.numel(), 1,
                     2, 40, 0, d, d)
    sd.sdpa_device_check()
    assert not out.any().item() and not dq.any().item()
    assert bool(t.isneginf(lse).all().item())


def test_backward_matches_across_calls_and_reuses_workspace():
    """Two calls on one workspace give the same gradients (the fp32 dQ
    accumulator is cleared by each call); the order of the floating-point
    reductions may differ, so equality is to 1e-6 of the scale."""
    q, k, v, do = _inputs(9500, 2, 4, 384, 384, 128)
    t = __import__("torch")
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    out, lse = sd.attention_with_lse(qd, kd, vd, 1)
    ws = t.empty(sd.sdpa_backward_workspace_size(2, 4, 384, 128), dtype=t.uint8, device="cuda")
    a = sd.attention_backward(qd, kd, vd, out, lse, dod, 1, workspace=ws)
    b = sd.attention_backward(qd, kd, vd, out, lse, dod, 1, workspace=ws)
    sd.sdpa_device_check()
    for x, y in zip(a, b):
        assert rel_err(host(x), host(y)) <= 1e-2 * TOL_BF16


def test_backward_workload_length():
    """The backward workload's full sequence (causal n8192 d128, values
    0.5 N(0,1), as bench.py --workload backward) on two of its heads: up to
    128 query steps per key tile, every row of every gradient."""
    w = synthetic.WORKLOADS["long_causal"]
    q, k, v, _ = synthetic.sdpa_inputs(w, b=1, h=2)
    do = synthetic.dout_input(w, b=1, h=2)
    _check(q, k, v, do, w.mask_kind, None)


def test_backward_long_causal():
    """Causal b1 h4 n4096 d128 (up to 32 key tiles per query tile): every
    row of every gradient checked against the oracle."""
    q, k, v, do = _inputs(9600, 1, 4, 4096, 4096, 128)
    errs = _check(q, k, v, do, 1, None)
    assert max(errs.values()) <= TOL_BF16


@pytest.mark.parametrize("r", [1, 64, 129, 300])
@pytest.mark.parametrize("mask", [0, 1, 3])
def test_backward_wide_head_restricted(r, mask):
    """Table 3, row (A): two heads of 256 at d_model 512 (dK, dV, dQ in two
    128-column chunks, one CTA each), with the restricted window."""
    b, h, n = 2, 2, 520
    q, k, v, do = _inputs(9250 + r + mask, b, h, n, n, 256)
    lens = np.array([n, 290], np.int32) if mask & 2 else None
    _check(q, k, v, do, mask, lens, r=r)


def test_backward_wide_head_long_causal():
    """d = 256, causal n = 2048 (16 key tiles, up to 32 query steps each)."""
    q, k, v, do = _inputs(9650, 1, 2, 2048, 2048, 256, std=0.5)
    _check(q, k, v, do, 1, None)


@pytest.mark.parametrize("r", [1, 64, 129, 300])
@pytest.mark.parametrize("mask", [0, 1, 3])
def test_backward_head512_restricted(r, mask):
    """Table 3, row (A): one head of 512 (64-key tiles, two CTAs per key
    tile for the two halves of d, 32-query steps), with the restricted window."""
    b, h, n = 2, 1, 520
    q, k, v, do = _inputs(9270 + r + mask, b, h, n, n, 512)
    lens = np.array([n, 290], np.int32) if mask & 2 else None
    _check(q, k, v, do, mask, lens, r=r)


def test_backward_head512_empty_rows():
    """d = 512: a batch whose every key is hidden gets zero gradients, and
    keys past a length get zero dK and dV."""
    q, k, v, do = _inputs(9280, 2, 1, 200, 200, 512)
    lens = np.array([0, 77], np.int32)
    out, lse, dq, dk, dv = _gpu_forward_backward(q, k, v, do, 2, lens)
    assert np.all(np.isneginf(lse[0])) and not np.isneginf(lse[1]).any()
    assert not dq[0].any() and not dk[0].any() and not dv[0].any()
    assert not dk[1, :, 77:].any() and not dv[1, :, 77:].any()
    _check(q, k, v, do, 2, lens)


def test_backward_head512_workload_length():
    """The 512-wide workload's full sequence (causal n8192 d512, values
    0.5 N(0,1), as bench.py --workload wide512) on one of its batch entries:
    128 key tiles with up to 256 query steps each, every row of every
    gradient."""
    w = synthetic.WORKLOADS["wide_d512"]
    q, k, v, _ = synthetic.sdpa_inputs(w, b=1, h=1)
    do = synthetic.dout_input(w, b=1, h=1)
    _check(q, k, v, do, w.mask_kind, None)


@pytest.mark.parametrize("d", [16, 32])
@pytest.mark.parametrize("n", [1, 65, 300])
def test_backward_small_heads(d, n):
    """Table 3's small heads: causal, padding and a window."""
    q, k, v, do = _inputs(9700 + d + n, 2, 3, n, n, d)
    _check(q, k, v, do, 1, None)
    _check(q, k, v, do, 2, np.array([n, max(1, n // 3)], np.int32))
    _check(q, k, v, do, 1, None, r=33)


@pytest.mark.parametrize("d_k", [16, 32])
@pytest.mark.parametrize("mask,n_q,n_k,r", [(0, 70, 200, 0), (1, 300, 300, 0), (2, 129, 257, 0),
                                            (3, 300, 300, 0), (1, 260, 260, 65)])
def test_backward_row_b_heads(d_k, mask, n_q, n_k, r):
    """Table 3, rows (B): keys of 16 or 32 against values of 64; dq and dk
    have d_k columns, dv has d_v."""
    rng = np.random.default_rng(9800 + d_k + 7 * mask + r)
    b, h, d_v = 2, 3, 64
    q, k = _rand(rng, (b, h, n_q, d_k)), _rand(rng, (b, h, n_k, d_k))
    v, do = _rand(rng, (b, h, n_k, d_v)), _rand(rng, (b, h, n_q, d_v))
    lens = np.array([n_k, max(1, n_k // 3)], np.int32) if mask & 2 else None
    errs = _check(q, k, v, do, mask, lens, r)
    assert set(errs) == {"dq", "dk", "dv"}


def test_backward_row_b_unscaled():
    """Scale 1 (the unscaled dot product of the paper's comparison) at d_k = 16, d_v = 64."""
    rng = np.random.default_rng(9850)
    q, k = _rand(rng, (1, 2, 200, 16), 0.3), _rand(rng, (1, 2, 200, 16))
    v, do = _rand(rng, (1, 2, 200, 64)), _rand(rng, (1, 2, 200, 64))
    _check(q, k, v, do, 1, None, scale=1.0)


def test_backward_rejects_bad_arguments():
    t = __import__("torch")
    x = t.zeros((1, 1, 64, 64), dtype=t.bfloat16, device="cuda")
    lse = t.zeros((1, 1, 64), dtype=t.float32, device="cuda")
    ws = t.empty(sd.sdpa_backward_workspace_size(1, 1, 64, 64), dtype=t.uint8, device="cuda")
    with pytest.raises(sd.SdpaError, match="WORKSPACE"):
        sd.sdpa_backward(x, x, x, x, x, lse, x, x, x, ws, ws.numel() - 16, 1, 1, 64, 64, 64, 64)
    # a head size outside Table 3
    x96 = t.zeros((1, 1, 64, 96), dtype=t.bfloat16, device="cuda")
    with pytest.raises(sd.SdpaError, match="UNSUPPORTED"):
        sd.sdpa_backward(x96, x96, x96, x96, x96, lse, x96, x96, x96, ws, ws.numel(), 1, 1,
                         64, 64, 96, 96)
    # 512-wide heads need the larger dQ accumulator
    x512 = t.zeros((1, 1, 64, 512), dtype=t.bfloat16, device="cuda")
    with pytest.raises(sd.SdpaError, match="WORKSPACE"):
        sd.sdpa_backward(x512, x512, x512, x512, x512, lse, x512, x512, x512, ws, ws.numel(), 1, 1,
                         64, 64, 512, 512)
    with pytest.raises(sd.SdpaError, match="INVALID_ARG"):
        sd.sdpa_backward(x, x, x, x, None, lse, x, x, x, ws, ws.numel(), 1, 1, 64, 64, 64, 64)
    # unequal head sizes other than Table 3's rows (B)
    x32 = t.zeros((1, 1, 64, 32), dtype=t.bfloat16, device="cuda")
    with pytest.raises(sd.SdpaError, match="UNSUPPORTED"):
        sd.sdpa_backward(x, x, x32, x32, x32, lse, x, x, x32, ws, ws.numel(), 1, 1, 64, 64, 64, 32)
