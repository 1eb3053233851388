"""Restricted self-attention (a neighbourhood of size r around each position)
on the tensor cores against the oracle, tolerance 2e-2 of the output scale."""
import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_BF16, dev, dev_int, host, parity_err

pytestmark = pytest.mark.gpu


def _rand(rng, shape, std=1.0):
    return synthetic.round_to_bf16(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def _gpu(q, k, v, mask, lens, r, scale=0.0):
    t = __import__("torch")
    b, h, n_q, d = q.shape
    n_k = k.shape[2]
    out = t.empty((b, h, n_q, d), dtype=t.bfloat16, device="cuda")
    sd.sdpa_forward_restricted(dev(q), dev(k), dev(v), out, b, h, n_q, n_k, d, d, mask,
                               None if lens is None else dev_int(lens), r, scale)
    sd.sdpa_device_check()
    return host(out)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("mask", [0, 1, 2, 3])
@pytest.mark.parametrize("r", [1, 2, 3, 64, 127, 128, 129, 300, 5000])
def test_restricted_shapes(d, mask, r):
    rng = np.random.default_rng(7000 + d + 10 * mask + r)
    b, h, n = 2, 2, 700
    n_k = n if mask & 1 else 650
    q, k, v = _rand(rng, (b, h, n, d)), _rand(rng, (b, h, n_k, d)), _rand(rng, (b, h, n_k, d))
    lens = np.array([n_k, 333], np.int32) if mask & 2 else None
    got = _gpu(q, k, v, mask, lens, r)
    ref = oracle.sdpa(q, k, v, mask, lens, window=r)
    assert parity_err(got, ref) <= TOL_BF16


def test_restricted_one_is_identity():
    rng = np.random.default_rng(71)
    q, k, v = _rand(rng, (1, 3, 300, 64)), _rand(rng, (1, 3, 300, 64)), _rand(rng, (1, 3, 300, 64))
    got = _gpu(q, k, v, 0, None, 1)
    assert np.array_equal(got, v.astype(np.float64))


def test_restricted_wide_equals_full():
    rng = np.random.default_rng(72)
    q, k, v = _rand(rng, (2, 2, 500, 128)), _rand(rng, (2, 2, 500, 128)), _rand(rng, (2, 2, 500, 128))
    wide = _gpu(q, k, v, 1, None, 2000)
    full = host(sd.attention(dev(q), dev(k), dev(v), 1))
    assert np.array_equal(wide, full)


def test_restricted_long_sequence():
    """Long causal sequence with a 1024-position neighbourhood (b2 h8
    n8192 d128): every output row under both measures, and every row's
    log-sum-exp to 1e-3."""
    t = __import__("torch")
    rng = np.random.default_rng(73)
    b, h, n, d, r = 2, 8, 8192, 128, 1024
    q, k, v = _rand(rng, (b, h, n, d), 0.5), _rand(rng, (b, h, n, d), 0.5), _rand(rng, (b, h, n, d), 0.5)
    got = _gpu(q, k, v, 1, None, r)
    assert parity_err(got, oracle.sdpa(q, k, v, 1, None, window=r)) <= TOL_BF16
    out = t.empty((b, h, n, d), dtype=t.bfloat16, device="cuda")
    lse = t.empty((b, h, n), dtype=t.float32, device="cuda")
    sd.sdpa_forward_lse(dev(q), dev(k), dev(v), out, lse, b, h, n, n, d, d, 1, None, r)
    sd.sdpa_device_check()
    assert np.array_equal(host(out), got)
    ref_lse = oracle.lse(q, k, 1, None, window=r)
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 1e-3
