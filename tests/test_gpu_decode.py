"""One decoding step over a K/V cache (split across CTAs on the CUDA cores)
against the oracle, tolerance 2e-2 of the output scale."""
import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_BF16, dev, dev_int, host, parity_err

pytestmark = pytest.mark.gpu


def _rand(rng, shape, std=1.0):
    return synthetic.round_to_bf16(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def _gpu(q, k, v, lens=None, scale=0.0):
    out = sd.decode_step(dev(q), dev(k), dev(v), None if lens is None else dev_int(lens), scale)
    sd.sdpa_device_check()
    return host(out)


@pytest.mark.parametrize("d_k,d_v", [(16, 16), (32, 32), (64, 64), (128, 128), (256, 256),
                                     (512, 512), (16, 64), (32, 64)])
@pytest.mark.parametrize("n_q", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("b,h,n_k", [(1, 1, 1), (2, 3, 37), (4, 2, 1000), (1, 4, 5000)])
def test_decode_shapes(d_k, d_v, n_q, b, h, n_k):
    """Every head shape of Table 3 (rows (A), (B), (C)), one to eight new
    queries, caches of 1 to 5000 keys (one or many splits)."""
    rng = np.random.default_rng(9000 + d_k + 3 * d_v + 10 * n_q + n_k)
    q, k, v = _rand(rng, (b, h, n_q, d_k)), _rand(rng, (b, h, n_k, d_k)), _rand(rng, (b, h, n_k, d_v))
    lens = rng.integers(0, n_k + 1, size=b).astype(np.int32)
    lens[0] = n_k
    got = _gpu(q, k, v, lens)
    ref = oracle.decode(q, k, v, lens)
    assert parity_err(got, ref) <= TOL_BF16
    got_full = _gpu(q, k, v, None)
    assert parity_err(got_full, oracle.decode(q, k, v)) <= TOL_BF16


def test_decode_edge_lengths():
    """Cache lengths 0 (nothing visible), shorter than n_q (early queries see
    nothing), one, and beyond n_k (clamped)."""
    rng = np.random.default_rng(91)
    b, h, n_q, n_k, d = 5, 2, 4, 700, 128
    q, k, v = _rand(rng, (b, h, n_q, d)), _rand(rng, (b, h, n_k, d)), _rand(rng, (b, h, n_k, d))
    lens = np.array([0, 2, 1, 699, 5000], np.int32)
    got = _gpu(q, k, v, lens)
    ref = oracle.decode(q, k, v, lens)
    assert np.array_equal(got[0], np.zeros_like(got[0]))
    assert np.array_equal(got[1, :, :2], np.zeros_like(got[1, :, :2]))
    assert parity_err(got, ref) <= TOL_BF16


def test_decode_matches_causal_attention_rows():
    """The last n_q rows of causal self-attention equal a decoding step."""
    rng = np.random.default_rng(92)
    b, h, n, d, n_q = 2, 4, 640, 64, 3
    q, k, v = _rand(rng, (b, h, n, d)), _rand(rng, (b, h, n, d)), _rand(rng, (b, h, n, d))
    full = host(sd.attention(dev(q), dev(k), dev(v), sd.SDPA_MASK_CAUSAL))
    step = _gpu(q[:, :, n - n_q:], k, v)
    assert parity_err(step, full[:, :, n - n_q:]) <= TOL_BF16


def test_decode_unscaled_and_sharp():
    """scale 1 with large queries: peaked weights that move the running max
    from tile to tile."""
    rng = np.random.default_rng(95)
    b, h, n_q, n_k, d = 2, 2, 4, 3000, 64
    q = _rand(rng, (b, h, n_q, d), 0.4)
    k = synthetic.round_to_bf16(_rand(rng, (b, h, n_k, d)) *
                                np.linspace(0.2, 2.0, n_k, dtype=np.float32)[None, None, :, None])
    v = _rand(rng, (b, h, n_k, d))
    got = _gpu(q, k, v, None, 1.0)
    assert parity_err(got, oracle.decode(q, k, v, None, 1.0)) <= TOL_BF16


@pytest.mark.parametrize("n_q", [1, 4, 8])
def test_decode_workload(n_q):
    """Decoding step at serving size: 32 sequences, 16 heads, d=128, caches of
    8192 positions filled to lengths in [4096, 8192]."""
    rng = np.random.default_rng(93 + n_q)
    b, h, n_k, d = 32, 16, 8192, 128
    q, k, v = _rand(rng, (b, h, n_q, d)), _rand(rng, (b, h, n_k, d)), _rand(rng, (b, h, n_k, d))
    lens = rng.integers(4096, n_k + 1, size=b).astype(np.int32)
    got = _gpu(q, k, v, lens)
    ref = oracle.decode(q, k, v, lens)
    assert parity_err(got, ref) <= TOL_BF16
