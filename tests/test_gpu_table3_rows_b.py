"""Smaller keys than values ("Attention Is All You Need", Table 3, rows (B):
d_k = 16 or 32 with d_v = 64, the rest as the base model) on the tensor
cores against the oracle, tolerance 2e-2 of the output scale."""
import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_BF16, dev, dev_int, host, parity_err

pytestmark = pytest.mark.gpu


def _rand(rng, shape, std=1.0):
    return synthetic.round_to_bf16(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


@pytest.mark.parametrize("d_k", [16, 32])
@pytest.mark.parametrize("mask,r", [(0, 0), (1, 0), (2, 0), (3, 0), (1, 77)])
def test_rows_b_attention(d_k, mask, r):
    rng = np.random.default_rng(15000 + d_k + 3 * mask + r)
    b, h, n, d_v = 2, 3, 300, 64
    n_k = n if (mask & 1) or r else 520
    q, k, v = _rand(rng, (b, h, n, d_k)), _rand(rng, (b, h, n_k, d_k)), _rand(rng, (b, h, n_k, d_v))
    lens = np.array([n_k, 150], np.int32) if mask & 2 else None
    lens_d = None if lens is None else dev_int(lens)
    out, lse = sd.attention_with_lse(dev(q), dev(k), dev(v), mask, lens_d, r)
    sd.sdpa_device_check()
    assert tuple(out.shape) == (b, h, n, d_v)
    window = r or None
    assert parity_err(host(out), oracle.sdpa(q, k, v, mask, lens, window=window)) <= TOL_BF16
    ref_lse = oracle.lse(q, k, mask, lens, window=window)
    got = lse.double().cpu().numpy()
    fin = ~np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(got), ~fin)
    assert np.abs(got[fin] - ref_lse[fin]).max() <= 1e-3


@pytest.mark.parametrize("d_k", [16, 32])
def test_rows_b_long_causal(d_k):
    rng = np.random.default_rng(15100 + d_k)
    q, k = _rand(rng, (1, 2, 2048, d_k)), _rand(rng, (1, 2, 2048, d_k))
    v = _rand(rng, (1, 2, 2048, 64))
    got = host(sd.attention(dev(q), dev(k), dev(v), sd.SDPA_MASK_CAUSAL))
    sd.sdpa_device_check()
    assert parity_err(got, oracle.sdpa(q, k, v, sd.SDPA_MASK_CAUSAL)) <= TOL_BF16


@pytest.mark.parametrize("d_k", [16, 32])
def test_rows_b_mha(d_k):
    """The rows' model: d_model 512, h = 8, d_v = 64, key padding."""
    rng = np.random.default_rng(15200 + d_k)
    b, n, dm, h, d_v = 3, 140, 512, 8, 64
    x = _rand(rng, (b, n, dm))
    wq, wk = (synthetic.round_to_bf16((rng.standard_normal((dm, h * d_k)) / np.sqrt(dm)).astype(np.float32))
              for _ in range(2))
    wv = synthetic.round_to_bf16((rng.standard_normal((dm, h * d_v)) / np.sqrt(dm)).astype(np.float32))
    wo = synthetic.round_to_bf16((rng.standard_normal((h * d_v, dm)) / np.sqrt(h * d_v)).astype(np.float32))
    lens = np.array([140, 99, 3], np.int32)
    y = sd.multi_head_attention(dev(x), dev(x), dev(wq), dev(wk), dev(wv), dev(wo), h,
                                sd.SDPA_MASK_PADDING, dev_int(lens))
    sd.sdpa_device_check()
    ref = oracle.mha(x, x, wq, wk, wv, wo, h, d_k, d_v, sd.SDPA_MASK_PADDING, lens)
    assert parity_err(host(y), ref) <= TOL_BF16
