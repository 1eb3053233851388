"""Wide heads, d_k = d_v in {256, 512} ("Attention Is All You Need", Table 3
rows (A): fewer, larger heads at a fixed model width), on the tensor cores
against the oracle, tolerance 2e-2 of the output scale; the log-sum-exp to
1e-3 absolute."""
import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_BF16, dev, dev_int, host, parity_err

pytestmark = pytest.mark.gpu


def _rand(rng, shape, std=1.0):
    return synthetic.round_to_bf16(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def _gpu(q, k, v, mask, lens, r=0, scale=0.0):
    t = __import__("torch")
    b, h, n_q, d = q.shape
    n_k = k.shape[2]
    out = t.full((b, h, n_q, d), 7.0, dtype=t.bfloat16, device="cuda")
    lse = t.zeros((b, h, n_q), dtype=t.float32, device="cuda")
    sd.sdpa_forward_lse(dev(q), dev(k), dev(v), out, lse, b, h, n_q, n_k, d, d, mask,
                        None if lens is None else dev_int(lens), r, scale)
    sd.sdpa_device_check()
    return host(out), lse.double().cpu().numpy()


def _check(q, k, v, mask, lens, r=0, scale=0.0):
    got, lse = _gpu(q, k, v, mask, lens, r, scale)
    window = r or None
    ref = oracle.sdpa(q, k, v, mask, lens, scale=scale, window=window)
    assert parity_err(got, ref) <= TOL_BF16
    ref_lse = oracle.lse(q, k, mask, lens, scale=scale, window=window)
    hidden = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), hidden)
    if (~hidden).any():
        assert np.abs(lse[~hidden] - ref_lse[~hidden]).max() <= 1e-3


@pytest.mark.parametrize("d", [256, 512])
@pytest.mark.parametrize("mask", [0, 1, 2, 3])
def test_wide_shapes(d, mask):
    rng = np.random.default_rng(11000 + d + mask)
    b, h, n = 2, 2, 300
    n_k = n if mask & 1 else 650
    q, k, v = _rand(rng, (b, h, n, d)), _rand(rng, (b, h, n_k, d)), _rand(rng, (b, h, n_k, d))
    lens = np.array([n_k, 133], np.int32) if mask & 2 else None
    _check(q, k, v, mask, lens)


@pytest.mark.parametrize("d", [256, 512])
@pytest.mark.parametrize("n", [1, 31, 33, 64, 65, 128, 129, 257])
def test_wide_ragged_causal(d, n):
    rng = np.random.default_rng(11100 + d + n)
    q, k, v = _rand(rng, (1, 2, n, d)), _rand(rng, (1, 2, n, d)), _rand(rng, (1, 2, n, d))
    _check(q, k, v, 1, None)


@pytest.mark.parametrize("d", [256, 512])
@pytest.mark.parametrize("n_k", [1, 63, 64, 65, 128, 191, 192, 193, 256, 320, 385, 448, 449, 512])
def test_wide_key_walk_lengths(d, n_k):
    """Key walks of 1 to 8 tiles of 64, whole and ragged, through the K and V
    stages (three of each at d = 256, the third in Q's shared memory; two of
    K and one of V at d = 512): cross-attention without a mask, then with
    key padding that ends the walk inside a tile."""
    rng = np.random.default_rng(11300 + d + n_k)
    b, h, n_q = 2, 1, 130
    q, k, v = _rand(rng, (b, h, n_q, d)), _rand(rng, (b, h, n_k, d)), _rand(rng, (b, h, n_k, d))
    _check(q, k, v, 0, None)
    _check(q, k, v, 2, np.array([n_k, max(0, n_k - 37)], np.int32))


@pytest.mark.parametrize("d", [256, 512])
@pytest.mark.parametrize("r", [1, 2, 63, 64, 200])
def test_wide_restricted(d, r):
    rng = np.random.default_rng(11200 + d + r)
    q, k, v = _rand(rng, (1, 2, 400, d)), _rand(rng, (1, 2, 400, d)), _rand(rng, (1, 2, 400, d))
    _check(q, k, v, 3, np.array([340], np.int32), r=r)


@pytest.mark.parametrize("d", [256, 512])
def test_wide_sharp_scores_and_scale(d):
    """Growing, sharp scores force O rescales; scale 1 is the unscaled form."""
    rng = np.random.default_rng(11300 + d)
    n = 500
    q = _rand(rng, (1, 2, n, d), 0.4)
    k = (_rand(rng, (1, 2, n, d)) * np.linspace(0.2, 2.0, n, dtype=np.float32)[None, None, :, None])
    k = synthetic.round_to_bf16(k.astype(np.float32))
    v = _rand(rng, (1, 2, n, d))
    _check(q, k, v, 1, None)
    _check(q, k, v, 0, None, scale=1.0 / d)


@pytest.mark.parametrize("d", [256, 512])
def test_wide_empty_keys_and_rows(d):
    """n_k = 0 writes zeros (lse -inf); a batch whose keys are all padded
    gives zero rows."""
    t = __import__("torch")
    rng = np.random.default_rng(11400 + d)
    q = _rand(rng, (1, 2, 40, d))
    kv = dev(np.ones((1, 2, 1, d), np.float32))
    out = t.full((1, 2, 40, d), 5.0, dtype=t.bfloat16, device="cuda")
    lse = t.zeros((1, 2, 40), dtype=t.float32, device="cuda")
    sd.sdpa_forward_lse(dev(q), kv, kv, out, lse, 1, 2, 40, 0, d, d)
    sd.sdpa_device_check()
    assert not out.any().item() and bool(t.isneginf(lse).all().item())
    q, k, v = _rand(rng, (2, 1, 70, d)), _rand(rng, (2, 1, 90, d)), _rand(rng, (2, 1, 90, d))
    lens = np.array([0, 90], np.int32)
    got, _ = _gpu(q, k, v, 2, lens)
    assert not got[0].any()
    _check(q, k, v, 2, lens)


def test_wide_long_causal():
    """Causal b1 h2 n2048 d256 (32 key tiles per query tile) in full."""
    rng = np.random.default_rng(11500)
    q, k, v = (_rand(rng, (1, 2, 2048, 256), 0.5) for _ in range(3))
    _check(q, k, v, 1, None)


def test_wide512_workload_full():
    """The one-head d = 512 workload at full size (b4 h1 n8192 causal, values
    0.5 N(0,1)), the benchmark's --workload wide512 launch: every output row
    under both measures and every row's log-sum-exp."""
    w = synthetic.WORKLOADS["wide_d512"]
    q, k, v, lens = synthetic.sdpa_inputs(w)
    _check(q, k, v, w.mask_kind, lens)


@pytest.mark.parametrize("h,d", [(1, 512), (2, 256)])
def test_table3_row_a_mha(h, d):
    """Multi-head attention at d_model = 512 with one head of 512 (Table 3,
    row (A)) and two heads of 256, key padding."""
    rng = np.random.default_rng(11600 + h)
    b, n, dm = 3, 200, 512
    xq = _rand(rng, (b, n, dm))
    wq, wk, wv = (synthetic.round_to_bf16((rng.standard_normal((dm, h * d)) / np.sqrt(dm))
                                          .astype(np.float32)) for _ in range(3))
    wo = synthetic.round_to_bf16((rng.standard_normal((h * d, dm)) / np.sqrt(h * d)).astype(np.float32))
    lens = np.array([200, 117, 5], np.int32)
    y = sd.multi_head_attention(dev(xq), dev(xq), dev(wq), dev(wk), dev(wv), dev(wo), h, 2,
                                dev_int(lens))
    sd.sdpa_device_check()
    ref = oracle.mha(xq, xq, wq, wk, wv, wo, h, d, d, 2, lens)
    assert parity_err(host(y), ref.reshape(b, n, dm)) <= TOL_BF16
