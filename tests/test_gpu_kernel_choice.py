"""Both tensor-core attention kernels at head sizes 16, 32, 64 and 128, each pinned
with sdpa_set_kernel_choice, against the oracle (2e-2 of the output scale,
whole tensor and every row):
the two-tile kernel (two 128-row query tiles per CTA, 128-key tiles) and the
one-tile kernel (one query tile per CTA; 64-key tiles and two CTAs per SM at
d = 64, 128; 32-key tiles and four CTAs per SM at d = 16, 32, and at d = 64
for short walks over many CTAs).
The library picks between them by shape; these tests keep both covered on
the same shapes, masks, windows and ragged tails."""
import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_BF16, dev, dev_int, host, parity_err

pytestmark = pytest.mark.gpu


def _rand(rng, shape, std=1.0):
    return synthetic.round_to_bf16(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


@pytest.mark.parametrize("kernel", ["two_tile", "one_tile"])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("mask,r", [(0, 0), (1, 0), (2, 0), (3, 0), (1, 100), (0, 257)])
def test_kernel_parity(kernel, d, mask, r):
    rng = np.random.default_rng(13000 + d + 7 * mask + r)
    b, h, n = 2, 3, 300
    n_k = n if (mask & 1) or r else 650
    q, k, v = _rand(rng, (b, h, n, d)), _rand(rng, (b, h, n_k, d)), _rand(rng, (b, h, n_k, d))
    lens = np.array([n_k, 201], np.int32) if mask & 2 else None
    lens_d = None if lens is None else dev_int(lens)
    t = __import__("torch")
    out = t.full((b, h, n, d), 9.0, dtype=t.bfloat16, device="cuda")
    lse = t.zeros((b, h, n), dtype=t.float32, device="cuda")
    with sd.kernel_choice(attention=kernel):
        sd.sdpa_forward_lse(dev(q), dev(k), dev(v), out, lse, b, h, n, n_k, d, d, mask, lens_d, r)
    sd.sdpa_device_check()
    window = r or None
    assert parity_err(host(out), oracle.sdpa(q, k, v, mask, lens, window=window)) <= TOL_BF16
    ref_lse = oracle.lse(q, k, mask, lens, window=window)
    got_lse = lse.double().cpu().numpy()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse))
    fin = ~np.isneginf(ref_lse)
    assert np.abs(got_lse[fin] - ref_lse[fin]).max() <= 1e-3


@pytest.mark.parametrize("keys", [32, 64])
@pytest.mark.parametrize("mask,r", [(0, 0), (1, 0), (2, 0), (3, 0), (1, 100), (0, 257), (3, 64)])
def test_one_tile_d64_key_tiles(keys, mask, r):
    """The one-tile kernel at d = 64 with each key tile (32: four CTAs per SM;
    64: two), pinned with sdpa_set_kernel_choice, against the oracle."""
    rng = np.random.default_rng(13300 + keys + 7 * mask + r)
    b, h, n, d = 2, 3, 333, 64
    n_k = n if (mask & 1) or r else 650
    q, k, v = _rand(rng, (b, h, n, d)), _rand(rng, (b, h, n_k, d)), _rand(rng, (b, h, n_k, d))
    lens = np.array([n_k, 95], np.int32) if mask & 2 else None
    lens_d = None if lens is None else dev_int(lens)
    t = __import__("torch")
    out = t.full((b, h, n, d), 9.0, dtype=t.bfloat16, device="cuda")
    lse = t.zeros((b, h, n), dtype=t.float32, device="cuda")
    with sd.kernel_choice(attention="one_tile", one_tile_keys=keys):
        sd.sdpa_forward_lse(dev(q), dev(k), dev(v), out, lse, b, h, n, n_k, d, d, mask, lens_d, r)
    sd.sdpa_device_check()
    window = r or None
    assert parity_err(host(out), oracle.sdpa(q, k, v, mask, lens, window=window)) <= TOL_BF16
    ref_lse = oracle.lse(q, k, mask, lens, window=window)
    got_lse = lse.double().cpu().numpy()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse))
    fin = ~np.isneginf(ref_lse)
    assert np.abs(got_lse[fin] - ref_lse[fin]).max() <= 1e-3


@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_both_kernels_on_long_causal(d):
    """b1 h2 n2048 causal, 16 key tiles of 128 per query tile at the end:
    each kernel against the oracle, every row under both measures, and every
    row's log-sum-exp to 1e-3."""
    t = __import__("torch")
    rng = np.random.default_rng(13100 + d)
    b, h, n = 1, 2, 2048
    q, k, v = (_rand(rng, (b, h, n, d), 0.5) for _ in range(3))
    ref = oracle.sdpa(q, k, v, sd.SDPA_MASK_CAUSAL)
    ref_lse = oracle.lse(q, k, sd.SDPA_MASK_CAUSAL)
    for kernel in ("two_tile", "one_tile"):
        out = t.empty((b, h, n, d), dtype=t.bfloat16, device="cuda")
        lse = t.empty((b, h, n), dtype=t.float32, device="cuda")
        with sd.kernel_choice(attention=kernel):
            sd.sdpa_forward_lse(dev(q), dev(k), dev(v), out, lse, b, h, n, n, d, d,
                                sd.SDPA_MASK_CAUSAL)
        sd.sdpa_device_check()
        assert parity_err(host(out), ref) <= TOL_BF16, kernel
        assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 1e-3, kernel


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("n", [3072, 3200])
def test_default_choice_either_side_of_the_crossover(d, n):
    """Unpinned: a 3072-key walk runs on the one-tile kernel and a 3200-key
    walk on the two-tile kernel; both against the oracle, causal with padding,
    the log-sum-exp of every row to 1e-3."""
    sd.sdpa_set_kernel_choice(0, 0, 0)
    rng = np.random.default_rng(13200 + d + n)
    b, h = 2, 1
    q, k, v = (_rand(rng, (b, h, n, d), 0.5) for _ in range(3))
    lens = np.array([n, n - 77], np.int32)
    mask = sd.SDPA_MASK_CAUSAL | sd.SDPA_MASK_PADDING
    t = __import__("torch")
    out = t.empty((b, h, n, d), dtype=t.bfloat16, device="cuda")
    lse = t.empty((b, h, n), dtype=t.float32, device="cuda")
    sd.sdpa_forward_lse(dev(q), dev(k), dev(v), out, lse, b, h, n, n, d, d, mask, dev_int(lens))
    sd.sdpa_device_check()
    assert parity_err(host(out), oracle.sdpa(q, k, v, mask, lens)) <= TOL_BF16
    assert np.abs(lse.double().cpu().numpy() - oracle.lse(q, k, mask, lens)).max() <= 1e-3
