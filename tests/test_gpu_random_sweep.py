"""A seeded random sweep over the entry points' argument space, against the
oracle under both measures of gpu_util (whole tensor and every row, 2e-2).

Each case draws batch and head counts, query and key lengths (ragged, often
not multiples of the tile sizes), a head shape of Table 3, a mask, sometimes
a restricted window, key-padding lengths (including 0 and lengths past n_k)
and a scale, so the library's own kernel and tile choices are exercised
away from the hand-picked shapes of the other tests."""
import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_BF16, dev, dev_int, host, parity_err

pytestmark = pytest.mark.gpu

HEADS = [(16, 16), (32, 32), (64, 64), (128, 128), (256, 256), (512, 512), (16, 64), (32, 64)]


def _rand(rng, shape, std=1.0):
    return synthetic.round_to_bf16(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def _case(seed):
    rng = np.random.default_rng(70000 + seed)
    d_k, d_v = HEADS[rng.integers(len(HEADS))]
    b = int(rng.integers(1, 4))
    h = int(rng.integers(1, 4))
    mask = int(rng.integers(0, 4))
    n_q = int(rng.integers(1, 700))
    n_k = n_q if mask & 1 else int(rng.integers(1, 900))
    window = int(rng.choice([0, 0, 1, 7, 100, 333])) if d_k == d_v else 0
    lens = None
    if mask & 2:
        lens = rng.integers(0, n_k + 40, size=b).astype(np.int32)
        lens[0] = n_k
    scale = float(rng.choice([0.0, 0.0, 1.0 / d_k, 0.3]))
    std = float(rng.choice([0.5, 1.0, 2.0]))
    q = _rand(rng, (b, h, n_q, d_k), std)
    k = _rand(rng, (b, h, n_k, d_k))
    v = _rand(rng, (b, h, n_k, d_v))
    return rng, (b, h, n_q, n_k, d_k, d_v, mask, window, lens, scale), (q, k, v)


@pytest.mark.parametrize("seed", range(40))
def test_forward_and_lse(seed):
    t = __import__("torch")
    _, (b, h, n_q, n_k, d_k, d_v, mask, window, lens, scale), (q, k, v) = _case(seed)
    out = t.full((b, h, n_q, d_v), 9.0, dtype=t.bfloat16, device="cuda")
    lse = t.zeros((b, h, n_q), dtype=t.float32, device="cuda")
    sd.sdpa_forward_lse(dev(q), dev(k), dev(v), out, lse, b, h, n_q, n_k, d_k, d_v, mask,
                        None if lens is None else dev_int(lens), window, scale)
    sd.sdpa_device_check()
    w = window or None
    ref = oracle.sdpa(q, k, v, mask, lens, scale=scale, window=w)
    assert parity_err(host(out), ref) <= TOL_BF16, (b, h, n_q, n_k, d_k, d_v, mask, window)
    ref_lse = oracle.lse(q, k, mask, lens, scale=scale, window=w)
    got_lse = lse.double().cpu().numpy()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse))
    fin = ~np.isneginf(ref_lse)
    if fin.any():
        assert np.abs(got_lse[fin] - ref_lse[fin]).max() <= 1e-3


@pytest.mark.parametrize("seed", range(24))
def test_backward(seed):
    rng, (b, h, n_q, n_k, d_k, d_v, mask, window, lens, scale), (q, k, v) = _case(seed)
    t = __import__("torch")
    do = _rand(rng, (b, h, n_q, d_v))
    w = window or None
    ref_out = oracle.sdpa(q, k, v, mask, lens, scale=scale, window=w)
    ref_lse = oracle.lse(q, k, mask, lens, scale=scale, window=w)
    out_in = synthetic.round_to_bf16(ref_out.astype(np.float32))
    lse_d = t.from_numpy(np.ascontiguousarray(ref_lse, dtype=np.float32)).cuda()
    lens_d = None if lens is None else dev_int(lens)
    dq, dk, dv = sd.attention_backward(dev(q), dev(k), dev(v), dev(out_in), lse_d, dev(do), mask,
                                       lens_d, window, scale)
    sd.sdpa_device_check()
    rq, rk, rv = oracle.backward(q, k, v, do, mask, lens, scale=scale, window=w, out=out_in)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert parity_err(host(g), r) <= TOL_BF16, (name, b, h, n_q, n_k, d_k, d_v, mask, window)


@pytest.mark.parametrize("seed", range(24))
def test_decode(seed):
    rng = np.random.default_rng(71000 + seed)
    d_k, d_v = HEADS[rng.integers(len(HEADS))]
    b, h = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    n_q = int(rng.integers(1, 9))
    n_k = int(rng.integers(1, 6000))
    lens = rng.integers(0, n_k + 50, size=b).astype(np.int32)
    scale = float(rng.choice([0.0, 1.0 / d_k]))
    q, k, v = _rand(rng, (b, h, n_q, d_k)), _rand(rng, (b, h, n_k, d_k)), _rand(rng, (b, h, n_k, d_v))
    got = sd.decode_step(dev(q), dev(k), dev(v), dev_int(lens), scale)
    sd.sdpa_device_check()
    assert parity_err(host(got), oracle.decode(q, k, v, lens, scale)) <= TOL_BF16, \
        (b, h, n_q, n_k, d_k, d_v)


@pytest.mark.parametrize("seed", range(12))
def test_multi_head(seed):
    rng = np.random.default_rng(72000 + seed)
    d_k, d_v = HEADS[rng.integers(len(HEADS))]
    h = int(rng.integers(1, 5))
    dm = int(rng.choice([64, 256, 520]))
    b = int(rng.integers(1, 4))
    mask = int(rng.integers(0, 4))
    n_q = int(rng.integers(1, 400))
    n_k = n_q if mask & 1 else int(rng.integers(1, 500))
    cross = n_k != n_q or bool(rng.integers(2))
    xq = _rand(rng, (b, n_q, dm))
    xkv = _rand(rng, (b, n_k, dm)) if cross else xq
    ws = [synthetic.round_to_bf16((rng.standard_normal(s) / np.sqrt(s[0])).astype(np.float32))
          for s in [(dm, h * d_k), (dm, h * d_k), (dm, h * d_v), (h * d_v, dm)]]
    lens = None
    if mask & 2:
        lens = rng.integers(0, n_k + 10, size=b).astype(np.int32)
    y = sd.multi_head_attention(dev(xq), dev(xkv), *[dev(a) for a in ws], h, mask,
                                None if lens is None else dev_int(lens))
    sd.sdpa_device_check()
    ref = oracle.mha(xq, xkv, *ws, h, d_k, d_v, mask, lens)
    assert parity_err(host(y), ref) <= TOL_BF16, (b, h, n_q, n_k, d_k, d_v, dm, mask)
