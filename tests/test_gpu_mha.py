"""Multi-head attention with tensor-core projections against the oracle, and
the projection GEMM on its own against a float64 matrix product."""
import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_BF16, dev, dev_int, host, parity_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sd.load_library()


@pytest.mark.parametrize("m,n,k", [(128, 256, 64), (300, 520, 136), (4096, 1536, 512),
                                   (1, 8, 8), (257, 64, 1024)])
def test_linear(m, n, k):
    rng = np.random.default_rng(m + n + k)
    x = synthetic.round_to_bf16(rng.standard_normal((m, k)).astype(np.float32))
    w = synthetic.round_to_bf16((rng.standard_normal((k, n)) / np.sqrt(k)).astype(np.float32))
    t = __import__("torch")
    y = t.empty((m, n), dtype=t.bfloat16, device="cuda")
    sd.linear_forward(dev(x), dev(w), y, m, n, k)
    sd.sdpa_device_check()
    ref = x.astype(np.float64) @ w.astype(np.float64)
    assert parity_err(host(y), ref) <= 1e-2


@pytest.mark.parametrize("bn", ["256", "128"])
@pytest.mark.parametrize("m,n,k", [(300, 520, 136), (257, 64, 1024), (1000, 712, 200), (128, 256, 64),
                                   (4096, 512, 512)])
def test_linear_each_tile_width(bn, m, n, k):
    """The projection GEMM with its tile width pinned (sdpa_set_kernel_choice)
    to 256 and 128 columns: ragged edges in m, n and k for both widths."""
    rng = np.random.default_rng(7 * m + n + k)
    x = synthetic.round_to_bf16(rng.standard_normal((m, k)).astype(np.float32))
    w = synthetic.round_to_bf16((rng.standard_normal((k, n)) / np.sqrt(k)).astype(np.float32))
    t = __import__("torch")
    y = t.full((m, n), 3.0, dtype=t.bfloat16, device="cuda")
    with sd.kernel_choice(gemm_bn=int(bn)):
        sd.linear_forward(dev(x), dev(w), y, m, n, k)
    sd.sdpa_device_check()
    ref = x.astype(np.float64) @ w.astype(np.float64)
    assert parity_err(host(y), ref) <= 1e-2


def _mha_gpu(w, xq, xkv, wq, wk, wv, wo, lens):
    y = sd.multi_head_attention(dev(xq), dev(xkv), dev(wq), dev(wk), dev(wv), dev(wo), w.h,
                                w.mask_kind, None if lens is None else dev_int(lens))
    sd.sdpa_device_check()
    return host(y)


def test_encoder_mha_workload():
    """Base-model encoder self-attention with projections: X [32,128,512],
    h=8, d_k=d_v=64, key padding lengths 64..128; every output row."""
    w = synthetic.WORKLOADS["enc_mha_base"]
    xq, xkv, wq, wk, wv, wo, lens = synthetic.mha_inputs(w)
    got = _mha_gpu(w, xq, xkv, wq, wk, wv, wo, lens)
    ref = oracle.mha(xq, xkv, wq, wk, wv, wo, w.h, w.d_k, w.d_v, w.mask_kind, lens)
    assert parity_err(got, ref) <= TOL_BF16


def test_cross_mha_workload():
    """Big-model cross-attention with projections: X_dec [32,256,1024],
    X_enc [32,384,1024], h=16, d_k=d_v=64, key padding 192..384; every
    output row."""
    w = synthetic.WORKLOADS["cross_big"]
    xq, xkv, wq, wk, wv, wo, lens = synthetic.mha_inputs(w)
    got = _mha_gpu(w, xq, xkv, wq, wk, wv, wo, lens)
    ref = oracle.mha(xq, xkv, wq, wk, wv, wo, w.h, w.d_k, w.d_v, w.mask_kind, lens)
    assert parity_err(got, ref) <= TOL_BF16


@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_mha_ragged_causal(d):
    rng = np.random.default_rng(22 + d)
    b, n, dm, h = 2, 300, 256, 2
    x = synthetic.round_to_bf16(rng.standard_normal((b, n, dm)).astype(np.float32))
    ws = [synthetic.round_to_bf16((rng.standard_normal(s) / np.sqrt(s[0])).astype(np.float32))
          for s in [(dm, h * d)] * 3 + [(h * d, dm)]]
    y = sd.multi_head_attention(dev(x), dev(x), *[dev(a) for a in ws], h, sd.SDPA_MASK_CAUSAL)
    sd.sdpa_device_check()
    ref = oracle.mha(x, x, *ws, h, d, d, sd.SDPA_MASK_CAUSAL)
    assert parity_err(host(y), ref) <= TOL_BF16


@pytest.mark.parametrize("h,d_k,d_v", [(1, 512, 512), (2, 256, 256), (4, 128, 128), (16, 32, 32),
                                       (32, 16, 16), (8, 16, 64), (8, 32, 64)])
@pytest.mark.parametrize("mask", [1, 2])
def test_mha_table3_heads(h, d_k, d_v, mask):
    """Multi-head attention at d_model 512 with Table 3's head shapes (rows
    (A) and (B), and two heads of 256): causal self-attention, and
    cross-attention with key padding, ragged lengths."""
    rng = np.random.default_rng(23 + h + d_k + 7 * d_v + mask)
    b, dm = 2, 512
    n_q = 300
    n_k = n_q if mask & 1 else 170
    xq = synthetic.round_to_bf16(rng.standard_normal((b, n_q, dm)).astype(np.float32))
    xkv = xq if mask & 1 else synthetic.round_to_bf16(
        rng.standard_normal((b, n_k, dm)).astype(np.float32))
    ws = [synthetic.round_to_bf16((rng.standard_normal(s) / np.sqrt(s[0])).astype(np.float32))
          for s in [(dm, h * d_k), (dm, h * d_k), (dm, h * d_v), (h * d_v, dm)]]
    lens = np.array([n_k, 97], np.int32) if mask & 2 else None
    y = sd.multi_head_attention(dev(xq), dev(xkv), *[dev(a) for a in ws], h, mask,
                                None if lens is None else dev_int(lens))
    sd.sdpa_device_check()
    ref = oracle.mha(xq, xkv, *ws, h, d_k, d_v, mask, lens)
    assert parity_err(host(y), ref) <= TOL_BF16
