"""sdpa_forward_host (through attention_from_host): pinned host inputs,
chunked copies overlapped with the attention calls on the library's three
streams.  Each (batch, head) is computed by the
same kernel as one device-side call, so the result must match it exactly,
and the oracle within the bf16 bar."""
import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_BF16, dev, dev_int, host, parity_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,mask,hc", [(64, 3, 4), (128, 1, 8), (128, 0, 3), (256, 2, 2)])
def test_attention_from_host(d, mask, hc):
    t = __import__("torch")
    rng = np.random.default_rng(12000 + d + mask + hc)
    b, h, n = 2, 6, 300
    q, k, v = (synthetic.round_to_bf16(rng.standard_normal((b, h, n, d)).astype(np.float32))
               for _ in range(3))
    lens = np.array([300, 120], np.int32) if mask & 2 else None
    lens_d = None if lens is None else dev_int(lens)
    qh, kh, vh = (t.from_numpy(x).to(t.bfloat16).pin_memory() for x in (q, k, v))
    oh = t.full((b, h, n, d), 3.0, dtype=t.bfloat16).pin_memory()
    qd, kd, vd = (t.empty_like(x, device="cuda") for x in (qh, kh, vh))
    od = t.empty((b, h, n, d), dtype=t.bfloat16, device="cuda")
    sd.attention_from_host(qh, kh, vh, oh, qd, kd, vd, od, mask, lens_d, heads_per_chunk=hc)
    t.cuda.current_stream().synchronize()
    sd.sdpa_device_check()
    whole = sd.attention(dev(q), dev(k), dev(v), mask, lens_d)
    sd.sdpa_device_check()
    got = oh.float().numpy().astype(np.float64)
    assert np.array_equal(got, host(whole))
    assert parity_err(got, oracle.sdpa(q, k, v, mask, lens)) <= TOL_BF16


def test_host_pipeline_pageable_and_repeated():
    """Pageable host buffers also work (each copy then blocks the host), and
    two calls in a row on one device reuse the library's streams and events."""
    t = __import__("torch")
    rng = np.random.default_rng(12100)
    b, h, n, d = 3, 4, 200, 64
    q, k, v = (synthetic.round_to_bf16(rng.standard_normal((b, h, n, d)).astype(np.float32))
               for _ in range(3))
    qd, kd, vd, od = (t.empty((b, h, n, d), dtype=t.bfloat16, device="cuda") for _ in range(4))
    ref = oracle.sdpa(q, k, v, sd.SDPA_MASK_CAUSAL)
    for pinned in (False, True):
        qh, kh, vh = (t.from_numpy(x).to(t.bfloat16) for x in (q, k, v))
        oh = t.zeros((b, h, n, d), dtype=t.bfloat16)
        if pinned:
            qh, kh, vh, oh = (x.pin_memory() for x in (qh, kh, vh, oh))
        sd.attention_from_host(qh, kh, vh, oh, qd, kd, vd, od, sd.SDPA_MASK_CAUSAL,
                               heads_per_chunk=3)
        t.cuda.current_stream().synchronize()
        sd.sdpa_device_check()
        assert parity_err(oh.float().numpy().astype(np.float64), ref) <= TOL_BF16
