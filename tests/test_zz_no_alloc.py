"""mha_forward_noalloc: multi-head attention for callers that cannot allocate
device memory (for example code inside a framework that owns the device
memory pool, or on a path that must not risk an allocation's device-wide
synchronisation).  It uses the library's static device workspace instead of a
caller-allocated one and runs the same kernels as mha_forward, so its results
must equal mha_forward's bit for bit, call after call, while the shared
workspace keeps the previous call's contents.

The file is named so that pytest collects it last: if it fails, a run that
stops at the first failure has already run every other test.  It passes on
its own in a fresh process too.
"""
import numpy as np
import pytest

import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import dev, dev_int

pytestmark = pytest.mark.gpu


def _weights(rng, dm, h, d):
    return [synthetic.round_to_bf16((rng.standard_normal(s) / np.sqrt(s[0])).astype(np.float32))
            for s in [(dm, h * d)] * 3 + [(h * d, dm)]]


def _case(seed, b, n_q, n_k, dm, h, d, cross):
    rng = np.random.default_rng(seed)
    xq = synthetic.round_to_bf16(rng.standard_normal((b, n_q, dm)).astype(np.float32))
    xkv = (synthetic.round_to_bf16(rng.standard_normal((b, n_k, dm)).astype(np.float32))
           if cross else xq)
    return xq, xkv, _weights(rng, dm, h, d)


def test_noalloc_matches_mha_forward_on_consecutive_calls():
    torch = pytest.importorskip("torch")
    cases = [  # (seed, b, n_q, n_k, d_model, h, d, mask, lengths, cross-attention)
        (1, 4, 128, 128, 512, 8, 64, sd.SDPA_MASK_PADDING, np.array([128, 64, 100, 77], np.int32), False),
        (2, 2, 300, 300, 256, 2, 128, sd.SDPA_MASK_CAUSAL, None, False),
        (3, 3, 128, 192, 512, 8, 64, sd.SDPA_MASK_PADDING, np.array([192, 5, 150], np.int32), True),
    ]
    prepared = []
    for seed, b, n_q, n_k, dm, h, d, mask, lens, cross in cases:
        assert sd.mha_workspace_size(b, n_q, n_k, h, d, d) <= sd.MHA_NOALLOC_MAX_WORKSPACE
        xq, xkv, ws = _case(seed, b, n_q, n_k, dm, h, d, cross)
        xqd = dev(xq)
        xkvd = dev(xkv) if cross else xqd
        wd = [dev(a) for a in ws]
        ld = None if lens is None else dev_int(lens)
        ref = sd.multi_head_attention(xqd, xkvd, *wd, h, mask, ld)      # caller-allocated workspace
        y = torch.empty((b, n_q, dm), dtype=torch.bfloat16, device="cuda")
        prepared.append((xqd, xkvd, wd, ld, ref, y, (b, n_q, n_k, dm, h, d, d, mask)))
    torch.cuda.synchronize()

    # One call sets the library up on this device.  Then every output buffer
    # exists before the device's free memory is read, nothing but the
    # no-allocation calls runs until it is read again, and the comparisons
    # (which may allocate inside torch) come after.
    xqd, xkvd, wd, ld, ref, y, dims = prepared[0]
    sd.mha_forward_noalloc(xqd, xkvd, *wd, y, *dims, ld)
    sd.sdpa_device_check()
    outs = [[torch.full_like(p[4], 3.0) for p in prepared] for _ in range(2)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for rnd in range(2):
        for (xqd, xkvd, wd, ld, ref, y, dims), out in zip(prepared, outs[rnd]):
            sd.mha_forward_noalloc(xqd, xkvd, *wd, out, *dims, ld)
            sd.sdpa_device_check()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before
    for rnd in range(2):
        for p, out in zip(prepared, outs[rnd]):
            assert torch.equal(out, p[4]), (rnd, p[6])


def test_noalloc_rejects_sizes_beyond_its_workspace():
    torch = pytest.importorskip("torch")
    b, n, dm, h, d = 9, 1024, 512, 8, 64
    assert sd.mha_workspace_size(b, n, n, h, d, d) > sd.MHA_NOALLOC_MAX_WORKSPACE
    x = torch.zeros((b, n, dm), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((dm, h * d), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((b, n, dm), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sd.SdpaError) as e:
        sd.mha_forward_noalloc(x, x, w, w, w, w, y, b, n, n, dm, h, d, d)
    assert e.value.status == 4   # SDPA_ERR_WORKSPACE
    # an argument mha_forward rejects gets mha_forward's status, even when too large
    with pytest.raises(sd.SdpaError) as e:
        sd.mha_forward_noalloc(x, x, w, w, w, None, y, b, n, n, dm, h, d, d)
    assert e.value.status == 1   # SDPA_ERR_INVALID_ARG
    torch.cuda.synchronize()
