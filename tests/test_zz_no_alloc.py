"""mha_forward_noalloc: multi-head attention for callers that cannot allocate
device memory (for example code inside a framework that owns the device
memory pool, or on a path that must not risk an allocation's device-wide
synchronisation).  It uses the library's static device workspace instead of a
caller-allocated one, so its results must equal those of mha_forward on the
same inputs, call after call, while the shared workspace keeps the previous
call's contents.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_BF16, dev, dev_int, host, rel_err

pytestmark = pytest.mark.gpu


def _inputs(seed, b, n, dm, h, d):
    rng = np.random.default_rng(seed)
    x = synthetic.round_to_bf16(rng.standard_normal((b, n, dm)).astype(np.float32))
    ws = [synthetic.round_to_bf16((rng.standard_normal(s) / np.sqrt(s[0])).astype(np.float32))
          for s in [(dm, h * d)] * 3 + [(h * d, dm)]]
    return x, ws


def test_noalloc_matches_mha_forward_on_consecutive_calls():
    torch = pytest.importorskip("torch")
    cases = [  # (seed, b, n, d_model, h, d, mask, lengths)
        (1, 4, 128, 512, 8, 64, sd.SDPA_MASK_PADDING, np.array([128, 64, 100, 77], np.int32)),
        (2, 2, 300, 256, 2, 128, sd.SDPA_MASK_CAUSAL, None),
    ]
    for seed, b, n, dm, h, d, mask, lens in cases:
        assert sd.mha_workspace_size(b, n, n, h, d, d) <= sd.MHA_NOALLOC_MAX_WORKSPACE
        x, ws = _inputs(seed, b, n, dm, h, d)
        xd, wd = dev(x), [dev(a) for a in ws]
        ld = None if lens is None else dev_int(lens)
        ref = sd.multi_head_attention(xd, xd, *wd, h, mask, ld)      # caller-allocated workspace
        y = torch.empty((b, n, dm), dtype=torch.bfloat16, device="cuda")
        sd.mha_forward_noalloc(xd, xd, *wd, y, b, n, n, dm, h, d, d, mask, ld)
        sd.sdpa_device_check()
        assert rel_err(host(y), host(ref)) <= TOL_BF16


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
    torch.cuda.synchronize()
