"""Failure detection without a GPU fault: a bounded wait that runs out.

A test-only copy of the attention kernels, compiled here with
SDPA_TEST_WITHHOLD_FIRST_S_COMMIT, never signals the first score tile of a
query tile (forward) or of a key tile (backward).  The softmax or compute
warps' wait on it gives up after its limit (about a second), the CTA aborts
cleanly (copies and MMAs in flight are drained, tensor memory is freed) and
sdpa_device_check() reports SDPA_ERR_DEVICE_TIMEOUT.  The
context stays usable: the same library then returns to normal operation and
the product library computes correct results.
"""
import os
import subprocess
import tempfile
import time

import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from transformer_scaled_dot_02_gb300 import build as sd_build
from gpu_util import TOL_BF16, dev, host, parity_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def faulty_lib():
    sd_build.build()
    d = tempfile.mkdtemp(prefix="sdpa_timeout_")
    nvcc = sd_build._nvcc()
    # every attention kernel carries the hook
    hooked = ["sdpa_tc.cu", "sdpa_one_tile.cu", "sdpa_bwd.cu", "sdpa_bwd_wide.cu"]
    objs = []
    for src in hooked:
        obj = os.path.join(d, src.replace(".cu", "_withhold.o"))
        subprocess.check_call([nvcc] + sd_build._flags() + ["-DSDPA_TEST_WITHHOLD_FIRST_S_COMMIT",
                              "-c", os.path.join(sd_build.CSRC, src), "-o", obj])
        objs.append(obj)
    others = [os.path.join(sd_build.BUILD_DIR, s.replace(".cu", ".o"))
              for s in sd_build.SOURCES if s not in hooked]
    lib_path = os.path.join(d, "libsdpa_withhold.so")
    subprocess.check_call([nvcc] + sd_build.ARCH + ["-shared", "-cudart", "static", "-o", lib_path]
                          + objs + others)
    return sd.load_library(lib_path)


@pytest.mark.parametrize("kernel,d", [("two_tile", 64), ("one_tile", 64), ("one_tile", 512)])
def test_bounded_wait_times_out_and_reports(faulty_lib, kernel, d, pin_kernels):
    """d = 512 runs the one-tile kernel's single-stage path (K in two
    halves): its producer also waits on the withheld commit and must drain
    its own copies before the CTA leaves."""
    import torch
    pin_kernels(attention=kernel, lib=faulty_lib)
    rng = np.random.default_rng(1)
    b, h, n = 1, 1, 128   # one query tile (two CTAs at d = 512, one per half of d_v)
    q = synthetic.round_to_bf16(rng.standard_normal((b, h, n, d)).astype(np.float32))
    qd = dev(q)
    out = torch.zeros((b, h, n, d), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    rc = faulty_lib.sdpa_forward(qd.data_ptr(), qd.data_ptr(), qd.data_ptr(), out.data_ptr(), b, h,
                                 n, n, d, d, 0, None, __import__("ctypes").c_float(0.0), stream)
    assert rc == 0
    st = faulty_lib.sdpa_device_check()
    elapsed = time.time() - t0
    assert st == 6, sd.STATUS_NAMES.get(st, st)   # SDPA_ERR_DEVICE_TIMEOUT
    assert elapsed < 30.0
    # the word was cleared by the check
    assert faulty_lib.sdpa_device_check() == 0
    # the context still works: the product library computes the right answer
    k = synthetic.round_to_bf16(rng.standard_normal((b, h, n, d)).astype(np.float32))
    v = synthetic.round_to_bf16(rng.standard_normal((b, h, n, d)).astype(np.float32))
    got = host(sd.attention(dev(q), dev(k), dev(v), sd.SDPA_MASK_CAUSAL))
    sd.sdpa_device_check()
    assert parity_err(got, oracle.sdpa(q, k, v, sd.SDPA_MASK_CAUSAL)) <= TOL_BF16


@pytest.mark.parametrize("d", [64, 512])
def test_backward_bounded_wait_times_out_and_reports(faulty_lib, d):
    """d = 64: one key tile, one CTA; d = 512: one 64-key tile, two CTAs
    (one per half of d)."""
    import ctypes
    import torch
    rng = np.random.default_rng(2)
    b, h = 1, 1
    n = 128 if d <= 256 else 64
    q, k, v, do = (synthetic.round_to_bf16(rng.standard_normal((b, h, n, d)).astype(np.float32))
                   for _ in range(4))
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    out, lse = sd.attention_with_lse(qd, kd, vd, sd.SDPA_MASK_CAUSAL)   # product library
    sd.sdpa_device_check()
    ws = torch.empty(sd.sdpa_backward_workspace_size(b, h, n, d), dtype=torch.uint8, device="cuda")
    g = [torch.empty_like(x) for x in (qd, kd, vd)]
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    rc = faulty_lib.sdpa_backward(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(),
                                  dod.data_ptr(), lse.data_ptr(), g[0].data_ptr(), g[1].data_ptr(),
                                  g[2].data_ptr(), ws.data_ptr(), ws.numel(), b, h, n, n, d, d,
                                  sd.SDPA_MASK_CAUSAL, None, 0, ctypes.c_float(0.0), stream)
    assert rc == 0
    st = faulty_lib.sdpa_device_check()
    assert st == 6, sd.STATUS_NAMES.get(st, st)   # SDPA_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 30.0
    assert faulty_lib.sdpa_device_check() == 0
    # the context still works: the product library's backward matches the oracle
    dq, dk, dv = sd.attention_backward(qd, kd, vd, out, lse, dod, sd.SDPA_MASK_CAUSAL)
    sd.sdpa_device_check()
    rq, rk, rv = oracle.backward(q, k, v, do, sd.SDPA_MASK_CAUSAL)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert parity_err(host(got), ref) <= TOL_BF16
