"""Stream order under programmatic dependent launch.

Every attention launch may start while the previous kernel in the stream
finishes; it must still read its inputs (Q, K, V and the key-padding
lengths) only after that kernel has completed.  Here torch kernels write the
inputs on the same stream immediately before each call, with no
synchronisation, and the values change every round: a read that ran ahead
would see the previous round's lengths or queries.
"""
import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_BF16, dev, host, parity_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernel,d,n", [("one_tile", 64, 384), ("two_tile", 64, 384), ("two_tile", 128, 640),
                                        ("one_tile", 512, 200)])
def test_inputs_written_just_before_the_call(kernel, d, n, pin_kernels):
    import torch
    pin_kernels(attention=kernel)
    rng = np.random.default_rng(40 + d)
    b, h = 3, 2
    q0 = synthetic.round_to_bf16(rng.standard_normal((b, h, n, d)).astype(np.float32))
    k = synthetic.round_to_bf16(rng.standard_normal((b, h, n, d)).astype(np.float32))
    v = synthetic.round_to_bf16(rng.standard_normal((b, h, n, d)).astype(np.float32))
    qd, kd, vd = dev(q0), dev(k), dev(v)
    qw = torch.empty_like(qd)
    lens_d = torch.zeros(b, dtype=torch.int32, device="cuda")
    out = torch.empty_like(qd)
    rounds = [np.array(x, np.int32) for x in ([n, 1, 77], [5, n, 131], [n // 2, 0, n])]
    for r, lens in enumerate(rounds):
        sign = 1.0 if r % 2 == 0 else -1.0
        # kernels on the current stream, right before the call
        torch.mul(qd, sign, out=qw)
        for i in range(b):
            lens_d[i:i + 1].fill_(int(lens[i]))
        sd.sdpa_forward(qw, kd, vd, out, b, h, n, n, d, d, sd.SDPA_MASK_PADDING, lens_d)
        got = host(out)
        sd.sdpa_device_check()
        ref = oracle.sdpa(q0 * np.float32(sign), k, v, sd.SDPA_MASK_PADDING, lens)
        assert parity_err(got, ref) <= TOL_BF16, (r, kernel)


def test_backward_inputs_written_just_before_the_call():
    import torch
    rng = np.random.default_rng(77)
    b, h, n, d = 2, 2, 300, 64
    q, k, v, do0 = (synthetic.round_to_bf16(rng.standard_normal((b, h, n, d)).astype(np.float32))
                    for _ in range(4))
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do0)
    out, lse = sd.attention_with_lse(qd, kd, vd, sd.SDPA_MASK_CAUSAL)
    dow = torch.empty_like(dod)
    for r, sign in enumerate((1.0, -1.0, 2.0)):
        torch.mul(dod, sign, out=dow)   # the upstream gradient, written just before the call
        dq, dk, dv = sd.attention_backward(qd, kd, vd, out, lse, dow, sd.SDPA_MASK_CAUSAL)
        sd.sdpa_device_check()
        rq, rk, rv = oracle.backward(q, k, v, do0 * np.float32(sign), sd.SDPA_MASK_CAUSAL)
        for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
            assert parity_err(host(got), ref) <= TOL_BF16, r
