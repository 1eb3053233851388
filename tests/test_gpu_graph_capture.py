"""The library's calls allocate nothing and never synchronise, so a stream
capture can record them: one CUDA graph with sdpa_forward (both kernels),
mha_forward and the backward replays to the eager results bit for bit."""
import numpy as np
import pytest

import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import dev, dev_int

pytestmark = pytest.mark.gpu


def test_graph_capture_replays_eager_results():
    t = __import__("torch")
    rng = np.random.default_rng(14000)

    def r(shape, std=1.0):
        return dev(synthetic.round_to_bf16(rng.standard_normal(shape).astype(np.float32) * np.float32(std)))

    q, k, v, do = r((2, 4, 300, 64)), r((2, 4, 300, 64)), r((2, 4, 300, 64)), r((2, 4, 300, 64))
    ql, kl, vl = r((1, 2, 3000, 128), 0.5), r((1, 2, 3000, 128), 0.5), r((1, 2, 3000, 128), 0.5)
    x = r((2, 130, 256))
    ws = [r(s, 1.0 / np.sqrt(s[0])) for s in [(256, 4 * 64)] * 3 + [(4 * 64, 256)]]
    lens = dev_int(np.array([130, 61], np.int32))
    out = t.empty_like(q)
    lse = t.empty((2, 4, 300), dtype=t.float32, device="cuda")
    out_l = t.empty_like(ql)
    y = t.empty_like(x)
    mha_ws = t.empty(sd.mha_workspace_size(2, 130, 130, 4, 64, 64), dtype=t.uint8, device="cuda")
    grads = [t.empty_like(a) for a in (q, k, v)]
    bwd_ws = t.empty(sd.sdpa_backward_workspace_size(2, 4, 300, 64), dtype=t.uint8, device="cuda")
    s = t.cuda.Stream()

    def calls():
        sd.sdpa_forward_lse(q, k, v, out, lse, 2, 4, 300, 300, 64, 64, sd.SDPA_MASK_CAUSAL, None, 0,
                            0.0, s)
        sd.sdpa_forward(ql, kl, vl, out_l, 1, 2, 3000, 3000, 128, 128, sd.SDPA_MASK_CAUSAL, None,
                        0.0, s)
        sd.mha_forward(x, x, *ws, y, mha_ws, mha_ws.numel(), 2, 130, 130, 256, 4, 64, 64,
                       sd.SDPA_MASK_PADDING, lens, 0.0, s)
        sd.sdpa_backward(q, k, v, out, do, lse, *grads, bwd_ws, bwd_ws.numel(), 2, 4, 300, 300, 64,
                         64, sd.SDPA_MASK_CAUSAL, None, 0, 0.0, s)

    s.wait_stream(t.cuda.current_stream())
    with t.cuda.stream(s):
        calls()
    s.synchronize()
    sd.sdpa_device_check()
    eager = [a.clone() for a in (out, lse, out_l, y, *grads)]
    for a in (out, lse, out_l, y, *grads):
        a.zero_()
    g = t.cuda.CUDAGraph()
    with t.cuda.graph(g, stream=s):
        calls()
    g.replay()
    g.replay()
    t.cuda.synchronize()
    sd.sdpa_device_check()
    for a, b in zip((out, lse, out_l, y), eager[:4]):
        assert t.equal(a, b)
    # dQ is accumulated with floating-point reductions whose order may vary
    for a, b in zip(grads, eager[4:]):
        assert (a.float() - b.float()).abs().max().item() <= 1e-2 * b.float().abs().max().item()
