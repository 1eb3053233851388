"""Runs one attention (or multi-head attention) shape a few times through the
C ABI, for profiling a single kernel launch under a profiler.

    python -m transformer_scaled_dot_02_gb300.profile --b 4 --h 16 --n 8192 --d 128 --mask 1
    python -m transformer_scaled_dot_02_gb300.profile --mha --b 32 --n 128 --d-model 512 --h 8
    python -m transformer_scaled_dot_02_gb300.profile --decode --b 32 --h 16 --n 1 --nk 8192 --d 128
    python -m transformer_scaled_dot_02_gb300.profile --restricted 1024 --b 4 --h 16 --n 8192 --mask 1
    python -m transformer_scaled_dot_02_gb300.profile --backward --b 4 --h 16 --n 8192 --mask 1
    python -m transformer_scaled_dot_02_gb300.profile --gemm 16384,4096,4096

Inputs are seeded N(0,1) bf16 values made on the device; nothing is checked.
Prints the mean call time measured with CUDA events after one warm-up call;
for plain attention and the backward also TFLOP/s, counting
2 b h n_q n_k (d_k + d_v) FLOP per forward (S, O) and
2 b h n_q n_k (3 d_k + 2 d_v) per backward (S, dP, dV, dK, dQ), halved when
causal.
"""
from __future__ import annotations

import argparse

import torch

import transformer_scaled_dot_02_gb300 as sd


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--b", type=int, default=4)
    ap.add_argument("--h", type=int, default=16)
    ap.add_argument("--n", type=int, default=8192, help="query length (and key length)")
    ap.add_argument("--nk", type=int, default=0, help="key length if different (not causal)")
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--dv", type=int, default=0, help="value size if different from --d")
    ap.add_argument("--mask", type=int, default=1)
    ap.add_argument("--len-lo", type=int, default=0, help="padding lengths uniform in [lo, nk]")
    ap.add_argument("--mha", action="store_true", help="multi-head attention with projections")
    ap.add_argument("--decode", action="store_true", help="one decoding step: --n new queries, --nk cache")
    ap.add_argument("--restricted", type=int, default=0, help="neighbourhood size r (restricted)")
    ap.add_argument("--backward", action="store_true", help="the gradients (after one forward)")
    ap.add_argument("--gemm", default="", help="M,N,K: one projection Y = X W on its own")
    ap.add_argument("--d-model", type=int, default=512)
    ap.add_argument("--iters", type=int, default=3)
    a = ap.parse_args()

    torch.manual_seed(0)
    dev = torch.device("cuda", 0)
    n_q = a.n
    n_k = a.nk or a.n
    d_v = a.dv or a.d
    lens = None
    if (a.mask & 2) or (a.decode and a.len_lo):
        lo = a.len_lo or n_k // 2
        lens = torch.randint(lo, n_k + 1, (a.b,), dtype=torch.int32, device=dev)
    sd.load_library()
    gemm_mnk = [int(x) for x in a.gemm.split(",")] if a.gemm else None
    if gemm_mnk:
        gm, gn, gk = gemm_mnk
        x = (torch.randn(gm, gk, device=dev) * 0.1).to(torch.bfloat16)
        w = (torch.randn(gk, gn, device=dev) * 0.1).to(torch.bfloat16)
        y = torch.empty(gm, gn, dtype=torch.bfloat16, device=dev)

        def run():
            sd.linear_forward(x, w, y, gm, gn, gk)
    elif a.decode:
        q = torch.randn(a.b, a.h, n_q, a.d, device=dev).to(torch.bfloat16)
        k = torch.randn(a.b, a.h, n_k, a.d, device=dev).to(torch.bfloat16)
        v = torch.randn(a.b, a.h, n_k, d_v, device=dev).to(torch.bfloat16)
        out = torch.empty(a.b, a.h, n_q, d_v, dtype=torch.bfloat16, device=dev)
        work = torch.empty(max(1, sd.sdpa_decode_workspace_size(a.b, a.h, n_q, n_k, d_v)),
                           dtype=torch.uint8, device=dev)

        def run():
            sd.sdpa_decode(q, k, v, out, work, work.numel(), a.b, a.h, n_q, n_k, a.d, d_v, lens)
    elif a.mha:
        dm = a.d_model
        xq = torch.randn(a.b, n_q, dm, device=dev).to(torch.bfloat16)
        xkv = xq if n_k == n_q else torch.randn(a.b, n_k, dm, device=dev).to(torch.bfloat16)
        ws = [(torch.randn(*s, device=dev) / s[0] ** 0.5).to(torch.bfloat16)
              for s in [(dm, a.h * a.d)] * 3 + [(a.h * a.d, dm)]]
        work = torch.empty(sd.mha_workspace_size(a.b, n_q, n_k, a.h, a.d, a.d), dtype=torch.uint8,
                           device=dev)

        def run():
            sd.multi_head_attention(xq, xkv, *ws, a.h, a.mask, lens, workspace=work)
    elif a.backward:
        q, k, v, dout = (torch.randn(a.b, a.h, n, d, device=dev).to(torch.bfloat16)
                         for n, d in ((n_q, a.d), (n_k, a.d), (n_k, d_v), (n_q, d_v)))
        out, lse = sd.attention_with_lse(q, k, v, a.mask, lens, a.restricted)
        grads = [torch.empty_like(x) for x in (q, k, v)]
        work = torch.empty(sd.sdpa_backward_workspace_size(a.b, a.h, n_q, a.d), dtype=torch.uint8,
                           device=dev)

        def run():
            sd.sdpa_backward(q, k, v, out, dout, lse, *grads, work, work.numel(), a.b, a.h, n_q,
                             n_k, a.d, d_v, a.mask, lens, a.restricted)
    else:
        q = torch.randn(a.b, a.h, n_q, a.d, device=dev).to(torch.bfloat16)
        k = torch.randn(a.b, a.h, n_k, a.d, device=dev).to(torch.bfloat16)
        v = torch.randn(a.b, a.h, n_k, d_v, device=dev).to(torch.bfloat16)
        out = torch.empty(a.b, a.h, n_q, d_v, dtype=torch.bfloat16, device=dev)

        def run():
            if a.restricted:
                sd.sdpa_forward_restricted(q, k, v, out, a.b, a.h, n_q, n_k, a.d, d_v, a.mask, lens,
                                           a.restricted)
            else:
                sd.sdpa_forward(q, k, v, out, a.b, a.h, n_q, n_k, a.d, d_v, a.mask, lens)

    run()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(a.iters):
        run()
    e.record()
    torch.cuda.synchronize()
    sd.sdpa_device_check()
    ms = s.elapsed_time(e) / a.iters
    line = "mean %.4f ms per call over %d calls" % (ms, a.iters)
    if gemm_mnk:
        line += ", %.1f TFLOP/s" % (2.0 * gm * gn * gk / (ms * 1e-3) / 1e12)
    elif a.decode:
        # K and V caches read once (the whole capacity when no lengths are given)
        line += ", %.0f GB/s of K/V" % (2.0 * a.b * a.h * n_k * (a.d + d_v) / (ms * 1e-3) / 1e9)
    elif not (a.mha or a.decode or a.restricted):
        # 2 n_q n_k per unit of head size: S and O in the forward; S, dP, dV, dK, dQ in the backward
        units = 3 * a.d + 2 * d_v if a.backward else a.d + d_v
        flops = 2 * units * a.b * a.h * n_q * n_k * (0.5 if a.mask & 1 else 1)
        line += ", %.1f TFLOP/s" % (flops / (ms * 1e-3) / 1e12)
    print(line)


if __name__ == "__main__":
    main()
