"""Seeded synthetic inputs for the attention workloads.

This module is the only code shared by the CPU oracle's tests and the CUDA
path: it draws random numbers and rounds them to the storage type, and holds
none of the attention arithmetic.  Values are returned as float32 numpy arrays
whose entries are exactly representable in the workload's storage type
(bf16 values are float32 samples rounded to nearest-even), so both sides see
bit-identical inputs.

Generator: numpy's PCG64 seeded through ``SeedSequence([seed, stream])``.
One stream per tensor keeps each tensor independent of the shapes of the
others.  Shapes and distributions follow the Transformer's base model
(d_model=512, h=8, d_k=d_v=64) and big model (d_model=1024, h=16)
("Attention Is All You Need", section 3.2.2 and Table 3).
"""
from __future__ import annotations

import dataclasses
import numpy as np

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_PADDING = 2

# Stream ids inside one config's seed.
_STREAM = {"q": 1, "k": 2, "v": 3, "xq": 4, "xkv": 5, "wq": 6, "wk": 7,
           "wv": 8, "wo": 9, "len": 10, "dout": 11}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    b: int
    h: int
    n_q: int
    n_k: int
    d_k: int
    d_v: int
    mask_kind: int
    dtype: str                 # "f32" or "bf16": storage and I/O type
    value_scale: float = 1.0   # Q/K/V (or X) = value_scale * N(0,1)
    len_range: tuple | None = None   # key-padding lengths, closed range
    d_model: int | None = None       # set for the multi-head (projection) form
    seed: int = 0
    window: int = 0                  # r of restricted self-attention (0: none)

    @property
    def causal(self) -> bool:
        return bool(self.mask_kind & MASK_CAUSAL)


# The five workloads: shapes of the base and big models, synthetic values.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 1, 16, 16, 64, 64, MASK_NONE, "f32", seed=1000),
    "tiny_f32_causal": Workload("tiny_f32_causal", 1, 1, 16, 16, 64, 64, MASK_CAUSAL, "f32", seed=1000),
    "enc_mha_base": Workload("enc_mha_base", 32, 8, 128, 128, 64, 64, MASK_PADDING, "bf16",
                             len_range=(64, 128), d_model=512, seed=1001),
    "dec_causal_base": Workload("dec_causal_base", 16, 8, 512, 512, 64, 64, MASK_CAUSAL, "bf16",
                                seed=1002),
    "cross_big": Workload("cross_big", 32, 16, 256, 384, 64, 64, MASK_PADDING, "bf16",
                          len_range=(192, 384), d_model=1024, seed=1003),
    "long_causal": Workload("long_causal", 4, 16, 8192, 8192, 128, 128, MASK_CAUSAL, "bf16",
                            value_scale=0.5, seed=1004),
    # the widened rows: restricted self-attention (section 4's r), one
    # decoding step against 8192-token caches, and Table 3's single 512-wide head
    "long_restricted": Workload("long_restricted", 4, 16, 8192, 8192, 128, 128, MASK_CAUSAL,
                                "bf16", value_scale=0.5, seed=1005, window=1024),
    "decode_big": Workload("decode_big", 32, 16, 1, 8192, 128, 128, MASK_NONE, "bf16", seed=1006),
    "wide_d512": Workload("wide_d512", 4, 1, 8192, 8192, 512, 512, MASK_CAUSAL, "bf16",
                          value_scale=0.5, seed=1007),
}


def rng(seed: int, stream: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _STREAM[stream]])))


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    nan = np.isnan(x)
    out = rounded.astype(np.uint32).view(np.float32)
    if nan.any():
        out = out.copy()
        out[nan] = np.float32(np.nan)
    return out


def normal(seed: int, stream: str, shape, std: float = 1.0, dtype: str = "bf16") -> np.ndarray:
    x = rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return round_to_bf16(x) if dtype == "bf16" else x


def kv_lengths(w: Workload, b: int | None = None) -> np.ndarray | None:
    if not (w.mask_kind & MASK_PADDING):
        return None
    lo, hi = w.len_range if w.len_range is not None else (w.n_k, w.n_k)
    return rng(w.seed, "len").integers(lo, hi + 1, size=(b or w.b,), dtype=np.int64).astype(np.int32)


def sdpa_inputs(w: Workload, seed: int | None = None, b: int | None = None, h: int | None = None):
    """Q [b,h,n_q,d_k], K [b,h,n_k,d_k], V [b,h,n_k,d_v] (BHSD, float32 arrays) and lengths."""
    s = w.seed if seed is None else seed
    b = w.b if b is None else b
    h = w.h if h is None else h
    q = normal(s, "q", (b, h, w.n_q, w.d_k), w.value_scale, w.dtype)
    k = normal(s, "k", (b, h, w.n_k, w.d_k), w.value_scale, w.dtype)
    v = normal(s, "v", (b, h, w.n_k, w.d_v), w.value_scale, w.dtype)
    lens = kv_lengths(dataclasses.replace(w, seed=s), b)
    return q, k, v, lens


def dout_input(w: Workload, seed: int | None = None, b: int | None = None, h: int | None = None,
               n_q: int | None = None) -> np.ndarray:
    """Upstream gradient dO [b,h,n_q,d_v] ~ N(0,1) in the workload's storage type."""
    s = w.seed if seed is None else seed
    return normal(s, "dout", (w.b if b is None else b, w.h if h is None else h,
                              w.n_q if n_q is None else n_q, w.d_v), 1.0, w.dtype)


def mha_inputs(w: Workload, seed: int | None = None):
    """X_q [b,n_q,d_model], X_kv [b,n_k,d_model] ~ N(0,1); W^Q,W^K [d_model,h*d_k],
    W^V [d_model,h*d_v], W^O [h*d_v,d_model] ~ N(0, 1/d_model); lengths.

    For self-attention (n_q == n_k and no separate encoder memory) X_kv is X_q.
    """
    assert w.d_model is not None
    s = w.seed if seed is None else seed
    dm = w.d_model
    std_w = float(1.0 / np.sqrt(dm))
    xq = normal(s, "xq", (w.b, w.n_q, dm), w.value_scale, w.dtype)
    self_attn = w.name.startswith("enc")
    xkv = xq if self_attn else normal(s, "xkv", (w.b, w.n_k, dm), w.value_scale, w.dtype)
    wq = normal(s, "wq", (dm, w.h * w.d_k), std_w, w.dtype)
    wk = normal(s, "wk", (dm, w.h * w.d_k), std_w, w.dtype)
    wv = normal(s, "wv", (dm, w.h * w.d_v), std_w, w.dtype)
    wo = normal(s, "wo", (w.h * w.d_v, dm), std_w, w.dtype)
    lens = kv_lengths(dataclasses.replace(w, seed=s))
    return xq, xkv, wq, wk, wv, wo, lens
