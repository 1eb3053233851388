"""Python binding of libsdpa: fused scaled dot-product and multi-head attention
on one GB300 GPU.

The functions below carry the names of the C entry points in include/sdpa.h
and only marshal arguments: every step of the computation runs in the CUDA
kernels of libsdpa.so.  Tensor arguments may be torch tensors (their
``data_ptr()`` is passed) or raw device addresses as ints.  ``stream`` defaults
to PyTorch's current CUDA stream.

There is no fallback: if libsdpa.so is missing or fails to load, importing the
functions raises, and every call returns the library's status as an exception.

The library picks kernels and tile sizes from the shapes;
``sdpa_set_kernel_choice`` (or the ``kernel_choice`` context manager) pins
them for tests and tuning (include/sdpa.h gives the defaults).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsdpa.so")

SDPA_MASK_NONE = 0
SDPA_MASK_CAUSAL = 1
SDPA_MASK_PADDING = 2

STATUS_NAMES = {0: "SDPA_OK", 1: "SDPA_ERR_INVALID_ARG", 2: "SDPA_ERR_UNSUPPORTED",
                3: "SDPA_ERR_UNSUPPORTED_DEVICE", 4: "SDPA_ERR_WORKSPACE", 5: "SDPA_ERR_CUDA",
                6: "SDPA_ERR_DEVICE_TIMEOUT"}

# Every symbol include/sdpa.h declares.
EXPORTS = ("sdpa_forward", "sdpa_forward_restricted", "sdpa_forward_lse", "sdpa_forward_host",
           "sdpa_backward_workspace_size", "sdpa_backward", "sdpa_forward_f32",
           "sdpa_decode_workspace_size", "sdpa_decode", "mha_workspace_size",
           "mha_forward",
           "mha_forward_noalloc", "linear_forward", "sdpa_set_kernel_choice", "sdpa_device_check",
           "sdpa_status_string")

# Size of the static workspace behind mha_forward_noalloc (SDPA_MHA_NOALLOC_MAX_WORKSPACE).
MHA_NOALLOC_MAX_WORKSPACE = 32 << 20


class SdpaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, STATUS_NAMES.get(status, "status %d" % status)))


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Loads libsdpa.so (built by ``build.build()``) and declares its ABI."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError("libsdpa.so not built (%s); run transformer_scaled_dot_02_gb300.build" % p)
    lib = ctypes.CDLL(p)
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    attn = [P, P, P, P, I, I, I, I, I, I, I, P, F, P]
    lib.sdpa_forward.argtypes = attn
    lib.sdpa_forward.restype = I
    lib.sdpa_forward_restricted.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, I, F, P]
    lib.sdpa_forward_restricted.restype = I
    lib.sdpa_forward_lse.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, P, I, F, P]
    lib.sdpa_forward_lse.restype = I
    lib.sdpa_backward_workspace_size.argtypes = [I, I, I, I]
    lib.sdpa_backward_workspace_size.restype = SZ
    lib.sdpa_backward.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, I, I, I, P, I, F,
                                  P]
    lib.sdpa_backward.restype = I
    lib.sdpa_forward_host.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, F, I, P]
    lib.sdpa_forward_host.restype = I
    lib.sdpa_forward_f32.argtypes = attn
    lib.sdpa_forward_f32.restype = I
    lib.sdpa_decode_workspace_size.argtypes = [I, I, I, I, I]
    lib.sdpa_decode_workspace_size.restype = SZ
    lib.sdpa_decode.argtypes = [P, P, P, P, P, SZ, I, I, I, I, I, I, P, F, P]
    lib.sdpa_decode.restype = I
    lib.mha_workspace_size.argtypes = [I, I, I, I, I, I]
    lib.mha_workspace_size.restype = SZ
    lib.mha_forward.argtypes = [P, P, P, P, P, P, P, P, SZ, I, I, I, I, I, I, I, I, P, F, P]
    lib.mha_forward.restype = I
    lib.mha_forward_noalloc.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, F, P]
    lib.mha_forward_noalloc.restype = I
    lib.linear_forward.argtypes = [P, P, P, I, I, I, P]
    lib.linear_forward.restype = I
    lib.sdpa_set_kernel_choice.argtypes = [I, I, I]
    lib.sdpa_set_kernel_choice.restype = I
    lib.sdpa_device_check.argtypes = []
    lib.sdpa_device_check.restype = I
    lib.sdpa_status_string.argtypes = [I]
    lib.sdpa_status_string.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != 0:
        raise SdpaError(status, where)


def sdpa_forward(q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind=SDPA_MASK_NONE,
                 kv_lengths=None, scale=0.0, stream=None) -> None:
    """bf16 attention, BHSD tensors (see include/sdpa.h)."""
    _check(load_library().sdpa_forward(_addr(q), _addr(k), _addr(v), _addr(out), b, h, n_q, n_k,
                                       d_k, d_v, mask_kind, _addr(kv_lengths), float(scale),
                                       _stream(stream)), "sdpa_forward")


def sdpa_forward_restricted(q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind=SDPA_MASK_NONE,
                            kv_lengths=None, r=1, scale=0.0, stream=None) -> None:
    """bf16 restricted self-attention: query i sees keys i-(r-1)//2 .. i+r//2."""
    _check(load_library().sdpa_forward_restricted(_addr(q), _addr(k), _addr(v), _addr(out), b, h,
                                                  n_q, n_k, d_k, d_v, mask_kind,
                                                  _addr(kv_lengths), int(r), float(scale),
                                                  _stream(stream)), "sdpa_forward_restricted")


def sdpa_forward_lse(q, k, v, out, lse, b, h, n_q, n_k, d_k, d_v, mask_kind=SDPA_MASK_NONE,
                     kv_lengths=None, r=0, scale=0.0, stream=None) -> None:
    """sdpa_forward (r = 0) or the restricted form (r >= 1) that also writes
    each row's natural log-sum-exp into lse [b, h, n_q] fp32."""
    _check(load_library().sdpa_forward_lse(_addr(q), _addr(k), _addr(v), _addr(out), _addr(lse), b,
                                           h, n_q, n_k, d_k, d_v, mask_kind, _addr(kv_lengths),
                                           int(r), float(scale), _stream(stream)),
           "sdpa_forward_lse")


def sdpa_backward_workspace_size(b, h, n_q, d) -> int:
    return int(load_library().sdpa_backward_workspace_size(b, h, n_q, d))


def sdpa_backward(q, k, v, out, dout, lse, dq, dk, dv, workspace, ws_bytes, b, h, n_q, n_k, d_k,
                  d_v, mask_kind=SDPA_MASK_NONE, kv_lengths=None, r=0, scale=0.0,
                  stream=None) -> None:
    """Gradients dq, dk, dv of attention given dout and the forward's lse."""
    _check(load_library().sdpa_backward(_addr(q), _addr(k), _addr(v), _addr(out), _addr(dout),
                                        _addr(lse), _addr(dq), _addr(dk), _addr(dv),
                                        _addr(workspace), int(ws_bytes), b, h, n_q, n_k, d_k, d_v,
                                        mask_kind, _addr(kv_lengths), int(r), float(scale),
                                        _stream(stream)), "sdpa_backward")


def sdpa_forward_f32(q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind=SDPA_MASK_NONE,
                     kv_lengths=None, scale=0.0, stream=None) -> None:
    """fp32 attention, BHSD tensors (see include/sdpa.h)."""
    _check(load_library().sdpa_forward_f32(_addr(q), _addr(k), _addr(v), _addr(out), b, h, n_q,
                                           n_k, d_k, d_v, mask_kind, _addr(kv_lengths),
                                           float(scale), _stream(stream)), "sdpa_forward_f32")


def sdpa_decode_workspace_size(b, h, n_q, n_k, d_v) -> int:
    return int(load_library().sdpa_decode_workspace_size(b, h, n_q, n_k, d_v))


def sdpa_decode(q, k, v, out, workspace, ws_bytes, b, h, n_q, n_k, d_k, d_v, kv_lengths=None,
                scale=0.0, stream=None) -> None:
    """One decoding step over bf16 K/V caches (see include/sdpa.h)."""
    _check(load_library().sdpa_decode(_addr(q), _addr(k), _addr(v), _addr(out), _addr(workspace),
                                      int(ws_bytes), b, h, n_q, n_k, d_k, d_v, _addr(kv_lengths),
                                      float(scale), _stream(stream)), "sdpa_decode")


def decode_step(q, k, v, kv_lengths=None, scale=0.0, workspace=None, stream=None):
    """Allocates the output (and, if needed, the workspace) with torch and
    calls sdpa_decode on q [b,h,n_q,d_k], k [b,h,n_k,d_k], v [b,h,n_k,d_v]
    bf16 tensors."""
    import torch
    b, h, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    need = sdpa_decode_workspace_size(b, h, n_q, n_k, d_v)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    out = torch.empty((b, h, n_q, d_v), dtype=q.dtype, device=q.device)
    sdpa_decode(q, k, v, out, workspace, 0 if workspace is None else workspace.numel(), b, h, n_q,
                n_k, d_k, d_v, kv_lengths, scale, stream)
    return out


def mha_workspace_size(b, n_q, n_k, h, d_k, d_v) -> int:
    return int(load_library().mha_workspace_size(b, n_q, n_k, h, d_k, d_v))


def mha_forward(xq, xkv, wq, wk, wv, wo, y, workspace, ws_bytes, b, n_q, n_k, d_model, h, d_k,
                d_v, mask_kind=SDPA_MASK_NONE, kv_lengths=None, scale=0.0, stream=None) -> None:
    """Multi-head attention with projections (see include/sdpa.h)."""
    _check(load_library().mha_forward(_addr(xq), _addr(xkv), _addr(wq), _addr(wk), _addr(wv),
                                      _addr(wo), _addr(y), _addr(workspace), int(ws_bytes), b, n_q,
                                      n_k, d_model, h, d_k, d_v, mask_kind, _addr(kv_lengths),
                                      float(scale), _stream(stream)), "mha_forward")


def mha_forward_noalloc(xq, xkv, wq, wk, wv, wo, y, b, n_q, n_k, d_model, h, d_k, d_v,
                        mask_kind=SDPA_MASK_NONE, kv_lengths=None, scale=0.0, stream=None) -> None:
    """mha_forward without a workspace argument, for callers that cannot
    allocate device memory: the library's static device workspace (at most
    MHA_NOALLOC_MAX_WORKSPACE bytes) is used instead.  Calls that overlap on
    the GPU share that workspace and must be ordered by the caller (see
    include/sdpa.h)."""
    _check(load_library().mha_forward_noalloc(_addr(xq), _addr(xkv), _addr(wq), _addr(wk),
                                              _addr(wv), _addr(wo), _addr(y), b, n_q, n_k,
                                              d_model, h, d_k, d_v, mask_kind, _addr(kv_lengths),
                                              float(scale), _stream(stream)),
           "mha_forward_noalloc")


def linear_forward(x, w, y, m, n, k, stream=None) -> None:
    """y = x w for row-major bf16 matrices (see include/sdpa.h)."""
    _check(load_library().linear_forward(_addr(x), _addr(w), _addr(y), m, n, k, _stream(stream)),
           "linear_forward")


ATTENTION_KERNELS = {None: 0, "one_tile": 1, "two_tile": 2}


def sdpa_set_kernel_choice(attention_kernel=0, one_tile_keys=0, gemm_bn=0, lib=None) -> None:
    """Pins kernel choices for every later call (0: choose by shape)."""
    _check((lib or load_library()).sdpa_set_kernel_choice(attention_kernel, one_tile_keys, gemm_bn),
           "sdpa_set_kernel_choice")


class kernel_choice:
    """Context manager: ``with kernel_choice(attention="one_tile", one_tile_keys=32): ...``
    pins the choices inside the block and returns them to the shapes after it."""

    def __init__(self, attention=None, one_tile_keys=0, gemm_bn=0, lib=None):
        self.args = (ATTENTION_KERNELS[attention], int(one_tile_keys), int(gemm_bn))
        self.lib = lib

    def __enter__(self):
        sdpa_set_kernel_choice(*self.args, lib=self.lib)
        return self

    def __exit__(self, *exc):
        sdpa_set_kernel_choice(0, 0, 0, lib=self.lib)
        return False


def sdpa_device_check() -> None:
    """Synchronises the device; raises if a kernel gave up on a bounded wait."""
    _check(load_library().sdpa_device_check(), "sdpa_device_check")


def sdpa_status_string(status: int) -> str:
    return load_library().sdpa_status_string(status).decode()


# ---------------------------------------------------------------- conveniences
def attention(q, k, v, mask_kind=SDPA_MASK_NONE, kv_lengths=None, scale=0.0, stream=None):
    """Allocates the output with torch and calls sdpa_forward (bf16) or
    sdpa_forward_f32 (fp32) on BHSD tensors q [b,h,n_q,d_k], k, v."""
    import torch
    b, h, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    out = torch.empty((b, h, n_q, d_v), dtype=q.dtype, device=q.device)
    fn = sdpa_forward if q.dtype == torch.bfloat16 else sdpa_forward_f32
    fn(q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind, kv_lengths, scale, stream)
    return out


def multi_head_attention(xq, xkv, wq, wk, wv, wo, h, mask_kind=SDPA_MASK_NONE, kv_lengths=None,
                         scale=0.0, workspace=None, stream=None):
    """Allocates the output (and, if not given, the workspace) with torch and
    calls mha_forward."""
    import torch
    b, n_q, d_model = xq.shape
    n_k = xkv.shape[1]
    d_k = wq.shape[1] // h
    d_v = wv.shape[1] // h
    need = mha_workspace_size(b, n_q, n_k, h, d_k, d_v)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=xq.device)
    y = torch.empty((b, n_q, d_model), dtype=xq.dtype, device=xq.device)
    mha_forward(xq, xkv, wq, wk, wv, wo, y, workspace, workspace.numel() * workspace.element_size(),
                b, n_q, n_k, d_model, h, d_k, d_v, mask_kind, kv_lengths, scale, stream)
    return y


def attention_with_lse(q, k, v, mask_kind=SDPA_MASK_NONE, kv_lengths=None, r=0, scale=0.0,
                       stream=None):
    """Allocates out [b,h,n_q,d_v] and lse [b,h,n_q] with torch and calls
    sdpa_forward_lse on bf16 BHSD tensors; returns (out, lse)."""
    import torch
    b, h, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    out = torch.empty((b, h, n_q, d_v), dtype=q.dtype, device=q.device)
    lse = torch.empty((b, h, n_q), dtype=torch.float32, device=q.device)
    sdpa_forward_lse(q, k, v, out, lse, b, h, n_q, n_k, d_k, d_v, mask_kind, kv_lengths, r, scale,
                     stream)
    return out, lse


def attention_backward(q, k, v, out, lse, dout, mask_kind=SDPA_MASK_NONE, kv_lengths=None, r=0,
                       scale=0.0, workspace=None, stream=None):
    """Allocates dq, dk, dv (and, if not given, the workspace) with torch and
    calls sdpa_backward; returns (dq, dk, dv)."""
    import torch
    b, h, n_q, d = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    need = sdpa_backward_workspace_size(b, h, n_q, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    sdpa_backward(q, k, v, out, dout, lse, dq, dk, dv, workspace,
                  workspace.numel() * workspace.element_size(), b, h, n_q, n_k, d, d_v, mask_kind,
                  kv_lengths, r, scale, stream)
    return dq, dk, dv




def sdpa_forward_host(q_host, k_host, v_host, out_host, q_dev, k_dev, v_dev, out_dev, b, h, n_q,
                      n_k, d_k, d_v, mask_kind=SDPA_MASK_NONE, kv_lengths=None, scale=0.0,
                      heads_per_chunk=0, stream=None) -> None:
    """bf16 attention over host buffers, chunked and pipelined inside the
    library (see include/sdpa.h)."""
    _check(load_library().sdpa_forward_host(
        _addr(q_host), _addr(k_host), _addr(v_host), _addr(out_host), _addr(q_dev), _addr(k_dev),
        _addr(v_dev), _addr(out_dev), b, h, n_q, n_k, d_k, d_v, mask_kind, _addr(kv_lengths),
        float(scale), int(heads_per_chunk or 0), _stream(stream)), "sdpa_forward_host")


def attention_from_host(qh, kh, vh, oh, qd, kd, vd, od, mask_kind=SDPA_MASK_NONE, kv_lengths=None,
                        scale=0.0, heads_per_chunk=None, stream=None):
    """Attention over pinned HOST tensors qh/kh/vh [b,h,n,d] bf16 -> oh, with
    qd/kd/vd/od caller-owned device buffers of the same shapes: one call of
    sdpa_forward_host (the library pipelines the chunks' copies and kernels
    on its own streams).  `stream` (default: the current stream) waits for
    the last copy back.  kv_lengths: device int32 [b] or None."""
    b, h, n_q, d_k = qh.shape
    n_k, d_v = kh.shape[2], vh.shape[3]
    sdpa_forward_host(qh, kh, vh, oh, qd, kd, vd, od, b, h, n_q, n_k, d_k, d_v, mask_kind,
                      kv_lengths, scale, heads_per_chunk or 0, stream)
