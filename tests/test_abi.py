"""The C-ABI library builds, loads and exports every symbol include/sdpa.h
declares; host-side argument checks return their documented codes.

No compute runs here: calls either fail validation on the host or, on a
machine without a GPU, stop at the device check.  Calls that pass placeholder
addresses run only where no GPU is visible.
"""
import ctypes
import os
import re

import pytest

import transformer_scaled_dot_02_gb300 as sd
from transformer_scaled_dot_02_gb300 import build as sd_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa.h")

OK, INVALID, UNSUPPORTED, NODEV, WORKSPACE = 0, 1, 2, 3, 4


def _gpu_visible():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="module")
def lib():
    sd_build.build()
    return sd.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M))


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert names == set(sd.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in sd.STATUS_NAMES.items():
        assert sd.sdpa_status_string(code) == name
    assert sd.sdpa_status_string(99) == "SDPA_ERR_UNKNOWN"


def test_workspace_size_formula(lib):
    def r256(x):
        return (x + 255) // 256 * 256
    for (b, nq, nk, h, dk, dv) in [(32, 128, 128, 8, 64, 64), (32, 256, 384, 16, 64, 64),
                                   (1, 1, 1, 1, 64, 64), (3, 17, 5, 2, 128, 128)]:
        want = r256(b * nq * h * dk * 2) + r256(b * nk * h * dk * 2) + r256(b * nk * h * dv * 2) \
            + r256(b * nq * h * dv * 2)
        assert sd.mha_workspace_size(b, nq, nk, h, dk, dv) == want
    assert sd.mha_workspace_size(-1, 1, 1, 1, 64, 64) == 0


# Placeholder device addresses: 16-byte aligned, never dereferenced because
# every call below is rejected before any CUDA work.
A = 0x10000
MIS = 0x10008


def _attn(lib, fn, **kw):
    args = dict(q=A, k=A, v=A, out=A, b=1, h=1, n_q=16, n_k=16, d_k=64, d_v=64, mask=0,
                lens=None, scale=0.0)
    args.update(kw)
    return getattr(lib, fn)(args["q"], args["k"], args["v"], args["out"], args["b"], args["h"],
                            args["n_q"], args["n_k"], args["d_k"], args["d_v"], args["mask"],
                            args["lens"], ctypes.c_float(args["scale"]), None)


@pytest.mark.parametrize("fn", ["sdpa_forward", "sdpa_forward_f32"])
def test_attention_argument_checks(lib, fn):
    assert _attn(lib, fn, q=None) == INVALID
    assert _attn(lib, fn, out=MIS) == INVALID            # 16-byte alignment
    assert _attn(lib, fn, b=0) == INVALID
    assert _attn(lib, fn, n_q=-1) == INVALID
    assert _attn(lib, fn, d_k=0) == INVALID
    assert _attn(lib, fn, mask=4) == INVALID
    assert _attn(lib, fn, mask=1, n_q=16, n_k=17) == INVALID   # causal needs n_q == n_k
    assert _attn(lib, fn, mask=2, lens=None) == INVALID        # padding needs lengths
    assert _attn(lib, fn, mask=2, lens=A + 2) == INVALID       # int32 alignment
    assert _attn(lib, fn, scale=-1.0) == INVALID
    assert _attn(lib, fn, scale=float("nan")) == INVALID
    assert _attn(lib, fn, scale=float("inf")) == INVALID


def test_restricted_argument_checks(lib):
    def call(**kw):
        a = dict(q=A, out=A, n_q=16, n_k=16, d=64, mask=0, lens=None, r=3)
        a.update(kw)
        return lib.sdpa_forward_restricted(a["q"], A, A, a["out"], 1, 1, a["n_q"], a["n_k"], a["d"],
                                           a["d"], a["mask"], a["lens"], a["r"], ctypes.c_float(0.0),
                                           None)
    assert call(r=0) == INVALID
    assert call(r=-5) == INVALID
    assert call(q=None) == INVALID
    assert call(mask=1, n_k=17) == INVALID
    assert call(d=48) == UNSUPPORTED


def test_decode_argument_checks(lib):
    def call(**kw):
        a = dict(q=A, out=A, ws=A, ws_bytes=1 << 30, b=2, h=2, n_q=1, n_k=4096, d=128, lens=None)
        a.update(kw)
        return lib.sdpa_decode(a["q"], A, A, a["out"], a["ws"], a["ws_bytes"], a["b"], a["h"],
                               a["n_q"], a["n_k"], a["d"], a["d"], a["lens"], ctypes.c_float(0.0),
                               None)
    assert call(q=None) == INVALID
    assert call(out=MIS) == INVALID
    assert call(n_q=0) == INVALID
    assert call(lens=A + 2) == INVALID
    assert call(n_q=9) == UNSUPPORTED
    assert call(d=96) == UNSUPPORTED
    need = sd.sdpa_decode_workspace_size(2, 2, 1, 4096, 128)
    assert need > 0
    assert call(ws=None) == WORKSPACE
    assert call(ws_bytes=need - 1) == WORKSPACE
    # a short cache needs no workspace: one split
    assert sd.sdpa_decode_workspace_size(1024, 16, 1, 256, 128) == 0


def test_unsupported_shapes(lib):
    assert _attn(lib, "sdpa_forward", d_k=48, d_v=48) == UNSUPPORTED
    assert _attn(lib, "sdpa_forward", d_k=8, d_v=8) == UNSUPPORTED
    assert _attn(lib, "sdpa_forward", d_k=64, d_v=128) == UNSUPPORTED
    assert _attn(lib, "sdpa_forward", d_k=384, d_v=384) == UNSUPPORTED
    assert _attn(lib, "sdpa_forward", d_k=1024, d_v=1024) == UNSUPPORTED
    assert _attn(lib, "sdpa_forward", d_k=256, d_v=512) == UNSUPPORTED
    assert _attn(lib, "sdpa_forward", d_k=64, d_v=16) == UNSUPPORTED
    assert _attn(lib, "sdpa_forward", d_k=32, d_v=128) == UNSUPPORTED
    assert _attn(lib, "sdpa_forward_f32", d_k=129, d_v=64) == UNSUPPORTED
    assert _attn(lib, "sdpa_forward_f32", b=70000, h=1) == UNSUPPORTED


def _mha(lib, **kw):
    args = dict(xq=A, xkv=A, wq=A, wk=A, wv=A, wo=A, y=A, ws=A, ws_bytes=1 << 30, b=2, n_q=8,
                n_k=8, d_model=64, h=1, d_k=64, d_v=64, mask=0, lens=None, scale=0.0)
    args.update(kw)
    return lib.mha_forward(args["xq"], args["xkv"], args["wq"], args["wk"], args["wv"],
                           args["wo"], args["y"], args["ws"], args["ws_bytes"], args["b"],
                           args["n_q"], args["n_k"], args["d_model"], args["h"], args["d_k"],
                           args["d_v"], args["mask"], args["lens"], ctypes.c_float(args["scale"]),
                           None)


def test_mha_argument_checks(lib):
    assert _mha(lib, wo=None) == INVALID
    assert _mha(lib, y=MIS) == INVALID
    assert _mha(lib, h=0) == INVALID
    assert _mha(lib, mask=1, n_k=9) == INVALID
    assert _mha(lib, mask=2) == INVALID
    assert _mha(lib, d_k=48, d_v=48) == UNSUPPORTED
    assert _mha(lib, d_model=60) == UNSUPPORTED
    assert _mha(lib, ws=None) == WORKSPACE
    assert _mha(lib, ws=MIS) == WORKSPACE
    need = sd.mha_workspace_size(2, 8, 8, 1, 64, 64)
    assert _mha(lib, ws_bytes=need - 1) == WORKSPACE


def test_linear_argument_checks(lib):
    assert lib.linear_forward(None, A, A, 4, 8, 8, None) == INVALID
    assert lib.linear_forward(A, A, MIS, 4, 8, 8, None) == INVALID
    assert lib.linear_forward(A, A, A, 0, 8, 8, None) == INVALID
    assert lib.linear_forward(A, A, A, 4, 12, 8, None) == UNSUPPORTED
    assert lib.linear_forward(A, A, A, 4, 8, 12, None) == UNSUPPORTED


@pytest.mark.skipif(_gpu_visible(), reason="valid placeholder arguments would reach a real GPU")
def test_valid_arguments_without_gpu_report_no_device(lib):
    assert _attn(lib, "sdpa_forward") == NODEV
    assert _attn(lib, "sdpa_forward", d_k=16, d_v=64) == NODEV    # Table 3, row (B)
    assert _attn(lib, "sdpa_forward", d_k=512, d_v=512) == NODEV
    assert _attn(lib, "sdpa_forward_f32", d_k=1, d_v=1) == NODEV
    assert lib.sdpa_forward_restricted(A, A, A, A, 1, 1, 16, 16, 64, 64, 0, None, 3,
                                       ctypes.c_float(0.0), None) == NODEV
    assert _mha(lib) == NODEV
    assert lib.linear_forward(A, A, A, 4, 8, 8, None) == NODEV
    assert lib.sdpa_decode(A, A, A, A, A, 1 << 30, 2, 2, 1, 4096, 128, 128, None,
                           ctypes.c_float(0.0), None) == NODEV
    assert lib.sdpa_device_check() == NODEV


def test_kernel_choice_accepts_only_documented_values(lib):
    """sdpa_set_kernel_choice is host-only: valid pins are taken, others
    rejected with SDPA_ERR_INVALID_ARG; the test leaves every choice to the
    shapes again."""
    try:
        for args in [(0, 0, 0), (1, 0, 0), (2, 32, 0), (1, 64, 256), (0, 0, 128)]:
            assert lib.sdpa_set_kernel_choice(*args) == OK, args
        for args in [(3, 0, 0), (-1, 0, 0), (0, 16, 0), (0, 128, 0), (0, 0, 64), (0, 0, 512)]:
            assert lib.sdpa_set_kernel_choice(*args) == INVALID, args
    finally:
        assert lib.sdpa_set_kernel_choice(0, 0, 0) == OK


def test_noalloc_limit_matches_the_header():
    """The binding's copy of the static workspace size is the header's value."""
    text = open(HEADER).read()
    m = re.search(r"#define\s+SDPA_MHA_NOALLOC_MAX_WORKSPACE\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "SDPA_MHA_NOALLOC_MAX_WORKSPACE not found"
    assert int(m.group(1)) << int(m.group(2)) == sd.MHA_NOALLOC_MAX_WORKSPACE


def test_host_pipeline_argument_checks(lib):
    """sdpa_forward_host: null host pointers and a negative chunk size are
    rejected on the host; valid arguments stop at the device check here."""
    def call(**kw):
        a = dict(qh=A, kh=A, vh=A, oh=A, hc=0, d=64)
        a.update(kw)
        return lib.sdpa_forward_host(a["qh"], a["kh"], a["vh"], a["oh"], A, A, A, A, 2, 4, 128, 128,
                                     a["d"], a["d"], 0, None, ctypes.c_float(0.0), a["hc"], None)
    assert call(qh=None) == INVALID
    assert call(oh=None) == INVALID
    assert call(hc=-1) == INVALID
    assert call(d=48) == UNSUPPORTED
    if not _gpu_visible():
        assert call() == NODEV
