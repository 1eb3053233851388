"""Helpers shared by the GPU parity tests: device copies and the error
measures.

Two measures, both held to the same bar (1e-4 for fp32 inputs, 2e-2 for bf16
inputs with fp32 accumulation):
  - whole tensor: max|gpu - ref| / max|ref| over the compared entries, the
    absolute error relative to the output's scale;
  - per row: for every row i (every index but the last: one query's output
    row, or one key's row of dK and dV), max_c|gpu_ic - ref_ic| / s_i with
    s_i = max(max_c|ref_ic|, 1e-4 max|ref|).  The floor is the fp32 bar: a
    row whose exact value is far below its terms (a one-hot softmax row of
    dQ, where dS cancels to about 1e-6 of the tensor's scale) keeps the fp32
    rounding of those terms, about 1e-7 of the tensor's scale, and no
    arithmetic resolves it further.  A row that must be zero (a query that
    sees no key, a hidden key) is thereby held to 1e-4 of the tensor's scale
    times the bar.
The whole-tensor figure alone is set by the largest rows.  In a long causal
output the first rows are single value rows (|O| about max|V|) while rows
thousands of keys long average down to a few hundredths of that, so a dropped
key tile or a zeroed row far down the sequence would pass it.  The per-row
figure holds every row to its own scale.
"""
import numpy as np

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def torch():
    import torch as _t
    return _t


def dev(a, dtype="bf16"):
    t = torch()
    x = t.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if dtype == "bf16":
        x = x.to(t.bfloat16)
    return x.cuda()


def dev_int(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host(x):
    return x.float().cpu().numpy().astype(np.float64)


def _pair(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite output"
    return got, ref


def rel_err(got, ref):
    """Whole-tensor error: max|got - ref| / max|ref| (absolute if ref is 0)."""
    got, ref = _pair(got, ref)
    scale = np.abs(ref).max() if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    if scale == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / scale)


ROW_FLOOR = 1e-4   # floor of a row's scale, as a fraction of the tensor's


def row_errs(got, ref):
    """Per-row errors: max_c|got_ic - ref_ic| / max(max_c|ref_ic|, ROW_FLOOR
    max|ref|) for every row (absolute if the whole reference is 0),
    flattened over the leading axes."""
    got, ref = _pair(got, ref)
    if ref.size == 0:
        return np.zeros(0)
    g = got.reshape(-1, got.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    scale = np.maximum(np.abs(r).max(axis=1), ROW_FLOOR * np.abs(r).max())
    err = np.abs(g - r).max(axis=1)
    return np.where(scale > 0, err / np.where(scale > 0, scale, 1.0), err)


def row_err(got, ref):
    """The largest per-row error."""
    e = row_errs(got, ref)
    return float(e.max()) if e.size else 0.0


def parity_err(got, ref):
    """The larger of the whole-tensor and the per-row error; the parity bar
    applies to this figure."""
    return max(rel_err(got, ref), row_err(got, ref))
