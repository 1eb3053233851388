"""Helpers shared by the GPU parity tests: device copies and the error
measure.  The error is max|gpu - ref| / max|ref| over the compared entries
(absolute error relative to the output scale); the bars are 1e-4 for fp32
inputs and 2e-2 for bf16 inputs with fp32 accumulation."""
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


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite output"
    scale = np.abs(ref).max()
    if scale == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / scale)
