"""fp32 attention on the CUDA cores against the oracle (tolerance 1e-4
relative to the output scale), and the pages' worked examples exactly."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synthetic
import transformer_scaled_dot_02_gb300 as sd
from gpu_util import TOL_F32, dev, dev_int, host, parity_err

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sd.load_library()


def _run(q, k, v, mask=0, lens=None, scale=0.0):
    t = sd.attention(dev(q, "f32"), dev(k, "f32"), dev(v, "f32"), mask,
                     None if lens is None else dev_int(lens), scale)
    sd.sdpa_device_check()
    return host(t)


@pytest.mark.parametrize("name", ["tiny_f32", "tiny_f32_causal"])
def test_tiny_config(name):
    w = synthetic.WORKLOADS[name]
    q, k, v, lens = synthetic.sdpa_inputs(w)
    got = _run(q, k, v, w.mask_kind, lens)
    ref = oracle.sdpa(q, k, v, w.mask_kind, lens)
    assert parity_err(got, ref) <= TOL_F32


def test_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_dk1.json")))
    q = np.array([[[g["q"]]]], np.float32)
    k = np.array([[[[math.log(3.0)], [0.0]]]], np.float32)
    v = np.array([[[[2.0], [6.0]]]], np.float32)
    out = _run(q, k, v)
    assert abs(out[0, 0, 0, 0] - g["output"]) < 1e-6
    w = _run(q, k, np.eye(2, dtype=np.float32)[None, None])
    assert np.allclose(w[0, 0, 0], g["weights"], atol=1e-6)
    masked = _run(q, k, v, sd.SDPA_MASK_PADDING, np.array([1], np.int32))
    assert masked[0, 0, 0, 0] == g["masked_second_key"]["output"]
    causal = _run(np.ones((1, 1, 2, 1), np.float32), k, v, sd.SDPA_MASK_CAUSAL)
    assert causal[0, 0, 0, 0] == g["masked_second_key"]["output"]
    assert abs(causal[0, 0, 1, 0] - g["output"]) < 1e-6


def test_toy_rows():
    g = json.load(open(os.path.join(GOLDEN, "toy_rows_fig2.json")))
    vals = np.array(g["values"], np.float32).reshape(1, 1, -1, 1)
    for row in g["rows"]:
        k = np.log(np.array(row["weights"], np.float32)).reshape(1, 1, -1, 1)
        out = _run(np.ones((1, 1, 1, 1), np.float32), k, vals, scale=1.0)
        assert abs(out[0, 0, 0, 0] - row["output"]) < 1e-4


@pytest.mark.parametrize("d_k,d_v", [(1, 1), (3, 5), (64, 64), (100, 37), (128, 128)])
@pytest.mark.parametrize("mask", [0, 1, 2, 3])
def test_shapes_and_masks(d_k, d_v, mask):
    rng = np.random.default_rng(100 + d_k + 7 * mask)
    b, h, n = 2, 3, 45
    n_q = n
    n_k = n if mask & 1 else 61
    q = rng.standard_normal((b, h, n_q, d_k)).astype(np.float32)
    k = rng.standard_normal((b, h, n_k, d_k)).astype(np.float32)
    v = rng.standard_normal((b, h, n_k, d_v)).astype(np.float32)
    lens = np.array([n_k, 7], np.int32) if mask & 2 else None
    got = _run(q, k, v, mask, lens)
    ref = oracle.sdpa(q, k, v, mask, lens)
    assert parity_err(got, ref) <= TOL_F32


def test_degenerate_lengths():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((3, 1, 20, 8)).astype(np.float32)
    k = rng.standard_normal((3, 1, 33, 8)).astype(np.float32)
    v = rng.standard_normal((3, 1, 33, 8)).astype(np.float32)
    lens = np.array([0, 1, 99], np.int32)       # none visible, one, clamped to n_k
    got = _run(q, k, v, sd.SDPA_MASK_PADDING, lens)
    ref = oracle.sdpa(q, k, v, sd.SDPA_MASK_PADDING, lens)
    assert np.array_equal(got[0], np.zeros_like(got[0]))
    assert parity_err(got, ref) <= TOL_F32
