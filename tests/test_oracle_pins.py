"""The CPU oracle against values and properties fixed by the pages and by
mathematics (see oracle_pins.py for the source of each pin)."""
import numpy as np
import pytest

import oracle
import synthetic
from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle.default())


def test_oracle_rejects_bad_arguments():
    q = np.zeros((1, 1, 3, 2), np.float32)
    k = np.zeros((1, 1, 4, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.sdpa(q, k, k, oracle.MASK_CAUSAL)        # causal needs n_q == n_k
    with pytest.raises(ValueError):
        oracle.sdpa(q, k, k, oracle.MASK_PADDING, None)  # padding needs lengths


def test_threads_do_not_change_results():
    w = synthetic.WORKLOADS["dec_causal_base"]
    q, k, v, _ = synthetic.sdpa_inputs(w, b=1, h=2)
    one = oracle.sdpa(q[:, :, :64], k[:, :, :64], v[:, :, :64], oracle.MASK_CAUSAL, threads=1)
    many = oracle.sdpa(q[:, :, :64], k[:, :, :64], v[:, :, :64], oracle.MASK_CAUSAL, threads=5)
    assert np.array_equal(one, many)


def test_generator_score_variance():
    """Footnote to Eq. (1): for independent N(0,1) components q.k has variance
    d_k, so q.k / sqrt(d_k) has variance 1 on the synthetic inputs."""
    for name in ("dec_causal_base", "long_causal"):
        w = synthetic.WORKLOADS[name]
        q = synthetic.normal(w.seed, "q", (4096, w.d_k), 1.0, w.dtype).astype(np.float64)
        k = synthetic.normal(w.seed, "k", (4096, w.d_k), 1.0, w.dtype).astype(np.float64)
        s = (q * k).sum(1) / np.sqrt(w.d_k)
        assert abs(s.var() - 1.0) < 0.08, s.var()
        assert abs(s.mean()) < 0.05


def test_generator_is_deterministic_and_bf16_exact():
    w = synthetic.WORKLOADS["enc_mha_base"]
    a = synthetic.mha_inputs(w)
    b = synthetic.mha_inputs(w)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    bits = a[0].view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0)          # bf16 values in float32 storage
    lens = a[-1]
    assert lens.min() >= 64 and lens.max() <= 128 and lens.shape == (32,)
