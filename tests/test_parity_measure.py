"""The parity measures of the GPU tests, checked on the CPU against planted
mistakes made from the oracle's own output.

A long causal output has large first rows (row 0 is the value row V[0]) and
small late rows (rows thousands of keys long average the values down).  The
whole-tensor error max|got - ref| / max|ref| is set by the first rows, so a
mistake confined to late rows stays under its bar; the per-row error holds
each row to its own scale and must reject it.  The mistakes are made with the
oracle itself: a row whose last key tile (the 128-key tile holding the
diagonal) was dropped is the attention of that row over the keys before the
tile, i.e. the oracle with a key-padding length at the tile's start.
"""
import numpy as np

import oracle
import synthetic
from gpu_util import TOL_BF16, parity_err, rel_err, row_err

MASK_CAUSAL, MASK_PADDING = 1, 2
TILE = 128


def _inputs(n=2048, d=128, h=2, seed=4242):
    w = synthetic.Workload("measure_check", 1, h, n, n, d, d, MASK_CAUSAL, "bf16",
                           value_scale=0.5, seed=seed)
    q, k, v, _ = synthetic.sdpa_inputs(w)
    return q, k, v


def _without_diagonal_tile(q, k, v, rows):
    """Rows of head 0 recomputed without the key tile that holds their diagonal."""
    out = {}
    for start in sorted({(i // TILE) * TILE for i in rows}):
        lens = np.array([start], np.int32)
        part = oracle.sdpa(q[:, :1], k[:, :1], v[:, :1], MASK_CAUSAL | MASK_PADDING, lens)
        for i in rows:
            if (i // TILE) * TILE == start:
                out[i] = part[0, 0, i]
    return out


def test_exact_output_passes_both_measures():
    q, k, v = _inputs(n=300, d=64)
    ref = oracle.sdpa(q, k, v, MASK_CAUSAL)
    assert rel_err(ref, ref) == 0.0 and row_err(ref, ref) == 0.0
    # rounding the oracle's output to bf16 stays far inside both bars
    assert parity_err(synthetic.round_to_bf16(ref.astype(np.float32)), ref) <= TOL_BF16 / 4


def test_dropped_diagonal_tile_is_caught_by_the_row_measure_only():
    q, k, v = _inputs()
    ref = oracle.sdpa(q, k, v, MASK_CAUSAL)
    for rows in ([2047], [1000], list(range(1920, 2048))):
        bad = ref.copy()
        for i, row in _without_diagonal_tile(q, k, v, rows).items():
            bad[0, 0, i] = row
        assert rel_err(bad, ref) <= TOL_BF16, rows        # the whole-tensor bar misses it
        assert row_err(bad, ref) > 5 * TOL_BF16, rows     # the per-row bar does not
        assert parity_err(bad, ref) > TOL_BF16


def test_halved_late_rows_are_caught_by_the_row_measure_only():
    """Rows past the middle of the sequence at half their value (a softmax
    denominator counted twice in the later key tiles, say)."""
    q, k, v = _inputs()
    ref = oracle.sdpa(q, k, v, MASK_CAUSAL)
    bad = ref.copy()
    bad[:, :, 1024:] *= 0.5
    assert rel_err(bad, ref) <= TOL_BF16
    assert row_err(bad, ref) >= 0.5 - 1e-12


def test_dropped_tile_moves_the_log_sum_exp_past_its_bar():
    """The log-sum-exp check (1e-3 absolute) sees the dropped tile too: the
    tile's keys carry at least 1/16 of row 2047's weight."""
    q, k, v = _inputs()
    full = oracle.lse(q[:, :1], k[:, :1], MASK_CAUSAL)[0, 0, 2047]
    cut = oracle.lse(q[:, :1], k[:, :1], MASK_CAUSAL | MASK_PADDING, np.array([1920], np.int32))[0, 0, 2047]
    assert full - cut > 1e-2


def test_rows_are_floored_at_the_fp32_bar():
    """A row's scale is floored at 1e-4 of the tensor's: a row that must be
    zero is held to that, and a nearly-zero row is not held to less."""
    ref = np.zeros((2, 3, 4))
    ref[1] = 1.0
    got = ref.copy()
    assert row_err(got, ref) == 0.0
    got[0, 1, 2] = 1e-3     # a row that must be zero is not
    assert abs(row_err(got, ref) - 10.0) < 1e-9
    assert rel_err(got, ref) == 1e-3
    got = ref.copy()
    ref2 = ref.copy()
    ref2[0, 0, 0] = 1e-9    # a row far below the floor, off by 1e-6 of the tensor's scale
    got[0, 0, 0] = 1e-6
    assert abs(row_err(got, ref2) - (1e-6 - 1e-9) / 1e-4) < 1e-12
    # the whole reference zero: absolute
    assert row_err(np.full((2, 3), 1e-3), np.zeros((2, 3))) == 1e-3


def test_gradient_rows_with_a_dropped_tile_are_caught():
    """dQ rows of the last query tile computed without their diagonal key tile
    (the gradient of the attention over the keys before it) fail the per-row
    bar; dK and dV of keys that lost one query's contribution too."""
    q, k, v = _inputs(n=1024, d=64, h=1, seed=77)
    do = synthetic.normal(77, "dout", q.shape)
    dq, dk, dv = oracle.backward(q, k, v, do, MASK_CAUSAL)
    cq, _, _ = oracle.backward(q, k, v, do, MASK_CAUSAL | MASK_PADDING, np.array([896], np.int32))
    bad = dq.copy()
    bad[0, 0, 896:] = cq[0, 0, 896:]
    assert row_err(bad, dq) > 5 * TOL_BF16
    # dV of key 0 without the last query's share (P_{1023,0} dO_1023)
    o_last = oracle.sdpa(q, k, np.eye(1024, dtype=np.float32)[None, None], MASK_CAUSAL,
                         rows=np.array([1023]))[0]
    bad = dv.copy()
    bad[0, 0, 1023] -= o_last[1023] * do[0, 0, 1023]
    assert row_err(bad, dv) >= 1.0 - 1e-9
