"""Invariant pins for the oracle's OsciReset statistics and window-end reset
("Resumo Técnico: TetraJet-v2", §2B: dist_M accumulates the master weight's
movement, dist_Q the movement of its quantized value; at the end of a window a
weight whose ratio dist_Q / dist_M exceeds the threshold goes back to its
current quantized value and the statistics restart).

Each check follows from that definition alone, with the tensor quantizer (pinned
elsewhere) as a step:
  - no update moves nothing and resets nothing;
  - on a grid where every FP32 sum is exact, dist_M is the sum of |delta|;
  - dist_Q is the running sum of |xhat_t - xhat_(t-1)| over the quantizer's
    own outputs;
  - the reset moves exactly the weights with dist_Q > threshold * dist_M, to
    the last xhat, clears both statistics, and a second reset moves nothing.
"""
import numpy as np
import pytest

import oracle

FMTS = [oracle.NVFP4, oracle.MXFP4, oracle.NVFP4_2LEVEL]


def _grid_weights(rows, cols, seed):
    """Weights and updates that are small multiples of 2^-8: every FP32 sum
    and difference below stays exact."""
    g = np.random.default_rng(seed)
    w0 = (g.integers(-512, 513, (rows, cols)) * 2.0 ** -8).astype(np.float32)
    deltas = [(g.integers(-3, 4, (rows, cols)) * 2.0 ** -8).astype(np.float32)
              for _ in range(6)]
    return w0, deltas


@pytest.mark.parametrize("fmt", FMTS)
def test_no_update_moves_nothing(fmt):
    w0, _ = _grid_weights(16, 256, 1)
    st = oracle.OsciState(w0, fmt)
    codes0, scales0 = st.codes.copy(), st.scales.copy()
    for t in range(1, 4):
        st.step(np.zeros_like(w0), offset=t)
    assert not st.dist_m.any() and not st.dist_q.any()
    assert np.array_equal(st.codes, codes0) and np.array_equal(st.scales, scales0)
    assert np.array_equal(st.master.view(np.uint32), w0.view(np.uint32))
    assert st.reset(4.0) == 0
    assert np.array_equal(st.master.view(np.uint32), w0.view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rounding", [oracle.RNE, oracle.SR])
def test_statistics_follow_their_definition(fmt, rounding):
    rows, cols = 16, 256
    w0, deltas = _grid_weights(rows, cols, 2)
    seed = 9
    st = oracle.OsciState(w0, fmt, rounding, seed)
    # the quantizer's own outputs, step by step (offset 0 at initialisation)
    w = w0.copy()
    xh_prev = oracle.quantize(w, fmt, rounding, seed, 0, want_xhat=True)["row"]["xhat"]
    dq = np.zeros_like(w0)
    for t, d in enumerate(deltas, start=1):
        out = st.step(d, offset=t)
        w = (w + d).astype(np.float32)
        xh = oracle.quantize(w, fmt, rounding, seed, t, want_xhat=True)["row"]["xhat"]
        assert np.array_equal(out["xhat"].view(np.uint32), xh.view(np.uint32))
        dq = (dq + np.abs(xh - xh_prev)).astype(np.float32)
        xh_prev = xh
    dm_exact = sum(np.abs(d.astype(np.float64)) for d in deltas)
    assert np.array_equal(st.master.view(np.uint32), w.view(np.uint32))
    assert np.array_equal(st.dist_m.astype(np.float64), dm_exact)
    assert np.array_equal(st.dist_q.view(np.uint32), dq.view(np.uint32))

    # the window-end reset
    thr = np.float32(4.0)
    hit = st.dist_q > (thr * st.dist_m).astype(np.float32)
    assert hit.any() and not hit.all()
    master_before = st.master.copy()
    n = st.reset(float(thr))
    assert n == int(hit.sum())
    assert np.array_equal(st.master[hit].view(np.uint32), xh_prev[hit].view(np.uint32))
    assert np.array_equal(st.master[~hit].view(np.uint32), master_before[~hit].view(np.uint32))
    assert not st.dist_q.any() and not st.dist_m.any()
    assert st.reset(float(thr)) == 0
