"""Property-based pins of the oracle over random small shapes (hypothesis):
each property is fixed by the pages' definitions or by plain library routines,
never by the oracle itself.

  layout     UBEP section 2.3 / StrataCL Appendix D: counts are a bincount,
             offsets its exclusive cumsum, and the slot order is the stable
             sort of the flattened expert ids
  dispatch   every receive row is its source token's row
  combine    HyperParallel-MoE section 2.2: within the fp32 bound of the
             binary64 weighted sum
  coalesced  RailWave section 3.1: one row per distinct (rank, token), rank
             segments in token order; the pre-reduced rows of small-integer
             payloads sum exactly
"""
import numpy as np
import pytest

import oracle

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

SETTINGS = settings(max_examples=60, deadline=None)


@st.composite
def routing(draw):
    R = draw(st.integers(1, 6))
    El = draw(st.integers(1, 5))
    E = R * El
    T = draw(st.integers(0, 40))
    k = draw(st.integers(1, 6))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, E, (T, k)).astype(np.int32)
    return T, k, E, R, idx, rng


@SETTINGS
@given(routing())
def test_layout_is_a_stable_counting_sort(case):
    T, k, E, R, idx, _ = case
    counts, offs, roffs, slot_of, src_of = oracle.layout(idx, E, R)
    flat = idx.ravel()
    assert counts.tolist() == np.bincount(flat, minlength=E).tolist()
    assert offs.tolist() == [0] + np.cumsum(np.bincount(flat, minlength=E)).tolist()
    assert roffs.tolist() == offs[:: E // R].tolist()
    order = np.argsort(flat, kind="stable")
    assert np.array_equal(src_of, order)
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    assert np.array_equal(slot_of.ravel(), inv)


@SETTINGS
@given(routing(), st.integers(1, 4))
def test_dispatch_rows_are_source_rows(case, h8):
    T, k, E, R, idx, rng = case
    H = 8 * h8
    x = rng.integers(0, 1 << 16, (T, H)).astype(np.uint16)
    _, _, _, slot_of, src_of = oracle.layout(idx, E, R)
    recv = oracle.dispatch(x, slot_of)
    assert np.array_equal(recv, x[src_of // k]) if T else recv.size == 0


@SETTINGS
@given(routing())
def test_combine_within_fp32_bound(case):
    T, k, E, R, idx, rng = case
    H = 16
    _, _, _, slot_of, _ = oracle.layout(idx, E, R)
    yv = rng.standard_normal((T * k, H)).astype(np.float32)
    y = (yv.view(np.uint32) >> 16).astype(np.uint16)         # truncation: any bf16 will do
    w = rng.random((T, k), dtype=np.float32)
    out = oracle.combine(y, slot_of, w, "f32")
    yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    terms = w.astype(np.float64)[:, :, None] * yf[slot_of] if T else np.zeros((0, k, H))
    exact = terms.sum(axis=1)
    bound = k * 2.0 ** -24 / (1 - k * 2.0 ** -24) * np.abs(terms).sum(axis=1)
    assert np.all(np.abs(out - exact) <= bound)


@SETTINGS
@given(routing())
def test_coalesced_rows_are_distinct_rank_token_pairs(case):
    T, k, E, R, idx, rng = case
    El = E // R
    _, _, _, slot_of, _ = oracle.layout(idx, E, R)
    counts, offs, crow, src, expand = oracle.layout_coalesced(idx, E, R, slot_of)
    pairs = sorted({(int(e) // El, t) for t in range(T) for e in idx[t]})
    assert int(offs[-1]) == len(pairs)
    assert [(int(idx.ravel()[p]) // El, int(p) // k) for p in src] == pairs
    for t in range(T):
        for j in range(k):
            r = int(idx[t, j]) // El
            assert crow[t, j] == pairs.index((r, t))
    assert np.array_equal(expand[slot_of.ravel()], crow.ravel())


@SETTINGS
@given(routing())
def test_coalesced_combine_of_integer_payload_is_exact(case):
    T, k, E, R, idx, rng = case
    H = 8
    _, _, _, slot_of, _ = oracle.layout(idx, E, R)
    _, offs, crow, _, _ = oracle.layout_coalesced(idx, E, R, slot_of)
    yv = rng.integers(-4, 5, (T * k, H)).astype(np.float32)
    y = (yv.view(np.uint32) >> 16).astype(np.uint16)          # small integers are exact in bf16
    w = rng.choice(np.array([0.5, 1.0, 2.0], np.float32), (T, k))
    part = oracle.combine_coalesced_pre(y, slot_of, w, crow, int(offs[-1]))
    out = oracle.combine_coalesced_post(part, crow, "f32")
    exact = (w[:, :, None].astype(np.float64) * yv[slot_of]).sum(axis=1) if T else np.zeros((0, H))
    assert np.array_equal(out.astype(np.float64), exact)
