"""Pins for the oracle's expert parallelism across W real ranks.

UBEP section 2.3 / Figure 2 and section 4: each receiver's region is
partitioned by source rank and expert, and Phase 5 reorders the tokens
contiguously per expert using the per-source counts.  StrataCL Appendix D:
counts and token-local offsets are the metadata combine reuses.  Reading: a
receiver holds, per local expert, the rows of source 0, source 1, ..., each in
the source's (token, slot) order.

Pins, none of which calls the function it pins:
  * numpy's stable argsort of all ranks' ids, concatenated rank by rank, is
    the receive order: the receive buffers laid end to end are the single-GPU
    stable order (expert, global token, slot), cut at the ranks' first experts;
  * per-source bincounts give the counts each receiver gets;
  * a Python sort of (local expert, source, t, j) tuples on tiny inputs;
  * the combine: float64 closed form within the fp32 bound, and the
    identity-expert round trip with weights summing to one returns x.
"""
import numpy as np
import pytest

import oracle
from workloads.gen import random_case, make_workload, bf16_bits_to_f32

U = 2.0 ** -24


def ranks(seed, W, T_per, H, k, E):
    """W ranks' inputs; T_per gives each rank's token count (0 allowed)."""
    out = []
    for s, T in enumerate(T_per):
        w = random_case(seed * 100 + s, T, H, k, E, W)
        out.append(w)
    return out


CASES = [  # (seed, W, tokens per rank, H, k, E)
    (1, 2, [5, 7], 16, 2, 4),
    (2, 4, [30, 0, 17, 9], 8, 3, 8),
    (3, 3, [40, 40, 40], 24, 8, 12),
    (4, 8, [64] * 8, 8, 2, 8),
    (5, 1, [50], 16, 4, 6),
    (6, 2, [1, 1], 8, 1, 2),
]


@pytest.mark.parametrize("case", CASES, ids=[f"W{c[1]}_k{c[4]}_E{c[5]}" for c in CASES])
def test_receive_buffers_are_the_stable_order_of_all_tokens(case):
    seed, W, T_per, H, k, E = case
    rk = ranks(seed, W, T_per, H, k, E)
    counts, recv, src = oracle.ep_dispatch([r.topk_idx for r in rk], [r.x for r in rk], E)
    idx = np.concatenate([r.topk_idx for r in rk]).reshape(-1)
    x = np.concatenate([r.x for r in rk])
    order = np.argsort(idx, kind="stable")           # global pair ids in receive order
    El = E // W
    cuts = np.searchsorted(idx[order], np.arange(W + 1) * El, side="left")
    for d in range(W):
        want = order[cuts[d]:cuts[d + 1]]
        assert np.array_equal(src[d], want)
        assert np.array_equal(recv[d], x[want // k])


@pytest.mark.parametrize("case", CASES, ids=[f"W{c[1]}_k{c[4]}_E{c[5]}" for c in CASES])
def test_counts_are_per_source_bincounts(case):
    seed, W, T_per, H, k, E = case
    rk = ranks(seed, W, T_per, H, k, E)
    counts, recv, _ = oracle.ep_dispatch([r.topk_idx for r in rk], [r.x for r in rk], E)
    El = E // W
    assert counts.shape == (W, W, El)
    for s, r in enumerate(rk):
        bc = np.bincount(r.topk_idx.reshape(-1), minlength=E)
        for d in range(W):
            assert np.array_equal(counts[d, s], bc[d * El:(d + 1) * El])
    for d in range(W):
        assert counts[d].sum() == len(recv[d])


def test_receiver_order_brute_force():
    W, E, k = 3, 6, 2
    rk = ranks(9, W, [4, 3, 5], 8, k, E)
    _, recv, src = oracle.ep_dispatch([r.topk_idx for r in rk], [r.x for r in rk], E)
    El = E // W
    base = np.cumsum([0] + [r.T for r in rk])
    for d in range(W):
        rows = []
        for s, r in enumerate(rk):
            for t in range(r.T):
                for j in range(k):
                    e = int(r.topk_idx[t, j])
                    if e // El == d:
                        rows.append((e % El, s, t, j))
        rows.sort()
        assert [int(v) for v in src[d]] == [(base[s] + t) * k + j for _, s, t, j in rows]


def test_hand_worked_two_ranks():
    """W = 2, E = 4 (experts 0, 1 on rank 0; 2, 3 on rank 1), k = 2.
    rank 0: t0 -> (2, 0), t1 -> (1, 2);  rank 1: t0 -> (0, 3), t1 -> (2, 2).
    Receiver 0, expert 0: r0.t0.j1, r1.t0.j0; expert 1: r0.t1.j0.
    Receiver 1, expert 2: r0.t0.j0, r0.t1.j1, r1.t1.j0, r1.t1.j1; expert 3: r1.t0.j1."""
    i0 = np.array([[2, 0], [1, 2]], np.int32)
    i1 = np.array([[0, 3], [2, 2]], np.int32)
    x0 = np.array([[1], [2]], np.uint16)
    x1 = np.array([[3], [4]], np.uint16)
    counts, recv, src = oracle.ep_dispatch([i0, i1], [x0, x1], 4)
    assert src[0].tolist() == [1, 4, 2]
    assert src[1].tolist() == [0, 3, 6, 7, 5]
    assert recv[0].ravel().tolist() == [1, 3, 2]
    assert recv[1].ravel().tolist() == [1, 2, 4, 4, 3]
    assert counts[0].tolist() == [[1, 1], [1, 0]]     # receiver 0: [source][local expert]
    assert counts[1].tolist() == [[2, 0], [2, 1]]


@pytest.mark.parametrize("case", CASES, ids=[f"W{c[1]}_k{c[4]}_E{c[5]}" for c in CASES])
def test_combine_within_fp32_bound_of_exact(case):
    seed, W, T_per, H, k, E = case
    rk = ranks(seed, W, T_per, H, k, E)
    _, recv, src = oracle.ep_dispatch([r.topk_idx for r in rk], [r.x for r in rk], E)
    rng = np.random.default_rng(seed)
    y = [((rng.integers(0, 1 << 16, size=a.shape, dtype=np.uint32) & 0xBFFF) | 0x3C00)
         .astype(np.uint16) for a in recv]           # finite, |y| in [2^-7, 2^1)
    outs = oracle.ep_combine([r.topk_idx for r in rk], [r.topk_w for r in rk], y, E, "f32")
    # float64 closed form: row of pair i is found through the dispatch's src_pair
    allsrc = np.concatenate(src)
    ally = np.concatenate(y).reshape(-1, H) if len(allsrc) else np.zeros((0, H), np.uint16)
    row_of = np.empty(len(allsrc), np.int64)
    row_of[allsrc] = np.arange(len(allsrc))
    w = np.concatenate([r.topk_w for r in rk]).reshape(-1, k).astype(np.float64)
    yv = bf16_bits_to_f32(ally).astype(np.float64)
    T = w.shape[0]
    terms = w[:, :, None] * yv[row_of.reshape(T, k)] if T else np.zeros((0, k, H))
    exact, mag = terms.sum(axis=1), np.abs(terms).sum(axis=1)
    got = np.concatenate(outs).astype(np.float64) if T else np.zeros((0, H))
    gamma = k * U / (1 - k * U)
    assert np.all(np.abs(got - exact) <= gamma * mag)


@pytest.mark.parametrize("name,T", [("mixtral", 96), ("dsv3_decode", 24), ("glm45_air", 32)])
def test_identity_expert_round_trip(name, T):
    """Each rank's tokens come back to it: with the received rows as the
    experts' outputs and weights summing to one (within fp32), the combine
    returns every rank's x (x * (1 +- few 2^-24) rounds back to x)."""
    W = 4
    rk = [make_workload(name, seed=s, T=T) for s in range(W)]
    E = rk[0].E
    _, recv, _ = oracle.ep_dispatch([r.topk_idx for r in rk], [r.x for r in rk], E)
    outs = oracle.ep_combine([r.topk_idx for r in rk], [r.topk_w for r in rk], recv, E)
    for r, o in zip(rk, outs):
        nz = (r.x & 0x7FFF) != 0
        assert np.array_equal(o[nz], r.x[nz])
        assert np.all(bf16_bits_to_f32(o[~nz]) == 0)


def test_out_of_range_id_is_rejected():
    i0 = np.array([[0, 4]], np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.ep_dispatch([i0, i0], [np.zeros((1, 8), np.uint16)] * 2, 4)


def test_combine_accumulates_in_slot_order():
    """k = 3, unit weights, the token's rows hold (2^25, -2^25, 1) in slot
    order on two receivers: fp32 in slot order gives 0 + 1 = 1; the reverse
    order would give 1 - 2^25 = -2^25 (rounded), then 0."""
    big = np.float32(2.0 ** 25)
    i0 = np.array([[0, 2, 3]], np.int32)            # expert 0 on rank 0; 2, 3 on rank 1
    i1 = np.zeros((0, 3), np.int32)
    w = [np.ones((1, 3), np.float32), np.ones((0, 3), np.float32)]
    bits = lambda v: (np.array([[v]], np.float32).view(np.uint32) >> 16).astype(np.uint16)  # noqa: E731
    y = [bits(big), np.concatenate([bits(-big), bits(1.0)])]
    out = oracle.ep_combine([i0, i1], w, y, 4, "f32")
    assert out[0][0, 0] == 1.0
