"""Pins for the oracle's layout (count -> exclusive scan -> stable slot map).

What the layout must be is fixed by the pages (UBEP section 2.3: per-expert
counts, offsets, contiguous per-expert reordering; StrataCL Appendix D:
per-expert counts, prefix-sum offsets, token-local offsets) plus the stated
order inside an expert (source token, then k slot).  These tests check the
oracle against library routines and brute force, never against itself.
"""
import numpy as np
import pytest

import oracle
from workloads.gen import CONFIG_ORDER, make_workload, random_case


def _cases():
    out = []
    for name in CONFIG_ORDER:
        w = make_workload(name)
        out.append((name, w.topk_idx, w.E, w.R))
    for s, (T, k, E, R) in enumerate([(1, 1, 1, 1), (1, 8, 4, 2), (7, 3, 5, 5), (33, 2, 16, 4),
                                      (100, 8, 8, 1), (257, 4, 256, 32), (64, 6, 3, 3)]):
        w = random_case(100 + s, T, 16, k, E, R)
        out.append((f"fuzz{s}", w.topk_idx, E, R))
    return out


CASES = _cases()


@pytest.mark.parametrize("name,idx,E,R", CASES, ids=[c[0] for c in CASES])
def test_counts_and_offsets_match_library(name, idx, E, R):
    counts, offs, roffs, _, _ = oracle.layout(idx, E, R)
    ref = np.bincount(idx.ravel(), minlength=E)
    assert np.array_equal(counts, ref)
    assert counts.sum() == idx.size
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(ref)]))
    assert np.all(np.diff(offs) >= 0) and offs[-1] == idx.size
    assert np.array_equal(roffs, offs[:: E // R])


@pytest.mark.parametrize("name,idx,E,R", CASES, ids=[c[0] for c in CASES])
def test_slot_map_is_stable_counting_sort(name, idx, E, R):
    """The stable order (expert, token, slot) is a stable sort of the flattened
    expert ids: src_of is numpy's stable argsort, slot_of its inverse."""
    _, _, _, slot_of, src_of = oracle.layout(idx, E, R)
    flat = idx.ravel()
    ref = np.argsort(flat, kind="stable").astype(np.int32)
    assert np.array_equal(src_of, ref)
    inv = np.empty_like(ref)
    inv[ref] = np.arange(flat.size, dtype=np.int32)
    assert np.array_equal(slot_of.ravel(), inv)
    # every (token, slot) pair appears exactly once
    assert np.array_equal(np.sort(slot_of.ravel()), np.arange(flat.size))


@pytest.mark.parametrize("name,idx,E,R", [c for c in CASES if c[1].size <= 4096],
                         ids=[c[0] for c in CASES if c[1].size <= 4096])
def test_slot_map_brute_force(name, idx, E, R):
    """O(N^2) definition: slot = offset(e) + #earlier pairs (lexicographic) with e."""
    counts, offs, _, slot_of, _ = oracle.layout(idx, E, R)
    flat = idx.ravel().astype(np.int64)
    n = flat.size
    same = flat[None, :] == flat[:, None]
    earlier = np.arange(n)[None, :] < np.arange(n)[:, None]
    rank = (same & earlier).sum(axis=1)
    below = np.array([(flat < e).sum() for e in flat])
    assert np.array_equal(slot_of.ravel(), below + rank)


@pytest.mark.parametrize("name,idx,E,R", CASES, ids=[c[0] for c in CASES])
def test_rank_segments_hold_their_experts(name, idx, E, R):
    _, offs, roffs, _, src_of = oracle.layout(idx, E, R)
    flat = idx.ravel()
    El = E // R
    exp_of_slot = flat[src_of]
    assert np.all(np.diff(exp_of_slot) >= 0)          # expert-contiguous
    for r in range(R):
        seg = exp_of_slot[roffs[r]:roffs[r + 1]]
        assert np.all((seg >= r * El) & (seg < (r + 1) * El))
    for e in range(E):                                   # source order inside an expert
        assert np.all(np.diff(src_of[offs[e]:offs[e + 1]]) > 0)


def test_hand_worked_example():
    # T=3 tokens, k=2, E=4 experts on R=2 ranks (experts 0,1 on rank 0; 2,3 on rank 1)
    idx = np.array([[2, 0], [1, 2], [0, 0]], np.int32)
    counts, offs, roffs, slot_of, src_of = oracle.layout(idx, 4, 2)
    assert counts.tolist() == [3, 1, 2, 0]
    assert offs.tolist() == [0, 3, 4, 6, 6]
    assert roffs.tolist() == [0, 4, 6]
    # expert 0 receives (t0,j1), (t2,j0), (t2,j1) -> slots 0,1,2; expert 1: (t1,j0) -> 3;
    # expert 2: (t0,j0), (t1,j1) -> 4,5
    assert slot_of.tolist() == [[4, 0], [3, 5], [1, 2]]
    assert src_of.tolist() == [1, 4, 5, 2, 0, 3]


def test_duplicate_expert_in_one_token():
    idx = np.array([[1, 1, 1], [0, 1, 0]], np.int32)
    counts, offs, _, slot_of, _ = oracle.layout(idx, 2, 1)
    assert counts.tolist() == [2, 4]
    assert slot_of.tolist() == [[2, 3, 4], [0, 5, 1]]


def test_empty_input():
    idx = np.zeros((0, 4), np.int32)
    counts, offs, roffs, slot_of, src_of = oracle.layout(idx, 8, 2)
    assert counts.tolist() == [0] * 8 and offs.tolist() == [0] * 9 and roffs.tolist() == [0] * 3
    assert slot_of.shape == (0, 4) and src_of.shape == (0,)


@pytest.mark.parametrize("bad", [-1, 8, 1 << 30])
def test_bad_index_rejected(bad):
    idx = np.array([[0, 1], [2, bad]], np.int32)
    with pytest.raises(oracle.OracleError) as ei:
        oracle.layout(idx, 8, 2)
    assert ei.value.status == oracle.ERR_BAD_INDEX


def test_experts_not_divisible_by_ranks_rejected():
    with pytest.raises(oracle.OracleError) as ei:
        oracle.layout(np.zeros((2, 2), np.int32), 6, 4)
    assert ei.value.status == oracle.ERR_INVALID_ARG
