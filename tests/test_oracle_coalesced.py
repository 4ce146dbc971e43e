"""Pins for the oracle's rank-coalesced layout and dispatch: one receive row per
(token, distinct destination rank) (UBEP section 2.3: a token may go to
several experts; RailWave section 3.1: token coalescing), checked against a
set-based numpy brute force and invariants, never against itself."""
import numpy as np
import pytest

import oracle
from workloads.gen import CONFIG_ORDER, make_workload, random_case


def _cases():
    out = []
    for name in CONFIG_ORDER:
        w = make_workload(name, T=min(512, make_workload(name).T))
        out.append((name, w))
    for s, (T, k, E, R) in enumerate([(1, 1, 1, 1), (7, 4, 8, 2), (50, 8, 64, 8), (33, 6, 12, 3),
                                      (20, 5, 5, 5), (40, 3, 4, 1)]):
        out.append((f"fuzz{s}", random_case(400 + s, T, 16, k, E, R)))
    return out


CASES = _cases()


def brute(idx, E, R):
    T, k = idx.shape
    El = E // R
    pairs = []                       # (rank, token, first j) of every distinct (token, rank)
    for t in range(T):
        seen = {}
        for j in range(k):
            r = int(idx[t, j]) // El
            if r not in seen:
                seen[r] = j
                pairs.append((r, t, j))
    pairs.sort()                     # rank-major, then token
    row_of = {(r, t): c for c, (r, t, _) in enumerate(pairs)}
    crow = np.array([[row_of[(int(idx[t, j]) // El, t)] for j in range(k)] for t in range(T)],
                    np.int32).reshape(T, k)
    counts = np.bincount([p[0] for p in pairs], minlength=R).astype(np.int32)
    src = np.array([t * k + j for (_, t, j) in pairs], np.int32)
    return counts, crow, src


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_coalesced_layout_matches_brute_force(name, w):
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    counts, offs, crow, src, expand = oracle.layout_coalesced(w.topk_idx, w.E, w.R, slot_of)
    bc, bcrow, bsrc = brute(w.topk_idx, w.E, w.R)
    assert np.array_equal(counts, bc)
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(bc)]))
    assert np.array_equal(crow, bcrow)
    assert np.array_equal(src, bsrc)
    # expand: slot s of the plain layout reads the coalesced row of its pair
    assert np.array_equal(expand[slot_of.ravel()], crow.ravel())


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_coalesced_invariants(name, w):
    _, _, _, slot_of, src_of = oracle.layout(w.topk_idx, w.E, w.R)
    counts, offs, crow, src, expand = oracle.layout_coalesced(w.topk_idx, w.E, w.R, slot_of)
    El = w.E // w.R
    ranks = w.topk_idx // El
    distinct = sum(len(set(r)) for r in ranks.tolist())
    assert offs[-1] == distinct <= w.topk_idx.size
    tok = src // w.k
    for r in range(w.R):                      # token order inside each rank segment
        seg = tok[offs[r]:offs[r + 1]]
        assert np.all(np.diff(seg) > 0)
        assert np.all(ranks.ravel()[src[offs[r]:offs[r + 1]]] == r)
    # an expert's slots all read rows of its own rank's segment
    eidx = w.topk_idx.ravel()[src_of]
    rr = eidx // El
    assert np.all((expand >= offs[rr]) & (expand < offs[rr + 1]))


def test_coalesced_hand_worked():
    # E=4 on R=2 (experts 0,1 -> rank 0; 2,3 -> rank 1)
    idx = np.array([[0, 1], [2, 0], [3, 2]], np.int32)
    _, _, _, slot_of, _ = oracle.layout(idx, 4, 2)
    counts, offs, crow, src, expand = oracle.layout_coalesced(idx, 4, 2, slot_of)
    # token 0 -> {rank 0}; token 1 -> {rank 1, rank 0}; token 2 -> {rank 1}
    assert counts.tolist() == [2, 2] and offs.tolist() == [0, 2, 4]
    assert crow.tolist() == [[0, 0], [2, 1], [3, 3]]
    assert src.tolist() == [0, 3, 2, 4]


@pytest.mark.parametrize("name,w", CASES[:5] + CASES[7:9], ids=[c[0] for c in CASES[:5] + CASES[7:9]])
def test_coalesced_dispatch_rows(name, w):
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    _, offs, crow, src, expand = oracle.layout_coalesced(w.topk_idx, w.E, w.R, slot_of)
    rc = oracle.dispatch_coalesced(w.x, crow, int(offs[-1]))
    assert np.array_equal(rc, w.x[src // w.k])
    # reading through expand reproduces the plain dispatch
    assert np.array_equal(rc[expand], oracle.dispatch(w.x, slot_of))
