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


# ------------------------------------------------------------ coalesced combine
# Return path of the coalesced dispatch: each rank pre-reduces the token's
# slots it holds into the token's coalesced row (bf16), then the token sums its
# rows in fp32.

import torch  # noqa: E402  (CPU only: an independent bf16 rounding)

from workloads.gen import bf16_bits_to_f32, expert_output  # noqa: E402


def torch_bf16_bits(f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def coalesced_combine(idx, E, R, y, w, out_dtype="bf16"):
    _, _, _, slot_of, _ = oracle.layout(idx, E, R)
    _, offs, crow, src, _ = oracle.layout_coalesced(idx, E, R, slot_of)
    part = oracle.combine_coalesced_pre(y, slot_of, w, crow, int(offs[-1]))
    return slot_of, crow, part, oracle.combine_coalesced_post(part, crow, out_dtype)


@pytest.mark.parametrize("T,k,E", [(40, 8, 16), (7, 3, 5), (100, 2, 1)])
def test_coalesced_combine_on_one_rank_is_plain_combine(T, k, E):
    w = random_case(510 + T, T, 24, k, E, 1)
    y = expert_output(T * k, 24, seed=T)
    slot_of, _, _, out = coalesced_combine(w.topk_idx, E, 1, y, w.topk_w)
    assert np.array_equal(out, oracle.combine(y, slot_of, w.topk_w, "bf16"))
    _, _, _, out32 = coalesced_combine(w.topk_idx, E, 1, y, w.topk_w, "f32")
    assert np.array_equal(out32, bf16_bits_to_f32(out))


def test_coalesced_combine_one_slot_per_rank():
    rng = np.random.default_rng(7)
    T, k, E, R, H = 50, 4, 24, 6, 32
    El = E // R
    idx = np.stack([rng.permutation(R)[:k] * El + rng.integers(0, El, k) for _ in range(T)])
    idx = idx.astype(np.int32)
    wts = rng.random((T, k), dtype=np.float32)
    y = expert_output(T * k, H, seed=11)
    slot_of, crow, part, out = coalesced_combine(idx, E, R, y, wts, "f32")
    yf = bf16_bits_to_f32(y)
    prod = wts[:, :, None] * yf[slot_of]               # one fp32 multiply per element
    assert np.array_equal(part[crow.ravel()].reshape(T, k, H), torch_bf16_bits(prod))
    acc = np.zeros((T, H), np.float32)
    for j in range(k):                                 # fp32 adds in slot order
        acc = acc + bf16_bits_to_f32(torch_bf16_bits(prod[:, j]))
    assert np.array_equal(out, acc)


@pytest.mark.parametrize("seed,T,k,E,R", [(1, 64, 8, 32, 4), (2, 30, 6, 12, 3), (3, 9, 5, 10, 10)])
def test_coalesced_combine_integer_payload_is_exact(seed, T, k, E, R):
    rng = np.random.default_rng(seed)
    H = 16
    idx = rng.integers(0, E, (T, k)).astype(np.int32)
    wts = rng.choice(np.array([0.5, 1.0, 2.0], np.float32), (T, k))
    yv = rng.integers(-4, 5, (T * k, H)).astype(np.float32)   # |sum| <= 64 in steps of 1/2
    y = torch_bf16_bits(yv)
    slot_of, crow, part, out = coalesced_combine(idx, E, R, y, wts, "f32")
    exact = np.einsum("tk,tkh->th", wts.astype(np.float64), yv[slot_of].astype(np.float64))
    assert np.array_equal(out.astype(np.float64), exact)
    El = E // R
    for t in range(T):                                 # each row holds its rank's share
        for r in set((idx[t] // El).tolist()):
            js = [j for j in range(k) if idx[t, j] // El == r]
            c = crow[t, js[0]]
            share = sum(np.float64(wts[t, j]) * yv[slot_of[t, j]] for j in js)
            assert np.array_equal(bf16_bits_to_f32(part[c]).astype(np.float64), share)


@pytest.mark.parametrize("name,w", CASES[:5], ids=[c[0] for c in CASES[:5]])
def test_coalesced_combine_within_bound_of_exact(name, w):
    y = expert_output(w.N, w.H, seed=w.seed + 5)
    slot_of, crow, part, out = coalesced_combine(w.topk_idx, w.E, w.R, y, w.topk_w, "f32")
    terms = w.topk_w.astype(np.float64)[:, :, None] * bf16_bits_to_f32(y)[slot_of]
    exact = terms.sum(axis=1)
    El = w.E // w.R
    ranks = w.topk_idx // El
    share_abs = np.zeros_like(exact)                   # sum over ranks of |rank share|
    for r in range(w.R):
        share_abs += np.abs((terms * (ranks == r)[:, :, None]).sum(axis=1))
    # bf16 rounding of each share (unit 2^-8) + fp32 chains of at most k terms
    bound = 2.0 ** -8 * share_abs * (1 + 2.0 ** -6) + 2 * w.k * 2.0 ** -24 * np.abs(terms).sum(axis=1)
    assert np.all(np.abs(out - exact) <= bound)
