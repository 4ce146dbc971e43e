"""Rank-coalesced layout and dispatch on the GPU vs the CPU oracle.

RailWave, section 3.1 (token coalescing): one receive row per token and
distinct destination rank.  The row map (rank counts and offsets, crow,
src_pair_c, expand) and the coalesced rows must be bit-identical to the
oracle's; rows past Nc in the caller's buffer must stay untouched.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from workloads.gen import CONFIG_ORDER, make_workload, random_case

pytestmark = pytest.mark.gpu


def cl():
    import combine_layout_moe_gb300 as m
    return m


@functools.lru_cache(maxsize=2)
def workload(name):
    return make_workload(name)


def i32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def bf16_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_coalesced(idx, E, R, err=None):
    m = cl()
    d = i32_dev(idx)
    lay = m.moe_layout(d, E, R, err_word=err)
    co = m.moe_layout_coalesced(d, lay.slot_of, E, R, err_word=err)
    torch.cuda.synchronize()
    return lay, co


def assert_coalesced_equal(idx, E, R):
    lay, co = gpu_coalesced(idx, E, R)
    slot_of = lay.slot_of.cpu().numpy()
    counts, offs, crow, src, expand = oracle.layout_coalesced(idx, E, R, slot_of)
    nc = int(offs[-1])
    assert np.array_equal(co.rank_counts_c.cpu().numpy(), counts)
    assert np.array_equal(co.rank_offsets_c.cpu().numpy(), offs)
    g = co.crow.cpu().numpy()
    assert np.array_equal(g, crow), f"crow differs at {np.flatnonzero(g.ravel() != crow.ravel())[:8]}"
    assert np.array_equal(co.src_pair_c.cpu().numpy()[:nc], src)
    assert np.array_equal(co.expand.cpu().numpy(), expand)
    return lay, co, nc


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_coalesced_layout_matches_oracle(name):
    w = workload(name)
    assert_coalesced_equal(w.topk_idx, w.E, w.R)


FUZZ = [  # (seed, T, k, E, R)
    (1, 1, 1, 1, 1), (2, 1, 8, 256, 32), (3, 3, 5, 7, 7), (4, 33, 2, 16, 4), (5, 100, 8, 8, 1),
    (6, 257, 4, 256, 32), (7, 4097, 3, 5, 5), (8, 5000, 8, 1024, 8), (9, 12345, 6, 64, 16),
    (10, 70000, 2, 2, 2), (11, 100000, 8, 128, 16), (12, 300000, 8, 256, 32),
    (13, 2049, 1, 3, 1), (14, 511, 16, 40, 10), (15, 40, 33, 9, 3), (16, 3000, 32, 64, 64),
    (17, 9000, 8, 1024, 1024),
]


@pytest.mark.parametrize("case", FUZZ, ids=[f"s{c[0]}_T{c[1]}_k{c[2]}_E{c[3]}_R{c[4]}" for c in FUZZ])
def test_coalesced_layout_fuzz(case):
    seed, T, k, E, R = case
    w = random_case(seed, T, 8, k, E, R)
    assert_coalesced_equal(w.topk_idx, E, R)


def test_coalesced_layout_same_rank_and_same_expert():
    T, k, E, R = 20000, 8, 64, 8
    idx = np.full((T, k), 17, np.int32)        # every slot on one expert: one row per token
    _, _, nc = assert_coalesced_equal(idx, E, R)
    assert nc == T
    idx = (np.arange(T * k, dtype=np.int32).reshape(T, k) % E)  # 8 consecutive experts: one rank
    _, _, nc = assert_coalesced_equal(idx, E, R)
    assert nc == T
    idx = (np.arange(k, dtype=np.int32)[None, :] * (E // R)).repeat(T, 0)  # one slot per rank
    _, _, nc = assert_coalesced_equal(idx, E, R)
    assert nc == T * k


def test_coalesced_layout_empty():
    m = cl()
    d = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    so = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    co = m.moe_layout_coalesced(d, so, 8, 2)
    recv = m.moe_dispatch_coalesced(torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"),
                                    co.crow, 0)
    torch.cuda.synchronize()
    assert co.rank_counts_c.cpu().tolist() == [0, 0]
    assert co.rank_offsets_c.cpu().tolist() == [0, 0, 0]
    assert recv.shape == (0, 64)


def test_coalesced_layout_is_deterministic():
    w = workload("glm45_air")
    _, a = gpu_coalesced(w.topk_idx, w.E, w.R)
    _, b = gpu_coalesced(w.topk_idx, w.E, w.R)
    nc = int(a.rank_offsets_c[-1])
    for name in ("rank_counts_c", "rank_offsets_c", "crow", "expand"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert torch.equal(a.src_pair_c[:nc], b.src_pair_c[:nc])  # the rest is never written


def test_coalesced_layout_bad_index_reported():
    m = cl()
    err = m.new_error_word()
    idx = np.zeros((64, 2), np.int32)
    idx[10, 1] = 8
    idx[20, 0] = -3
    d = i32_dev(idx)
    so = i32_dev(np.arange(128, dtype=np.int32).reshape(64, 2))
    co = m.moe_layout_coalesced(d, so, 8, 2, err_word=err)
    assert m.moe_read_error(err) & m.MOE_ERRBIT_BAD_INDEX
    crow = co.crow.cpu().numpy()
    assert crow[10, 1] == -1 and crow[20, 0] == -1
    # the valid pairs still get rows: 62 tokens with one rank, tokens 10 and 20 one each
    assert co.rank_offsets_c.cpu().numpy()[-1] == 64


# ----------------------------------------------------------------- dispatch

SENTINEL = 0x7F7F


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_coalesced_dispatch_matches_oracle(name):
    m = cl()
    w = workload(name)
    lay, co, nc = assert_coalesced_equal(w.topk_idx, w.E, w.R)
    rows = w.T * min(w.k, w.R)
    recv_c = torch.full((rows, w.H), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    x = bf16_dev(w.x)
    m.moe_dispatch_coalesced(x, co.crow, rows, recv_c=recv_c)
    got = bits(recv_c)
    ref = oracle.dispatch_coalesced(w.x, co.crow.cpu().numpy(), nc)
    assert np.array_equal(got[:nc], ref)
    assert (got[nc:] == SENTINEL).all()
    # expanding the coalesced rows gives the plain expert-major receive buffer
    plain = m.moe_dispatch(x, lay.slot_of)
    assert torch.equal(recv_c[co.expand.long()].view(torch.int16), plain.view(torch.int16))


PAYLOAD_FUZZ = [  # (seed, T, H, k, E, R)
    (21, 1, 8, 1, 1, 1), (22, 17, 24, 3, 12, 4), (23, 300, 1000, 8, 64, 8),
    (24, 2000, 2048, 2, 8, 8), (25, 700, 7176, 8, 256, 32), (26, 64, 4096, 32, 64, 16),
    (27, 5, 16384, 6, 6, 3),
]


@pytest.mark.parametrize("case", PAYLOAD_FUZZ, ids=[f"s{c[0]}_T{c[1]}_H{c[2]}_k{c[3]}" for c in PAYLOAD_FUZZ])
def test_coalesced_dispatch_fuzz(case):
    m = cl()
    seed, T, H, k, E, R = case
    w = random_case(seed, T, H, k, E, R)
    _, co, nc = assert_coalesced_equal(w.topk_idx, E, R)
    recv_c = m.moe_dispatch_coalesced(bf16_dev(w.x), co.crow, nc)
    ref = oracle.dispatch_coalesced(w.x, co.crow.cpu().numpy(), nc)
    assert np.array_equal(bits(recv_c), ref)


def test_coalesced_dispatch_bad_row_reported():
    m = cl()
    err = m.new_error_word()
    x = torch.ones((4, 64), dtype=torch.bfloat16, device="cuda")
    crow = i32_dev(np.array([[0, 0], [1, 2], [3, 3], [4, 6]], np.int32))  # 6 >= rows
    m.moe_dispatch_coalesced(x, crow, 6, err_word=err)
    assert m.moe_read_error(err) == m.MOE_ERRBIT_BAD_INDEX


def test_coalesced_dispatch_rejects_large_k():
    m = cl()
    x = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
    crow = torch.zeros((2, 33), dtype=torch.int32, device="cuda")
    with pytest.raises(m.MoeError) as ei:
        m.moe_dispatch_coalesced(x, crow, 2)
    assert ei.value.status == m.MOE_ERR_UNSUPPORTED
