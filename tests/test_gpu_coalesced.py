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


# ------------------------------------------------------------------ combine

def _coalesced_combine_case(w, y, out_dtype):
    m = cl()
    lay, co, nc = assert_coalesced_equal(w.topk_idx, w.E, w.R)
    rows = w.T * min(w.k, w.R)
    wt = torch.from_numpy(np.ascontiguousarray(w.topk_w)).cuda()
    out, part = m.moe_combine_coalesced(bf16_dev(y), lay.slot_of, wt, co, rows,
                                        out_dtype=out_dtype)
    slot_of, crow = lay.slot_of.cpu().numpy(), co.crow.cpu().numpy()
    ref_part = oracle.combine_coalesced_pre(y, slot_of, w.topk_w, crow, nc)
    assert np.array_equal(bits(part)[:nc], ref_part)
    ref = oracle.combine_coalesced_post(ref_part, crow,
                                        "bf16" if out_dtype == torch.bfloat16 else "f32")
    got = bits(out) if out_dtype == torch.bfloat16 else out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32 if got.dtype == np.float32 else np.uint16),
                          ref.view(np.uint32 if ref.dtype == np.float32 else np.uint16))
    return lay, co, out


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_coalesced_combine_matches_oracle(name):
    from workloads.gen import expert_output
    w = workload(name)
    _coalesced_combine_case(w, expert_output(w.N, w.H, seed=w.seed + 7), torch.bfloat16)


@pytest.mark.parametrize("name", ["tiny", "glm45_air"])
def test_coalesced_combine_f32_matches_oracle(name):
    from workloads.gen import expert_output
    w = workload(name)
    _coalesced_combine_case(w, expert_output(w.N, w.H, seed=w.seed + 9), torch.float32)


COMBINE_FUZZ = [  # (seed, T, H, k, E, R)
    (31, 1, 8, 1, 1, 1), (32, 17, 24, 3, 12, 4), (33, 300, 1000, 8, 64, 8),
    (34, 2000, 2048, 2, 8, 8), (35, 700, 7176, 8, 256, 32), (36, 64, 4096, 32, 64, 16),
    (37, 5, 16384, 6, 6, 3), (38, 900, 512, 16, 32, 1), (39, 3000, 128, 12, 48, 48),
]


@pytest.mark.parametrize("case", COMBINE_FUZZ, ids=[f"s{c[0]}_T{c[1]}_H{c[2]}_k{c[3]}_R{c[5]}" for c in COMBINE_FUZZ])
def test_coalesced_combine_fuzz(case):
    from workloads.gen import expert_output
    seed, T, H, k, E, R = case
    w = random_case(seed, T, H, k, E, R)
    _coalesced_combine_case(w, expert_output(T * k, H, seed=seed), torch.bfloat16)


def test_coalesced_combine_one_rank_equals_plain_combine():
    from workloads.gen import expert_output
    m = cl()
    w = random_case(41, 1500, 1024, 8, 16, 1)
    y = expert_output(w.N, w.H, seed=3)
    lay, co, out = _coalesced_combine_case(w, y, torch.bfloat16)
    wt = torch.from_numpy(np.ascontiguousarray(w.topk_w)).cuda()
    plain = m.moe_combine(bf16_dev(y), lay.slot_of, wt)
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))


def test_coalesced_combine_empty_and_bad_rows():
    m = cl()
    d = torch.zeros((0, 2), dtype=torch.int32, device="cuda")
    co = m.moe_layout_coalesced(d, d, 8, 2)
    out, _ = m.moe_combine_coalesced(torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"),
                                     d, torch.zeros((0, 2), dtype=torch.float32, device="cuda"),
                                     co, 0)
    torch.cuda.synchronize()
    assert out.shape == (0, 64)
    # a capacity below Nc: the rows past it are neither computed nor read
    err = m.new_error_word()
    idx = np.array([[0, 2], [1, 3], [2, 2]], np.int32)   # E=4, R=2: Nc = 5
    lay = m.moe_layout(i32_dev(idx), 4, 2)
    co = m.moe_layout_coalesced(i32_dev(idx), lay.slot_of, 4, 2)
    y = torch.ones((6, 64), dtype=torch.bfloat16, device="cuda")
    wt = torch.ones((3, 2), dtype=torch.float32, device="cuda")
    m.moe_combine_coalesced(y, lay.slot_of, wt, co, 3, err_word=err)
    assert m.moe_read_error(err) == m.MOE_ERRBIT_BAD_INDEX



# ------------------------------------------------------------ FP8 dispatch

@pytest.mark.parametrize("name", ["dsv3_prefill", "tiny", "dsv3_decode"])
def test_coalesced_dispatch_quant_matches_oracle(name):
    """Each coalesced row holds the token's codes and scales, as the plain
    FP8 dispatch writes them to every slot of that token."""
    m = cl()
    w = workload(name)
    lay, co, nc = assert_coalesced_equal(w.topk_idx, w.E, w.R)
    rows = w.T * min(w.k, w.R)
    q = torch.full((rows, w.H), 0x5A, dtype=torch.uint8, device="cuda")
    sc = torch.full((rows, w.H // 128), -1.0, dtype=torch.float32, device="cuda")
    m.moe_dispatch_quant_coalesced(bf16_dev(w.x), co.crow, rows, recv_q=q, recv_scales=sc)
    slot_of = lay.slot_of.cpu().numpy()
    rq, rs = oracle.dispatch_quant(w.x, slot_of)
    src = co.src_pair_c.cpu().numpy()[:nc]
    owner_slot = slot_of.ravel()[src]
    assert np.array_equal(q.cpu().numpy()[:nc], rq[owner_slot])
    assert np.array_equal(sc.cpu().numpy()[:nc], rs[owner_slot])
    assert (q.cpu().numpy()[nc:] == 0x5A).all() and (sc.cpu().numpy()[nc:] == -1.0).all()
