"""The persistent dispatch -> identity expert -> combine kernel against the CPU
oracle, in each readiness mode (UBEP section 3.4 / Figure 6: a word per block,
sentinel polling, a per-batch checksum, and the stop-and-wait barrier), and
its bounded waits: readiness that never arrives ends in MOE_ERR_TIMEOUT, not a
hang, and leaves every other token correct."""
import functools

import numpy as np
import pytest
import torch

import oracle
from workloads.gen import make_workload, random_case

pytestmark = pytest.mark.gpu

SENTINEL_BITS = 0xFFFF


def cl():
    import combine_layout_moe_gb300 as m
    return m


def _dev(w):
    x = torch.from_numpy(np.ascontiguousarray(w.x).view(np.int16)).cuda().view(torch.bfloat16)
    return x, torch.from_numpy(w.topk_w).cuda()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _modes():
    m = cl()
    return [("word2048", m.MOE_SYNC_WORD, 2048), ("word32", m.MOE_SYNC_WORD, 32),
            ("sentinel", m.MOE_SYNC_SENTINEL, 512), ("batch4096", m.MOE_SYNC_BATCH, 4096),
            ("batch512", m.MOE_SYNC_BATCH, 512), ("barrier", m.MOE_SYNC_BARRIER, 512)]


MODE_IDS = ["word2048", "word32", "sentinel", "batch4096", "batch512", "barrier"]


def _mode(name):
    return {n: (mode, g) for n, mode, g in _modes()}[name]


@functools.lru_cache(maxsize=4)
def _named(name):
    """A named workload, its slot map and the oracle's rows and outputs."""
    w = make_workload(name)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    ref_recv = oracle.dispatch(w.x, slot_of)
    refs = {kind: oracle.combine(ref_recv, slot_of, w.topk_w, kind) for kind in ("bf16", "f32")}
    return w, slot_of, ref_recv, refs


def _check(m, state, w, slot_of, recv, y, out, out_kind="bf16", cached=None):
    if cached is None:
        ref_recv = oracle.dispatch(w.x, slot_of)
        ref = oracle.combine(ref_recv, slot_of, w.topk_w, out_kind)
    else:
        ref_recv, ref = cached[0], cached[1][out_kind]
    if out_kind == "bf16":
        assert np.array_equal(_bits(out), ref)
    else:
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    if state.mode == m.MOE_SYNC_SENTINEL:
        # every reader wrote the sentinel back: ready for the next call
        assert (_bits(recv) == SENTINEL_BITS).all() and (_bits(y) == SENTINEL_BITS).all()
    else:
        assert np.array_equal(_bits(recv), ref_recv)
        assert np.array_equal(_bits(y), ref_recv)


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "glm45_air", "mixtral"])
@pytest.mark.parametrize("mode_name", MODE_IDS)
def test_flagged_matches_oracle(mode_name, name):
    m = cl()
    mode, G = _mode(mode_name)
    w, slot_of, ref_recv, refs = _named(name)
    x, wt = _dev(w)
    so = torch.from_numpy(slot_of).cuda()
    state = m.SyncState(w.T, w.H, w.k, mode, G)
    err = m.new_error_word()
    recv, y, out = m.moe_dispatch_combine_flagged(x, so, wt, state, err_word=err)
    assert m.moe_read_error(err) == 0
    _check(m, state, w, slot_of, recv, y, out, cached=(ref_recv, refs))
    # the same state again: the next epoch (or the reset sentinel), fp32 output
    recv, y, out = m.moe_dispatch_combine_flagged(x, so, wt, state, out_dtype=torch.float32,
                                                  err_word=err)
    assert m.moe_read_error(err) == 0 and state.epoch == 2
    _check(m, state, w, slot_of, recv, y, out, "f32", cached=(ref_recv, refs))


FUZZ = [(61, 1, 8, 1, 1, 1), (62, 37, 264, 3, 5, 5), (63, 129, 7176, 8, 16, 4),
        (64, 300, 1024, 32, 40, 8), (65, 2000, 128, 4, 8, 2)]


@pytest.mark.parametrize("case", FUZZ, ids=[f"s{c[0]}_T{c[1]}_H{c[2]}_k{c[3]}" for c in FUZZ])
@pytest.mark.parametrize("mode_name", MODE_IDS)
def test_flagged_fuzz(mode_name, case):
    m = cl()
    mode, G = _mode(mode_name)
    seed, T, H, k, E, R = case
    w = random_case(seed, T, H, k, E, R)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, E, R)
    x, wt = _dev(w)
    state = m.SyncState(T, H, k, mode, G)
    err = m.new_error_word()
    recv, y, out = m.moe_dispatch_combine_flagged(x, torch.from_numpy(slot_of).cuda(), wt,
                                                  state, err_word=err)
    assert m.moe_read_error(err) == 0
    _check(m, state, w, slot_of, recv, y, out)


@pytest.mark.parametrize("G", [16, 64, 256, 512, 1024, 8192, 16384])
def test_word_granularity_sweep(G):
    m = cl()
    w = make_workload("dsv3_decode", T=256)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    x, wt = _dev(w)
    state = m.SyncState(w.T, w.H, w.k, m.MOE_SYNC_WORD, G)
    err = m.new_error_word()
    recv, y, out = m.moe_dispatch_combine_flagged(x, torch.from_numpy(slot_of).cuda(), wt,
                                                  state, err_word=err)
    assert m.moe_read_error(err) == 0
    _check(m, state, w, slot_of, recv, y, out)


@pytest.mark.parametrize("mode_name", ["word2048", "word32", "sentinel", "batch512"])
def test_missing_readiness_times_out_cleanly(mode_name):
    """The producer of one pair publishes nothing: the readers of that row give
    up after their bound, the call returns, the error word says TIMEOUT, every
    other token is still correct, and the next normal call succeeds."""
    m = cl()
    mode, G = _mode(mode_name)
    w = make_workload("tiny")
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    x, wt = _dev(w)
    so = torch.from_numpy(slot_of).cuda()
    state = m.SyncState(w.T, w.H, w.k, mode, G)
    err = m.new_error_word()
    skip = 5 * w.k + 1                              # token 5, slot 1
    out = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    m.moe_dispatch_combine_flagged(x, so, wt, state, out=out, spin_limit_ns=2_000_000,
                                   fault_skip_pair=skip, err_word=err)
    assert m.moe_read_error(err) == m.MOE_ERRBIT_TIMEOUT
    ref = oracle.combine(oracle.dispatch(w.x, slot_of), slot_of, w.topk_w, "bf16")
    got = _bits(out)
    others = np.ones(w.T, bool)
    others[5] = False
    assert np.array_equal(got[others], ref[others])
    if mode == m.MOE_SYNC_SENTINEL:
        state.refill()                               # a failed call leaves stale rows behind
    _, _, out = m.moe_dispatch_combine_flagged(x, so, wt, state, err_word=err)
    assert m.moe_read_error(err) == 0
    assert np.array_equal(_bits(out), ref)


def test_sentinel_collision_is_reported_and_bounded():
    """A payload word equal to the sentinel: the producer reports it and its
    readers' waits run out instead of hanging."""
    m = cl()
    w = random_case(66, 16, 64, 2, 4, 2)
    xb = np.ascontiguousarray(w.x).copy()
    xb[3, 8:10] = SENTINEL_BITS                      # one aligned 32-bit word of token 3
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    state = m.SyncState(w.T, w.H, w.k, m.MOE_SYNC_SENTINEL, 512)
    err = m.new_error_word()
    m.moe_dispatch_combine_flagged(x, torch.from_numpy(slot_of).cuda(),
                                   torch.from_numpy(w.topk_w).cuda(), state,
                                   spin_limit_ns=2_000_000, err_word=err)
    bits = m.moe_read_error(err)
    assert bits & m.MOE_ERRBIT_SENTINEL and bits & m.MOE_ERRBIT_TIMEOUT


def test_flagged_rejects_bad_arguments():
    m = cl()
    w = random_case(67, 4, 64, 2, 4, 2)
    x, wt = _dev(w)
    so = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    state = m.SyncState(4, 64, 2, m.MOE_SYNC_WORD, 512)
    state.epoch = 0xFFFFFFFF                         # next epoch wraps to 1, still valid
    m.moe_dispatch_combine_flagged(x, so.clone(), wt, state)
    with pytest.raises(ValueError):
        m.SyncState(4, 64, 2, m.MOE_SYNC_BATCH, 256)  # batches are whole 512-byte blocks
    L = m._lib
    st = L.moe_dispatch_combine_flagged(4, 64, 2, x.data_ptr(), so.data_ptr(), wt.data_ptr(),
                                        x.data_ptr(), x.data_ptr(), x.data_ptr(), 0,
                                        m.MOE_SYNC_WORD, 512, state.words.data_ptr(), 0, 1000,
                                        -1, None, None)
    assert st == m.MOE_ERR_INVALID_ARG               # epoch 0
