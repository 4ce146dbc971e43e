"""The persistent Data-as-Flag kernel (dispatch -> identity expert -> combine
with per-row-chunk readiness words) against the CPU oracle, and its bounded
wait: a readiness word that never arrives ends in MOE_ERR_TIMEOUT, not a hang."""
import numpy as np
import pytest
import torch

import oracle
from workloads.gen import make_workload, random_case

pytestmark = pytest.mark.gpu


def cl():
    import combine_layout_moe_gb300 as m
    return m


def _dev(w):
    x = torch.from_numpy(np.ascontiguousarray(w.x).view(np.int16)).cuda().view(torch.bfloat16)
    return x, torch.from_numpy(w.topk_w).cuda()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "glm45_air", "mixtral"])
def test_flagged_matches_oracle(name):
    m = cl()
    w = make_workload(name)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    x, wt = _dev(w)
    so = torch.from_numpy(slot_of).cuda()
    flags = m.FlagWords(w.T, w.H, w.k)
    err = m.new_error_word()
    recv, out = m.moe_dispatch_combine_flagged(x, so, wt, flags, err_word=err)
    assert m.moe_read_error(err) == 0
    ref_recv = oracle.dispatch(w.x, slot_of)
    assert np.array_equal(_bits(recv), ref_recv)
    assert np.array_equal(_bits(out), oracle.combine(ref_recv, slot_of, w.topk_w, "bf16"))
    # the same words again, next epoch, fp32 output
    recv2, out2 = m.moe_dispatch_combine_flagged(x, so, wt, flags, out_dtype=torch.float32,
                                                 err_word=err)
    assert m.moe_read_error(err) == 0 and flags.epoch == 2
    assert np.array_equal(out2.cpu().numpy(), oracle.combine(ref_recv, slot_of, w.topk_w, "f32"))


@pytest.mark.parametrize("case", [(61, 1, 8, 1, 1, 1), (62, 37, 264, 3, 5, 5), (63, 129, 7176, 8, 16, 4),
                                  (64, 300, 1024, 32, 40, 8)])
def test_flagged_fuzz(case):
    m = cl()
    seed, T, H, k, E, R = case
    w = random_case(seed, T, H, k, E, R)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, E, R)
    x, wt = _dev(w)
    flags = m.FlagWords(T, H, k)
    err = m.new_error_word()
    recv, out = m.moe_dispatch_combine_flagged(x, torch.from_numpy(slot_of).cuda(), wt, flags,
                                               err_word=err)
    assert m.moe_read_error(err) == 0
    ref_recv = oracle.dispatch(w.x, slot_of)
    assert np.array_equal(_bits(recv), ref_recv)
    assert np.array_equal(_bits(out), oracle.combine(ref_recv, slot_of, w.topk_w, "bf16"))


def test_missing_readiness_word_times_out_cleanly():
    """The producer of one pair skips its word: the consumer's wait runs out
    after 2 ms, the call returns, the error word says TIMEOUT, every other token
    is still correct, and the next normal call succeeds."""
    m = cl()
    w = make_workload("tiny")
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    x, wt = _dev(w)
    so = torch.from_numpy(slot_of).cuda()
    flags = m.FlagWords(w.T, w.H, w.k)
    err = m.new_error_word()
    skip = 5 * w.k + 1                              # token 5, slot 1
    out = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    m.moe_dispatch_combine_flagged(x, so, wt, flags, out=out, spin_limit_ns=2_000_000,
                                   fault_skip_pair=skip, err_word=err)
    assert m.moe_read_error(err) == m.MOE_ERRBIT_TIMEOUT
    ref = oracle.combine(oracle.dispatch(w.x, slot_of), slot_of, w.topk_w, "bf16")
    got = _bits(out)
    others = np.ones(w.T, bool)
    others[5] = False
    assert np.array_equal(got[others], ref[others])
    recv, out = m.moe_dispatch_combine_flagged(x, so, wt, flags, err_word=err)
    assert m.moe_read_error(err) == 0
    assert np.array_equal(_bits(out), ref)


def test_flagged_rejects_bad_arguments():
    m = cl()
    w = random_case(65, 4, 64, 2, 4, 2)
    x, wt = _dev(w)
    so = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    flags = m.FlagWords(4, 64, 2)
    flags.epoch = 0xFFFFFFFF                      # next epoch wraps to 1, still valid
    m.moe_dispatch_combine_flagged(x, so.clone(), wt, flags)
    L = m._lib
    st = L.moe_dispatch_combine_flagged(4, 64, 2, x.data_ptr(), so.data_ptr(), wt.data_ptr(),
                                        x.data_ptr(), x.data_ptr(), 0, flags.words.data_ptr(),
                                        0, 1000, -1, None, None)
    assert st == m.MOE_ERR_INVALID_ARG            # epoch 0
