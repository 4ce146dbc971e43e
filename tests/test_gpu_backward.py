"""Backward kernels vs the CPU oracle (HyperParallel-MoE section 2.2: backward
Dispatch = gradient of forward Combine; backward Combine = gradient of forward
Dispatch).  dy and dx must be bit-identical; dw, an fp32 dot product over H
whose summation order is the kernel's, must lie within the fp32 error bound
(H-1) * 2^-24 * sum|y * dout| of the oracle's (binary64, exact products)."""
import functools

import numpy as np
import pytest
import torch

import oracle
from workloads.gen import make_workload, random_case, expert_output

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


def cl():
    import combine_layout_moe_gb300 as m
    return m


def bf16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@functools.lru_cache(maxsize=1)
def _named(name):
    w = make_workload(name)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    return w, slot_of, expert_output(w.N, w.H, seed=7), expert_output(w.T, w.H, seed=8)


def _fuzz(seed, T, H, k, E, R):
    w = random_case(seed, T, H, k, E, R)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, E, R)
    return w, slot_of, expert_output(w.N, H, seed=seed), expert_output(T, H, seed=seed + 1)


def _check_combine_backward(w, slot_of, y, dout):
    m = cl()
    err = m.new_error_word()
    dy, dw = m.moe_combine_backward(bf16_dev(dout), bf16_dev(y), torch.from_numpy(slot_of).cuda(),
                                    torch.from_numpy(w.topk_w).cuda(), err_word=err)
    assert m.moe_read_error(err) == 0
    rdy, rdw, mag = oracle.combine_backward(dout, y, slot_of, w.topk_w)
    assert np.array_equal(bits(dy), rdy)
    got = dw.cpu().numpy().astype(np.float64)
    bound = (w.H - 1) * U / (1 - (w.H - 1) * U) * mag
    assert np.all(np.abs(got - rdw) <= bound), np.max(np.abs(got - rdw) - bound)


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "dsv3_prefill", "glm45_air", "mixtral"])
def test_combine_backward_matches_oracle(name):
    _check_combine_backward(*_named(name))


# 5 <= k <= 8 takes the bulk-copy pipeline: fewer tokens than SMs (one or a
# few tokens per CTA), tokens split between two CTAs, k = 5..7, and one chunk
# per row as well as many
FUZZ = [(71, 1, 8, 1, 1, 1), (72, 33, 264, 3, 5, 5), (73, 100, 7176, 8, 16, 4),
        (74, 17, 1024, 16, 20, 4), (75, 9, 512, 32, 40, 8), (78, 777, 1000, 5, 10, 5),
        (79, 7, 4096, 6, 12, 3), (80, 3001, 136, 7, 7, 7), (81, 1, 16384, 8, 8, 2),
        # H = 262144: the pipeline's ring and stages exceed shared memory, so
        # the CTA-per-token kernel takes k = 8
        (82, 2, 262144, 8, 8, 2),
        # 9 <= k <= 16: the CTA-per-token kernel's 16-slot instance
        (83, 300, 2056, 9, 18, 6), (84, 64, 4096, 12, 48, 8)]


@pytest.mark.parametrize("case", FUZZ, ids=[f"T{c[1]}_H{c[2]}_k{c[3]}" for c in FUZZ])
def test_combine_backward_fuzz(case):
    _check_combine_backward(*_fuzz(*case))


@pytest.mark.parametrize("k", [4, 8])
def test_combine_backward_without_dw(k):
    m = cl()
    w, slot_of, y, dout = _fuzz(76, 400, 2048, k, 8, 2)
    dy, dw = m.moe_combine_backward(bf16_dev(dout), None, torch.from_numpy(slot_of).cuda(),
                                    torch.from_numpy(w.topk_w).cuda())
    assert dw is None
    assert np.array_equal(bits(dy), oracle.combine_backward(dout, None, slot_of, w.topk_w)[0])


def test_combine_backward_dw_is_deterministic():
    # dw's summation order is fixed (tokens split between two CTAs get exactly
    # two additions onto zero, whose order cannot change the result)
    m = cl()
    w, slot_of, y, dout = _named("dsv3_decode")
    args = (bf16_dev(dout), bf16_dev(y), torch.from_numpy(slot_of).cuda(),
            torch.from_numpy(w.topk_w).cuda())
    runs = [m.moe_combine_backward(*args)[1].cpu().numpy().view(np.uint32) for _ in range(3)]
    assert all(np.array_equal(runs[0], r) for r in runs[1:])


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "glm45_air", "mixtral"])
def test_dispatch_backward_matches_oracle(name):
    m = cl()
    w, slot_of, y, _ = _named(name)
    so = torch.from_numpy(slot_of).cuda()
    for dt, od in ((torch.bfloat16, "bf16"), (torch.float32, "f32")):
        dx = m.moe_dispatch_backward(bf16_dev(y), so, out_dtype=dt)
        ref = oracle.dispatch_backward(y, slot_of, od)
        got = bits(dx) if od == "bf16" else dx.cpu().numpy()
        assert np.array_equal(got.view(ref.dtype), ref)


@pytest.mark.parametrize("case", FUZZ + [(77, 9, 64, 40, 7, 7)],
                         ids=[f"T{c[1]}_H{c[2]}_k{c[3]}" for c in FUZZ + [(77, 9, 64, 40, 7, 7)]])
def test_dispatch_backward_fuzz(case):
    m = cl()
    w, slot_of, y, _ = _fuzz(*case)
    dx = m.moe_dispatch_backward(bf16_dev(y), torch.from_numpy(slot_of).cuda())
    assert np.array_equal(bits(dx), oracle.dispatch_backward(y, slot_of, "bf16"))


def test_combine_backward_bad_slot_reported_k8():
    m = cl()
    err = m.new_error_word()
    T, k, H = 300, 8, 512
    so = torch.arange(T * k, dtype=torch.int32, device="cuda").view(T, k)
    so[123, 5] = T * k + 7
    d = torch.ones((T, H), dtype=torch.bfloat16, device="cuda")
    yv = torch.ones((T * k, H), dtype=torch.bfloat16, device="cuda")
    m.moe_combine_backward(d, yv, so, torch.ones((T, k), device="cuda"), err_word=err)
    assert m.moe_read_error(err) == m.MOE_ERRBIT_BAD_INDEX


def test_backward_bad_slot_reported():
    m = cl()
    err = m.new_error_word()
    so = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device="cuda")
    d = torch.ones((2, 64), dtype=torch.bfloat16, device="cuda")
    yv = torch.ones((4, 64), dtype=torch.bfloat16, device="cuda")
    m.moe_combine_backward(d, yv, so, torch.ones((2, 2), device="cuda"), err_word=err)
    assert m.moe_read_error(err) == m.MOE_ERRBIT_BAD_INDEX
    m.moe_dispatch_backward(yv, so, err_word=err)
    assert m.moe_read_error(err) == m.MOE_ERRBIT_BAD_INDEX
