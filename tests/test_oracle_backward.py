"""Pins for the oracle's backward pass (HyperParallel-MoE section 2.2: backward
Dispatch is the gradient of forward Combine; backward Combine returns the
input-activation gradient).  Checked against torch autograd of a float64
forward combine, torch's bf16 rounding of fp32 products, numpy einsum, and the
unit-weight special case of the forward combine."""
import numpy as np
import pytest
import torch

import oracle
from workloads.gen import make_workload, random_case, expert_output, bf16_bits_to_f32


def _case(seed, T, H, k, E, R):
    w = random_case(seed, T, H, k, E, R)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, E, R)
    y = expert_output(w.N, H, seed=seed)
    dout = expert_output(T, H, seed=seed + 1)
    return w, slot_of, y, dout


CASES = [(300, 17, 64, 3, 5, 5), (301, 40, 256, 8, 16, 4), (302, 9, 136, 1, 2, 1),
         (303, 64, 1024, 2, 8, 8)]


@pytest.mark.parametrize("case", CASES)
def test_combine_backward_matches_autograd(case):
    w, slot_of, y, dout = _case(*case)
    dy, dw, mag = oracle.combine_backward(dout, y, slot_of, w.topk_w)
    # float64 forward combine, differentiated by torch autograd
    yt = torch.tensor(bf16_bits_to_f32(y), dtype=torch.float64, requires_grad=True)
    wt = torch.tensor(w.topk_w, dtype=torch.float64, requires_grad=True)
    so = torch.from_numpy(slot_of.astype(np.int64))
    out = (wt.unsqueeze(-1) * yt[so]).sum(dim=1)
    out.backward(torch.tensor(bf16_bits_to_f32(dout), dtype=torch.float64))
    # dy: the autograd gradient, then one fp32 rounding and one bf16 rounding
    g32 = yt.grad.to(torch.float32)
    assert torch.equal(torch.from_numpy(bf16_bits_to_f32(dy)),
                       g32.to(torch.bfloat16).to(torch.float32))
    # dw: exact up to binary64 rounding
    assert np.allclose(dw, wt.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(mag >= np.abs(dw) - 1e-12)


@pytest.mark.parametrize("case", CASES)
def test_combine_backward_dy_is_torch_rounded_product(case):
    w, slot_of, y, dout = _case(*case)
    dy, _, _ = oracle.combine_backward(dout, None, slot_of, w.topk_w)
    d = torch.from_numpy(bf16_bits_to_f32(dout))
    wt = torch.from_numpy(w.topk_w)
    ref = (wt.unsqueeze(-1) * d.unsqueeze(1)).to(torch.bfloat16)          # [T, k, H]
    ref = ref.view(torch.int16).numpy().view(np.uint16).reshape(-1, dout.shape[1])
    assert np.array_equal(dy[slot_of.ravel()], ref)


def test_combine_backward_dw_is_einsum():
    w, slot_of, y, dout = _case(304, 33, 512, 6, 12, 3)
    _, dw, _ = oracle.combine_backward(dout, y, slot_of, w.topk_w)
    yf = bf16_bits_to_f32(y).astype(np.float64)
    df = bf16_bits_to_f32(dout).astype(np.float64)
    assert np.allclose(dw, np.einsum("tkh,th->tk", yf[slot_of], df), rtol=1e-12, atol=1e-12)


def test_unit_weight_dy_is_dout():
    w, slot_of, y, dout = _case(305, 10, 64, 4, 4, 2)
    dy, _, _ = oracle.combine_backward(dout, None, slot_of, np.ones_like(w.topk_w))
    assert np.array_equal(dy[slot_of.ravel()], np.repeat(dout, w.k, axis=0))


@pytest.mark.parametrize("case", CASES)
def test_dispatch_backward_is_unit_weight_combine(case):
    w, slot_of, y, _ = _case(*case)
    for od in ("bf16", "f32"):
        dx = oracle.dispatch_backward(y, slot_of, od)
        assert np.array_equal(dx, oracle.combine(y, slot_of, np.ones_like(w.topk_w), od))


def test_dispatch_backward_of_dispatch_is_k_times_x():
    """drecv = dispatch(x): every token's k rows are copies of x[t], so dx is
    the fp32 sum of k copies; for k a power of two that is exact: k * x."""
    w = make_workload("tiny")                       # k = 2
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    dx = oracle.dispatch_backward(oracle.dispatch(w.x, slot_of), slot_of, "f32")
    assert np.array_equal(dx, 2.0 * bf16_bits_to_f32(w.x))


def test_backward_rejects_bad_slot():
    with pytest.raises(oracle.OracleError):
        oracle.dispatch_backward(np.zeros((2, 8), np.uint16), np.array([[0], [5]], np.int32))
