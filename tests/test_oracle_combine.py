"""Pins for the oracle's combine (router-weighted sum of the k expert outputs).

HyperParallel-MoE section 2.2 / 4.1: expert outputs are weighted by the routing
scores and the top-k contributions accumulated; RailWave section 3: combine uses
the saved dispatch metadata to return rows to token order.  The stated
precision is fp32 accumulation, one fused multiply-add per slot in slot order.
Pins: the float64 closed form within the fp32 error bound, one-hot weights,
the identity-expert round trip and torch's bf16 rounding of the fp32 result.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads.gen import make_workload, random_case, bf16_bits_to_f32

U = 2.0 ** -24


def _case(name, T=None):
    if name.startswith("fuzz"):
        s = int(name[4:])
        return random_case(200 + s, [33, 5, 64][s], [128, 264, 8][s], [8, 3, 1][s],
                           [16, 5, 2][s], [4, 5, 1][s])
    return make_workload(name, T=T)


CASES = [("tiny", None), ("dsv3_decode", 32), ("mixtral", 300), ("glm45_air", 40),
         ("fuzz0", None), ("fuzz1", None), ("fuzz2", None)]


@pytest.mark.parametrize("name,T", CASES)
def test_fp32_sum_within_error_bound_of_exact(name, T):
    w = _case(name, T)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    y = w.y()
    out = oracle.combine(y, slot_of, w.topk_w, "f32").astype(np.float64)
    exact, mag = oracle.combine_f64(y, slot_of, w.topk_w)
    k = w.k
    gamma = k * U / (1 - k * U)
    assert np.all(np.abs(out - exact) <= gamma * mag)


@pytest.mark.parametrize("name,T", CASES)
def test_bf16_output_is_rounded_fp32_output(name, T):
    w = _case(name, T)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    y = w.y()
    f = oracle.combine(y, slot_of, w.topk_w, "f32")
    b = oracle.combine(y, slot_of, w.topk_w, "bf16")
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, ref)


def test_one_hot_weights_select_one_slot():
    w = random_case(9, 20, 64, 4, 6, 2)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    y = w.y()
    for j0 in range(w.k):
        wt = np.zeros_like(w.topk_w)
        wt[:, j0] = 1.0
        out = oracle.combine(y, slot_of, wt, "bf16")
        assert np.array_equal(out, y[slot_of[:, j0]])
        out32 = oracle.combine(y, slot_of, wt, "f32")
        assert np.array_equal(out32, bf16_bits_to_f32(y[slot_of[:, j0]]))


@pytest.mark.parametrize("name,T", [("tiny", None), ("dsv3_decode", 64), ("mixtral", 512),
                                    ("glm45_air", 64), ("dsv3_prefill", 16)])
def test_identity_expert_round_trip(name, T):
    """combine(dispatch(x)) with identity experts and weights summing to one
    (within fp32) returns x exactly: x*(1 +- few*2^-24) rounds back to x."""
    w = make_workload(name, T=T)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    recv = oracle.dispatch(w.x, slot_of)
    out = oracle.combine(recv, slot_of, w.topk_w, "bf16")
    nz = (w.x & 0x7FFF) != 0
    assert np.array_equal(out[nz], w.x[nz])
    assert np.all(bf16_bits_to_f32(out[~nz]) == 0)


def test_slot_order_and_fp32_accumulation():
    """k=3, unit weights, y = (2^25, 1, -2^25): fp32 accumulation in slot order
    loses the 1 (2^25 + 1 rounds to 2^25) and returns 0; float64 returns 1."""
    big = np.float32(2.0 ** 25)
    vals = np.array([big, 1.0, -big], np.float32)
    y = (vals.view(np.uint32) >> 16).astype(np.uint16)[:, None]  # exact bf16 values
    slot_of = np.array([[0, 1, 2]], np.int32)
    wt = np.ones((1, 3), np.float32)
    assert oracle.combine(y, slot_of, wt, "f32")[0, 0] == 0.0
    assert oracle.combine_f64(y, slot_of, wt)[0][0, 0] == 1.0
    # the same three rows taken in the slot order (2^25, -2^25, 1) keep the 1
    assert oracle.combine(y, np.array([[0, 2, 1]], np.int32), wt, "f32")[0, 0] == 1.0


def test_weights_are_not_renormalised():
    y = np.array([[0x3F80], [0x4000]], np.uint16)               # 1.0, 2.0
    slot_of = np.array([[0, 1]], np.int32)
    wt = np.array([[0.5, 2.0]], np.float32)
    assert oracle.combine(y, slot_of, wt, "f32")[0, 0] == np.float32(4.5)


def test_empty_tokens():
    out = oracle.combine(np.zeros((0, 16), np.uint16), np.zeros((0, 2), np.int32),
                         np.zeros((0, 2), np.float32))
    assert out.shape == (0, 16)


def test_each_slot_is_one_fused_multiply_add():
    """k = 2, y = (1 + 2^-7, 1 + 2^-7) (exact bf16), w = (-1, 1 + 2^-23) (exact
    fp32).  The exact value of w1*y1 + w0*y0 is 2^-23 (1 + 2^-7) = 2^-23 +
    2^-30, which fp32 holds.  One fused multiply-add per slot keeps it: the
    running sum after slot 0 is -(1 + 2^-7) exactly, and slot 1 rounds the
    exact w1*y1 + acc once.  Rounding the product first (to 1 + 2^-7 + 2^-23,
    the 2^-30 lies below half an ulp at 1) and then adding would give 2^-23."""
    y = np.full((2, 8), 0x3F81, np.uint16)          # 1.0078125 = 1 + 2^-7
    slot_of = np.array([[0, 1]], np.int32)
    wt = np.array([[-1.0, 1.0 + 2.0 ** -23]], np.float32)
    assert float(wt[0, 1]) == 1.0 + 2.0 ** -23
    out = oracle.combine(y, slot_of, wt, "f32")
    assert np.all(out == np.float32(2.0 ** -23 + 2.0 ** -30))
    # one rounding to bf16: 2^-23 (1 + 2^-7) has 8 significant bits, so it is
    # exact in bf16: sign 0, biased exponent 127 - 23 = 104, fraction 0000001
    outb = oracle.combine(y, slot_of, wt, "bf16")
    assert np.all(outb == (104 << 7) | 1)
