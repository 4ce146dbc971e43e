"""Combine on the method's edge inputs, bit for bit against the oracle.

Every finite bf16 bit pattern (both zeros, every subnormal, up to the largest
finite value, 65280 patterns) goes through moe_combine as expert output, with
router weights 0, -0, 1, -1, 0.5, an fp32 subnormal, a weight whose products
overflow fp32, and mixes of them; outputs in bf16 and fp32.  Both sides do one
fused multiply-add per slot in slot order from +0 and round once, without
flushing subnormals, so the outputs must be identical bit patterns (overflow
included: it rounds to infinity on both sides)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

ALL = np.array([b for b in range(1 << 16) if (b >> 7) & 0xFF != 0xFF], np.uint16)
assert ALL.size == 65280                       # 2 x (2^15 - 128) finite patterns
H = ALL.size                                    # a multiple of 8


def _dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _check(y, slot_of, w):
    import combine_layout_moe_gb300 as m
    err = m.new_error_word()
    yd = _dev16(y)
    so = torch.from_numpy(np.ascontiguousarray(slot_of, np.int32)).cuda()
    wd = torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda()
    ob = m.moe_combine(yd, so, wd, err_word=err)
    of = m.moe_combine(yd, so, wd, out_dtype=torch.float32, err_word=err)
    assert m.moe_read_error(err) == 0
    gb = ob.view(torch.int16).cpu().numpy().view(np.uint16)
    gf = of.cpu().numpy().view(np.uint32)
    rb = oracle.combine(y, slot_of, w, "bf16")
    rf = oracle.combine(y, slot_of, w, "f32").view(np.uint32)
    for name, g, r in (("bf16", gb, rb), ("f32", gf, rf)):
        bad = np.flatnonzero(g.ravel() != r.ravel())
        assert bad.size == 0, f"{name}: {bad.size} differ, first at {bad[:4]}: " \
                              f"{g.ravel()[bad[:4]]} vs {r.ravel()[bad[:4]]}"


W1 = np.array([0.0, -0.0, 1.0, -1.0, 0.5, 1e-40, 3.0, 2.0 ** -126], np.float32)


def test_every_finite_bf16_times_edge_weights_k1():
    """k = 1: out = round(w * y) for every finite y and each edge weight
    (3 * the largest values overflows to infinity; 1e-40 * y is subnormal
    or zero; 2^-126 * y lands on the subnormal boundary)."""
    assert W1[5] != 0 and W1[5] < np.finfo(np.float32).tiny      # an fp32 subnormal
    T = W1.size
    y = np.tile(ALL, (T, 1))
    _check(y, np.arange(T, dtype=np.int32).reshape(T, 1), W1.reshape(T, 1))


W2 = np.array([[1.0, 1.0], [1.0, -1.0], [0.5, 0.5], [-1.0, 1e-40], [1e-40, 1e-40],
               [0.0, 1.0], [-0.0, -0.0], [1.0, 2.0 ** -24]], np.float32)


def test_every_finite_bf16_pairs_k2():
    """k = 2: slot 0 takes every pattern in order, slot 1 the same patterns
    reversed (the largest magnitudes meet the zeros, so no sum overflows);
    cancellations, signed zeros and subnormal sums included."""
    T = W2.shape[0]
    y = np.empty((2 * T, H), np.uint16)
    y[0::2] = ALL
    y[1::2] = ALL[::-1]
    slot_of = np.arange(2 * T, dtype=np.int32).reshape(T, 2)
    _check(y, slot_of, W2)


def test_random_finite_patterns_k8():
    """k = 8 over rows of random finite patterns (subnormals and zeros
    included) with weights drawn from the edge set and random fp32 values."""
    rng = np.random.default_rng(5)
    T, k, Hs = 64, 8, 4096
    # patterns up to 2^101 in magnitude: with |w| <= 1 no sum of eight can
    # overflow (an overflow could meet one of the other sign and give a NaN,
    # whose bits the two sides need not share)
    small = ALL[((ALL >> 7) & 0xFF) <= 127 + 100]
    y = small[rng.integers(0, small.size, size=(T * k, Hs))]
    edge = np.array([0.0, -0.0, 1.0, -1.0, 1e-40, 0.125], np.float32)
    w = np.where(rng.random((T, k)) < 0.5, edge[rng.integers(0, edge.size, (T, k))],
                 np.clip(rng.standard_normal((T, k)), -1, 1)).astype(np.float32)
    slot_of = rng.permutation(T * k).astype(np.int32).reshape(T, k)
    _check(y, slot_of, w.astype(np.float32))
