"""Pins for the oracle's bf16 dispatch and FP8-quantising dispatch.

Dispatch copies each token row to its k slots (UBEP section 2.3, Phase 2; the
receive buffer is packed without padding, RailWave section 3.2).  The FP8
variant follows the stated reading of UBEP Table 3's "W8A8": 1x128 blocks,
scale = amax/448, codes = e4m3_satfinite(x * (448/amax)).  The E4M3 encoder is
pinned against torch's float8_e4m3fn cast (an independent implementation) on
every code, every rounding midpoint and random inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads.gen import make_workload, random_case, bf16_bits_to_f32


def _row_source(idx):
    return np.argsort(idx.ravel(), kind="stable") // idx.shape[1]


@pytest.mark.parametrize("case", [("tiny", None), ("dsv3_decode", 64), ("mixtral", 256),
                                  ("glm45_air", 96), ("fuzz", 0), ("fuzz", 1)])
def test_dispatch_rows_equal_source_token(case):
    name, T = case
    if name == "fuzz":
        w = random_case(7 + T, 50, 64, 5, 6, 3)
    else:
        w = make_workload(name, T=T)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    recv = oracle.dispatch(w.x, slot_of)
    assert recv.shape == (w.N, w.H)
    assert np.array_equal(recv, w.x[_row_source(w.topk_idx)])


def test_dispatch_hand_worked():
    idx = np.array([[2, 0], [1, 2], [0, 0]], np.int32)
    x = np.array([[1, 2], [3, 4], [5, 6]], np.uint16)  # arbitrary bit patterns
    _, _, _, slot_of, _ = oracle.layout(idx, 4, 2)
    recv = oracle.dispatch(x, slot_of)
    assert recv.tolist() == [[1, 2], [5, 6], [5, 6], [3, 4], [1, 2], [3, 4]]


def test_dispatch_rejects_out_of_range_slot():
    x = np.zeros((2, 8), np.uint16)
    with pytest.raises(oracle.OracleError):
        oracle.dispatch(x, np.array([[0], [2]], np.int32))


# ---------------------------------------------------------------- E4M3 encoder

def _torch_e4m3(f: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.clip(f.astype(np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _all_code_values():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    return codes, vals


def test_e4m3_every_code_round_trips():
    codes, vals = _all_code_values()
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_e4m3_midpoints_and_neighbours_match_torch():
    codes, vals = _all_code_values()
    pos = np.unique(vals[vals >= 0]).astype(np.float64)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)          # exact in fp32
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(np.inf)), pos.astype(np.float32)])
    near = np.concatenate([near, -near])
    assert np.array_equal(oracle.e4m3_encode(near), _torch_e4m3(near))


def test_e4m3_random_and_saturating_match_torch():
    rng = np.random.default_rng(5)
    mant = rng.random(1 << 20, dtype=np.float32) + 1.0
    expo = rng.integers(-30, 12, size=mant.size)
    sign = rng.choice(np.array([-1.0, 1.0], np.float32), size=mant.size)
    f = (sign * np.ldexp(mant, expo)).astype(np.float32)
    f = np.concatenate([f, np.array([448, 449, 463.9, 464, 480, 1e30, np.inf, -np.inf,
                                     -0.0, 0.0, 2 ** -10, 2 ** -9, 1.5 * 2 ** -9,
                                     2.5 * 2 ** -9, 1e-45], np.float32)])
    assert np.array_equal(oracle.e4m3_encode(f), _torch_e4m3(f))


def test_e4m3_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(6)
    f = (rng.standard_normal(1 << 18).astype(np.float32) * 64).astype(np.float32)
    f = np.clip(f, -448, 448)
    ref = f.astype(ml.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(f), ref)


# --------------------------------------------------------- quantising dispatch

def _decode(q):
    return torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float32).numpy()


@pytest.mark.parametrize("case", [("dsv3_prefill", 48), ("tiny", None), ("fuzz", 0)])
def test_quant_block_invariants(case):
    name, T = case
    w = random_case(11, 40, 384, 3, 4, 2) if name == "fuzz" else make_workload(name, T=T)
    _, _, _, slot_of, src_of = oracle.layout(w.topk_idx, w.E, w.R)
    q, sc = oracle.dispatch_quant(w.x, slot_of)
    B = w.H // 128
    assert q.shape == (w.N, w.H) and sc.shape == (w.N, B)
    src_tok = _row_source(w.topk_idx)
    xf = bf16_bits_to_f32(w.x)[src_tok].reshape(w.N, B, 128).astype(np.float64)
    qv = _decode(q).reshape(w.N, B, 128).astype(np.float64)
    amax = np.abs(xf).max(axis=2)
    assert np.all(amax > 0)
    # scale is amax/448 to within one fp32 rounding
    assert np.allclose(sc, amax / 448.0, rtol=2 ** -23, atol=0)
    # the block's largest element encodes to +-448
    am = np.abs(xf).argmax(axis=2)
    top = np.take_along_axis(qv, am[..., None], axis=2)[..., 0]
    assert np.all(np.abs(top) == 448.0)
    # dequantised value is within half an E4M3 step (times the scale) of x,
    # plus three fp32 roundings of x
    aq = np.abs(qv)
    e = np.floor(np.log2(np.maximum(aq, 2.0 ** -6)))
    half_step = np.where(aq < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))
    err = np.abs(qv * sc[..., None].astype(np.float64) - xf)
    bound = half_step * sc[..., None] + np.abs(xf) * 4 * 2.0 ** -24
    assert np.all(err <= bound)
    # all k copies of a token are identical
    for t in range(min(w.T, 8)):
        rows = slot_of[t]
        assert all(np.array_equal(q[rows[0]], q[r]) and np.array_equal(sc[rows[0]], sc[r])
                   for r in rows)


def test_quant_zero_and_tiny_blocks():
    x = np.zeros((2, 384), np.uint16)
    x[0, 128:256] = 0x8000                                  # -0.0 block
    x[1, 0:128] = 0x3F80                                    # 1.0 block
    x[1, 128] = 0x0001                                      # amax ~9e-41: 448/amax overflows
    x[1, 129] = 0x8001
    x[1, 256:384] = 0x0000
    idx = np.array([[0], [1]], np.int32)
    _, _, _, slot_of, _ = oracle.layout(idx, 2, 1)
    q, sc = oracle.dispatch_quant(x, slot_of)
    assert sc[0].tolist() == [1.0, 1.0, 1.0]                # zero blocks: scale 1
    assert sc[1, 0] == np.float32(1.0 / 448.0)             # amax 1: 1/448 in fp32
    assert sc[1, 1:].tolist() == [1.0, 1.0]                # overflowing 448/amax, zero
    assert np.all(q[0, :128] == 0) and np.all(q[0, 128:256] == 0x80) and np.all(q[0, 256:] == 0)
    assert np.all(q[1, :128] == 0x7E)
    assert q[1, 128] == 0x00 and q[1, 129] == 0x80 and np.all(q[1, 130:] == 0)


def test_quant_rejects_ragged_hidden():
    with pytest.raises(oracle.OracleError):
        oracle.dispatch_quant(np.zeros((1, 200), np.uint16), np.zeros((1, 1), np.int32))
