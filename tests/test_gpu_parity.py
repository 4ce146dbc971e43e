"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Layout (counts, offsets, slot maps) and dispatched payloads (bf16 rows, E4M3
codes, fp32 scales) must be bit-identical.  Combine must be within 1 bf16 ulp
(ordered-integer distance of the bit patterns) of the oracle's fp32-accumulated
result; both sides do one fused multiply-add per slot in slot order, so the
tests also require exact equality.  Every named workload runs at its full size,
through the same entry points and launch configuration the benchmark times.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from workloads.gen import CONFIG_ORDER, make_workload, random_case, expert_output

pytestmark = pytest.mark.gpu


def cl():
    import combine_layout_moe_gb300 as m
    return m


@functools.lru_cache(maxsize=2)
def workload(name):
    return make_workload(name)


def bf16_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def i32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def run_layout(idx, E, R, err=None):
    m = cl()
    lay = m.moe_layout(i32_dev(idx), E, R, err_word=err)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in lay]


def assert_layout_equal(idx, E, R):
    g = run_layout(idx, E, R)
    o = oracle.layout(idx, E, R)
    for name, a, b in zip(["expert_counts", "expert_offsets", "rank_offsets", "slot_of", "src_of"],
                          g, o):
        assert a.shape == b.shape, name
        assert np.array_equal(a, b), f"{name} differs at {np.flatnonzero(a.ravel() != b.ravel())[:8]}"


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|ordered-int(a) - ordered-int(b)| for bf16 bit patterns."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + (x & 0x7FFF))
    return np.abs(ordered(a) - ordered(b))


# ------------------------------------------------------------------- layout

@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_layout_matches_oracle(name):
    w = workload(name)
    assert_layout_equal(w.topk_idx, w.E, w.R)


FUZZ = [  # (seed, T, k, E, R)
    (1, 1, 1, 1, 1), (2, 1, 8, 256, 32), (3, 3, 5, 7, 7), (4, 33, 2, 16, 4), (5, 100, 8, 8, 1),
    (6, 257, 4, 256, 32), (7, 4097, 3, 5, 5), (8, 5000, 8, 1024, 8), (9, 12345, 6, 64, 16),
    (10, 70000, 2, 2, 2), (11, 100000, 8, 128, 16), (12, 300000, 8, 256, 32),
    (13, 2049, 1, 3, 1), (14, 511, 16, 40, 10), (15, 40, 33, 9, 3),
    # around the one-cluster form (at most 16 tiles of ~1024 pairs; above 8 a
    # non-portable cluster): 8000 pairs with the largest expert count, 8192
    # pairs (8 tiles), 8193 (9), 12000 (12), 16384 (16) and 16385 (17 tiles:
    # the grid-barrier form)
    (16, 1000, 8, 1024, 8), (17, 4096, 2, 32, 4), (18, 8193, 1, 64, 4),
    (19, 1500, 8, 1024, 32), (20, 2048, 8, 256, 32), (21, 16385, 1, 16, 4),
]


# The form each straddling shape must take on a GB300 (clusters of 9..16 CTAs
# are non-portable sizes, which the launcher uses only where the GPU can place
# them; GB300 can): a silent fall-back to the grid barrier would still pass the
# parity check, so the form is checked as well.
FUZZ_FORM = {16: "CLUSTER", 17: "CLUSTER", 18: "CLUSTER", 19: "CLUSTER", 20: "CLUSTER",
             21: "COOPERATIVE", 1: "SINGLE", 2: "SINGLE", 3: "SINGLE", 5: "SINGLE",
             12: "COOPERATIVE"}


@pytest.mark.parametrize("case", FUZZ, ids=[f"s{c[0]}_T{c[1]}_k{c[2]}_E{c[3]}" for c in FUZZ])
def test_layout_fuzz(case):
    seed, T, k, E, R = case
    w = random_case(seed, T, 8, k, E, R)
    assert_layout_equal(w.topk_idx, E, R)
    if seed in FUZZ_FORM:
        m = cl()
        assert m.moe_layout_last_form() == getattr(m, "MOE_LAYOUT_FORM_" + FUZZ_FORM[seed])


def test_layout_all_one_expert_and_hot_expert():
    T, k, E = 20000, 4, 64
    idx = np.full((T, k), 17, np.int32)
    assert_layout_equal(idx, E, 8)
    idx[::3, 1] = 5
    assert_layout_equal(idx, E, 8)


def test_layout_is_deterministic():
    w = workload("glm45_air")
    a = run_layout(w.topk_idx, w.E, w.R)
    b = run_layout(w.topk_idx, w.E, w.R)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_layout_empty():
    m = cl()
    lay = m.moe_layout(torch.zeros((0, 4), dtype=torch.int32, device="cuda"), 8, 2)
    torch.cuda.synchronize()
    assert lay.expert_counts.cpu().tolist() == [0] * 8
    assert lay.expert_offsets.cpu().tolist() == [0] * 9
    assert lay.rank_offsets.cpu().tolist() == [0] * 3


@pytest.mark.parametrize("T", [64, 2048, 6000, 20000])  # one tile, clusters of 4 and 12, the grid barrier
def test_layout_bad_index_reported(T):
    m = cl()
    err = m.new_error_word()
    idx = np.zeros((T, 2), np.int32)
    idx[10, 1] = 8
    idx[T - 20, 0] = -3
    m.moe_layout(i32_dev(idx), 8, 2, err_word=err)
    assert m.moe_read_error(err) & m.MOE_ERRBIT_BAD_INDEX
    assert m.moe_read_error(err) == 0          # cleared by the first read
    m.moe_layout(i32_dev(np.zeros((T, 2), np.int32)), 8, 2, err_word=err)
    assert m.moe_read_error(err) == 0


def test_invalid_arguments_rejected():
    m = cl()
    idx = i32_dev(np.zeros((4, 2), np.int32))
    with pytest.raises(m.MoeError) as ei:
        m.moe_layout(idx, 6, 4)                # E % R != 0
    assert ei.value.status == m.MOE_ERR_INVALID_ARG
    x = torch.zeros((4, 12), dtype=torch.bfloat16, device="cuda")
    so = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(m.MoeError):
        m.moe_dispatch(x, so)                  # H % 8 != 0
    with pytest.raises(m.MoeError):
        m.moe_dispatch_quant(torch.zeros((4, 192), dtype=torch.bfloat16, device="cuda"), so)
    with pytest.raises(m.MoeError) as ei:
        m.moe_layout(i32_dev(np.zeros((4, 2), np.int32)), 2048, 2)
    assert ei.value.status == m.MOE_ERR_UNSUPPORTED


# ----------------------------------------------------------------- dispatch

@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_dispatch_bf16_matches_oracle(name):
    m = cl()
    w = workload(name)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    lay = m.moe_layout(i32_dev(w.topk_idx), w.E, w.R)
    recv = m.moe_dispatch(bf16_dev(w.x), lay.slot_of)
    ref = oracle.dispatch(w.x, slot_of)
    got = bits(recv)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("name", ["dsv3_prefill", "tiny", "dsv3_decode"])
def test_dispatch_quant_matches_oracle(name):
    m = cl()
    w = workload(name)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    lay = m.moe_layout(i32_dev(w.topk_idx), w.E, w.R)
    q, sc = m.moe_dispatch_quant(bf16_dev(w.x), lay.slot_of)
    rq, rs = oracle.dispatch_quant(w.x, slot_of)
    gq = q.cpu().numpy()
    assert np.array_equal(gq, rq), f"{(gq != rq).sum()} code bytes differ"
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), rs.view(np.uint32))


PAYLOAD_FUZZ = [  # (seed, T, H, k, E, R)
    (21, 1, 128, 1, 1, 1), (22, 37, 384, 3, 6, 2), (23, 300, 896, 8, 32, 4),
    (24, 129, 7168, 5, 10, 5), (25, 1000, 4096, 2, 8, 8), (26, 17, 1280, 16, 4, 1),
]


@pytest.mark.parametrize("case", PAYLOAD_FUZZ, ids=[f"s{c[0]}_T{c[1]}_H{c[2]}_k{c[3]}" for c in PAYLOAD_FUZZ])
def test_dispatch_and_quant_fuzz(case):
    m = cl()
    seed, T, H, k, E, R = case
    w = random_case(seed, T, H, k, E, R)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, E, R)
    lay = m.moe_layout(i32_dev(w.topk_idx), E, R)
    x = bf16_dev(w.x)
    assert np.array_equal(bits(m.moe_dispatch(x, lay.slot_of)), oracle.dispatch(w.x, slot_of))
    q, sc = m.moe_dispatch_quant(x, lay.slot_of)
    rq, rs = oracle.dispatch_quant(w.x, slot_of)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("H", [8, 24, 136, 1000, 7176])
def test_dispatch_ragged_hidden(H):
    """Rows whose 16-byte vector count is not a multiple of the warp's chunk."""
    m = cl()
    w = random_case(30 + H, 65, H, 3, 5, 1)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, 5, 1)
    lay = m.moe_layout(i32_dev(w.topk_idx), 5, 1)
    assert np.array_equal(bits(m.moe_dispatch(bf16_dev(w.x), lay.slot_of)),
                          oracle.dispatch(w.x, slot_of))


def test_e4m3_conversion_every_bf16_value():
    """Blocks of 127 values plus one 448 have amax 448 and reciprocal exactly 1,
    so the codes are the E4M3 encodings of the bf16 values themselves: every
    finite bf16 pattern with |x| <= 448 goes through the kernel's conversion."""
    m = cl()
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = (allb.astype(np.uint32) << 16).view(np.float32)
    vals = allb[np.isfinite(f) & (np.abs(f) <= 448.0)]
    nblk = -(-vals.size // 127)
    x = np.zeros((nblk, 128), np.uint16)
    flat = np.zeros(nblk * 127, np.uint16)
    flat[:vals.size] = vals
    x[:, :127] = flat.reshape(nblk, 127)
    x[:, 127] = 0x43E0                                  # 448.0
    T = nblk
    idx = np.zeros((T, 1), np.int32)
    _, _, _, slot_of, _ = oracle.layout(idx, 1, 1)
    q, sc = m.moe_dispatch_quant(bf16_dev(x), i32_dev(slot_of))
    rq, rs = oracle.dispatch_quant(x, slot_of)
    assert np.all(rs == 1.0)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(sc.cpu().numpy(), rs)


def test_quant_zero_and_tiny_blocks_on_gpu():
    m = cl()
    x = np.zeros((2, 384), np.uint16)
    x[0, 128:256] = 0x8000
    x[1, 0:128] = 0x3F80
    x[1, 128] = 0x0001
    x[1, 129] = 0x8001
    idx = np.array([[0], [1]], np.int32)
    _, _, _, slot_of, _ = oracle.layout(idx, 2, 1)
    q, sc = m.moe_dispatch_quant(bf16_dev(x), i32_dev(slot_of))
    rq, rs = oracle.dispatch_quant(x, slot_of)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(sc.cpu().numpy(), rs)


def test_dispatch_bad_slot_reported():
    m = cl()
    err = m.new_error_word()
    x = torch.ones((4, 64), dtype=torch.bfloat16, device="cuda")
    so = i32_dev(np.array([[0, 1], [2, 3], [4, 5], [6, 8]], np.int32))  # 8 >= T*k
    m.moe_dispatch(x, so, err_word=err)
    assert m.moe_read_error(err) == m.MOE_ERRBIT_BAD_INDEX


# ------------------------------------------------------------------ combine

def _combine_case(name):
    w = workload(name)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    return w, slot_of, expert_output(w.N, w.H, seed=w.seed)


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_combine_bf16_matches_oracle(name):
    m = cl()
    w, slot_of, y = _combine_case(name)
    out = m.moe_combine(bf16_dev(y), i32_dev(slot_of), torch.from_numpy(w.topk_w).cuda())
    got = bits(out)
    ref = oracle.combine(y, slot_of, w.topk_w, "bf16")
    d = ulp_distance(got, ref)
    assert d.max() <= 1, f"max ulp distance {d.max()}"
    assert np.array_equal(got, ref), f"{(d > 0).sum()} elements differ by 1 ulp"


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "mixtral"])
def test_combine_f32_matches_oracle(name):
    m = cl()
    w, slot_of, y = _combine_case(name)
    out = m.moe_combine(bf16_dev(y), i32_dev(slot_of), torch.from_numpy(w.topk_w).cuda(),
                        out_dtype=torch.float32)
    ref = oracle.combine(y, slot_of, w.topk_w, "f32")
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


COMBINE_FUZZ = [(41, 1, 8, 1, 1, 1), (42, 50, 264, 3, 5, 5), (43, 333, 2048, 8, 64, 8),
                (44, 77, 7176, 6, 12, 3), (45, 9, 64, 40, 7, 7), (46, 2000, 4096, 2, 8, 8),
                # k > 32 (the register fallback): several row batches, ragged H
                (47, 300, 7168, 40, 256, 32), (48, 50, 1000, 64, 64, 8), (49, 33, 2056, 33, 33, 11)]


@pytest.mark.parametrize("case", COMBINE_FUZZ, ids=[f"s{c[0]}_T{c[1]}_H{c[2]}_k{c[3]}" for c in COMBINE_FUZZ])
def test_combine_fuzz(case):
    m = cl()
    seed, T, H, k, E, R = case
    w = random_case(seed, T, H, k, E, R)
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, E, R)
    y = expert_output(w.N, H, seed=seed)
    for dt, od in ((torch.bfloat16, "bf16"), (torch.float32, "f32")):
        out = m.moe_combine(bf16_dev(y), i32_dev(slot_of), torch.from_numpy(w.topk_w).cuda(),
                            out_dtype=dt)
        ref = oracle.combine(y, slot_of, w.topk_w, od)
        got = bits(out) if od == "bf16" else out.cpu().numpy()
        assert np.array_equal(got.view(ref.dtype), ref)


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "glm45_air", "mixtral"])
def test_round_trip_identity_expert(name):
    """combine(dispatch(x)) with identity experts and weights summing to 1 is x."""
    m = cl()
    w = workload(name)
    lay = m.moe_layout(i32_dev(w.topk_idx), w.E, w.R)
    x = bf16_dev(w.x)
    recv = m.moe_dispatch(x, lay.slot_of)
    out = m.moe_combine(recv, lay.slot_of, torch.from_numpy(w.topk_w).cuda())
    got, ref = bits(out), w.x
    nz = (ref & 0x7FFF) != 0
    assert np.array_equal(got[nz], ref[nz])


def test_combine_bad_slot_reported():
    m = cl()
    err = m.new_error_word()
    y = torch.ones((8, 64), dtype=torch.bfloat16, device="cuda")
    so = i32_dev(np.array([[0, 1], [2, 3], [4, 5], [6, -1]], np.int32))
    w = torch.ones((4, 2), dtype=torch.float32, device="cuda")
    m.moe_combine(y, so, w, err_word=err)
    assert m.moe_read_error(err) == m.MOE_ERRBIT_BAD_INDEX


# ------------------------------------------------------- layout + dispatch

@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_layout_dispatch_matches_oracle(name):
    """The combined call, whose dispatch reads x while the layout still runs,
    gives the layout and rows of the two calls made in turn."""
    m = cl()
    w = workload(name)
    lay, recv = m.moe_layout_dispatch(bf16_dev(w.x), i32_dev(w.topk_idx), w.E, w.R)
    torch.cuda.synchronize()
    o = oracle.layout(w.topk_idx, w.E, w.R)
    for a, b in zip(lay, o):
        assert np.array_equal(a.cpu().numpy(), b)
    assert np.array_equal(bits(recv), oracle.dispatch(w.x, o[3]))


@pytest.mark.parametrize("case", [(71, 1, 8, 1, 1, 1), (72, 300, 1000, 33, 64, 8),
                                  (73, 5000, 2048, 8, 256, 32), (74, 0, 64, 2, 4, 2)])
def test_layout_dispatch_fuzz(case):
    m = cl()
    seed, T, H, k, E, R = case
    w = random_case(seed, T, H, k, E, R)
    lay, recv = m.moe_layout_dispatch(bf16_dev(w.x), i32_dev(w.topk_idx), E, R)
    torch.cuda.synchronize()
    o = oracle.layout(w.topk_idx, E, R)
    assert np.array_equal(lay.slot_of.cpu().numpy(), o[3])
    assert np.array_equal(bits(recv), oracle.dispatch(w.x, o[3]))


# Shapes of the single-kernel layout + dispatch (every CTA counts the whole
# batch itself; at most 16384 pairs, each CTA's share of x resident in shared
# memory): one token, ragged H, rows split in two units, k = 32 with the
# largest expert count, fewer units than SMs, a 2048-token decode batch (the
# largest share of x a CTA holds), and k = 5.  (seed, T, H, k, E, R)
FUSED = [(81, 1, 8, 1, 1, 1), (82, 7, 7176, 8, 256, 32), (83, 1024, 7168, 8, 256, 32),
         (84, 2048, 7168, 8, 256, 32), (85, 500, 12288, 4, 64, 8), (86, 512, 1000, 32, 1024, 16),
         (87, 3000, 512, 5, 7, 7), (88, 160, 4096, 2, 8, 8)]


@pytest.mark.parametrize("case", FUSED, ids=[f"s{c[0]}_T{c[1]}_H{c[2]}_k{c[3]}" for c in FUSED])
@pytest.mark.parametrize("aligned_ids", [True, False])
def test_layout_dispatch_single_kernel(case, aligned_ids):
    m = cl()
    seed, T, H, k, E, R = case
    w = random_case(seed, T, H, k, E, R)
    if aligned_ids:
        idx = i32_dev(w.topk_idx)
    else:  # ids 4 bytes past a 16-byte boundary: the kernel's scalar path
        buf = torch.zeros(T * k + 1, dtype=torch.int32, device="cuda")
        buf[1:] = i32_dev(w.topk_idx).view(-1)
        idx = buf[1:].view(T, k)
        assert idx.data_ptr() % 16 == 4
    err = m.new_error_word()
    lay, recv = m.moe_layout_dispatch(bf16_dev(w.x), idx, E, R, err_word=err)
    assert m.moe_layout_last_form() == m.MOE_LAYOUT_FORM_FUSED
    torch.cuda.synchronize()
    assert m.moe_read_error(err) == 0
    o = oracle.layout(w.topk_idx, E, R)
    for name, a, b in zip(["expert_counts", "expert_offsets", "rank_offsets", "slot_of", "src_of"],
                          lay, o):
        assert np.array_equal(a.cpu().numpy(), b), name
    assert np.array_equal(bits(recv), oracle.dispatch(w.x, o[3]))


def test_layout_dispatch_single_kernel_bad_id():
    m = cl()
    w = random_case(89, 300, 256, 4, 16, 4)
    idx = w.topk_idx.copy()
    idx[7, 2] = 16          # one past the last expert
    idx[200, 0] = -3
    err = m.new_error_word()
    lay, recv = m.moe_layout_dispatch(bf16_dev(w.x), i32_dev(idx), 16, 4, err_word=err)
    assert m.moe_layout_last_form() == m.MOE_LAYOUT_FORM_FUSED
    assert m.moe_read_error(err) == m.MOE_ERRBIT_BAD_INDEX
    so = lay.slot_of.cpu().numpy()
    assert so[7, 2] == -1 and so[200, 0] == -1
    # the valid pairs still take the slots of the stable order over valid ids
    good = (idx >= 0) & (idx < 16)
    order = np.argsort(np.where(good, idx, 1 << 20).ravel(), kind="stable")[:good.sum()]
    want = np.full(idx.size, -1, np.int64)
    want[order] = np.arange(good.sum())
    assert np.array_equal(so.ravel(), want)


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "dsv3_prefill", "glm45_air", "mixtral"])
def test_layout_dispatch_quant_matches_oracle(name):
    """The combined FP8 call, whose dispatch loads and quantises x while the
    layout still runs: the layout, codes and scales of the two calls in turn."""
    m = cl()
    w = workload(name)
    err = m.new_error_word()
    lay, q, sc = m.moe_layout_dispatch_quant(bf16_dev(w.x), i32_dev(w.topk_idx), w.E, w.R,
                                             err_word=err)
    assert m.moe_read_error(err) == 0
    o = oracle.layout(w.topk_idx, w.E, w.R)
    for a, b in zip(lay, o):
        assert np.array_equal(a.cpu().numpy(), b)
    rq, rs = oracle.dispatch_quant(w.x, o[3])
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(sc.cpu().numpy(), rs)


@pytest.mark.parametrize("case", [(91, 1, 128, 1, 1, 1), (92, 3000, 1024, 3, 12, 4),
                                  (93, 20000, 256, 8, 64, 8), (94, 0, 128, 2, 4, 2)])
def test_layout_dispatch_quant_fuzz(case):
    m = cl()
    seed, T, H, k, E, R = case
    w = random_case(seed, T, H, k, E, R)
    lay, q, sc = m.moe_layout_dispatch_quant(bf16_dev(w.x), i32_dev(w.topk_idx), E, R)
    torch.cuda.synchronize()
    o = oracle.layout(w.topk_idx, E, R)
    assert np.array_equal(lay.slot_of.cpu().numpy(), o[3])
    rq, rs = oracle.dispatch_quant(w.x, o[3])
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(sc.cpu().numpy(), rs)
