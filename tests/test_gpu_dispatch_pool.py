"""The dispatch kernels' shared pool of work (a CTA or warp takes a fixed
share, then draws the rest from a counter of the launch): every unit is copied
(and, FP8, every item quantised) exactly once whichever CTA or warp draws it,
on shapes that take the fixed share by percentage and by the whole units of
an equal split; the counter's slot is clean again for the next launch, for
the replays of a captured graph, and after more launches than there are
slots, from two streams at once.  Launches with few units per CTA take a
static split instead (no pool).  Each receive buffer is compared bit for bit
with the oracle's dispatch."""
import numpy as np
import pytest
import torch

import oracle
from workloads.gen import random_case

pytestmark = pytest.mark.gpu


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _case(seed, T, H, k, E):
    w = random_case(seed, T, H, k, E, 1)
    slot_of = oracle.layout(w.topk_idx, E, 1)[3]
    return w, slot_of


# (T, H, k, E): 8192 one-chunk rows (about 9 units per CTA: half of them
# drawn); 20000 rows of two unequal chunks (44 units per CTA); 3000 rows of two
# chunks (about 6.6 units per CTA: a static split, no pool); 911 single units
# (fewer units than CTAs could run)
SHAPES = [(8192, 256, 4, 32), (20000, 7168, 1, 4), (3000, 7168, 3, 24), (911, 64, 2, 8)]


@pytest.mark.parametrize("T,H,k,E", SHAPES)
def test_every_unit_copied_once(T, H, k, E):
    import combine_layout_moe_gb300 as m
    w, slot_of = _case(31, T, H, k, E)
    so = torch.from_numpy(slot_of).cuda()
    err = m.new_error_word()
    recv = torch.empty((T * k, H), dtype=torch.bfloat16, device="cuda")
    for rep in range(4):
        x = w.x if rep % 2 == 0 else w.x ^ np.uint16(0x0100 * (rep + 1))
        recv.fill_(float("nan"))
        m.moe_dispatch(_bf16(x), so, recv=recv, err_word=err)
        torch.cuda.synchronize()
        assert m.moe_read_error(err) == 0
        assert np.array_equal(_bits(recv).reshape(T * k, H), oracle.dispatch(x, slot_of)), rep


def test_graph_replays_reuse_a_clean_slot():
    import combine_layout_moe_gb300 as m
    T, H, k, E = SHAPES[0]
    w, slot_of = _case(32, T, H, k, E)
    so = torch.from_numpy(slot_of).cuda()
    err = m.new_error_word()
    x = _bf16(w.x)
    recv = torch.empty((T * k, H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.moe_dispatch(x, so, recv=recv, err_word=err)   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.moe_dispatch(x, so, recv=recv, err_word=err)
    for rep in range(4):
        xr = w.x ^ np.uint16(0x0010 * (rep + 1))
        x.copy_(_bf16(xr))
        recv.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert m.moe_read_error(err) == 0
        assert np.array_equal(_bits(recv).reshape(T * k, H), oracle.dispatch(xr, slot_of)), rep


def test_more_launches_than_slots_on_two_streams():
    """1100 launches per stream (the slot table holds 1024), the two streams'
    launches free to overlap; each stream's buffer is checked every 100
    launches and at the end."""
    import combine_layout_moe_gb300 as m
    T, H, k, E = 8192, 64, 2, 8    # about 9 units per CTA: the pool
    cases = [_case(40 + i, T, H, k, E) for i in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    errs = [m.new_error_word() for _ in range(2)]
    xs = [_bf16(w.x) for w, _ in cases]
    sos = [torch.from_numpy(so).cuda() for _, so in cases]
    recvs = [torch.empty((T * k, H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    want = [oracle.dispatch(w.x, so) for w, so in cases]
    torch.cuda.synchronize()
    for it in range(1100):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                if it % 100 == 99:
                    recvs[i].fill_(float("nan"))
                m.moe_dispatch(xs[i], sos[i], recv=recvs[i], err_word=errs[i], stream=streams[i])
        if it % 100 == 99:
            torch.cuda.synchronize()
            for i in range(2):
                assert m.moe_read_error(errs[i]) == 0
                assert np.array_equal(_bits(recvs[i]).reshape(T * k, H), want[i]), (it, i)


# FP8 (T, H, k, E): 20000 tokens of one 256-channel item (5 rounds of the
# resident warps: the pool); 6000 tokens of 7168 channels (about 9 rounds)
FP8_SHAPES = [(20000, 256, 8, 64), (6000, 7168, 3, 24)]


@pytest.mark.parametrize("T,H,k,E", FP8_SHAPES)
def test_fp8_every_item_once(T, H, k, E):
    import combine_layout_moe_gb300 as m
    w, slot_of = _case(51, T, H, k, E)
    so = torch.from_numpy(slot_of).cuda()
    err = m.new_error_word()
    q = torch.empty((T * k, H), dtype=torch.uint8, device="cuda")
    sc = torch.empty((T * k, H // 128), dtype=torch.float32, device="cuda")
    for rep in range(3):
        x = w.x if rep == 0 else w.x ^ np.uint16(0x0010 * rep)
        q.fill_(0x5A)
        sc.fill_(-1.0)
        m.moe_dispatch_quant(_bf16(x), so, recv_q=q, recv_scales=sc, err_word=err)
        torch.cuda.synchronize()
        assert m.moe_read_error(err) == 0
        rq, rs = oracle.dispatch_quant(x, slot_of)
        assert np.array_equal(q.cpu().numpy(), rq), rep
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), rs.view(np.uint32)), rep


def test_fp8_graph_replays_reuse_a_clean_slot():
    import combine_layout_moe_gb300 as m
    T, H, k, E = FP8_SHAPES[0]
    w, slot_of = _case(52, T, H, k, E)
    so = torch.from_numpy(slot_of).cuda()
    err = m.new_error_word()
    x = _bf16(w.x)
    q = torch.empty((T * k, H), dtype=torch.uint8, device="cuda")
    sc = torch.empty((T * k, H // 128), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.moe_dispatch_quant(x, so, recv_q=q, recv_scales=sc, err_word=err)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.moe_dispatch_quant(x, so, recv_q=q, recv_scales=sc, err_word=err)
    for rep in range(3):
        xr = w.x ^ np.uint16(0x0020 * (rep + 1))
        x.copy_(_bf16(xr))
        q.fill_(0x5A)
        g.replay()
        torch.cuda.synchronize()
        assert m.moe_read_error(err) == 0
        rq, rs = oracle.dispatch_quant(xr, slot_of)
        assert np.array_equal(q.cpu().numpy(), rq), rep
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), rs.view(np.uint32)), rep
