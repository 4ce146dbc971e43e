"""Expert parallelism across ranks on the GPU: W virtual ranks in one process
run the phases of combine_layout_moe_gb300.ep (layout with R = W, dispatch,
the receiver's reorder, the reverse reorder, combine) through the library's
kernels, the all-to-alls done by copying each segment into its receiver's
buffer.  Receive buffers, local expert offsets and combined outputs must be
bit-identical to the oracle's expert-parallel dispatch and combine."""
import numpy as np
import pytest
import torch

import oracle
from workloads.gen import make_workload, random_case, expert_output

pytestmark = pytest.mark.gpu


def bf16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _run(ins, E, H):
    import combine_layout_moe_gb300 as m
    from combine_layout_moe_gb300 import ep
    W = len(ins)
    err = m.new_error_word()
    ys = {}

    def expert(recv, offs):        # each receiver's own synthetic outputs
        d = len(ys)
        ys[d] = expert_output(recv.shape[0], H, seed=300 + d)
        return bf16_dev(ys[d])

    recv, offs, outs = ep.virtual_step([bf16_dev(w.x) for w in ins],
                                       [torch.from_numpy(w.topk_idx).cuda() for w in ins],
                                       [torch.from_numpy(w.topk_w).cuda() for w in ins], E,
                                       expert=expert, ops=ep.LibraryOps(err))
    torch.cuda.synchronize()
    assert m.moe_read_error(err) == 0
    counts, o_recv, _ = oracle.ep_dispatch([w.topk_idx for w in ins], [w.x for w in ins], E)
    o_out = oracle.ep_combine([w.topk_idx for w in ins], [w.topk_w for w in ins],
                              [ys[d] for d in range(W)], E)
    for d in range(W):
        assert np.array_equal(bits(recv[d]).reshape(o_recv[d].shape), o_recv[d]), d
        want = np.concatenate([[0], np.cumsum(counts[d].sum(axis=0))])
        assert np.array_equal(offs[d].cpu().numpy(), want), d
        assert np.array_equal(bits(outs[d]).reshape(o_out[d].shape), o_out[d]), d


@pytest.mark.parametrize("name,W,T", [("mixtral", 8, 4096), ("mixtral", 2, 4096),
                                      ("dsv3_decode", 8, 256), ("glm45_air", 4, 512),
                                      ("dsv3_prefill", 32, 64)])
def test_virtual_ranks_match_oracle(name, W, T):
    """The workloads' routing recipes, W ranks of T tokens each (rank s draws
    with seed s), experts spread over the W ranks."""
    ins = [make_workload(name, seed=s, T=T) for s in range(W)]
    _run(ins, ins[0].E, ins[0].H)


@pytest.mark.parametrize("W,T_per,H,k,E", [(2, [300, 0], 24, 3, 4), (3, [1, 2, 3], 8, 1, 3),
                                           (4, [100, 7, 0, 250], 1000, 8, 1024),
                                           (16, [64] * 16, 136, 5, 32)])
def test_virtual_ranks_fuzz(W, T_per, H, k, E):
    ins = [random_case(600 + s, T_per[s], H, k, E, W) for s in range(W)]
    _run(ins, E, H)


def test_reorder_round_trip_and_offsets():
    """to-expert then to-source returns the rows; offsets as documented."""
    import combine_layout_moe_gb300 as m
    W, El, H = 5, 3, 64
    rng = np.random.default_rng(1)
    cnt = rng.integers(0, 9, size=(W, El)).astype(np.int32)
    cnt[2] = 0
    rows = int(cnt.sum())
    src = bf16_dev(rng.integers(0, 1 << 16, size=(rows, H), dtype=np.uint32)
                   .astype(np.uint16) & 0x7F7F)
    rc = torch.from_numpy(cnt).cuda()
    offs = torch.empty(El + 1, dtype=torch.int32, device="cuda")
    fwd = m.moe_ep_reorder(src, rc, local_expert_offsets=offs)
    back = m.moe_ep_reorder(fwd, rc, to_source=True)
    torch.cuda.synchronize()
    assert torch.equal(back.view(torch.int16), src.view(torch.int16))
    assert offs.cpu().tolist() == [0] + np.cumsum(cnt.sum(axis=0)).tolist()
    # row by row: source-major segment (s, el) lands at the expert-major start
    s_start = np.concatenate([[0], np.cumsum(cnt.reshape(-1))])
    e_start = np.concatenate([[0], np.cumsum(cnt.T.reshape(-1))])
    a, b = bits(src), bits(fwd)
    for s in range(W):
        for el in range(El):
            n = cnt[s, el]
            i0, j0 = s_start[s * El + el], e_start[el * W + s]
            assert np.array_equal(b[j0:j0 + n], a[i0:i0 + n])


def test_reorder_rejects_counts_that_do_not_add_up():
    import combine_layout_moe_gb300 as m
    err = m.new_error_word()
    rc = torch.tensor([[2, 1], [0, 3]], dtype=torch.int32, device="cuda")
    src = torch.zeros((5, 8), dtype=torch.bfloat16, device="cuda")   # counts sum to 6
    dst = torch.full((5, 8), 7.0, dtype=torch.bfloat16, device="cuda")
    m.moe_ep_reorder(src, rc, out=dst, err_word=err)
    assert m.moe_read_error(err) == m.MOE_ERRBIT_BAD_INDEX
    assert torch.all(dst == 7.0)                                      # nothing copied
    neg = torch.tensor([[3, -1], [0, 3]], dtype=torch.int32, device="cuda")
    m.moe_ep_reorder(src, neg, out=dst, err_word=err)
    assert m.moe_read_error(err) == m.MOE_ERRBIT_BAD_INDEX


def test_reorder_empty():
    import combine_layout_moe_gb300 as m
    rc = torch.zeros((3, 2), dtype=torch.int32, device="cuda")
    offs = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    out = m.moe_ep_reorder(torch.zeros((0, 8), dtype=torch.bfloat16, device="cuda"), rc,
                           local_expert_offsets=offs)
    torch.cuda.synchronize()
    assert out.shape == (0, 8) and offs.cpu().tolist() == [0, 0, 0]


@pytest.mark.parametrize("name,W,T", [("dsv3_prefill", 8, 128), ("glm45_air", 4, 256),
                                      ("mixtral", 2, 1024)])
def test_virtual_ranks_fp8_dispatch(name, W, T):
    """The FP8 dispatch across ranks: every receiver holds the E4M3 codes and
    fp32 scales of its tokens in the bf16 path's receive order (codes and
    scales reordered as rows of H and H / 128 * 4 bytes); the return path is
    bf16."""
    import combine_layout_moe_gb300 as m
    from combine_layout_moe_gb300 import ep
    ins = [make_workload(name, seed=s, T=T) for s in range(W)]
    E, H, k = ins[0].E, ins[0].H, ins[0].k
    err = m.new_error_word()
    ys = {}

    def expert(recv, offs):
        d = len(ys)
        ys[d] = expert_output(recv[0].shape[0], H, seed=400 + d)
        return bf16_dev(ys[d])

    recv, offs, outs = ep.virtual_step([bf16_dev(w.x) for w in ins],
                                       [torch.from_numpy(w.topk_idx).cuda() for w in ins],
                                       [torch.from_numpy(w.topk_w).cuda() for w in ins], E,
                                       expert=expert, ops=ep.LibraryOps(err), quant=True)
    torch.cuda.synchronize()
    assert m.moe_read_error(err) == 0
    counts, _, src = oracle.ep_dispatch([w.topk_idx for w in ins], [w.x for w in ins], E)
    tq = np.concatenate([oracle.dispatch_quant(w.x, np.arange(w.T, dtype=np.int32)[:, None])[0]
                         for w in ins])
    ts = np.concatenate([oracle.dispatch_quant(w.x, np.arange(w.T, dtype=np.int32)[:, None])[1]
                         for w in ins])
    o_out = oracle.ep_combine([w.topk_idx for w in ins], [w.topk_w for w in ins],
                              [ys[d] for d in range(W)], E)
    for d in range(W):
        tok = src[d] // k
        assert np.array_equal(recv[d][0].cpu().numpy(), tq[tok]), d
        assert np.array_equal(recv[d][1].cpu().numpy(), ts[tok]), d
        want = np.concatenate([[0], np.cumsum(counts[d].sum(axis=0))])
        assert np.array_equal(offs[d].cpu().numpy(), want), d
        assert np.array_equal(bits(outs[d]).reshape(o_out[d].shape), o_out[d]), d


@pytest.mark.parametrize("shape,dtype", [((37, 1), torch.float32), ((50, 56), torch.float32),
                                         ((30, 3), torch.float32), ((64, 7168), torch.uint8),
                                         ((20, 12), torch.int32)])
def test_reorder_rows_of_any_width(shape, dtype):
    """moe_ep_reorder_rows on 4-byte rows (one fp32 scale), scale rows of a
    7168-channel token, 12-byte rows (4-byte copies), FP8 code rows, and
    48-byte rows: round trip and the expert-major placement."""
    import combine_layout_moe_gb300 as m
    W, El = 3, 2
    rng = np.random.default_rng(3)
    cnt = rng.integers(0, 8, size=(W, El)).astype(np.int32)
    rows = int(cnt.sum())
    full = (rows,) + shape[1:]
    src = torch.from_numpy(rng.integers(0, 100, size=full).astype(
        {torch.float32: np.float32, torch.uint8: np.uint8, torch.int32: np.int32}[dtype])).cuda()
    rc = torch.from_numpy(cnt).cuda()
    fwd = m.moe_ep_reorder_rows(src, rc)
    back = m.moe_ep_reorder_rows(fwd, rc, to_source=True)
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    s_start = np.concatenate([[0], np.cumsum(cnt.reshape(-1))])
    e_start = np.concatenate([[0], np.cumsum(cnt.T.reshape(-1))])
    a, b = src.cpu().numpy(), fwd.cpu().numpy()
    for s in range(W):
        for el in range(El):
            n = cnt[s, el]
            assert np.array_equal(b[e_start[el * W + s]:e_start[el * W + s] + n],
                                  a[s_start[s * El + el]:s_start[s * El + el] + n])
