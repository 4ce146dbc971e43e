"""Expert parallelism across real ranks, host side, on CPU: two (and three)
gloo ranks run the exchange of combine_layout_moe_gb300.ep -- the counts
all-to-all, the split sizes read back to the host, the all-to-all-v of the
rows there and back -- with the local steps (layout, dispatch, reorder,
combine) replaced by CPU stand-ins.  The receive buffers, expert offsets and
combined outputs must equal the oracle's expert-parallel dispatch and combine
of all ranks' tokens.

The stand-ins: layout, dispatch and combine are the oracle's single-rank
functions; the reorder is written out below from its contract (source-major
segments -> expert-major).  The CUDA kernels behind the same phases are
checked against the oracle on the GPU (tests/test_gpu_ep.py)."""
import os
import socket
from types import SimpleNamespace

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from workloads.gen import random_case, expert_output


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


class CpuOps:
    """CPU stand-ins for the library's local steps (test scaffolding)."""

    def layout(self, topk_idx, E, W):
        c, o, ro, so, src = oracle.layout(topk_idx.numpy(), E, W)
        t = torch.from_numpy
        return SimpleNamespace(expert_counts=t(c), expert_offsets=t(o), rank_offsets=t(ro),
                               slot_of=t(so), src_of=t(src))

    def dispatch(self, x, slot_of):
        return _bf16(oracle.dispatch(_bits(x), slot_of.numpy()))

    def dispatch_quant(self, x, slot_of):
        q, sc = oracle.dispatch_quant(_bits(x), slot_of.numpy())
        return torch.from_numpy(q), torch.from_numpy(sc)

    def reorder(self, src, recv_counts, to_source, with_offsets):
        cnt = recv_counts.numpy().astype(np.int64)
        W, El = cnt.shape
        s_start = np.concatenate([[0], np.cumsum(cnt.reshape(-1))])[:-1].reshape(W, El)
        e_start = np.concatenate([[0], np.cumsum(cnt.T.reshape(-1))])[:-1].reshape(El, W).T
        perm = np.empty(int(cnt.sum()), np.int64)       # source-major row -> expert-major row
        for s in range(W):
            for el in range(El):
                n = cnt[s, el]
                perm[s_start[s, el]:s_start[s, el] + n] = e_start[s, el] + np.arange(n)
        bf = src.dtype == torch.bfloat16
        a = _bits(src) if bf else src.numpy()
        out = np.empty_like(a)
        if to_source:
            out[:] = a[perm]
        else:
            out[perm] = a
        offs = None
        if with_offsets:
            offs = torch.from_numpy(np.append(e_start[0], cnt.sum()).astype(np.int32))
        return (_bf16(out) if bf else torch.from_numpy(out)), offs

    def combine(self, y, slot_of, topk_w):
        return _bf16(oracle.combine(_bits(y), slot_of.numpy(), topk_w.numpy(), "bf16"))


def _inputs(W, T_per, H, k, E):
    return [random_case(500 + s, T_per[s], H, k, E, W) for s in range(W)]


def _rank_main(rank, W, port, T_per, H, k, E, q, quant=False):
    import torch.distributed as dist
    from combine_layout_moe_gb300 import ep
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=W)
    try:
        ins = _inputs(W, T_per, H, k, E)
        me = ins[rank]
        epl = ep.ExpertParallel(E, ops=CpuOps())
        recv, offs, handle = epl.dispatch(_bf16(me.x), torch.from_numpy(me.topk_idx), quant=quant)
        rows = recv[0].shape[0] if quant else recv.shape[0]
        # an expert that is not the identity: each receiver's own rows
        y = _bf16(expert_output(rows, H, seed=900 + rank))
        out = epl.combine(y, handle, torch.from_numpy(me.topk_w))
        got = (recv[0].numpy(), recv[1].numpy()) if quant else _bits(recv)
        q.put((rank, got, offs.numpy(), _bits(out), handle[1].recv_splits,
               handle[0].send_splits))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, repr(e)))
    finally:
        dist.destroy_process_group()


def _port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.mark.parametrize("W,T_per,H,k,E", [(2, [37, 23], 16, 2, 4), (2, [40, 0], 8, 3, 8),
                                           (3, [11, 29, 5], 24, 8, 6)])
def test_exchange_over_gloo_matches_oracle(W, T_per, H, k, E):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_rank_main, args=(r, W, port, T_per, H, k, E, q))
             for r in range(W)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(W):
        item = q.get(timeout=120)
        res[item[0]] = item
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(W):
        assert len(res[r]) > 2, res[r][1]
    ins = _inputs(W, T_per, H, k, E)
    counts, recv, _ = oracle.ep_dispatch([w.topk_idx for w in ins], [w.x for w in ins], E)
    El = E // W
    ys = [expert_output(len(recv[d]), H, seed=900 + d) for d in range(W)]
    outs = oracle.ep_combine([w.topk_idx for w in ins], [w.topk_w for w in ins], ys, E)
    for d in range(W):
        _, g_recv, g_offs, g_out, recv_splits, send_splits = res[d]
        assert np.array_equal(g_recv.reshape(recv[d].shape), recv[d])
        # local expert offsets: the expert-major start of each local expert
        want = np.concatenate([[0], np.cumsum(counts[d].sum(axis=0))])
        assert np.array_equal(g_offs, want)
        assert recv_splits == counts[d].sum(axis=1).tolist()
        assert send_splits == [int(counts[dd, d].sum()) for dd in range(W)]
        assert np.array_equal(g_out.reshape(outs[d].shape), outs[d])
        assert El >= 1


def test_virtual_step_on_cpu_stand_ins_matches_oracle():
    """The single-process driver (the exchange done by copies) with the same
    stand-ins: the phases compose to the oracle's result."""
    from combine_layout_moe_gb300 import ep
    W, H, k, E = 4, 8, 2, 8
    ins = _inputs(W, [9, 0, 14, 3], H, k, E)
    ys = {}

    def expert(recv, offs):
        d = len(ys)
        ys[d] = expert_output(recv.shape[0], H, seed=700 + d)
        return _bf16(ys[d])

    recv, offs, outs = ep.virtual_step([_bf16(w.x) for w in ins],
                                       [torch.from_numpy(w.topk_idx) for w in ins],
                                       [torch.from_numpy(w.topk_w) for w in ins], E,
                                       expert=expert, ops=CpuOps())
    _, o_recv, _ = oracle.ep_dispatch([w.topk_idx for w in ins], [w.x for w in ins], E)
    o_out = oracle.ep_combine([w.topk_idx for w in ins], [w.topk_w for w in ins],
                              [ys[d] for d in range(W)], E)
    for d in range(W):
        assert np.array_equal(_bits(recv[d]).reshape(o_recv[d].shape), o_recv[d])
        assert np.array_equal(_bits(outs[d]).reshape(o_out[d].shape), o_out[d])


@pytest.mark.parametrize("W,T_per,H,k,E", [(2, [37, 23], 256, 2, 4), (3, [11, 29, 0], 128, 8, 6)])
def test_fp8_exchange_over_gloo_matches_oracle(W, T_per, H, k, E):
    """The FP8 dispatch across ranks (UBEP Table 3: W8A8): each receiver gets
    the E4M3 codes and fp32 scales of the tokens routed to it, in the receive
    order of the bf16 path; the combine's return path is bf16 as before."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_rank_main, args=(r, W, port, T_per, H, k, E, q, True))
             for r in range(W)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(W):
        item = q.get(timeout=120)
        res[item[0]] = item
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(W):
        assert len(res[r]) > 2, res[r][1]
    ins = _inputs(W, T_per, H, k, E)
    counts, recv, src = oracle.ep_dispatch([w.topk_idx for w in ins], [w.x for w in ins], E)
    # each token's codes and scales: the oracle's FP8 dispatch of the token
    # alone (one slot per token); a received row holds its source token's
    tq, ts = [], []
    for w in ins:
        a, b = oracle.dispatch_quant(w.x, np.arange(w.T, dtype=np.int32).reshape(w.T, 1))
        tq.append(a)
        ts.append(b)
    tq, ts = np.concatenate(tq), np.concatenate(ts)
    ys = [expert_output(len(recv[d]), H, seed=900 + d) for d in range(W)]
    outs = oracle.ep_combine([w.topk_idx for w in ins], [w.topk_w for w in ins], ys, E)
    for d in range(W):
        _, (g_q, g_s), g_offs, g_out, _, _ = res[d]
        tok = src[d] // k
        assert np.array_equal(g_q, tq[tok])
        assert np.array_equal(g_s, ts[tok])
        assert np.array_equal(g_offs, np.concatenate([[0], np.cumsum(counts[d].sum(axis=0))]))
        assert np.array_equal(g_out.reshape(outs[d].shape), outs[d])


def test_virtual_step_fp8_needs_an_expert():
    """The FP8 receive buffers are (codes, scales) pairs: without an expert
    returning bf16 rows there is nothing to send back."""
    from combine_layout_moe_gb300 import ep
    ins = _inputs(2, [4, 4], 128, 2, 4)
    with pytest.raises(ValueError):
        ep.virtual_step([_bf16(w.x) for w in ins], [torch.from_numpy(w.topk_idx) for w in ins],
                        [torch.from_numpy(w.topk_w) for w in ins], 4, ops=CpuOps(), quant=True)


@pytest.mark.parametrize("T_per", [[13], [0]])
def test_single_rank_is_the_local_path(T_per):
    """W = 1: the exchange is the identity and the receive order is the
    rank's own dispatch order; empty batches pass through."""
    from combine_layout_moe_gb300 import ep
    H, k, E = 8, 3, 5
    ins = _inputs(1, T_per, H, k, E)
    ys = {}

    def expert(recv, offs):
        ys[0] = expert_output(recv.shape[0], H, seed=710)
        return _bf16(ys[0])

    recv, offs, outs = ep.virtual_step([_bf16(ins[0].x)], [torch.from_numpy(ins[0].topk_idx)],
                                       [torch.from_numpy(ins[0].topk_w)], E, expert=expert,
                                       ops=CpuOps())
    _, o_recv, _ = oracle.ep_dispatch([ins[0].topk_idx], [ins[0].x], E)
    assert np.array_equal(_bits(recv[0]).reshape(o_recv[0].shape), o_recv[0])
    # one rank: the expert-major receive order is the layout's own slot order
    assert np.array_equal(o_recv[0], oracle.dispatch(ins[0].x, oracle.layout(ins[0].topk_idx, E, 1)[3]))
    o_out = oracle.ep_combine([ins[0].topk_idx], [ins[0].topk_w], [ys[0]], E)
    assert np.array_equal(_bits(outs[0]).reshape(o_out[0].shape), o_out[0])
    assert offs[0].tolist() == [0] + np.cumsum(np.bincount(ins[0].topk_idx.ravel(), minlength=E)).tolist()
