"""Expert-parallel dispatch and combine across real ranks (one GPU each).

UBEP, section 2.3 / Figure 2 and section 4: each rank counts its tokens per
destination expert, sends every token to the rank of each expert it chose, and
the receiver, from the per-expert counts of every source, reorders the rows
contiguously per expert (Phase 5) into a receive region partitioned by source
and expert.  StrataCL Appendix D: the same counts and token-local offsets
bring the expert outputs back for combine.

Experts are spread over the W ranks of a process group in contiguous blocks of
El = E / W.  One step, on every rank:

  send      moe_layout with R = W over the rank's own tokens, then
            moe_dispatch (or moe_dispatch_quant: E4M3 codes and fp32 scales,
            UBEP Table 3's W8A8): the rank segments of the dispatched buffer
            are the rows for each destination rank, already in (local expert,
            token, slot) order
  exchange  an all-to-all of each rank's El counts per destination, read back
            to the host as the split sizes, then an all-to-all-v of the rows
  receive   moe_ep_reorder (moe_ep_reorder_rows for the FP8 codes and
            scales): source-major rows -> expert-major
  (experts run on the expert-major rows)
  return    moe_ep_reorder back to source-major, the reverse all-to-all-v;
            each rank then holds its own rows in its own dispatch order
  finish    moe_combine with the rank's slot map and router weights

The exchange goes through torch.distributed (NCCL on GPUs, whose all-to-all
is grouped point-to-point sends and receives); every other step is one of
the library's kernels.  The functions below are the phases; `ExpertParallel`
runs them with a process group, and `virtual_step` runs W ranks' phases in one
process on one GPU, the exchange done by copying each segment to its
receiver's buffer.  The local operations are taken from an `ops` object
(default: the CUDA library), so the exchange logic can be exercised on CPU
ranks with stand-ins.
"""
from __future__ import annotations

from typing import List, NamedTuple, Optional

import torch


class LibraryOps:
    """The local steps, on the CUDA library's kernels."""

    def __init__(self, err_word: Optional[torch.Tensor] = None):
        import combine_layout_moe_gb300 as m
        self.m = m
        self.err = err_word

    def layout(self, topk_idx, E, W):
        return self.m.moe_layout(topk_idx, E, W, err_word=self.err)

    def dispatch(self, x, slot_of):
        return self.m.moe_dispatch(x, slot_of, err_word=self.err)

    def dispatch_quant(self, x, slot_of):
        return self.m.moe_dispatch_quant(x, slot_of, err_word=self.err)

    def reorder(self, src, recv_counts, to_source, with_offsets):
        offs = None
        if with_offsets:
            offs = torch.empty(recv_counts.shape[1] + 1, dtype=torch.int32, device=src.device)
        if src.dtype == torch.bfloat16 and src.dim() == 2:
            dst = self.m.moe_ep_reorder(src, recv_counts, to_source=to_source,
                                        local_expert_offsets=offs, err_word=self.err)
        else:  # FP8 codes or scales: rows of any width
            dst = self.m.moe_ep_reorder_rows(src, recv_counts, to_source=to_source,
                                             local_expert_offsets=offs, err_word=self.err)
        return dst, offs

    def combine(self, y, slot_of, topk_w):
        return self.m.moe_combine(y, slot_of, topk_w, err_word=self.err)


class SendState(NamedTuple):
    layout: object               # the rank's Layout over its own tokens, R = W
    send: object                 # [T*k, H] bf16 rows, rank-segmented; or with FP8 a
                                 # (codes uint8 [T*k, H], scales fp32 [T*k, H/128]) pair
    send_counts: torch.Tensor    # [W, El] int32: rows for each destination's local experts
    send_splits: List[int]       # rows for each destination rank


class Received(NamedTuple):
    recv: object                         # [rows, H] expert-major (bf16, or the FP8 pair)
    local_expert_offsets: torch.Tensor   # [El+1] int32: each local expert's first row
    recv_counts: torch.Tensor            # [W, El] int32: rows from each source per local expert
    recv_splits: List[int]               # rows from each source rank


def send(x, topk_idx, E: int, W: int, ops, quant: bool = False) -> SendState:
    """Layout with R = W over this rank's tokens, then the dispatch (bf16, or
    FP8 codes and scales with `quant`); host readback of the rank offsets as
    the split sizes."""
    lay = ops.layout(topk_idx, E, W)
    rows = ops.dispatch_quant(x, lay.slot_of) if quant else ops.dispatch(x, lay.slot_of)
    ro = lay.rank_offsets.cpu().tolist()
    return SendState(lay, rows, lay.expert_counts.view(W, E // W),
                     [ro[d + 1] - ro[d] for d in range(W)])


def receive(land, recv_counts, ops) -> Received:
    """Source-major rows that arrived -> the expert-major receive buffer (an
    FP8 pair is reordered part by part on the same counts)."""
    if isinstance(land, tuple):
        codes, offs = ops.reorder(land[0], recv_counts, False, True)
        scales, _ = ops.reorder(land[1], recv_counts, False, False)
        recv = (codes, scales)
    else:
        recv, offs = ops.reorder(land, recv_counts, False, True)
    splits = recv_counts.sum(dim=1).cpu().tolist()
    return Received(recv, offs, recv_counts, [int(v) for v in splits])


def give_back(y, received: Received, ops):
    """Expert outputs (expert-major, the receive order) -> source-major, ready
    for the reverse exchange."""
    back, _ = ops.reorder(y, received.recv_counts, True, False)
    return back


def finish(y_own, state: SendState, topk_w, ops):
    """This rank's rows back in its own dispatch order -> the combined tokens."""
    return ops.combine(y_own, state.layout.slot_of, topk_w)


# ------------------------------------------------------------------ exchange

def exchange_counts(send_counts: torch.Tensor, group=None) -> torch.Tensor:
    """All-to-all of the [W, El] counts: row d goes to rank d; returns the
    [W, El] matrix whose row s came from rank s."""
    import torch.distributed as dist
    out = torch.empty_like(send_counts)
    dist.all_to_all_single(out, send_counts.contiguous(), group=group)
    return out


def exchange_rows(rows: torch.Tensor, send_splits, recv_splits, group=None) -> torch.Tensor:
    """All-to-all-v of rows: send_splits[d] rows to rank d, recv_splits[s]
    rows from rank s, received source by source."""
    import torch.distributed as dist
    out = rows.new_empty((int(sum(recv_splits)),) + tuple(rows.shape[1:]))
    dist.all_to_all_single(out, rows.contiguous(), output_split_sizes=list(recv_splits),
                           input_split_sizes=list(send_splits), group=group)
    return out


class ExpertParallel:
    """Dispatch and combine of one rank of a process group of W ranks, each
    holding E / W experts.

        ep = ExpertParallel(E)
        recv, offsets, handle = ep.dispatch(x, topk_idx)
        y = experts(recv, offsets)          # expert-major rows
        out = ep.combine(y, handle, topk_w)
    """

    def __init__(self, E: int, group=None, ops=None):
        import torch.distributed as dist
        self.group = group
        self.W = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if E % self.W != 0:
            raise ValueError(f"E = {E} experts do not divide over {self.W} ranks")
        self.E = E
        self.ops = ops if ops is not None else LibraryOps()

    def dispatch(self, x, topk_idx, quant: bool = False):
        """Returns (the expert-major receive buffer: bf16 rows, or with
        `quant` an (E4M3 codes, fp32 scales) pair; local expert offsets;
        the handle combine needs)."""
        st = send(x, topk_idx, self.E, self.W, self.ops, quant)
        recv_counts = exchange_counts(st.send_counts, self.group)
        recv_splits = recv_counts.sum(dim=1).cpu().tolist()
        if quant:
            land = tuple(exchange_rows(part, st.send_splits, recv_splits, self.group)
                         for part in st.send)
        else:
            land = exchange_rows(st.send, st.send_splits, recv_splits, self.group)
        rc = receive(land, recv_counts, self.ops)
        return rc.recv, rc.local_expert_offsets, (st, rc)

    def combine(self, y, handle, topk_w):
        st, rc = handle
        back = give_back(y, rc, self.ops)
        own = exchange_rows(back, rc.recv_splits, st.send_splits, self.group)
        return finish(own, st, topk_w, self.ops)


def virtual_step(xs, idxs, ws, E: int, expert=None, ops=None, quant: bool = False):
    """W ranks' dispatch -> experts -> combine in one process (one GPU): the
    same phases as ExpertParallel, with the all-to-alls done by copying each
    rank's segments into its receivers' buffers.  `expert(recv, offsets)`
    maps a rank's expert-major rows to its bf16 outputs (default: the
    received rows themselves; required with `quant`, whose receive buffers
    are (codes, scales) pairs).  Returns (per-rank receive buffers, per-rank
    local expert offsets, per-rank combined outputs)."""
    W = len(xs)
    ops = ops if ops is not None else LibraryOps()
    if quant and expert is None:
        raise ValueError("an FP8 dispatch needs an expert that returns bf16 rows")
    states = [send(x, i, E, W, ops, quant) for x, i in zip(xs, idxs)]
    # counts: receiver d gets row d of every source's [W, El] matrix
    recv_counts = [torch.stack([states[s].send_counts[d] for s in range(W)]) for d in range(W)]
    cut = [[0] + list(torch.tensor(st.send_splits).cumsum(0).tolist()) for st in states]

    def segments(part_of, d):
        return torch.cat([part_of(states[s].send)[cut[s][d]:cut[s][d + 1]] for s in range(W)])

    if quant:
        lands = [(segments(lambda p: p[0], d), segments(lambda p: p[1], d)) for d in range(W)]
    else:
        lands = [segments(lambda p: p, d) for d in range(W)]
    recs = [receive(lands[d], recv_counts[d], ops) for d in range(W)]
    ys = [r.recv if expert is None else expert(r.recv, r.local_expert_offsets) for r in recs]
    backs = [give_back(ys[d], recs[d], ops) for d in range(W)]
    bcut = [[0] + list(torch.tensor(r.recv_splits).cumsum(0).tolist()) for r in recs]
    owns = [torch.cat([backs[d][bcut[d][s]:bcut[d][s + 1]] for d in range(W)])
            for s in range(W)]
    outs = [finish(owns[s], states[s], ws[s], ops) for s in range(W)]
    return [r.recv for r in recs], [r.local_expert_offsets for r in recs], outs
