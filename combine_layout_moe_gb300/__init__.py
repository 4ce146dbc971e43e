"""GB300 MoE expert-parallel layout / dispatch / combine.

A thin ctypes binding over the C ABI of libmoe_ep.so (include/moe_ep.h).  The
functions carry the C names and only marshal arguments: they check dtypes and
shapes, allocate outputs with torch when none are given, and pass raw device
pointers and the current CUDA stream.  Every step of the path runs in the
library's sm_103a kernels; there is no CPU or PyTorch fallback.  If the
library is missing, importing this package fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_ep.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_BAD_INDEX, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, \
    MOE_ERR_UNSUPPORTED, MOE_ERR_INTEGRITY = range(7)
MOE_OUT_BF16, MOE_OUT_F32 = 0, 1
MOE_ERRBIT_BAD_INDEX, MOE_ERRBIT_TIMEOUT, MOE_ERRBIT_SENTINEL, MOE_ERRBIT_CHECKSUM = 0x1, 0x2, 0x4, 0x8
MOE_ERRBIT_LAUNCH = 0x10
MOE_LAYOUT_FORM_NONE, MOE_LAYOUT_FORM_SINGLE, MOE_LAYOUT_FORM_CLUSTER, \
    MOE_LAYOUT_FORM_COOPERATIVE, MOE_LAYOUT_FORM_FUSED = range(5)
MOE_SYNC_WORD, MOE_SYNC_SENTINEL, MOE_SYNC_BATCH, MOE_SYNC_BARRIER = range(4)
MOE_EP_TO_EXPERT, MOE_EP_TO_SOURCE = 0, 1
MOE_MAX_EXPERTS = 1024

# Every symbol the header declares, with its ctypes signature.
_P, _I, _SZ, _U32P = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
SIGNATURES = {
    "moe_abi_version": ([], ctypes.c_int),
    "moe_status_string": ([_I], ctypes.c_char_p),
    "moe_layout_workspace_bytes": ([_I, _I, _I], ctypes.c_size_t),
    "moe_layout": ([_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _U32P, _P], ctypes.c_int),
    "moe_dispatch": ([_I, _I, _I, _P, _P, _P, _U32P, _P], ctypes.c_int),
    "moe_layout_dispatch": ([_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _U32P,
                             _P], ctypes.c_int),
    "moe_dispatch_quant": ([_I, _I, _I, _P, _P, _P, _P, _U32P, _P], ctypes.c_int),
    "moe_layout_dispatch_quant": ([_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _SZ, _U32P, _P], ctypes.c_int),
    "moe_combine": ([_I, _I, _I, _P, _P, _P, _P, _I, _U32P, _P], ctypes.c_int),
    "moe_read_error": ([_U32P, _I, _P, ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
    "moe_layout_noalloc": ([_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _U32P, _P], ctypes.c_int),
    "moe_sync_words": ([_I, _I, _I, _I, _I], ctypes.c_size_t),
    "moe_layout_last_form": ([], ctypes.c_int),
    "moe_e4m3_encode_bits": ([ctypes.c_uint32, ctypes.c_uint32, _P, _P], ctypes.c_int),
    "moe_ep_reorder": ([_I, _I, _I, _P, _I, _P, _P, _I, _P, _U32P, _P], ctypes.c_int),
    "moe_ep_reorder_rows": ([_I, _I, _I, _P, _I, _P, _P, _I, _P, _U32P, _P], ctypes.c_int),
    "moe_combine_backward": ([_I, _I, _I, _P, _P, _P, _P, _P, _P, _U32P, _P], ctypes.c_int),
    "moe_dispatch_backward": ([_I, _I, _I, _P, _P, _P, _I, _U32P, _P], ctypes.c_int),
    "moe_layout_coalesced": ([_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _U32P, _P],
                             ctypes.c_int),
    "moe_dispatch_coalesced": ([_I, _I, _I, _P, _P, _I, _P, _U32P, _P], ctypes.c_int),
    "moe_dispatch_quant_coalesced": ([_I, _I, _I, _P, _P, _I, _P, _P, _U32P, _P], ctypes.c_int),
    "moe_combine_coalesced": ([_I, _I, _I, _P, _P, _P, _P, _I, _P, _P, _I, _U32P, _P],
                              ctypes.c_int),
    "moe_dispatch_combine_flagged": ([_I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P,
                                      ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int64, _U32P,
                                      _P], ctypes.c_int),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
            "or `python combine_layout_moe_gb300/build.py` first")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib.moe_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def _stream(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _want(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def moe_abi_version() -> int:
    return _lib.moe_abi_version()


def moe_status_string(status: int) -> str:
    return _lib.moe_status_string(status).decode()


def moe_e4m3_encode_bits(first: int, count: int, out: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The quantised dispatch's E4M3 encoding of the fp32 values with bit
    patterns first .. first + count - 1 (uint8 device tensor [count])."""
    if out is None:
        out = torch.empty(count, dtype=torch.uint8, device="cuda")
    _check(_lib.moe_e4m3_encode_bits(first & 0xffffffff, count, _ptr(out), _stream(stream)),
           "moe_e4m3_encode_bits")
    return out


def moe_layout_last_form() -> int:
    """MOE_LAYOUT_FORM_* of the layout kernel this host thread launched last."""
    return int(_lib.moe_layout_last_form())


def new_error_word(device=None) -> torch.Tensor:
    """A zero-filled device word for the kernels' error bits (int32 storage)."""
    return torch.zeros(4, dtype=torch.int32, device=device or "cuda")


def moe_layout_workspace_bytes(T: int, k: int, E: int) -> int:
    return int(_lib.moe_layout_workspace_bytes(T, k, E))


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A layout workspace: zero-filled once, as moe_layout requires; reusable
    for every later call whose moe_layout_workspace_bytes fits in it."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


class Layout(NamedTuple):
    expert_counts: torch.Tensor   # int32 [E]
    expert_offsets: torch.Tensor  # int32 [E+1]
    rank_offsets: torch.Tensor    # int32 [R+1]
    slot_of: torch.Tensor         # int32 [T, k]
    src_of: torch.Tensor          # int32 [T*k]


def moe_layout(topk_idx: torch.Tensor, E: int, R: int, *, workspace: Optional[torch.Tensor] = None,
               err_word: Optional[torch.Tensor] = None, out: Optional[Layout] = None,
               stream: Optional[torch.cuda.Stream] = None) -> Layout:
    """Count, scan and stable slot map of top-k router output (see moe_ep.h)."""
    if topk_idx.dim() != 2:
        raise ValueError("topk_idx must be [T, k]")
    T, k = topk_idx.shape
    _want(topk_idx, "topk_idx", torch.int32)
    dev = topk_idx.device
    if out is None:
        out = Layout(torch.empty(E, dtype=torch.int32, device=dev),
                     torch.empty(E + 1, dtype=torch.int32, device=dev),
                     torch.empty(R + 1, dtype=torch.int32, device=dev),
                     torch.empty((T, k), dtype=torch.int32, device=dev),
                     torch.empty(T * k, dtype=torch.int32, device=dev))
    need = moe_layout_workspace_bytes(T, k, E)
    if workspace is None:
        workspace = new_workspace(need, dev)
    _check(_lib.moe_layout(T, k, E, R, _ptr(topk_idx), _ptr(out.expert_counts),
                           _ptr(out.expert_offsets), _ptr(out.rank_offsets), _ptr(out.slot_of),
                           _ptr(out.src_of), _ptr(workspace), workspace.numel() *
                           workspace.element_size(), _ptr(err_word), _stream(stream)),
           "moe_layout")
    return out


def moe_layout_noalloc(topk_idx: torch.Tensor, E: int, R: int, *, out: Layout,
                       err_word: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None) -> Layout:
    """moe_layout for callers that cannot allocate: the outputs are passed in
    (`out`) and the library's fixed device scratch array replaces the
    workspace, so the call allocates nothing."""
    T, k = topk_idx.shape
    _want(topk_idx, "topk_idx", torch.int32)
    _check(_lib.moe_layout_noalloc(T, k, E, R, _ptr(topk_idx), _ptr(out.expert_counts),
                                   _ptr(out.expert_offsets), _ptr(out.rank_offsets),
                                   _ptr(out.slot_of), _ptr(out.src_of), _ptr(err_word),
                                   _stream(stream)), "moe_layout_noalloc")
    return out


class CoalescedLayout(NamedTuple):
    rank_counts_c: torch.Tensor   # int32 [R]
    rank_offsets_c: torch.Tensor  # int32 [R+1]; [R] = Nc
    crow: torch.Tensor            # int32 [T, k]
    src_pair_c: torch.Tensor      # int32 [T*k]; first Nc entries written
    expand: torch.Tensor          # int32 [T*k]


def moe_layout_coalesced(topk_idx: torch.Tensor, slot_of: torch.Tensor, E: int, R: int, *,
                         workspace: Optional[torch.Tensor] = None,
                         err_word: Optional[torch.Tensor] = None,
                         out: Optional[CoalescedLayout] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> CoalescedLayout:
    """One row per (token, distinct destination rank); expand maps plain slots
    to those rows (see moe_ep.h)."""
    if topk_idx.dim() != 2:
        raise ValueError("topk_idx must be [T, k]")
    T, k = topk_idx.shape
    _want(topk_idx, "topk_idx", torch.int32)
    _want(slot_of, "slot_of", torch.int32, (T, k))
    dev = topk_idx.device
    if out is None:
        out = CoalescedLayout(torch.empty(R, dtype=torch.int32, device=dev),
                              torch.empty(R + 1, dtype=torch.int32, device=dev),
                              torch.empty((T, k), dtype=torch.int32, device=dev),
                              torch.empty(T * k, dtype=torch.int32, device=dev),
                              torch.empty(T * k, dtype=torch.int32, device=dev))
    need = moe_layout_workspace_bytes(T, k, R)
    if workspace is None:
        workspace = new_workspace(need, dev)
    _check(_lib.moe_layout_coalesced(T, k, E, R, _ptr(topk_idx), _ptr(slot_of),
                                     _ptr(out.rank_counts_c), _ptr(out.rank_offsets_c),
                                     _ptr(out.crow), _ptr(out.src_pair_c), _ptr(out.expand),
                                     _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _ptr(err_word), _stream(stream)), "moe_layout_coalesced")
    return out


def moe_dispatch_coalesced(x: torch.Tensor, crow: torch.Tensor, rows: int, *,
                           recv_c: Optional[torch.Tensor] = None,
                           err_word: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """recv_c[crow[t, j]] = x[t], each coalesced row written once; `rows` is
    recv_c's capacity (at least Nc; T * min(k, R) always suffices)."""
    T, H = x.shape
    k = crow.shape[1]
    _want(x, "x", torch.bfloat16)
    _want(crow, "crow", torch.int32, (T, k))
    if recv_c is None:
        recv_c = torch.empty((rows, H), dtype=torch.bfloat16, device=x.device)
    elif recv_c.shape[0] < rows:
        raise ValueError("recv_c has fewer than `rows` rows")
    _check(_lib.moe_dispatch_coalesced(T, H, k, _ptr(x), _ptr(crow), rows, _ptr(recv_c),
                                       _ptr(err_word), _stream(stream)), "moe_dispatch_coalesced")
    return recv_c


def moe_dispatch_quant_coalesced(x: torch.Tensor, crow: torch.Tensor, rows: int, *,
                                 recv_q: Optional[torch.Tensor] = None,
                                 recv_scales: Optional[torch.Tensor] = None,
                                 err_word: Optional[torch.Tensor] = None,
                                 stream: Optional[torch.cuda.Stream] = None):
    """E4M3 codes and fp32 scales of each token, written once per coalesced
    row.  Returns (recv_q uint8 [rows, H], recv_scales fp32 [rows, H/128])."""
    T, H = x.shape
    k = crow.shape[1]
    _want(x, "x", torch.bfloat16)
    _want(crow, "crow", torch.int32, (T, k))
    if recv_q is None:
        recv_q = torch.empty((rows, H), dtype=torch.uint8, device=x.device)
    if recv_scales is None:
        recv_scales = torch.empty((rows, H // 128), dtype=torch.float32, device=x.device)
    if recv_q.shape[0] < rows or recv_scales.shape[0] < rows:
        raise ValueError("recv_q / recv_scales have fewer than `rows` rows")
    _check(_lib.moe_dispatch_quant_coalesced(T, H, k, _ptr(x), _ptr(crow), rows, _ptr(recv_q),
                                             _ptr(recv_scales), _ptr(err_word), _stream(stream)),
           "moe_dispatch_quant_coalesced")
    return recv_q, recv_scales


def moe_combine_coalesced(y: torch.Tensor, slot_of: torch.Tensor, topk_w: torch.Tensor,
                          co: CoalescedLayout, rows: int, *,
                          partial: Optional[torch.Tensor] = None,
                          out: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                          err_word: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None):
    """Per-rank pre-reduction into `partial` (bf16 [rows, H]), then the sum of
    each token's distinct coalesced rows.  Returns (out, partial)."""
    T, k = slot_of.shape
    H = y.shape[1]
    _want(y, "y", torch.bfloat16)
    _want(slot_of, "slot_of", torch.int32, (T, k))
    _want(topk_w, "topk_w", torch.float32, (T, k))
    if partial is None:
        partial = torch.empty((rows, H), dtype=torch.bfloat16, device=y.device)
    elif partial.shape[0] < rows:
        raise ValueError("partial has fewer than `rows` rows")
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=y.device)
    code = MOE_OUT_F32 if out.dtype == torch.float32 else MOE_OUT_BF16
    _check(_lib.moe_combine_coalesced(T, H, k, _ptr(y), _ptr(slot_of), _ptr(topk_w),
                                      _ptr(co.crow), rows, _ptr(partial), _ptr(out), code,
                                      _ptr(err_word), _stream(stream)), "moe_combine_coalesced")
    return out, partial


def moe_layout_dispatch(x: torch.Tensor, topk_idx: torch.Tensor, E: int, R: int, *,
                        workspace: Optional[torch.Tensor] = None,
                        out: Optional[Layout] = None, recv: Optional[torch.Tensor] = None,
                        err_word: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None):
    """moe_layout then moe_dispatch (bf16), the dispatch's first loads of x
    overlapping the layout.  Returns (Layout, recv)."""
    if topk_idx.dim() != 2:
        raise ValueError("topk_idx must be [T, k]")
    T, k = topk_idx.shape
    H = x.shape[1]
    _want(topk_idx, "topk_idx", torch.int32)
    _want(x, "x", torch.bfloat16, (T, H))
    dev = topk_idx.device
    if out is None:
        out = Layout(torch.empty(E, dtype=torch.int32, device=dev),
                     torch.empty(E + 1, dtype=torch.int32, device=dev),
                     torch.empty(R + 1, dtype=torch.int32, device=dev),
                     torch.empty((T, k), dtype=torch.int32, device=dev),
                     torch.empty(T * k, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = new_workspace(moe_layout_workspace_bytes(T, k, E), dev)
    if recv is None:
        recv = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
    _check(_lib.moe_layout_dispatch(T, H, k, E, R, _ptr(topk_idx), _ptr(x),
                                    _ptr(out.expert_counts), _ptr(out.expert_offsets),
                                    _ptr(out.rank_offsets), _ptr(out.slot_of), _ptr(out.src_of),
                                    _ptr(recv), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _ptr(err_word), _stream(stream)), "moe_layout_dispatch")
    return out, recv


def moe_layout_dispatch_quant(x: torch.Tensor, topk_idx: torch.Tensor, E: int, R: int, *,
                              workspace: Optional[torch.Tensor] = None,
                              out: Optional[Layout] = None,
                              recv_q: Optional[torch.Tensor] = None,
                              recv_scales: Optional[torch.Tensor] = None,
                              err_word: Optional[torch.Tensor] = None,
                              stream: Optional[torch.cuda.Stream] = None):
    """moe_layout then moe_dispatch_quant, the FP8 dispatch's first loads and
    quantisation of x overlapping the layout.  Returns (Layout, recv_q uint8
    [T*k, H], recv_scales fp32 [T*k, H/128])."""
    if topk_idx.dim() != 2:
        raise ValueError("topk_idx must be [T, k]")
    T, k = topk_idx.shape
    H = x.shape[1]
    _want(topk_idx, "topk_idx", torch.int32)
    _want(x, "x", torch.bfloat16, (T, H))
    dev = topk_idx.device
    if out is None:
        out = Layout(torch.empty(E, dtype=torch.int32, device=dev),
                     torch.empty(E + 1, dtype=torch.int32, device=dev),
                     torch.empty(R + 1, dtype=torch.int32, device=dev),
                     torch.empty((T, k), dtype=torch.int32, device=dev),
                     torch.empty(T * k, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = new_workspace(moe_layout_workspace_bytes(T, k, E), dev)
    if recv_q is None:
        recv_q = torch.empty((T * k, H), dtype=torch.uint8, device=dev)
    if recv_scales is None:
        recv_scales = torch.empty((T * k, H // 128), dtype=torch.float32, device=dev)
    _check(_lib.moe_layout_dispatch_quant(T, H, k, E, R, _ptr(topk_idx), _ptr(x),
                                          _ptr(out.expert_counts), _ptr(out.expert_offsets),
                                          _ptr(out.rank_offsets), _ptr(out.slot_of),
                                          _ptr(out.src_of), _ptr(recv_q), _ptr(recv_scales),
                                          _ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          _ptr(err_word), _stream(stream)),
           "moe_layout_dispatch_quant")
    return out, recv_q, recv_scales


def moe_dispatch(x: torch.Tensor, slot_of: torch.Tensor, *, recv: Optional[torch.Tensor] = None,
                 err_word: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """recv[slot_of[t, j]] = x[t] (bf16 rows)."""
    T, H = x.shape
    k = slot_of.shape[1]
    _want(x, "x", torch.bfloat16)
    _want(slot_of, "slot_of", torch.int32, (T, k))
    if recv is None:
        recv = torch.empty((T * k, H), dtype=torch.bfloat16, device=x.device)
    _want(recv, "recv", torch.bfloat16, (T * k, H))
    _check(_lib.moe_dispatch(T, H, k, _ptr(x), _ptr(slot_of), _ptr(recv), _ptr(err_word),
                             _stream(stream)), "moe_dispatch")
    return recv


def moe_dispatch_quant(x: torch.Tensor, slot_of: torch.Tensor, *,
                       recv_q: Optional[torch.Tensor] = None,
                       recv_scales: Optional[torch.Tensor] = None,
                       err_word: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None):
    """Dispatch with fused FP8-E4M3 1x128 block quantisation.
    Returns (recv_q uint8 [T*k, H], recv_scales float32 [T*k, H/128])."""
    T, H = x.shape
    k = slot_of.shape[1]
    _want(x, "x", torch.bfloat16)
    _want(slot_of, "slot_of", torch.int32, (T, k))
    if recv_q is None:
        recv_q = torch.empty((T * k, H), dtype=torch.uint8, device=x.device)
    if recv_scales is None:
        recv_scales = torch.empty((T * k, H // 128), dtype=torch.float32, device=x.device)
    _want(recv_q, "recv_q", torch.uint8, (T * k, H))
    _want(recv_scales, "recv_scales", torch.float32, (T * k, H // 128))
    _check(_lib.moe_dispatch_quant(T, H, k, _ptr(x), _ptr(slot_of), _ptr(recv_q),
                                   _ptr(recv_scales), _ptr(err_word), _stream(stream)),
           "moe_dispatch_quant")
    return recv_q, recv_scales


def moe_combine(y: torch.Tensor, slot_of: torch.Tensor, topk_w: torch.Tensor, *,
                out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
                err_word: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """out[t] = sum_j topk_w[t, j] * y[slot_of[t, j]] with fp32 accumulation."""
    T, k = slot_of.shape
    H = y.shape[1]
    _want(y, "y", torch.bfloat16, (T * k, H))
    _want(slot_of, "slot_of", torch.int32)
    _want(topk_w, "topk_w", torch.float32, (T, k))
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out_dtype must be bfloat16 or float32")
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=y.device)
    _want(out, "out", out_dtype, (T, H))
    code = MOE_OUT_BF16 if out_dtype == torch.bfloat16 else MOE_OUT_F32
    _check(_lib.moe_combine(T, H, k, _ptr(y), _ptr(slot_of), _ptr(topk_w), _ptr(out), code,
                            _ptr(err_word), _stream(stream)), "moe_combine")
    return out


def moe_combine_backward(dout: torch.Tensor, y: Optional[torch.Tensor], slot_of: torch.Tensor,
                         topk_w: torch.Tensor, *, dy: Optional[torch.Tensor] = None,
                         dw: Optional[torch.Tensor] = None, want_dw: bool = True,
                         err_word: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None):
    """Gradient of moe_combine.  Returns (dy bf16 [T*k, H], dw fp32 [T, k] or None)."""
    T, H = dout.shape
    k = slot_of.shape[1]
    _want(dout, "dout", torch.bfloat16)
    _want(slot_of, "slot_of", torch.int32, (T, k))
    _want(topk_w, "topk_w", torch.float32, (T, k))
    if y is not None:
        _want(y, "y", torch.bfloat16, (T * k, H))
    if dy is None:
        dy = torch.empty((T * k, H), dtype=torch.bfloat16, device=dout.device)
    _want(dy, "dy", torch.bfloat16, (T * k, H))
    if want_dw and y is not None and dw is None:
        dw = torch.empty((T, k), dtype=torch.float32, device=dout.device)
    if not want_dw or y is None:
        dw = None
    _check(_lib.moe_combine_backward(T, H, k, _ptr(dout), _ptr(y), _ptr(slot_of), _ptr(topk_w),
                                     _ptr(dy), _ptr(dw), _ptr(err_word), _stream(stream)),
           "moe_combine_backward")
    return dy, dw


def moe_dispatch_backward(drecv: torch.Tensor, slot_of: torch.Tensor, *,
                          out_dtype: torch.dtype = torch.bfloat16,
                          dx: Optional[torch.Tensor] = None,
                          err_word: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Gradient of moe_dispatch: dx[t] = sum_j drecv[slot_of[t, j]]."""
    T, k = slot_of.shape
    H = drecv.shape[1]
    _want(drecv, "drecv", torch.bfloat16, (T * k, H))
    _want(slot_of, "slot_of", torch.int32)
    if dx is None:
        dx = torch.empty((T, H), dtype=out_dtype, device=drecv.device)
    _want(dx, "dx", out_dtype, (T, H))
    code = MOE_OUT_BF16 if out_dtype == torch.bfloat16 else MOE_OUT_F32
    _check(_lib.moe_dispatch_backward(T, H, k, _ptr(drecv), _ptr(slot_of), _ptr(dx), code,
                                      _ptr(err_word), _stream(stream)), "moe_dispatch_backward")
    return dx


def moe_sync_words(T: int, H: int, k: int, mode: int, block_bytes: int) -> int:
    return int(_lib.moe_sync_words(T, H, k, mode, block_bytes))


SENTINEL_WORD = -1  # every 32-bit word 0xFFFFFFFF (two bf16 0xFFFF NaNs)


class SyncState:
    """What moe_dispatch_combine_flagged keeps between calls for one shape:
    the readiness words (zero-filled once) with a fresh epoch per call and, for
    MOE_SYNC_SENTINEL, recv and y filled with the sentinel."""

    def __init__(self, T: int, H: int, k: int, mode: int = MOE_SYNC_WORD,
                 block_bytes: int = 2048, device=None):
        dev = device or "cuda"
        n = moe_sync_words(T, H, k, mode, block_bytes)
        if n == 0 and mode != MOE_SYNC_SENTINEL:
            raise ValueError(f"invalid granularity {block_bytes} for mode {mode}")
        self.mode, self.block_bytes = mode, block_bytes
        self.words = torch.zeros(max(n, 2), dtype=torch.int32, device=dev)
        self.epoch = 0
        self.recv = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
        self.y = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
        if mode == MOE_SYNC_SENTINEL:
            self.refill()

    def refill(self) -> None:
        """Sentinel-fill recv and y (needed again after a call that failed)."""
        self.recv.view(torch.int16).fill_(SENTINEL_WORD)
        self.y.view(torch.int16).fill_(SENTINEL_WORD)

    def next_epoch(self) -> int:
        self.epoch = (self.epoch % 0xFFFFFFFF) + 1
        return self.epoch


def moe_dispatch_combine_flagged(x: torch.Tensor, slot_of: torch.Tensor, topk_w: torch.Tensor,
                                 state: SyncState, *, out_dtype: torch.dtype = torch.bfloat16,
                                 out: Optional[torch.Tensor] = None,
                                 spin_limit_ns: int = 1_000_000_000, fault_skip_pair: int = -1,
                                 err_word: Optional[torch.Tensor] = None,
                                 stream: Optional[torch.cuda.Stream] = None):
    """Dispatch, identity expert and combine in one persistent kernel; the
    expert and combine phases learn that rows have arrived through
    `state.mode`.  Returns (recv, y, out)."""
    T, H = x.shape
    k = slot_of.shape[1]
    _want(x, "x", torch.bfloat16)
    _want(slot_of, "slot_of", torch.int32, (T, k))
    _want(topk_w, "topk_w", torch.float32, (T, k))
    _want(state.recv, "recv", torch.bfloat16, (T * k, H))
    _want(state.y, "y", torch.bfloat16, (T * k, H))
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=x.device)
    _want(out, "out", out_dtype, (T, H))
    code = MOE_OUT_BF16 if out_dtype == torch.bfloat16 else MOE_OUT_F32
    _check(_lib.moe_dispatch_combine_flagged(T, H, k, _ptr(x), _ptr(slot_of), _ptr(topk_w),
                                             _ptr(state.recv), _ptr(state.y), _ptr(out), code,
                                             state.mode, state.block_bytes, _ptr(state.words),
                                             state.next_epoch(), int(spin_limit_ns),
                                             int(fault_skip_pair), _ptr(err_word),
                                             _stream(stream)), "moe_dispatch_combine_flagged")
    return state.recv, state.y, out


def moe_read_error(err_word: torch.Tensor, clear: bool = True,
                   stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise, read (and clear) the error word; returns the error bits."""
    bits = ctypes.c_uint32(0)
    st = _lib.moe_read_error(_ptr(err_word), 1 if clear else 0, _stream(stream),
                             ctypes.byref(bits))
    if st == MOE_ERR_CUDA or st == MOE_ERR_INVALID_ARG:
        _check(st, "moe_read_error")
    return int(bits.value)


__all__ = [
    "Layout", "MoeError", "moe_abi_version", "moe_status_string", "new_error_word", "new_workspace",
    "moe_layout_workspace_bytes", "moe_layout", "moe_layout_noalloc", "moe_dispatch", "moe_dispatch_quant",
    "moe_layout_dispatch", "moe_layout_dispatch_quant",
    "moe_combine", "moe_read_error", "moe_sync_words", "SyncState",
    "moe_combine_backward", "moe_dispatch_backward",
    "CoalescedLayout", "moe_layout_coalesced", "moe_dispatch_coalesced", "moe_dispatch_quant_coalesced",
    "moe_combine_coalesced",
    "moe_dispatch_combine_flagged", "moe_ep_reorder", "moe_layout_last_form",
    "moe_e4m3_encode_bits", "moe_ep_reorder_rows", "LIB_PATH",
    "SIGNATURES",
]


def moe_ep_reorder(src: torch.Tensor, recv_counts: torch.Tensor, *, to_source: bool = False,
                   out: Optional[torch.Tensor] = None,
                   local_expert_offsets: Optional[torch.Tensor] = None,
                   err_word: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Source-major received rows -> expert-major (to_source False), or back
    (True); recv_counts is the [W, El] int32 device matrix of rows each source
    sent for each local expert (see moe_ep.h)."""
    if recv_counts.dim() != 2:
        raise ValueError("recv_counts must be [W, El]")
    W, El = recv_counts.shape
    rows, H = src.shape
    _want(src, "src", torch.bfloat16)
    _want(recv_counts, "recv_counts", torch.int32)
    if out is None:
        out = torch.empty_like(src)
    _want(out, "out", torch.bfloat16, (rows, H))
    if local_expert_offsets is not None:
        _want(local_expert_offsets, "local_expert_offsets", torch.int32, (El + 1,))
    _check(_lib.moe_ep_reorder(W, El, H, _ptr(recv_counts), rows, _ptr(src), _ptr(out),
                               MOE_EP_TO_SOURCE if to_source else MOE_EP_TO_EXPERT,
                               _ptr(local_expert_offsets), _ptr(err_word), _stream(stream)),
           "moe_ep_reorder")
    return out


def moe_ep_reorder_rows(src: torch.Tensor, recv_counts: torch.Tensor, *, to_source: bool = False,
                        out: Optional[torch.Tensor] = None,
                        local_expert_offsets: Optional[torch.Tensor] = None,
                        err_word: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """moe_ep_reorder for rows of any contiguous payload (the first dimension
    indexes rows; a row's size must be a multiple of 4 bytes)."""
    if recv_counts.dim() != 2:
        raise ValueError("recv_counts must be [W, El]")
    W, El = recv_counts.shape
    _want(recv_counts, "recv_counts", torch.int32)
    if not src.is_cuda or not src.is_contiguous() or src.dim() < 1:
        raise ValueError("src must be a contiguous CUDA tensor of rows")
    rows = src.shape[0]
    row_bytes = (src.numel() // rows if rows else int(torch.tensor(src.shape[1:]).prod())) * \
        src.element_size()
    if out is None:
        out = torch.empty_like(src)
    if out.shape != src.shape or out.dtype != src.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like src")
    if local_expert_offsets is not None:
        _want(local_expert_offsets, "local_expert_offsets", torch.int32, (El + 1,))
    _check(_lib.moe_ep_reorder_rows(W, El, row_bytes, _ptr(recv_counts), rows, _ptr(src),
                                    _ptr(out), MOE_EP_TO_SOURCE if to_source else
                                    MOE_EP_TO_EXPERT, _ptr(local_expert_offsets),
                                    _ptr(err_word), _stream(stream)), "moe_ep_reorder_rows")
    return out
