"""CPU oracle for MoE expert-parallel layout, dispatch and combine.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, the smoke check in
__graft_entry__ and bench.py's CPU-baseline / reference leg may import this.
The CUDA library (combine_layout_moe_gb300) never imports it, and the two share
no code.  The arithmetic lives in moe_oracle.c (plain C, -ffp-contract=off);
this module compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, ERR_INVALID_ARG, ERR_BAD_INDEX = 0, 1, 2
E4M3_MAX = 448.0


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/liboracle.so (single-threaded, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        compile_to(_SRC, tmp)
        os.replace(tmp, _LIB)
    return _LIB


_lib: Optional[ctypes.CDLL] = None


def _bind(path: str) -> ctypes.CDLL:
    """Load a compiled oracle library and declare its C signatures."""
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    L.oracle_layout.argtypes = [I, I, I, I, P, P, P, P, P, P]
    L.oracle_dispatch.argtypes = [I, I, I, P, P, P]
    L.oracle_dispatch_quant.argtypes = [I, I, I, P, P, P, P]
    L.oracle_combine.argtypes = [I, I, I, P, P, P, P, I]
    L.oracle_combine_f64.argtypes = [I, I, I, P, P, P, P, P]
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    L.oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.oracle_e4m3_encode_array.argtypes = [P, P, ctypes.c_int64]
    L.oracle_e4m3_encode_array.restype = None
    L.oracle_f32_to_bf16_array.argtypes = [P, P, ctypes.c_int64]
    L.oracle_f32_to_bf16_array.restype = None
    L.oracle_combine_backward.argtypes = [I, I, I, P, P, P, P, P, P, P]
    L.oracle_dispatch_backward.argtypes = [I, I, I, P, P, P, I]
    L.oracle_layout_coalesced.argtypes = [I, I, I, I, P, P, P, P, P, P, P]
    L.oracle_dispatch_coalesced.argtypes = [I, I, I, P, P, P]
    L.oracle_combine_coalesced_pre.argtypes = [I, I, I, P, P, P, P, I, P]
    L.oracle_combine_coalesced_post.argtypes = [I, I, I, P, P, I, P, I]
    L.oracle_ep_dispatch.argtypes = [I, P, I, I, I, P, P, P, P, P, P]
    L.oracle_ep_combine.argtypes = [I, P, I, I, I, P, P, P, P, I]
    for f in ("oracle_layout", "oracle_dispatch", "oracle_dispatch_quant",
              "oracle_combine", "oracle_combine_f64", "oracle_abi_version",
              "oracle_combine_backward", "oracle_dispatch_backward",
              "oracle_layout_coalesced", "oracle_dispatch_coalesced",
              "oracle_combine_coalesced_pre", "oracle_combine_coalesced_post",
              "oracle_ep_dispatch", "oracle_ep_combine"):
        getattr(L, f).restype = ctypes.c_int
    return L


def compile_to(src: str, out: str) -> None:
    """Compile an oracle source file with the oracle's flags."""
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
                    "-fPIC", "-shared", "-Wall", "-Wextra", "-o", out, src, "-lm"],
                   check=True)


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        _lib = _bind(_LIB)
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__({1: "invalid argument", 2: "expert or slot index out of range"}.get(
            status, f"status {status}"))
        self.status = status


def _check(st: int):
    if st != OK:
        raise OracleError(st)


def layout(topk_idx: np.ndarray, E: int, R: int):
    """Returns (expert_counts[E], expert_offsets[E+1], rank_offsets[R+1],
    slot_of[T,k], src_of[T*k]) as int32 arrays."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offs = np.empty(E + 1, np.int32)
    roffs = np.empty(R + 1, np.int32)
    slot_of = np.empty((T, k), np.int32)
    src_of = np.empty(T * k, np.int32)
    _check(lib().oracle_layout(T, k, E, R, _p(idx), _p(counts), _p(offs), _p(roffs),
                               _p(slot_of), _p(src_of)))
    return counts, offs, roffs, slot_of, src_of


def dispatch(x_bf16: np.ndarray, slot_of: np.ndarray) -> np.ndarray:
    """x: uint16 bf16 bits [T,H]; returns recv uint16 [T*k, H]."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    T, H = x.shape
    k = so.shape[1]
    recv = np.empty((T * k, H), np.uint16)
    _check(lib().oracle_dispatch(T, H, k, _p(x), _p(so), _p(recv)))
    return recv


def dispatch_quant(x_bf16: np.ndarray, slot_of: np.ndarray):
    """Returns (recv_q uint8 [T*k, H], recv_scales float32 [T*k, H/128])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    T, H = x.shape
    k = so.shape[1]
    q = np.empty((T * k, H), np.uint8)
    sc = np.empty((T * k, max(H // 128, 1)), np.float32)
    _check(lib().oracle_dispatch_quant(T, H, k, _p(x), _p(so), _p(q), _p(sc)))
    return q, sc


def combine(y_bf16: np.ndarray, slot_of: np.ndarray, topk_w: np.ndarray,
            out_dtype: str = "bf16") -> np.ndarray:
    """y: uint16 bf16 bits [T*k, H] in receive order.  Returns uint16 bf16 bits
    [T,H] (out_dtype 'bf16') or float32 [T,H] ('f32')."""
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    T, k = so.shape
    H = y.shape[1]
    if out_dtype == "bf16":
        out = np.empty((T, H), np.uint16)
        code = 0
    elif out_dtype == "f32":
        out = np.empty((T, H), np.float32)
        code = 1
    else:
        raise ValueError(out_dtype)
    _check(lib().oracle_combine(T, H, k, _p(y), _p(so), _p(w), _p(out), code))
    return out


def combine_f64(y_bf16: np.ndarray, slot_of: np.ndarray, topk_w: np.ndarray):
    """Float64 weighted sum and sum of |terms| (for the fp32 error bound)."""
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    T, k = so.shape
    H = y.shape[1]
    out = np.empty((T, H), np.float64)
    mag = np.empty((T, H), np.float64)
    _check(lib().oracle_combine_f64(T, H, k, _p(y), _p(so), _p(w), _p(out), _p(mag)))
    return out, mag


def combine_backward(dout_bf16: np.ndarray, y_bf16, slot_of: np.ndarray, topk_w: np.ndarray):
    """Returns (dy uint16 bf16 bits [T*k, H], dw float64 [T,k] or None,
    dw_abs_sum float64 [T,k] or None).  y may be None (no dw)."""
    d = np.ascontiguousarray(dout_bf16, dtype=np.uint16)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    T, H = d.shape
    k = so.shape[1]
    dy = np.empty((T * k, H), np.uint16)
    if y_bf16 is None:
        _check(lib().oracle_combine_backward(T, H, k, _p(d), None, _p(so), _p(w), _p(dy), None,
                                             None))
        return dy, None, None
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    dw = np.empty((T, k), np.float64)
    mag = np.empty((T, k), np.float64)
    _check(lib().oracle_combine_backward(T, H, k, _p(d), _p(y), _p(so), _p(w), _p(dy), _p(dw),
                                         _p(mag)))
    return dy, dw, mag


def dispatch_backward(drecv_bf16: np.ndarray, slot_of: np.ndarray, out_dtype: str = "bf16"):
    """dx[t] = sum_j drecv[slot_of[t,j]]; uint16 bf16 bits or float32 [T, H]."""
    dr = np.ascontiguousarray(drecv_bf16, dtype=np.uint16)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    T, k = so.shape
    H = dr.shape[1]
    out = np.empty((T, H), np.uint16 if out_dtype == "bf16" else np.float32)
    _check(lib().oracle_dispatch_backward(T, H, k, _p(dr), _p(so), _p(out),
                                          0 if out_dtype == "bf16" else 1))
    return out


def layout_coalesced(topk_idx: np.ndarray, E: int, R: int, slot_of: np.ndarray):
    """Returns (rank_counts_c[R], rank_offsets_c[R+1], crow[T,k], src_pair_c[Nc],
    expand[T*k])."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(R, np.int32)
    offs = np.empty(R + 1, np.int32)
    crow = np.empty((T, k), np.int32)
    src = np.full(T * k, -1, np.int32)
    expand = np.empty(T * k, np.int32)
    _check(lib().oracle_layout_coalesced(T, k, E, R, _p(idx), _p(so), _p(counts), _p(offs),
                                         _p(crow), _p(src), _p(expand)))
    return counts, offs, crow, src[: offs[-1]].copy(), expand


def dispatch_coalesced(x_bf16: np.ndarray, crow: np.ndarray, n_rows: int) -> np.ndarray:
    """recv_c[crow[t, j]] = x[t]; uint16 [n_rows, H]."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    cr = np.ascontiguousarray(crow, dtype=np.int32)
    T, H = x.shape
    k = cr.shape[1]
    out = np.zeros((max(T * k, 1), H), np.uint16)
    _check(lib().oracle_dispatch_coalesced(T, H, k, _p(x), _p(cr), _p(out)))
    return out[:n_rows]


def combine_coalesced_pre(y_bf16: np.ndarray, slot_of: np.ndarray, topk_w: np.ndarray,
                          crow: np.ndarray, n_rows: int) -> np.ndarray:
    """partial[c] = bf16(sum over the slots of row c of w * y), uint16 [n_rows, H]."""
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    cr = np.ascontiguousarray(crow, dtype=np.int32)
    T, k = so.shape
    H = y.shape[1]
    part = np.zeros((max(n_rows, 1), H), np.uint16)
    _check(lib().oracle_combine_coalesced_pre(T, H, k, _p(y), _p(so), _p(w), _p(cr), n_rows,
                                              _p(part)))
    return part[:n_rows]


def combine_coalesced_post(partial: np.ndarray, crow: np.ndarray, out_dtype: str = "bf16"):
    """out[t] = sum over the token's distinct coalesced rows of partial (fp32)."""
    p = np.ascontiguousarray(partial, dtype=np.uint16)
    cr = np.ascontiguousarray(crow, dtype=np.int32)
    T, k = cr.shape
    H = p.shape[1]
    out = np.empty((T, H), np.uint16 if out_dtype == "bf16" else np.float32)
    _check(lib().oracle_combine_coalesced_post(T, H, k, _p(p), _p(cr), p.shape[0], _p(out),
                                               0 if out_dtype == "bf16" else 1))
    return out


def ep_dispatch(idx_per_rank, x_per_rank, E: int):
    """Expert-parallel dispatch across W = len(idx_per_rank) ranks.  Each
    rank's ids are int32 [T_s, k] and rows uint16 bf16 bits [T_s, H].  Returns
    (recv_counts int32 [W(receiver), W(source), El], recv per receiver: a list
    of uint16 [rows_d, H], src_pair per receiver: a list of int64 global pair
    indices t*k + j, t counted over the ranks' tokens in rank order)."""
    W = len(idx_per_rank)
    k = idx_per_rank[0].shape[1]
    H = x_per_rank[0].shape[1]
    tok_off = np.zeros(W + 1, np.int64)
    tok_off[1:] = np.cumsum([a.shape[0] for a in idx_per_rank])
    idx = np.ascontiguousarray(np.concatenate(idx_per_rank).reshape(-1, k), dtype=np.int32)
    x = np.ascontiguousarray(np.concatenate(x_per_rank).reshape(-1, H), dtype=np.uint16)
    N = idx.size
    counts = np.empty((W, W, max(E // W, 1)), np.int32)
    base = np.empty(W + 1, np.int64)
    src_pair = np.empty(max(N, 1), np.int64)
    recv = np.empty((max(N, 1), H), np.uint16)
    _check(lib().oracle_ep_dispatch(W, _p(tok_off), k, E, H, _p(idx), _p(x), _p(counts),
                                    _p(base), _p(src_pair), _p(recv)))
    return (counts, [recv[base[d]:base[d + 1]] for d in range(W)],
            [src_pair[base[d]:base[d + 1]] for d in range(W)])


def ep_combine(idx_per_rank, w_per_rank, y_per_receiver, E: int, out_dtype: str = "bf16"):
    """The return path: y_per_receiver[d] holds receiver d's expert outputs in
    its receive order (as ep_dispatch lays recv out).  Returns each rank's
    combined rows: a list of uint16 bf16 bits [T_s, H] ('bf16') or float32
    ('f32')."""
    W = len(idx_per_rank)
    k = idx_per_rank[0].shape[1]
    H = y_per_receiver[0].shape[1]
    tok_off = np.zeros(W + 1, np.int64)
    tok_off[1:] = np.cumsum([a.shape[0] for a in idx_per_rank])
    idx = np.ascontiguousarray(np.concatenate(idx_per_rank).reshape(-1, k), dtype=np.int32)
    w = np.ascontiguousarray(np.concatenate(w_per_rank).reshape(-1, k), dtype=np.float32)
    y = np.ascontiguousarray(np.concatenate(y_per_receiver).reshape(-1, H), dtype=np.uint16)
    T = int(tok_off[W])
    out = np.empty((T, H), np.uint16 if out_dtype == "bf16" else np.float32)
    _check(lib().oracle_ep_combine(W, _p(tok_off), k, E, H, _p(idx), _p(w), _p(y), _p(out),
                                   0 if out_dtype == "bf16" else 1))
    return [out[tok_off[s]:tok_off[s + 1]] for s in range(W)]


def e4m3_encode(f: np.ndarray) -> np.ndarray:
    """Elementwise E4M3 (satfinite, nearest-even) codes of float32 values."""
    flat = np.ascontiguousarray(f, dtype=np.float32).ravel()
    q = np.empty(flat.size, np.uint8)
    lib().oracle_e4m3_encode_array(_p(flat), _p(q), flat.size)
    return q.reshape(np.shape(f))


def f32_to_bf16(f: np.ndarray) -> np.ndarray:
    """Elementwise float32 -> bf16 bits (nearest, ties to even)."""
    flat = np.ascontiguousarray(f, dtype=np.float32).ravel()
    b = np.empty(flat.size, np.uint16)
    lib().oracle_f32_to_bf16_array(_p(flat), _p(b), flat.size)
    return b.reshape(np.shape(f))
