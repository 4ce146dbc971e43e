"""Seeded synthetic workloads shaped like the pages' MoE expert-parallel cases.

Five named shapes, each standing in for a workload the pages measure on real
models and clusters (their routing traces and weights are not available):

  tiny          T=128,   H=256,  top-2, E=8,   R=2   (parity-only case)
  dsv3_decode   T=1024,  H=7168, top-8, E=256, R=32  (DeepSeek-V3-style decode batch,
                near-uniform routing; StrataCL section 8 uses 4096 tokens, H=7168, top-8)
  dsv3_prefill  T=8192,  H=7168, top-8, E=256, R=32  (HyperParallel-MoE section 6 setup:
                8192 tokens per rank, H=7168, top-8; Zipf(1.1) expert popularity; FP8 payload)
  glm45_air     T=16384, H=4096, top-8, E=128, R=16  (RailWave's GLM-4.5-Air replay stand-in:
                8 groups of 16 experts, node-limited to 4 groups, Zipf(1.2) skew)
  mixtral       T=65536, H=4096, top-2, E=8,   R=8   (one hot expert, logit bias +2.0)

Recipe (all streams derive from one integer seed through numpy's SeedSequence):
  x       = bf16_rne(N(0,1) float32)                      stream 0, row-major [T, H]
  logits  = N(0,1) float32 [T, E]                         stream 1
  bias    = -s * ln(1 + pi(e)), pi a permutation of E     stream 2 (Zipf cases)
            +2.0 on expert 0                              (hot-expert case)
  groups  : score(g) = sum of the two largest biased logits in g; keep the best
            `topk_groups`, mask the rest to -inf          (group-limited case)
  topk    = stable descending sort of biased logits, first k (ties -> lower id)
  weights = softmax over the k chosen biased logits, in float64, stored float32
  y       = expert outputs in receive order: bf16 with random sign and mantissa and
            exponent in [2^-7, 2^2]                       stream 3

Nothing here implements layout, dispatch or combine: these are inputs only.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# name -> shape and routing recipe
CONFIGS = {
    "tiny": dict(T=128, H=256, k=2, E=8, R=2, routing="uniform", payload="bf16"),
    "dsv3_decode": dict(T=1024, H=7168, k=8, E=256, R=32, routing="uniform", payload="bf16"),
    "dsv3_prefill": dict(T=8192, H=7168, k=8, E=256, R=32, routing="zipf", zipf_s=1.1,
                         payload="fp8"),
    "glm45_air": dict(T=16384, H=4096, k=8, E=128, R=16, routing="group", zipf_s=1.2,
                      groups=8, topk_groups=4, payload="bf16"),
    "mixtral": dict(T=65536, H=4096, k=2, E=8, R=8, routing="hot", hot_bias=2.0,
                    payload="bf16"),
}
CONFIG_ORDER = ["tiny", "dsv3_decode", "dsv3_prefill", "glm45_air", "mixtral"]

_CHUNK = 1 << 22  # elements per generation chunk (keeps temporaries small)


def _streams(seed: int, n: int = 4):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def _f32_to_bf16_bits_inplace(f: np.ndarray, out: np.ndarray) -> None:
    """Round float32 to bf16 bit patterns (nearest, ties to even) for input data."""
    u = f.view(np.uint32)
    lsb = (u >> 16) & np.uint32(1)
    u += np.uint32(0x7FFF)
    u += lsb
    u >>= 16
    out[...] = u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 values (exact)."""
    return (b.astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """bf16 bit patterns of N(0,1) float32 draws, generated in chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        f = rng.standard_normal(e - s, dtype=np.float32)
        _f32_to_bf16_bits_inplace(f, out[s:e])
    return out.reshape(shape)


def expert_output(N: int, H: int, seed: int = 0) -> np.ndarray:
    """Synthetic expert outputs y[N, H] (bf16 bits) in receive order.

    Random sign and 7-bit mantissa, exponent uniform over 2^-7 .. 2^2, so rows of
    different slots differ everywhere (a wrong slot is always visible).
    """
    rng = _streams(seed)[3]
    n = N * H
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        r = rng.integers(0, 1 << 32, size=e - s, dtype=np.uint32)
        sign = (r >> 31) << 15
        mant = r & np.uint32(0x7F)
        expo = (np.uint32(120) + ((r >> 8) % np.uint32(10))) << 7
        out[s:e] = (sign | expo | mant).astype(np.uint16)
    return out.reshape(N, H)


def _route(cfg: dict, T: int, rng_logits, rng_perm):
    E, k = cfg["E"], cfg["k"]
    logits = rng_logits.standard_normal((T, E), dtype=np.float32)
    bias = np.zeros(E, dtype=np.float64)
    if cfg["routing"] in ("zipf", "group"):
        perm = rng_perm.permutation(E)
        bias = -cfg["zipf_s"] * np.log1p(perm.astype(np.float64))
    elif cfg["routing"] == "hot":
        bias[0] = cfg["hot_bias"]
    biased = logits + bias.astype(np.float32)
    select = biased
    if cfg["routing"] == "group":
        G, keep = cfg["groups"], cfg["topk_groups"]
        per = biased.reshape(T, G, E // G)
        srt = np.sort(per, axis=2)
        score = srt[:, :, -1] + srt[:, :, -2]
        best = np.argsort(-score, axis=1, kind="stable")[:, :keep]
        allowed = np.zeros((T, G), dtype=bool)
        np.put_along_axis(allowed, best, True, axis=1)
        select = np.where(np.repeat(allowed, E // G, axis=1), biased, np.float32(-np.inf))
    order = np.argsort(-select, axis=1, kind="stable")[:, :k].astype(np.int32)
    chosen = np.take_along_axis(biased, order, axis=1).astype(np.float64)
    ex = np.exp(chosen - chosen.max(axis=1, keepdims=True))
    w = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    return np.ascontiguousarray(order), np.ascontiguousarray(w)


@dataclass
class Workload:
    name: str
    T: int
    H: int
    k: int
    E: int
    R: int
    payload: str
    topk_idx: np.ndarray          # int32 [T, k]
    topk_w: np.ndarray            # float32 [T, k]
    seed: int = 0
    _x: Optional[np.ndarray] = field(default=None, repr=False)

    @property
    def N(self) -> int:
        return self.T * self.k

    @property
    def x(self) -> np.ndarray:
        """Hidden states, bf16 bit patterns uint16 [T, H] (drawn on first use)."""
        if self._x is None:
            self._x = normal_bf16(_streams(self.seed)[0], (self.T, self.H))
        return self._x

    def y(self) -> np.ndarray:
        """Expert outputs in receive order, bf16 bits uint16 [T*k, H]."""
        return expert_output(self.N, self.H, self.seed)


def make_workload(name: str, seed: int = 0, T: Optional[int] = None) -> Workload:
    """Build a named workload; `T` overrides the token count (same recipe)."""
    cfg = CONFIGS[name]
    T = cfg["T"] if T is None else int(T)
    _, rl, rp, _ = _streams(seed)
    idx, w = _route(cfg, T, rl, rp)
    return Workload(name=name, T=T, H=cfg["H"], k=cfg["k"], E=cfg["E"], R=cfg["R"],
                    payload=cfg["payload"], topk_idx=idx, topk_w=w, seed=seed)


def random_case(seed: int, T: int, H: int, k: int, E: int, R: int,
                payload: str = "bf16") -> Workload:
    """Fuzz case: experts drawn uniformly with replacement (a token may pick the
    same expert in several of its k slots), weights uniform in [0, 1)."""
    rx, rl, _, _ = _streams(seed)
    idx = rl.integers(0, E, size=(T, k), dtype=np.int32)
    w = rl.random((T, k), dtype=np.float32)
    wl = Workload(name=f"fuzz{seed}", T=T, H=H, k=k, E=E, R=R, payload=payload,
                  topk_idx=np.ascontiguousarray(idx), topk_w=np.ascontiguousarray(w),
                  seed=seed)
    return wl


def device_inputs(w: Workload, device, seed: Optional[int] = None):
    """x [T, H] and expert outputs y [T*k, H], bf16 tensors drawn on `device`
    with torch's seeded generator, for benchmarks whose inputs are too large
    to draw quickly on the host.  Same distributions as `Workload.x` (N(0,1)
    rounded to bf16, nearest-even) and `expert_output` (random sign, 7-bit
    mantissa, exponent uniform over 2^-7 .. 2^2), not the same values."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(w.seed if seed is None else seed) * 7919 + 17)
    x = torch.randn((w.T, w.H), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    r = torch.randint(0, 1 << 31, (w.N, w.H), generator=g, device=device, dtype=torch.int32)
    sign = (r & 1) << 15
    mant = (r >> 1) & 0x7F
    expo = (120 + (r >> 8) % 10) << 7
    y = (sign | expo | mant).to(torch.int16).view(torch.bfloat16)
    return x, y
