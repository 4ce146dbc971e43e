"""Benchmark: MoE expert-parallel dispatch + combine on one GB300 (or N replicas).

One step = the whole hot path over one batch: layout (count, scan, slot map)
-> dispatch (bf16 row scatter, or the fused FP8 variant for FP8 workloads) ->
combine (router-weighted fp32 gather-reduce, bf16 out) of synthetic expert
outputs.  The headline workload is the largest of the target's single-GPU
workloads: Mixtral-style, T=65536, H=4096, top-2 of E=8 experts on R=8
virtual ranks, one hot expert.  The line then carries a `per_config` block:
the DeepSeek-V3-style decode (T=1024, H=7168, top-8 of 256, R=32) and prefill
(T=8192, FP8 dispatch) workloads, the GLM-4.5-Air-style workload (T=16384,
H=4096, top-8 of 128, R=16) and the headline's own figures, each through the
same timed loop, with its dispatch and combine times, algorithmic bytes and
fraction of the measured HBM peak, and the oracle's time per operation on one
host core.

Timing: W untimed warm-up steps, then exactly K timed steps between a barrier
and a device synchronisation.  Every step flushes L2 twice, outside the CUDA
events that bracket each segment on the launching stream: a 2xL2 buffer is
written before layout+dispatch (dispatch then pays for evicting dirty lines,
as its own writes would), and a 4xL2 buffer is read before combine
(combine starts from a cold, clean L2 and is not charged for dispatch's
write-backs).  value = tokens per second over all ranks (weak scaling: each
rank runs its own replica).  SM clocks and clock-event reasons are sampled
through NVML about every millisecond inside each timed region.  `e2e` repeats
the step through the public API with each step's inputs copied from pinned
host memory and its combined output copied back, pipelined over three streams.

--variant coalesced times the rank-coalesced path instead: layout ->
coalesced layout -> coalesced dispatch (one row per token and destination
rank; FP8 codes and scales for FP8 workloads), then the coalesced combine
(per-rank pre-reduction and the per-token sum).  The default line is the plain
path.

--impl reference times the CPU oracle (the plain C statement of the method) on
the same metric: every step is a bounded sample of the same workload recipe.

Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "dispatch+combine tokens/s"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "mixtral"
# the workloads the target names (configs 1-4), measured after the headline
PER_CONFIG = "dsv3_decode,dsv3_prefill,glm45_air,mixtral"
PER_CONFIG_MIN_STEPS = 500


# ------------------------------------------------------------------ bytes

def kernel_bytes(name: str, T: int, H: int, k: int, E: int, R: int = 1) -> int:
    """Algorithmic bytes one launch must move (HBM reads + writes), per kernel.

    layout_count   reads topk_idx once
    layout_assign  reads topk_idx, writes slot_of and src_of, counts and offsets
    layout_dispatch  both of the above
    dispatch_bf16  reads x and slot_of once, writes k copies of every row
    dispatch_fp8   reads x and slot_of, writes k copies of the codes and scales
    combine        reads k rows per token, slot_of and weights, writes one row
    combine_backward  reads dout and the k rows of y, writes the k rows of dy
                   and dw
    dispatch_backward  reads the k rows of drecv per token, writes dx
    The coalesced kernels also depend on Nc, the number of coalesced rows:
    dispatch_coalesced  reads x and crow, writes Nc rows
    dispatch_fp8_coalesced  reads x and crow, writes Nc rows of codes and scales
    combine_coalesced   reads k rows per token, slot_of, weights and crow,
                        writes the Nc pre-reduced rows and one row per token
    """
    N = T * k
    if name == "layout_count":
        return 4 * N
    if name == "layout_assign":
        return 12 * N + 4 * (2 * E + 1 + R + 1)
    if name == "dispatch_bf16":
        return 2 * T * H + 4 * N + 2 * N * H
    if name == "dispatch_fp8":
        return 2 * T * H + 4 * N + N * H + 4 * N * (H // 128)
    if name == "combine":
        return 2 * N * H + 8 * N + 2 * T * H
    if name == "layout_dispatch":
        return 12 * N + 4 * (2 * E + 1 + R + 1) + 2 * T * H + 4 * N + 2 * N * H
    if name == "combine_backward":   # reads dout, k rows of y, slot_of, w; writes dy, dw
        return 2 * T * H + 2 * N * H + 2 * N * H + 12 * N
    if name == "dispatch_backward":  # the unit-weight combine of drecv
        return 2 * N * H + 4 * N + 2 * T * H
    raise KeyError(name)


def coalesced_bytes(name: str, T: int, H: int, k: int, Nc: int) -> int:
    N = T * k
    if name == "dispatch_coalesced":
        return 2 * T * H + 4 * N + 2 * Nc * H
    if name == "dispatch_fp8_coalesced":
        return 2 * T * H + 4 * N + Nc * H + 4 * Nc * (H // 128)
    if name == "combine_coalesced":
        return 2 * N * H + 12 * N + 2 * Nc * H + 2 * T * H
    if name == "layout_coalesced":  # reads ids and slot_of; writes crow, src_pair_c, expand
        return 20 * N
    raise KeyError(name)


def step_bytes(T, H, k, E, R, fp8: bool) -> int:
    d = "dispatch_fp8" if fp8 else "dispatch_bf16"
    return sum(kernel_bytes(n, T, H, k, E, R)
               for n in ("layout_count", "layout_assign", d, "combine"))


# ------------------------------------------------------------------ host helpers

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def allreduce_max(x: float) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi; summary() keeps
    only the samples taken between mark_start() and mark_stop()."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []
        self._t = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            deadline = time.perf_counter() + 5.0
            while not self.lines and time.perf_counter() < deadline and self.proc.poll() is None:
                time.sleep(0.02)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_stop(self):
        self.t1 = time.perf_counter()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        for ts, ln in self.lines:
            if self.t0 is not None and not (self.t0 <= ts <= (self.t1 or ts)):
                continue
            p = [c.strip() for c in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, p[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_smi_id(torch, dev) -> str:
    """nvidia-smi id of a torch device (its UUID when torch exposes it)."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


def measured_peak_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summaries, if that kernel's source is unchanged since the counters were
    taken; else None.  Entries are keyed "kernel@workload" (a capture of a
    smaller case of the same workload states how it was scaled)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(f"{kernel}@{workload}")
        src = os.path.join(ROOT, rec["source"])
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if sha != rec["source_sha256"]:
            return None
        return rec
    except (OSError, KeyError, ValueError, TypeError, AttributeError):
        return None


# ------------------------------------------------------------------ CPU oracle

def oracle_step(w, y_np, fp8: bool, x_np=None):
    import oracle
    x_np = w.x if x_np is None else x_np
    counts, offs, roffs, slot_of, src_of = oracle.layout(w.topk_idx, w.E, w.R)
    if fp8:
        oracle.dispatch_quant(x_np, slot_of)
    else:
        oracle.dispatch(x_np, slot_of)
    oracle.combine(y_np, slot_of, w.topk_w, "bf16")


def host_info():
    """The host's logical CPU count and CPU model (from /proc/cpuinfo)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            fields = {}
            for ln in f:
                if ":" in ln:
                    k_, v_ = (t.strip() for t in ln.split(":", 1))
                    fields.setdefault(k_, v_)
        model = fields.get("model name") or fields.get("Model Name")
        if model is None and "CPU part" in fields:
            model = f"implementer {fields.get('CPU implementer')} part {fields['CPU part']}"
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu": model}


def cpu_baseline_table(args):
    """The oracle's time per operation on every workload, on one host core:
    the median of 3 runs of each (layout, dispatch of the workload's payload,
    combine).  One JSON line per (workload, operation)."""
    import oracle
    from workloads.gen import make_workload, expert_output, CONFIGS, CONFIG_ORDER
    host = host_info()
    for name in CONFIG_ORDER:
        w = make_workload(name)
        y = expert_output(w.N, w.H, seed=w.seed)
        fp8 = CONFIGS[name]["payload"] == "fp8"
        _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
        ops = [("layout", lambda: oracle.layout(w.topk_idx, w.E, w.R)),
               ("dispatch_fp8" if fp8 else "dispatch_bf16",
                (lambda: oracle.dispatch_quant(w.x, slot_of)) if fp8
                else (lambda: oracle.dispatch(w.x, slot_of))),
               ("combine", lambda: oracle.combine(y, slot_of, w.topk_w, "bf16"))]
        for op, fn in ops:
            ts = []
            for _ in range(3):
                t0 = time.perf_counter()
                fn()
                ts.append(time.perf_counter() - t0)
            med = statistics.median(ts)
            print(json.dumps({"workload": name, "op": op, "oracle_median_ms": round(1e3 * med, 3),
                              "tokens_per_s": round(w.T / med, 1), "cores": 1,
                              "host": host}), flush=True)


def cpu_baseline(name: str, budget_s: float = 12.0, w=None, x_np=None, y_np=None):
    """The oracle on the host, single-threaded, over whole steps of the workload
    until `budget_s` of CPU work (at least one step).  `w`, `x_np`, `y_np`: the
    workload and the bit patterns of the inputs the GPU step used (drawn here
    when not given)."""
    from workloads.gen import make_workload, expert_output, CONFIGS
    w = make_workload(name) if w is None else w
    y = expert_output(w.N, w.H, seed=w.seed) if y_np is None else y_np
    x = w.x if x_np is None else x_np
    fp8 = CONFIGS[name]["payload"] == "fp8"
    steps, t0 = 0, time.perf_counter()
    while True:
        oracle_step(w, y, fp8, x)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": steps * w.T / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "host": host_info(),
            "sample": f"{steps} whole {name} steps (T={w.T}: layout + "
                      f"{'fp8 ' if fp8 else ''}dispatch + combine), single-threaded C, "
                      f"{el:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from workloads.gen import make_workload, expert_output, CONFIGS
    name = args.config
    full = CONFIGS[name]["T"]
    Ts = max(1, min(full, args.ref_tokens))
    w = make_workload(name, T=Ts)
    y = expert_output(w.N, w.H, seed=w.seed)
    fp8 = CONFIGS[name]["payload"] == "fp8"
    _ = w.x
    for _ in range(args.warmup):
        oracle_step(w, y, fp8)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, y, fp8)
    el = time.perf_counter() - t0
    value = args.steps * Ts / el
    c = CONFIGS[name]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8-e4m3 + bf16" if fp8 else "bf16", "data": "synthetic",
        "config": {"workload": f"{name} T={c['T']} H={c['H']} k={c['k']} E={c['E']} R={c['R']}",
                   "sample_tokens_per_step": Ts},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "host": host_info(),
                         "sample": f"each step: the {name} recipe at T={Ts} tokens "
                                   f"(layout + {'fp8 ' if fp8 else ''}dispatch + combine)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

class NvmlClocks:
    """Samples the SM clock and the clock-event reasons of one GPU through NVML
    (read-only queries, via ctypes on the driver's libnvidia-ml) on a thread,
    every ~1 ms while a window is open, so that a timed region of a few
    milliseconds still gets samples.  Unavailable NVML leaves no samples."""
    NVML_CLOCK_SM = 1
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str):
        import ctypes
        self.ok = False
        self.samples = []      # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self._stop = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
            self._lib, self._h, self._ct = lib, h, ctypes
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _one(self):
        ct = self._ct
        c = ct.c_uint()
        r = ct.c_ulonglong(0)
        if self._lib.nvmlDeviceGetClockInfo(self._h, self.NVML_CLOCK_SM, ct.byref(c)) != 0:
            return None
        if self._reasons is not None:
            self._reasons(self._h, ct.byref(r))
        return float(c.value), int(r.value)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def _run(self):
        while not self._stop.is_set():
            s = self._one()
            if s is not None:
                self.samples.append(s)
            time.sleep(0.001)

    def __exit__(self, *a):
        if self._stop is not None:
            self._stop.set()
            self._t.join(timeout=2)
            s = self._one()      # and one at the end of the window
            if s is not None:
                self.samples.append(s)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml"}
        bits = 0
        for _, r in self.samples:
            bits |= r
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_min_mhz": min(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASON_BITS.items() if bits & b),
                "samples": len(self.samples), "source": "nvml, ~1 ms, inside the timed region"}


def _ms_list(evs, a, b):
    return [e[a].elapsed_time(e[b]) for e in evs]


class StepBench:
    """Buffers and launch arguments of one workload's step, all resident in
    HBM, and the timed loop over it.

    A step is layout -> dispatch -> combine.  The front segment (A1-A4, or
    A1-A3 + A5 for an FP8 workload) is timed by one event pair; so is the
    combine.  Before the front, a 2xL2 buffer is written (the dispatch pays
    for evicting dirty lines, as its own writes eventually would); before the
    combine, a 4xL2 buffer is read (the combine starts from a cold, clean L2
    and is not charged for the dispatch's write-backs).  Both flushes sit
    outside the events."""

    def __init__(self, name, dev, seed, variant, m, stream=None):
        import torch
        import ctypes
        from workloads.gen import make_workload, CONFIGS, device_inputs
        self.name, self.dev, self.m = name, dev, m
        self.coal = variant == "coalesced"
        self.fp8 = CONFIGS[name]["payload"] == "fp8"
        w = make_workload(name, seed=seed)
        self.w = w
        T, H, k, E, R, N = w.T, w.H, w.k, w.E, w.R, w.N
        self.T, self.H, self.k, self.E, self.R, self.N = T, H, k, E, R, N
        self.x, self.y = device_inputs(w, dev)
        self.idx = torch.from_numpy(w.topk_idx).to(dev)
        self.wt = torch.from_numpy(w.topk_w).to(dev)
        self.err = m.new_error_word(dev)
        self.ws = m.new_workspace(m.moe_layout_workspace_bytes(T, k, E), dev)
        lay = m.Layout(torch.empty(E, dtype=torch.int32, device=dev),
                       torch.empty(E + 1, dtype=torch.int32, device=dev),
                       torch.empty(R + 1, dtype=torch.int32, device=dev),
                       torch.empty((T, k), dtype=torch.int32, device=dev),
                       torch.empty(T * k, dtype=torch.int32, device=dev))
        self.lay = lay
        rows = T * min(k, R)   # coalesced rows: at most one per token and rank
        self.rows = rows
        nrecv = rows if self.coal else N
        self.recv = self.recv_q = self.recv_s = None
        if self.fp8:
            self.recv_q = torch.empty((nrecv, H), dtype=torch.uint8, device=dev)
            self.recv_s = torch.empty((nrecv, H // 128), dtype=torch.float32, device=dev)
        else:
            self.recv = torch.empty((nrecv, H), dtype=torch.bfloat16, device=dev)
        if self.coal:
            self.partial = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
            self.wsc = m.new_workspace(m.moe_layout_workspace_bytes(T, k, R), dev)
            self.co = m.CoalescedLayout(torch.empty(R, dtype=torch.int32, device=dev),
                                        torch.empty(R + 1, dtype=torch.int32, device=dev),
                                        torch.empty((T, k), dtype=torch.int32, device=dev),
                                        torch.empty(T * k, dtype=torch.int32, device=dev),
                                        torch.empty(T * k, dtype=torch.int32, device=dev))
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
        # Reading 2xL2 once leaves some of the dispatch's dirty lines resident
        # on GB300 (combine then pays ~1.6 us of their write-back); one read of
        # 4xL2 evicts them all.
        self.flush_r = torch.zeros(max(4 * l2, 512 << 20), dtype=torch.uint8, device=dev)
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)

        # The step calls the C ABI directly with pre-marshalled arguments, so
        # host time between launches stays far below the GPU time of a step.
        L = m._lib
        self.L = L
        cs = ctypes.c_void_p(self.stream.cuda_stream)
        P = lambda t: t.data_ptr()  # noqa: E731
        self.lay_args = (T, k, E, R, P(self.idx), P(lay.expert_counts), P(lay.expert_offsets),
                         P(lay.rank_offsets), P(lay.slot_of), P(lay.src_of), P(self.ws),
                         self.ws.numel(), P(self.err), cs)
        x, y, err, wt = self.x, self.y, self.err, self.wt
        if self.fp8 and self.coal:
            co = self.co
            self.disp = (L.moe_dispatch_quant_coalesced,
                         (T, H, k, P(x), P(co.crow), rows, P(self.recv_q), P(self.recv_s),
                          P(err), cs))
        elif self.fp8:
            self.disp = (L.moe_dispatch_quant, (T, H, k, P(x), P(lay.slot_of), P(self.recv_q),
                                                P(self.recv_s), P(err), cs))
        elif self.coal:
            self.disp = (L.moe_dispatch_coalesced, (T, H, k, P(x), P(self.co.crow), rows,
                                                    P(self.recv), P(err), cs))
        else:
            self.disp = (L.moe_dispatch, (T, H, k, P(x), P(lay.slot_of), P(self.recv), P(err),
                                          cs))
        if self.coal:
            co = self.co
            self.coal_args = (T, k, E, R, P(self.idx), P(lay.slot_of), P(co.rank_counts_c),
                              P(co.rank_offsets_c), P(co.crow), P(co.src_pair_c), P(co.expand),
                              P(self.wsc), self.wsc.numel(), P(err), cs)
            self.comb = (L.moe_combine_coalesced, (T, H, k, P(y), P(lay.slot_of), P(wt),
                                                   P(co.crow), rows, P(self.partial), P(self.out),
                                                   m.MOE_OUT_BF16, P(err), cs))
        else:
            self.comb = (L.moe_combine, (T, H, k, P(y), P(lay.slot_of), P(wt), P(self.out),
                                         m.MOE_OUT_BF16, P(err), cs))
        # layout then dispatch as one call where the library offers it (bf16):
        # the dispatch's first loads of x overlap the layout
        self.fused_front = not self.fp8 and not self.coal
        self.front_args = (T, H, k, E, R, P(self.idx), P(x), P(lay.expert_counts),
                           P(lay.expert_offsets), P(lay.rank_offsets), P(lay.slot_of),
                           P(lay.src_of), P(self.recv) if self.fused_front else None, P(self.ws),
                           self.ws.numel(), P(err), cs)
        # FP8: layout then the FP8 dispatch as one call, the dispatch's first
        # loads and quantisation of x overlapping the layout
        self.fused_front_quant = self.fp8 and not self.coal
        self.front_quant_args = (T, H, k, E, R, P(self.idx), P(x), P(lay.expert_counts),
                                 P(lay.expert_offsets), P(lay.rank_offsets), P(lay.slot_of),
                                 P(lay.src_of), P(self.recv_q) if self.fp8 else None,
                                 P(self.recv_s) if self.fp8 else None, P(self.ws),
                                 self.ws.numel(), P(err), cs)
        self.d_name = (("dispatch_fp8_coalesced" if self.fp8 else "dispatch_coalesced")
                       if self.coal else ("dispatch_fp8" if self.fp8 else "dispatch_bf16"))
        self.c_name = "combine_coalesced" if self.coal else "combine"

    # -- launches
    def _call(self, fn, a):
        st = fn(*a)
        if st != self.m.MOE_OK:
            raise self.m.MoeError(st, fn.__name__)

    def layout_only(self):
        self._call(self.L.moe_layout, self.lay_args)
        if self.coal:
            self._call(self.L.moe_layout_coalesced, self.coal_args)

    def dispatch_only(self):
        self._call(*self.disp)

    def front(self):
        if self.fused_front:
            self._call(self.L.moe_layout_dispatch, self.front_args)
        elif self.fused_front_quant:
            self._call(self.L.moe_layout_dispatch_quant, self.front_quant_args)
        else:
            self.layout_only()
            self.dispatch_only()

    def combine_only(self):
        self._call(*self.comb)

    def dirty_flush(self):
        self.flush.fill_(0)

    def clean_flush(self):
        import torch
        self.flush_r.view(torch.int64).sum()

    def launches_per_step(self):
        # layout, dispatch, combine (layout and dispatch are one kernel when
        # moe_layout_dispatch takes its single-kernel form); the coalesced
        # step adds the coalesced layout (a second launch when k does not
        # divide 32)
        if self.coal:
            return 4 if 32 % self.k == 0 else 5
        if self.fused_front:
            self.front()
            if self.m.moe_layout_last_form() == self.m.MOE_LAYOUT_FORM_FUSED:
                return 2
        return 3

    def step(self, ev=None):
        st = self.stream
        self.dirty_flush()
        if ev:
            ev[0].record(st)
        self.front()
        if ev:
            ev[1].record(st)
        self.clean_flush()
        if ev:
            ev[2].record(st)
        self.combine_only()
        if ev:
            ev[3].record(st)

    def check_errors(self, where):
        bits = self.m.moe_read_error(self.err)
        if bits:
            raise RuntimeError(f"device error bits {bits:#x} {where} ({self.name})")

    def timed(self, steps, warmup, clocks_uuid=None):
        """W warm-up steps, then exactly `steps` timed steps between a barrier
        and a device synchronisation; then a breakdown pass (an event pair
        around the layout and around the dispatch, outside the timed steps)."""
        import torch
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        self.check_errors("during warm-up")
        self.Nc = int(self.co.rank_offsets_c[self.R].item()) if self.coal else self.N
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        nv = NvmlClocks(clocks_uuid) if clocks_uuid else None
        barrier()
        torch.cuda.synchronize()
        with (nv if nv is not None else _Null()):
            t0 = time.perf_counter()
            for i in range(steps):
                self.step(ev[i])
            torch.cuda.synchronize()
            wall = time.perf_counter() - t0
        barrier()
        self.check_errors("in the timed steps")
        t_front = _ms_list(ev, 0, 1)
        t_comb = _ms_list(ev, 2, 3)
        nsplit = max(3, min(steps, 200))
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nsplit)]
        for i in range(nsplit):
            self.dirty_flush()
            evs[i][0].record(self.stream)
            self.layout_only()
            evs[i][1].record(self.stream)
            self.dispatch_only()
            evs[i][2].record(self.stream)
        torch.cuda.synchronize()
        self.check_errors("in the breakdown pass")
        return {"t_front": t_front, "t_comb": t_comb, "t_layout": _ms_list(evs, 0, 1),
                "t_disp": _ms_list(evs, 1, 2), "wall": wall,
                "clocks": nv.summary() if nv is not None else None}

    def bytes_of(self, name):
        T, H, k, E, R = self.T, self.H, self.k, self.E, self.R
        if self.coal:
            if name == "front":
                return (kernel_bytes("layout_assign", T, H, k, E, R) +
                        coalesced_bytes("layout_coalesced", T, H, k, self.Nc) +
                        coalesced_bytes(self.d_name, T, H, k, self.Nc))
            return coalesced_bytes(name, T, H, k, self.Nc)
        if name == "front":
            return kernel_bytes("layout_assign", T, H, k, E, R) + kernel_bytes(self.d_name, T, H,
                                                                               k, E, R)
        return kernel_bytes(name, T, H, k, E, R)


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def _frac(nbytes, ms, peak):
    gbs = nbytes / (ms / 1000.0) / 1e9
    return {"ms": ms, "bytes": nbytes, "gbs": gbs, "frac": gbs / peak}


def per_config_entry(b: StepBench, r: dict, peak: float) -> dict:
    """The in-step figures of one workload: the front segment (the pages'
    dispatch, A1-A4/A5: layout and dispatch), the dispatch kernel alone (the
    breakdown pass), and the combine (timed steps), each with its algorithmic
    bytes and the fraction of the measured HBM peak."""
    front = statistics.mean(r["t_front"])
    comb = statistics.mean(r["t_comb"])
    disp = statistics.mean(r["t_disp"])
    steps = len(r["t_front"])
    return {
        "workload": f"{b.name} T={b.T} H={b.H} k={b.k} E={b.E} R={b.R}",
        "payload": "fp8-e4m3" if b.fp8 else "bf16",
        "steps": steps,
        "tokens_per_s": b.T * steps / (sum(r["t_front"]) + sum(r["t_comb"])) * 1000.0,
        "ms_per_step": front + comb,
        "dispatch": dict(_frac(b.bytes_of("front"), front, peak),
                         what="layout + dispatch in the timed steps (A1-A4 or A1-A3 + A5)",
                         call="moe_layout_dispatch" if b.fused_front else
                              "moe_layout_dispatch_quant" if b.fused_front_quant else
                              f"moe_layout + {b.disp[0].__name__}"),
        "dispatch_kernel": dict(_frac(b.bytes_of(b.d_name), disp, peak),
                                what="the dispatch kernel alone, breakdown pass"),
        "layout_ms": statistics.mean(r["t_layout"]),
        "combine": dict(_frac(b.bytes_of(b.c_name), comb, peak),
                        what="combine in the timed steps"),
    }


def oracle_op_times(name, x_bits, y_bits, w, budget_s=1.0):
    """The oracle's time per operation on the full workload, on one host core:
    each op once, repeated (median of up to 3) while it stays under
    `budget_s` in total."""
    import oracle
    from workloads.gen import CONFIGS
    fp8 = CONFIGS[name]["payload"] == "fp8"
    _, _, _, slot_of, _ = oracle.layout(w.topk_idx, w.E, w.R)
    ops = [("layout", lambda: oracle.layout(w.topk_idx, w.E, w.R)),
           ("dispatch_fp8" if fp8 else "dispatch_bf16",
            (lambda: oracle.dispatch_quant(x_bits, slot_of)) if fp8
            else (lambda: oracle.dispatch(x_bits, slot_of))),
           ("combine", lambda: oracle.combine(y_bits, slot_of, w.topk_w, "bf16"))]
    res = {}
    for op, fn in ops:
        ts = []
        while len(ts) < 3 and (not ts or sum(ts) < budget_s):
            t0 = time.perf_counter()
            fn()
            ts.append(time.perf_counter() - t0)
        med = statistics.median(ts)
        res[op] = {"ms": 1e3 * med, "tokens_per_s": w.T / med, "reps": len(ts)}
    return res


def host_bits(t):
    """uint16 numpy bit patterns of a bf16 device tensor."""
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_gpu(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if (world > 1 or args.ep_nccl) and not dist.is_initialized():
        import datetime
        dist.init_process_group("nccl", timeout=datetime.timedelta(seconds=180))
    if world > 1 or args.ep_nccl or args.ep_virtual > 1:
        return run_gpu_ep(args, rank, world, local)
    dev = torch.device("cuda", local)

    import combine_layout_moe_gb300 as m

    name = args.config
    uuid = gpu_smi_id(torch, dev)
    peak, peak_kind = measured_peak_gbs()
    b = StepBench(name, dev, args.seed + rank, args.variant, m)
    T, H, k, E, R, N = b.T, b.H, b.k, b.E, b.R, b.N
    coal, fp8 = b.coal, b.fp8

    smi = ClockSampler(uuid).__enter__()   # nvidia-smi, over every timed region
    smi.mark_start()
    r = b.timed(args.steps, args.warmup, clocks_uuid=uuid)
    t_front, t_comb = r["t_front"], r["t_comb"]
    t_step = [a + c for a, c in zip(t_front, t_comb)]
    total_ms = allreduce_max(sum(t_step))
    ms_per_step = total_ms / args.steps
    value = world * T * args.steps / (total_ms / 1000.0)

    # roofline of the dominant kernel: combine is timed alone inside the timed
    # steps; dispatch (when it dominates) in the breakdown pass.
    avg_d, avg_c = statistics.mean(r["t_disp"]), statistics.mean(t_comb)
    if avg_c >= avg_d:
        dom, dom_ms, source = b.c_name, avg_c, "timed steps"
    else:
        dom, dom_ms, source = b.d_name, avg_d, "breakdown pass (one event pair per kernel)"
    dom_bytes = b.bytes_of(dom)
    achieved = dom_bytes / (dom_ms / 1000.0) / 1e9
    kern_name = {"dispatch_bf16": "dispatch_bulk_kernel", "dispatch_fp8": "dispatch_fp8_kernel",
                 "combine": "combine_bulk_kernel",
                 "dispatch_coalesced": "dispatch_bulk_kernel<coalesced>",
                 "dispatch_fp8_coalesced": "dispatch_fp8_kernel<coalesced>",
                 "combine_coalesced": "combine_bulk_kernel<coalesced>"}[dom]
    tr = None if coal else recorded_traffic(kern_name, name)
    traffic = tr.get("dram_bytes_per_launch") if tr is not None else None

    launches = b.launches_per_step() * args.steps
    e2e = e2e_leg(b, args, world)
    headline = per_config_entry(b, r, peak)
    headline["clocks"] = r["clocks"]
    x_host = y_host = None
    want_cpu = not args.no_cpu_baseline and world == 1 and rank == 0 and not coal
    if want_cpu:
        x_host, y_host = host_bits(b.x), host_bits(b.y)
    w_head = b.w
    Nc = b.Nc
    del b
    torch.cuda.empty_cache()

    # the other workloads of the target (configs 1-4), each through the same
    # timed loop and L2 regime, one after the other
    per_config = {name: headline}
    host_inputs = {name: (w_head, x_host, y_host)}
    if not args.no_per_config and not coal:
        for other in args.per_config.split(","):
            if not other or other == name:
                continue
            bo = StepBench(other, dev, args.seed + rank, "plain", m)
            # the other workloads are context for the headline: timed over at
            # least PER_CONFIG_MIN_STEPS steps, so a short headline run (the
            # decode step is ~55 us of GPU time) still gives stable averages
            ro = bo.timed(max(args.steps, PER_CONFIG_MIN_STEPS), max(args.warmup, 20),
                          clocks_uuid=uuid)
            per_config[other] = per_config_entry(bo, ro, peak)
            per_config[other]["clocks"] = ro["clocks"]
            if want_cpu:
                host_inputs[other] = (bo.w, host_bits(bo.x), host_bits(bo.y))
            del bo
            torch.cuda.empty_cache()
    smi.mark_stop()
    smi.__exit__(None, None, None)

    if rank != 0:
        return
    clocks = r["clocks"] or {"samples": 0}
    if not clocks.get("samples"):
        clocks = smi.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8-e4m3 + bf16" if fp8 else "bf16", "data": "synthetic",
        "config": {"workload": f"{name} T={T} H={H} k={k} E={E} R={R}",
                   "tokens_per_step": T, "variant": args.variant,
                   "l2": "flushed every step outside the events: 2xL2 written before layout+"
                         "dispatch, 4xL2 read before combine",
                   "inputs": "routing from workloads/gen.py (seed 0); x ~ N(0,1) and the expert "
                             "outputs drawn on the device with torch's seeded generator",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": kern_name, "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)", "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "traffic_source": tr.get("capture") if tr is not None else None,
                     "algorithmic_bytes": dom_bytes, "duration_ms": dom_ms,
                     "duration_source": source},
        "segments_ms": {"layout+" + b_dname(fp8, coal): statistics.mean(t_front),
                        "combine": avg_c},
        "kernels_ms": {"layout": statistics.mean(r["t_layout"]), b_dname(fp8, coal): avg_d,
                       "combine": avg_c},
        "step_hbm_gbs": (None if coal else
                         step_bytes(T, H, k, E, R, fp8) / (ms_per_step / 1000.0) / 1e9),
        "wall_ms_per_step_incl_flush": 1000.0 * r["wall"] / args.steps,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "clocks_window": smi.summary(),
        "per_config": per_config,
    }
    if coal:
        line["config"]["coalesced_rows"] = {"N": N, "Nc": Nc}
    if want_cpu:
        wh, xh, yh = host_inputs[name]
        line["cpu_baseline"] = cpu_baseline(name, args.cpu_budget, wh, xh, yh)
        for nm, (wo, xo, yo) in host_inputs.items():
            per_config[nm]["oracle_1core"] = oracle_op_times(nm, xo, yo, wo)
    print(json.dumps(line), flush=True)


def run_gpu_ep(args, rank, world, local):
    """Expert parallelism across ranks.  Under torchrun (N > 1) each GPU is
    one rank of W = N: it holds T tokens of the workload (drawn with seed
    seed + rank) and E / W of the experts, and a step is layout (R = W) ->
    dispatch -> the counts all-to-all and the rows' all-to-all-v over NCCL ->
    the receiver's reorder -> identity experts -> the reverse reorder and
    all-to-all-v -> combine.  With --ep-virtual W on one GPU the W ranks run
    in one process and the exchange is a device copy of each segment.  The
    timed step brackets the whole of it with CUDA events on the current
    stream (the host reads the split sizes back twice per step, as any
    all-to-all-v must); value = W x T tokens over the MAX over ranks."""
    import torch
    import combine_layout_moe_gb300 as m
    from combine_layout_moe_gb300 import ep
    from workloads.gen import make_workload, device_inputs

    dev = torch.device("cuda", local)
    name = args.config
    virtual = world == 1 and not args.ep_nccl
    W = args.ep_virtual if virtual else world
    err = m.new_error_word(dev)
    ops = ep.LibraryOps(err)
    mine = range(W) if virtual else [rank]
    ws_, xs, idxs, wts = [], [], [], []
    for r in mine:
        w = make_workload(name, seed=args.seed + r)
        x, _ = device_inputs(w, dev)
        ws_.append(w)
        xs.append(x)
        idxs.append(torch.from_numpy(w.topk_idx).to(dev))
        wts.append(torch.from_numpy(w.topk_w).to(dev))
    T, H, k, E = ws_[0].T, ws_[0].H, ws_[0].k, ws_[0].E
    if E % W:
        raise SystemExit(f"{name}: E = {E} experts do not divide over {W} ranks")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    epl = None if virtual else ep.ExpertParallel(E, ops=ops)

    def step():
        if virtual:
            return ep.virtual_step(xs, idxs, wts, E, ops=ops)[2]
        recv, offs, handle = epl.dispatch(xs[0], idxs[0])
        return [epl.combine(recv, handle, wts[0])]

    for _ in range(args.warmup):
        outs = step()
    torch.cuda.synchronize()
    bits = m.moe_read_error(err)
    if bits:
        raise RuntimeError(f"device error bits {bits:#x} during warm-up")
    # identity experts and weights summing to one: each rank's tokens come back
    for x, o in zip(xs, outs):
        nz = x != 0
        if not torch.equal(o[nz].view(torch.int16), x[nz].view(torch.int16)):
            raise RuntimeError("expert-parallel round trip did not return x")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    nv = NvmlClocks(gpu_smi_id(torch, dev))
    barrier()
    torch.cuda.synchronize()
    with nv:
        for a, b in ev:
            flush.fill_(0)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
    barrier()
    total_ms = allreduce_max(sum(a.elapsed_time(b) for a, b in ev))
    ms = total_ms / args.steps
    if rank != 0:
        return
    tokens = W * T
    peak, peak_kind = measured_peak_gbs()
    line = {
        "metric": METRIC, "value": tokens / (ms / 1000.0), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{name} T={T} per rank H={H} k={k} E={E}",
                   "parallelism": (f"ep{W} virtual ranks on one GPU (exchange by device copy)"
                                   if virtual else f"ep{W}: experts over {W} GPUs, NCCL "
                                                   "all-to-all-v"),
                   "tokens_per_step": tokens,
                   "l2": "2xL2 written before each step, outside the events"},
        "step": "layout (R = W) -> dispatch -> counts all-to-all -> rows all-to-all-v -> "
                "receiver reorder -> identity experts -> reverse reorder -> rows all-to-all-v "
                "-> combine",
        "roofline": None,
        "roofline_note": f"the step includes the exchange and two host readbacks of split "
                         f"sizes; the local kernels' fractions of HBM peak ({peak_kind} "
                         f"{peak} GB/s) are in the single-GPU line",
        "gpu_launches": (5 if not virtual else 5 * W) * args.steps,  # layout, dispatch, 2 reorders, combine
        "clocks": nv.summary(),
    }
    print(json.dumps(line), flush=True)


def b_dname(fp8, coal):
    return (("dispatch_fp8_coalesced" if fp8 else "dispatch_coalesced") if coal
            else ("dispatch_fp8" if fp8 else "dispatch_bf16"))


def e2e_leg(b: StepBench, args, world):
    """The step through the public API with host buffers: every step copies its
    inputs from pinned host memory and reads its combined output back.  Steps
    are pipelined on three streams (H2D of step i+1 and D2H of step i-1
    overlap step i's kernels), with double-buffered device inputs and
    outputs.  No flush here: one step's footprint (x, recv, y, out) is larger
    than L2.  A step's inputs (x, topk_idx, topk_w) sit in one pinned host slab
    and go over in one copy, into one device slab that the calls take views
    of: each separate small copy cost the host link ~7.5 us per step."""
    import torch
    m, dev, stream = b.m, b.dev, b.stream
    T, H, k, E, R = b.T, b.H, b.k, b.E, b.R
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    XB, IB, WB = T * H * 2, T * k * 4, T * k * 4
    in_h = torch.empty(XB + IB + WB, dtype=torch.uint8).pin_memory()
    in_h[:XB].copy_(b.x.view(torch.uint8).reshape(-1).cpu())
    in_h[XB:XB + IB].copy_(torch.from_numpy(b.w.topk_idx.view(np.uint8).reshape(-1)))
    in_h[XB + IB:].copy_(torch.from_numpy(b.w.topk_w.view(np.uint8).reshape(-1)))
    in_d = [torch.empty(XB + IB + WB, dtype=torch.uint8, device=dev) for _ in range(2)]
    out_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xb = [d[:XB].view(torch.bfloat16).view(T, H) for d in in_d]
    ib = [d[XB:XB + IB].view(torch.int32).view(T, k) for d in in_d]
    wb = [d[XB + IB:].view(torch.float32).view(T, k) for d in in_d]
    ob = [b.out, torch.empty_like(b.out)]
    y, lay, ws, err = b.y, b.lay, b.ws, b.err
    rq = (dict(recv_q=b.recv_q, recv_scales=b.recv_s) if b.fp8
          else (dict(recv_c=b.recv) if b.coal else dict(recv=b.recv)))
    steps = max(1, min(args.steps, args.e2e_steps))

    def run(n):
        h2d_done = [torch.cuda.Event() for _ in range(n)]
        comp_done = [torch.cuda.Event() for _ in range(n)]
        d2h_done = [torch.cuda.Event() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(h2d_s)
        for i in range(n):
            j = i % 2
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(comp_done[i - 2])
                in_d[j].copy_(in_h, non_blocking=True)
                h2d_done[i].record(h2d_s)
            stream.wait_event(h2d_done[i])
            if i >= 2:
                stream.wait_event(d2h_done[i - 2])
            if b.fused_front:
                m.moe_layout_dispatch(xb[j], ib[j], E, R, workspace=ws, out=lay, err_word=err,
                                      stream=stream, **rq)
                m.moe_combine(y, lay.slot_of, wb[j], out=ob[j], err_word=err, stream=stream)
            elif b.coal:
                co = b.co
                m.moe_layout(ib[j], E, R, workspace=ws, err_word=err, out=lay, stream=stream)
                m.moe_layout_coalesced(ib[j], lay.slot_of, E, R, workspace=b.wsc, err_word=err,
                                       out=co, stream=stream)
                if b.fp8:
                    m.moe_dispatch_quant_coalesced(xb[j], co.crow, b.rows, err_word=err,
                                                   stream=stream, **rq)
                else:
                    m.moe_dispatch_coalesced(xb[j], co.crow, b.rows, err_word=err,
                                             stream=stream, **rq)
                m.moe_combine_coalesced(y, lay.slot_of, wb[j], co, b.rows, partial=b.partial,
                                        out=ob[j], err_word=err, stream=stream)
            else:
                m.moe_layout_dispatch_quant(xb[j], ib[j], E, R, workspace=ws, out=lay,
                                            err_word=err, stream=stream, **rq)
                m.moe_combine(y, lay.slot_of, wb[j], out=ob[j], err_word=err, stream=stream)
            comp_done[i].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(comp_done[i])
                out_h[j].copy_(ob[j], non_blocking=True)
                d2h_done[i].record(d2h_s)
        d2h_s.wait_event(d2h_done[n - 1])
        t1.record(d2h_s)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    run(3)  # warm-up
    e2e_ms = allreduce_max(run(steps)) / steps
    b.check_errors("in the e2e leg")
    # the last output read back must be the combine of the resident inputs
    if b.coal:
        ref, _ = m.moe_combine_coalesced(y, lay.slot_of, b.wt, b.co, b.rows, partial=b.partial)
    else:
        ref = m.moe_combine(y, lay.slot_of, b.wt)
    torch.cuda.synchronize()
    if not torch.equal(out_h[(steps - 1) % 2].view(torch.int16), ref.cpu().view(torch.int16)):
        raise RuntimeError("e2e output differs from the combine of the resident inputs")
    return {"value": world * T / (e2e_ms / 1000.0), "unit": UNIT,
            "h2d_bytes_per_step": in_h.numel(), "d2h_bytes_per_step": b.out.numel() * 2,
            "ms_per_step": e2e_ms, "steps": steps,
            "how": "public API; one H2D copy per step (x, topk_idx, topk_w in one pinned "
                   "slab); H2D of step i+1 and D2H of step i-1 overlap step i's kernels "
                   "(three streams, double-buffered inputs/outputs); one step's footprint "
                   "exceeds L2"}


# ------------------------------------------------------------------ kernel table

def run_table(args):
    """Every entry point alone, on every workload: each launch follows a write
    of 2xL2 and a read of 4xL2 (cold, clean L2), bracketed by CUDA events on
    its stream; 5 warm-ups, then args.table_reps launches.  Prints one JSON
    line per (workload, kernel): median and minimum time, algorithmic bytes,
    achieved GB/s and the fraction of the measured HBM peak."""
    import torch
    import combine_layout_moe_gb300 as m
    from workloads.gen import make_workload, expert_output, CONFIGS, CONFIG_ORDER

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    fw = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    fr = torch.zeros(max(4 * l2, 512 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = measured_peak_gbs()
    names = CONFIG_ORDER if args.table_all else [args.config]
    for name in names:
        w = make_workload(name)
        T, H, k, E, R, N = w.T, w.H, w.k, w.E, w.R, w.N
        bf = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)  # noqa: E731
        x, y = bf(w.x), bf(expert_output(N, H, seed=w.seed))
        dout = bf(expert_output(T, H, seed=w.seed + 1))
        idx = torch.from_numpy(w.topk_idx).to(dev)
        wt = torch.from_numpy(w.topk_w).to(dev)
        err = m.new_error_word(dev)
        ws = m.new_workspace(m.moe_layout_workspace_bytes(T, k, E), dev)
        wsc = m.new_workspace(m.moe_layout_workspace_bytes(T, k, R), dev)
        lay = m.moe_layout(idx, E, R, workspace=ws, err_word=err)
        co = m.moe_layout_coalesced(idx, lay.slot_of, E, R, workspace=wsc, err_word=err)
        torch.cuda.synchronize()
        Nc = int(co.rank_offsets_c[R].item())
        rows = T * min(k, R)
        recv = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        rq = torch.empty((N, H), dtype=torch.uint8, device=dev)
        rs = torch.empty((N, H // 128), dtype=torch.float32, device=dev)
        rc = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
        part = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        dy = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        dw = torch.empty((T, k), dtype=torch.float32, device=dev)
        kw = dict(err_word=err, stream=stream)
        ops = [
            ("layout", lambda: m.moe_layout(idx, E, R, workspace=ws, out=lay, **kw),
             kernel_bytes("layout_assign", T, H, k, E, R)),
            ("layout_dispatch", lambda: m.moe_layout_dispatch(x, idx, E, R, workspace=ws, out=lay,
                                                              recv=recv, **kw),
             kernel_bytes("layout_dispatch", T, H, k, E, R)),
            ("dispatch_bf16", lambda: m.moe_dispatch(x, lay.slot_of, recv=recv, **kw),
             kernel_bytes("dispatch_bf16", T, H, k, E, R)),
            ("combine", lambda: m.moe_combine(y, lay.slot_of, wt, out=out, **kw),
             kernel_bytes("combine", T, H, k, E, R)),
            ("combine_backward", lambda: m.moe_combine_backward(dout, y, lay.slot_of, wt, dy=dy,
                                                                dw=dw, **kw),
             kernel_bytes("combine_backward", T, H, k, E, R)),
            ("dispatch_backward", lambda: m.moe_dispatch_backward(y, lay.slot_of, dx=out, **kw),
             kernel_bytes("dispatch_backward", T, H, k, E, R)),
            ("layout_coalesced", lambda: m.moe_layout_coalesced(idx, lay.slot_of, E, R,
                                                                workspace=wsc, out=co, **kw),
             coalesced_bytes("layout_coalesced", T, H, k, Nc)),
            ("dispatch_coalesced", lambda: m.moe_dispatch_coalesced(x, co.crow, rows, recv_c=rc,
                                                                    **kw),
             coalesced_bytes("dispatch_coalesced", T, H, k, Nc)),
            ("combine_coalesced", lambda: m.moe_combine_coalesced(y, lay.slot_of, wt, co, rows,
                                                                  partial=part, out=out, **kw),
             coalesced_bytes("combine_coalesced", T, H, k, Nc)),
        ]
        if H % 128 == 0:
            ops.insert(3, ("dispatch_fp8", lambda: m.moe_dispatch_quant(x, lay.slot_of, recv_q=rq,
                                                                        recv_scales=rs, **kw),
                           kernel_bytes("dispatch_fp8", T, H, k, E, R)))
            ops.insert(-1, ("dispatch_fp8_coalesced",
                            lambda: m.moe_dispatch_quant_coalesced(x, co.crow, rows, recv_q=rq,
                                                                   recv_scales=rs, **kw),
                            coalesced_bytes("dispatch_fp8_coalesced", T, H, k, Nc)))
        if args.table_flagged:
            # A7: dispatch -> identity expert -> combine in one kernel, per
            # readiness mode and granularity, against the same three steps as
            # separate launches (the expert is torch's copy of recv into y)
            yf = torch.empty_like(y)
            nb_f = 4 * T * H + 8 * N * H
            ops = [("separate", lambda: (m.moe_dispatch(x, lay.slot_of, recv=recv, **kw),
                                         yf.copy_(recv),
                                         m.moe_combine(yf, lay.slot_of, wt, out=out, **kw)), nb_f)]
            for mode, grans in ((m.MOE_SYNC_BARRIER, (2048,)), (m.MOE_SYNC_BATCH, (2048, 4096, 8192)),
                                (m.MOE_SYNC_WORD, (2048, 4096, 8192)), (m.MOE_SYNC_SENTINEL, (2048,))):
                for g in grans:
                    label = {m.MOE_SYNC_BARRIER: "barrier", m.MOE_SYNC_BATCH: f"batch_{g}",
                             m.MOE_SYNC_WORD: f"word_{g}", m.MOE_SYNC_SENTINEL: "sentinel"}[mode]
                    ops.append((f"flagged_{label}", (mode, g), nb_f))
        for op, fn, nbytes in ops:
            state = None
            if isinstance(fn, tuple):
                state = m.SyncState(T, H, k, fn[0], fn[1], device=dev)
                fn = (lambda st: lambda: m.moe_dispatch_combine_flagged(x, lay.slot_of, wt, st,
                                                                         out=out, **kw))(state)
            evs = []
            for i in range(5 + args.table_reps):
                fw.fill_(0)
                fr.view(torch.int64).sum()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                if i >= 5:
                    evs.append((a, b))
            torch.cuda.synchronize()
            us = sorted(a.elapsed_time(b) * 1000.0 for a, b in evs)
            med = statistics.median(us)
            bits = m.moe_read_error(err)
            if bits:
                raise RuntimeError(f"device error bits {bits:#x} in {name}/{op}")
            gbs = nbytes / (med * 1e-6) / 1e9
            del state
            print(json.dumps({"workload": name, "kernel": op, "median_us": round(med, 2),
                              "min_us": round(us[0], 2), "algorithmic_bytes": nbytes,
                              "gbs": round(gbs, 1), "frac": round(gbs / peak, 3),
                              "peak": f"{peak_kind} hbm_gbs {peak}",
                              "rows": {"N": N, "Nc": Nc}}), flush=True)
        del x, y, dout, recv, rq, rs, rc, part, out, dy, ops
        torch.cuda.empty_cache()


def run_profile_op(args):
    """One entry point on one workload, for an ncu capture: args.warmup
    launches, then args.steps launches, each after a write of 2xL2 and a read
    of 4xL2 and bracketed by CUDA events; prints the median.  Only the buffers
    that entry point needs are allocated.  --shape T,H,k,E,R replaces the
    workload by a uniform random routing of that shape."""
    import torch
    import combine_layout_moe_gb300 as m
    from workloads.gen import make_workload, random_case, device_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.shape:
        T, H, k, E, R = (int(v) for v in args.shape.split(","))
        w = random_case(args.seed, T, H, k, E, R)
        name = f"random T={T} H={H} k={k} E={E} R={R}"
    else:
        w = make_workload(args.config, seed=args.seed)
        T, H, k, E, R = w.T, w.H, w.k, w.E, w.R
        name = f"{args.config} T={T} H={H} k={k} E={E} R={R}"
    N = T * k
    x, y = device_inputs(w, dev)
    idx = torch.from_numpy(w.topk_idx).to(dev)
    wt = torch.from_numpy(w.topk_w).to(dev)
    err = m.new_error_word(dev)
    ws = m.new_workspace(m.moe_layout_workspace_bytes(T, k, E), dev)
    lay = m.moe_layout(idx, E, R, workspace=ws, err_word=err)
    kw = dict(err_word=err)
    op = args.profile_op
    if op in ("layout_coalesced", "dispatch_coalesced", "combine_coalesced"):
        wsc = m.new_workspace(m.moe_layout_workspace_bytes(T, k, R), dev)
        co = m.moe_layout_coalesced(idx, lay.slot_of, E, R, workspace=wsc, err_word=err)
        rows = T * min(k, R)
    if op == "layout":
        fn = lambda: m.moe_layout(idx, E, R, workspace=ws, out=lay, **kw)  # noqa: E731
    elif op == "layout_dispatch":
        recv = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        fn = lambda: m.moe_layout_dispatch(x, idx, E, R, workspace=ws, out=lay, recv=recv,  # noqa: E731
                                           **kw)
    elif op == "dispatch":
        recv = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        fn = lambda: m.moe_dispatch(x, lay.slot_of, recv=recv, **kw)  # noqa: E731
    elif op == "layout_dispatch_quant":
        rq = torch.empty((N, H), dtype=torch.uint8, device=dev)
        rs = torch.empty((N, H // 128), dtype=torch.float32, device=dev)
        fn = lambda: m.moe_layout_dispatch_quant(x, idx, E, R, workspace=ws, out=lay,  # noqa: E731
                                                 recv_q=rq, recv_scales=rs, **kw)
    elif op == "dispatch_fp8":
        rq = torch.empty((N, H), dtype=torch.uint8, device=dev)
        rs = torch.empty((N, H // 128), dtype=torch.float32, device=dev)
        fn = lambda: m.moe_dispatch_quant(x, lay.slot_of, recv_q=rq, recv_scales=rs, **kw)  # noqa: E731
    elif op == "combine":
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        fn = lambda: m.moe_combine(y, lay.slot_of, wt, out=out, **kw)  # noqa: E731
    elif op == "combine_backward":
        dout = torch.empty((T, H), dtype=torch.bfloat16, device=dev).normal_()
        dy = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        dw = torch.empty((T, k), dtype=torch.float32, device=dev)
        fn = lambda: m.moe_combine_backward(dout, y, lay.slot_of, wt, dy=dy, dw=dw, **kw)  # noqa: E731
    elif op == "dispatch_backward":
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        fn = lambda: m.moe_dispatch_backward(y, lay.slot_of, dx=out, **kw)  # noqa: E731
    elif op == "layout_coalesced":
        fn = lambda: m.moe_layout_coalesced(idx, lay.slot_of, E, R, workspace=wsc, out=co, **kw)  # noqa: E731
    elif op == "dispatch_coalesced":
        rc = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
        fn = lambda: m.moe_dispatch_coalesced(x, co.crow, rows, recv_c=rc, **kw)  # noqa: E731
    elif op == "combine_coalesced":
        part = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        fn = lambda: m.moe_combine_coalesced(y, lay.slot_of, wt, co, rows, partial=part,  # noqa: E731
                                             out=out, **kw)
    elif op == "ep_reorder":
        # the receiver's reorder of R ranks' rows: the counts of a receiver
        # that gets this workload's tokens from each of R sources, one local
        # expert per source slice (E / R of them)
        El = E // R
        cnt = lay.expert_counts.view(R, El)
        src = y[:N]
        dst = torch.empty_like(src)
        fn = lambda: m.moe_ep_reorder(src, cnt, out=dst, **kw)  # noqa: E731
    else:
        raise SystemExit(f"unknown --profile-op {op}")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    fw = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    fr = torch.zeros(4 * l2, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()  # the input draw's temporaries: keep the footprint small
    evs = []
    for i in range(args.warmup + args.steps):
        fw.fill_(0)
        fr.view(torch.int64).sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        if i >= args.warmup:
            evs.append((a, b))
    torch.cuda.synchronize()
    bits = m.moe_read_error(err)
    if bits:
        raise RuntimeError(f"device error bits {bits:#x}")
    us = sorted(a.elapsed_time(b) * 1000.0 for a, b in evs)
    print(json.dumps({"profile_op": op, "workload": name, "launches": len(us),
                      "median_us": statistics.median(us), "min_us": us[0],
                      "layout_form": m.moe_layout_last_form()}), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=4000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default=DEFAULT_WORKLOAD)
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--cpu-budget", type=float, default=12.0)
    p.add_argument("--ref-tokens", type=int, default=2048,
                   help="tokens per oracle step in --impl reference")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--per-config", default=PER_CONFIG,
                   help="comma-separated workloads timed after the headline, each through "
                        "the same loop, reported in the line's per_config block")
    p.add_argument("--no-per-config", action="store_true")
    p.add_argument("--profile-op", default=None,
                   help="time one entry point alone on --config (or --shape), for ncu "
                        "captures: layout, layout_dispatch, layout_dispatch_quant, dispatch, "
                        "dispatch_fp8, combine, "
                        "combine_backward, dispatch_backward, layout_coalesced, "
                        "dispatch_coalesced, combine_coalesced, ep_reorder")
    p.add_argument("--shape", default=None, help="with --profile-op: T,H,k,E,R of a uniform "
                                                 "random routing instead of --config")
    p.add_argument("--ep-nccl", action="store_true",
                   help="run the expert-parallel step through an NCCL process group even with "
                        "one rank (under torchrun), to exercise the exchange on one GPU")
    p.add_argument("--ep-virtual", type=int, default=1,
                   help="on one GPU: time expert parallelism over W virtual ranks (the "
                        "exchange done by device copies) instead of the single-GPU step")
    p.add_argument("--variant", choices=["plain", "coalesced"], default="plain",
                   help="plain: the hot path; coalesced: the rank-coalesced path")
    p.add_argument("--table", action="store_true",
                   help="time every entry point alone after a flush (one JSON line each) "
                        "on --config, or on every workload with --table-all")
    p.add_argument("--table-all", action="store_true")
    p.add_argument("--table-flagged", action="store_true",
                   help="with --table: the single-kernel Data-as-Flag variant per readiness "
                        "mode and granularity, against separate launches")
    p.add_argument("--table-reps", type=int, default=50)
    p.add_argument("--cpu-baseline-table", action="store_true",
                   help="the oracle's time per operation on every workload, one host core "
                        "(median of 3); no GPU")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.profile_op:
        run_profile_op(args)
    elif args.cpu_baseline_table:
        cpu_baseline_table(args)
    elif args.table or args.table_all or args.table_flagged:
        run_table(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)
    try:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass


if __name__ == "__main__":
    main()
