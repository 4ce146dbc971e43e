"""bench.py host logic on the CPU: the max-over-ranks reduction across two gloo
ranks, the algorithmic byte model, and the reference arm's JSON line."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    v = bench.allreduce_max(10.0 * (rank + 1))
    bench.barrier()
    q.put((rank, v))
    dist.destroy_process_group()


def test_allreduce_max_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 20.0), (1, 20.0)]


def test_allreduce_single_process_is_identity():
    assert bench.allreduce_max(3.5) == 3.5


def test_byte_model_dsv3_decode():
    T, H, k, E, R = 1024, 7168, 8, 256, 32
    assert bench.kernel_bytes("dispatch_bf16", T, H, k, E, R) == 2 * T * H * (1 + k) + 4 * T * k
    assert bench.kernel_bytes("combine", T, H, k, E, R) == 2 * T * H * (1 + k) + 8 * T * k
    # ~132 MB each; 19.5 us at 6787 GB/s
    assert abs(bench.kernel_bytes("combine", T, H, k, E, R) / 1e6 - 132.19) < 0.01
    fp8 = bench.kernel_bytes("dispatch_fp8", 8192, 7168, 8, 256, 32)
    assert fp8 == 2 * 8192 * 7168 + 4 * 65536 + 65536 * 7168 + 4 * 65536 * 56


def test_byte_model_backward_and_coalesced():
    T, H, k, E, R = 1024, 7168, 8, 256, 32
    N = T * k
    # dy is a k-row scatter of dout; dw reads the same k rows of y
    assert bench.kernel_bytes("combine_backward", T, H, k, E, R) == \
        2 * T * H + 2 * N * H + 2 * N * H + 12 * N
    # dx is the unit-weight combine: no weights read
    assert bench.kernel_bytes("dispatch_backward", T, H, k, E, R) == \
        bench.kernel_bytes("combine", T, H, k, E, R) - 4 * N
    assert bench.kernel_bytes("layout_dispatch", T, H, k, E, R) == \
        bench.kernel_bytes("layout_assign", T, H, k, E, R) + \
        bench.kernel_bytes("dispatch_bf16", T, H, k, E, R)
    Nc = 7464
    assert bench.coalesced_bytes("dispatch_coalesced", T, H, k, Nc) == 2 * T * H + 4 * N + 2 * Nc * H
    # with one row per slot, the coalesced combine moves the plain combine's
    # bytes plus the rows it pre-reduces and the coalesced row map
    assert bench.coalesced_bytes("combine_coalesced", T, H, k, N) == \
        bench.kernel_bytes("combine", T, H, k, E, R) + 2 * N * H + 4 * N


def test_reference_arm_prints_one_json_line():
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--config", "tiny", "--steps", "3", "--warmup", "3"])
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["higher_is_better"] is True


def test_warmup_below_three_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "2"])


def test_host_info_reports_core_count():
    h = bench.host_info()
    assert h["nproc"] == os.cpu_count() and h["nproc"] >= 1
    assert h["cpu"] is None or isinstance(h["cpu"], str)
