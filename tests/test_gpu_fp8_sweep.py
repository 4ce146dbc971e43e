"""The quantised dispatch's channel encoding on every fp32 input.

moe_dispatch_quant scales each channel by 448 / amax in fp32 and encodes the
product to E4M3 (nearest-even, saturating): the products reach fp32 values
anywhere near the format's rounding midpoints, not only bf16 ones.  Through
moe_e4m3_encode_bits (the same device routine) every fp32 bit pattern that is
not a NaN -- zeros, subnormals, normals, infinities, both signs: 2^32 - 2^24 +
2 patterns -- is encoded on the GPU and compared with the oracle's encoder,
written from the OCP FP8 E4M3 definition (bias 7, no infinities, largest
finite 448, subnormal step 2^-9, ties to even).  The oracle side runs in a
pool of spawned host processes."""
import multiprocessing as mp

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28          # patterns per GPU launch
SLICE = 1 << 24          # patterns per host task


def _oracle_slice(first: int) -> np.ndarray:
    import oracle
    u = (np.arange(SLICE, dtype=np.uint64) + np.uint64(first)).astype(np.uint32)
    return oracle.e4m3_encode(u.view(np.float32))


def test_every_fp32_pattern_encodes_as_the_oracle():
    import combine_layout_moe_gb300 as m
    ctx = mp.get_context("spawn")
    codes = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    with ctx.Pool(processes=min(16, max(2, mp.cpu_count()))) as pool:
        for c in range((1 << 32) // CHUNK):
            first = c * CHUNK
            pending = pool.map_async(_oracle_slice, range(first, first + CHUNK, SLICE))
            m.moe_e4m3_encode_bits(first, CHUNK, out=codes)
            got = codes.cpu().numpy()
            want = np.concatenate(pending.get(timeout=600))
            u = (np.arange(CHUNK, dtype=np.uint64) + np.uint64(first)).astype(np.uint32)
            nan = ((u & 0x7F800000) == 0x7F800000) & ((u & 0x007FFFFF) != 0)
            bad = np.flatnonzero((got != want) & ~nan)
            assert bad.size == 0, (f"{bad.size} patterns differ, first {u[bad[:4]]}: "
                                   f"{got[bad[:4]]} vs {want[bad[:4]]}")
            # NaNs stay NaNs (code 0x7F or 0xFF)
            assert np.all((got[nan] & 0x7F) == 0x7F)
