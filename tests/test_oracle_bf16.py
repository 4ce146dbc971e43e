"""Pin for the oracle's float32 -> bf16 rounding (nearest, ties to even)
against torch's bfloat16 cast, an independent implementation."""
import numpy as np
import torch

import oracle


def _torch_bf16(f):
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_random_and_special_values_match_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    ties = ((rng.integers(0, 1 << 16, size=4096, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 3.4028235e38, -3.4028235e38,
                        1e-45, -1e-45, 1.1754942e-38, 1.0, 1.00390625, 1.01171875],
                       np.float32)
    f = np.concatenate([f, ties[np.isfinite(ties)], special])
    assert np.array_equal(oracle.f32_to_bf16(f), _torch_bf16(f))


def test_nan_stays_nan():
    b = oracle.f32_to_bf16(np.array([np.nan], np.float32))[0]
    assert (b & 0x7F80) == 0x7F80 and (b & 0x007F) != 0
