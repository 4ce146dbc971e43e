"""The synthetic workloads have the shapes and routing structure they stand in for."""
import numpy as np
import pytest

from workloads.gen import CONFIGS, CONFIG_ORDER, make_workload, random_case, expert_output


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_shapes_types_and_weights(name):
    w = make_workload(name)
    c = CONFIGS[name]
    assert (w.T, w.H, w.k, w.E, w.R) == (c["T"], c["H"], c["k"], c["E"], c["R"])
    assert w.topk_idx.dtype == np.int32 and w.topk_idx.shape == (w.T, w.k)
    assert w.topk_w.dtype == np.float32 and w.topk_w.shape == (w.T, w.k)
    assert w.topk_idx.min() >= 0 and w.topk_idx.max() < w.E
    # top-k without replacement: distinct experts per token
    s = np.sort(w.topk_idx, axis=1)
    assert np.all(s[:, 1:] != s[:, :-1])
    assert np.all(w.topk_w > 0)
    assert np.abs(w.topk_w.astype(np.float64).sum(1) - 1).max() < 8 * 2.0 ** -24 * w.k


def test_deterministic():
    a = make_workload("glm45_air", T=512)
    b = make_workload("glm45_air", T=512)
    assert np.array_equal(a.topk_idx, b.topk_idx) and np.array_equal(a.topk_w, b.topk_w)
    assert np.array_equal(a.x, b.x)
    c = make_workload("glm45_air", seed=1, T=512)
    assert not np.array_equal(a.topk_idx, c.topk_idx)


def test_group_limited_routing():
    w = make_workload("glm45_air")
    groups = w.topk_idx // (w.E // CONFIGS["glm45_air"]["groups"])
    per_tok = np.array([len(set(r)) for r in groups])
    assert per_tok.max() <= CONFIGS["glm45_air"]["topk_groups"]


def test_skews():
    m = make_workload("mixtral")
    frac = np.bincount(m.topk_idx.ravel(), minlength=8)[0] / m.topk_idx.size
    assert 0.35 < frac < 0.5                         # one hot expert, ~40% of slots
    d = make_workload("dsv3_decode")
    c = np.bincount(d.topk_idx.ravel(), minlength=256)
    assert c.max() / c.mean() < 2.0                  # near-uniform decode routing
    p = make_workload("dsv3_prefill")
    c = np.bincount(p.topk_idx.ravel(), minlength=256)
    assert c.max() / c.mean() > 10                   # Zipf-skewed prefill


def test_hidden_states_are_bf16_normal():
    w = make_workload("dsv3_decode", T=64)
    f = (w.x.astype(np.uint32) << 16).view(np.float32)
    assert abs(f.mean()) < 0.02 and abs(f.std() - 1) < 0.02


def test_expert_output_and_fuzz():
    y = expert_output(64, 32, seed=1)
    f = (y.astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.isfinite(f)) and np.all(np.abs(f) >= 2.0 ** -7) and np.all(np.abs(f) < 8)
    r = random_case(0, 10, 16, 4, 3, 1)
    assert r.topk_idx.max() < 3 and r.x.shape == (10, 16)
