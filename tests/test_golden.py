"""The oracle reproduces its stored outputs on the seeded tiny workload
(tests/golden/tiny_oracle.json, written by tests/golden/make_golden.py), and
the stored layout agrees with numpy's bincount/cumsum of the stored inputs."""
import json
import os

import numpy as np

from workloads.gen import make_workload

HERE = os.path.dirname(os.path.abspath(__file__))


def _load():
    with open(os.path.join(HERE, "golden", "tiny_oracle.json")) as f:
        return json.load(f)


def test_oracle_reproduces_golden():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "make_golden", os.path.join(HERE, "golden", "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    assert mod.compute() == _load()


def test_golden_layout_consistent_with_library():
    g = _load()
    w = make_workload("tiny")
    c = np.bincount(w.topk_idx.ravel(), minlength=w.E)
    assert g["expert_counts"] == c.tolist()
    assert g["expert_offsets"] == [0] + np.cumsum(c).tolist()
    assert g["rank_offsets"] == g["expert_offsets"][:: w.E // w.R]
