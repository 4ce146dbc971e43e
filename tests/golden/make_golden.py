"""Writes tests/golden/tiny_oracle.json: the oracle's outputs on the seeded
`tiny` workload (T=128, H=256, top-2, E=8 over R=2 ranks), so that a change of
platform, compiler or oracle arithmetic shows up as a diff.

Calls only oracle/ and the input generators.  What each stored field computes:
  layout      UBEP section 2.3 (counts, offsets, contiguous per-expert reorder),
              StrataCL Appendix D (prefix-sum offsets, token-local offsets)
  dispatch    UBEP section 2.3 Phase 2 (each token to each chosen expert)
  quant       UBEP Table 3 (W8A8), with the 1x128 amax/448 reading
  combine     HyperParallel-MoE section 2.2 (weighted by routing scores)
  backward    HyperParallel-MoE section 2.2 / Figure 2(b) (backward Dispatch
              is the gradient of the forward Combine, and the reverse)
  coalesced   RailWave section 3.1 (token coalescing: one row per token and
              destination rank; the return path pre-reduced per rank)
Run:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from workloads.gen import expert_output, make_workload  # noqa: E402


def digest(a) -> str:
    return hashlib.sha256(a.tobytes()).hexdigest()


def compute():
    w = make_workload("tiny")
    counts, offs, roffs, slot_of, src_of = oracle.layout(w.topk_idx, w.E, w.R)
    recv = oracle.dispatch(w.x, slot_of)
    q, sc = oracle.dispatch_quant(w.x, slot_of)
    y = w.y()
    out_b = oracle.combine(y, slot_of, w.topk_w, "bf16")
    out_f = oracle.combine(y, slot_of, w.topk_w, "f32")
    dout = expert_output(w.T, w.H, seed=w.seed + 1)
    dy, dw, _ = oracle.combine_backward(dout, y, slot_of, w.topk_w)
    dx = oracle.dispatch_backward(y, slot_of)
    c_counts, c_offs, crow, src_c, expand = oracle.layout_coalesced(w.topk_idx, w.E, w.R,
                                                                    slot_of)
    nc = int(c_offs[-1])
    recv_c = oracle.dispatch_coalesced(w.x, crow, nc)
    part = oracle.combine_coalesced_pre(y, slot_of, w.topk_w, crow, nc)
    out_c = oracle.combine_coalesced_post(part, crow)
    return {
        "workload": "tiny seed 0 (T=128, H=256, k=2, E=8, R=2)",
        "inputs_sha256": {"x": digest(w.x), "topk_idx": digest(w.topk_idx),
                          "topk_w": digest(w.topk_w), "y": digest(y)},
        "expert_counts": counts.tolist(),
        "expert_offsets": offs.tolist(),
        "rank_offsets": roffs.tolist(),
        "slot_of_first16": slot_of.ravel()[:16].tolist(),
        "sha256": {"slot_of": digest(slot_of), "src_of": digest(src_of),
                   "recv_bf16": digest(recv), "recv_e4m3": digest(q),
                   "recv_scales": digest(sc), "combine_bf16": digest(out_b),
                   "combine_f32": digest(out_f), "dy": digest(dy),
                   "dw_f64": digest(dw), "dx": digest(dx), "crow": digest(crow),
                   "src_pair_c": digest(src_c), "expand": digest(expand),
                   "recv_coalesced": digest(recv_c), "partial": digest(part),
                   "combine_coalesced": digest(out_c)},
        "coalesced_rank_counts": c_counts.tolist(),
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(compute(), f, indent=1)
        f.write("\n")
