"""The oracle's pins have teeth: each plausible mistake, planted in a temporary
copy of the oracle's C source on the CPU, makes at least one pin fail."""
import os

import numpy as np
import pytest

import oracle
import test_oracle_combine as tc
import test_oracle_dispatch as td
import test_oracle_layout as tl
import test_oracle_bf16 as tb
import test_oracle_backward as tbw
import test_oracle_coalesced as tco
import test_oracle_ep as tep

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "moe_oracle.c")

MUTANTS = {
    # layout: walk the k slots backwards (unstable inside a token)
    "slot_order": ("for (int j = 0; j < k; ++j) {\n            int64_t i = (int64_t)t * k + j;\n            int e = topk_idx[i];\n            int32_t s = cursor[e]++;",
                   "for (int j = k - 1; j >= 0; --j) {\n            int64_t i = (int64_t)t * k + j;\n            int e = topk_idx[i];\n            int32_t s = cursor[e]++;"),
    # layout: rank offsets indexed by rank instead of first expert of the rank
    "rank_index": ("rank_offsets[r] = expert_offsets[r * El];", "rank_offsets[r] = expert_offsets[r];"),
    # layout: each expert starts at the previous expert's offset (scan shifted by one)
    "shifted_scan": ("cursor[e] = expert_offsets[e];", "cursor[e] = e > 0 ? expert_offsets[e - 1] : 0;"),
    # e4m3: ties away from zero
    "e4m3_ties": ("double r = nearbyint(frac8);", "double r = round(frac8);"),
    # e4m3: exponent bias 8
    "e4m3_bias": ("code = ((uint32_t)(ee + 7) << 3) | (uint32_t)r;", "code = ((uint32_t)(ee + 8) << 3) | (uint32_t)r;"),
    # quant: scale divisor off (E5M2's max instead of E4M3's)
    "quant_scale": ("srow[b] = amax / 448.0f;", "srow[b] = amax / 57344.0f;"),
    # combine: the slot index dropped (always slot 0 of the token)
    "combine_index": ("float v = bf16_to_f32(y[(int64_t)slot_of[i] * H + h]);",
                      "float v = bf16_to_f32(y[(int64_t)slot_of[(int64_t)t * k] * H + h]);"),
    # combine: weight and value of neighbouring slots swapped
    "combine_weight": ("acc = fmaf(topk_w[i], v, acc);", "acc = fmaf(topk_w[(int64_t)t * k + (j + 1) % k], v, acc);"),
    # combine: product rounded before the add (two roundings per slot, not one)
    "combine_unfused": ("acc = fmaf(topk_w[i], v, acc);", "acc = acc + topk_w[i] * v;"),
    # backward: dy scaled by the weight of the wrong slot
    "dy_weight": ("const float w = topk_w[i];\n            double acc = 0.0, mag = 0.0;",
                  "const float w = topk_w[(int64_t)t * k];\n            double acc = 0.0, mag = 0.0;"),
    # backward: dx skips the last slot
    "dx_drop": ("            for (int j = 0; j < k; ++j)\n                acc = acc + bf16_to_f32(",
                "            for (int j = 0; j + 1 < k; ++j)\n                acc = acc + bf16_to_f32("),
    # coalesced: tokens coalesced per expert instead of per rank
    "coalesced_key": ("            for (int jj = j - 1; jj >= 0; --jj)\n                if (topk_idx[(int64_t)t * k + jj] / El == r)\n                    owner_j = jj;",
                      "            for (int jj = j - 1; jj >= 0; --jj)\n                if (topk_idx[(int64_t)t * k + jj] == topk_idx[i])\n                    owner_j = jj;"),
    # coalesced combine: each rank returns only its first slot's contribution
    "pre_first_only": ("for (int jj = j; jj < k; ++jj) {", "for (int jj = j; jj < j + 1; ++jj) {"),
    # coalesced combine: the token adds its row once per slot, not once per row
    "post_duplicates": ("if (first)\n                    acc = acc + bf16_to_f32(partial",
                        "if (1)\n                    acc = acc + bf16_to_f32(partial"),
    # expert parallelism: a receiver takes its sources in reverse order
    "ep_source_order": ("            for (int s = 0; s < W; ++s) {\n                int32_t cnt = 0;",
                        "            for (int s = W - 1; s >= 0; --s) {\n                int32_t cnt = 0;"),
    # expert parallelism: counts filed [source][receiver] instead of [receiver][source]
    "ep_counts_index": ("recv_counts[((int64_t)d * W + s) * El + el] = cnt;",
                        "recv_counts[((int64_t)s * W + d) * El + el] = cnt;"),
    # expert parallelism: the return path sums a token's slots in reverse order
    "ep_combine_order": ("            for (int j = 0; j < k; ++j) {\n                const int64_t i = t * k + j;\n                acc = fmaf(topk_w[i], bf16_to_f32(y[row_of[i] * H + h]), acc);",
                         "            for (int j = k - 1; j >= 0; --j) {\n                const int64_t i = t * k + j;\n                acc = fmaf(topk_w[i], bf16_to_f32(y[row_of[i] * H + h]), acc);"),
    # bf16: ties rounded up instead of to even
    "bf16_ties": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))", "if (lower >= 0x8000u)"),
}


def _pins():
    lay = tl.CASES
    pins = []
    for c in lay[:8]:
        pins += [lambda c=c: tl.test_counts_and_offsets_match_library(*c),
                 lambda c=c: tl.test_slot_map_is_stable_counting_sort(*c),
                 lambda c=c: tl.test_rank_segments_hold_their_experts(*c)]
    pins += [tl.test_hand_worked_example, tl.test_duplicate_expert_in_one_token,
             td.test_e4m3_every_code_round_trips, td.test_e4m3_midpoints_and_neighbours_match_torch,
             td.test_quant_zero_and_tiny_blocks, td.test_dispatch_hand_worked,
             lambda: td.test_quant_block_invariants(("fuzz", 0)),
             lambda: td.test_dispatch_rows_equal_source_token(("fuzz", 0)),
             tc.test_one_hot_weights_select_one_slot, tc.test_weights_are_not_renormalised,
             tc.test_each_slot_is_one_fused_multiply_add,
             lambda: tc.test_bf16_output_is_rounded_fp32_output("fuzz0", None),
             tb.test_random_and_special_values_match_torch,
             lambda: tbw.test_combine_backward_matches_autograd(tbw.CASES[1]),
             lambda: tbw.test_dispatch_backward_is_unit_weight_combine(tbw.CASES[1]),
             tco.test_coalesced_hand_worked,
             lambda: tco.test_coalesced_layout_matches_brute_force(*tco.CASES[7]),
             lambda: tco.test_coalesced_combine_integer_payload_is_exact(1, 64, 8, 32, 4),
             lambda: tco.test_coalesced_combine_on_one_rank_is_plain_combine(40, 8, 16),
             lambda: tep.test_receive_buffers_are_the_stable_order_of_all_tokens(tep.CASES[2]),
             lambda: tep.test_counts_are_per_source_bincounts(tep.CASES[1]),
             tep.test_hand_worked_two_ranks, tep.test_combine_accumulates_in_slot_order]
    return pins


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    oracle.compile_to(str(path), so)
    monkeypatch.setattr(oracle, "_lib", oracle._bind(so))
    failed = 0
    for pin in _pins():
        try:
            pin()
        except (AssertionError, oracle.OracleError, IndexError, ValueError):
            failed += 1
    assert failed > 0, f"no pin caught mutation {name}"


def test_unmutated_oracle_passes_all_pins():
    for pin in _pins():
        pin()
