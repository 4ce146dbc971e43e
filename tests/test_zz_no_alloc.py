"""moe_layout_noalloc, the layout entry point for callers that cannot allocate
device memory (for example code given fixed buffers by a framework that owns
all allocation).  It must produce exactly what moe_layout produces, call after
call, although every call reuses the same fixed scratch array in the library.
Collected last on purpose: it runs after every other test in a full run."""
import ctypes

import numpy as np
import pytest
import torch

from workloads.gen import make_workload, random_case

pytestmark = pytest.mark.gpu


def _empty_layout(m, T, k, E, R):
    dev = "cuda"
    return m.Layout(torch.full((E,), -5, dtype=torch.int32, device=dev),
                    torch.full((E + 1,), -5, dtype=torch.int32, device=dev),
                    torch.full((R + 1,), -5, dtype=torch.int32, device=dev),
                    torch.full((T, k), -5, dtype=torch.int32, device=dev),
                    torch.full((T * k,), -5, dtype=torch.int32, device=dev))


def _noalloc_via_abi(m, idx, E, R, out, err):
    T, k = idx.shape
    st = m._lib.moe_layout_noalloc(T, k, E, R, idx.data_ptr(), out.expert_counts.data_ptr(),
                                   out.expert_offsets.data_ptr(), out.rank_offsets.data_ptr(),
                                   out.slot_of.data_ptr(), out.src_of.data_ptr(),
                                   err.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == m.MOE_OK, m.moe_status_string(st)


def test_noalloc_layout_matches_moe_layout_on_consecutive_calls():
    import combine_layout_moe_gb300 as m
    import oracle
    # the grid-barrier form (which uses the fixed array), clusters of 8 and 16
    # CTAs (which do not), then the grid-barrier form again
    cases = [(make_workload("glm45_air"), m.MOE_LAYOUT_FORM_COOPERATIVE),
             (make_workload("dsv3_decode"), m.MOE_LAYOUT_FORM_CLUSTER),
             (random_case(78, 2048, 8, 8, 256, 32), m.MOE_LAYOUT_FORM_CLUSTER),
             (random_case(77, 3000, 8, 6, 40, 8), m.MOE_LAYOUT_FORM_COOPERATIVE)]
    err = m.new_error_word()
    for w, form in cases:                             # two and more calls in a row
        idx = torch.from_numpy(w.topk_idx).cuda()
        ref = m.moe_layout(idx, w.E, w.R)
        got = _empty_layout(m, w.T, w.k, w.E, w.R)
        _noalloc_via_abi(m, idx, w.E, w.R, got, err)
        assert m.moe_layout_last_form() == form
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
        # and against the oracle directly: counts, offsets, rank offsets,
        # slot map and its inverse
        for a, b in zip(got, oracle.layout(w.topk_idx, w.E, w.R)):
            assert np.array_equal(a.cpu().numpy().reshape(b.shape), b)
    assert m.moe_read_error(err) == 0


def test_noalloc_layout_repeated_same_input_and_python_binding():
    import combine_layout_moe_gb300 as m
    w = make_workload("mixtral")
    idx = torch.from_numpy(w.topk_idx).cuda()
    ref = m.moe_layout(idx, w.E, w.R)
    import oracle
    want = oracle.layout(w.topk_idx, w.E, w.R)
    for _ in range(2):
        got = m.moe_layout_noalloc(idx, w.E, w.R, out=_empty_layout(m, w.T, w.k, w.E, w.R))
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(got, ref))
        assert all(np.array_equal(a.cpu().numpy().reshape(b.shape), b) for a, b in zip(got, want))


def test_noalloc_rejects_tables_beyond_the_fixed_scratch():
    import combine_layout_moe_gb300 as m
    assert m.moe_layout_workspace_bytes(600000, 8, 1024) > 256 * 1024
    idx = torch.zeros((600000, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(m.MoeError) as ei:
        m.moe_layout_noalloc(idx, 1024, 8, out=_empty_layout(m, 600000, 8, 1024, 8))
    assert ei.value.status == m.MOE_ERR_UNSUPPORTED
