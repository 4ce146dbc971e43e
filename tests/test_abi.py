"""The C ABI library loads without a GPU, exports every symbol include/moe_ep.h
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_ep.h")


@pytest.fixture(scope="module")
def m():
    import __graft_entry__
    __graft_entry__._cuda_build_module().build()
    import combine_layout_moe_gb300 as pkg
    return pkg


def declared():
    text = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)


def test_header_declares_entry_points():
    names = declared()
    for n in ("moe_layout", "moe_dispatch", "moe_dispatch_quant", "moe_combine",
              "moe_layout_workspace_bytes", "moe_read_error", "moe_status_string",
              "moe_abi_version"):
        assert n in names


def test_every_declared_symbol_is_exported(m):
    lib = ctypes.CDLL(m.LIB_PATH)
    for n in declared():
        assert hasattr(lib, n), n
        assert n in m.SIGNATURES, f"binding lacks {n}"


def test_status_strings_and_version(m):
    assert m.moe_abi_version() == 2
    assert m.moe_status_string(0) == "ok"
    assert "range" in m.moe_status_string(m.MOE_ERR_BAD_INDEX)
    assert m.moe_status_string(99) == "unknown status"


def test_workspace_bytes(m):
    assert m.moe_layout_workspace_bytes(1024, 8, 256) >= 256
    assert m.moe_layout_workspace_bytes(0, 8, 256) == 256      # the barrier counter only
    assert m.moe_layout_workspace_bytes(-1, 8, 256) == 0
    assert m.moe_layout_workspace_bytes(1 << 28, 8, 256) == 0      # T*k >= 2^31
    assert m.moe_layout_workspace_bytes(16, 2, 4096) == 0          # E above the maximum
    # barrier counter + tile table, capped at 128 tiles x E int32
    assert m.moe_layout_workspace_bytes(1 << 20, 8, 256) == 256 + 128 * 256 * 4


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced


@pytest.mark.parametrize("args", [
    (-1, 2, 8, 2),      # T < 0
    (4, 0, 8, 2),       # k < 1
    (4, 2, 6, 4),       # E % R
    (4, 2, 8, 0),       # R < 1
    (1 << 28, 8, 8, 2),  # T*k >= 2^31
])
def test_layout_rejects_bad_sizes(m, args):
    T, k, E, R = args
    st = m._lib.moe_layout(T, k, E, R, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None,
                           None)
    assert st == m.MOE_ERR_INVALID_ARG


def test_layout_rejects_small_workspace_and_misalignment(m):
    L = m._lib
    assert L.moe_layout(1024, 8, 256, 32, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, None,
                        None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_layout(4, 2, 8, 2, FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None,
                        None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_layout(4, 2, 8, 2, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None,
                        None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_layout(4, 2, 2048, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None,
                        None) == m.MOE_ERR_UNSUPPORTED


def test_payload_calls_reject_bad_shapes_and_alignment(m):
    L = m._lib
    bad = m.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch(4, 12, 2, FAKE, FAKE, FAKE, None, None) == bad          # H % 8
    assert L.moe_dispatch(4, 64, 2, FAKE + 8, FAKE, FAKE, None, None) == bad      # x align
    assert L.moe_dispatch(4, 64, 2, FAKE, FAKE, None, None, None) == bad          # null recv
    assert L.moe_dispatch_quant(4, 192, 2, FAKE, FAKE, FAKE, FAKE, None, None) == bad
    assert L.moe_dispatch_quant(4, 256, 2, FAKE, FAKE, FAKE, FAKE + 4, None, None) == bad
    assert L.moe_combine(4, 64, 2, FAKE, FAKE, FAKE, FAKE, 2, None, None) == bad  # dtype
    assert L.moe_combine(4, 64, 2, FAKE, FAKE, FAKE, FAKE + 8, 0, None, None) == bad
    assert L.moe_combine(4, 64, 0, FAKE, FAKE, FAKE, FAKE, 0, None, None) == bad
    assert L.moe_read_error(None, 1, None, None) == bad
    # flagged variant: (mode, granularity, epoch, spin limit) -> status
    def flagged(k, mode, G, epoch, spin):
        return L.moe_dispatch_combine_flagged(4, 64, k, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0,
                                              mode, G, FAKE, epoch, spin, -1, None, None)
    assert flagged(2, m.MOE_SYNC_WORD, 512, 0, 10) == bad               # epoch 0
    assert flagged(2, m.MOE_SYNC_WORD, 512, 1, 0) == bad                # no spin limit
    assert flagged(2, m.MOE_SYNC_WORD, 48, 1, 10) == bad                # 48 does not divide 512
    assert flagged(2, m.MOE_SYNC_WORD, 1000, 1, 10) == bad              # not a multiple of 512
    assert flagged(2, m.MOE_SYNC_BATCH, 256, 1, 10) == bad              # batches of whole blocks
    assert flagged(2, 4, 512, 1, 10) == bad                             # no such mode
    assert flagged(40, m.MOE_SYNC_WORD, 512, 1, 10) == m.MOE_ERR_UNSUPPORTED
    # words per mode: two hops x rows x blocks (BATCH: 64-bit words)
    T, H, k = 1024, 7168, 8
    assert m.moe_sync_words(T, H, k, m.MOE_SYNC_WORD, 2048) == 2 * T * k * 7
    assert m.moe_sync_words(T, H, k, m.MOE_SYNC_WORD, 32) == 2 * T * k * 448
    assert m.moe_sync_words(T, H, k, m.MOE_SYNC_BATCH, 4096) == 4 * T * k * 4
    assert m.moe_sync_words(T, H, k, m.MOE_SYNC_BARRIER, 512) == 2
    assert m.moe_sync_words(T, H, k, m.MOE_SYNC_SENTINEL, 512) == 0
    assert m.moe_sync_words(T, H, k, m.MOE_SYNC_WORD, 24) == 0
    # backward: k above 32, dw without y, bad output dtype
    assert L.moe_combine_backward(4, 64, 40, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                  None) == m.MOE_ERR_UNSUPPORTED
    assert L.moe_combine_backward(4, 64, 2, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, None) == bad
    assert L.moe_dispatch_backward(4, 64, 2, FAKE, FAKE, FAKE, 3, None, None) == bad


def test_coalesced_calls_reject_bad_arguments(m):
    L = m._lib
    bad = m.MOE_ERR_INVALID_ARG
    ws = 1 << 20
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, None, None)
    assert L.moe_layout_coalesced(4, 2, 6, 4, *args) == bad                 # E % R
    assert L.moe_layout_coalesced(4, 2, 2048, 2, *args) == m.MOE_ERR_UNSUPPORTED
    assert L.moe_layout_coalesced(4, 2, 8, 2, FAKE, None, *args[2:]) == bad  # null slot_of
    assert L.moe_layout_coalesced(4, 2, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE + 2, FAKE, FAKE,
                                  FAKE, ws, None, None) == bad              # crow alignment
    # the workspace is sized by the rank count: 128 tiles x R int32 at most
    need = m.moe_layout_workspace_bytes(1 << 20, 8, 32)
    assert L.moe_layout_coalesced(1 << 20, 8, 256, 32, *args[:8], need - 4, None,
                                  None) == bad
    assert L.moe_dispatch_coalesced(4, 12, 2, FAKE, FAKE, 8, FAKE, None, None) == bad  # H % 8
    assert L.moe_dispatch_coalesced(4, 64, 2, FAKE, FAKE, -1, FAKE, None, None) == bad
    assert L.moe_dispatch_coalesced(4, 64, 2, FAKE, FAKE, 8, FAKE + 8, None, None) == bad
    assert L.moe_dispatch_coalesced(4, 64, 40, FAKE, FAKE, 8, FAKE, None,
                                    None) == m.MOE_ERR_UNSUPPORTED
    # coalesced combine: bad dtype, k above 32, misaligned partial
    cargs = (FAKE, FAKE, FAKE, FAKE, 8)
    assert L.moe_combine_coalesced(4, 64, 2, *cargs, FAKE, FAKE, 2, None, None) == bad
    assert L.moe_combine_coalesced(4, 64, 40, *cargs, FAKE, FAKE, 0, None,
                                   None) == m.MOE_ERR_UNSUPPORTED
    assert L.moe_combine_coalesced(4, 64, 2, *cargs, FAKE + 8, FAKE, 0, None, None) == bad
    assert L.moe_combine_coalesced(4, 64, 2, FAKE, FAKE, FAKE, FAKE, -1, FAKE, FAKE, 0, None,
                                   None) == bad
    # coalesced FP8 dispatch: H % 128, k above 32
    assert L.moe_dispatch_quant_coalesced(4, 192, 2, FAKE, FAKE, 8, FAKE, FAKE, None, None) == bad
    assert L.moe_dispatch_quant_coalesced(4, 256, 40, FAKE, FAKE, 8, FAKE, FAKE, None,
                                          None) == m.MOE_ERR_UNSUPPORTED
