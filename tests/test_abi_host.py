"""C-ABI checks that need no GPU: the library builds, loads and exports every
function ``include/gqa_decode.h`` declares, and the host-side argument checks
return the documented status before anything touches the device."""
import ctypes
import os
import re

import pytest

import decode_attention_gb300 as gqa
from decode_attention_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_decode.h")

# Aligned addresses that are never dereferenced: every call below fails its host
# checks (or is an empty batch) before any CUDA call.
FAKE = 0x10000
SLIDING = (32, 16, 256)
GLOBAL = (32, 4, 512)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return gqa.load_library()


def test_header_declares_the_exported_api():
    assert declared_functions() == sorted(_native.EXPORTED_SYMBOLS)


def test_binding_constants_match_the_header():
    defines = dict(re.findall(r"#define (GQA_[A-Z_]+) (\d+)u?\b", open(HEADER).read()))
    for name, value in [("GQA_MAX_SEQ", gqa.GQA_MAX_SEQ), ("GQA_PAGE_SIZE", gqa.PAGE_SIZE),
                        ("GQA_MAX_QUERIES_SLIDING", gqa.GQA_MAX_QUERIES_SLIDING),
                        ("GQA_MAX_QUERIES_GLOBAL", gqa.GQA_MAX_QUERIES_GLOBAL),
                        ("GQA_DEVICE_WAIT_TIMEOUT", gqa.GQA_DEVICE_WAIT_TIMEOUT),
                        ("GQA_DEVICE_BAD_PAGE", gqa.GQA_DEVICE_BAD_PAGE),
                        ("GQA_DEVICE_BAD_LENGTH", gqa.GQA_DEVICE_BAD_LENGTH)]:
        assert int(defines[name]) == value, name


def test_binding_kernel_and_test_mode_codes_match_the_header():
    text = open(HEADER).read()
    kernels = dict(re.findall(r"(GQA_KERNEL_[A-Z_0-9]+) = (\d+)", text))
    assert {k: int(v) for k, v in kernels.items()} == {
        "GQA_KERNEL_NONE": gqa.GQA_KERNEL_NONE, "GQA_KERNEL_SPLIT_DECODE": gqa.GQA_KERNEL_SPLIT_DECODE,
        "GQA_KERNEL_TCGEN05": gqa.GQA_KERNEL_TCGEN05}
    defines = dict(re.findall(r"#define (GQA_TEST_[A-Z_]+) (\d+)u?\b", text))
    assert int(defines["GQA_TEST_SINGLE_PIECE"]) == gqa.GQA_TEST_SINGLE_PIECE
    assert int(defines["GQA_TEST_STALL"]) == gqa.GQA_TEST_STALL


def test_test_mode_round_trip(lib):
    assert gqa.gqa_get_test_mode() == 0
    assert gqa.gqa_set_test_mode(gqa.GQA_TEST_SINGLE_PIECE | 0x80) == 0
    assert gqa.gqa_get_test_mode() == gqa.GQA_TEST_SINGLE_PIECE   # unknown bits dropped
    assert gqa.gqa_set_test_mode(0) == gqa.GQA_TEST_SINGLE_PIECE
    assert gqa.gqa_get_test_mode() == 0


def test_keqv_kernel_query_refuses_bad_sizes(lib):
    # refused before the device is queried
    assert lib.gqa_decode_keqv_kernel(4, 1024, *SLIDING) == gqa.GQA_KERNEL_NONE
    assert lib.gqa_decode_keqv_kernel(0, 1024, *GLOBAL) == gqa.GQA_KERNEL_NONE
    assert lib.gqa_decode_keqv_kernel(4, 0, *GLOBAL) == gqa.GQA_KERNEL_NONE
    assert lib.gqa_decode_keqv_kernel(4, 262145, *GLOBAL) == gqa.GQA_KERNEL_NONE


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in [(0, "GQA_OK"), (1, "GQA_ERR_INVALID_ARGUMENT"), (2, "GQA_ERR_UNSUPPORTED"),
                       (3, "GQA_ERR_WORKSPACE"), (4, "GQA_ERR_CUDA")]:
        assert gqa.gqa_status_string(code) == name
    assert gqa.gqa_status_string(99) == "GQA_ERR_UNKNOWN"


def test_workspace_size(lib):
    s = gqa.gqa_workspace_size(64, 32768, *SLIDING, 1024)
    g = gqa.gqa_workspace_size(16, 131072, *GLOBAL, 0)
    assert s > 0 and g > 0 and s % 256 == 0 and g % 256 == 0
    # grows with the batch, independent of the sequence capacity
    assert gqa.gqa_workspace_size(65, 32768, *SLIDING, 1024) > s
    assert gqa.gqa_workspace_size(64, 10, *SLIDING, 1024) == s
    # outside the domain -> 0
    assert gqa.gqa_workspace_size(1, 100, 32, 8, 256, 0) == 0
    assert gqa.gqa_workspace_size(257, 100, *SLIDING, 0) == 0
    assert gqa.gqa_workspace_size(1, 0, *SLIDING, 0) == 0
    assert gqa.gqa_workspace_size(1, 262145, *SLIDING, 0) == 0
    assert gqa.gqa_workspace_size(1, 100, *SLIDING, -1) == 0


def call_decode(lib, B=2, S=64, geo=SLIDING, window=0, q=FAKE, k=FAKE, v=FAKE, lens=FAKE,
                out=FAKE, dtype=1, ws=None, ws_bytes=0):
    H, KVH, D = geo
    return lib.gqa_decode(q, k, v, lens, B, S, H, KVH, D, window, out, dtype, ws, ws_bytes, None)


def call_paged(lib, B=2, P=8, max_pages=4, page_size=16, geo=GLOBAL, window=0, q=FAKE, kp=FAKE,
               vp=FAKE, bt=FAKE, lens=FAKE, out=FAKE, dtype=0):
    H, KVH, D = geo
    return lib.gqa_decode_paged(q, kp, vp, bt, lens, B, P, max_pages, page_size, H, KVH, D, window,
                                out, dtype, None, 0, None)


def test_unsupported_geometry(lib):
    assert call_decode(lib, geo=(32, 8, 256)) == gqa.GQA_ERR_UNSUPPORTED
    assert call_decode(lib, geo=(16, 4, 512)) == gqa.GQA_ERR_UNSUPPORTED
    assert call_decode(lib, geo=(32, 4, 256)) == gqa.GQA_ERR_UNSUPPORTED
    assert call_paged(lib, geo=(32, 16, 512)) == gqa.GQA_ERR_UNSUPPORTED


def test_invalid_arguments(lib):
    E = gqa.GQA_ERR_INVALID_ARGUMENT
    assert call_decode(lib, q=None) == E
    assert call_decode(lib, k=None) == E
    assert call_decode(lib, v=None) == E
    assert call_decode(lib, lens=None) == E
    assert call_decode(lib, out=None) == E
    assert call_decode(lib, q=FAKE + 8) == E          # q not 16-byte aligned
    assert call_decode(lib, k=FAKE + 2) == E
    assert call_decode(lib, out=FAKE + 4) == E
    assert call_decode(lib, lens=FAKE + 2) == E       # int32 misaligned
    assert call_decode(lib, B=-1) == E
    assert call_decode(lib, B=257) == E
    assert call_decode(lib, S=0) == E
    assert call_decode(lib, S=262145) == E
    assert call_decode(lib, window=-5) == E
    assert call_decode(lib, dtype=7) == E


def test_invalid_paged_arguments(lib):
    E = gqa.GQA_ERR_INVALID_ARGUMENT
    assert call_paged(lib, page_size=32) == E
    assert call_paged(lib, P=0) == E
    assert call_paged(lib, max_pages=0) == E
    assert call_paged(lib, max_pages=16385) == E       # 16 * max_pages above the shape domain
    assert call_paged(lib, bt=None) == E
    assert call_paged(lib, kp=FAKE + 8) == E
    assert call_paged(lib, bt=FAKE + 2) == E


def test_empty_batch_is_a_no_op(lib):
    # B == 0: nothing to read or write, nothing enqueued (pointers are not examined)
    assert call_decode(lib, B=0, q=None, k=None, v=None, lens=None, out=None) == gqa.GQA_OK
    assert call_paged(lib, B=0, q=None, kp=None, vp=None, bt=None, lens=None, out=None) == gqa.GQA_OK


def test_other_entry_points_reject_null(lib):
    assert lib.gqa_workspace_init(None, 1024, None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert lib.gqa_device_status(None, None, None) == gqa.GQA_ERR_INVALID_ARGUMENT


def test_python_binding_validates_before_calling():
    import torch
    q = torch.zeros(2, 32, 256, dtype=torch.bfloat16)
    k = torch.zeros(2, 8, 16, 256, dtype=torch.bfloat16)
    lens = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError):     # CPU tensors are refused, no fallback
        gqa.gqa_decode(q, k, k, lens, 1024)


def test_check_inputs_host_lengths():
    # contiguous cache: lengths must lie in [0, capacity]
    assert gqa.gqa_check_inputs_host([0, 1, 64], capacity=64, window=0) == -1
    assert gqa.gqa_check_inputs_host([3, 65, 1], capacity=64, window=0) == 1
    assert gqa.gqa_check_inputs_host([-1], capacity=64, window=16) == 0
    assert gqa.gqa_check_inputs_host([], capacity=64, window=0) == -1


def test_check_inputs_host_pages_only_attended():
    # paged: only the pages covering [lo, L) must be valid; later entries (-1 in
    # inputs.page_table) and pages before a sliding window are not looked at
    P = 10
    bt = [[0, 1, 2, -1, -1],
          [-7, 9, 3, 4, -1]]          # page 0 of sequence 1 is bad but lies before its window
    assert gqa.gqa_check_inputs_host([40, 64], capacity=80, window=40, block_table=bt,
                                     num_pages=P) == -1
    # the same table with full history: sequence 1 attends page 0 -> bad
    assert gqa.gqa_check_inputs_host([40, 64], capacity=80, window=0, block_table=bt,
                                     num_pages=P) == 1
    # a page id equal to P is out of range
    assert gqa.gqa_check_inputs_host([17], capacity=80, window=0, block_table=[[0, P, 0, 0, 0]],
                                     num_pages=P) == 0
    # L = 48 covers pages 0..2 exactly; entry 3 = -1 is not attended
    assert gqa.gqa_check_inputs_host([48], capacity=80, window=0, block_table=[[5, 6, 7, -1, -1]],
                                     num_pages=P) == -1


def test_check_inputs_host_matches_generated_tables():
    import numpy as np
    from decode_attention_gb300 import inputs
    wl = inputs.WORKLOADS["paged_mixed_b256"]
    lens = wl.lengths(np.random.default_rng(wl.seed))
    table, P = inputs.page_table(lens, wl.seed, max_pages=(wl.S + 15) // 16)
    for window in (0, 1024):
        assert gqa.gqa_check_inputs_host(lens, wl.S, window, table, P) == -1
    # one attended page out of range is found
    bad = table.copy()
    b = int(np.argmax(lens))
    bad[b, (int(lens[b]) - 1) // 16] = P
    assert gqa.gqa_check_inputs_host(lens, wl.S, 0, bad, P) == b


def test_check_inputs_host_rejects_bad_sizes(lib):
    first = ctypes.c_int(5)
    assert lib.gqa_check_inputs_host(None, 2, 64, 0, None, 0, 0, ctypes.byref(first)) == \
        gqa.GQA_ERR_INVALID_ARGUMENT
    assert first.value == -1
    lens = (ctypes.c_int32 * 1)(4)
    assert lib.gqa_check_inputs_host(lens, 1, 0, 0, None, 0, 0, None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert lib.gqa_check_inputs_host(lens, 1, 64, -1, None, 0, 0, None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert lib.gqa_check_inputs_host(lens, 1, 64, 0, lens, 0, 3, None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert lib.gqa_check_inputs_host(lens, 1, 64, 0, None, 0, 0, None) == gqa.GQA_OK


def test_ring_argument_checks(lib):
    F = FAKE
    H, KVH, D = SLIDING
    st = gqa.GQA_ERR_INVALID_ARGUMENT
    # window must lie in [1, C]; C in [1, GQA_MAX_SEQ]
    assert lib.gqa_decode_ring(F, F, F, F, 2, 1024, H, KVH, D, 0, F, 1, None, 0, None) == st
    assert lib.gqa_decode_ring(F, F, F, F, 2, 1024, H, KVH, D, 1025, F, 1, None, 0, None) == st
    assert lib.gqa_decode_ring(F, F, F, F, 2, 0, H, KVH, D, 1, F, 1, None, 0, None) == st
    assert lib.gqa_decode_ring(F, F, F, F, 2, 262145, H, KVH, D, 1024, F, 1, None, 0, None) == st
    assert lib.gqa_decode_ring(F, None, F, F, 2, 1024, H, KVH, D, 1024, F, 1, None, 0, None) == st
    assert lib.gqa_decode_ring(F, F, F, F, 2, 1024, 32, 8, 256, 1024, F, 1, None, 0, None) == \
        gqa.GQA_ERR_UNSUPPORTED
    assert lib.gqa_decode_ring(None, None, None, None, 0, 1024, H, KVH, D, 1024, None, 1, None, 0,
                               None) == gqa.GQA_OK


def test_keqv_argument_checks(lib):
    F = FAKE
    H, KVH, D = GLOBAL
    # values = keys only on the global geometry
    assert lib.gqa_decode_keqv(F, F, F, F, 2, 64, *SLIDING, F, 1, None, 0, None) == \
        gqa.GQA_ERR_UNSUPPORTED
    assert lib.gqa_decode_keqv(F, F, None, F, 2, 64, H, KVH, D, F, 1, None, 0, None) == \
        gqa.GQA_ERR_INVALID_ARGUMENT
    assert lib.gqa_decode_keqv(F, F, F, F, 2, 0, H, KVH, D, F, 1, None, 0, None) == \
        gqa.GQA_ERR_INVALID_ARGUMENT
    assert lib.gqa_decode_keqv(None, None, None, None, 0, 64, H, KVH, D, None, 1, None, 0,
                               None) == gqa.GQA_OK
    assert lib.gqa_decode_keqv_paged(F, F, F, F, F, 2, 4, 4, 8, H, KVH, D, F, 1, None, 0, None) == \
        gqa.GQA_ERR_INVALID_ARGUMENT   # page size must be 16
    assert lib.gqa_decode_keqv_paged(F, F, F, F, F, 2, 4, 4, 16, *SLIDING, F, 1, None, 0, None) == \
        gqa.GQA_ERR_UNSUPPORTED


def test_prepare_argument_checks(lib):
    F = FAKE
    H, KVH, D = SLIDING
    bad = gqa.GQA_ERR_INVALID_ARGUMENT
    assert lib.gqa_prepare_decode(F, F, F, F, F, F, 2, 32, 8, 256, F, F, F, 64, 0, None) == \
        gqa.GQA_ERR_UNSUPPORTED
    # values = keys (v_raw NULL) exists on the global geometry only
    assert lib.gqa_prepare_decode(F, F, None, F, F, F, 2, H, KVH, D, F, F, F, 64, 0, None) == \
        gqa.GQA_ERR_UNSUPPORTED
    assert lib.gqa_prepare_decode(F, F, F, F, F, F, 2, H, KVH, D, F, F, F, 0, 0, None) == bad
    assert lib.gqa_prepare_decode(F, F, F, F, F, F, 2, H, KVH, D, F, F, F, 64, 2, None) == bad
    assert lib.gqa_prepare_decode(F, F, F, F, F, F, 2, H, KVH, D, F, None, F, 64, 0, None) == bad
    assert lib.gqa_prepare_decode(F + 2, F, F, F, F, F, 2, H, KVH, D, F, F, F, 64, 0, None) == bad
    assert lib.gqa_prepare_decode(None, None, None, None, None, None, 0, H, KVH, D, None, None,
                                  None, 64, 0, None) == gqa.GQA_OK
    assert lib.gqa_prepare_decode_paged(F, F, F, F, F, F, F, 2, 4, 4, 8, H, KVH, D, F, F, F,
                                        None) == bad
