"""gqa_decode_noalloc: the decode call for callers that cannot allocate device
memory (for example a plugin layer handed only one operator's tensors, or a
runtime whose device memory all belongs to a fixed pool).  It runs on the
library's fixed device scratch array instead of a workspace.

The GPU tests call it through the C ABI (ctypes binding) twice in a row and
compare each result with gqa_decode's on the same inputs, within the parity
tolerance the other tests use, and once with the fp64 oracle.  They also check that
a call changes neither the device's free memory nor torch's allocator, and that the
fixed scratch's status word reports a clamped length.  This file is collected last,
and it needs no state from the other tests (it passes alone in a fresh process too).
"""
import numpy as np
import pytest
import torch

import decode_attention_gb300 as gqa
from decode_attention_gb300 import inputs
from tests.helpers import TOL_MAX_ABS, TOL_REL_L2, assert_parity, oracle_contiguous

needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def close(a: torch.Tensor, b: torch.Tensor):
    a64 = a.double().cpu().numpy()
    b64 = b.double().cpu().numpy()
    max_abs = float(np.abs(a64 - b64).max())
    denom = float(np.linalg.norm(b64)) or 1.0
    rel = float(np.linalg.norm(a64 - b64)) / denom
    assert max_abs <= TOL_MAX_ABS, max_abs
    assert rel <= TOL_REL_L2, rel


def test_argument_checks_need_no_gpu():
    lib = gqa.load_library()
    F = 0x10000
    # unsupported geometry, bad sizes and null pointers are refused before any CUDA call
    assert lib.gqa_decode_noalloc(F, F, F, F, 2, 64, 32, 8, 256, 0, F, 1, None) == gqa.GQA_ERR_UNSUPPORTED
    assert lib.gqa_decode_noalloc(F, F, F, F, 2, 0, 32, 16, 256, 0, F, 1, None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert lib.gqa_decode_noalloc(None, F, F, F, 2, 64, 32, 16, 256, 0, F, 1, None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert lib.gqa_decode_noalloc(None, None, None, None, 0, 64, 32, 16, 256, 0, None, 1, None) == gqa.GQA_OK


@pytest.mark.gpu
@needs_gpu
@pytest.mark.parametrize("layer,lens", [
    ("sliding", [0, 1, 17, 1024, 1025, 2500, 3000, 64]),
    ("global", [1, 33, 700, 4097, 0, 5000]),
])
def test_matches_gqa_decode_on_two_calls(layer, lens):
    geo = inputs.geometry(layer)
    S = max(lens)
    case = inputs.contiguous_case(len(lens), S, geo["H"], geo["KVH"], geo["D"], lens, seed=77,
                                  device="cuda")
    ref = gqa.gqa_decode(case["q"], case["k"], case["v"], case["seq_lens"], geo["window"],
                         out_dtype=torch.float32)
    outs = []
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        gqa.gqa_decode_noalloc(case["q"], case["k"], case["v"], case["seq_lens"], geo["window"], out)
        torch.cuda.synchronize()
        close(out, ref)
        outs.append(out)
    close(outs[1], outs[0])
    # the fp64 oracle, independently of gqa_decode (the two share their kernels)
    for b, r in oracle_contiguous(case, geo["window"]).items():
        assert_parity(outs[1][b], r, f"{layer} b={b} L={lens[b]}")
    # bf16 output through the same scratch: the round-to-nearest-even of the fp32
    # result (bf16 cannot meet the fp32 max-abs gate at |o| ~ 4)
    out16 = torch.empty(ref.shape, dtype=torch.bfloat16, device="cuda")
    gqa.gqa_decode_noalloc(case["q"], case["k"], case["v"], case["seq_lens"], geo["window"], out16)
    torch.cuda.synchronize()
    assert torch.equal(out16, outs[0].to(torch.bfloat16))


@pytest.mark.gpu
@needs_gpu
def test_rejects_calls_larger_than_the_scratch():
    # decodeGQA with B = 256 needs more than GQA_NOALLOC_SCRATCH_BYTES on any GPU
    geo = inputs.geometry("global")
    B, S = 256, 16
    q = torch.zeros(B, geo["H"], geo["D"], dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(B, S, geo["KVH"], geo["D"], dtype=torch.bfloat16, device="cuda")
    lens = torch.full((B,), S, dtype=torch.int32, device="cuda")
    out = torch.empty(B, geo["H"], geo["D"], dtype=torch.float32, device="cuda")
    with pytest.raises(gqa.GQAError) as e:
        gqa.gqa_decode_noalloc(q, k, k, lens, 0, out)
    assert e.value.status == gqa.GQA_ERR_WORKSPACE


@pytest.mark.gpu
@needs_gpu
def test_decode_global_with_fewer_dynamic_slots():
    # decodeGQA with B = 64 fits the scratch with only part of the dynamic-chunk
    # slots gqa_decode has (about 610 of 912 on 152 SMs): the kernel sizes its
    # chunks to that bound, and the result must not change beyond rounding
    geo = inputs.geometry("global")
    B, S = 64, 8192
    lens = np.random.default_rng(5).integers(6000, S + 1, B).tolist()
    case = inputs.contiguous_case(B, S, geo["H"], geo["KVH"], geo["D"], lens, seed=78, device="cuda")
    ref = gqa.gqa_decode(case["q"], case["k"], case["v"], case["seq_lens"], 0, out_dtype=torch.float32)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        gqa.gqa_decode_noalloc(case["q"], case["k"], case["v"], case["seq_lens"], 0, out)
        torch.cuda.synchronize()
        close(out, ref)


@pytest.mark.gpu
@needs_gpu
def test_larger_call_after_a_smaller_one():
    # The scratch layout depends on the call's shape.  A small call leaves its
    # split-softmax partials and partial lists in the scratch where a larger call
    # puts other things; the larger call rewrites every partial list and slot it
    # reads, so the leftovers must not change its result.
    geo = inputs.geometry("global")
    small = [3000, 4097, 5000]
    c1 = inputs.contiguous_case(len(small), max(small), geo["H"], geo["KVH"], geo["D"], small,
                                seed=79, device="cuda")
    out1 = torch.empty(len(small), geo["H"], geo["D"], dtype=torch.float32, device="cuda")
    gqa.gqa_decode_noalloc(c1["q"], c1["k"], c1["v"], c1["seq_lens"], 0, out1)
    B, S = 48, 4096
    lens = np.random.default_rng(6).integers(1, S + 1, B).tolist()
    c2 = inputs.contiguous_case(B, S, geo["H"], geo["KVH"], geo["D"], lens, seed=80, device="cuda")
    ref = gqa.gqa_decode(c2["q"], c2["k"], c2["v"], c2["seq_lens"], 0, out_dtype=torch.float32)
    out = torch.full_like(ref, float("nan"))
    gqa.gqa_decode_noalloc(c2["q"], c2["k"], c2["v"], c2["seq_lens"], 0, out)
    torch.cuda.synchronize()
    close(out, ref)


@pytest.mark.gpu
@needs_gpu
def test_a_call_allocates_no_device_memory():
    geo = inputs.geometry("global")
    lens = [3000, 8192, 17]
    case = inputs.contiguous_case(len(lens), 8192, geo["H"], geo["KVH"], geo["D"], lens, seed=81,
                                  device="cuda")
    out = torch.empty(len(lens), geo["H"], geo["D"], dtype=torch.float32, device="cuda")
    # the first call loads the kernels (module loading may take device memory)
    gqa.gqa_decode_noalloc(case["q"], case["k"], case["v"], case["seq_lens"], 0, out)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for _ in range(3):
        gqa.gqa_decode_noalloc(case["q"], case["k"], case["v"], case["seq_lens"], 0, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
    for key in ("allocation.all.allocated", "segment.all.allocated"):
        assert stats1.get(key, 0) == stats0.get(key, 0), key


@pytest.mark.gpu
@needs_gpu
def test_status_word_reports_a_clamped_length():
    geo = inputs.geometry("sliding")
    B, S = 2, 1024
    case = inputs.contiguous_case(B, S, geo["H"], geo["KVH"], geo["D"], [S, S], seed=82, device="cuda")
    out = torch.empty(B, geo["H"], geo["D"], dtype=torch.float32, device="cuda")
    gqa.gqa_noalloc_status()   # start from a clear word
    gqa.gqa_decode_noalloc(case["q"], case["k"], case["v"], case["seq_lens"], geo["window"], out)
    assert gqa.gqa_noalloc_status() == 0
    bad = torch.tensor([S + 5, S], dtype=torch.int32, device="cuda")   # above the capacity
    gqa.gqa_decode_noalloc(case["q"], case["k"], case["v"], bad, geo["window"], out)
    assert gqa.gqa_noalloc_status() == gqa.GQA_DEVICE_BAD_LENGTH
    # the read cleared the word; the clamped call equals the call at the capacity
    ref = out.clone()
    gqa.gqa_decode_noalloc(case["q"], case["k"], case["v"], case["seq_lens"], geo["window"], out)
    assert gqa.gqa_noalloc_status() == 0
    assert torch.equal(out, ref)
