"""The timeout exit of the kernels, made to happen on purpose (GQA_TEST_STALL).

Every wait in the kernels gives up after a time limit, raises the status word's
GQA_DEVICE_WAIT_TIMEOUT bit and takes an exit in which every role leaves, the copies
(and, on the tcgen05 kernel, the tensor-core work) in flight are drained and TMEM is
released.  In the test mode GQA_TEST_STALL each CTA's producer, after issuing its
first tile, waits on a barrier that nothing completes; that wait gives up after 1 ms.
Nothing faults and nothing waits without a limit.

Each case makes one stalled call and checks that
  * it ends (well within the 2 s a wait would take to give up in normal use),
  * the status word reports GQA_DEVICE_WAIT_TIMEOUT,
and then, on the same workspace, that a normal call matches the fp64 oracle and
leaves the status word clear.  Covered: the split-KV kernel on contiguous and paged
caches (both geometries), the tcgen05 multi-query kernel (both geometries), both
kernels of the single K=V cache, and gqa_decode_noalloc's fixed scratch.
"""
import contextlib
import time

import numpy as np
import pytest
import torch

import decode_attention_gb300 as gqa
import oracle
from decode_attention_gb300 import inputs
from tests.helpers import (GLOBAL, SLIDING, assert_parity, keqv_tcgen05_capacity,
                           oracle_contiguous, oracle_paged)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

GEOS = {"sliding": SLIDING, "global": GLOBAL}


@contextlib.contextmanager
def mode(flags):
    prev = gqa.gqa_set_test_mode(flags)
    try:
        yield
    finally:
        gqa.gqa_set_test_mode(prev)


def stalled(call, read_status):
    """Run call() in the stall mode; return the status word it left."""
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with mode(gqa.GQA_TEST_STALL):
        call()
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    flags = read_status()
    assert elapsed < 1.0, f"the stalled call took {elapsed:.2f} s"
    assert flags & gqa.GQA_DEVICE_WAIT_TIMEOUT, f"status word {flags:#x}"
    return flags


def check_contiguous(case, window, out):
    for b, r in oracle_contiguous(case, window).items():
        assert_parity(out[b], r, f"b={b}")


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_split_kernel_contiguous(layer):
    geo = GEOS[layer]
    lens = [1, 700, 3000, 5000]
    case = inputs.contiguous_case(len(lens), 5000, geo["H"], geo["KVH"], geo["D"], lens, 900,
                                  device="cuda")
    ws = gqa.new_workspace(len(lens), 5000, geo["H"], geo["KVH"], geo["D"], geo["window"])
    out = torch.empty(len(lens), geo["H"], geo["D"], dtype=torch.float32, device="cuda")

    def call():
        gqa.gqa_decode(case["q"], case["k"], case["v"], case["seq_lens"], geo["window"], out=out,
                       workspace=ws)

    stalled(call, lambda: gqa.gqa_device_status(ws))
    out.fill_(float("nan"))
    call()
    torch.cuda.synchronize()
    check_contiguous(case, geo["window"], out)
    assert gqa.gqa_device_status(ws) == 0


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_split_kernel_paged(layer):
    geo = GEOS[layer]
    lens = [40, 1500, 4100]
    case = inputs.paged_case(len(lens), geo["H"], geo["KVH"], geo["D"], lens, 901, device="cuda")

    def call():
        return gqa.gqa_decode_paged(case["q"], case["k_pages"], case["v_pages"], case["block_table"],
                                    case["seq_lens"], geo["window"], out_dtype=torch.float32)

    stalled(call, gqa.gqa_device_status)   # the library-owned workspace
    out = call()
    torch.cuda.synchronize()
    ref = oracle_paged(case, geo["window"])
    for b in range(len(lens)):
        assert_parity(out[b], ref[b], f"b={b}")
    assert gqa.gqa_device_status() == 0


@pytest.mark.parametrize("layer,T", [("sliding", 8), ("global", 4), ("global", 2)])
def test_tcgen05_multi_query_kernel(layer, T):
    geo = GEOS[layer]
    lens = [T - 1, 300, 2000, 3000]
    case = inputs.mq_case(len(lens), T, 3000, geo["H"], geo["KVH"], geo["D"], lens, 902 + T,
                          device="cuda")
    ws = torch.empty(gqa.gqa_workspace_size_mq(len(lens), T, geo["H"], geo["KVH"], geo["D"]),
                     dtype=torch.uint8, device="cuda")
    gqa.gqa_workspace_init(ws)

    def call():
        return gqa.gqa_decode_mq(case["q"], case["k"], case["v"], case["seq_lens"], geo["window"],
                                 out_dtype=torch.float32, workspace=ws)

    stalled(call, lambda: gqa.gqa_device_status(ws))
    out = call()
    torch.cuda.synchronize()
    ref = oracle.gqa_decode_mq_f64(inputs.bf16_bits(case["q"]), inputs.bf16_bits(case["k"]),
                                   inputs.bf16_bits(case["v"]), np.asarray(lens), geo["window"])
    for b in range(len(lens)):
        for t in range(T):
            assert_parity(out[b, t], ref[b, t], f"b={b} t={t}")
    assert gqa.gqa_device_status(ws) == 0


@pytest.mark.parametrize("roomy", [False, True], ids=["split_kernel", "tcgen05_kernel"])
def test_keqv_kernels(roomy):
    H, KVH, D = GLOBAL["H"], GLOBAL["KVH"], GLOBAL["D"]
    lens = [1, 2500, 3000]
    want = gqa.GQA_KERNEL_TCGEN05 if roomy else gqa.GQA_KERNEL_SPLIT_DECODE
    S = keqv_tcgen05_capacity(len(lens), 3000) if roomy else 3000
    assert gqa.gqa_decode_keqv_kernel(len(lens), S) == want
    case = inputs.contiguous_case(len(lens), S, H, KVH, D, lens, 905, device="cuda")
    w_k = inputs.k_norm_weight_bf16(D, 906, device="cuda")

    def call():
        return gqa.gqa_decode_keqv(case["q"], case["v"], w_k, case["seq_lens"],
                                   out_dtype=torch.float32)

    stalled(call, gqa.gqa_device_status)
    out = call()
    torch.cuda.synchronize()
    v = case["v"][:, :max(lens)].contiguous()
    ref = oracle.gqa_decode_keqv_f64(inputs.bf16_bits(case["q"]), inputs.bf16_bits(v),
                                     inputs.bf16_bits(w_k), np.asarray(lens), 0)
    for b in range(len(lens)):
        assert_parity(out[b], ref[b], f"b={b}")
    assert gqa.gqa_device_status() == 0


def test_noalloc_fixed_scratch():
    geo = SLIDING
    lens = [900, 2000, 4096]
    case = inputs.contiguous_case(len(lens), 4096, geo["H"], geo["KVH"], geo["D"], lens, 907,
                                  device="cuda")
    out = torch.empty(len(lens), geo["H"], geo["D"], dtype=torch.float32, device="cuda")
    gqa.gqa_noalloc_status()   # start from a clear word

    def call():
        gqa.gqa_decode_noalloc(case["q"], case["k"], case["v"], case["seq_lens"], geo["window"], out)

    stalled(call, gqa.gqa_noalloc_status)
    out.fill_(float("nan"))
    call()
    torch.cuda.synchronize()
    check_contiguous(case, geo["window"], out)
    assert gqa.gqa_noalloc_status() == 0


def test_test_mode_is_restored():
    assert gqa.gqa_get_test_mode() == 0
