"""Parity of repeated calls made on a cold L2 cache: every call follows a write larger
than L2, and every call's output is checked against the fp64 oracle.

One warm call can hide a race between a CTA's one-time setup and its first tiles.
With L2 flushed, the first tiles and any setup that reads global memory both wait on
DRAM, and either may finish first. Such a race once gave wrong rows in the single
K=V kernel, and the status word stayed clean (covered in test_gpu_keqv.py). This file
runs the same check on the other entry points:
- the single-token kernel, both geometries, on contiguous and paged caches;
- the multi-query kernel, both geometries.
The batches are spread over every CTA, with ragged lengths and a sequence split into
dynamic chunks.
"""
import numpy as np
import pytest
import torch

import decode_attention_gb300 as gqa
import oracle
from decode_attention_gb300 import inputs
from tests.helpers import GLOBAL, SLIDING, assert_parity, cuda_case, oracle_contiguous, oracle_paged

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

GEOS = {"sliding": SLIDING, "global": GLOBAL}
LENS = [2914, 1371, 5003, 17, 4096, 640]
CALLS = 8


def cold_calls(call):
    """CALLS outputs of call(), each made after a 256 MB write (twice the L2 cache)."""
    flush = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(CALLS):
        flush.add_(1)
        outs.append(call())
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_cold_calls_contiguous(layer):
    geo = GEOS[layer]
    c = cuda_case(len(LENS), max(LENS), geo, LENS, seed=700)
    ref = oracle_contiguous(c, geo["window"])
    outs = cold_calls(lambda: gqa.gqa_decode(c["q"], c["k"], c["v"], c["seq_lens"], geo["window"],
                                             out_dtype=torch.float32))
    for k, out in enumerate(outs):
        for b in range(len(LENS)):
            assert_parity(out[b], ref[b], f"{layer} cold call {k} b={b} L={LENS[b]}")
    assert gqa.gqa_device_status() == 0


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_cold_calls_paged(layer):
    geo = GEOS[layer]
    c = inputs.paged_case(len(LENS), geo["H"], geo["KVH"], geo["D"], LENS, seed=701, device="cuda")
    ref = oracle_paged(c, geo["window"])
    outs = cold_calls(lambda: gqa.gqa_decode_paged(c["q"], c["k_pages"], c["v_pages"], c["block_table"],
                                                   c["seq_lens"], geo["window"],
                                                   out_dtype=torch.float32))
    for k, out in enumerate(outs):
        for b in range(len(LENS)):
            assert_parity(out[b], ref[b], f"{layer} paged cold call {k} b={b} L={LENS[b]}")
    assert gqa.gqa_device_status() == 0


@pytest.mark.parametrize("layer,T", [("sliding", 8), ("global", 4)])
def test_cold_calls_multi_query(layer, T):
    geo = GEOS[layer]
    c = inputs.mq_case(len(LENS), T, max(LENS), geo["H"], geo["KVH"], geo["D"], LENS, seed=702,
                       device="cuda")
    ref = oracle.gqa_decode_mq_f64(inputs.bf16_bits(c["q"]), inputs.bf16_bits(c["k"]),
                                   inputs.bf16_bits(c["v"]), np.asarray(LENS), geo["window"])
    outs = cold_calls(lambda: gqa.gqa_decode_mq(c["q"], c["k"], c["v"], c["seq_lens"], geo["window"],
                                                out_dtype=torch.float32))
    for k, out in enumerate(outs):
        for b in range(len(LENS)):
            for t in range(T):
                assert_parity(out[b, t], ref[b, t], f"{layer} T={T} cold call {k} b={b} t={t}")
    assert gqa.gqa_device_status() == 0
