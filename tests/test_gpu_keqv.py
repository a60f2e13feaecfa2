"""GPU parity of the single K=V global cache (gqa_decode_keqv / _paged) against the
fp64 oracle, which derives every key as rope(w_k * v, s) in double precision.

Covers ragged lengths that span many 32-position tiles and several CTAs per
segment, a sequence reaching position 131074 (where the rotation angle of the
fastest pair is ~1.3e5 rad, so the kernel's fp64 angle reduction matters), the
paged form, NaN in every cache row past the sequence end, and the bf16 output.

The library runs a K=V call on one of two kernels, chosen by the cache capacity
(tiles of 128 positions per CTA): the mma.sync streaming kernel for small caches,
the tcgen05 kernel for large ones.  Every test runs twice with the same lengths: in
a cache sized to them ("tight") and in one large enough for the tcgen05 kernel
("roomy").
"""
import numpy as np
import pytest
import torch

import decode_attention_gb300 as gqa
import oracle
from decode_attention_gb300 import inputs
from tests.helpers import BF16_NAN, GLOBAL, assert_parity, keqv_tcgen05_capacity

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

H, KVH, D = GLOBAL["H"], GLOBAL["KVH"], GLOBAL["D"]


def capacity(B, S, roomy):
    """S (the library runs the split-KV kernel there), or a roomy capacity: the
    smallest one at or above S that the library routes to the tcgen05 kernel."""
    if not roomy:
        assert gqa.gqa_decode_keqv_kernel(B, S) == gqa.GQA_KERNEL_SPLIT_DECODE
        return S
    return keqv_tcgen05_capacity(B, S)


def case(lens, S, seed):
    c = inputs.contiguous_case(len(lens), S, H, KVH, D, lens, seed, device="cuda")
    c["w_k"] = inputs.k_norm_weight_bf16(D, inputs.tensor_seed(seed, "w_k"), device="cuda")
    return c


def oracle_keqv(c, lens):
    # the oracle reads rows below each length only: pass the rows up to the longest
    v = c["v"][:, :max(1, max(lens))].contiguous()
    return oracle.gqa_decode_keqv_f64(inputs.bf16_bits(c["q"]), inputs.bf16_bits(v),
                                      inputs.bf16_bits(c["w_k"]), np.asarray(lens), 0)


def check(out, ref, lens, what):
    for b in range(len(lens)):
        if lens[b] == 0:
            assert torch.all(out[b] == 0), f"{what}: empty sequence must give zeros"
            continue
        assert_parity(out[b], ref[b], f"{what} b={b} L={lens[b]}")
    assert gqa.gqa_device_status() == 0


ROOMY = pytest.mark.parametrize("roomy", [False, True], ids=["tight", "roomy"])


@ROOMY
def test_keqv_contiguous_ragged(roomy):
    lens = [0, 1, 17, 31, 32, 33, 1023, 2500, 3000]
    c = case(lens, capacity(len(lens), 3000, roomy), seed=400)
    out = gqa.gqa_decode_keqv(c["q"], c["v"], c["w_k"], c["seq_lens"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(out, oracle_keqv(c, lens), lens, "keqv contiguous")


@ROOMY
def test_keqv_long_positions(roomy):
    """A sequence of 131075 positions: keys at rotation angles up to ~1.3e5 rad.  (One
    sequence alone never fills enough tiles per CTA for the tcgen05 kernel: the roomy
    form adds a short second one.)"""
    lens = [131075, 3] if roomy else [131075]
    c = case(lens, capacity(len(lens), 131080, roomy), seed=401)
    out = gqa.gqa_decode_keqv(c["q"], c["v"], c["w_k"], c["seq_lens"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(out, oracle_keqv(c, lens), lens, "keqv long")


@ROOMY
def test_keqv_rows_past_the_end_are_never_read(roomy):
    lens = [5, 700, 1601]
    c = case(lens, capacity(len(lens), 1700, roomy), seed=402)
    nan = torch.tensor(BF16_NAN, dtype=torch.int16).view(torch.bfloat16).item()
    for b, L in enumerate(lens):
        c["v"][b, L:] = nan
    out = gqa.gqa_decode_keqv(c["q"], c["v"], c["w_k"], c["seq_lens"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(out, oracle_keqv(c, lens), lens, "keqv poisoned")


@ROOMY
def test_keqv_paged(roomy):
    lens = [1, 16, 17, 900, 2049]
    S = max(lens)
    c = case(lens, S, seed=403)
    # the capacity of a paged call is max_pages * 16 positions
    bt, P = inputs.page_table(lens, 403, max_pages=(capacity(len(lens), S, roomy) + 15) // 16,
                              spare_pages=5)
    pool = torch.full((P, 16, KVH, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    for b, L in enumerate(lens):
        for j in range((L + 15) // 16):
            n = min(16, L - 16 * j)
            pool[bt[b, j], :n] = c["v"][b, 16 * j:16 * j + n]
    out = gqa.gqa_decode_keqv_paged(c["q"], pool, c["w_k"], torch.as_tensor(bt, device="cuda"),
                                    c["seq_lens"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(out, oracle_keqv(c, lens), lens, "keqv paged")


@ROOMY
def test_keqv_bf16_output_is_the_rounded_fp32_output(roomy):
    lens = [40, 1500]
    c = case(lens, capacity(len(lens), 1500, roomy), seed=404)
    out32 = gqa.gqa_decode_keqv(c["q"], c["v"], c["w_k"], c["seq_lens"], out_dtype=torch.float32)
    out16 = gqa.gqa_decode_keqv(c["q"], c["v"], c["w_k"], c["seq_lens"], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out16, out32.to(torch.bfloat16))


@ROOMY
def test_keqv_cold_calls_agree_with_the_oracle_every_time(roomy):
    """Twelve calls in a row, each after a write larger than the L2 cache, so every
    CTA's first tile comes from DRAM as fast as the one-time setup of its tables does.
    Every call's output is checked: the rotation angles of the first tiles must not
    depend on which of the two finishes first."""
    lens = [2914, 1371]
    c = case(lens, capacity(len(lens), 3000, roomy), seed=405)
    ref = oracle_keqv(c, lens)
    flush = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty((len(lens), H, D), dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(12):
        flush.add_(1)
        gqa.gqa_decode_keqv(c["q"], c["v"], c["w_k"], c["seq_lens"], out=out)
        outs.append(out.clone())
    torch.cuda.synchronize()
    for k, o in enumerate(outs):
        check(o, ref, lens, f"keqv cold call {k}")
