"""GPU parity of the single K=V global cache (gqa_decode_keqv / _paged) against the
fp64 oracle, which derives every key as rope(w_k * v, s) in double precision.

Covers ragged lengths that span many 32-position tiles and several CTAs per
segment, a sequence reaching position 131074 (where the rotation angle of the
fastest pair is ~1.3e5 rad, so the kernel's fp64 angle reduction matters), the
paged form, NaN in every cache row past the sequence end, and the bf16 output.
"""
import numpy as np
import pytest
import torch

import decode_attention_gb300 as gqa
import oracle
from decode_attention_gb300 import inputs
from tests.helpers import BF16_NAN, GLOBAL, assert_parity

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

H, KVH, D = GLOBAL["H"], GLOBAL["KVH"], GLOBAL["D"]


def case(lens, S, seed):
    c = inputs.contiguous_case(len(lens), S, H, KVH, D, lens, seed, device="cuda")
    c["w_k"] = inputs.k_norm_weight_bf16(D, inputs.tensor_seed(seed, "w_k"), device="cuda")
    return c


def oracle_keqv(c, lens):
    return oracle.gqa_decode_keqv_f64(inputs.bf16_bits(c["q"]), inputs.bf16_bits(c["v"]),
                                      inputs.bf16_bits(c["w_k"]), np.asarray(lens), 0)


def check(out, ref, lens, what):
    for b in range(len(lens)):
        if lens[b] == 0:
            assert torch.all(out[b] == 0), f"{what}: empty sequence must give zeros"
            continue
        assert_parity(out[b], ref[b], f"{what} b={b} L={lens[b]}")
    assert gqa.gqa_device_status() == 0


def test_keqv_contiguous_ragged():
    lens = [0, 1, 17, 31, 32, 33, 1023, 2500, 3000]
    c = case(lens, 3000, seed=400)
    out = gqa.gqa_decode_keqv(c["q"], c["v"], c["w_k"], c["seq_lens"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(out, oracle_keqv(c, lens), lens, "keqv contiguous")


def test_keqv_long_positions():
    """One sequence of 131075 positions: keys at rotation angles up to ~1.3e5 rad."""
    lens = [131075]
    c = case(lens, 131080, seed=401)
    out = gqa.gqa_decode_keqv(c["q"], c["v"], c["w_k"], c["seq_lens"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(out, oracle_keqv(c, lens), lens, "keqv long")


def test_keqv_rows_past_the_end_are_never_read():
    lens = [5, 700, 1601]
    c = case(lens, 1700, seed=402)
    nan = torch.tensor(BF16_NAN, dtype=torch.int16).view(torch.bfloat16).item()
    for b, L in enumerate(lens):
        c["v"][b, L:] = nan
    out = gqa.gqa_decode_keqv(c["q"], c["v"], c["w_k"], c["seq_lens"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(out, oracle_keqv(c, lens), lens, "keqv poisoned")


def test_keqv_paged():
    lens = [1, 16, 17, 900, 2049]
    S = max(lens)
    c = case(lens, S, seed=403)
    bt, P = inputs.page_table(lens, 403, max_pages=(S + 15) // 16, spare_pages=5)
    pool = torch.full((P, 16, KVH, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    for b, L in enumerate(lens):
        for j in range((L + 15) // 16):
            n = min(16, L - 16 * j)
            pool[bt[b, j], :n] = c["v"][b, 16 * j:16 * j + n]
    out = gqa.gqa_decode_keqv_paged(c["q"], pool, c["w_k"], torch.as_tensor(bt, device="cuda"),
                                    c["seq_lens"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    check(out, oracle_keqv(c, lens), lens, "keqv paged")


def test_keqv_bf16_output_is_the_rounded_fp32_output():
    lens = [40, 1500]
    c = case(lens, 1500, seed=404)
    out32 = gqa.gqa_decode_keqv(c["q"], c["v"], c["w_k"], c["seq_lens"], out_dtype=torch.float32)
    out16 = gqa.gqa_decode_keqv(c["q"], c["v"], c["w_k"], c["seq_lens"], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out16, out32.to(torch.bfloat16))
