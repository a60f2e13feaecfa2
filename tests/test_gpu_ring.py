"""GPU parity of gqa_decode_ring (window-capped ring-buffer cache, position s at row
s mod C) against the fp64 ring oracle, through the C ABI.

Covers the retrofit's window sizes (1024, 2048, 4096, 8192 with C = window), a ring
longer than its window, lengths below, at and across multiples of C (so pieces
split at the wrap), both geometries, NaN in every row the window does not reach,
and the bf16 output.
"""
import numpy as np
import pytest
import torch

import decode_attention_gb300 as gqa
import oracle
from decode_attention_gb300 import inputs
from tests.helpers import BF16_NAN, GLOBAL, SLIDING, assert_parity

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

GEOS = {"sliding": SLIDING, "global": GLOBAL}


def ring_case(B, C, geo, lens, seed):
    return inputs.contiguous_case(B, C, geo["H"], geo["KVH"], geo["D"], lens, seed, device="cuda")


def oracle_ring(case, window):
    return oracle.gqa_decode_ring_f64(
        inputs.bf16_bits(case["q"]), inputs.bf16_bits(case["k"]), inputs.bf16_bits(case["v"]),
        case["seq_lens"].cpu().numpy(), window)


def run_ring(case, window, out_dtype=torch.float32):
    out = gqa.gqa_decode_ring(case["q"], case["k"], case["v"], case["seq_lens"], window,
                              out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out


def check(case, window, out, what):
    ref = oracle_ring(case, window)
    for b in range(ref.shape[0]):
        assert_parity(out[b], ref[b], f"{what} b={b} L={int(case['seq_lens'][b])}")
    assert gqa.gqa_device_status() == 0


@pytest.mark.parametrize("window", [1024, 2048, 4096, 8192])
def test_retrofit_windows_ring_equal_to_window(window):
    """Sliding geometry, C = window (each layer's cache capped at its window)."""
    lens = [1, 17, window - 1, window, window + 1, 3 * window + 77]
    case = ring_case(len(lens), window, SLIDING, lens, seed=300 + window // 1024)
    out = run_ring(case, window)
    check(case, window, out, f"ring W=C={window}")


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_ring_longer_than_window(layer):
    geo = GEOS[layer]
    C, W = 1100, 1024
    lens = [0, 1, 1099, 1100, 1101, 2200, 2201, 5555, 262144]
    case = ring_case(len(lens), C, geo, lens, seed=310)
    out = run_ring(case, W)
    check(case, W, out, f"{layer} ring C={C} W={W}")


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_ring_rows_outside_the_window_are_never_read(layer):
    """Every row that holds no attended position is bf16 NaN."""
    geo = GEOS[layer]
    C, W = 640, 600
    lens = [600, 640, 641, 1239, 1240, 1281, 7000]
    case = ring_case(len(lens), C, geo, lens, seed=311)
    nan = torch.tensor(BF16_NAN, dtype=torch.int16).view(torch.bfloat16).item()
    for b, L in enumerate(lens):
        keep = {s % C for s in range(max(0, L - W), L)}
        drop = torch.tensor([r for r in range(C) if r not in keep], dtype=torch.long, device="cuda")
        if drop.numel():
            case["k"][b, drop] = nan
            case["v"][b, drop] = nan
    out = run_ring(case, W)
    check(case, W, out, f"{layer} poisoned ring")


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_ring_many_sequences_split_across_ctas(layer):
    """A batch large enough that static units and dynamic chunks cross the wrap."""
    geo = GEOS[layer]
    C = W = 2048
    rng = np.random.default_rng(312)
    B = 24
    lens = rng.integers(1, 6 * C, B).tolist()
    case = ring_case(B, C, geo, lens, seed=312)
    out = run_ring(case, W)
    check(case, W, out, f"{layer} ring batch")


def test_ring_bf16_output_is_the_rounded_fp32_output():
    C = W = 1024
    lens = [5, 1024, 3333]
    case = ring_case(len(lens), C, SLIDING, lens, seed=313)
    out32 = run_ring(case, W, torch.float32)
    out16 = run_ring(case, W, torch.bfloat16)
    assert torch.equal(out16, out32.to(torch.bfloat16))
