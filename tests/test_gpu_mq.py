"""GPU parity of the multi-query decode (gqa_decode_mq / gqa_decode_mq_paged, the
tcgen05 kernel) against the fp64 multi-query oracle, through the C ABI.

Query t of a T-token step sits at position L - T + t and attends with its own
causal (and sliding-window) mask.  Covers both geometries at every supported T,
lengths below, at and across tile (128) and window boundaries, sequences shorter
than T, NaN in every row outside the attended union, paged caches with a bad page
seen by one query only, batches large enough for dynamic chunks and the combine
kernel, the bf16 output, and agreement with the single-query path at T = 1.
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
MAX_T = {"sliding": gqa.GQA_MAX_QUERIES_SLIDING, "global": gqa.GQA_MAX_QUERIES_GLOBAL}


def mq_case(B, T, S, geo, lens, seed):
    return inputs.mq_case(B, T, S, geo["H"], geo["KVH"], geo["D"], lens, seed, device="cuda")


def oracle_mq(case, window):
    return oracle.gqa_decode_mq_f64(
        inputs.bf16_bits(case["q"]), inputs.bf16_bits(case["k"]), inputs.bf16_bits(case["v"]),
        case["seq_lens"].cpu().numpy(), window)


def run_mq(case, window, out_dtype=torch.float32):
    out = gqa.gqa_decode_mq(case["q"], case["k"], case["v"], case["seq_lens"], window,
                            out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out


def check(out, ref, lens, what):
    for b in range(ref.shape[0]):
        for t in range(ref.shape[1]):
            assert_parity(out[b, t], ref[b, t], f"{what} b={b} L={lens[b]} t={t}")


def union_range(L, T, window):
    hi = L
    lo = max(0, L - T + 1 - window) if window > 0 else 0
    return lo, hi


@pytest.mark.parametrize("layer,T", [("sliding", 1), ("sliding", 2), ("sliding", 5),
                                     ("sliding", 8), ("global", 1), ("global", 2),
                                     ("global", 3), ("global", 4)])
def test_mq_matches_oracle(layer, T):
    geo = GEOS[layer]
    W = geo["window"]
    S = 1400
    lens = [1, T, T + 1, 127, 128, 129, 300, 1031, 1024 + T, 1400]
    if T > 1:
        lens[0] = T - 1   # the first queries sit before the start
    case = mq_case(len(lens), T, S, geo, lens, seed=400 + T)
    out = run_mq(case, W)
    check(out, oracle_mq(case, W), lens, f"{layer} T={T}")
    assert gqa.gqa_device_status() == 0


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_mq_rows_outside_the_union_are_never_used(layer):
    """bf16 NaN in every cache row outside [L - T + 1 - W, L) (or past L)."""
    geo = GEOS[layer]
    T, W, S = MAX_T[layer], geo["window"], 1500
    lens = [5, 130, 1030, 1100, 1500]
    case = mq_case(len(lens), T, S, geo, lens, seed=410)
    nan = torch.tensor(BF16_NAN, dtype=torch.int16).view(torch.bfloat16).item()
    for b, L in enumerate(lens):
        lo, hi = union_range(L, T, W)
        for name in ("k", "v"):
            case[name][b, :lo] = nan
            case[name][b, hi:] = nan
    out = run_mq(case, W)
    check(out, oracle_mq(case, W), lens, f"{layer} poisoned")


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_mq_batch_with_dynamic_chunks(layer):
    """Enough work per CTA that pieces split segments (combine kernel, dynamic chunks)."""
    geo = GEOS[layer]
    T, W = MAX_T[layer], geo["window"]
    rng = np.random.default_rng(420)
    B = 12 if layer == "global" else 40
    S = 12000 if layer == "global" else 3000
    lens = rng.integers(1, S + 1, B).tolist()
    case = mq_case(B, T, S, geo, lens, seed=420)
    out = run_mq(case, W)
    check(out, oracle_mq(case, W), lens, f"{layer} batch")


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_mq_single_query_agrees_with_decode(layer):
    """T = 1 is the ordinary decode step (two different kernels, same result up to
    rounding)."""
    geo = GEOS[layer]
    lens = [1, 200, 1500, 4000]
    case = mq_case(len(lens), 1, 4000, geo, lens, seed=430)
    out_mq = run_mq(case, geo["window"])
    out_1 = gqa.gqa_decode(case["q"][:, 0].contiguous(), case["k"], case["v"], case["seq_lens"],
                           geo["window"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert float((out_mq[:, 0] - out_1).abs().max()) < 1e-4


def test_mq_empty_sequences_are_zero():
    geo = GLOBAL
    lens = [0, 3, 0]
    case = mq_case(len(lens), 4, 64, geo, lens, seed=440)
    out = run_mq(case, 0)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    check(out, oracle_mq(case, 0), lens, "empty")


def test_mq_bf16_output_is_the_rounded_fp32_output():
    geo = SLIDING
    lens = [7, 900, 1300]
    case = mq_case(len(lens), 4, 1300, geo, lens, seed=450)
    out32 = run_mq(case, geo["window"], torch.float32)
    out16 = run_mq(case, geo["window"], torch.bfloat16)
    assert torch.equal(out16, out32.to(torch.bfloat16))


# ---------------------------------------------------------------------------
# paged caches
# ---------------------------------------------------------------------------

def paged_mq(B, T, geo, lens, seed, spare=0):
    return inputs.paged_mq_case(B, T, geo["H"], geo["KVH"], geo["D"], lens, seed, device="cuda",
                                spare_pages=spare)


def oracle_paged_mq(case, window):
    return oracle.gqa_decode_mq_paged_f64(
        inputs.bf16_bits(case["q"]), inputs.bf16_bits(case["k_pages"]),
        inputs.bf16_bits(case["v_pages"]), case["block_table"].cpu().numpy(),
        case["seq_lens"].cpu().numpy(), window)


def run_paged_mq(case, window):
    out = gqa.gqa_decode_mq_paged(case["q"], case["k_pages"], case["v_pages"],
                                  case["block_table"], case["seq_lens"], window,
                                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_mq_paged_matches_oracle(layer):
    geo = GEOS[layer]
    T, W = MAX_T[layer], geo["window"]
    lens = [2, 17, 128, 129, 1040, 2100]
    case = paged_mq(len(lens), T, geo, lens, seed=460, spare=5)
    out = run_paged_mq(case, W)
    check(out, oracle_paged_mq(case, W), lens, f"{layer} paged")
    assert gqa.gqa_device_status() == 0


def test_mq_paged_bad_page_hits_only_the_query_that_sees_it():
    """A bad id on the page that holds only position L - 1 (its first slot): the last
    query's outputs are NaN, every other query is exact, and the status bit is set."""
    geo = GLOBAL
    T = 3
    lens = [49, 300]   # L - 1 = 48: first slot of page 3
    case = paged_mq(len(lens), T, geo, lens, seed=470)
    case["block_table"][0, 3] = case["k_pages"].shape[0] + 7
    out = run_paged_mq(case, 0)
    assert torch.all(torch.isnan(out[0, T - 1]))
    ref = oracle_paged_mq(case, 0)
    check(out[:, :T - 1], ref[:, :T - 1], lens, "bad page, earlier queries")
    check(out[1:], ref[1:], lens[1:], "bad page, other sequence")
    assert gqa.gqa_device_status() & gqa.GQA_DEVICE_BAD_PAGE


def test_mq_rejects_bad_query_counts():
    geo = GLOBAL
    case = mq_case(1, 1, 16, geo, [4], seed=480)
    for T in (0, gqa.GQA_MAX_QUERIES_GLOBAL + 1):
        q = torch.zeros((1, max(T, 1), geo["H"], geo["D"]), dtype=torch.bfloat16, device="cuda")
        lib = gqa.load_library()
        out = torch.empty((1, max(T, 1), geo["H"], geo["D"]), dtype=torch.float32, device="cuda")
        st = lib.gqa_decode_mq(q.data_ptr(), case["k"].data_ptr(), case["v"].data_ptr(),
                               case["seq_lens"].data_ptr(), 1, T, 16, geo["H"], geo["KVH"],
                               geo["D"], 0, out.data_ptr(), gqa.GQA_OUT_F32, None, 0, None)
        assert st == gqa.GQA_ERR_INVALID_ARGUMENT
