"""GPU parity: libgqadecode.so (through the C ABI) against the fp64 oracle.

Sizes here keep the oracle within seconds while spanning many 32-position tiles,
several CTAs per (b, kvh) segment (so the split-softmax combine runs) and ragged
tails; full-size workloads are in test_gpu_workloads.py.
"""
import numpy as np
import pytest
import torch

import decode_attention_gb300 as gqa
from decode_attention_gb300 import inputs
from tests.helpers import (GLOBAL, SLIDING, assert_parity, attended, cuda_case, errors,
                           oracle_contiguous, oracle_paged, poison_outside_window)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

GEOS = {"sliding": SLIDING, "global": GLOBAL}


def run(case, window, out_dtype=torch.float32, workspace=None):
    out = gqa.gqa_decode(case["q"], case["k"], case["v"], case["seq_lens"], window,
                         out_dtype=out_dtype, workspace=workspace)
    torch.cuda.synchronize()
    return out


def check_against_oracle(case, window, out, what):
    ref = oracle_contiguous(case, window)
    worst = (0.0, 0.0)
    for b, r in ref.items():
        ma, rl = assert_parity(out[b], r, f"{what} b={b} L={int(case['seq_lens'][b])}")
        worst = (max(worst[0], ma), max(worst[1], rl))
    return worst


def status_clean():
    assert gqa.gqa_device_status() == 0


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_small_batch_parity(layer):
    geo = GEOS[layer]
    lens = [1, 17, 1023, 1024, 1025, 1300]
    case = cuda_case(len(lens), 1300, geo, lens, seed=101)
    out = run(case, geo["window"])
    worst = check_against_oracle(case, geo["window"], out, layer)
    print(f"{layer}: worst max-abs {worst[0]:.2e} rel-L2 {worst[1]:.2e}")
    status_clean()


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_edge_lengths(layer):
    geo = GEOS[layer]
    lens = [0, 1, 2, 15, 16, 17, 31, 32, 33, 1023, 1024, 1025, 1040, 2100]
    case = cuda_case(len(lens), 2100, geo, lens, seed=102)
    out = run(case, geo["window"])
    assert torch.all(out[0] == 0), "L = 0 must give zeros"
    check_against_oracle(case, geo["window"], out, f"{layer} edges")
    status_clean()


@pytest.mark.parametrize("layer", ["sliding", "global"])
@pytest.mark.parametrize("window", [0, 1, 16, 1024, 2048, 8192])
def test_any_window(layer, window):
    """The window is a runtime parameter; both geometries accept any value."""
    geo = GEOS[layer]
    lens = [1, 16, 700, 3000, 9000]
    case = cuda_case(len(lens), 9000, geo, lens, seed=103 + window)
    out = run(case, window)
    check_against_oracle(case, window, out, f"{layer} W={window}")


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_bf16_output_is_rounded_fp32_output(layer):
    geo = GEOS[layer]
    lens = [5, 999, 2048, 3333]
    case = cuda_case(len(lens), 3333, geo, lens, seed=104)
    o32 = run(case, geo["window"], torch.float32)
    o16 = run(case, geo["window"], torch.bfloat16)
    assert torch.equal(o16, o32.to(torch.bfloat16))
    ref = oracle_contiguous(case, geo["window"])
    for b, r in ref.items():
        _, rel = errors(o16[b], r)
        assert rel <= 5e-3


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_deterministic(layer):
    geo = GEOS[layer]
    lens = [4000, 3, 2500, 1024]
    case = cuda_case(len(lens), 4000, geo, lens, seed=105)
    a = run(case, geo["window"])
    b = run(case, geo["window"])
    assert torch.equal(a, b)


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_rows_outside_the_range_are_never_used(layer):
    """NaN in every cache row before the window or at/after L changes nothing."""
    geo = GEOS[layer]
    lens = [1, 30, 1024, 1500, 2600]
    case = cuda_case(len(lens), 2600, geo, lens, seed=106)
    clean = run(case, geo["window"])
    poison_outside_window(case["k"], case["v"], lens, geo["window"])
    dirty = run(case, geo["window"])
    assert torch.isfinite(dirty).all()
    assert torch.equal(clean, dirty)


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_caller_workspace_matches_library_workspace(layer):
    geo = GEOS[layer]
    lens = [700, 2000, 1]
    case = cuda_case(len(lens), 2000, geo, lens, seed=107)
    a = run(case, geo["window"])
    ws = gqa.new_workspace(len(lens), 2000, geo["H"], geo["KVH"], geo["D"], geo["window"])
    b = run(case, geo["window"], workspace=ws)
    c = run(case, geo["window"], workspace=ws)    # the workspace is reusable as left
    assert torch.equal(a, b) and torch.equal(a, c)
    assert gqa.gqa_device_status(ws) == 0
    small = ws[: ws.numel() // 2]
    with pytest.raises(gqa.GQAError) as e:
        run(case, geo["window"], workspace=small)
    assert e.value.status == gqa.GQA_ERR_WORKSPACE


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_lengths_beyond_capacity_are_clamped_and_flagged(layer):
    geo = GEOS[layer]
    S = 600
    case = cuda_case(2, S, geo, [S, S], seed=108)
    ref = run(case, geo["window"])
    case["seq_lens"] = torch.tensor([S + 50, S], dtype=torch.int32, device="cuda")
    out = run(case, geo["window"])
    assert torch.equal(out, ref)
    assert gqa.gqa_device_status() & gqa.GQA_DEVICE_BAD_LENGTH
    status_clean()


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_max_batch(layer):
    geo = GEOS[layer]
    rng = np.random.default_rng(7)
    lens = rng.integers(0, 200, size=256).astype(np.int32)
    lens[0], lens[255] = 200, 0
    case = cuda_case(256, 200, geo, lens, seed=109)
    out = run(case, geo["window"])
    check_against_oracle(case, geo["window"], out, f"{layer} B=256")


def test_max_sequence_global():
    """S = 262144 (the top of the shape domain), one sequence, full history."""
    geo = GLOBAL
    case = cuda_case(1, 262144, geo, [262144], seed=110)
    out = run(case, 0)
    check_against_oracle(case, 0, out, "global S=262144")
    del case
    torch.cuda.empty_cache()


def test_all_lengths_zero():
    case = cuda_case(3, 64, SLIDING, [0, 0, 0], seed=111)
    out = run(case, 1024)
    assert torch.all(out == 0)


def test_empty_batch():
    q = torch.empty(0, 32, 256, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(0, 16, 16, 256, dtype=torch.bfloat16, device="cuda")
    lens = torch.empty(0, dtype=torch.int32, device="cuda")
    out = gqa.gqa_decode(q, k, k, lens, 1024)
    assert out.shape == (0, 32, 256)


def test_k_and_v_may_alias():
    case = cuda_case(2, 300, GLOBAL, [300, 77], seed=112)
    case["v"] = case["k"]
    out = run(case, 0)
    check_against_oracle(case, 0, out, "aliased k/v")


# ---------------------------------------------------------------------------
# paged cache
# ---------------------------------------------------------------------------

def paged(lens, geo, seed, spare=5, max_pages=None):
    return inputs.paged_case(len(lens), geo["H"], geo["KVH"], geo["D"], lens, seed,
                             max_pages=max_pages, device="cuda", spare_pages=spare)


def run_paged(case, window, out_dtype=torch.float32):
    out = gqa.gqa_decode_paged(case["q"], case["k_pages"], case["v_pages"], case["block_table"],
                               case["seq_lens"], window, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_paged_parity(layer):
    geo = GEOS[layer]
    lens = [0, 1, 15, 16, 17, 1023, 1025, 1039, 2500, 4097]
    case = paged(lens, geo, seed=120, max_pages=300)
    out = run_paged(case, geo["window"])
    ref = oracle_paged(case, geo["window"])
    for b in range(len(lens)):
        assert_parity(out[b], ref[b], f"paged {layer} b={b} L={lens[b]}")
    status_clean()


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_paged_matches_contiguous(layer):
    """Same rows through a permuted page table give the same result (the tile
    boundaries differ, so agreement is to fp32 rounding, not bitwise)."""
    geo = GEOS[layer]
    lens = [3000, 1, 1100, 48]
    contig = cuda_case(len(lens), 3000, geo, lens, seed=121)
    bt, P = inputs.page_table(lens, 121, spare_pages=3)
    kp = torch.full((P, 16, geo["KVH"], geo["D"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = kp.clone()
    for b, L in enumerate(lens):
        for j in range((L + 15) // 16):
            n = min(16, L - 16 * j)
            kp[bt[b, j], :n] = contig["k"][b, 16 * j:16 * j + n]
            vp[bt[b, j], :n] = contig["v"][b, 16 * j:16 * j + n]
    case = dict(q=contig["q"], k_pages=kp, v_pages=vp, block_table=torch.as_tensor(bt, device="cuda"),
                seq_lens=contig["seq_lens"])
    a = run(contig, geo["window"])
    b = run_paged(case, geo["window"])
    assert torch.isfinite(b).all()
    assert (a - b).abs().max().item() <= 1e-5


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_paged_bad_page_gives_nan_and_flag(layer):
    geo = GEOS[layer]
    lens = [200, 200, 200]
    case = paged(lens, geo, seed=122)
    good = run_paged(case, geo["window"])
    bt = case["block_table"].clone()
    bt[1, 12] = case["k_pages"].shape[0] + 3    # attended page of sequence 1 (window >= 200)
    case["block_table"] = bt
    out = run_paged(case, geo["window"])
    assert torch.isnan(out[1]).all()
    assert torch.equal(out[0], good[0]) and torch.equal(out[2], good[2])
    assert gqa.gqa_device_status() & gqa.GQA_DEVICE_BAD_PAGE
    status_clean()


def test_paged_unread_entries_may_hold_anything():
    """Entries past the last page, and pages wholly before the window, are never read."""
    geo = SLIDING
    lens = [3000, 1500]
    case = paged(lens, geo, seed=123)
    good = run_paged(case, 1024)
    bt = case["block_table"].clone()
    bt[0, : (3000 - 1024) // 16] = -99            # pages entirely before the window
    bt[1, (1500 + 15) // 16:] = 10 ** 9          # past the last page
    case["block_table"] = bt
    out = run_paged(case, 1024)
    assert torch.equal(out, good)
    status_clean()
