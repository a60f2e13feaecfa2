"""Shared helpers for the GPU parity tests (CUDA path vs the fp64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from decode_attention_gb300 import inputs

# Parity gate for floating-point outputs (the target stated for the attention
# core): max absolute error 1e-2 and relative L2 error 5e-3 against the fp64
# oracle, applied to fp32 output.
TOL_MAX_ABS = 1e-2
TOL_REL_L2 = 5e-3

# Tighter regression budget derived from the arithmetic (fp32 scores and
# accumulation, exp2 with ~2^-22 relative error, P applied to ~16 bits on the
# tensor-core path): errors of order 1e-5 are expected, 1e-3 flags a defect long
# before the gate would.
BUDGET_MAX_ABS = 1e-3

BF16_NAN = 0x7FC0

SLIDING = inputs.SLIDING
GLOBAL = inputs.GLOBAL


def errors(gpu: torch.Tensor, ref: np.ndarray):
    g = gpu.detach().float().cpu().double().numpy()
    diff = np.abs(g - ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel_l2 = float(np.linalg.norm(g - ref) / denom) if denom > 0 else float(np.linalg.norm(g - ref))
    return max_abs, rel_l2


def assert_parity(gpu: torch.Tensor, ref: np.ndarray, what: str = ""):
    assert np.all(np.isfinite(gpu.float().cpu().numpy())), f"{what}: non-finite output"
    max_abs, rel_l2 = errors(gpu, ref)
    assert max_abs <= TOL_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {TOL_MAX_ABS}"
    assert rel_l2 <= TOL_REL_L2, f"{what}: rel-L2 {rel_l2:.3e} > {TOL_REL_L2}"
    assert max_abs <= BUDGET_MAX_ABS, f"{what}: max-abs {max_abs:.3e} above the fp32 budget"
    return max_abs, rel_l2


def attended(L: int, window: int):
    return (max(0, L - window) if window > 0 else 0), L


def oracle_contiguous(case: dict, window: int, batches=None) -> np.ndarray:
    """Oracle output for (a subset of) the sequences of a contiguous case.

    Only the attended rows of each sampled sequence are copied to the host; the
    oracle receives them with pos_base = first attended position, so its own
    window logic decides what to read.
    """
    lens = case["seq_lens"].cpu().numpy()
    B = len(lens)
    batches = range(B) if batches is None else batches
    out = {}
    for b in batches:
        L = int(lens[b])
        lo = max(0, L - window) if window > 0 else 0
        lo_copy = min(lo, L)
        qb = inputs.bf16_bits(case["q"][b:b + 1])
        hi_copy = max(L, lo_copy + 1)   # keep at least one row so shapes are non-empty
        S_cap = case["k"].shape[1]
        hi_copy = min(hi_copy, S_cap)
        lo_copy = min(lo_copy, hi_copy - 1) if hi_copy > 0 else 0
        kb = inputs.bf16_bits(case["k"][b:b + 1, lo_copy:hi_copy])
        vb = inputs.bf16_bits(case["v"][b:b + 1, lo_copy:hi_copy])
        out[b] = oracle.gqa_decode_f64(qb, kb, vb, [L], window, pos_base=lo_copy)[0]
    return out


def oracle_paged(case: dict, window: int) -> np.ndarray:
    return oracle.gqa_decode_paged_f64(
        inputs.bf16_bits(case["q"]), inputs.bf16_bits(case["k_pages"]),
        inputs.bf16_bits(case["v_pages"]), case["block_table"].cpu().numpy(),
        case["seq_lens"].cpu().numpy(), window)


def poison_outside_window(k: torch.Tensor, v: torch.Tensor, lens, window: int):
    """Set every cache row outside [lo_b, L_b) to bf16 NaN (in place)."""
    nan = torch.tensor(BF16_NAN, dtype=torch.int16).view(torch.bfloat16).item()
    for b, L in enumerate(list(lens)):
        lo, hi = attended(int(L), window)
        k[b, :lo] = nan
        v[b, :lo] = nan
        k[b, hi:] = nan
        v[b, hi:] = nan


def cuda_case(B, S, geo, lens, seed):
    return inputs.contiguous_case(B, S, geo["H"], geo["KVH"], geo["D"], lens, seed, device="cuda")


def keqv_tcgen05_capacity(B: int, S: int) -> int:
    """The smallest cache capacity >= S (at most GQA_MAX_SEQ) for which the library
    runs a K=V call of B sequences on the tcgen05 kernel (gqa_decode_keqv_kernel)."""
    import decode_attention_gb300 as gqa
    lo, hi = S, gqa.GQA_MAX_SEQ
    assert gqa.gqa_decode_keqv_kernel(B, hi) == gqa.GQA_KERNEL_TCGEN05, "no capacity takes tcgen05"
    while lo < hi:
        mid = (lo + hi) // 2
        if gqa.gqa_decode_keqv_kernel(B, mid) == gqa.GQA_KERNEL_TCGEN05:
            hi = mid
        else:
            lo = mid + 1
    return lo
