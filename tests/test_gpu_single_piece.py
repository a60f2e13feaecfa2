"""Split-KV versus one piece per segment (GQA_TEST_SINGLE_PIECE).

A normal call cuts each (sequence, KV head) segment into pieces on several CTAs and
merges their softmax partials with the log-sum-exp rule.  In the test mode
GQA_TEST_SINGLE_PIECE one CTA computes every segment in one piece, with no partials
and no merge.  The two must agree up to rounding, independently of the oracle's
tolerance:
  * the single-query calls (slidingDecodeGQA on CUDA cores with fp32 weights,
    decodeGQA on mma.sync): max-abs <= 1e-5;
  * the multi-query and K=V calls apply each softmax weight p = 2^(s - m) as a bf16
    hi + lo pair relative to a reference max m that moves with the piece boundaries.
    Each side then carries up to 2^-17 relative error per weight, so the two differ
    by at most 2 * 2^-17 * max|v| (the weights sum to 1): max-abs <= 2^-16 * max|v|
    (8.4e-5 at |v| = 5.5), which is above 1e-5.
The workspace's per-segment partial lists (the library's internal layout: int4
(first static unit, static pieces, first dynamic chunk, dynamic chunks) per segment
at byte 256) show that the normal call did split and the single-piece one did not.
Both are also checked against the fp64 oracle.
"""
import contextlib

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
AGREE = 1e-5


@contextlib.contextmanager
def mode(flags):
    prev = gqa.gqa_set_test_mode(flags)
    try:
        yield
    finally:
        gqa.gqa_set_test_mode(prev)


def pieces(ws, segments):
    """Pieces per segment from the workspace's partial lists."""
    e = ws[256:256 + 16 * segments].view(torch.int32).reshape(segments, 4).cpu().numpy()
    return e[:, 1] + e[:, 3]


def both(call, ws, segments):
    """(normal output, single-piece output), checking the piece counts."""
    normal = call().clone()
    torch.cuda.synchronize()
    split = pieces(ws, segments)
    with mode(gqa.GQA_TEST_SINGLE_PIECE):
        single = call().clone()
    torch.cuda.synchronize()
    one = pieces(ws, segments)
    assert split.max() > 1, "the normal call must split some segment"
    assert np.all(one <= 1), "the single-piece call must not split"
    return normal, single


def agree(a, b, what, vmax=None):
    """Within AGREE, or (vmax given: hi + lo weights) within 2^-16 * vmax."""
    bound = AGREE if vmax is None else 2.0 ** -16 * vmax
    d = (a.double() - b.double()).abs().max().item()
    print(f"{what}: split vs single piece max-abs {d:.2e} (bound {bound:.1e})")
    assert d <= bound, f"{what}: {d:.2e}"


@pytest.mark.parametrize("layer,lens", [
    ("sliding", [2048]),                      # the single-sequence sliding step
    ("sliding", [2048, 5000, 900, 1]),
    ("global", [8192, 5000]),
    ("global", [1, 31, 4097, 8000, 2500]),
])
def test_contiguous(layer, lens):
    geo = GEOS[layer]
    B, S = len(lens), max(lens)
    case = inputs.contiguous_case(B, S, geo["H"], geo["KVH"], geo["D"], lens, 950 + B, device="cuda")
    ws = gqa.new_workspace(B, S, geo["H"], geo["KVH"], geo["D"], geo["window"])

    def call():
        return gqa.gqa_decode(case["q"], case["k"], case["v"], case["seq_lens"], geo["window"],
                              out_dtype=torch.float32, workspace=ws)

    normal, single = both(call, ws, B * geo["KVH"])
    agree(normal, single, f"{layer} {lens}")
    for b, r in oracle_contiguous(case, geo["window"]).items():
        assert_parity(single[b], r, f"single b={b}")
        assert_parity(normal[b], r, f"normal b={b}")
    assert gqa.gqa_device_status(ws) == 0


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_paged(layer):
    geo = GEOS[layer]
    lens = [3000, 6001, 77]
    B = len(lens)
    case = inputs.paged_case(B, geo["H"], geo["KVH"], geo["D"], lens, 960, device="cuda")
    ws = gqa.new_workspace(B, 6016, geo["H"], geo["KVH"], geo["D"], geo["window"])

    def call():
        return gqa.gqa_decode_paged(case["q"], case["k_pages"], case["v_pages"], case["block_table"],
                                    case["seq_lens"], geo["window"], out_dtype=torch.float32,
                                    workspace=ws)

    normal, single = both(call, ws, B * geo["KVH"])
    agree(normal, single, f"paged {layer}")
    ref = oracle_paged(case, geo["window"])
    for b in range(B):
        assert_parity(single[b], ref[b], f"single b={b}")


@pytest.mark.parametrize("layer,T", [("global", 4), ("sliding", 8)])
def test_multi_query(layer, T):
    geo = GEOS[layer]
    lens = [6000, 2000, 3]
    B = len(lens)
    case = inputs.mq_case(B, T, 6000, geo["H"], geo["KVH"], geo["D"], lens, 970 + T, device="cuda")
    ws = torch.empty(gqa.gqa_workspace_size_mq(B, T, geo["H"], geo["KVH"], geo["D"]),
                     dtype=torch.uint8, device="cuda")
    gqa.gqa_workspace_init(ws)

    def call():
        return gqa.gqa_decode_mq(case["q"], case["k"], case["v"], case["seq_lens"], geo["window"],
                                 out_dtype=torch.float32, workspace=ws)

    normal, single = both(call, ws, B * geo["KVH"])
    agree(normal, single, f"multi-query {layer} T={T}", case["v"].float().abs().max().item())
    ref = oracle.gqa_decode_mq_f64(inputs.bf16_bits(case["q"]), inputs.bf16_bits(case["k"]),
                                   inputs.bf16_bits(case["v"]), np.asarray(lens), geo["window"])
    for b in range(B):
        for t in range(T):
            assert_parity(single[b, t], ref[b, t], f"single b={b} t={t}")


@pytest.mark.parametrize("roomy", [False, True], ids=["split_kernel", "tcgen05_kernel"])
def test_keqv(roomy):
    H, KVH, D = GLOBAL["H"], GLOBAL["KVH"], GLOBAL["D"]
    lens = [7000, 3000]
    B = len(lens)
    want = gqa.GQA_KERNEL_TCGEN05 if roomy else gqa.GQA_KERNEL_SPLIT_DECODE
    S = keqv_tcgen05_capacity(B, 7000) if roomy else 7000
    assert gqa.gqa_decode_keqv_kernel(B, S) == want
    case = inputs.contiguous_case(B, S, H, KVH, D, lens, 980, device="cuda")
    w_k = inputs.k_norm_weight_bf16(D, 981, device="cuda")
    ws = gqa.new_workspace(B, S, H, KVH, D, 0)

    def call():
        return gqa.gqa_decode_keqv(case["q"], case["v"], w_k, case["seq_lens"],
                                   out_dtype=torch.float32, workspace=ws)

    normal, single = both(call, ws, B * KVH)
    agree(normal, single, f"keqv {'tcgen05' if roomy else 'split'}",
          case["v"][:, :max(lens)].float().abs().max().item())
    v = case["v"][:, :max(lens)].contiguous()
    ref = oracle.gqa_decode_keqv_f64(inputs.bf16_bits(case["q"]), inputs.bf16_bits(v),
                                     inputs.bf16_bits(w_k), np.asarray(lens), 0)
    for b in range(B):
        assert_parity(single[b], ref[b], f"single b={b}")
