"""GPU parity of the decode-step producer (gqa_prepare_decode[_paged]) against the
fp64 oracle: q = rope(q_norm(q_raw)), k = rope(k_norm(k_raw)), v = v_norm(v_raw) at
position L - 1, written as bf16 to q_out and to the new token's cache slot.

Gate (from the arithmetic): the kernel computes in fp32 (relative error ~1e-6 on
unit-RMS heads) and rounds to bf16 once, so every output lies within half a bf16
ulp of the exact value plus 4e-6.  Every cache element other than the new
token's slot must keep its sentinel value.
"""
import numpy as np
import pytest
import torch

import decode_attention_gb300 as gqa
import oracle
from decode_attention_gb300 import inputs
from tests.helpers import GLOBAL, SLIDING, assert_parity

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

GEOS = {"sliding": SLIDING, "global": GLOBAL}
ROPE = {"sliding": (oracle.SLIDING_ROPE_PAIRS, oracle.SLIDING_ROPE_THETA),
        "global": (oracle.GLOBAL_ROPE_PAIRS, oracle.GLOBAL_ROPE_THETA)}
SENTINEL = 7.0


def raw_case(B, geo, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    H, KVH, D = geo["H"], geo["KVH"], geo["D"]
    scale = 0.2 + 5 * torch.rand((B, H, 1), generator=g, device="cuda")
    q = (torch.randn((B, H, D), generator=g, device="cuda") * scale).to(torch.bfloat16)
    k = (torch.randn((B, KVH, D), generator=g, device="cuda") * scale[:, :KVH]).to(torch.bfloat16)
    v = (torch.randn((B, KVH, D), generator=g, device="cuda") * 2).to(torch.bfloat16)
    w_q = inputs.k_norm_weight_bf16(D, seed + 1, device="cuda")
    w_k = inputs.k_norm_weight_bf16(D, seed + 2, device="cuda")
    return q, k, v, w_q, w_k


def oracle_of(layer, q, k, v, w_q, w_k, lens):
    n_rot, theta = ROPE[layer]
    bits = inputs.bf16_bits
    return oracle.prepare_decode_f64(bits(q), bits(k), None if v is None else bits(v), bits(w_q),
                                     bits(w_k), np.asarray(lens), n_rot, theta)


def assert_rounded(gpu, ref, what):
    g = gpu.float().cpu().double().numpy()
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    err = np.abs(g - ref)
    bound = 0.5 * ulp + 4e-6
    worst = float(np.max(err - bound))
    assert worst <= 0, f"{what}: an output lies {worst:.3e} beyond its bf16 rounding bound"


def sentinel_like(shape):
    return torch.full(shape, SENTINEL, dtype=torch.bfloat16, device="cuda")


@pytest.mark.parametrize("layer", ["sliding", "global"])
@pytest.mark.parametrize("ring", [False, True])
def test_prepare_contiguous_and_ring(layer, ring):
    geo = GEOS[layer]
    H, KVH, D = geo["H"], geo["KVH"], geo["D"]
    rows = 1024
    lens = [0, 1, 2, 17, 1024] + ([1025, 131075, 262144] if ring else [999])
    B = len(lens)
    q, k, v, w_q, w_k = raw_case(B, geo, seed=500 + ring)
    kc, vc = sentinel_like((B, rows, KVH, D)), sentinel_like((B, rows, KVH, D))
    q_out = sentinel_like((B, H, D))
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    gqa.gqa_prepare_decode(q, k, v, w_q, w_k, seq, q_out, kc, vc, ring=ring)
    torch.cuda.synchronize()
    rq, rk, rv = oracle_of(layer, q, k, v, w_q, w_k, lens)
    touched = torch.zeros((B, rows), dtype=torch.bool, device="cuda")
    for b, L in enumerate(lens):
        if L < 1:
            assert torch.all(q_out[b] == SENTINEL), "no token: q_out untouched"
            continue
        row = (L - 1) % rows if ring else L - 1
        assert_rounded(q_out[b], rq[b], f"{layer} q b={b}")
        assert_rounded(kc[b, row], rk[b], f"{layer} k b={b}")
        assert_rounded(vc[b, row], rv[b], f"{layer} v b={b}")
        touched[b, row] = True
    assert torch.all(kc[~touched] == SENTINEL) and torch.all(vc[~touched] == SENTINEL)


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_prepare_paged(layer):
    geo = GEOS[layer]
    H, KVH, D = geo["H"], geo["KVH"], geo["D"]
    lens = [1, 16, 17, 700, 4097]
    B = len(lens)
    bt, P = inputs.page_table(lens, 501, max_pages=(max(lens) + 15) // 16, spare_pages=3)
    bt = bt.copy()
    bt[2, 1] = P + 4   # sequence 2's new token (position 16) has a bad page: no write
    q, k, v, w_q, w_k = raw_case(B, geo, seed=502)
    kp, vp = sentinel_like((P, 16, KVH, D)), sentinel_like((P, 16, KVH, D))
    q_out = sentinel_like((B, H, D))
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    gqa.gqa_prepare_decode_paged(q, k, v, w_q, w_k, torch.as_tensor(bt, device="cuda"), seq, q_out,
                                 kp, vp)
    torch.cuda.synchronize()
    rq, rk, rv = oracle_of(layer, q, k, v, w_q, w_k, lens)
    touched = torch.zeros((P, 16), dtype=torch.bool, device="cuda")
    for b, L in enumerate(lens):
        assert_rounded(q_out[b], rq[b], f"{layer} paged q b={b}")
        page, slot = int(bt[b, (L - 1) // 16]), (L - 1) % 16
        if not 0 <= page < P:
            continue
        assert_rounded(kp[page, slot], rk[b], f"{layer} paged k b={b}")
        assert_rounded(vp[page, slot], rv[b], f"{layer} paged v b={b}")
        touched[page, slot] = True
    assert torch.all(kp[~touched] == SENTINEL) and torch.all(vp[~touched] == SENTINEL)


def test_prepare_values_equal_keys():
    """Global layer with one K=V cache: only v_norm(k_raw) is written."""
    geo = GLOBAL
    H, KVH, D = geo["H"], geo["KVH"], geo["D"]
    lens = [3, 4096, 131072]
    B, rows = len(lens), 131072
    q, k, _, w_q, w_k = raw_case(B, geo, seed=503)
    vc = sentinel_like((B, rows, KVH, D))
    q_out = sentinel_like((B, H, D))
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    gqa.gqa_prepare_decode(q, k, None, w_q, w_k, seq, q_out, None, vc)
    torch.cuda.synchronize()
    rq, _, rv = oracle_of("global", q, k, None, w_q, w_k, lens)
    for b, L in enumerate(lens):
        assert_rounded(q_out[b], rq[b], f"keqv q b={b}")
        assert_rounded(vc[b, L - 1], rv[b], f"keqv v b={b}")
        vc[b, L - 1] = SENTINEL
    assert torch.all(vc == SENTINEL)


def test_prepare_then_decode_reads_the_new_token():
    """Producer then attention core on a window-capped ring: the decode sees the
    token the producer wrote (checked with the oracle on the produced tensors)."""
    geo = SLIDING
    H, KVH, D = geo["H"], geo["KVH"], geo["D"]
    C = W = 1024
    lens = [1, 700, 1024, 1025, 5000]
    B = len(lens)
    ring = inputs.contiguous_case(B, C, H, KVH, D, lens, seed=504, device="cuda")
    q_raw, k_raw, v_raw, w_q, w_k = raw_case(B, geo, seed=505)
    q = torch.empty_like(ring["q"])
    gqa.gqa_prepare_decode(q_raw, k_raw, v_raw, w_q, w_k, ring["seq_lens"], q, ring["k"], ring["v"],
                           ring=True)
    out = gqa.gqa_decode_ring(q, ring["k"], ring["v"], ring["seq_lens"], W, out_dtype=torch.float32)
    torch.cuda.synchronize()
    bits = inputs.bf16_bits
    ref = oracle.gqa_decode_ring_f64(bits(q), bits(ring["k"]), bits(ring["v"]), np.asarray(lens), W)
    for b in range(B):
        assert_parity(out[b], ref[b], f"pipeline b={b}")
    assert gqa.gqa_device_status() == 0
