"""Seeded synthetic inputs for the decode attention core.

This module is the only code shared by the CUDA path's tests/benchmark and the
fp64 oracle's tests.  It draws inputs; it holds none of the attention
arithmetic.

Recipe (gemma-4-31B Model Spec: ``attn.qk_norm`` and ``attn.v_norm`` rows of the
"Compute-graph nodes" table, eps 1e-6; "Tensors of the main nodes" table,
``attn.core`` row, for the shapes):

* every head vector of q, k and v is drawn N(0, 1) in fp32, divided by its root
  mean square sqrt(mean(x^2) + 1e-6) (unit weight), then rounded to bf16
  (round-to-nearest-even) -- the state in which the attention core receives
  them after the per-head norms;
* sequence lengths come from ``numpy.random.default_rng(seed)``;
* tensor values come from ``torch.Generator(device).manual_seed(seed * 16 + id)``
  with a fixed id per tensor, drawn in fixed-size chunks so the values depend on
  the seed, the shape and the device only;
* paged caches use 16-position pages whose physical ids are a seeded random
  permutation; block-table entries past a sequence's last page hold -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

# Layer geometries of the Model Spec's two attention-core rows.
SLIDING = dict(H=32, KVH=16, D=256, window=1024)  # slidingDecodeGQA
GLOBAL = dict(H=32, KVH=4, D=512, window=0)       # decodeGQA
PAGE_SIZE = 16                                    # "Shape domain" row of "At a glance"

_RMS_EPS = 1e-6
_CHUNK_ELEMS = 1 << 27

_TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "k_pages": 4, "v_pages": 5, "w_k": 6}


def rms_normalised_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """bf16 tensor whose last-dim vectors are N(0,1) draws scaled to unit RMS."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if out.numel() == 0:
        return out
    d = shape[-1]
    rows = out.numel() // d
    flat = out.view(rows, d)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    step = max(1, _CHUNK_ELEMS // d)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = torch.randn((r1 - r0, d), generator=gen, device=device, dtype=torch.float32)
        x = x * torch.rsqrt(x.square().mean(dim=-1, keepdim=True) + _RMS_EPS)
        flat[r0:r1].copy_(x)
    return out


def k_norm_weight_bf16(D: int, seed: int, device="cpu") -> torch.Tensor:
    """Synthetic k_norm weight [D] (bf16): 1 + 0.25 * N(0, 1), a learned per-channel
    scale around 1 (the checkpoint's values are not available)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.randn((D,), generator=gen, device=device, dtype=torch.float32)
    return (1.0 + 0.25 * x).to(torch.bfloat16)


def tensor_seed(seed: int, name: str) -> int:
    return int(seed) * 16 + _TENSOR_IDS[name]


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 numpy view (on the host) of a bf16 tensor's bit patterns."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------
# Sequence lengths of the five benchmark workloads
# ----------------------------------------------------------------------------

def lengths_fixed(value: int, batch: int):
    return lambda rng: np.full(batch, value, dtype=np.int32)


def lengths_uniform(lo: int, hi: int, batch: int):
    """Integers uniform on [lo, hi] inclusive."""
    return lambda rng: rng.integers(lo, hi, size=batch, endpoint=True).astype(np.int32)


def lengths_lognormal(median: float, sigma: float, lo: int, hi: int, batch: int):
    """round(exp(ln(median) + sigma * z)), z ~ N(0, 1), clipped to [lo, hi]."""
    def draw(rng):
        z = rng.standard_normal(batch)
        x = np.rint(np.exp(math.log(median) + sigma * z))
        return np.clip(x, lo, hi).astype(np.int32)
    return draw


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: a geometry (or two, for the paged mix) and lengths."""
    name: str
    description: str
    B: int
    S: int                   # cache capacity in positions (contiguous) / max length (paged)
    seed: int
    lengths: object = field(repr=False)
    layers: tuple = ()       # ("sliding",) / ("global",) / ("sliding", "global")
    paged: bool = False
    rings: tuple = ()        # windows of ring-cache sliding calls (ring length = window)
    keqv: bool = False       # global layer over a single K=V cache (values only)
    step: bool = False       # each ring call is preceded by the decode-step producer
    queries: int = 0         # > 0: multi-query calls with this many new tokens per sequence

    def seq_lens(self) -> np.ndarray:
        return self.lengths(np.random.default_rng(self.seed))


WORKLOADS = {
    w.name: w for w in [
        Workload("sliding_b1_s2048", "slidingDecodeGQA single step, B=1, seq_len 2048",
                 B=1, S=2048, seed=0, lengths=lengths_fixed(2048, 1), layers=("sliding",)),
        Workload("global_b8_s8192", "decodeGQA, B=8, seq_lens uniform on [1, 8192]",
                 B=8, S=8192, seed=1, lengths=lengths_uniform(1, 8192, 8), layers=("global",)),
        Workload("sliding_b64_s32768", "slidingDecodeGQA batched, B=64, seq_lens uniform on [1, 32768]",
                 B=64, S=32768, seed=2, lengths=lengths_uniform(1, 32768, 64), layers=("sliding",)),
        Workload("global_b16_s131072", "decodeGQA long context, B=16, seq_lens uniform on [65536, 131072]",
                 B=16, S=131072, seed=3, lengths=lengths_uniform(65536, 131072, 16),
                 layers=("global",)),
        Workload("paged_mixed_b256", "paged mixed batch, B=256, lognormal seq_lens (median 4096, "
                 "sigma 1) clipped to [1, 65536]; one sliding and one global call",
                 B=256, S=65536, seed=4, lengths=lengths_lognormal(4096, 1.0, 1, 65536, 256),
                 layers=("sliding", "global"), paged=True),
        # One block of the progressive-window retrofit ("Retrofit Plan: Gemma 4 31B IT ->
        # Progressive Multi-Scale SWA with Block Attention Residuals", §3.3): four
        # sliding layers with windows 1024, 2048, 4096, 8192, each over its own
        # window-capped ring cache, at the batched sliding shape's lengths.
        Workload("retrofit_block_b64", "progressive-window sliding block, B=64, seq_lens uniform "
                 "on [1, 32768]; four ring-cache calls, windows 1024/2048/4096/8192",
                 B=64, S=32768, seed=6, lengths=lengths_uniform(1, 32768, 64),
                 layers=("sliding",), rings=(1024, 2048, 4096, 8192)),
        # One sliding layer's decode step: the producer (norms, rope, append at L - 1)
        # then the attention core over a window-capped ring, at the batched sliding
        # shape's lengths.
        Workload("sliding_step_b64", "sliding layer decode step, B=64, seq_lens uniform on "
                 "[1, 32768]: producer (q/k/v norms, rope, ring append) then the attention core "
                 "over a 1024-row ring", B=64, S=32768, seed=9,
                 lengths=lengths_uniform(1, 32768, 64), layers=("sliding",), rings=(1024,),
                 step=True),
        # The long-context global shape over a single K=V cache: keys derived from the
        # cached values in the kernel (Model Spec "What to watch for": values = keys).
        Workload("global_keqv_b16_s131072", "decodeGQA long context over a single K=V cache, "
                 "B=16, seq_lens uniform on [65536, 131072]", B=16, S=131072, seed=7,
                 lengths=lengths_uniform(65536, 131072, 16), layers=("global",), keqv=True),
        # mid-size: a cache large enough for the tcgen05 K=V kernel, small enough for a
        # full profiler capture
        Workload("global_keqv_b16_s24576", "decodeGQA over a single K=V cache, B=16, seq_lens "
                 "uniform on [12288, 24576]", B=16, S=24576, seed=13,
                 lengths=lengths_uniform(12288, 24576, 16), layers=("global",), keqv=True),
        Workload("global_keqv_b8_s8192", "decodeGQA over a single K=V cache, B=8, seq_lens "
                 "uniform on [1, 8192]", B=8, S=8192, seed=8, lengths=lengths_uniform(1, 8192, 8),
                 layers=("global",), keqv=True),
        # Multi-query steps ("Gemma 4 31B-it Text Architecture", "Inference behavior":
        # new query positions attend to the cache with the same masks): T new tokens
        # per sequence, e.g. a speculative-decoding verify step of T - 1 draft tokens
        # plus one.  The same length draws as the single-query shapes.
        Workload("global_mq4_b16_s131072", "decodeGQA long context, 4 new tokens per sequence "
                 "(multi-query), B=16, seq_lens uniform on [65536, 131072]", B=16, S=131072,
                 seed=10, lengths=lengths_uniform(65536, 131072, 16), layers=("global",),
                 queries=4),
        Workload("sliding_mq8_b64_s32768", "slidingDecodeGQA batched, 8 new tokens per sequence "
                 "(multi-query), B=64, seq_lens uniform on [1, 32768]", B=64, S=32768, seed=11,
                 lengths=lengths_uniform(1, 32768, 64), layers=("sliding",), queries=8),
        Workload("global_mq4_b8_s8192", "decodeGQA, 4 new tokens per sequence (multi-query), B=8, "
                 "seq_lens uniform on [1, 8192]", B=8, S=8192, seed=12,
                 lengths=lengths_uniform(1, 8192, 8), layers=("global",), queries=4),
        # One new token through the multi-query entry point, at the single-query shapes'
        # seeds and lengths (a one-token call runs the single-query kernel).
        Workload("global_mq1_b8_s8192", "decodeGQA, B=8, seq_lens uniform on [1, 8192], one "
                 "new token through the multi-query entry point", B=8, S=8192, seed=1,
                 lengths=lengths_uniform(1, 8192, 8), layers=("global",), queries=1),
        Workload("global_mq1_b16_s131072", "decodeGQA long context, B=16, seq_lens uniform on "
                 "[65536, 131072], one new token through the multi-query entry point", B=16,
                 S=131072, seed=3, lengths=lengths_uniform(65536, 131072, 16),
                 layers=("global",), queries=1),
        # Smaller instance of the paged mixed batch for profiler captures: the first 16
        # lengths of the B=256 draw (same seed), 16-position pages in a random order,
        # 3.2 GB of pools.
        Workload("paged_mixed_b16", "paged mixed batch, B=16, lognormal seq_lens (median 4096, "
                 "sigma 1) clipped to [1, 65536]; one sliding and one global call (profiling size)",
                 B=16, S=65536, seed=4, lengths=lengths_lognormal(4096, 1.0, 1, 65536, 16),
                 layers=("sliding", "global"), paged=True),
        # Smaller instance of the batched sliding shape for profiler captures: the same
        # bytes per call as sliding_b64_s32768 (every sequence reads its full 1024-position
        # window) with a 2 GB cache instead of 34 GB.
        Workload("sliding_b64_s2048", "slidingDecodeGQA batched, B=64, every seq_len 2048 "
                 "(profiling size)", B=64, S=2048, seed=5, lengths=lengths_fixed(2048, 64),
                 layers=("sliding",)),
    ]
}


def geometry(layer: str) -> dict:
    return dict(SLIDING if layer == "sliding" else GLOBAL)


# ----------------------------------------------------------------------------
# Case builders
# ----------------------------------------------------------------------------

def raw_projections(B: int, H: int, KVH: int, D: int, seed: int, device="cpu") -> dict:
    """Synthetic projection outputs for the decode-step producer: q_raw [B,H,D],
    k_raw, v_raw [B,KVH,D] drawn N(0,1) times a per-head scale in [0.2, 5.2), and
    the q_norm / k_norm weights [D]."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 16 + 7)
    scale = 0.2 + 5.0 * torch.rand((B, H, 1), generator=gen, device=device)
    q = (torch.randn((B, H, D), generator=gen, device=device) * scale).to(torch.bfloat16)
    k = (torch.randn((B, KVH, D), generator=gen, device=device) * scale[:, :KVH]).to(torch.bfloat16)
    v = (torch.randn((B, KVH, D), generator=gen, device=device) * 2.0).to(torch.bfloat16)
    return dict(q_raw=q, k_raw=k, v_raw=v, w_q=k_norm_weight_bf16(D, int(seed) * 16 + 8, device),
                w_k=k_norm_weight_bf16(D, int(seed) * 16 + 9, device))


def keqv_case(B: int, S: int, H: int, KVH: int, D: int, seq_lens, seed: int,
              device="cpu") -> dict:
    """q [B,H,D], the value cache v [B,S,KVH,D], k_norm weight w_k [D] (bf16) and
    seq_lens [B]: a single K=V cache (no k tensor)."""
    lens = torch.as_tensor(np.asarray(seq_lens, dtype=np.int32), device=device)
    return dict(
        q=rms_normalised_bf16((B, H, D), tensor_seed(seed, "q"), device),
        v=rms_normalised_bf16((B, S, KVH, D), tensor_seed(seed, "v"), device),
        w_k=k_norm_weight_bf16(D, tensor_seed(seed, "w_k"), device),
        seq_lens=lens,
    )


def contiguous_case(B: int, S: int, H: int, KVH: int, D: int, seq_lens, seed: int,
                    device="cpu") -> dict:
    """q [B,H,D], k/v [B,S,KVH,D] (bf16) and seq_lens [B] (int32, on ``device``)."""
    lens = torch.as_tensor(np.asarray(seq_lens, dtype=np.int32), device=device)
    return dict(
        q=rms_normalised_bf16((B, H, D), tensor_seed(seed, "q"), device),
        k=rms_normalised_bf16((B, S, KVH, D), tensor_seed(seed, "k"), device),
        v=rms_normalised_bf16((B, S, KVH, D), tensor_seed(seed, "v"), device),
        seq_lens=lens,
    )


def page_table(seq_lens, seed: int, max_pages: int | None = None,
               page_size: int = PAGE_SIZE, spare_pages: int = 0):
    """Seeded random page assignment.

    Returns (block_table int32 [B, max_pages], P).  Sequence b owns
    ceil(L_b / page_size) pages; the physical ids of all owned pages are a random
    permutation of [0, P) with P = total owned pages + ``spare_pages``.  Entries
    past a sequence's last page are -1.
    """
    lens = np.asarray(seq_lens, dtype=np.int64)
    need = (lens + page_size - 1) // page_size
    if max_pages is None:
        max_pages = max(1, int(need.max()) if len(need) else 1)
    total = int(need.sum())
    P = max(1, total + int(spare_pages))
    rng = np.random.default_rng(seed + 1_000_003)
    perm = rng.permutation(P).astype(np.int32)
    bt = np.full((len(lens), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, P


def paged_case(B: int, H: int, KVH: int, D: int, seq_lens, seed: int, max_pages: int | None = None,
               device="cpu", spare_pages: int = 0, table=None) -> dict:
    """q [B,H,D], page pools [P,16,KVH,D] (bf16), block_table [B,max_pages], seq_lens [B]."""
    if table is None:
        table = page_table(seq_lens, seed, max_pages, PAGE_SIZE, spare_pages)
    bt, P = table
    lens = torch.as_tensor(np.asarray(seq_lens, dtype=np.int32), device=device)
    return dict(
        q=rms_normalised_bf16((B, H, D), tensor_seed(seed, "q"), device),
        k_pages=rms_normalised_bf16((P, PAGE_SIZE, KVH, D), tensor_seed(seed, "k_pages"), device),
        v_pages=rms_normalised_bf16((P, PAGE_SIZE, KVH, D), tensor_seed(seed, "v_pages"), device),
        block_table=torch.as_tensor(bt, device=device),
        seq_lens=lens,
    )



def mq_case(B: int, T: int, S: int, H: int, KVH: int, D: int, seq_lens, seed: int,
            device="cpu") -> dict:
    """Multi-query step: q [B,T,H,D] (T new tokens per sequence), k/v [B,S,KVH,D]
    (bf16) already holding the new tokens' rows, seq_lens [B] (lengths after them)."""
    case = contiguous_case(B, S, H, KVH, D, seq_lens, seed, device)
    case["q"] = rms_normalised_bf16((B, T, H, D), tensor_seed(seed, "q"), device)
    return case


def paged_mq_case(B: int, T: int, H: int, KVH: int, D: int, seq_lens, seed: int,
                  max_pages: int | None = None, device="cpu", spare_pages: int = 0,
                  table=None) -> dict:
    """paged_case with a multi-query q [B,T,H,D]."""
    case = paged_case(B, H, KVH, D, seq_lens, seed, max_pages, device, spare_pages, table)
    case["q"] = rms_normalised_bf16((B, T, H, D), tensor_seed(seed, "q"), device)
    return case
