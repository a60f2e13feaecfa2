// Decode-step producer: the nodes ahead of the attention core for one new token
// per sequence.
//
// "Gemma 4 31B-it Text Architecture", decoder listing: Q = rope(q_norm(Q)),
// K = rope(k_norm(K_raw)), V = v_norm(V_raw) (V_raw = K_raw on global layers), and
// the new K/V are appended to the cache before attention.  gemma-4-31B Model Spec
// rows: attn.qk_norm, per head y = x / sqrt(mean(x^2) + 1e-6) * w; attn.v_norm, the
// same without w; attn.rope, pairs (i, i + D/2), i < n_rot, rotated by
// pos * theta^(-2i/D) (sliding: 128 pairs, theta 1e4; global: 64 pairs, theta 1e6).
// The token's position is L - 1 with L = seq_lens[b] counting the new token.
//
// Grid (sequence, group of 8 head vectors): each warp of a CTA takes one of the
// sequence's H + 2 KVH head vectors (q heads, then k, then v).  It loads its vector
// first; meanwhile the CTA's first n_rot threads reduce the angles pos * f_i mod
// 2 pi in fp64 (pos * f_i reaches 2.6e5 rad) and take sincosf of the remainder.
// Lane l holds the elements (i, i + D/2) of its pairs, so the rotation needs no
// shuffles.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace gqa {

constexpr int kPrepareThreads = 256;
constexpr int kPrepareMaxRot = 128;

struct PrepareParams {
    const __nv_bfloat16* q_raw;   // [B, H, D]
    const __nv_bfloat16* k_raw;   // [B, KVH, D]
    const __nv_bfloat16* v_raw;   // [B, KVH, D], or null: values = keys (v = v_norm(k_raw))
    const __nv_bfloat16* w_q;     // [D]
    const __nv_bfloat16* w_k;     // [D]
    const int32_t* seq_lens;      // [B], lengths after the append
    __nv_bfloat16* q_out;         // [B, H, D]
    __nv_bfloat16* k_cache;       // contiguous [B, rows, KVH, D] or pool [P, 16, KVH, D]; null if values = keys
    __nv_bfloat16* v_cache;       // same layout as k_cache
    const int32_t* block_table;   // [B, max_pages] (paged only)
    int B, H, KVH;
    int rows;                     // contiguous: rows per sequence
    int ring;                     // contiguous: 1 = position s at row s mod rows, 0 = row s
    int max_pages, num_pages;     // paged
    int n_rot;                    // rotated pairs
    double freq[kPrepareMaxRot];  // theta^(-2i/D), i < n_rot
};

template <int D, bool kPaged>
__global__ void __launch_bounds__(kPrepareThreads)
    gqa_prepare_kernel(const PrepareParams p) {
    constexpr int kHalf = D / 2;
    constexpr int kPer = kHalf / 32;   // elements per lane in each half
    __shared__ float2 cs[kPrepareMaxRot];

    // inputs may come from the kernel before this one in the stream
    ptx::grid_dependency_wait();
    ptx::allow_dependent_launch();

    const int b = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int vec = blockIdx.y * (kPrepareThreads / 32) + warp;   // head vector of this warp
    const int L = p.seq_lens[b];
    const int pos = L - 1;
    if (pos < 0) return;   // no new token
    // cache slot of the new token: null when it lies outside the cache
    size_t row_base = 0;   // element offset of (slot, kv head 0)
    bool have_slot = true;
    if (kPaged) {
        const int pg = pos >> 4;
        const int page = pg < p.max_pages ? p.block_table[static_cast<size_t>(b) * p.max_pages + pg] : -1;
        have_slot = page >= 0 && page < p.num_pages;
        row_base = (static_cast<size_t>(page) * 16 + (pos & 15)) * p.KVH * D;
    } else {
        const int row = p.ring ? pos % p.rows : pos;
        have_slot = p.ring || pos < p.rows;
        row_base = (static_cast<size_t>(b) * p.rows + row) * p.KVH * D;
    }

    const bool keqv = p.v_raw == nullptr;
    const int n_vec = p.H + 2 * p.KVH;   // q heads, then k heads, then v heads
    const bool is_q = vec < p.H;
    const bool is_k = !is_q && vec < p.H + p.KVH;
    const int kvh = is_q ? 0 : (is_k ? vec - p.H : vec - p.H - p.KVH);
    // does this warp write anything?  (no cache slot, or k on a K=V layer: no)
    const bool active = vec < n_vec && (is_q || (have_slot && !(is_k && keqv)));
    const __nv_bfloat16* src = nullptr;
    __nv_bfloat16* dst = nullptr;
    if (active) {
        if (is_q) {
            src = p.q_raw + (static_cast<size_t>(b) * p.H + vec) * D;
            dst = p.q_out + (static_cast<size_t>(b) * p.H + vec) * D;
        } else {
            const __nv_bfloat16* raw = (is_k || keqv) ? p.k_raw : p.v_raw;
            src = raw + (static_cast<size_t>(b) * p.KVH + kvh) * D;
            dst = (is_k ? p.k_cache : p.v_cache) + row_base + static_cast<size_t>(kvh) * D;
        }
    }
    // lane holds elements [kPer l, kPer l + kPer) of each half; loads first
    float x[2][kPer];
    if (active) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < kPer; e += 2) {
                const __nv_bfloat162 t =
                    *reinterpret_cast<const __nv_bfloat162*>(src + h * kHalf + kPer * lane + e);
                x[h][e] = __low2float(t);
                x[h][e + 1] = __high2float(t);
            }
    }
    if (tid < p.n_rot) {
        const double a = static_cast<double>(pos) * p.freq[tid];
        const double turns = rint(a * 0.15915494309189535);   // 1 / (2 pi)
        const double r = fma(-turns, 6.283185307179586, a);
        float sn, c;
        sincosf(static_cast<float>(r), &sn, &c);
        cs[tid] = make_float2(c, sn);
    }
    __syncthreads();
    if (!active) return;

    float ss = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < kPer; ++e) ss = fmaf(x[h][e], x[h][e], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = 1.0f / sqrtf(ss / static_cast<float>(D) + 1e-6f);
    const bool weighted = is_q || is_k;
    const __nv_bfloat16* w = is_q ? p.w_q : p.w_k;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            x[h][e] *= inv;
            if (weighted) x[h][e] *= __bfloat162float(w[h * kHalf + kPer * lane + e]);
        }
    if (weighted) {
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int i = kPer * lane + e;
            if (i < p.n_rot) {
                const float2 r = cs[i];
                const float x0 = x[0][e], x1 = x[1][e];
                x[0][e] = x0 * r.x - x1 * r.y;
                x[1][e] = x1 * r.x + x0 * r.y;
            }
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < kPer; e += 2)
            *reinterpret_cast<__nv_bfloat162*>(dst + h * kHalf + kPer * lane + e) =
                __floats2bfloat162_rn(x[h][e], x[h][e + 1]);
}

}  // namespace gqa
