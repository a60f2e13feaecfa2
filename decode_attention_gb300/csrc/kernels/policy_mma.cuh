// Tensor-core arithmetic for the decode attention core: the two contractions
// (scores Q K^T and the weighted sum P V) run as warp-level bf16 mma
// (m16n8k16, fp32 accumulate) on tiles staged in shared memory.
//
// Instantiated for decodeGQA (g = 8 query heads per KV head, D = 512) and for
// slidingDecodeGQA (g = 2, D = 256), the two attn.core rows of the gemma-4-31B
// Model Spec ("Compute-graph nodes").  The g heads of a KV head fill rows
// 0..g-1 of the 16-row A operand; the remaining rows are zero.  Even with most
// rows idle the tensor pipe does the arithmetic in a few instructions per
// position, where the CUDA cores would spend ~25 per position per head pair on
// unpacking and FMAs.
//
// Per tile of 32 positions and consumer warp w (of 8):
//   scores  S[h, pos] = Q[h, :] . K[pos, :] for positions [8(w%4), 8(w%4)+8) and
//           the half (w/4) of the head dimension (A = Q from registers, B = K
//           rows via ldmatrix); the two half sums go to shared memory in log2
//           units;
//   softmax every warp reads all 32 scores of its heads, so all warps hold the
//           same running max/normaliser;
//   P.V     O[h, d] += P[h, pos] V[pos, d] for the warp's D/8-wide slice of d
//           (B = V rows via ldmatrix.trans).  P is split into bf16 hi + lo parts
//           placed in rows 0-7 and 8-15 of the A operand, so one mma applies
//           P to ~16 significant bits at no extra cost; O = rows 0-7 + rows 8-15.
// K/V rows outside the valid range of a tile are masked: scores to -inf, the
// V fragments to 0 (0 * NaN would poison the sum).
#pragma once

#include "decode_kernel.cuh"

namespace gqa {

template <int kG, int kD, int kStages>
struct MmaPolicy {
    static constexpr int G = kG, D = kD, TP = 32, STAGES = kStages, NC = 8;
    static_assert(G >= 1 && G <= 8, "heads fill rows 0..G-1 of the A operand");
    static constexpr int kDSlice = D / NC;          // output dims per warp
    static constexpr int kNTiles = kDSlice / 8;     // n-tiles of 8 dims per warp
    static_assert(kNTiles % 2 == 0, "n-tiles are loaded in pairs");
    static constexpr int kKSteps = D / 16 / 2;      // k-steps over half of the head dim
    static constexpr int kSStride = 40;             // padded row of the score tile
    static constexpr bool kSwizzle128 = true;       // ldmatrix needs the 128-byte swizzle
    static constexpr int kBoxRows = 16;             // TMA box height on a contiguous cache
    // every warp holds the full running max/normaliser and its own slice of the
    // output, so results are stored straight from registers
    static constexpr bool kDirectEpilogue = true;
    // split segments are merged by the combine kernel (16 KB partials: its many blocks
    // share the merges better than one CTA per segment)
    static constexpr bool kMergeInKernel = false;
    static constexpr bool kKeqV = false;   // separate K and V tiles

    struct Scratch {
        alignas(16) float S[2][2][G][kSStride];   // [tile parity][half of D][head][position]
    };

    struct State {
        uint32_t qa[kKSteps][2];   // A fragments of Q (rows 0-7) for this warp's half of D
        float acc[kNTiles][4];     // rows gid (hi part) and gid+8 (lo part)
        float m;                   // running max of head gid (log2 units)
        float l;                   // this lane's share of the normaliser of head gid
    };

    __device__ static __forceinline__ void begin(State& st, const __nv_bfloat16* q_heads, int warp,
                                                 int lane) {
        const int gid = lane >> 2, t4 = lane & 3;
        const bool real = gid < G;   // rows G..7 of A are zero
        // q_heads: the g query heads of the KV head, [G][D] bf16 in shared memory
        const uint32_t* qrow =
            reinterpret_cast<const uint32_t*>(q_heads + (real ? gid : 0) * D + (warp >> 2) * (D / 2));
#pragma unroll
        for (int kk = 0; kk < kKSteps; ++kk) {
            st.qa[kk][0] = real ? qrow[(kk * 16 + 2 * t4) / 2] : 0u;
            st.qa[kk][1] = real ? qrow[(kk * 16 + 8 + 2 * t4) / 2] : 0u;
        }
#pragma unroll
        for (int n = 0; n < kNTiles; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) st.acc[n][e] = 0.0f;
        st.m = -INFINITY;
        st.l = 0.0f;
    }

    // Byte address of the 16-byte unit (row, 8-element column group `grp`) of a tile.
    __device__ static __forceinline__ uint32_t unit_addr(uint32_t tile, int row, int grp) {
        const int box = row >> 4, r = row & 15;
        const int chunk = grp >> 3, unit = grp & 7;
        return tile + box * (16 * D * 2) + chunk * kChunkBytes + r * 128 + ((unit ^ (r & 7)) << 4);
    }

    __device__ static __forceinline__ uint32_t pack_bf16(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }

    __device__ static __forceinline__ void tile(State& st, uint32_t k_tile, uint32_t v_tile, int vlo,
                                                int vhi, Scratch& sc, uint32_t t_idx, int warp,
                                                int lane) {
        const int gid = lane >> 2, t4 = lane & 3;
        float(*S)[G][kSStride] = sc.S[t_idx & 1];

        // ---- half scores for positions [8(w%4), 8(w%4)+8), dims [256(w/4), +256) ----
        {
            float c[2][4];   // two independent accumulation chains
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) c[i][e] = 0.0f;
            const int row = (warp & 3) * 8 + (lane & 7);
            const int mat = lane >> 3;
            const int grp0 = (warp >> 2) * (D / 2 / 8);
#pragma unroll
            for (int k2 = 0; k2 < kKSteps / 2; ++k2) {
                uint32_t b0, b1, b2, b3;
                ptx::ldmatrix_x4(unit_addr(k_tile, row, grp0 + k2 * 4 + mat), b0, b1, b2, b3);
                ptx::mma_bf16_16816(c[0], st.qa[2 * k2][0], 0u, st.qa[2 * k2][1], 0u, b0,
                                    b1);
                ptx::mma_bf16_16816(c[1], st.qa[2 * k2 + 1][0], 0u,
                                    st.qa[2 * k2 + 1][1], 0u, b2, b3);
            }
            const int pos = (warp & 3) * 8 + 2 * t4;
            float s0 = (c[0][0] + c[1][0]) * kLog2e;
            float s1 = (c[0][1] + c[1][1]) * kLog2e;
            if (pos < vlo || pos >= vhi) s0 = -INFINITY;
            if (pos + 1 < vlo || pos + 1 >= vhi) s1 = -INFINITY;
            if (gid < G) *reinterpret_cast<float2*>(&S[warp >> 2][gid][pos]) = make_float2(s0, s1);
        }
        ptx::named_barrier_sync(1, NC * 32);
        softmax_pv(st, S, v_tile, vlo, vhi, warp, lane);
    }

    // Online softmax over the 32 half-score pairs of tile S (heads in rows 0..G-1),
    // then P.V for this warp's D/8-wide slice of the output.  St holds acc, m, l.
    template <class St>
    __device__ static __forceinline__ void softmax_pv(St& st, const float (*S)[G][kSStride],
                                                      uint32_t v_tile, int vlo, int vhi, int warp,
                                                      int lane) {
        const int gid = lane >> 2, t4 = lane & 3;
        // ---- online softmax over the 32 positions of head gid (rows >= G stay empty) ----
        float sv[2][4];
        const int hrow = gid < G ? gid : 0;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const float2 x0 = *reinterpret_cast<const float2*>(&S[0][hrow][16 * ks + 2 * t4]);
            const float2 x1 = *reinterpret_cast<const float2*>(&S[1][hrow][16 * ks + 2 * t4]);
            const float2 y0 = *reinterpret_cast<const float2*>(&S[0][hrow][16 * ks + 8 + 2 * t4]);
            const float2 y1 = *reinterpret_cast<const float2*>(&S[1][hrow][16 * ks + 8 + 2 * t4]);
            const bool real = gid < G;
            sv[ks][0] = real ? x0.x + x1.x : -INFINITY;
            sv[ks][1] = real ? x0.y + x1.y : -INFINITY;
            sv[ks][2] = real ? y0.x + y1.x : -INFINITY;
            sv[ks][3] = real ? y0.y + y1.y : -INFINITY;
        }
        float tmax = -INFINITY;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
#pragma unroll
            for (int e = 0; e < 4; ++e) tmax = fmaxf(tmax, sv[ks][e]);
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float m_new = fmaxf(st.m, tmax);
        const bool none = (m_new == -INFINITY);
        const float alpha = none ? 1.0f : exp2f(st.m - m_new);
        uint32_t a[2][4];
        float psum = 0.0f;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            float pv[4], hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                pv[e] = none ? 0.0f : exp2f(sv[ks][e] - m_new);
                psum += pv[e];
                hi[e] = __bfloat162float(__float2bfloat16_rn(pv[e]));
                lo[e] = pv[e] - hi[e];
            }
            a[ks][0] = pack_bf16(hi[0], hi[1]);   // row gid,   cols 2t, 2t+1
            a[ks][1] = pack_bf16(lo[0], lo[1]);   // row gid+8, cols 2t, 2t+1
            a[ks][2] = pack_bf16(hi[2], hi[3]);   // row gid,   cols 2t+8, 2t+9
            a[ks][3] = pack_bf16(lo[2], lo[3]);   // row gid+8, cols 2t+8, 2t+9
        }
        st.l = st.l * alpha + psum;
        st.m = m_new;
#pragma unroll
        for (int n = 0; n < kNTiles; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) st.acc[n][e] *= alpha;

        // ---- P.V for dims [64w, 64w+64) ----
        const bool partial = (vlo > 0) || (vhi < TP);
        const int mat = lane >> 3, r8 = lane & 7;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            // validity of the positions this lane's B registers hold
            const int pa = 16 * ks + 2 * t4, pb = pa + 8;
            uint32_t mask_a = 0xffffffffu, mask_b = 0xffffffffu;
            if (partial) {
                mask_a = ((pa >= vlo && pa < vhi) ? 0x0000ffffu : 0u) |
                         ((pa + 1 >= vlo && pa + 1 < vhi) ? 0xffff0000u : 0u);
                mask_b = ((pb >= vlo && pb < vhi) ? 0x0000ffffu : 0u) |
                         ((pb + 1 >= vlo && pb + 1 < vhi) ? 0xffff0000u : 0u);
            }
            const int row = 16 * ks + (mat & 1) * 8 + r8;
#pragma unroll
            for (int jj = 0; jj < kNTiles / 2; ++jj) {
                const int grp = (warp * kDSlice + 16 * jj) / 8 + (mat >> 1);
                uint32_t b0, b1, b2, b3;
                ptx::ldmatrix_x4_trans(unit_addr(v_tile, row, grp), b0, b1, b2, b3);
                b0 &= mask_a;
                b1 &= mask_b;
                b2 &= mask_a;
                b3 &= mask_b;
                ptx::mma_bf16_16816(st.acc[2 * jj], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b0, b1);
                ptx::mma_bf16_16816(st.acc[2 * jj + 1], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b2,
                                    b3);
            }
        }
    }

    // The piece's result for head gid, dims [warp D/8, +D/8) of this warp: the
    // normalised output (slot < 0; the piece is the whole segment) or the partial
    // (acc, m, l) at workspace slot `slot`.  A bad page turns it into NaN.
    template <class St>
    __device__ static __forceinline__ void store(const St& st, const DecodeParams& p,
                                                 size_t out_base, int slot, bool bad, int warp,
                                                 int lane) {
        const int gid = lane >> 2, t4 = lane & 3;
        float l = st.l;
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if (gid >= G) return;
        const float nan = __uint_as_float(0x7fc00000u);
        if (slot < 0) {
            const float inv = 1.0f / l;
#pragma unroll
            for (int n = 0; n < kNTiles; ++n) {
                const int d = warp * kDSlice + n * 8 + 2 * t4;
                const float x = (st.acc[n][0] + st.acc[n][2]) * inv;
                const float y = (st.acc[n][1] + st.acc[n][3]) * inv;
                store_out2(p, out_base + gid * D + d, bad ? nan : x, bad ? nan : y);
            }
        } else {
            float* wacc = p.ws_acc + static_cast<size_t>(slot) * G * D + gid * D;
#pragma unroll
            for (int n = 0; n < kNTiles; ++n) {
                const int d = warp * kDSlice + n * 8 + 2 * t4;
                *reinterpret_cast<float2*>(wacc + d) =
                    bad ? make_float2(nan, nan)
                        : make_float2(st.acc[n][0] + st.acc[n][2], st.acc[n][1] + st.acc[n][3]);
            }
            if (warp == 0 && t4 == 0) {
                float* ml = p.ws_ml + (static_cast<size_t>(slot) * G + gid) * 2;
                ml[0] = bad ? 0.0f : st.m;
                ml[1] = bad ? nan : l;
            }
        }
    }

    __device__ static __forceinline__ void end(State& st, float* acc_out, float* m_out, float* l_out,
                                               Scratch& sc, int warp, int lane) {
        (void)sc;
        const int gid = lane >> 2, t4 = lane & 3;
        float l = st.l;
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if (gid < G) {
#pragma unroll
            for (int n = 0; n < kNTiles; ++n) {
                const int d = warp * kDSlice + n * 8 + 2 * t4;
                *reinterpret_cast<float2*>(&acc_out[gid * D + d]) =
                    make_float2(st.acc[n][0] + st.acc[n][2], st.acc[n][1] + st.acc[n][3]);
            }
        }
        if (warp == 0 && t4 == 0 && gid < G) {
            m_out[gid] = st.m;
            l_out[gid] = l;
        }
        ptx::named_barrier_sync(1, NC * 32);
    }
};

using GlobalMma = MmaPolicy<8, 512, 3>;    // decodeGQA
using SlidingMma = MmaPolicy<2, 256, 6>;   // slidingDecodeGQA

}  // namespace gqa
