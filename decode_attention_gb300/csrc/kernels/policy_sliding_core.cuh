// CUDA-core arithmetic for slidingDecodeGQA (g = 2 query heads per KV head,
// D = 256), gemma-4-31B Model Spec, "Compute-graph nodes", attn.core row with
// Op Spec slidingDecodeGQA.
//
// At 2 heads per KV row the work is 1 FMA per byte of K/V (scores + P.V), far
// below what the CUDA cores sustain at HBM rate, so no tensor core is used.
//
// Shared-memory tiles are plain row-major [position][256] bf16 (no swizzle):
// lane l reads bytes [16l, 16l+16) of a row, so a row is one conflict-free
// 512-byte read, and the TMA moves whole 512-byte rows (one 32-position box per
// tensor and tile on a contiguous cache).
//
// Layout per consumer warp w (of 8) and tile of 64 positions: the warp owns the
// 8 positions [8w, 8w+8); lane l owns head-dim elements [8l, 8l+8) of every
// row.  The 16 dot products of a tile (8 positions x 2 heads) are reduced
// across lanes with a reduce-scatter butterfly (15 shuffles), after which lane
// l holds the score of position l/4, head (l/2)%2.  Each warp keeps its own
// online-softmax state (m, l, acc); the 8 states are merged through shared
// memory when a piece ends.  Two warps per scheduler, and 8 positions per warp
// per tile, keep the shuffle and shared-memory latency chains overlapped.
// Scores are kept in log2 units (q is pre-multiplied by log2(e)), so every
// exponential is exp2.  The products run on packed fp32 pairs (fma.rn.f32x2: the
// two halves of a bf16x2 word, widened exactly), two fp32 FMAs per instruction;
// each score sums its even and its odd products in two chains.
#pragma once

#include "decode_kernel.cuh"

namespace gqa {

struct SlidingCore {
    static constexpr int G = 2, D = 256, TP = 64, STAGES = 3, NC = 8;
    static constexpr int kPosPerWarp = TP / NC;   // 8
    static constexpr bool kSwizzle128 = false;    // plain [position][D] tiles
    static constexpr int kBoxRows = 64;           // TMA box height on a contiguous cache
    static constexpr bool kDirectEpilogue = false;   // warps merge through shared memory
    // split segments are merged in the main kernel (small partials), not by the
    // combine kernel
    static constexpr bool kMergeInKernel = true;
    static constexpr bool kKeqV = false;   // separate K and V tiles
    static_assert(kPosPerWarp == 8, "reduce-scatter below assumes 8 positions x 2 heads");

    struct Scratch {
        alignas(16) float wacc[NC][G][D];   // float4 stores
        float wm[NC][G];
        float wl[NC][G];
    };

    struct State {
        uint64_t q[G][4];     // q[h][8*lane + 2e, + 2e + 1] * log2(e), packed fp32 pairs
        uint64_t acc[G][4];   // unnormalised output, dims 8*lane + 2e, + 2e + 1 (pairs)
        float m[G];           // running max (log2 units), same in every lane
        float l[G];           // running normaliser, same in every lane
    };

    __device__ static __forceinline__ void begin(State& st, const __nv_bfloat16* q_heads, int warp,
                                                 int lane) {
        (void)warp;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const uint4 raw = *reinterpret_cast<const uint4*>(q_heads + h * D + lane * 8);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                st.q[h][e] = ptx::f2_pack(bf16lo(w[e]) * kLog2e, bf16hi(w[e]) * kLog2e);
                st.acc[h][e] = ptx::f2_pack(0.0f, 0.0f);
            }
            st.m[h] = -INFINITY;
            st.l[h] = 0.0f;
        }
    }

    // Address of this lane's 16 bytes of row `row` of a tile.
    __device__ static __forceinline__ uint32_t row_addr(uint32_t tile, int row, int lane) {
        return tile + row * (D * 2) + lane * 16;
    }

    __device__ static __forceinline__ void tile(State& st, uint32_t k_tile, uint32_t v_tile, int vlo,
                                                int vhi, Scratch& sc, uint32_t t_idx, int warp,
                                                int lane) {
        (void)sc;
        (void)t_idx;
        const int row0 = warp * kPosPerWarp;

        // ---- scores: 8 positions x 2 heads, partial sums over this lane's 8 dims ----
        float v[16];
#pragma unroll
        for (int j = 0; j < kPosPerWarp; ++j) {
            const uint4 raw = ptx::lds128(row_addr(k_tile, row0 + j, lane));
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
            // even and odd products of each head in the two halves of a pair
            uint64_t s0 = ptx::f2_mul(st.q[0][0], ptx::f2_from_bf16x2(w[0]));
            uint64_t s1 = ptx::f2_mul(st.q[1][0], ptx::f2_from_bf16x2(w[0]));
#pragma unroll
            for (int e = 1; e < 4; ++e) {
                const uint64_t kk = ptx::f2_from_bf16x2(w[e]);
                s0 = ptx::f2_fma(st.q[0][e], kk, s0);
                s1 = ptx::f2_fma(st.q[1][e], kk, s1);
            }
            const float2 a0 = ptx::f2_unpack(s0), a1 = ptx::f2_unpack(s1);
            v[2 * j] = a0.x + a0.y;
            v[2 * j + 1] = a1.x + a1.y;
        }
        // ---- reduce-scatter: lane l ends with the full score of index l >> 1 ----
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const bool up = lane & 16;
            const float send = up ? v[i] : v[i + 8];
            const float keep = up ? v[i + 8] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool up = lane & 8;
            const float send = up ? v[i] : v[i + 4];
            const float keep = up ? v[i + 4] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const bool up = lane & 4;
            const float send = up ? v[i] : v[i + 2];
            const float keep = up ? v[i + 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        {
            const bool up = lane & 2;
            const float send = up ? v[0] : v[1];
            const float keep = up ? v[1] : v[0];
            v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        float s = v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
        // lane holds position row0 + (lane >> 2), head (lane >> 1) & 1
        const int my_pos = row0 + (lane >> 2);
        const int my_head = (lane >> 1) & 1;
        if (my_pos < vlo || my_pos >= vhi) s = -INFINITY;

        // ---- online softmax (per head; lanes with equal bit 1 share a head) ----
        float tmax = s;
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
        const float tmax_other = __shfl_xor_sync(0xffffffffu, tmax, 2);
        const float tm0 = my_head == 0 ? tmax : tmax_other;
        const float tm1 = my_head == 0 ? tmax_other : tmax;
        const float mn0 = fmaxf(st.m[0], tm0), mn1 = fmaxf(st.m[1], tm1);
        const float a0 = (mn0 == -INFINITY) ? 1.0f : exp2f(st.m[0] - mn0);
        const float a1 = (mn1 == -INFINITY) ? 1.0f : exp2f(st.m[1] - mn1);
        const float m_mine = my_head == 0 ? mn0 : mn1;
        const float pr = (s == -INFINITY) ? 0.0f : exp2f(s - m_mine);
        float psum = pr;
        psum += __shfl_xor_sync(0xffffffffu, psum, 4);
        psum += __shfl_xor_sync(0xffffffffu, psum, 8);
        psum += __shfl_xor_sync(0xffffffffu, psum, 16);
        const float psum_other = __shfl_xor_sync(0xffffffffu, psum, 2);
        const float ps0 = my_head == 0 ? psum : psum_other;
        const float ps1 = my_head == 0 ? psum_other : psum;
        st.l[0] = st.l[0] * a0 + ps0;
        st.l[1] = st.l[1] * a1 + ps1;
        st.m[0] = mn0;
        st.m[1] = mn1;

        // ---- P.V ----
        {
            const uint64_t aa0 = ptx::f2_pack(a0, a0), aa1 = ptx::f2_pack(a1, a1);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                st.acc[0][e] = ptx::f2_mul(st.acc[0][e], aa0);
                st.acc[1][e] = ptx::f2_mul(st.acc[1][e], aa1);
            }
        }
#pragma unroll
        for (int j = 0; j < kPosPerWarp; ++j) {
            const float p0 = __shfl_sync(0xffffffffu, pr, j * 4 + 0);
            const float p1 = __shfl_sync(0xffffffffu, pr, j * 4 + 2);
            uint4 raw = ptx::lds128(row_addr(v_tile, row0 + j, lane));
            const bool valid = (row0 + j >= vlo) && (row0 + j < vhi);
            if (!valid) raw = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
            const uint64_t pp0 = ptx::f2_pack(p0, p0), pp1 = ptx::f2_pack(p1, p1);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint64_t xx = ptx::f2_from_bf16x2(w[e]);
                st.acc[0][e] = ptx::f2_fma(pp0, xx, st.acc[0][e]);
                st.acc[1][e] = ptx::f2_fma(pp1, xx, st.acc[1][e]);
            }
        }
    }

    // Merge the 4 warps' states into acc_out[G][D], m_out[G], l_out[G].
    __device__ static __forceinline__ void end(State& st, float* acc_out, float* m_out, float* l_out,
                                               Scratch& sc, int warp, int lane) {
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                sc.wm[warp][h] = st.m[h];
                sc.wl[warp][h] = st.l[h];
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float4* dst = reinterpret_cast<float4*>(&sc.wacc[warp][h][lane * 8]);
            const float2 x0 = ptx::f2_unpack(st.acc[h][0]), x1 = ptx::f2_unpack(st.acc[h][1]);
            const float2 x2 = ptx::f2_unpack(st.acc[h][2]), x3 = ptx::f2_unpack(st.acc[h][3]);
            dst[0] = make_float4(x0.x, x0.y, x1.x, x1.y);
            dst[1] = make_float4(x2.x, x2.y, x3.x, x3.y);
        }
        ptx::named_barrier_sync(1, NC * 32);
        const int tid = warp * 32 + lane;
        for (int i = tid; i < G * D; i += NC * 32) {
            const int h = i / D, d = i % D;
            float M = sc.wm[0][h];
#pragma unroll
            for (int w = 1; w < NC; ++w) M = fmaxf(M, sc.wm[w][h]);
            float a = 0.0f, l = 0.0f;
#pragma unroll
            for (int w = 0; w < NC; ++w) {
                const float f = (sc.wm[w][h] == -INFINITY) ? 0.0f : exp2f(sc.wm[w][h] - M);
                a = fmaf(f, sc.wacc[w][h][d], a);
                l = fmaf(f, sc.wl[w][h], l);
            }
            acc_out[i] = a;
            if (d == 0) {
                m_out[h] = M;
                l_out[h] = l;
            }
        }
        ptx::named_barrier_sync(1, NC * 32);
    }
};

}  // namespace gqa
