// Tensor-core arithmetic for decodeGQA over a single K=V cache.
//
// On the global layers keys and values come from the same projection: V =
// v_norm(K_raw) and K = rope(k_norm(K_raw)) (gemma-4-31B Model Spec, "What to
// watch for"; decoder listing of the "Gemma 4 31B-it Text Architecture" page).
// Both norms divide K_raw by the same root mean square, so with the cached value
// row v at position s and the layer's k_norm weight w,
//     k = rope(w * v, s),
// where the global layers' rope (Model Spec, `attn.rope` row for layers 5, 11,
// ..., 59) rotates the pairs (i, i + 256), i < 64, by s * 1e6^(-2i/512) and
// leaves every other coordinate alone.  Only v is cached and read, half the
// bytes of separate K and V.
//
// Scores per tile of 32 positions, warp w (of 8) owning positions 8(w%4)..+8 and
// the half h = w/4 of the head dimension:
//   unrotated dims [256h + 64, 256h + 256): <q * w, v> with B = the v tile itself
//       and A = q * w split into bf16 hi (rows 0-7) and lo (rows 8-15), so the
//       sum of the two row groups carries ~16 significant bits (A is staged in
//       shared memory once per piece and read with ldmatrix: 48 more registers
//       per thread would not fit the 168 a 9-warp CTA can have);
//   rotated dims [256h, 256h + 64): <q, k_rot> with k_rot derived for the tile in
//       shared memory (bf16 hi and lo tiles, two mma each).
// Rotation angles: a helper warp computes, for every tile a few stages ahead,
// cos/sin of pos0 * f_i (reduced mod 2 pi in fp64, then sincosf); the consumers
// combine them with cos/sin of j * f_i for row j (a table built once per CTA) by
// the angle-addition formulas.  The softmax and P.V are those of MmaPolicy, on
// the v tile.
#pragma once

#include "decode_kernel.cuh"
#include "policy_mma.cuh"

namespace gqa {

struct MmaKeqV {
    using Base = MmaPolicy<8, 512, 4>;
    static constexpr int G = 8, D = 512, TP = 32, STAGES = 4, NC = 8;
    static constexpr int kDSlice = Base::kDSlice, kNTiles = Base::kNTiles;
    static constexpr int kSStride = Base::kSStride;
    static constexpr bool kSwizzle128 = true;
    static constexpr int kBoxRows = 16;
    static constexpr bool kDirectEpilogue = true;
    // split segments are merged by the combine kernel (16 KB partials: its many blocks
    // share the merges better than one CTA per segment)
    static constexpr bool kMergeInKernel = false;
    static constexpr bool kKeqV = true;              // only the value tile is loaded
    static constexpr int kRot = 64;                  // rotated pairs (i, i + D/2), i < kRot
    static constexpr int kHalf = D / 2;
    static constexpr int kRotDims = 2 * kRot;        // columns of the derived tile
    static constexpr int kPlainSteps = (kHalf - kRot) / 16;   // 12 k-steps per half
    static constexpr int kRotSteps = kRot / 16;               // 4 k-steps per half
    static constexpr int kRotTileBytes = TP * kRotDims * 2;   // one bf16 tile, 8 KB
    static constexpr int kPlainCols = 2 * (kHalf - kRot);     // 384 unrotated dims
    static constexpr int kQtStride = kPlainCols * 2 + 16;     // padded row: ldmatrix rows hit distinct banks
    static_assert(NC * 32 == TP * (kRot / 8), "one thread per (row, 8 pairs) of the derived tile");

    struct Scratch {
        alignas(16) float S[2][2][G][kSStride];       // [tile parity][half of D][head][position]
        alignas(128) uint8_t krot[2][kRotTileBytes];  // derived rotated keys: [hi, lo]
        alignas(128) uint8_t qt[16 * kQtStride];      // q * w of the piece: rows 0-7 hi, 8-15 lo
        alignas(16) float2 cs_base[STAGES][kRot];     // cos, sin of pos0 * f_i, per stage
        alignas(16) float2 cs_step[TP][kRot];         // cos, sin of j * f_i
        alignas(16) float w[D];                       // k_norm weight
    };

    struct State {
        uint32_t qr[kRotSteps][2];     // A fragments of q (rows 0-7), rotated dims
        float acc[kNTiles][4];         // rows gid (hi part) and gid+8 (lo part) of P.V
        float m;                       // running max of head gid (log2 units)
        float l;                       // this lane's share of the normaliser of head gid
    };

    // Byte address of 16-byte unit `grp` of `row` in a derived tile: the swizzled
    // [box of 16 rows][64-column chunk][16 rows][128 B] layout of the K/V tiles.
    __device__ static __forceinline__ uint32_t rot_addr(uint32_t tile, int row, int grp) {
        const int box = row >> 4, r = row & 15;
        const int chunk = grp >> 3, unit = grp & 7;
        return tile + box * (16 * kRotDims * 2) + chunk * kChunkBytes + r * 128 +
               ((unit ^ (r & 7)) << 4);
    }

    // Once per CTA (all consumer threads, then a consumer barrier): the weight and the
    // table of cos/sin(j f_i).  Only the consumers read them, after that barrier.
    __device__ static __forceinline__ void init(Scratch& sc, const DecodeParams& p, int tid) {
        constexpr int kThreads = NC * 32;
        for (int i = tid; i < D; i += kThreads) sc.w[i] = __bfloat162float(p.w_k[i]);
        for (int e = tid; e < TP * kRot; e += kThreads) {
            const int j = e / kRot, i = e - (e / kRot) * kRot;
            const double f = p.rope_freq[i];
            float sn, cs;
            sincosf(static_cast<float>(static_cast<double>(j) * f), &sn, &cs);   // |angle| < 32
            sc.cs_step[j][i] = make_float2(cs, sn);
        }
        ptx::named_barrier_sync(1, kThreads);
    }

    // Column of unrotated dim d (256h + 64 <= d < 256h + 256) in the staged q * w tile.
    __device__ static __forceinline__ int plain_col(int d) {
        return (d / kHalf) * (kHalf - kRot) + (d % kHalf) - kRot;
    }

    // Every consumer warp calls this at the first tile of a piece.  The staged q * w
    // is written cooperatively (each thread its own 12 columns); it is read only
    // after the tile's first consumer barrier, and the previous piece's readers have
    // all passed that piece's last score barrier.
    __device__ static __forceinline__ void begin(State& st, const __nv_bfloat16* q_heads,
                                                 Scratch& sc, int warp, int lane) {
        const int gid = lane >> 2, t4 = lane & 3;
        const int h = warp >> 2;
        const int tid = warp * 32 + lane;
        {
            // thread tid: head tid / 32, unrotated dims of both halves, 12 at stride 32
            const int head = tid >> 5, c0 = tid & 31;
            const __nv_bfloat16* qrow = q_heads + head * D;
            uint8_t* hi_row = sc.qt + head * kQtStride;
            uint8_t* lo_row = sc.qt + (head + 8) * kQtStride;
#pragma unroll
            for (int k = 0; k < kPlainCols / 32; ++k) {
                const int col = c0 + 32 * k;
                const int d = (col / (kHalf - kRot)) * kHalf + kRot + col % (kHalf - kRot);
                const float x = __bfloat162float(qrow[d]) * sc.w[d];
                const __nv_bfloat16 hi = __float2bfloat16_rn(x);
                const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
                reinterpret_cast<__nv_bfloat16*>(hi_row)[col] = hi;
                reinterpret_cast<__nv_bfloat16*>(lo_row)[col] = lo;
            }
        }
        const __nv_bfloat16* qrow = q_heads + gid * D;   // G = 8: every row is a head
        // rotated dims of this half: q itself (its weight is in the derived keys)
        const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow);
#pragma unroll
        for (int ks = 0; ks < kRotSteps; ++ks) {
            const int d = h * kHalf + ks * 16 + 2 * t4;
            st.qr[ks][0] = q32[d / 2];
            st.qr[ks][1] = q32[(d + 8) / 2];
        }
#pragma unroll
        for (int n = 0; n < kNTiles; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) st.acc[n][e] = 0.0f;
        st.m = -INFINITY;
        st.l = 0.0f;
    }

    // Helper warp: cos/sin of pos0 * f_i for the tile in stage `stage`, lane l taking
    // i = 2l and 2l + 1 (f = f_2l, f_2l+1, which the lane holds in registers: the helper
    // runs from the first tile on, before the consumers' one-time setup has finished).
    // pos0 * f_i reaches 2.6e5 rad, far past fp32's exact range, so the angle is reduced
    // mod 2 pi in fp64 first.
    __device__ static __forceinline__ void tile_angles(Scratch& sc, int stage, int pos0,
                                                       const double (&f)[2], int lane) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int i = 2 * lane + t;
            const double a = static_cast<double>(pos0) * f[t];
            const double turns = rint(a * 0.15915494309189535);   // 1 / (2 pi)
            const double r = fma(-turns, 6.283185307179586, a);
            float sn, cs;
            sincosf(static_cast<float>(r), &sn, &cs);
            sc.cs_base[stage][i] = make_float2(cs, sn);
        }
    }

    // Derived rotated keys of the tile: thread (lane p, row group g) takes the pairs
    // i = 2p, 2p + 1 in rows g, g + 8, g + 16, g + 24, so the lanes of a warp read and
    // write consecutive words of one row (no bank conflicts).
    __device__ static __forceinline__ void derive_keys(Scratch& sc, uint32_t v_tile, int stage,
                                                       int tid) {
        constexpr int kThreads = NC * 32;
        const int p = tid & 31, g = tid >> 5;
        const int i = 2 * p;
        const float4 base = *reinterpret_cast<const float4*>(&sc.cs_base[stage][i]);   // i, i + 1
        const float2 w_lo = *reinterpret_cast<const float2*>(&sc.w[i]);
        const float2 w_hi = *reinterpret_cast<const float2*>(&sc.w[kHalf + i]);
        const uint32_t hi_tile = ptx::smem_addr(&sc.krot[0][0]);
        const uint32_t lo_tile = ptx::smem_addr(&sc.krot[1][0]);
        const int byte_in_unit = (i & 7) * 2;
#pragma unroll
        for (int k = 0; k < TP / 8; ++k) {
            const int j = g + 8 * k;
            const uint32_t vx = ptx::lds32(Base::unit_addr(v_tile, j, i / 8) + byte_in_unit);
            const uint32_t vy = ptx::lds32(Base::unit_addr(v_tile, j, (kHalf + i) / 8) + byte_in_unit);
            const float4 step = *reinterpret_cast<const float4*>(&sc.cs_step[j][i]);
            float r0[2], r1[2];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const float bc = t == 0 ? base.x : base.z, bs = t == 0 ? base.y : base.w;
                const float sc_ = t == 0 ? step.x : step.z, ss = t == 0 ? step.y : step.w;
                const float c = bc * sc_ - bs * ss;   // cos((pos0 + j) f_i)
                const float sn = bs * sc_ + bc * ss;  // sin((pos0 + j) f_i)
                const float x = (t == 0 ? w_lo.x : w_lo.y) * (t == 0 ? bf16lo(vx) : bf16hi(vx));
                const float y = (t == 0 ? w_hi.x : w_hi.y) * (t == 0 ? bf16lo(vy) : bf16hi(vy));
                r0[t] = x * c - y * sn;
                r1[t] = y * c + x * sn;
            }
            const __nv_bfloat162 h0 = __floats2bfloat162_rn(r0[0], r0[1]);
            const __nv_bfloat162 h1 = __floats2bfloat162_rn(r1[0], r1[1]);
            const __nv_bfloat162 l0 =
                __floats2bfloat162_rn(r0[0] - __low2float(h0), r0[1] - __high2float(h0));
            const __nv_bfloat162 l1 =
                __floats2bfloat162_rn(r1[0] - __low2float(h1), r1[1] - __high2float(h1));
            // columns: m = i for the first coordinates, 64 + i for the second
            ptx::sts32(rot_addr(hi_tile, j, i / 8) + byte_in_unit, *reinterpret_cast<const uint32_t*>(&h0));
            ptx::sts32(rot_addr(lo_tile, j, i / 8) + byte_in_unit, *reinterpret_cast<const uint32_t*>(&l0));
            ptx::sts32(rot_addr(hi_tile, j, (kRot + i) / 8) + byte_in_unit,
                       *reinterpret_cast<const uint32_t*>(&h1));
            ptx::sts32(rot_addr(lo_tile, j, (kRot + i) / 8) + byte_in_unit,
                       *reinterpret_cast<const uint32_t*>(&l1));
        }
        ptx::named_barrier_sync(1, kThreads);
    }

    __device__ static __forceinline__ void tile(State& st, uint32_t v_tile, int vlo, int vhi,
                                                Scratch& sc, uint32_t t_idx, int warp, int lane) {
        const int gid = lane >> 2, t4 = lane & 3;
        const int tid = warp * 32 + lane;
        float(*S)[G][kSStride] = sc.S[t_idx & 1];
        derive_keys(sc, v_tile, static_cast<int>(t_idx % STAGES), tid);

        // ---- half scores for positions [8(w%4), +8), dims [256 h, +256) ----
        {
            float c[2][4];   // two independent accumulation chains
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) c[i][e] = 0.0f;
            const int row = (warp & 3) * 8 + (lane & 7);
            const int mat = lane >> 3;
            const int h = warp >> 2;
            // rotated dims: derived tile columns [64 h, 64 h + 64), hi then lo
            const uint32_t hi_tile = ptx::smem_addr(&sc.krot[0][0]);
            const uint32_t lo_tile = ptx::smem_addr(&sc.krot[1][0]);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const uint32_t tile = part == 0 ? hi_tile : lo_tile;
#pragma unroll
                for (int k2 = 0; k2 < kRotSteps / 2; ++k2) {
                    uint32_t b0, b1, b2, b3;
                    ptx::ldmatrix_x4(rot_addr(tile, row, h * (kRot / 8) + k2 * 4 + mat), b0, b1,
                                     b2, b3);
                    ptx::mma_bf16_16816(c[0], st.qr[2 * k2][0], 0u, st.qr[2 * k2][1], 0u, b0, b1);
                    ptx::mma_bf16_16816(c[1], st.qr[2 * k2 + 1][0], 0u, st.qr[2 * k2 + 1][1], 0u,
                                        b2, b3);
                }
            }
            // unrotated dims: the value tile, columns [256 h + 64, 256 h + 256); A from
            // the staged q * w (lanes 0-15 address rows 0-15 at k, lanes 16-31 at k + 8)
            const int grp0 = (h * kHalf + kRot) / 8;
            const uint32_t qt = ptx::smem_addr(sc.qt) + (lane & 15) * kQtStride +
                                (plain_col(h * kHalf + kRot) + (lane >> 4) * 8) * 2;
#pragma unroll
            for (int k2 = 0; k2 < kPlainSteps / 2; ++k2) {
                uint32_t b0, b1, b2, b3, a[2][4];
                ptx::ldmatrix_x4(Base::unit_addr(v_tile, row, grp0 + k2 * 4 + mat), b0, b1, b2, b3);
                ptx::ldmatrix_x4(qt + (2 * k2) * 32, a[0][0], a[0][1], a[0][2], a[0][3]);
                ptx::ldmatrix_x4(qt + (2 * k2 + 1) * 32, a[1][0], a[1][1], a[1][2], a[1][3]);
                ptx::mma_bf16_16816(c[0], a[0][0], a[0][1], a[0][2], a[0][3], b0, b1);
                ptx::mma_bf16_16816(c[1], a[1][0], a[1][1], a[1][2], a[1][3], b2, b3);
            }
            const int pos = (warp & 3) * 8 + 2 * t4;
            // rows gid (hi of q * w, and q) + rows gid + 8 (lo of q * w)
            float s0 = ((c[0][0] + c[0][2]) + (c[1][0] + c[1][2])) * kLog2e;
            float s1 = ((c[0][1] + c[0][3]) + (c[1][1] + c[1][3])) * kLog2e;
            if (pos < vlo || pos >= vhi) s0 = -INFINITY;
            if (pos + 1 < vlo || pos + 1 >= vhi) s1 = -INFINITY;
            *reinterpret_cast<float2*>(&S[h][gid][pos]) = make_float2(s0, s1);
        }
        ptx::named_barrier_sync(1, NC * 32);
        Base::softmax_pv(st, S, v_tile, vlo, vhi, warp, lane);
    }

    __device__ static __forceinline__ void store(const State& st, const DecodeParams& p,
                                                 size_t out_base, int slot, bool bad, int warp,
                                                 int lane) {
        Base::store(st, p, out_base, slot, bad, warp, lane);
    }
};

}  // namespace gqa
