// Split-KV decode attention for sm_103a: one persistent kernel per call.
//
// Operation (gemma-4-31B Model Spec, "Compute-graph nodes", the two attn.core
// rows): o[b,h] = softmax over the attended positions s of <q[b,h], k[b,s,h/g]>
// (scale 1), applied to v[b,s,h/g].  Attended positions are [lo_b, L_b) with
// lo_b = max(0, L_b - window) for sliding layers and 0 for global layers (masks
// of the "Gemma 4 31B-it Text Architecture" page, "Compact form", with the
// current token appended before attention).
//
// Work decomposition.  A "segment" is one (b, kvh) pair with its n_b attended
// positions; all g query heads of that KV head are served from one read of its
// K/V rows.  The segments are laid end to end (b-major, then kvh) into one index
// space of N = KVH * sum_b n_b positions, and CTA i of the grid takes the equal
// share [floor(i N / G), floor((i+1) N / G)).  Every CTA derives this plan
// itself from seq_lens (no planning kernel, no host read of device data).  The
// piece of a segment that falls inside one CTA is a "partial"; a segment that
// lies inside one CTA is written straight to the output, otherwise each CTA
// stores its (m, l, acc) softmax partial in the workspace at slot i + u and the
// last CTA to finish a segment (an atomic ticket, no waiting) merges the
// partials with the log-sum-exp rule and writes the output.
//
// Data movement.  One producer warp streams K and V tiles of TP positions through
// a ring of shared-memory stages with TMA (one 4-D box = 16 positions x D per
// tensor, 128-byte swizzled), completion counted on mbarriers.  The consumer
// warps run the policy's arithmetic (CUDA cores or warp mma) on each stage and
// release it.  Every wait is bounded (~2 s); a wait that gives up sets a status
// bit and the kernel runs to its end without further waits or global writes.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace gqa {

constexpr int kBoxRows = 16;         // positions per TMA box (= one 16-position page)
constexpr int kChunkElems = 64;      // bf16 per 128-byte swizzle row
constexpr int kChunkBytes = 2048;    // one chunk of a box: 16 rows x 128 B
constexpr int kMaxBatch = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // a wait gives up after 2 s
constexpr uint32_t kWaitMaxRounds = 1u << 24;        // ... or after this many polling rounds

// Status bits (same values as the public header's GQA_DEVICE_* macros).
constexpr uint32_t kFlagWaitTimeout = 1u;
constexpr uint32_t kFlagBadPage = 2u;
constexpr uint32_t kFlagBadLength = 4u;

struct DecodeParams {
    const __nv_bfloat16* q;       // [B, H, D]
    const int32_t* seq_lens;      // [B]
    const int32_t* block_table;   // [B, max_pages] (paged only)
    void* out;                    // [B, H, D], bf16 or fp32
    float* ws_acc;                // [slots, G, D]
    float* ws_ml;                 // [slots, G, 2]
    uint32_t* ws_counters;        // [B * KVH]
    uint32_t* ws_flags;           // device status word
    int B, H, KVH;
    int capacity;                 // S, or 16 * max_pages
    int window;                   // 0 = full history
    int num_pages;                // P (paged)
    int max_pages;                // block-table row length (paged)
    int out_f32;                  // 1: fp32 output, 0: bf16
};

// Unpack 2 x bf16 (low half first) to fp32.
__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ---------------------------------------------------------------------------
// Plan: per-sequence attended ranges and their prefix sums (shared memory).
// ---------------------------------------------------------------------------

struct PlanSmem {
    int lo[kMaxBatch];
    int n[kMaxBatch];
    long long pref[kMaxBatch + 1];   // pref[b] = KVH * sum_{b' < b} n_b'
};

struct Partial {
    int b, kvh;
    int p0, p1;               // positions [p0, p1) of this CTA's piece
    long long seg_start;      // flattened index of the segment's first position
    int seg_len;              // n_b
};

// Walks the partials of one CTA's flattened range [pos, end).
struct PartialIter {
    long long pos, end;
    int b;
    __device__ PartialIter(long long begin, long long stop) : pos(begin), end(stop), b(0) {}
    __device__ __forceinline__ bool next(const PlanSmem& pl, int B, int KVH, Partial& pt) {
        if (pos >= end) return false;
        while (b < B - 1 && pl.pref[b + 1] <= pos) ++b;
        const long long rel = pos - pl.pref[b];
        const int nb = pl.n[b];
        const int kvh = static_cast<int>(rel / nb);
        const int off = static_cast<int>(rel - static_cast<long long>(kvh) * nb);
        const long long avail = end - pos;
        const int take = static_cast<int>(avail < (nb - off) ? avail : (nb - off));
        pt.b = b;
        pt.kvh = kvh;
        pt.p0 = pl.lo[b] + off;
        pt.p1 = pt.p0 + take;
        pt.seg_start = pl.pref[b] + static_cast<long long>(kvh) * nb;
        pt.seg_len = nb;
        pos += take;
        return true;
    }
};

// CTA whose share contains flattened position x (shares are floor(i N / G)).
__device__ __forceinline__ int cta_of(long long x, long long N, int G) {
    return static_cast<int>(((x + 1) * G - 1) / N);
}

// ---------------------------------------------------------------------------
// Kernel shared memory
// ---------------------------------------------------------------------------

template <class Pol>
struct alignas(1024) KernelSmem {
    static constexpr int kTileBytes = Pol::TP * Pol::D * 2;
    uint8_t kv[Pol::STAGES][2][kTileBytes];   // [stage][K, V][box][chunk][16 rows][128 B]
    alignas(8) uint64_t full[Pol::STAGES];
    alignas(8) uint64_t empty[Pol::STAGES];
    PlanSmem plan;
    alignas(16) float acc[Pol::G][Pol::D];    // merged partial of the current piece
    float m[Pol::G];
    float l[Pol::G];
    alignas(16) typename Pol::Scratch scratch;
    int abort_flag;
    int last_flag;
};

// Bounded mbarrier wait.  Returns false when the CTA is aborting or the wait
// timed out (which starts the abort).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, uint32_t* flags) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t round = 0;; ++round) {
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        // time limit, with an iteration cap in case the timer does not advance
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs || round > kWaitMaxRounds) {
            *abort_flag = 1;
            atomicOr(flags, kFlagWaitTimeout);
            return false;
        }
    }
}

// Time-bounded wait that ignores the abort flag (used to drain copies in flight).
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t round = 0; !ptx::mbar_try_wait(bar, parity); ++round) {
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs || round > 32u * kWaitMaxRounds) return;
    }
}

__device__ __forceinline__ void store_out(const DecodeParams& p, size_t idx, float x) {
    if (p.out_f32)
        static_cast<float*>(p.out)[idx] = x;
    else
        static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(x);
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

template <class Pol, bool kPaged>
__global__ void __launch_bounds__((Pol::NC + 1) * 32, 1)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
    constexpr int G = Pol::G, D = Pol::D, TP = Pol::TP, STAGES = Pol::STAGES, NC = Pol::NC;
    constexpr int kConsumerThreads = NC * 32;
    constexpr int kBoxBytes = kBoxRows * D * 2;
    constexpr int kBoxesPerTile = TP / kBoxRows;
    constexpr int kChunksPerRow = D / kChunkElems;
    static_assert(TP % kBoxRows == 0, "tile must be whole boxes");

    extern __shared__ uint8_t smem_raw[];
    KernelSmem<Pol>& sm = *reinterpret_cast<KernelSmem<Pol>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int B = p.B, KVH = p.KVH, H = p.H;
    const int cta = blockIdx.x;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sm.full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sm.empty[s]), NC);
        }
        ptx::fence_mbar_init();
        sm.abort_flag = 0;
    }
    if (warp == NC && lane == 0) {
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }

    // ---- plan: attended ranges, clamped lengths, prefix sums ----
    for (int b = tid; b < B; b += blockDim.x) {
        int L = p.seq_lens[b];
        if (L < 0 || L > p.capacity) {
            if (cta == 0) atomicOr(p.ws_flags, kFlagBadLength);
            L = L < 0 ? 0 : p.capacity;
        }
        const int lo = (p.window > 0 && L > p.window) ? L - p.window : 0;
        sm.plan.lo[b] = lo;
        sm.plan.n[b] = L - lo;
    }
    __syncthreads();
    if (warp == 0) {
        // each lane sums 8 consecutive sequences, then a warp-wide inclusive scan
        constexpr int kPer = kMaxBatch / 32;
        long long local[kPer];
        long long run = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int b = lane * kPer + j;
            local[j] = run;
            run += (b < B) ? static_cast<long long>(sm.plan.n[b]) * KVH : 0;
        }
        long long incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long t = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += t;
        }
        const long long excl = incl - run;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int b = lane * kPer + j;
            if (b <= B) sm.plan.pref[b] = excl + local[j];
        }
        if (lane == 31 && B == kMaxBatch) sm.plan.pref[kMaxBatch] = incl;
    }
    __syncthreads();

    const long long N = sm.plan.pref[B];

    // sequences with nothing to attend produce zeros (the empty sum)
    for (int b = cta; b < B; b += gridDim.x) {
        if (sm.plan.n[b] != 0) continue;
        const size_t base = static_cast<size_t>(b) * H * D;
        for (int i = tid; i < H * D; i += blockDim.x) store_out(p, base + i, 0.0f);
    }
    // Work is shared by min(grid, N) CTAs so that every share is non-empty: the
    // arrival count of a segment split over CTAs [first, last] must see one
    // piece from each of them.
    const int num_ctas = N < static_cast<long long>(gridDim.x) ? static_cast<int>(N) : gridDim.x;
    if (cta >= num_ctas) return;

    const long long c_begin = static_cast<long long>(cta) * N / num_ctas;
    const long long c_end = static_cast<long long>(cta + 1) * N / num_ctas;

    const uint32_t kv_base = ptx::smem_addr(&sm.kv[0][0][0]);
    constexpr uint32_t kStageBytes = 2u * KernelSmem<Pol>::kTileBytes;

    if (warp == NC) {
        // ================= producer: one thread issues all TMA =================
        if (lane != 0) return;
        const uint64_t policy = ptx::policy_evict_first();
        PartialIter it(c_begin, c_end);
        Partial pt;
        uint32_t t_idx = 0;
        bool ok = true;
        while (ok && it.next(sm.plan, B, KVH, pt)) {
            const int t_first = kPaged ? (pt.p0 & ~(kBoxRows - 1)) : pt.p0;
            const int chunk0 = pt.kvh * kChunksPerRow;
            const int32_t* bt_row =
                kPaged ? p.block_table + static_cast<size_t>(pt.b) * p.max_pages : nullptr;
            for (int t = t_first; t < pt.p1; t += TP) {
                const int s = t_idx % STAGES;
                const uint32_t ph = (t_idx / STAGES) & 1u;
                if (!wait_bounded(ptx::smem_addr(&sm.empty[s]), ph ^ 1u, &sm.abort_flag,
                                  p.ws_flags)) {
                    ok = false;
                    break;
                }
                int nbox = 0;
#pragma unroll
                for (int j = 0; j < kBoxesPerTile; ++j) nbox += (t + j * kBoxRows < pt.p1) ? 1 : 0;
                const uint32_t full_bar = ptx::smem_addr(&sm.full[s]);
                ptx::mbar_arrive_expect_tx(full_bar, static_cast<uint32_t>(nbox) * 2u * kBoxBytes);
                const uint32_t k_dst = kv_base + s * kStageBytes;
                const uint32_t v_dst = k_dst + KernelSmem<Pol>::kTileBytes;
                for (int j = 0; j < nbox; ++j) {
                    if (kPaged) {
                        int page = bt_row[(t >> 4) + j];
                        if (page < 0 || page >= p.num_pages) page = 0;   // flagged by the consumers
                        ptx::tma_load_4d(k_dst + j * kBoxBytes, &tm_k, full_bar, 0, 0, chunk0, page,
                                         policy);
                        ptx::tma_load_4d(v_dst + j * kBoxBytes, &tm_v, full_bar, 0, 0, chunk0, page,
                                         policy);
                    } else {
                        const int row = t + j * kBoxRows;
                        ptx::tma_load_4d(k_dst + j * kBoxBytes, &tm_k, full_bar, 0, row, chunk0,
                                         pt.b, policy);
                        ptx::tma_load_4d(v_dst + j * kBoxBytes, &tm_v, full_bar, 0, row, chunk0,
                                         pt.b, policy);
                    }
                }
                ++t_idx;
            }
        }
        if (!ok) {
            // let every copy already issued land before the CTA exits
            const uint32_t first = t_idx > static_cast<uint32_t>(STAGES) ? t_idx - STAGES : 0u;
            for (uint32_t tt = first; tt < t_idx; ++tt)
                wait_drain(ptx::smem_addr(&sm.full[tt % STAGES]), (tt / STAGES) & 1u);
        }
        return;
    }

    // ===================== consumers =====================
    typename Pol::State st;
    PartialIter it(c_begin, c_end);
    Partial pt;
    uint32_t t_idx = 0;
    bool aborted = false;
    while (it.next(sm.plan, B, KVH, pt)) {
        const int t_first = kPaged ? (pt.p0 & ~(kBoxRows - 1)) : pt.p0;
        const __nv_bfloat16* q_heads = p.q + (static_cast<size_t>(pt.b) * H + pt.kvh * G) * D;
        Pol::begin(st, q_heads, warp, lane);
        bool bad = false;
        const int32_t* bt_row =
            kPaged ? p.block_table + static_cast<size_t>(pt.b) * p.max_pages : nullptr;
        for (int t = t_first; t < pt.p1; t += TP) {
            const int s = t_idx % STAGES;
            const uint32_t ph = (t_idx / STAGES) & 1u;
            if (!aborted &&
                !wait_bounded(ptx::smem_addr(&sm.full[s]), ph, &sm.abort_flag, p.ws_flags))
                aborted = true;
            const int vlo = (pt.p0 > t ? pt.p0 : t) - t;
            const int vhi = (pt.p1 < t + TP ? pt.p1 : t + TP) - t;
            if (kPaged) {
                for (int j = vlo >> 4; j <= (vhi - 1) >> 4; ++j) {
                    const int page = bt_row[(t >> 4) + j];
                    bad |= (page < 0 || page >= p.num_pages);
                }
            }
            const uint32_t k_tile = kv_base + s * kStageBytes;
            const uint32_t v_tile = k_tile + KernelSmem<Pol>::kTileBytes;
            Pol::tile(st, k_tile, v_tile, vlo, vhi, sm.scratch, t_idx, warp, lane);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sm.empty[s]));
            ++t_idx;
        }
        // merged (m, l, acc) of this piece -> sm.m, sm.l, sm.acc (ends with a consumer barrier)
        Pol::end(st, &sm.acc[0][0], sm.m, sm.l, sm.scratch, warp, lane);

        // ---------------- epilogue ----------------
        if (bad && tid == 0) atomicOr(p.ws_flags, kFlagBadPage);
        const int u = pt.b * KVH + pt.kvh;
        const long long seg_end = pt.seg_start + pt.seg_len;
        const int first = cta_of(pt.seg_start, N, num_ctas);
        const int last = cta_of(seg_end - 1, N, num_ctas);
        const size_t out_base = (static_cast<size_t>(pt.b) * H + pt.kvh * G) * D;
        const float nan = __uint_as_float(0x7fc00000u);
        if (first == last) {
            if (!aborted) {
                for (int i = tid; i < G * D; i += kConsumerThreads) {
                    const int h = i / D;
                    store_out(p, out_base + i, bad ? nan : (&sm.acc[0][0])[i] / sm.l[h]);
                }
            }
        } else {
            const size_t slot = static_cast<size_t>(cta) + u;
            if (!aborted) {
                float* wacc = p.ws_acc + slot * G * D;
                for (int i = tid; i < G * D; i += kConsumerThreads)
                    wacc[i] = bad ? nan : (&sm.acc[0][0])[i];
                if (tid < G) {
                    p.ws_ml[(slot * G + tid) * 2 + 0] = bad ? 0.0f : sm.m[tid];
                    p.ws_ml[(slot * G + tid) * 2 + 1] = bad ? nan : sm.l[tid];
                }
                __threadfence();
            }
            ptx::named_barrier_sync(1, kConsumerThreads);
            if (tid == 0) {
                int is_last = 0;
                if (!aborted && !sm.abort_flag) {
                    const unsigned nparts = static_cast<unsigned>(last - first + 1);
                    is_last = atomicInc(p.ws_counters + u, nparts - 1u) == nparts - 1u;
                }
                sm.last_flag = is_last;
            }
            ptx::named_barrier_sync(1, kConsumerThreads);
            if (sm.last_flag) {
                __threadfence();
                // log-sum-exp merge of the partials of segment u, in CTA order
                for (int i = tid; i < G * D; i += kConsumerThreads) {
                    const int h = i / D;
                    float M = -INFINITY;
                    for (int j = first; j <= last; ++j)
                        M = fmaxf(M, __ldcg(p.ws_ml + ((static_cast<size_t>(j) + u) * G + h) * 2));
                    float num = 0.0f, den = 0.0f;
                    for (int j = first; j <= last; ++j) {
                        const size_t sl = static_cast<size_t>(j) + u;
                        const float w = exp2f(__ldcg(p.ws_ml + (sl * G + h) * 2) - M);
                        num += w * __ldcg(p.ws_acc + sl * G * D + i);
                        den += w * __ldcg(p.ws_ml + (sl * G + h) * 2 + 1);
                    }
                    store_out(p, out_base + i, num / den);
                }
            }
        }
        // sm.acc / sm.last_flag are reused by the next piece
        ptx::named_barrier_sync(1, kConsumerThreads);
    }
}

}  // namespace gqa
