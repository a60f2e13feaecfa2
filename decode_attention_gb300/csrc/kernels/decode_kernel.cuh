// Split-KV decode attention for sm_103a: one persistent kernel per call.
//
// Operation (gemma-4-31B Model Spec, "Compute-graph nodes", the two attn.core
// rows): o[b,h] = softmax over the attended positions s of <q[b,h], k[b,s,h/g]>
// (scale 1), applied to v[b,s,h/g].  Attended positions are [lo_b, L_b) with
// lo_b = max(0, L_b - window) for sliding layers and 0 for global layers (masks
// of the "Gemma 4 31B-it Text Architecture" page, "Compact form", with the
// current token appended before attention).
//
// Work decomposition.  A "segment" u = (b, kvh) is one KV head of one sequence
// with its n_b attended positions; all g query heads of that KV head are served
// from one read of its K/V rows.  Each segment is split into a static head
// (its first sn_b positions) and a dynamic tail of dn_b chunks of c_dyn
// positions (dn_b grows with n_b; short segments have none).
//   * The static heads of all segments, laid end to end (b-major, then kvh),
//     form an index space of Ns positions; CTA i owns the static unit
//     [floor(i Ns / Ge), floor((i+1) Ns / Ge)), Ge = min(grid, Ns).
//   * The dynamic chunks (a few per CTA in total) are claimed with an atomic
//     counter by whichever CTA finishes its static unit first; this absorbs the
//     uneven per-SM memory bandwidth without letting any one segment collect
//     many pieces.
// Every CTA derives the plan itself from seq_lens (no planning kernel, no host
// read of device data).  The piece of a segment inside one unit is a
// "partial".  A segment with a single partial is written straight to the
// output; otherwise each partial stores its (m, l, acc) softmax state in the
// workspace (static unit j at slot j + u, dynamic chunk k at slot
// dyn_slot_base + k), and the partials are merged -- static units in order, then
// the segment's dynamic chunks in order -- with the log-sum-exp rule:
//   * policies with small partials (kMergeInKernel: slidingDecodeGQA, 2 KB) merge
//     in this kernel: each partial counts itself on the segment's arrival counter,
//     and the CTA whose partial completes the count merges them all, writes the
//     output and zeroes the counter for the next call;
//   * the others leave it to the combine kernel (combine_kernel.cuh), launched
//     right behind this one, whose many blocks share the larger merges.
// Which CTA processes a unit, or merges a segment, does not change the
// arithmetic, so results are bit-reproducible.
//
// Data movement.  One producer thread walks the schedule and streams K and V
// tiles of TP positions through a ring of shared-memory stages with TMA (4-D
// boxes of one KV head's rows: 16 positions = one page, or the policy's box
// height on a contiguous cache; 128-byte swizzled where the policy reads the
// tile with ldmatrix), completion counted on mbarriers; with each stage it publishes a descriptor (segment, valid rows,
// first/last tile of a partial, workspace slot).  The consumer warps follow the
// descriptors: policy arithmetic (CUDA cores or warp mma) per tile, epilogue
// after the last tile of a partial.  Every wait is bounded (~2 s): a wait that
// gives up raises a status bit and all consumer warps leave together.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace gqa {

constexpr int kPageRows = 16;         // positions per page = TMA box height on a paged cache
constexpr int kChunkElems = 64;       // bf16 per 128-byte swizzle row
constexpr int kChunkBytes = 2048;     // one chunk of a box: 16 rows x 128 B
constexpr int kMaxBatch = 256;
constexpr int kMaxDynUnits = 2048;    // bound on dynamic chunks (sizes the workspace)
constexpr int kDynChunksPerCta = 8;   // bound on dynamic chunks per CTA
constexpr int kDynSmallPerCta = 4;    // chunks per CTA when the work is small
constexpr int kDynMinSpan = 5;        // segment positions per chunk, in chunk lengths, at least
constexpr int kDynTailPerCta = 2;     // short chunks (claimed last) per CTA
constexpr int kDynTailRatio = 4;      // long / short chunk length
constexpr int kDynFraction = 7;       // about 1/7 of the work is dynamic: covers the spread
                                      // of per-SM memory throughput (~13% between SMs)
constexpr int kDynMinChunk = 256;     // positions: fewer pieces to merge per segment (global
                                      // B=8, S=8192: 1.5% faster than 128; 512 is 5% slower)
constexpr int kDynMinShare = 256;     // positions per CTA below which all work is static
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // a wait gives up after 2 s
constexpr uint32_t kWaitMaxRounds = 1u << 24;        // ... or after this many polling rounds

// Status bits (same values as the public header's GQA_DEVICE_* macros).
constexpr uint32_t kFlagWaitTimeout = 1u;
constexpr uint32_t kFlagBadPage = 2u;
constexpr uint32_t kFlagBadLength = 4u;

// Test modes (same values as the public header's GQA_TEST_* macros).
//   kTestSinglePiece: one CTA streams every segment, so each segment is one piece
//     written straight to the output (no split, no combine).
//   kTestStall: each producer, after issuing its first tile, waits on a barrier
//     that nothing completes; the wait gives up after kTestStallNs, which takes the
//     timeout exit of every role.
constexpr uint32_t kTestSinglePiece = 1u;
constexpr uint32_t kTestStall = 2u;
constexpr uint64_t kTestStallNs = 1000000ull;   // 1 ms

struct DecodeParams {
    const __nv_bfloat16* q;       // [B, H, D]
    const int32_t* seq_lens;      // [B]
    const int32_t* block_table;   // [B, max_pages] (paged only)
    void* out;                    // [B, H, D], bf16 or fp32
    float* ws_acc;                // [slots, G, D]
    float* ws_ml;                 // [slots, G, 2]
    int4* ws_segs;                // [B * KVH] partial list per segment (SegmentParts)
    uint32_t* ws_flags;           // device status word
    uint32_t* ws_claim;           // dynamic-chunk claim counter (zero between calls)
    uint32_t* ws_seg_count;       // [B * KVH] partials stored per segment (in-kernel merge;
                                  // zero between calls)
    uint32_t* ws_done;            // producers finished (in-kernel merge; zero between calls)
    int dyn_slot_base;            // first workspace slot of the dynamic chunks (> grid + B*KVH - 2)
    int max_dyn;                  // dynamic-chunk slots the workspace holds (<= kMaxDynUnits)
    int B, H, KVH;
    int capacity;                 // S, or 16 * max_pages (GQA_MAX_SEQ for a ring)
    int ring;                     // > 0: contiguous ring of `ring` rows, position s at row s mod ring
    int window;                   // 0 = full history
    int num_pages;                // P (paged)
    int max_pages;                // block-table row length (paged)
    int out_f32;                  // 1: fp32 output, 0: bf16
    int T;                        // query tokens per sequence, at positions L - T .. L - 1
                                  // (0 or 1: the single decode token at L - 1)
    uint32_t test_flags;          // kTestSinglePiece / kTestStall (0 in normal use)
    // single K=V cache (policies with kKeqV): the k_norm weight [D] and the rotary
    // frequencies theta^(-2i/D) of the rotated pairs, in fp64
    const __nv_bfloat16* w_k;
    double rope_freq[64];
    // the tensor-core single K=V path: the scores' B operand of every segment,
    // [B, KVH, 2 G, D] bf16 in the workspace (rows [0, G): q * w hi, rows [G, 2 G): lo,
    // with the raw q and zeros on the rotated dims)
    __nv_bfloat16* keqv_operand;
};

// Unpack 2 x bf16 (low half first) to fp32.
__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ---------------------------------------------------------------------------
// Threads per CTA: NC consumer warps, the producer warp, and for the single K=V
// cache a helper warp that prepares per-tile rotation angles.
template <class Pol>
constexpr int block_threads() {
    return (Pol::NC + 1 + (Pol::kKeqV ? 1 : 0)) * 32;
}

// ---------------------------------------------------------------------------
// Plan (shared memory): per-sequence ranges, static/dynamic split, prefix sums
// ---------------------------------------------------------------------------

struct PlanSmem {
    int lo[kMaxBatch];               // first attended position
    int n[kMaxBatch];                // attended positions
    int sn[kMaxBatch];               // static head length of each segment of sequence b
    // (chunk counts and their prefixes are at most kMaxDynUnits; static tiles at most
    // B KVH 2^18 / 16 < 2^32: narrow types keep the plan within the multi-query kernel's
    // shared-memory budget)
    uint16_t dn[kMaxBatch];          // long dynamic chunks of each segment of sequence b
    uint16_t dn1[kMaxBatch];         // short dynamic chunks of each segment of sequence b
    uint32_t spref[kMaxBatch + 1];   // KVH * sum_{b' < b} st_b' (static tiles, below)
    uint16_t dpref[kMaxBatch + 1];   // KVH * sum_{b' < b} dn_b'
    uint16_t dpref1[kMaxBatch + 1];  // KVH * sum_{b' < b} dn1_b'
    long long n_static;              // Ns: static tiles in total
    int unit;                        // positions per tile: the static head of a segment is
                                     // st_b = ceil(sn_b / unit) tiles, all whole but the last
    int n_dyn;                       // dynamic chunks in total (long, then short)
    int n_dyn0;                      // long dynamic chunks
    int c_dyn;                       // positions per long dynamic chunk
    int c_dyn1;                      // positions per short dynamic chunk
    int g_eff;                       // static units (= CTAs with work)
};

// Largest b in [0, B) with pref[b] <= x (pref non-decreasing, pref[B] > x).
template <class T>
__device__ __forceinline__ int upper_seq(const T* pref, int B, long long x) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<long long>(pref[mid]) <= x)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// floor(a / b) for a >= 0, b > 0: one 32-bit division when a fits 32 bits (always,
// for the sizes of this kernel's plan; the 64-bit division is a long software
// routine on the critical path of every CTA's start).
__device__ __forceinline__ long long div_floor(long long a, long long b) {
    if ((static_cast<unsigned long long>(a) >> 32) == 0 && (static_cast<unsigned long long>(b) >> 32) == 0)
        return static_cast<long long>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
    return a / b;
}

// Static tiles of each segment of sequence b.
__device__ __forceinline__ int static_tiles(const PlanSmem& pl, int b) {
    return (pl.sn[b] + pl.unit - 1) / pl.unit;
}
// First static tile of unit j.  The static heads of all segments, concatenated in
// (b, kvh) order and counted in tiles, are split evenly over the units: a unit
// boundary never falls inside a tile, so no tile is read by two CTAs.
__device__ __forceinline__ long long static_unit_begin(const PlanSmem& pl, int j) {
    return div_floor(static_cast<long long>(j) * pl.n_static, pl.g_eff);
}
// static unit containing static tile x (units are floor(j Ns / Ge))
__device__ __forceinline__ int static_unit_of(const PlanSmem& pl, long long x) {
    return static_cast<int>(div_floor((x + 1) * pl.g_eff - 1, pl.n_static));
}

// The partials of segment (b, kvh): static units first_s..first_s+ns_parts-1,
// then dynamic chunks dk0..dk0+nd_parts-1.
struct SegmentParts {
    int first_s, ns_parts, dk0, nd_parts, dyn_base;
    __device__ __forceinline__ SegmentParts(const PlanSmem& pl, int b, int kvh, int dyn_slot_base)
        : dyn_base(dyn_slot_base) {
        const int st = static_tiles(pl, b);
        const long long ss = pl.spref[b] + static_cast<long long>(kvh) * st;
        first_s = static_unit_of(pl, ss);
        ns_parts = static_unit_of(pl, ss + st - 1) - first_s + 1;
        // the dynamic slots of a segment are contiguous: its long chunks, then its
        // short ones (whatever order they are claimed in)
        nd_parts = pl.dn[b] + pl.dn1[b];
        dk0 = pl.dpref[b] + pl.dpref1[b] + kvh * nd_parts;
    }
    __device__ __forceinline__ int count() const { return ns_parts + nd_parts; }
    __device__ __forceinline__ size_t slot(int j, int u) const {
        return j < ns_parts ? static_cast<size_t>(first_s + j) + u
                            : static_cast<size_t>(dyn_base) + dk0 + (j - ns_parts);
    }
};

// One piece of a CTA's work: positions [p0, p1) of segment (b, kvh), whose partial
// goes to workspace slot `slot`; unit_end marks the last piece of the static unit and
// every dynamic chunk (the producer claims the next chunk one tile before its end).
struct Piece {
    int b, kvh, p0, p1, slot;
    bool unit_end;
};

// The CTA's pieces in order: the pieces of consecutive segments in its static unit
// [x, stop) (static tiles of `tile` positions), then dynamic chunks claimed through the
// counter (a claim may already be in flight in `claimed`, -1 when not).  Fills `pc` and
// returns true, or returns false when no piece is left.  One call site per producer
// keeps the producer's code (and its instruction-cache footprint) small.
__device__ __forceinline__ bool next_piece(const PlanSmem& pl, const DecodeParams& p, int cta,
                                           int tile, bool dynamic, long long& x, long long stop,
                                           int& claimed, Piece& pc) {
    const int B = p.B, KVH = p.KVH;
    if (x < stop) {
        const int b = upper_seq(pl.spref, B, x);
        const int st = static_tiles(pl, b);
        const long long rel = x - pl.spref[b];
        const int kvh = static_cast<int>(div_floor(rel, st));
        const int k0 = static_cast<int>(rel - static_cast<long long>(kvh) * st);
        const int take = static_cast<int>(stop - x < st - k0 ? stop - x : st - k0);
        x += take;
        const int e = k0 + take == st ? pl.sn[b] : (k0 + take) * tile;
        pc.b = b;
        pc.kvh = kvh;
        pc.p0 = pl.lo[b] + k0 * tile;
        pc.p1 = pl.lo[b] + e;
        pc.slot = cta + b * KVH + kvh;
        pc.unit_end = x >= stop;
        return true;
    }
    if (!dynamic) return false;
    if (claimed < 0) claimed = static_cast<int>(atomicAdd(p.ws_claim, 1u));
    const int k = claimed;
    claimed = -1;
    if (k >= pl.n_dyn) return false;
    // chunk k: long chunks first, then the short ones; a segment's tail is its long
    // chunks followed by its short ones
    const bool is_long = k < pl.n_dyn0;
    const int kk = is_long ? k : k - pl.n_dyn0;
    const uint16_t* pref = is_long ? pl.dpref : pl.dpref1;
    const int b = upper_seq(pref, B, kk);
    const int per = is_long ? pl.dn[b] : pl.dn1[b];
    const int rel = kk - pref[b];
    const int kvh = rel / per;
    const int idx = rel - kvh * per;
    const int len = is_long ? pl.c_dyn : pl.c_dyn1;
    const int local = is_long ? idx : pl.dn[b] + idx;
    pc.b = b;
    pc.kvh = kvh;
    pc.p0 = pl.lo[b] + pl.sn[b] + (is_long ? 0 : pl.dn[b] * pl.c_dyn) + idx * len;
    pc.p1 = pc.p0 + len;
    pc.slot = p.dyn_slot_base + pl.dpref[b] + pl.dpref1[b] + kvh * (pl.dn[b] + pl.dn1[b]) + local;
    pc.unit_end = true;
    return true;
}

// What the producer publishes with every stage.
struct TileDesc {
    int b, kvh;
    int t;          // first cache row of the tile
    int pos0;       // position held by that row
    int vlo, vhi;   // rows [vlo, vhi) of the tile are attended positions of this partial
    int slot;       // workspace slot of the partial
    int flags;
};
constexpr int kDescFirst = 1;   // first tile of a partial
constexpr int kDescLast = 2;    // last tile of a partial
constexpr int kDescDone = 4;    // no more tiles: consumers leave

// ---------------------------------------------------------------------------
// Kernel shared memory
// ---------------------------------------------------------------------------

template <class Pol>
struct alignas(1024) KernelSmem {
    static constexpr int kTileBytes = Pol::TP * Pol::D * 2;
    static constexpr int kTensors = Pol::kKeqV ? 1 : 2;   // K and V tiles, or the value tile only
    uint8_t kv[Pol::STAGES][kTensors][kTileBytes];   // [stage][K, V][box][chunk][16 rows][128 B]
    alignas(8) uint64_t full[Pol::STAGES];
    alignas(8) uint64_t empty[Pol::STAGES];
    TileDesc desc[Pol::STAGES];
    alignas(8) uint64_t q_empty[2];           // q buffer free (consumer warps arrive)
    alignas(8) uint64_t ready[Pol::STAGES];   // K=V: the stage's rotation angles are ready
    alignas(8) uint64_t stall_bar;            // kTestStall: a barrier nothing completes
    PlanSmem plan;
    // q of the next pieces (bf16, [G][D]), copied in by the producer with the
    // first tile of each piece; double-buffered over pieces
    alignas(128) __nv_bfloat16 q[2][Pol::G * Pol::D];
    // merged partial of the current piece (policies that merge their warps' results
    // through shared memory; the others store straight from registers)
    alignas(16) float acc[Pol::kDirectEpilogue ? 1 : Pol::G][Pol::kDirectEpilogue ? 4 : Pol::D];
    float m[Pol::G];
    float l[Pol::G];
    typename Pol::Scratch scratch;   // each policy aligns its own members (16 B or more)
    int abort_flag;
    int merge_last;                  // this CTA stored the last partial of the segment
};

// Bounded mbarrier wait.  Returns false when the CTA is aborting or the wait
// timed out after limit_ns (which starts the abort).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, uint32_t* flags,
                                             uint64_t limit_ns = kWaitLimitNs) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t round = 0;; ++round) {
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        // time limit, with an iteration cap in case the timer does not advance
        if (ptx::globaltimer_ns() - t0 > limit_ns || round > kWaitMaxRounds) {
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

// Two consecutive outputs starting at idx (a multiple of 2).
__device__ __forceinline__ void store_out2(const DecodeParams& p, size_t idx, float x, float y) {
    if (p.out_f32)
        *reinterpret_cast<float2*>(static_cast<float*>(p.out) + idx) = make_float2(x, y);
    else
        *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + idx) =
            __floats2bfloat162_rn(x, y);
}

// Four consecutive outputs starting at idx (a multiple of 4).
__device__ __forceinline__ void store_out4(const DecodeParams& p, size_t idx, float4 x) {
    if (p.out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(p.out) + idx) = x;
    } else {
        __nv_bfloat162* o =
            reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + idx);
        o[0] = __floats2bfloat162_rn(x.x, x.y);
        o[1] = __floats2bfloat162_rn(x.z, x.w);
    }
}

// ---------------------------------------------------------------------------
// Plan computation, by warps 0..7: lane l of warp w owns sequence b = 32 w + l.
// Every thread of the CTA calls it (the other warps only take part in its CTA
// barriers); it ends with a barrier after which the plan is complete.  Lengths are
// clamped to [0, capacity].  The tail of each segment becomes dynamic chunks:
// long ones of c_dyn positions, then short ones of c_dyn1 ~ c_dyn / 4, all whole
// tiles of `unit` positions.  At most cap = min(kDynChunksPerCta * grid,
// max_dyn) chunks exist (the slots the workspace holds); kDynTailPerCta * grid
// of them (at most half) are kept for the short ones, the rest bound the long.
//  - Long: with much work per CTA, c_dyn is chosen so that about 1/kDynFraction
//    of the work is dynamic, about one chunk per F = kDynFraction c_dyn positions
//    of a segment; with little, chunks keep their minimum length and number about
//    kDynSmallPerCta per CTA (F = N / (kDynSmallPerCta grid)), at most
//    1/kDynMinSpan of the work.
//  - Short: claimed after every long one.  When the long chunks run out, CTAs
//    still differ by up to one long chunk of work; the short ones even that out,
//    so the last CTA ends about one short chunk after the others.
// The T (T1) chunks per kv head are spread over the sequences in proportion to
// their lengths; together they never take more than half of a segment.
//
// Only the chunk counts are bounded, so c_dyn, F and T may be rounded freely:
// they are taken in float (every thread of every CTA computes the same values).
// The counts themselves are integers: n_b <= 2^18, B <= 256, KVH <= 16, so every
// sum fits 32 bits.
//
// Three passes, one sequence per lane: (1) lengths, ranges and a warp scan of n;
// (2) the chunk sizing from the total, each sequence's split and warp scans of
// its tile and chunk counts; (3) the prefix arrays.  The warps' sums cross over
// through `xsum` (32 words of shared memory that nothing else uses meanwhile; the
// caller passes the first stage buffer, which no copy has been issued to yet).
// One short pass per warp instead of one warp walking eight sequences per lane
// keeps the plan's latency (and the code fetched cold on each SM) small.
// ---------------------------------------------------------------------------
constexpr int kPlanWarps = kMaxBatch / 32;   // 8

__device__ __forceinline__ void build_plan(PlanSmem& pl, const DecodeParams& p, int grid, int warp,
                                           int lane, int cta, int unit, uint32_t* xsum) {
    const int B = p.B, KVH = p.KVH;
    const int b = warp * 32 + lane;
    const bool plan_warp = warp < kPlanWarps;
    const bool in_batch = plan_warp && b < B;
    // ---- pass 1: clamped lengths, attended ranges, warp scan of n ----
    int n = 0, nincl = 0;
    if (plan_warp) {
        int x = in_batch ? __ldg(p.seq_lens + b) : 0;
        if (x < 0 || x > p.capacity) {
            if (in_batch && cta == 0) atomicOr(p.ws_flags, kFlagBadLength);
            x = x < 0 ? 0 : p.capacity;
        }
        // union of the queries' ranges: query 0 (position x - T) starts the
        // earliest window, the last query ends at x
        const int span = p.window > 0 ? p.window + (p.T > 1 ? p.T - 1 : 0) : 0;
        const int lo = (span > 0 && x > span) ? x - span : 0;
        n = in_batch ? x - lo : 0;
        if (in_batch) {
            pl.lo[b] = lo;
            pl.n[b] = n;
        }
        nincl = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, nincl, off);
            if (lane >= off) nincl += t;
        }
        if (lane == 31) xsum[warp] = static_cast<uint32_t>(nincl);
    }
    __syncthreads();
    // ---- pass 2: chunk sizing (every plan thread alike), this sequence's split ----
    uint32_t st_incl = 0;
    int d_incl = 0, d1_incl = 0, st_own = 0, d_own = 0, d1_own = 0;
    bool single = false;
    int c = kDynMinChunk, c1 = kDynMinChunk;
    if (plan_warp) {
        uint32_t tot = 0, nbase = 0;
#pragma unroll
        for (int w = 0; w < kPlanWarps; ++w) {
            const uint32_t v = xsum[w];
            tot += v;
            nbase += w < warp ? v : 0u;
        }
        const uint32_t N = tot * static_cast<uint32_t>(KVH);
        const uint32_t ugrid = static_cast<uint32_t>(grid);
        const uint32_t g = N < ugrid ? N : ugrid;
        const uint32_t cdyn = static_cast<uint32_t>(kDynChunksPerCta) * ugrid;
        const uint32_t cap = cdyn < static_cast<uint32_t>(p.max_dyn) ? cdyn : static_cast<uint32_t>(p.max_dyn);
        // the short chunks' slots are set aside first (at most half of them)
        const uint32_t tail_want = static_cast<uint32_t>(kDynTailPerCta) * ugrid;
        const uint32_t tail_cap = tail_want < cap / 2 ? tail_want : cap / 2;
        const uint32_t long_cap = cap - tail_cap;
        // floor(N / g) >= kDynMinShare; none in the single-piece test mode
        single = (p.test_flags & kTestSinglePiece) != 0;
        const bool use_dyn = !single && g > 0 && N >= static_cast<uint32_t>(kDynMinShare) * g &&
                             long_cap > 0;
        int T = 0;
        if (use_dyn) {
            const float Nf = static_cast<float>(N);
            // chunk length: at least kDynMinChunk, about N / (kDynFraction cap), whole tiles
            const int cf = static_cast<int>(ceilf(Nf / static_cast<float>(kDynFraction * long_cap)));
            c = ((cf + unit - 1) / unit) * unit;
            c = c < kDynMinChunk ? kDynMinChunk : c;
            const uint32_t csmall = static_cast<uint32_t>(kDynSmallPerCta) * ugrid;
            const float small = static_cast<float>(csmall < long_cap ? csmall : long_cap);
            const float cff = static_cast<float>(c);
            const float F = fmaxf(fminf(ceilf(Nf / small), kDynFraction * cff), kDynMinSpan * cff);
            const int t = static_cast<int>(static_cast<float>(tot) / F + 0.5f);
            const int tmax = static_cast<int>(long_cap) / KVH;
            T = t < tmax ? t : tmax;
        }
        // short chunks of c1 ~ c / kDynTailRatio positions, about kDynTailPerCta per CTA,
        // claimed after the long ones: when the long chunks run out, CTAs still differ
        // by up to one long chunk of work, and the short ones even that out
        c1 = c;
        int T1 = 0;
        if (T > 0) {
            // (never below kDynMinChunk: shorter pieces cost more in their epilogue
            // and claim than they gain in balance)
            c1 = (c / kDynTailRatio) / unit * unit;
            if (c1 >= kDynMinChunk) {
                const int want = (static_cast<int>(tail_cap) + KVH / 2) / KVH;
                const int room = static_cast<int>(cap) / KVH - T;
                T1 = want < room ? want : room;
            } else {
                c1 = c;
            }
        }
        // sequence b gets d_b = f(P_b + n_b) - f(P_b) long chunks per kv head, P_b the sum
        // of n over the sequences before b and f(x) = floor(x * (T / sum n)): f is
        // monotone and f(sum n) <= T, so the d_b are >= 0 and add up to at most T; the
        // same with T1 for the short ones.  Together they take at most half a segment.
        int d = 0, d1 = 0;
        if (T > 0 && n > 0) {
            const float r = static_cast<float>(T) / static_cast<float>(tot);
            const float x0 = static_cast<float>(nbase + static_cast<uint32_t>(nincl - n));
            const float x1 = static_cast<float>(nbase + static_cast<uint32_t>(nincl));
            d = __float2int_rd(__fmul_rn(x1, r)) - __float2int_rd(__fmul_rn(x0, r));
            int h = __float2int_rd(static_cast<float>(n) * (1.0f / static_cast<float>(2 * c)));
            h -= (h * 2 * c > n) ? 1 : 0;   // floor(n / 2c)
            d = d < h ? d : h;
            if (T1 > 0) {
                const float r1 = static_cast<float>(T1) / static_cast<float>(tot);
                d1 = __float2int_rd(__fmul_rn(x1, r1)) - __float2int_rd(__fmul_rn(x0, r1));
                const int left = n - 2 * d * c;   // >= 0
                int h1 = __float2int_rd(static_cast<float>(left) * (1.0f / static_cast<float>(2 * c1)));
                h1 -= (h1 * 2 * c1 > left) ? 1 : 0;
                d1 = d1 < h1 ? d1 : h1;
            }
        }
        const int sn = n - d * c - d1 * c1;
        if (in_batch) {
            pl.sn[b] = sn;
            pl.dn[b] = static_cast<uint16_t>(d);
            pl.dn1[b] = static_cast<uint16_t>(d1);
        }
        st_own = ((sn + unit - 1) / unit) * KVH;
        d_own = d * KVH;
        d1_own = d1 * KVH;
        st_incl = static_cast<uint32_t>(st_own);
        d_incl = d_own;
        d1_incl = d1_own;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t ts = __shfl_up_sync(0xffffffffu, st_incl, off);
            const int td = __shfl_up_sync(0xffffffffu, d_incl, off);
            const int td1 = __shfl_up_sync(0xffffffffu, d1_incl, off);
            if (lane >= off) {
                st_incl += ts;
                d_incl += td;
                d1_incl += td1;
            }
        }
        if (lane == 31) {   // (words 0 .. 7 are still being read: these are 8 .. 31)
            xsum[8 + warp] = st_incl;
            xsum[16 + warp] = static_cast<uint32_t>(d_incl);
            xsum[24 + warp] = static_cast<uint32_t>(d1_incl);
        }
    }
    __syncthreads();
    // ---- pass 3: exclusive prefixes over the sequences (entry B holds the totals) ----
    if (plan_warp) {
        uint32_t sb = 0, st_tot = 0;
        int db = 0, d_tot = 0, d1b = 0, d1_tot = 0;
#pragma unroll
        for (int w = 0; w < kPlanWarps; ++w) {
            const uint32_t vs = xsum[8 + w];
            const int vd = static_cast<int>(xsum[16 + w]), vd1 = static_cast<int>(xsum[24 + w]);
            st_tot += vs;
            d_tot += vd;
            d1_tot += vd1;
            if (w < warp) {
                sb += vs;
                db += vd;
                d1b += vd1;
            }
        }
        if (b <= B) {
            pl.spref[b] = sb + st_incl - static_cast<uint32_t>(st_own);
            pl.dpref[b] = static_cast<uint16_t>(db + d_incl - d_own);
            pl.dpref1[b] = static_cast<uint16_t>(d1b + d1_incl - d1_own);
        }
        if (warp == 0 && lane == 0) {
            if (B == kMaxBatch) {
                pl.spref[kMaxBatch] = st_tot;
                pl.dpref[kMaxBatch] = static_cast<uint16_t>(d_tot);
                pl.dpref1[kMaxBatch] = static_cast<uint16_t>(d1_tot);
            }
            pl.n_static = static_cast<long long>(st_tot);
            pl.unit = unit;
            pl.n_dyn0 = d_tot;
            pl.n_dyn = d_tot + d1_tot;
            pl.c_dyn = c;
            pl.c_dyn1 = c1;
            const uint32_t units = single ? 1u : static_cast<uint32_t>(grid);   // single piece: CTA 0 takes all
            pl.g_eff = static_cast<int>(st_tot < units ? st_tot : units);
        }
        // xsum lies in a stage buffer that TMA writes next: order these generic-proxy
        // accesses before those async-proxy writes
        ptx::fence_proxy_async_smem();
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// In-kernel merge of a segment's partials
// ---------------------------------------------------------------------------

constexpr int kMergeBatch = 16;   // partials whose loads are in flight together

// Output = the log-sum-exp merge of the segment's partials, in the fixed order of
// SegmentParts: with M = max_j m_j, o = sum_j 2^(m_j - M) acc_j / sum_j 2^(m_j - M) l_j
// (m in log2 units), evaluated as a running merge over batches of partials.  A
// partial that saw no key (m = -inf) weighs 0; no key at all gives the empty sum, 0;
// a NaN normaliser (bad page) stays NaN.  Thread t owns the outputs [2t, 2t + 2) of
// the segment's G x D (kThreads = G D / 2).  The partials were stored by other SMs:
// loads bypass L1.
template <int G, int D, int kThreads>
__device__ __forceinline__ void merge_segment(const DecodeParams& p, const SegmentParts& sp, int u,
                                              size_t out_base, int tid) {
    static_assert(G * D == 2 * kThreads, "two outputs per thread");
    const int nparts = sp.count();
    const int h = (2 * tid) / D;
    const float2* acc2 = reinterpret_cast<const float2*>(p.ws_acc);
    const float2* ml2 = reinterpret_cast<const float2*>(p.ws_ml);
    float M = -INFINITY, den = 0.0f, nx = 0.0f, ny = 0.0f;
    for (int j0 = 0; j0 < nparts; j0 += kMergeBatch) {
        float2 mlj[kMergeBatch], aj[kMergeBatch];
#pragma unroll
        for (int q = 0; q < kMergeBatch; ++q) {
            mlj[q] = make_float2(-INFINITY, 0.0f);
            aj[q] = make_float2(0.0f, 0.0f);
            if (j0 + q < nparts) {
                const size_t sl = sp.slot(j0 + q, u);
                mlj[q] = __ldcg(ml2 + sl * G + h);
                aj[q] = __ldcg(acc2 + sl * (G * D / 2) + tid);
            }
        }
#pragma unroll
        for (int q = 0; q < kMergeBatch; ++q) {
            if (j0 + q >= nparts) break;
            const float Mn = fmaxf(M, mlj[q].x);
            const float sc = M == -INFINITY ? 0.0f : exp2f(M - Mn);
            const float w = mlj[q].x == -INFINITY ? 0.0f : exp2f(mlj[q].x - Mn);
            den = den * sc + w * mlj[q].y;
            nx = nx * sc + w * aj[q].x;
            ny = ny * sc + w * aj[q].y;
            M = Mn;
        }
    }
    const float inv = den == 0.0f ? 0.0f : 1.0f / den;
    store_out2(p, out_base + 2 * static_cast<size_t>(tid), nx * inv, ny * inv);
}

// After this CTA's consumers stored a partial of segment u: count it, and if it was
// the segment's last, merge all of them into the output.  Every consumer thread
// calls this; `last` is a shared-memory flag.  One thread counts, with release
// semantics (the CTA's partial stores, ordered before it by the barrier, are
// visible to the merging CTA) and acquire semantics (if it completes the count, the
// other CTAs' partials are visible here; the barrier after it passes that on).
template <int G, int D, int kThreads>
__device__ __forceinline__ void count_and_merge(const DecodeParams& p, const SegmentParts& sp,
                                                int u, size_t out_base, int tid, volatile int* last) {
    ptx::named_barrier_sync(1, kThreads);
    if (tid == 0)
        *last = ptx::atom_add_acq_rel_gpu(p.ws_seg_count + u, 1u) ==
                        static_cast<uint32_t>(sp.count() - 1)
                    ? 1
                    : 0;
    ptx::named_barrier_sync(1, kThreads);
    if (!*last) return;
    merge_segment<G, D, kThreads>(p, sp, u, out_base, tid);
    if (tid == 0) p.ws_seg_count[u] = 0u;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

template <class Pol, bool kPaged>
__global__ void __launch_bounds__(block_threads<Pol>(), 1)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
    constexpr int G = Pol::G, D = Pol::D, TP = Pol::TP, STAGES = Pol::STAGES, NC = Pol::NC;
    constexpr int kConsumerThreads = NC * 32;
    // TMA boxes: one page on a paged cache, Pol::kBoxRows positions on a contiguous one
    constexpr int kBoxRows = kPaged ? kPageRows : Pol::kBoxRows;
    constexpr int kBoxBytes = kBoxRows * D * 2;
    constexpr int kBoxesPerTile = TP / kBoxRows;
    constexpr int kChunksPerRow = D / kChunkElems;
    static_assert(TP % kBoxRows == 0, "tile must be whole boxes");
    static_assert(block_threads<Pol>() >= 32 * kPlanWarps, "the plan takes eight warps");

    extern __shared__ uint8_t smem_raw[];
    // aligned to 1024 B by pointer arithmetic on smem_raw, so that the compiler still
    // sees shared-memory accesses through sm
    KernelSmem<Pol>& sm = *reinterpret_cast<KernelSmem<Pol>*>(smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u));

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int B = p.B, KVH = p.KVH, H = p.H;
    const int cta = blockIdx.x;
    PlanSmem& pl = sm.plan;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sm.full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sm.empty[s]), NC);
        }
        ptx::mbar_init(ptx::smem_addr(&sm.q_empty[0]), NC);
        ptx::mbar_init(ptx::smem_addr(&sm.q_empty[1]), NC);
        if (Pol::kKeqV)
            for (int s = 0; s < STAGES; ++s) ptx::mbar_init(ptx::smem_addr(&sm.ready[s]), 1);
        ptx::mbar_init(ptx::smem_addr(&sm.stall_bar), 1);
        ptx::fence_mbar_init();
        sm.abort_flag = 0;
    }
    if (warp == NC && lane == 0) {
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }
    // Everything above touches no global memory; from here on inputs written by
    // earlier kernels in the stream are read.
    ptx::grid_dependency_wait();
    ptx::allow_dependent_launch();

    // ---- plan: clamped lengths, attended ranges, static/dynamic split ----
    build_plan(pl, p, gridDim.x, warp, lane, cta, TP, reinterpret_cast<uint32_t*>(&sm.kv[0][0][0]));

    // Work that no tile waits for: zeros for the sequences with nothing to attend (the
    // empty sum) and the partial list of every segment, which the combine kernel reads
    // (each CTA a slice).  The consumer warps do it while the first tiles load; a CTA without
    // work does it with all of its threads and leaves.
    const bool has_work = cta < pl.g_eff;   // (false also for an all-empty batch)
    if (!has_work || warp < NC) {
        const int nt = has_work ? kConsumerThreads : static_cast<int>(blockDim.x);
        for (int b = cta; b < B; b += gridDim.x) {
            if (pl.n[b] != 0) continue;
            const size_t base = static_cast<size_t>(b) * H * D;
            for (int i = tid; i < H * D; i += nt) store_out(p, base + i, 0.0f);
        }
        // (policies that merge in this kernel do not need the lists; they are written
        // anyway, off the critical path, as a record of how each segment was split)
        const int U = B * KVH;
        const int u_end = (cta + 1) * U / static_cast<int>(gridDim.x);   // < 2^31: U <= 4096
        for (int u = cta * U / static_cast<int>(gridDim.x) + tid; u < u_end; u += nt) {
            const int b = u / KVH, kvh = u - (u / KVH) * KVH;
            int4 e = make_int4(0, 0, 0, 0);
            if (pl.n[b] != 0 && pl.g_eff > 0) {
                const SegmentParts sp(pl, b, kvh, p.dyn_slot_base);
                e = make_int4(sp.first_s, sp.ns_parts, sp.dk0, sp.nd_parts);
            }
            p.ws_segs[u] = e;
        }
    }
    if (!has_work) return;

    const uint32_t kv_base = ptx::smem_addr(&sm.kv[0][0][0]);
    constexpr int kTensors = KernelSmem<Pol>::kTensors;
    constexpr uint32_t kStageBytes = kTensors * KernelSmem<Pol>::kTileBytes;

    if (warp == NC) {
        // ================= producer: one thread walks the schedule =================
        if (lane != 0) return;
        const uint64_t policy = ptx::policy_evict_first();
        uint32_t t_idx = 0;
        bool ok = true;

        // Dynamic chunks are claimed one ahead: the claim for the next chunk is
        // issued before the last tile of the current unit, so its latency
        // overlaps the wait for a free stage.
        const bool dynamic = pl.n_dyn > 0;
        int claimed = -1;   // result of the claim in flight, -1 when none
        uint32_t q_n = 0;   // pieces started (q buffer q_n & 1)
        constexpr uint32_t kQBytes = G * D * 2;

        // Streams the tiles of positions [p0, p1) of segment (b, kvh); returns false on abort.
        auto emit_piece = [&](int b, int kvh, int p0, int p1, int slot, bool unit_end) -> bool {
            // the piece's q goes to buffer q_n & 1 once the consumers are done with
            // the q the buffer held two pieces ago
            const uint32_t qb = q_n & 1u;
            if (!wait_bounded(ptx::smem_addr(&sm.q_empty[qb]), ((q_n >> 1) & 1u) ^ 1u,
                              &sm.abort_flag, p.ws_flags))
                return false;
            ++q_n;
            const int chunk0 = kvh * kChunksPerRow;
            const int32_t* bt_row =
                kPaged ? p.block_table + static_cast<size_t>(b) * p.max_pages : nullptr;
            bool first = true;
            // runs [a, e) of positions held in consecutive rows: the whole piece,
            // or on a ring the parts between multiples of the ring length
            for (int a = p0; a < p1;) {
                const int base = p.ring > 0 ? (a / p.ring) * p.ring : 0;   // row = position - base
                const int e = p.ring > 0 && base + p.ring < p1 ? base + p.ring : p1;
                const int t_first = kPaged ? (a & ~(kPageRows - 1)) : a;
                for (int t = t_first; t < e; t += TP) {
                    const bool last = (t + TP >= e) && (e == p1);
                    if (dynamic && unit_end && last)
                        claimed = static_cast<int>(atomicAdd(p.ws_claim, 1u));
                    const int s = t_idx % STAGES;
                    const uint32_t ph = (t_idx / STAGES) & 1u;
                    if (!wait_bounded(ptx::smem_addr(&sm.empty[s]), ph ^ 1u, &sm.abort_flag,
                                      p.ws_flags))
                        return false;
                    const int row0 = t - base;
                    TileDesc& d = sm.desc[s];
                    d.b = b;
                    d.kvh = kvh;
                    d.t = row0;
                    d.pos0 = t;
                    d.vlo = (a > t ? a : t) - t;
                    d.vhi = (e < t + TP ? e : t + TP) - t;
                    d.slot = slot;
                    d.flags = (first ? kDescFirst : 0) | (last ? kDescLast : 0);
                    int nbox = 0;
#pragma unroll
                    for (int j = 0; j < kBoxesPerTile; ++j) nbox += (t + j * kBoxRows < e) ? 1 : 0;
                    const uint32_t full_bar = ptx::smem_addr(&sm.full[s]);
                    ptx::mbar_arrive_expect_tx(full_bar,
                                               static_cast<uint32_t>(nbox * kTensors) * kBoxBytes +
                                                   (first ? kQBytes : 0u));
                    if (first)
                        ptx::bulk_copy_g2s(ptx::smem_addr(&sm.q[qb][0]),
                                           p.q + (static_cast<size_t>(b) * H + kvh * G) * D,
                                           kQBytes, full_bar);
                    // the value tile is the stage's last tensor
                    const uint32_t k_dst = kv_base + s * kStageBytes;
                    const uint32_t v_dst = k_dst + (kTensors - 1) * KernelSmem<Pol>::kTileBytes;
                    for (int j = 0; j < nbox; ++j) {
                        if (kPaged) {
                            int page = bt_row[(row0 >> 4) + j];
                            if (page < 0 || page >= p.num_pages) page = 0;   // flagged by the consumers
                            // swizzled map: (elem, slot, chunk, page); plain map: (elem, kvh, slot, page)
                            const int c1 = Pol::kSwizzle128 ? 0 : kvh;
                            const int c2 = Pol::kSwizzle128 ? chunk0 : 0;
                            if (!Pol::kKeqV)
                                ptx::tma_load_4d(k_dst + j * kBoxBytes, &tm_k, full_bar, 0, c1, c2, page, policy);
                            ptx::tma_load_4d(v_dst + j * kBoxBytes, &tm_v, full_bar, 0, c1, c2, page, policy);
                        } else {
                            // rows past the end of the cache (a run's last tile) read as zeros
                            const int row = row0 + j * kBoxRows;
                            // swizzled map: (elem, position, chunk, seq); plain map: (elem, kvh, position, seq)
                            const int c1 = Pol::kSwizzle128 ? row : kvh;
                            const int c2 = Pol::kSwizzle128 ? chunk0 : row;
                            if (!Pol::kKeqV)
                                ptx::tma_load_4d(k_dst + j * kBoxBytes, &tm_k, full_bar, 0, c1, c2, b, policy);
                            ptx::tma_load_4d(v_dst + j * kBoxBytes, &tm_v, full_bar, 0, c1, c2, b, policy);
                        }
                    }
                    first = false;
                    ++t_idx;
                    // test mode: wait for a barrier that nothing completes (times out)
                    if ((p.test_flags & kTestStall) && t_idx == 1 &&
                        !wait_bounded(ptx::smem_addr(&sm.stall_bar), 0u, &sm.abort_flag, p.ws_flags,
                                      kTestStallNs))
                        return false;
                }
                a = e;
            }
            return true;
        };

        // ---- the static unit of this CTA, then dynamic chunks ----
        long long x = static_unit_begin(pl, cta);
        const long long stop = static_unit_begin(pl, cta + 1);
        Piece pc;
        while (ok && next_piece(pl, p, cta, TP, dynamic, x, stop, claimed, pc))
            ok = emit_piece(pc.b, pc.kvh, pc.p0, pc.p1, pc.slot, pc.unit_end);
        if (ok) {
            // end-of-work descriptor (a plain arrival, no bytes)
            const int s = t_idx % STAGES;
            const uint32_t ph = (t_idx / STAGES) & 1u;
            if (wait_bounded(ptx::smem_addr(&sm.empty[s]), ph ^ 1u, &sm.abort_flag, p.ws_flags)) {
                sm.desc[s].flags = kDescDone;
                ptx::mbar_arrive(ptx::smem_addr(&sm.full[s]));
            }
        } else {
            // let every copy already issued land before the CTA exits
            const uint32_t first = t_idx > static_cast<uint32_t>(STAGES) ? t_idx - STAGES : 0u;
            for (uint32_t tt = first; tt < t_idx; ++tt)
                wait_drain(ptx::smem_addr(&sm.full[tt % STAGES]), (tt / STAGES) & 1u);
        }
        if (Pol::kMergeInKernel && dynamic) {
            // no combine kernel follows: the last producer to finish claiming zeroes
            // the claim counter for the next call
            if (ptx::atom_add_acq_rel_gpu(p.ws_done, 1u) == static_cast<uint32_t>(pl.g_eff - 1)) {
                atomicExch(p.ws_claim, 0u);
                atomicExch(p.ws_done, 0u);
            }
        }
        return;
    }

    if constexpr (Pol::kKeqV) {
        if (warp == NC + 1) {
            // ====== helper: the rotation angles of every tile, a few stages ahead ======
            // (its frequencies come from the parameters: the consumers' setup of the
            // scratch tables is not ordered before this warp's first tile)
            const double f[2] = {p.rope_freq[2 * lane], p.rope_freq[2 * lane + 1]};
            for (uint32_t t_idx = 0;; ++t_idx) {
                const int s = t_idx % STAGES;
                const uint32_t ph = (t_idx / STAGES) & 1u;
                const bool ok = __all_sync(0xffffffffu, wait_bounded(ptx::smem_addr(&sm.full[s]), ph,
                                                                    &sm.abort_flag, p.ws_flags));
                if (!ok) return;
                const TileDesc d = sm.desc[s];
                if (!(d.flags & kDescDone)) Pol::tile_angles(sm.scratch, s, d.pos0, f, lane);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sm.ready[s]));
                if (d.flags & kDescDone) return;
            }
        }
    }

    // ===================== consumers: follow the descriptors =====================
    typename Pol::State st;
    if constexpr (Pol::kKeqV) Pol::init(sm.scratch, p, tid);   // ends in a consumer barrier
    uint32_t t_idx = 0;
    uint32_t q_n = 0;   // pieces started (q buffer q_n & 1)
    bool bad = false;
    const float nan = __uint_as_float(0x7fc00000u);
    while (true) {
        const int s = t_idx % STAGES;
        const uint32_t ph = (t_idx / STAGES) & 1u;
        bool ok = wait_bounded(ptx::smem_addr(&sm.full[s]), ph, &sm.abort_flag, p.ws_flags);
        if constexpr (Pol::kKeqV)
            ok = ok && wait_bounded(ptx::smem_addr(&sm.ready[s]), ph, &sm.abort_flag, p.ws_flags);
        // all consumer warps take the same exit decision
        if (ptx::named_barrier_or(2, kConsumerThreads, !ok)) break;
        const TileDesc d = sm.desc[s];
        if (d.flags & kDescDone) break;
        if (d.flags & kDescFirst) {
            // q arrived with this tile; release the buffer once every lane has read it
            const uint32_t qb = q_n & 1u;
            if constexpr (Pol::kKeqV)
                Pol::begin(st, &sm.q[qb][0], sm.scratch, warp, lane);
            else
                Pol::begin(st, &sm.q[qb][0], warp, lane);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sm.q_empty[qb]));
            ++q_n;
            bad = false;
        }
        if (kPaged) {
            const int32_t* bt_row = p.block_table + static_cast<size_t>(d.b) * p.max_pages;
            for (int j = d.vlo >> 4; j <= (d.vhi - 1) >> 4; ++j) {
                const int page = bt_row[(d.t >> 4) + j];
                bad |= (page < 0 || page >= p.num_pages);
            }
        }
        const uint32_t k_tile = kv_base + s * kStageBytes;
        const uint32_t v_tile = k_tile + (kTensors - 1) * KernelSmem<Pol>::kTileBytes;
        if constexpr (Pol::kKeqV)
            Pol::tile(st, v_tile, d.vlo, d.vhi, sm.scratch, t_idx, warp, lane);
        else
            Pol::tile(st, k_tile, v_tile, d.vlo, d.vhi, sm.scratch, t_idx, warp, lane);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sm.empty[s]));
        ++t_idx;
        if (!(d.flags & kDescLast)) continue;

        // ---------------- epilogue of a partial ----------------
        if (bad && tid == 0) atomicOr(p.ws_flags, kFlagBadPage);
        const SegmentParts sp(pl, d.b, d.kvh, p.dyn_slot_base);
        const int nparts = sp.count();
        const size_t out_base = (static_cast<size_t>(d.b) * H + d.kvh * G) * D;
        const int seg_u = d.b * p.KVH + d.kvh;
        if constexpr (Pol::kDirectEpilogue) {
            // each warp stores its own share of the result from registers: the
            // output when the piece is the whole segment, else the partial
            Pol::store(st, p, out_base, nparts == 1 ? -1 : d.slot, bad, warp, lane);
            if constexpr (Pol::kMergeInKernel)
                if (nparts > 1)
                    count_and_merge<G, D, kConsumerThreads>(p, sp, seg_u, out_base, tid, &sm.merge_last);
        } else {
            // merged (m, l, acc) of this piece -> sm.m, sm.l, sm.acc (ends with a
            // consumer barrier)
            Pol::end(st, &sm.acc[0][0], sm.m, sm.l, sm.scratch, warp, lane);
            const float4* acc4 = reinterpret_cast<const float4*>(&sm.acc[0][0]);
            const float4 nan4 = make_float4(nan, nan, nan, nan);
            if (nparts == 1) {
                for (int i4 = tid; i4 < G * D / 4; i4 += kConsumerThreads) {
                    const float inv = 1.0f / sm.l[(i4 * 4) / D];
                    const float4 a = acc4[i4];
                    store_out4(p, out_base + static_cast<size_t>(i4) * 4,
                               bad ? nan4 : make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv));
                }
            } else {
                const size_t slot = static_cast<size_t>(d.slot);
                float4* wacc4 = reinterpret_cast<float4*>(p.ws_acc + slot * G * D);
                for (int i4 = tid; i4 < G * D / 4; i4 += kConsumerThreads)
                    wacc4[i4] = bad ? nan4 : acc4[i4];
                if (tid < G) {
                    p.ws_ml[(slot * G + tid) * 2 + 0] = bad ? 0.0f : sm.m[tid];
                    p.ws_ml[(slot * G + tid) * 2 + 1] = bad ? nan : sm.l[tid];
                }
                if constexpr (Pol::kMergeInKernel)
                    count_and_merge<G, D, kConsumerThreads>(p, sp, seg_u, out_base, tid, &sm.merge_last);
            }
            // sm.acc is reused by the next piece
            ptx::named_barrier_sync(1, kConsumerThreads);
        }
    }
}

}  // namespace gqa
