// Multi-query decode attention on the 5th-generation tensor cores (tcgen05).
//
// Operation ("Gemma 4 31B-it Text Architecture", "Inference behavior: Prefill,
// Cache, and Long Context" and "Compact form"; gemma-4-31B Model Spec, the two
// attn.core rows): a step appends T new tokens per sequence to the cache, then
// query t, at position p = L - T + t, attends to the keys s <= p (full layers) or
// p - W < s <= p (sliding layers), with scale 1; the g query heads of a KV head
// share its keys and values.  A query at a negative position sees nothing (o = 0).
//
// Orientation.  A segment (b, kvh) has R = T * g query rows (r = t * g + h, at
// most 32).  Tiles of 128 positions fill the M dimension of a cta_group::1 mma,
// so both contractions run transposed:
//   scores  S^T[pos, r]  = sum_d K[pos, d] Q[r, d]          A = K tile (K-major),
//                                                          B = Q (K-major)
//   P.V     O^T[d, r]   += sum_pos V^T[d, pos] P^T[pos, r]  A = the V tile read
//                                                          MN-major, B = P (K-major)
// with N = R rounded up to 16.  S^T (two buffers) and O^T (D/128 blocks of 128
// head-dim lanes) live in TMEM.  One K or V stage is 128 positions x 64 head-dim
// elements (16 KB, 128-byte swizzled, exactly what TMA writes); the P.V mma of a
// 128-wide head-dim block reads two adjacent stages.
//
// Warp roles (352 threads; 384 over a K=V cache).  Warp 0, lane 0: the producer.  It
// walks the same schedule as the single-query kernel (static units, then claimed dynamic
// chunks)
// and streams the tiles in the order K(0), K(1), V(0), K(2), V(1), ...: the scores
// of tile i+1 are computed while the softmax of tile i runs.  K blocks go to one
// stage ring and V blocks to another, each consumed in order by one warp (with two
// consumers on one ring, a one-bit phase wait could see the other consumer's
// earlier fill of the same stage).  It also loads each piece's Q with TMA (box: 64
// elements x g heads x T tokens) into the Q buffer, once the previous piece's last
// scores are done.  Warp 1: owns the TMEM allocation; lane 0 issues the scores' mma.
// Warp 10: lane 0 issues the P.V mma, and the whole warp zeroes the V rows of a tile
// that lie outside its sequence's attended range before they are read (0 * NaN
// would poison the sum).  A tcgen05.mma costs its issuing thread about 75 cycles
// whatever N is up to 128, so two issuing warps keep the tensor core busier.
// Warps 2..9: thread j of lane quarter warp % 4 owns TMEM lane j, i.e. position j
// of the tile's scores and head-dim element j of each O^T block; they run the
// softmax and the epilogue, the two warps of a quarter splitting the query rows
// (two warps per scheduler hide each other's latencies).  Over a K=V cache, warp 11
// (lane 0) streams the V blocks from tile descriptors the producer hands it, warps
// 2..5 run the softmax (one per quarter, all query rows) and warps 6..9 derive each
// tile's rotated keys into TMEM while the softmax of the tile before runs.
//
// Where the configuration has two O^T buffers in TMEM, pieces alternate between them: a
// piece's output is written after the next tile's P has been published, so the softmax
// warps never wait for the last P.V of a piece before starting the next one.  With one
// buffer, a piece's output is written before the next piece's first P.V.
//
// Softmax.  Each query row keeps a reference max m (log2 units) that all threads
// share; P = exp2(s - m), and m moves only when a score of the tile exceeds it by
// more than kMqTau (then the O^T columns and the normaliser shares are rescaled
// by exp2(m_old - m_new)).  P <= 2^kMqTau keeps every fp32 sum finite.  P is
// applied as a bf16 hi part and a bf16 lo part, rows [0, NMAX) and [NMAX, 2 NMAX) of
// the mma's B operand, whose two O^T columns are summed at the end: about 16
// significant bits.  The epilogue of a piece writes the
// normalised output, or the partial (acc, m, l) that the combine kernel merges.
//
// Every wait is bounded; a wait that gives up raises the status word's timeout
// bit, the roles leave together, in-flight copies and mma are drained, and TMEM is
// released before the CTA exits.
#pragma once

#include <type_traits>

#include <cuda_fp16.h>

#include "decode_kernel.cuh"

namespace gqa {

constexpr int kMqTile = 128;                       // positions per tile (mma M)
constexpr int kMqStageBytes = kMqTile * 128;       // 128 rows x 64 bf16
constexpr float kMqTau = 24.0f;                    // rescale threshold, log2 units
constexpr int kMqPLbo = 144;                       // P core matrices along positions (padded
                                                   // from 128 B so stores hit distinct banks)
constexpr int kMqPSbo = (kMqTile / 8) * kMqPLbo;   // P 8-row groups: 2304 B
constexpr int kMqVq = 8;                // tile descriptors in flight to the V producer

constexpr int tmem_cols_for(int cols) {
    int c = 32;
    while (c < cols) c *= 2;
    return c;
}

template <int kD, int kG, int kMaxT, int kKStages, int kVStages, int kObufs, bool kKeqV = false,
          int kRStages = 0>
struct MqCfg {
    static constexpr int D = kD, G = kG, MAXT = kMaxT, OBUFS = kObufs;
    // stage rings, each consumed in order by one warp: K (scores warp), V (P.V warp) and,
    // over a single K=V cache, R (the rotated dims, read by the softmax warps to
    // derive the rotated keys)
    static constexpr bool KEQV = kKeqV;
    static constexpr int KST = kKStages, VST = kVStages, RST = kRStages;
    static constexpr int STAGES = kKStages + kVStages + kRStages;
    static constexpr int NSUB = D / 64;                 // stages per tile of one tensor
    static constexpr int NB = D / 128;                  // 128-wide head-dim blocks of O^T
    static constexpr int RMAX = G * MAXT;               // query rows of a segment
    static constexpr int NMAX = RMAX <= 16 ? 16 : 32;   // mma N bound
    static constexpr int QATOM = NMAX * 128;            // Q rows of one 64-element column block
    static constexpr int QBYTES = NSUB * QATOM;
    // P^T rows: the bf16 hi parts in [0, PLO), the lo parts in [PLO, 2 PLO); this is the
    // P.V mma's N.  Over a K=V cache only the RMAX query rows (and their lo parts) exist.
    static constexpr int PLO = KEQV ? RMAX : NMAX;
    static constexpr int PROWS = 2 * PLO;
    static constexpr int PBYTES = (PROWS / 8) * kMqPSbo;
    static constexpr int TMEM_S = 0;                    // S^T buffers: columns [0, 2 NMAX)
    static constexpr int TMEM_O = 2 * NMAX;             // O^T: OBUFS piece buffers of NB blocks
    static constexpr int OBUF = NB * PROWS;             // of PROWS columns (hi part, lo part)
    // K=V: the derived rotated keys of a tile, the A operand of the rotated k-steps:
    // 128 rows x 128 bf16 (rotated dims i and D/2 + i, i < 64), hi then lo
    static constexpr int TMEM_KROT = TMEM_O + OBUFS * OBUF;
    static constexpr int KROT_COLS = KEQV ? 128 : 0;
    // K=V: the key of tile row j (the TMEM lane) on rotated pair i is R(j f_i) (w * v):
    // per pair group m (pairs i = 2m, 2m + 1), fp32 at columns 8m + t (t = i - 2m):
    // cos(j f_i) w_i, then at + 2: -sin(j f_i) w_{D/2+i}, + 4: cos(j f_i) w_{D/2+i},
    // + 6: sin(j f_i) w_i
    static constexpr int TMEM_TRIG = TMEM_KROT + KROT_COLS;
    static constexpr int TRIG_COLS = KEQV ? 256 : 0;
    // Warp roles: 0 producer, 1 scores mma (and TMEM owner), then the softmax warps (8,
    // two per TMEM lane quarter; over a K=V cache 4, one per quarter), then over a K=V
    // cache 8 key-deriving warps (two per quarter), then the P.V warp and, over a K=V
    // cache, the V producer.
    static constexpr int SMX_WARPS = KEQV ? 4 : 8;
    static constexpr int SMX_THREADS = 32 * SMX_WARPS;
    static constexpr int DRV_WARPS = KEQV ? 8 : 0;
    static constexpr int DRV_THREADS = 32 * DRV_WARPS;
    static constexpr int PV_WARP = 2 + SMX_WARPS + DRV_WARPS;
    static constexpr int NK = KEQV ? NSUB - 2 : NSUB;   // stages of a K block
    // Over a K=V cache a second producer warp streams the V blocks, so that waits on the
    // V ring (paced by the P.V warp) never hold up the K and R rings.
    static constexpr bool SPLIT_V = KEQV;
    // On a contiguous cache, a tile at the end of its sequence loads only the 16-row boxes
    // that hold attended rows.  Sliding segments span at most W + T - 1 positions (1031
    // for T = 8: 9 tiles, the last one 7 rows), so about a tenth of their tile rows would
    // be unattended; global segments are long, and the extra branch in the producer's
    // stage loop cost them more (3-7%) than it saved.
    static constexpr bool RAGGED = (D == 256);
    static constexpr int V_WARP = PV_WARP + 1;          // the V producer (SPLIT_V)
    static constexpr int THREADS = 32 * (PV_WARP + 1 + (SPLIT_V ? 1 : 0));
    static constexpr int TMEM_COLS = tmem_cols_for(TMEM_TRIG + TRIG_COLS);
    static_assert(TMEM_TRIG + TRIG_COLS <= 512, "TMEM holds 512 columns");
    static_assert(OBUFS == 1 || OBUFS == 2, "one or two O^T buffers");
    static_assert(!KEQV || (D == 512 && G == 8 && MAXT == 1 && RST >= 2 && RST % 2 == 0),
                  "K=V: decodeGQA, one query, whole tiles of R blocks");
    static_assert(VST % 2 == 0, "a P.V block reads two adjacent stages");
    static_assert(NSUB % 2 == 0 && RMAX <= 32, "geometry");
    // query rows fill the mma N bound; over a K=V cache the scores' B operand holds
    // the hi and the lo parts of q * w as 2 RMAX rows
    static_assert(RMAX == NMAX || (KEQV && 2 * RMAX == NMAX), "query rows fill the mma N bound");
    static_assert(PROWS % 16 == 0, "the P.V mma's N is a multiple of 16");
};

using MqGlobal = MqCfg<512, 8, 4, 4, 4, 1>;     // decodeGQA, T <= 4
using MqGlobal2 = MqCfg<512, 8, 2, 4, 6, 2>;   // decodeGQA, T <= 2: smaller Q and P, more stages
using MqSliding = MqCfg<256, 2, 8, 4, 6, 2>;   // slidingDecodeGQA, T <= 8
using MqKeqV = MqCfg<512, 8, 1, 6, 4, 1, true, 2>;   // decodeGQA over a single K=V cache (one
                                                     // O^T buffer: TMEM holds the rotation factors;
                                                     // the R ring holds two tiles)

// Rotation data of the K=V key derivation in shared memory (the per-row factors of
// R(j f_i) live in TMEM): per tile, cos and sin of t f_i for the tile's first position t.
struct MqRopeTables {
    float2 base[64];
};
struct MqNoTables {};


struct MqTile {
    int b, kvh;
    int t;          // position of tile row 0 (= its cache row on a contiguous cache)
    int vlo, vhi;   // rows [vlo, vhi) belong to this piece
    int zlo, zhi;   // rows outside [zlo, zhi) lie outside the sequence's attended range
    int slot;       // workspace slot of the piece
    int flags;      // kDescFirst / kDescLast of the piece, kDescDone
    int ob;         // O^T buffer of the piece (pieces alternate)
};

constexpr int kMqKindK = 0, kMqKindV = 1, kMqKindDone = 2, kMqKindR = 3, kMqKindDoneR = 4;

template <class Cfg>
struct alignas(1024) MqSmem {
    uint8_t stage[Cfg::STAGES][kMqStageBytes];   // K ring, then V ring: [128 rows][128 B], swizzled
    // [column block][NMAX rows][128 B], swizzled.  Over a K=V cache the column blocks of
    // the rotated dims (0 and NSUB/2) hold R(-t f) q of the current tile instead (f16 hi
    // rows [0, G), lo rows [G, 2 G)), written per tile by the key-deriving warps
    uint8_t q[Cfg::QBYTES];
    uint8_t pm[2][Cfg::PBYTES];                   // P^T [buffer], core-matrix layout
    alignas(8) uint64_t full[Cfg::STAGES];
    alignas(8) uint64_t empty[Cfg::STAGES];
    alignas(8) uint64_t q_empty;      // the last scores of the piece holding Q are done
    alignas(8) uint64_t s_full[2];    // scores of tile i in S buffer i % 2 (+ its tile)
    alignas(8) uint64_t p_full[2];    // P of tile i written (softmax warps)
    alignas(8) uint64_t p_empty[2];   // P.V of tile i no longer reads P buffer i % 2
    alignas(8) uint64_t o_ready[2];   // P.V of tile i complete
    alignas(8) uint64_t s_empty[2];   // the softmax warps have read S buffer i % 2
    alignas(8) uint64_t drain[2];     // the two mma warps' final commits
    alignas(8) uint64_t stall_bar;    // test mode kTestStall: a barrier nothing completes
    int kind[Cfg::KST];               // K ring: a K block or the end-of-work marker
    MqTile desc[Cfg::KST];            // tile of a K block (its first stage)
    int rkind[Cfg::KEQV ? Cfg::RST : 1];       // R ring: an R block or the end-of-work marker
    MqTile rdesc[Cfg::KEQV ? Cfg::RST : 1];    // tile of an R block (its first stage)
    alignas(8) uint64_t krot_full;             // K=V: the derived keys of the next tile are in TMEM
    alignas(8) uint64_t krot_empty;            // K=V: the rotated mma of the last tile completed
    alignas(8) uint64_t r_full[2];             // K=V: the rotated mma of tile i (S buffer i % 2) completed
    // K=V: tiles whose V blocks the V producer issues, in order (FIFO from the producer)
    MqTile vq[Cfg::SPLIT_V ? kMqVq : 1];
    alignas(8) uint64_t vq_full[Cfg::SPLIT_V ? kMqVq : 1];
    alignas(8) uint64_t vq_empty[Cfg::SPLIT_V ? kMqVq : 1];
    alignas(16) std::conditional_t<Cfg::KEQV, MqRopeTables, MqNoTables> rope;
    MqTile s_desc[2];                 // tile whose scores are in S buffer j
    MqTile p_desc[2];                 // tile whose P is in P buffer j
    int pv_stop;                      // index of the first tile that does not exist (set
                                      // with the last p_full; larger until then)
    PlanSmem plan;
    float red[4][Cfg::NMAX];
    uint32_t red_bad[Cfg::SMX_WARPS];
    float epi_m[Cfg::NMAX];   // the finished piece whose epilogue is pending: reference max,
    float epi_l[Cfg::NMAX];   // normaliser and bad-page bits per query row
    uint32_t epi_bad;
    uint32_t tmem_base;
    int abort_flag;
};

// The Q operand of segment (b, kvh) into the Q buffer at qdst, completing on bar: the
// q rows of the KV head's group (elements, rows, ...), or over a K=V cache the scores
// operand [B, KVH, 2 G, D] of the segment except its rotated column blocks.  Not
// inlined: the producer services a pending Q load from every wait, and one out-of-line
// copy keeps its code (fetched cold at the start of each CTA) small.
template <class Cfg>
__device__ __noinline__ void mq_load_q(uint32_t qdst, const CUtensorMap* tm_q, uint32_t bar, int b,
                                       int kvh, uint64_t policy) {
    for (int c = 0; c < Cfg::NSUB; ++c) {
        if (Cfg::KEQV && (c == 0 || c == Cfg::NSUB / 2)) continue;
        if (Cfg::KEQV)
            ptx::tma_load_4d(qdst + c * Cfg::QATOM, tm_q, bar, 64 * c, 0, kvh, b, policy);
        else
            ptx::tma_load_4d(qdst + c * Cfg::QATOM, tm_q, bar, 64 * c, kvh * Cfg::G, 0, b, policy);
    }
}

// The producer's pending Q load: the Q operand of the newest piece, issued once the
// previous piece's last scores are done (q_empty), completing on that piece's first K
// stage (bar).
struct MqPendingQ {
    bool pend;
    uint32_t issued;      // pieces whose Q load was issued
    int b, kvh;
    uint32_t bar;         // full barrier the load completes on
    uint32_t empty_bar;   // q_empty
    uint32_t dst;         // the Q buffer
    const CUtensorMap* map;
    uint64_t policy;
};

// Issues the pending Q load if the Q buffer is free (piece n = issued may overwrite it
// once the last scores of piece n - 1 are done).
template <class Cfg>
__device__ __forceinline__ void mq_service_q(MqPendingQ& qs) {
    if (qs.pend && ptx::mbar_try_wait(qs.empty_bar, (qs.issued & 1u) ^ 1u)) {
        mq_load_q<Cfg>(qs.dst, qs.map, qs.bar, qs.b, qs.kvh, qs.policy);
        qs.pend = false;
        ++qs.issued;
    }
}

// The producer's bounded wait on barrier bar (or, with bar == 0, for the pending Q load
// to go out), servicing the pending Q load meanwhile.  False when the CTA is aborting or
// the wait timed out (which starts the abort).  Out of line: one copy serves every wait
// site of the producer, whose code is fetched cold at the start of each CTA.
template <class Cfg>
__device__ __noinline__ bool mq_poll_servicing(uint32_t bar, uint32_t parity, MqPendingQ& qs,
                                               volatile int* abort_flag, uint32_t* flags) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t round = 0;; ++round) {
        mq_service_q<Cfg>(qs);
        for (int i = 0; i < 8; ++i)
            if (bar ? ptx::mbar_try_wait(bar, parity) : !qs.pend) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs || round > kWaitMaxRounds) {
            *abort_flag = 1;
            atomicOr(flags, kFlagWaitTimeout);
            return false;
        }
    }
}

// Byte offset of P^T element (query row r, tile position j): K-major, no swizzle.
__device__ __forceinline__ uint32_t mq_p_off(int r, int j) {
    return (j >> 3) * kMqPLbo + (r >> 3) * kMqPSbo + (r & 7) * 16 + (j & 7) * 2;
}

template <class Cfg, bool kPaged>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    gqa_mq_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k16,
                  const __grid_constant__ CUtensorMap tm_v16, const DecodeParams p) {
    constexpr int D = Cfg::D, G = Cfg::G, NSUB = Cfg::NSUB, NB = Cfg::NB, STAGES = Cfg::STAGES;
    constexpr int KST = Cfg::KST, VST = Cfg::VST;
    constexpr int NMAX = Cfg::NMAX;
    static_assert(Cfg::THREADS >= 32 * kPlanWarps, "the plan takes eight warps");

    extern __shared__ uint8_t smem_raw[];
    // aligned to 1024 B by pointer arithmetic on smem_raw, so that the compiler still
    // sees shared-memory accesses through sm
    MqSmem<Cfg>& sm = *reinterpret_cast<MqSmem<Cfg>*>(smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u));

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int B = p.B, KVH = p.KVH, H = p.H;
    const int T = p.T > 1 ? p.T : 1;
    const int R = T * G;
    const int N = (R + 15) & ~15;   // mma N
    const int cta = blockIdx.x;
    PlanSmem& pl = sm.plan;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sm.full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sm.empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&sm.q_empty), 1);
        for (int j = 0; j < 2; ++j) {
            ptx::mbar_init(ptx::smem_addr(&sm.s_full[j]), 2);   // mma commit + the tile's descriptor
            ptx::mbar_init(ptx::smem_addr(&sm.p_full[j]), Cfg::SMX_WARPS);   // one arrival per softmax warp
            ptx::mbar_init(ptx::smem_addr(&sm.p_empty[j]), 1);
            ptx::mbar_init(ptx::smem_addr(&sm.o_ready[j]), 1);
            ptx::mbar_init(ptx::smem_addr(&sm.s_empty[j]), Cfg::SMX_WARPS);   // one per softmax warp
            ptx::mbar_init(ptx::smem_addr(&sm.drain[j]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&sm.krot_full), Cfg::KEQV ? Cfg::DRV_WARPS : 1);   // one per key-deriving warp
        ptx::mbar_init(ptx::smem_addr(&sm.krot_empty), 1);   // the rotated mma's commit
        ptx::mbar_init(ptx::smem_addr(&sm.r_full[0]), 1);
        ptx::mbar_init(ptx::smem_addr(&sm.r_full[1]), 1);
        for (int k = 0; k < (Cfg::SPLIT_V ? kMqVq : 0); ++k) {
            ptx::mbar_init(ptx::smem_addr(&sm.vq_full[k]), 1);
            ptx::mbar_init(ptx::smem_addr(&sm.vq_empty[k]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&sm.stall_bar), 1);
        sm.pv_stop = 0x7fffffff;
        ptx::fence_mbar_init();
        sm.abort_flag = 0;
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        if (!kPaged && Cfg::RAGGED) {
            ptx::prefetch_tensormap(&tm_k16);
            ptx::prefetch_tensormap(&tm_v16);
        }
        ptx::prefetch_tensormap(&tm_q);
    }
    ptx::grid_dependency_wait();
    ptx::allow_dependent_launch();

    build_plan(pl, p, gridDim.x, warp, lane, cta, kMqTile, reinterpret_cast<uint32_t*>(&sm.stage[0][0]));

    // Work that no tile waits for: zeros for the sequences with nothing to attend (all T
    // queries) and the partial list of every segment for the combine kernel (each CTA a
    // slice).  The softmax warps do it while the first tiles load (bookkeeping() below);
    // a CTA without work does it with all of its threads and leaves.
    auto bookkeeping = [&](int t0, int nt) {
        for (int b = cta; b < B; b += gridDim.x) {
            if (pl.n[b] != 0) continue;
            const size_t base = static_cast<size_t>(b) * T * H * D;
            for (int i = t0; i < T * H * D; i += nt) store_out(p, base + i, 0.0f);
        }
        const int U = B * KVH;
        const int u_end = (cta + 1) * U / static_cast<int>(gridDim.x);   // < 2^31: U <= 4096
        for (int u = cta * U / static_cast<int>(gridDim.x) + t0; u < u_end; u += nt) {
            const int b = u / KVH, kvh = u - (u / KVH) * KVH;
            int4 e = make_int4(0, 0, 0, 0);
            if (pl.n[b] != 0 && pl.g_eff > 0) {
                const SegmentParts sp(pl, b, kvh, p.dyn_slot_base);
                e = make_int4(sp.first_s, sp.ns_parts, sp.dk0, sp.nd_parts);
            }
            p.ws_segs[u] = e;
        }
    };
    if (cta >= pl.g_eff) {   // (also for an all-empty batch)
        bookkeeping(tid, static_cast<int>(blockDim.x));
        return;
    }

    if (warp == 1) ptx::tmem_alloc(ptx::smem_addr(&sm.tmem_base), Cfg::TMEM_COLS);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t stage0 = ptx::smem_addr(&sm.stage[0][0]);
    // Stage q of the K ring is stage[q % KST]; stage q of the V ring is stage[KST + q % VST].
    constexpr int RST1 = Cfg::RST > 0 ? Cfg::RST : 1;
    auto kst = [&](uint32_t q) { return static_cast<int>(q % KST); };
    auto vst = [&](uint32_t q) { return KST + static_cast<int>(q % VST); };
    auto rstg = [&](uint32_t q) { return KST + VST + static_cast<int>(q % RST1); };
    // bounded wait (whole warp) for K-ring (v = false) or V-ring stage q to be full
    auto wait_full = [&](bool v, uint32_t q) -> bool {
        const int s = v ? vst(q) : kst(q);
        const uint32_t ph = (q / (v ? VST : KST)) & 1u;
        return __all_sync(0xffffffffu, wait_bounded(ptx::smem_addr(&sm.full[s]), ph, &sm.abort_flag,
                                                     p.ws_flags));
    };

    if (warp == 0) {
        // ============================ producer ============================
        if (lane == 0) {
            const uint64_t policy = ptx::policy_evict_first();
            // Q rows: the query rows, or over a K=V cache the hi and lo rows of q * w on the
            // unrotated dims (the rotated dims' blocks hold R(-t f) q, written per tile)
            const uint32_t q_bytes = static_cast<uint32_t>((Cfg::KEQV ? (NSUB - 2) * 2 * R : NSUB * R) * 128);
            constexpr uint32_t kPageBytes = kPageRows * 128;
            uint32_t kseq = 0, vseq = 0, rseq = 0;   // stages issued on the K, V and R rings
            uint32_t vpush = 0;                      // K=V: tiles handed to the V producer
            const uint64_t policy_keep = ptx::policy_evict_normal();
            uint32_t n_piece = 0;    // pieces started (O^T buffer n_piece & 1)
            bool ok = true;
            // Q of the newest piece, when its load still waits for the previous piece's
            // last scores: the load completes on the full barrier of the piece's first K
            // stage, which already expects its bytes.  Every wait of the producer keeps
            // servicing it, so the K stages of the piece stream meanwhile.
            MqPendingQ qs;
            qs.pend = false;
            qs.issued = 0;
            qs.b = qs.kvh = 0;
            qs.bar = 0;
            qs.empty_bar = ptx::smem_addr(&sm.q_empty);
            qs.dst = ptx::smem_addr(&sm.q[0]);
            qs.map = &tm_q;
            qs.policy = policy;
            auto service_q = [&]() { mq_service_q<Cfg>(qs); };
            // Bounded wait on a stage barrier (or, with bar == 0, for the pending Q to be
            // issued) that services the pending Q while it waits.  Over a K=V cache the
            // polling loop is out of line (one copy for the producer's many wait sites:
            // 1387 -> 1358 us on global_keqv_b16_s131072); the multi-query configurations
            // keep it inline (out of line they were 4-6% slower, the pending-Q state then
            // living in local memory).
            auto wait_servicing = [&](uint32_t bar, uint32_t parity) -> bool {
                service_q();
                if (bar ? ptx::mbar_try_wait(bar, parity) : !qs.pend) return true;
                if constexpr (Cfg::KEQV) {
                    return mq_poll_servicing<Cfg>(bar, parity, qs, &sm.abort_flag, p.ws_flags);
                } else {
                    const uint64_t t0 = ptx::globaltimer_ns();
                    for (uint32_t round = 0;; ++round) {
                        service_q();
                        for (int i = 0; i < 8; ++i)
                            if (bar ? ptx::mbar_try_wait(bar, parity) : !qs.pend) return true;
                        if (sm.abort_flag) return false;
                        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs || round > kWaitMaxRounds) {
                            sm.abort_flag = 1;
                            atomicOr(p.ws_flags, kFlagWaitTimeout);
                            return false;
                        }
                    }
                }
            };
            const bool dynamic = pl.n_dyn > 0;
            int claimed = -1;
            MqTile prev;
            bool have_prev = false;

            // One block of tile d: its K rows (NK stages), V rows (NSUB stages) or, on a K=V
            // cache, the rotated dims (R, 2 stages); or an end-of-work marker on the K or
            // the R ring.  Over a K=V cache, the K and R blocks are the first read of the
            // value tile (kept in L2 for the V block's second read); the R block holds the
            // column blocks of dims [0, 64) and [D/2, D/2 + 64), the K block the others.
            auto emit_block = [&](const MqTile& d, int kind) -> bool {
                const int32_t* bt_row =
                    kPaged ? p.block_table + static_cast<size_t>(d.b) * p.max_pages : nullptr;
                // paged: load the pages that hold attended positions of the sequence
                const int npage = kPaged ? (d.zhi + kPageRows - 1) / kPageRows : 0;
                const int ring = (kind == kMqKindV) ? 1 : (kind == kMqKindR || kind == kMqKindDoneR) ? 2 : 0;
                const int nst = ring == 1 ? NSUB : ring == 2 ? 2 : Cfg::NK;
                const uint64_t pol = (Cfg::KEQV && ring != 1) ? policy_keep : policy;
                for (int sub = 0; sub < nst; ++sub) {
                    uint32_t& seq = ring == 1 ? vseq : ring == 2 ? rseq : kseq;
                    const int s = ring == 1 ? vst(seq) : ring == 2 ? rstg(seq) : kst(seq);
                    const uint32_t ph = (seq / (ring == 1 ? VST : ring == 2 ? RST1 : KST)) & 1u;
                    if (!wait_servicing(ptx::smem_addr(&sm.empty[s]), ph ^ 1u)) return false;
                    if (ring == 0) sm.kind[s] = kind;
                    if (ring == 2) sm.rkind[s - KST - VST] = kind;
                    const uint32_t full_bar = ptx::smem_addr(&sm.full[s]);
                    if (kind == kMqKindDone || kind == kMqKindDoneR) {
                        ptx::mbar_arrive(full_bar);
                        ++seq;
                        continue;
                    }
                    const bool with_q = kind == kMqKindK && sub == 0 && (d.flags & kDescFirst);
                    // at most one Q load pending: the previous piece's goes out first
                    if (with_q && !wait_servicing(0u, 0u)) return false;
                    if (sub == 0 && ring == 0) sm.desc[s] = d;
                    if (sub == 0 && ring == 2) sm.rdesc[s - KST - VST] = d;
                    // (RAGGED) a tile at the end of its sequence (fewer than 128 rows attended)
                    // loads only the 16-row boxes that hold attended rows; the rows after them
                    // keep stale data, which the masks and the P.V warp's fix-up exclude
                    const int nrag =
                        (!kPaged && Cfg::RAGGED && d.zhi < kMqTile) ? (d.zhi + kPageRows - 1) / kPageRows : 0;
                    const uint32_t bytes =
                        (kPaged ? static_cast<uint32_t>(npage) * kPageBytes
                                : (nrag > 0 ? static_cast<uint32_t>(nrag) * kPageBytes : kMqStageBytes)) +
                        (with_q ? q_bytes : 0u);
                    ptx::mbar_arrive_expect_tx(full_bar, bytes);
                    if (with_q) {
                        qs.pend = true;
                        qs.b = d.b;
                        qs.kvh = d.kvh;
                        qs.bar = full_bar;
                    }
                    const CUtensorMap* map = kind == kMqKindK ? &tm_k : &tm_v;
                    const uint32_t dst = stage0 + s * kMqStageBytes;
                    // column block of the stage: K=V K blocks skip blocks 0 and NSUB/2
                    int cb = sub;
                    if (Cfg::KEQV && ring == 0) cb = sub + 1 + (sub >= NSUB / 2 - 1 ? 1 : 0);
                    if (ring == 2) cb = sub * (NSUB / 2);
                    const int chunk = d.kvh * NSUB + cb;
                    if (kPaged) {
                        for (int j = 0; j < npage; ++j) {
                            int page = bt_row[(d.t >> 4) + j];
                            if (page < 0 || page >= p.num_pages) page = 0;   // flagged by the softmax warps
                            ptx::tma_load_4d(dst + j * kPageBytes, map, full_bar, 0, 0, chunk, page, pol);
                        }
                    } else if (Cfg::RAGGED && nrag > 0) {
                        const CUtensorMap* map16 = kind == kMqKindK ? &tm_k16 : &tm_v16;
                        for (int j = 0; j < nrag; ++j)
                            ptx::tma_load_4d(dst + j * kPageBytes, map16, full_bar, 0, d.t + j * kPageRows,
                                             chunk, d.b, pol);
                    } else {
                        // rows past the end of the cache read as zeros
                        ptx::tma_load_4d(dst, map, full_bar, 0, d.t, chunk, d.b, pol);
                    }
                    ++seq;
                    service_q();
                }
                return true;
            };
            // K=V: hands tile d (or, flagged kDescDone, the end of work) to the V producer.
            auto push_v = [&](const MqTile& d) -> bool {
                const uint32_t k = vpush % kMqVq;
                if (!wait_servicing(ptx::smem_addr(&sm.vq_empty[k]), ((vpush / kMqVq) & 1u) ^ 1u))
                    return false;
                sm.vq[k] = d;
                ptx::mbar_arrive(ptx::smem_addr(&sm.vq_full[k]));   // releases the descriptor
                ++vpush;
                return true;
            };
            // Tiles arrive in order.  Multi-query: K(i), then V(i - 1).  K=V: K(i), tile i to
            // the V producer, then R(i).  R(i) waits for the derivation of tile i - 1 to free
            // the R ring; the scores warp does not wait for any derivation, so K(i) goes out
            // first and the K stream runs ahead of the derivation.
            auto emit_tile = [&](MqTile nxt) -> bool {
                if constexpr (Cfg::KEQV) {
                    if (!(emit_block(nxt, kMqKindK) && push_v(nxt) && emit_block(nxt, kMqKindR)))
                        return false;
                } else {
                    if (!emit_block(nxt, kMqKindK)) return false;
                    if (have_prev && !emit_block(prev, kMqKindV)) return false;
                    prev = nxt;
                    have_prev = true;
                }
                return true;
            };
            uint32_t tiles_emitted = 0;
            // The tiles of positions [p0, p1) of segment (b, kvh).
            auto emit_piece = [&](int b, int kvh, int p0, int p1, int slot, bool unit_end) -> bool {
                const uint32_t ob = n_piece & 1u;
                ++n_piece;
                const int lo = pl.lo[b], L = lo + pl.n[b];
                const int t_first = kPaged ? (p0 & ~(kPageRows - 1)) : p0;
                for (int t = t_first; t < p1; t += kMqTile) {
                    const bool last = t + kMqTile >= p1;
                    if (dynamic && unit_end && last)
                        claimed = static_cast<int>(atomicAdd(p.ws_claim, 1u));
                    MqTile d;
                    d.b = b;
                    d.kvh = kvh;
                    d.t = t;
                    d.vlo = (p0 > t ? p0 : t) - t;
                    d.vhi = (p1 < t + kMqTile ? p1 : t + kMqTile) - t;
                    d.zlo = lo > t ? lo - t : 0;
                    d.zhi = L < t + kMqTile ? L - t : kMqTile;
                    d.slot = slot;
                    d.flags = (t == t_first ? kDescFirst : 0) | (last ? kDescLast : 0);
                    d.ob = Cfg::OBUFS == 2 ? static_cast<int>(ob) : 0;
                    if (!emit_tile(d)) return false;
                    // test mode: wait for a barrier that nothing completes (times out)
                    // (after the piece's Q load has gone out, so that every copy the
                    // producer drains on the way out completes)
                    if ((p.test_flags & kTestStall) && ++tiles_emitted == 1) {
                        if (!wait_servicing(0u, 0u)) return false;
                        if (!wait_bounded(ptx::smem_addr(&sm.stall_bar), 0u, &sm.abort_flag, p.ws_flags,
                                          kTestStallNs))
                            return false;
                    }
                }
                return true;
            };

            // the static unit of this CTA, then dynamic chunks (as in the single-query kernel);
            // one call site of emit_piece keeps the producer's code small
            long long x = static_unit_begin(pl, cta);
            const long long stop = static_unit_begin(pl, cta + 1);
            Piece pc;
            while (ok && next_piece(pl, p, cta, kMqTile, dynamic, x, stop, claimed, pc))
                ok = emit_piece(pc.b, pc.kvh, pc.p0, pc.p1, pc.slot, pc.unit_end);
            // end of work: end-of-work markers where the next K (and R) block would be,
            // then the blocks still owed
            if (ok) {
                MqTile none;
                none.b = none.kvh = none.t = none.vlo = none.vhi = none.zlo = none.zhi = 0;
                none.slot = none.ob = 0;
                none.flags = kDescDone;
                if constexpr (Cfg::KEQV) {
                    ok = emit_block(none, kMqKindDoneR);
                    if (ok) ok = emit_block(none, kMqKindDone);
                    if (ok) ok = push_v(none);
                } else {
                    ok = emit_block(none, kMqKindDone);
                    if (ok && have_prev) ok = emit_block(prev, kMqKindV);
                }
            }
            if (!ok) {
                // let every copy already issued land before the CTA exits
                for (uint32_t tt = kseq > static_cast<uint32_t>(KST) ? kseq - KST : 0u; tt < kseq; ++tt)
                    wait_drain(ptx::smem_addr(&sm.full[kst(tt)]), (tt / KST) & 1u);
                for (uint32_t tt = vseq > static_cast<uint32_t>(VST) ? vseq - VST : 0u; tt < vseq; ++tt)
                    wait_drain(ptx::smem_addr(&sm.full[vst(tt)]), (tt / VST) & 1u);
                for (uint32_t tt = rseq > static_cast<uint32_t>(RST1) ? rseq - RST1 : 0u; tt < rseq; ++tt)
                    wait_drain(ptx::smem_addr(&sm.full[rstg(tt)]), (tt / RST1) & 1u);
            }
        }
    } else if (warp == 1) {
        // =================== scores: S^T[pos, r] = K Q^T (lane 0 issues) ===================
        const uint32_t idesc_s = ptx::idesc_bf16_f32(kMqTile, N, 0, 0);
        for (uint32_t i = 0;; ++i) {
            // tile i's K block (or the end-of-work marker) on the K ring
            uint32_t seq = i * Cfg::NK;
            if (!wait_full(false, seq)) break;
            ptx::tc_fence_after();
            const bool done = sm.kind[kst(seq)] == kMqKindDone;
            const MqTile d = sm.desc[kst(seq)];
            // S buffer i % 2 is free once the softmax warps have read tile i - 2
            if (!__all_sync(0xffffffffu, wait_bounded(ptx::smem_addr(&sm.s_empty[i & 1u]),
                                                      ((i >> 1) & 1u) ^ 1u, &sm.abort_flag, p.ws_flags)))
                break;
            ptx::tc_fence_after();
            if (done) {
                // release the end-of-work stages; the softmax warps learn there is no tile i
                bool ok = true;
                for (int sub = 0; sub < Cfg::NK && ok; ++sub) {
                    if (sub > 0) ok = wait_full(false, seq);
                    if (ok && lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sm.empty[kst(seq)]));
                    ++seq;
                }
                if (ok && lane == 0) {
                    sm.s_desc[i & 1u].flags = kDescDone;
                    ptx::mbar_arrive(ptx::smem_addr(&sm.s_full[i & 1u]));
                    ptx::mbar_arrive(ptx::smem_addr(&sm.s_full[i & 1u]));
                }
                break;
            }
            const uint32_t s_col = tmem + Cfg::TMEM_S + (i & 1u) * NMAX;
            const uint32_t qbase = ptx::smem_addr(&sm.q[0]);
            bool ok = true;
            for (int sub = 0; sub < Cfg::NK; ++sub) {
                if (sub > 0) {
                    ok = wait_full(false, seq);
                    if (!ok) break;
                    ptx::tc_fence_after();
                }
                const int s = kst(seq);
                // column block of the stage (K=V: blocks 0 and NSUB/2 are the rotated dims)
                const int cb = Cfg::KEQV ? sub + 1 + (sub >= NSUB / 2 - 1 ? 1 : 0) : sub;
                if (lane == 0) {
                    const uint32_t a0 = stage0 + s * kMqStageBytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = ptx::smem_desc(a0 + kk * 32, 16, 1024, ptx::kSwizzle128B);
                        const uint64_t bq = ptx::smem_desc(qbase + cb * Cfg::QATOM + kk * 32, 16, 1024,
                                                           ptx::kSwizzle128B);
                        ptx::umma_ss(s_col, a, bq, idesc_s, (sub | kk) != 0 ? 1u : 0u);
                    }
                    ptx::umma_commit(ptx::smem_addr(&sm.empty[s]));
                }
                __syncwarp();
                ++seq;
            }
            if (!ok) break;
            // (over a K=V cache the rotated dims are added by a softmax thread once the
            // keys are derived, so this warp moves on to the next tile's K block)
            if (lane == 0) {
                if (d.flags & kDescLast) ptx::umma_commit(ptx::smem_addr(&sm.q_empty));
                ptx::umma_commit(ptx::smem_addr(&sm.s_full[i & 1u]));
                sm.s_desc[i & 1u] = d;
                ptx::mbar_arrive(ptx::smem_addr(&sm.s_full[i & 1u]));
            }
            __syncwarp();
        }
        // every mma issued has completed before TMEM is released
        if (lane == 0) {
            ptx::umma_commit(ptx::smem_addr(&sm.drain[0]));
            wait_drain(ptx::smem_addr(&sm.drain[0]), 0u);
        }
        __syncwarp();
    } else if (warp == Cfg::PV_WARP) {
        // ========= P.V: O^T[d, r] += V^T[d, pos] P^T[pos, r] (lane 0 issues) + V fix-up =========
        // P^T holds the bf16 hi parts in rows [0, PLO) and the lo parts in rows
        // [PLO, 2 PLO): one mma applies P to ~16 significant bits.
        const uint32_t idesc_o = ptx::idesc_bf16_f32(kMqTile, Cfg::PROWS, 1, 0);
        for (uint32_t i = 0;; ++i) {
            if (!__all_sync(0xffffffffu, wait_bounded(ptx::smem_addr(&sm.p_full[i & 1u]), (i >> 1) & 1u,
                                                      &sm.abort_flag, p.ws_flags)))
                break;
            ptx::tc_fence_after();
            // no tile i (the flag names the tile: it may be set while tile i - 1's P
            // is read)
            if (static_cast<int>(i) >= sm.pv_stop) break;
            const MqTile d = sm.p_desc[i & 1u];
            const bool fix = d.zlo > 0 || d.zhi < kMqTile;
            const uint32_t pbase = ptx::smem_addr(&sm.pm[i & 1u][0]);
            uint32_t seq = i * NSUB;   // tile i's V block on the V ring
            bool ok = true;
            for (int mb = 0; mb < NB; ++mb) {
                // the two stages of head-dim block mb (adjacent: seq is even, VST even)
                ok = wait_full(true, seq) && wait_full(true, seq + 1);
                if (!ok) break;
                const int s = vst(seq);
                if (fix) {
                    // rows outside the attended range of the sequence may hold anything
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t st = stage0 + (s + h) * kMqStageBytes;
                        for (int row = lane; row < kMqTile; row += 32) {
                            if (row >= d.zlo && row < d.zhi) continue;
                            const uint32_t ra = st + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
                            for (int u = 0; u < 8; ++u) ptx::sts128(ra + u * 16, 0u, 0u, 0u, 0u);
                        }
                    }
                    ptx::fence_proxy_async_smem();
                }
                __syncwarp();
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t a0 = stage0 + s * kMqStageBytes;
                    const uint32_t o_col = tmem + Cfg::TMEM_O + d.ob * Cfg::OBUF + mb * Cfg::PROWS;
#pragma unroll
                    for (int kk = 0; kk < kMqTile / 16; ++kk) {
                        const uint64_t a = ptx::smem_desc(a0 + kk * 2048, kMqStageBytes, 1024,
                                                          ptx::kSwizzle128B);
                        const uint64_t bp = ptx::smem_desc(pbase + kk * 2 * kMqPLbo, kMqPLbo, kMqPSbo,
                                                           ptx::kSwizzleNone);
                        ptx::umma_ss(o_col, a, bp, idesc_o, ((d.flags & kDescFirst) && kk == 0) ? 0u : 1u);
                    }
                    ptx::umma_commit(ptx::smem_addr(&sm.empty[s]));
                    ptx::umma_commit(ptx::smem_addr(&sm.empty[s + 1]));
                }
                __syncwarp();
                seq += 2;
            }
            if (!ok) break;
            if (lane == 0) {
                ptx::umma_commit(ptx::smem_addr(&sm.o_ready[i & 1u]));
                ptx::umma_commit(ptx::smem_addr(&sm.p_empty[i & 1u]));
            }
            __syncwarp();
        }
        if (lane == 0) {
            ptx::umma_commit(ptx::smem_addr(&sm.drain[1]));
            wait_drain(ptx::smem_addr(&sm.drain[1]), 0u);
        }
        __syncwarp();
    } else if (Cfg::SPLIT_V && warp == Cfg::V_WARP) {
        // ========== K=V: V producer, tile i's V blocks in tile order (lane 0) ==========
        // The tiles come from the producer through the descriptor FIFO.
        if (lane == 0) {
            const uint64_t policy = ptx::policy_evict_first();
            constexpr uint32_t kPageBytes = kPageRows * 128;
            uint32_t vseq = 0;   // stages issued on the V ring
            bool ok = true;
            for (uint32_t n = 0; ok; ++n) {
                const uint32_t k = n % kMqVq;
                ok = wait_bounded(ptx::smem_addr(&sm.vq_full[k]), (n / kMqVq) & 1u, &sm.abort_flag,
                                  p.ws_flags);
                if (!ok) break;
                const MqTile d = sm.vq[k];
                ptx::mbar_arrive(ptx::smem_addr(&sm.vq_empty[k]));
                if (d.flags & kDescDone) break;
                const int32_t* bt_row =
                    kPaged ? p.block_table + static_cast<size_t>(d.b) * p.max_pages : nullptr;
                // paged: the pages that hold attended positions of the sequence
                const int npage = kPaged ? (d.zhi + kPageRows - 1) / kPageRows : 0;
                // a tile at the end of its sequence: only the 16-row boxes with attended rows
                const int nrag =
                    (!kPaged && Cfg::RAGGED && d.zhi < kMqTile) ? (d.zhi + kPageRows - 1) / kPageRows : 0;
                for (int sub = 0; sub < NSUB; ++sub) {
                    const int s = vst(vseq);
                    ok = wait_bounded(ptx::smem_addr(&sm.empty[s]), ((vseq / VST) & 1u) ^ 1u,
                                      &sm.abort_flag, p.ws_flags);
                    if (!ok) break;
                    const uint32_t vfull = ptx::smem_addr(&sm.full[s]);
                    ptx::mbar_arrive_expect_tx(
                        vfull, kPaged ? static_cast<uint32_t>(npage) * kPageBytes
                                      : (nrag > 0 ? static_cast<uint32_t>(nrag) * kPageBytes : kMqStageBytes));
                    const uint32_t dst = stage0 + s * kMqStageBytes;
                    const int chunk = d.kvh * NSUB + sub;
                    if (kPaged) {
                        for (int j = 0; j < npage; ++j) {
                            int page = bt_row[(d.t >> 4) + j];
                            if (page < 0 || page >= p.num_pages) page = 0;   // flagged by the softmax warps
                            ptx::tma_load_4d(dst + j * kPageBytes, &tm_v, vfull, 0, 0, chunk, page, policy);
                        }
                    } else if (Cfg::RAGGED && nrag > 0) {
                        for (int j = 0; j < nrag; ++j)
                            ptx::tma_load_4d(dst + j * kPageBytes, &tm_v16, vfull, 0, d.t + j * kPageRows,
                                             chunk, d.b, policy);
                    } else {
                        // rows past the end of the cache read as zeros
                        ptx::tma_load_4d(dst, &tm_v, vfull, 0, d.t, chunk, d.b, policy);
                    }
                    ++vseq;
                }
            }
            if (!ok) {
                // let every copy already issued land before the CTA exits
                for (uint32_t tt = vseq > static_cast<uint32_t>(VST) ? vseq - VST : 0u; tt < vseq; ++tt)
                    wait_drain(ptx::smem_addr(&sm.full[vst(tt)]), (tt / VST) & 1u);
            }
        }
        __syncwarp();
    } else if (Cfg::KEQV && warp >= 2 + Cfg::SMX_WARPS) {
        // ======= K=V: key derivation (warps 6..13, two per TMEM lane quarter) =======
        // Thread j of lane quarter q owns TMEM lane j = tile row j, the two warps of a
        // quarter halves h of its 64 rotated pairs.  For tile i (first
        // position t) the keys on the rotated dims are rope(w * v, t + j): pair i of the
        // row rotated by (t + j) f_i.  R((t + j) f) = R(t f) R(j f), and
        // <q, R(t f) y> = <R(-t f) q, y>, so the keys here are R(j f) (w * v), with factors
        // that do not depend on the tile (TRIG columns, set once per CTA), and the scores'
        // B operand on those dims is R(-t f) q, rotated once per tile (8 heads x 64 pairs).
        // Both are written as f16 hi + lo parts (~22 significant bits each; |values| stay
        // far below the f16 range), so the rotated dims lose nothing to the split.
        if constexpr (Cfg::KEQV) {
            constexpr int kDThreads = Cfg::DRV_THREADS;
            const int q4 = warp & 3;
            const int h = (warp - 2 - Cfg::SMX_WARPS) >> 2;   // half of the pairs
            const int j = 32 * q4 + lane;
            const int did = tid - 64 - Cfg::SMX_THREADS;   // 0 .. kDThreads - 1
            const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q4) << 16);
            // the factors of row j: cos and sin of j f_i (|j f_i| < 128) times the k_norm
            // weights of the pair's two dims
            {
#pragma unroll 1
                for (int c16 = 8 * h; c16 < 8 * h + 8; ++c16) {   // 16 columns = 2 pair groups
                    uint32_t cols[16];
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const int i = 4 * c16 + 2 * g + t;
                            float sn, cs;
                            sincosf(static_cast<float>(static_cast<double>(j) * p.rope_freq[i]), &sn, &cs);
                            const float wa = __bfloat162float(p.w_k[i]);
                            const float wb = __bfloat162float(p.w_k[D / 2 + i]);
                            cols[8 * g + t] = __float_as_uint(cs * wa);
                            cols[8 * g + 2 + t] = __float_as_uint(-sn * wb);
                            cols[8 * g + 4 + t] = __float_as_uint(cs * wb);
                            cols[8 * g + 6 + t] = __float_as_uint(sn * wa);
                        }
                    }
                    ptx::tmem_st16(lane_addr + Cfg::TMEM_TRIG + 16 * c16, cols);
                }
                ptx::tmem_wait_st();
            }
            // R(-t f) q: thread did takes head r = did / 32 and pairs [2 (did % 32), + 2)
            const int qr = did >> 5;
            const int qp = (did & 31) * 2;
            float qa[2] = {0.f, 0.f}, qb[2] = {0.f, 0.f};
            int seg_b = -1, seg_kvh = -1;
            const uint32_t qrot = ptx::smem_addr(&sm.q[0]);   // column blocks 0 and NSUB/2
            // byte offset of elements [qp, qp + 2) of row rr in a swizzled column block
            auto qrot_off = [&](int rr) -> uint32_t {
                return static_cast<uint32_t>((rr >> 3) * 1024 + (rr & 7) * 128 +
                                             ((((qp >> 3) ^ (rr & 7)) << 4) | ((qp & 7) * 2)));
            };
            ptx::named_barrier_sync(4, kDThreads);
            for (uint32_t ti = 0;; ++ti) {
                const uint32_t q0 = 2u * ti;
                // the tile's two R stages, and the keys' TMEM and the q buffer free (the
                // rotated mma of the previous tile completed)
                const bool okd =
                    wait_bounded(ptx::smem_addr(&sm.full[rstg(q0)]), (q0 / RST1) & 1u, &sm.abort_flag,
                                 p.ws_flags) &&
                    wait_bounded(ptx::smem_addr(&sm.full[rstg(q0 + 1)]), ((q0 + 1) / RST1) & 1u,
                                 &sm.abort_flag, p.ws_flags) &&
                    wait_bounded(ptx::smem_addr(&sm.krot_empty), (ti & 1u) ^ 1u, &sm.abort_flag,
                                 p.ws_flags);
                if (ptx::named_barrier_or(4, kDThreads, !okd)) break;
                ptx::tc_fence_after();
                const int rs = rstg(q0) - KST - VST;
                if (sm.rkind[rs] == kMqKindDoneR) break;
                const MqTile d = sm.rdesc[rs];
                if (d.b != seg_b || d.kvh != seg_kvh) {
                    // a new segment: this thread's q values of the rotated dims
                    seg_b = d.b;
                    seg_kvh = d.kvh;
                    const __nv_bfloat16* qrow =
                        p.q + (static_cast<size_t>(d.b) * H + d.kvh * G + qr) * D + qp;
                    const uint32_t xa = *reinterpret_cast<const uint32_t*>(qrow);
                    const uint32_t xb = *reinterpret_cast<const uint32_t*>(qrow + D / 2);
                    qa[0] = bf16lo(xa);
                    qa[1] = bf16hi(xa);
                    qb[0] = bf16lo(xb);
                    qb[1] = bf16hi(xb);
                }
                // cos, sin of t f_i: the angle reaches 2.6e5 rad, so it is reduced mod 2 pi
                // in fp64 before sincosf
                if (did < 64) {
                    const double ang = static_cast<double>(d.t) * p.rope_freq[did];
                    const double turns = rint(ang * 0.15915494309189535);   // 1 / (2 pi)
                    const double rr = fma(-turns, 6.283185307179586, ang);
                    float sn, cs;
                    sincosf(static_cast<float>(rr), &sn, &cs);
                    sm.rope.base[did] = make_float2(cs, sn);
                }
                ptx::named_barrier_sync(5, kDThreads);
                // R(-t f) q: (a, b) -> (a cos + b sin, b cos - a sin); f16 hi rows [0, G),
                // lo rows [G, 2 G); block 0 holds dims i, block 1 dims D/2 + i
                {
                    float ra[2], rb[2];
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const float2 cs = sm.rope.base[qp + t];
                        ra[t] = qa[t] * cs.x + qb[t] * cs.y;
                        rb[t] = qb[t] * cs.x - qa[t] * cs.y;
                    }
                    const __half2 h0 = __floats2half2_rn(ra[0], ra[1]);
                    const __half2 h1 = __floats2half2_rn(rb[0], rb[1]);
                    const __half2 l0 = __floats2half2_rn(ra[0] - __low2float(h0), ra[1] - __high2float(h0));
                    const __half2 l1 = __floats2half2_rn(rb[0] - __low2float(h1), rb[1] - __high2float(h1));
                    constexpr uint32_t kYBlock = (NSUB / 2) * Cfg::QATOM;
                    ptx::sts32(qrot + qrot_off(qr), *reinterpret_cast<const uint32_t*>(&h0));
                    ptx::sts32(qrot + kYBlock + qrot_off(qr), *reinterpret_cast<const uint32_t*>(&h1));
                    ptx::sts32(qrot + qrot_off(G + qr), *reinterpret_cast<const uint32_t*>(&l0));
                    ptx::sts32(qrot + kYBlock + qrot_off(G + qr), *reinterpret_cast<const uint32_t*>(&l1));
                }
                // the keys of row j: y = R(j f) (w * v) per pair, as packed fp32 pairs of
                // adjacent pairs (2m, 2m + 1):
                //   y_a = (cos w_a) v_a + (-sin w_b) v_b,  y_b = (cos w_b) v_b + (sin w_a) v_a
                const uint32_t sx = stage0 + rstg(q0) * kMqStageBytes;       // dims [0, 64)
                const uint32_t sy = stage0 + rstg(q0 + 1) * kMqStageBytes;   // dims [D/2, D/2 + 64)
                const uint32_t rowoff = (j >> 3) * 1024 + (j & 7) * 128;
                {   // this warp's half of the pairs: [32 h, 32 h + 32), 8 pairs per round
                    // (a rolled loop: the kernel's roles share the SM's instruction caches)
                    // keys columns: dims i (x) at i / 2, dims D/2 + i (y) at 32 + i / 2; lo parts
                    // 64 later
                    const uint32_t kb = lane_addr + Cfg::TMEM_KROT + 16 * h;
#pragma unroll 1
                    for (int u = 0; u < 4; ++u) {   // pairs 32 h + 8 u .. + 8
                        uint32_t hx[4], hy[4], lx[4], ly[4];
                        uint32_t f[32];
                        const uint32_t tcol = lane_addr + Cfg::TMEM_TRIG + 4 * (32 * h + 8 * u);
                        ptx::tmem_ld16(tcol, *reinterpret_cast<uint32_t(*)[16]>(&f[0]));
                        ptx::tmem_ld16(tcol + 16, *reinterpret_cast<uint32_t(*)[16]>(&f[16]));
                        const uint32_t unit = static_cast<uint32_t>(((4 * h + u) ^ (j & 7)) << 4);
                        const uint4 vx4 = ptx::lds128(sx + rowoff + unit);
                        const uint4 vy4 = ptx::lds128(sy + rowoff + unit);
                        ptx::tmem_wait_ld();
                        const uint32_t vx[4] = {vx4.x, vx4.y, vx4.z, vx4.w};
                        const uint32_t vy[4] = {vy4.x, vy4.y, vy4.z, vy4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {   // pair group 16 h + 4 u + e
                            const uint32_t* c = &f[8 * e];
                            const uint64_t va = ptx::f2_from_bf16x2(vx[e]);
                            const uint64_t vb = ptx::f2_from_bf16x2(vy[e]);
                            const uint64_t ya = ptx::f2_fma(ptx::f2_pack(__uint_as_float(c[0]), __uint_as_float(c[1])), va,
                                                            ptx::f2_mul(ptx::f2_pack(__uint_as_float(c[2]), __uint_as_float(c[3])), vb));
                            const uint64_t yb = ptx::f2_fma(ptx::f2_pack(__uint_as_float(c[4]), __uint_as_float(c[5])), vb,
                                                            ptx::f2_mul(ptx::f2_pack(__uint_as_float(c[6]), __uint_as_float(c[7])), va));
                            // f16 hi + lo parts
                            const float2 fa = ptx::f2_unpack(ya), fb = ptx::f2_unpack(yb);
                            const __half2 h0 = __floats2half2_rn(fa.x, fa.y);
                            const __half2 h1 = __floats2half2_rn(fb.x, fb.y);
                            const float2 g0 = __half22float2(h0), g1 = __half22float2(h1);
                            const float2 ra = ptx::f2_unpack(ptx::f2_sub(ya, ptx::f2_pack(g0.x, g0.y)));
                            const float2 rb = ptx::f2_unpack(ptx::f2_sub(yb, ptx::f2_pack(g1.x, g1.y)));
                            const __half2 l0 = __floats2half2_rn(ra.x, ra.y);
                            const __half2 l1 = __floats2half2_rn(rb.x, rb.y);
                            hx[e] = *reinterpret_cast<const uint32_t*>(&h0);
                            hy[e] = *reinterpret_cast<const uint32_t*>(&h1);
                            lx[e] = *reinterpret_cast<const uint32_t*>(&l0);
                            ly[e] = *reinterpret_cast<const uint32_t*>(&l1);
                        }
                        ptx::tmem_st4(kb + 4 * u, hx);
                        ptx::tmem_st4(kb + 32 + 4 * u, hy);
                        ptx::tmem_st4(kb + 64 + 4 * u, lx);
                        ptx::tmem_st4(kb + 96 + 4 * u, ly);
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::fence_proxy_async_smem();   // R(-t f) q is read by the tensor core
                // every thread is done with the R stages and the angle table, and has
                // stored its keys and its part of R(-t f) q
                ptx::named_barrier_sync(5, kDThreads);
                if (did == 0) {
                    ptx::mbar_arrive(ptx::smem_addr(&sm.empty[rstg(q0)]));
                    ptx::mbar_arrive(ptx::smem_addr(&sm.empty[rstg(q0 + 1)]));
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sm.krot_full));
            }
        }
    } else {
        // ================ softmax and epilogue (warps 2..9, two per TMEM lane quarter;
        // over a K=V cache warps 2..5, one per quarter) ================
        // Thread j of lane quarter q (warp % 4) owns TMEM lane j: position j of the
        // tile's scores and head-dim element j of each O^T block.  Where two warps share
        // a quarter they split the query rows: warps 2..5 rows [0, RH), warps 6..9
        // [RH, 2 RH).  Over a K=V cache the G query rows' scores are the sum of a hi
        // column r and a lo column G + r.
        constexpr int RH = Cfg::KEQV ? Cfg::RMAX : NMAX / 2;   // rows per warp
        // the loops over head-dim blocks (rescale, epilogue) stay rolled where that costs no
        // registers: the kernel's roles share the SM's instruction caches, and smaller code
        // misses them less (with 32 query rows rolling them spills, so they are unrolled)
        constexpr int kBlockUnroll = Cfg::RMAX > 16 ? NB : 1;
        constexpr int kSmx = Cfg::SMX_THREADS;
        const int q4 = warp & 3;
        const int r0 = Cfg::KEQV ? 0 : ((warp - 2) >> 2) * RH;   // first row of this warp
        const int j = 32 * q4 + lane;
        const int sid = tid - 64;                    // 0 .. kSmx - 1 over the softmax warps
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q4) << 16);
        const float nan = __uint_as_float(0x7fc00000u);
        float m_ref[RH], l_part[RH];
#pragma unroll
        for (int k = 0; k < RH; ++k) {
            m_ref[k] = -INFINITY;
            l_part[k] = 0.0f;
        }
        uint32_t bad_q = 0;   // bit t: query t attended a bad page in this piece
        bookkeeping(sid, kSmx);
        // P rows past the query rows in use stay zero (the P.V mma reads PROWS rows)
        for (int i = sid; i < 2 * Cfg::PBYTES / 16; i += kSmx)
            ptx::sts128(ptx::smem_addr(&sm.pm[0][0]) + i * 16, 0u, 0u, 0u, 0u);
        ptx::named_barrier_sync(3, kSmx);
        // A finished piece whose output is still to be written: its last tile and
        // that tile's index; its reference max, normaliser and bad bits are in smem.
        bool epi_pending = false;
        MqTile epi;
        uint32_t epi_i = 0;
        epi.b = epi.kvh = epi.slot = epi.ob = 0;
        // Writes the pending piece's output: waits for its last P.V, then reads this
        // warp's rows of its O^T buffer and stores the normalised rows (a piece that is
        // its whole segment) or the partial (acc, m, l).  False when the CTA is aborting.
        auto finish_piece = [&]() -> bool {
            const bool okw = wait_bounded(ptx::smem_addr(&sm.o_ready[epi_i & 1u]), (epi_i >> 1) & 1u,
                                          &sm.abort_flag, p.ws_flags);
            if (ptx::named_barrier_or(1, kSmx, !okw)) return false;
            ptx::tc_fence_after();
            const uint32_t bad_all = sm.epi_bad;
            const SegmentParts sp(pl, epi.b, epi.kvh, p.dyn_slot_base);
            const bool direct = sp.count() == 1;
            // This code runs once per piece, and mostly cold: its loop over head-dim blocks
            // stays rolled, each row's scale is taken once, and each kind of piece stores
            // through one short path, so that few instruction lines are fetched.  (Fully
            // unrolled, with a division and both output types per element, the last
            // epilogue of a CTA took ~15 us on decodeGQA B=8, T=4.)
            if (r0 < R) {
                // per row k of this warp: direct pieces 1 / l (0 for a row that saw no key,
                // NaN for a bad page), partials 1 (NaN for a bad page)
                float scale[RH];
#pragma unroll
                for (int k = 0; k < RH; ++k) {
                    const int r = r0 + k;
                    const bool bad = r < R && ((bad_all >> (r / G)) & 1u);
                    const float lr = (direct && r < R) ? sm.epi_l[r] : 1.0f;
                    scale[k] = bad ? nan : (lr == 0.0f ? 0.0f : 1.0f / lr);
                }
                // row r0 + k is query token r0 / G + k / G (r0 is a multiple of G), head
                // k % G of the group: output row (b T + t) H + kvh G + g of [B, T, H, D]
                const size_t out_row0 = (static_cast<size_t>(epi.b) * T + r0 / G) * H + epi.kvh * G;
                float* const part0 = p.ws_acc + (static_cast<size_t>(epi.slot) * R + r0) * D;
#pragma unroll 1
                for (int mb = 0; mb < NB; ++mb) {
                    // row r's sum is its hi column r plus its lo column PLO + r
                    uint32_t oh[RH], ol[RH];
                    const uint32_t ob = lane_addr + Cfg::TMEM_O + epi.ob * Cfg::OBUF + mb * Cfg::PROWS + r0;
                    ptx::tmem_ld<RH>(ob, oh);
                    ptx::tmem_ld<RH>(ob + Cfg::PLO, ol);
                    ptx::tmem_wait_ld();
                    const int dd = mb * 128 + j;
                    if (!direct) {
                        float* const dst = part0 + dd;
#pragma unroll
                        for (int k = 0; k < RH; ++k)
                            if (r0 + k < R)
                                dst[static_cast<size_t>(k) * D] =
                                    (__uint_as_float(oh[k]) + __uint_as_float(ol[k])) * scale[k];
                    } else if (p.out_f32) {
                        float* const dst = static_cast<float*>(p.out) + out_row0 * D + dd;
#pragma unroll
                        for (int k = 0; k < RH; ++k)
                            if (r0 + k < R) {
                                const float acc = __uint_as_float(oh[k]) + __uint_as_float(ol[k]);
                                dst[static_cast<size_t>((k / G) * H + k % G) * D] =
                                    scale[k] == 0.0f ? 0.0f : acc * scale[k];
                            }
                    } else {
                        __nv_bfloat16* const dst = static_cast<__nv_bfloat16*>(p.out) + out_row0 * D + dd;
#pragma unroll
                        for (int k = 0; k < RH; ++k)
                            if (r0 + k < R) {
                                const float acc = __uint_as_float(oh[k]) + __uint_as_float(ol[k]);
                                dst[static_cast<size_t>((k / G) * H + k % G) * D] =
                                    __float2bfloat16_rn(scale[k] == 0.0f ? 0.0f : acc * scale[k]);
                            }
                    }
                }
            }
            if (!direct && sid < R) {
                const bool bad = (bad_all >> (sid / G)) & 1u;
                float* ml = p.ws_ml + (static_cast<size_t>(epi.slot) * R + sid) * 2;
                ml[0] = bad ? 0.0f : sm.epi_m[sid];
                ml[1] = bad ? nan : sm.epi_l[sid];
            }
            ptx::tc_fence_before();
            return true;
        };
        for (uint32_t i = 0;; ++i) {
            bool ok = wait_bounded(ptx::smem_addr(&sm.s_full[i & 1u]), (i >> 1) & 1u, &sm.abort_flag,
                                   p.ws_flags);
            if (ptx::named_barrier_or(1, kSmx, !ok)) break;
            ptx::tc_fence_after();
            const MqTile d = sm.s_desc[i & 1u];
            if (d.flags & kDescDone) {
                // no tile i: the P.V warp stops too (a pending piece is finished below).
                // Like a tile's P, the signal waits until the P.V warp is done with tile
                // i - 2, so p_full[i % 2] never runs two phases ahead of it.
                ok = wait_bounded(ptx::smem_addr(&sm.p_empty[i & 1u]), ((i >> 1) & 1u) ^ 1u,
                                  &sm.abort_flag, p.ws_flags);
                if (ptx::named_barrier_or(1, kSmx, !ok)) break;
                if (sid == 0) sm.pv_stop = static_cast<int>(i);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sm.p_full[i & 1u]));
                break;
            }
            if constexpr (Cfg::KEQV) {
                // The rotated dims of tile i: A = the keys R(j f) (w * v) derived into TMEM
                // (hi, then lo), B = R(-t f) q of the tile in the Q buffer's column blocks 0
                // and NSUB/2 (hi rows [0, G), lo rows [G, 2 G)), all f16.  One thread adds
                // them to S once the keys are derived; the unrotated part is complete.
                ok = wait_bounded(ptx::smem_addr(&sm.krot_full), i & 1u, &sm.abort_flag, p.ws_flags);
                if (ptx::named_barrier_or(1, kSmx, !ok)) break;
                ptx::tc_fence_after();
                if (sid == 0) {
                    const uint32_t idesc_r = ptx::idesc_f16_f32(kMqTile, N, 0, 0);
                    const uint32_t s_col = tmem + Cfg::TMEM_S + (i & 1u) * NMAX;
                    const uint32_t qbase = ptx::smem_addr(&sm.q[0]);
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t a_t = tmem + Cfg::TMEM_KROT + part * 64 + kk * 8;
                            const uint64_t bq = ptx::smem_desc(
                                qbase + (kk < 4 ? 0 : NSUB / 2) * Cfg::QATOM + (kk & 3) * 32, 16, 1024,
                                ptx::kSwizzle128B);
                            ptx::umma_ts(s_col, a_t, bq, idesc_r, 1u);
                        }
                    // the keys and R(-t f) q may be overwritten with the next tile's
                    ptx::umma_commit(ptx::smem_addr(&sm.krot_empty));
                    ptx::umma_commit(ptx::smem_addr(&sm.r_full[i & 1u]));
                    // the issuer sees its mma complete even when the CTA is aborting (TMEM
                    // is released only after every mma has completed)
                    wait_drain(ptx::smem_addr(&sm.r_full[i & 1u]), (i >> 1) & 1u);
                }
                ok = wait_bounded(ptx::smem_addr(&sm.r_full[i & 1u]), (i >> 1) & 1u, &sm.abort_flag,
                                  p.ws_flags);
                if (ptx::named_barrier_or(1, kSmx, !ok)) break;
                ptx::tc_fence_after();
            }
            if (d.flags & kDescFirst) {
#pragma unroll
                for (int k = 0; k < RH; ++k) {
                    m_ref[k] = -INFINITY;
                    l_part[k] = 0.0f;
                }
                bad_q = 0;
            }
            const int L = pl.lo[d.b] + pl.n[d.b];
            const int pos = d.t + j;
            const bool in_piece = j >= d.vlo && j < d.vhi;
            bool page_bad = false;
            if (kPaged && in_piece) {
                const int page = p.block_table[static_cast<size_t>(d.b) * p.max_pages + (pos >> 4)];
                page_bad = page < 0 || page >= p.num_pages;
            }
            // scores of position j for this warp's rows, log2 units, masked per query
            uint32_t sr[RH];
            if constexpr (Cfg::KEQV) {
                uint32_t sa[NMAX];
                ptx::tmem_ld<NMAX>(lane_addr + Cfg::TMEM_S + (i & 1u) * NMAX, sa);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < RH; ++k)
                    sr[k] = __float_as_uint(__uint_as_float(sa[r0 + k]) + __uint_as_float(sa[Cfg::RMAX + r0 + k]));
            } else {
                ptx::tmem_ld<RH>(lane_addr + Cfg::TMEM_S + (i & 1u) * NMAX + r0, sr);
                ptx::tmem_wait_ld();
            }
            // S buffer i % 2 may take the scores of tile i + 2
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sm.s_empty[i & 1u]));
            float s[RH];
            bool need = false;
#pragma unroll
            for (int k = 0; k < RH; ++k) {
                const int r = r0 + k;
                const int t = r / G;
                const int hi_t = L - T + t + 1;
                const int lo_t = (p.window > 0 && hi_t > p.window) ? hi_t - p.window : 0;
                const bool valid = r < R && in_piece && pos >= lo_t && pos < hi_t;
                if (valid && page_bad) bad_q |= 1u << t;
                s[k] = valid ? __uint_as_float(sr[k]) * kLog2e : -INFINITY;
                need |= s[k] > m_ref[k] + kMqTau;
            }
            if (ptx::named_barrier_or(2, kSmx, need)) {
                // new reference max of every row: the tile's max where it is larger
#pragma unroll
                for (int k = 0; k < RH; ++k) {
                    float mx = s[k];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    if (lane == 0) sm.red[q4][r0 + k] = mx;
                }
                ptx::named_barrier_sync(3, kSmx);
                float alpha[RH];
#pragma unroll
                for (int k = 0; k < RH; ++k) {
                    const int r = r0 + k;
                    const float mt = fmaxf(fmaxf(sm.red[0][r], sm.red[1][r]), fmaxf(sm.red[2][r], sm.red[3][r]));
                    const float mn = fmaxf(m_ref[k], mt);
                    alpha[k] = (m_ref[k] == -INFINITY || mn == -INFINITY) ? 0.0f : exp2f(m_ref[k] - mn);
                    m_ref[k] = mn;
                }
                ptx::named_barrier_sync(3, kSmx);
                if (!(d.flags & kDescFirst)) {
                    // O^T holds the earlier tiles of this piece: rescale it once their
                    // P.V is complete (the P.V of this tile waits for p_full)
                    const uint32_t ip = i - 1;
                    ok = wait_bounded(ptx::smem_addr(&sm.o_ready[ip & 1u]), (ip >> 1) & 1u,
                                      &sm.abort_flag, p.ws_flags);
                    if (ptx::named_barrier_or(1, kSmx, !ok)) break;
                    ptx::tc_fence_after();
#pragma unroll (kBlockUnroll)
                    for (int mb = 0; mb < NB; ++mb) {
                        // the hi column and the lo column of each row
#pragma unroll
                        for (int part = 0; part < 2; ++part) {
                            uint32_t o[RH];
                            const uint32_t ta = lane_addr + Cfg::TMEM_O + d.ob * Cfg::OBUF +
                                                mb * Cfg::PROWS + part * Cfg::PLO + r0;
                            ptx::tmem_ld<RH>(ta, o);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < RH; ++k)
                                o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha[k]);
                            ptx::tmem_st<RH>(ta, o);
                        }
                    }
                    ptx::tmem_wait_st();
#pragma unroll
                    for (int k = 0; k < RH; ++k) l_part[k] *= alpha[k];
                }
            }
            // P buffer i % 2 is free once the P.V of tile i - 2 is done
            ok = wait_bounded(ptx::smem_addr(&sm.p_empty[i & 1u]), ((i >> 1) & 1u) ^ 1u, &sm.abort_flag,
                              p.ws_flags);
            if (ptx::named_barrier_or(1, kSmx, !ok)) break;
            if (r0 < N) {
                // hi part in row r, lo part in row PLO + r; rows past R stay zero
                const uint32_t pb = ptx::smem_addr(&sm.pm[i & 1u][0]);
#pragma unroll
                for (int k = 0; k < RH; ++k) {
                    const float pv = s[k] != -INFINITY ? exp2f(s[k] - m_ref[k]) : 0.0f;
                    l_part[k] += pv;
                    const __nv_bfloat16 hb = __float2bfloat16_rn(pv);
                    const __nv_bfloat16 lb = __float2bfloat16_rn(pv - __bfloat162float(hb));
                    ptx::sts16(pb + mq_p_off(r0 + k, j), *reinterpret_cast<const uint16_t*>(&hb));
                    ptx::sts16(pb + mq_p_off(Cfg::PLO + r0 + k, j), *reinterpret_cast<const uint16_t*>(&lb));
                }
            }
            // one O^T buffer: the pending piece's output is read before this new piece's
            // first P.V overwrites it
            if (Cfg::OBUFS == 1 && (d.flags & kDescFirst) && epi_pending) {
                if (!finish_piece()) break;
                epi_pending = false;
            }
            if (sid == 0) sm.p_desc[i & 1u] = d;
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sm.p_full[i & 1u]));
            if (epi_pending) {
                if (!finish_piece()) break;
                epi_pending = false;
            }
            if (!(d.flags & kDescLast)) continue;

            // ---- the piece is complete: its normaliser now, its output after the next
            // tile's P (so the softmax of that tile does not wait for this P.V) ----
#pragma unroll
            for (int k = 0; k < RH; ++k) {
                float v = l_part[k];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0) sm.red[q4][r0 + k] = v;
            }
            const uint32_t bq = __reduce_or_sync(0xffffffffu, bad_q);
            if (lane == 0) sm.red_bad[warp - 2] = bq;
            ptx::named_barrier_sync(3, kSmx);
            if (sid < NMAX)
                sm.epi_l[sid] = (sm.red[0][sid] + sm.red[1][sid]) + (sm.red[2][sid] + sm.red[3][sid]);
            if (q4 == 0 && lane < RH) {
                float mk = 0.0f;
#pragma unroll
                for (int k = 0; k < RH; ++k)
                    if (k == lane) mk = m_ref[k];
                sm.epi_m[r0 + lane] = mk;
            }
            if (sid == 0) {
                uint32_t bad_all = 0;
                for (int w = 0; w < Cfg::SMX_WARPS; ++w) bad_all |= sm.red_bad[w];
                sm.epi_bad = bad_all;
                if (bad_all) atomicOr(p.ws_flags, kFlagBadPage);
            }
            ptx::named_barrier_sync(3, kSmx);
            epi = d;
            epi_i = i;
            epi_pending = true;
        }
        // (uniform: every exit from the loop above is a collective decision)
        if (epi_pending) finish_piece();
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

}  // namespace gqa
