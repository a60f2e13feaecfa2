// C ABI of libgqadecode.so: argument checks, workspace handling, TMA tensor
// maps and the kernel launch.  See include/gqa_decode.h for the contract.
//
// Operation: the decode-step attention core `attn.core` of gemma-4-31B (Model
// Spec, "Compute-graph nodes", the slidingDecodeGQA and decodeGQA rows; tensor
// shapes from "Tensors of the main nodes"; 16-position pages from "At a glance",
// Shape domain row).
#include <atomic>
#include <cstdint>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "gqa_decode.h"
#include "launch.h"

namespace {

using gqa::kMaxCtas;

enum class Geometry { kNone, kSliding, kGlobal };

Geometry geometry_of(int H, int KVH, int D) {
    if (H == 32 && KVH == 16 && D == 256) return Geometry::kSliding;   // slidingDecodeGQA
    if (H == 32 && KVH == 4 && D == 512) return Geometry::kGlobal;     // decodeGQA
    return Geometry::kNone;
}

int heads_per_kv(Geometry g) { return g == Geometry::kSliding ? 2 : 8; }

// RoPE base of the global layers (Model Spec, `attn.rope` row for layers 5, 11, ..., 59).
constexpr double kGlobalRopeTheta = 1.0e6;
// K=V calls whose cache holds at least this many 128-position tiles per CTA take the
// tcgen05 kernel (measured: ~13 tiles per CTA ran 40% faster on the mma.sync kernel,
// ~430 tiles per CTA 16% faster on the tcgen05 kernel)
constexpr int kKeqvTcTilesPerCta = 64;

// ---- workspace layout --------------------------------------------------------
// [0, 4)              status word (uint32)
// [64, 68)            dynamic-chunk claim counter (zero between calls)
// [128, 132)          producers finished (zero between calls)
// [256, 65792)        per-(b, kvh) partial lists, 4096 x int4
// [65792, 82176)      per-(b, kvh) partials stored, 4096 x uint32 (zero between calls)
// [ml_off, ...)       softmax partial (m, l): slots x G x 2 floats
// [acc_off, ...)      softmax partial acc:    slots x G x D floats
// slots = kMaxCtas + B * KVH + kMaxDynUnits bounds the partials one call can
// store: static unit j keeps its piece of segment u at slot j + u, dynamic
// chunk k at slot kMaxCtas + B * KVH + k.
// The status word and the counters must be zero before a call; every completed
// call leaves them so (gqa_device_status zeroes the whole header after a call
// that raised a status bit, e.g. one that timed out half-way).
constexpr size_t kFlagsOff = 0;
constexpr size_t kClaimOff = 64;
constexpr size_t kDoneOff = 128;
constexpr size_t kSegsOff = 256;
constexpr size_t kMaxSegments = static_cast<size_t>(GQA_MAX_BATCH) * 16;
constexpr size_t kSegCountOff = kSegsOff + kMaxSegments * 16;
constexpr size_t kHeaderBytes = kSegCountOff + kMaxSegments * 4;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WorkspaceLayout {
    size_t ml_off, acc_off, operand_off, total;
};

// G = query rows per segment.  On the decodeGQA geometry the workspace also holds the
// single K=V path's scores operand, [B, KVH, 16, 512] bf16.
WorkspaceLayout layout_for(int B, int KVH, int G, int D) {
    const size_t slots = static_cast<size_t>(kMaxCtas) + static_cast<size_t>(B) * KVH +
                         gqa::kMaxDynUnits;
    WorkspaceLayout w;
    w.ml_off = align256(kHeaderBytes);
    w.acc_off = align256(w.ml_off + slots * G * 2 * sizeof(float));
    w.operand_off = align256(w.acc_off + slots * G * D * sizeof(float));
    const size_t operand = (KVH == 4 && D == 512) ? static_cast<size_t>(B) * KVH * 16 * D * 2 : 0;
    w.total = align256(w.operand_off + operand);
    return w;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- per-device state -----------------------------------------------------------
constexpr int kMaxDevices = 64;

struct DeviceState {
    std::mutex mu;
    int sm_count = 0;
    void* ws = nullptr;          // library-owned workspace
    size_t ws_bytes = 0;
};

DeviceState g_dev[kMaxDevices];

// Test modes of the calls that follow (GQA_TEST_* bits; 0 in normal use).
std::atomic<uint32_t> g_test_mode{0};

// Whether a K=V call runs on the tcgen05 kernel.  Long histories do (derived keys in
// TMEM); short ones are latency-bound: the tcgen05 kernel's pipeline fill and per-piece
// steps cost more than they save there, and the mma.sync streaming kernel finishes
// first.  The host knows only the cache capacity, so the split is on capacity tiles
// (128 positions) per CTA.
bool keqv_long_history(int B, int capacity, int KVH, int grid) {
    const long long cap_tiles = static_cast<long long>(B) * capacity * KVH / 128;
    return cap_tiles >= static_cast<long long>(kKeqvTcTilesPerCta) * grid;
}

// CTAs of one persistent launch on the current device (its SM count), or 0.
int device_grid() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    DeviceState& ds = g_dev[dev];
    std::lock_guard<std::mutex> lock(ds.mu);
    if (ds.sm_count == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return 0;
        ds.sm_count = n;
    }
    return ds.sm_count < kMaxCtas ? ds.sm_count : kMaxCtas;
}

}  // namespace

namespace gqa {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn_ptr = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn_ptr = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return fn_ptr;
}

}  // namespace gqa

namespace {

struct CallShape {
    Geometry geo;
    int B, H, KVH, D, window;
    int T = 1;   // query tokens per sequence
};

// Query tokens one multi-query call may carry for a geometry.
bool queries_ok(Geometry geo, int T) {
    return T >= 1 && T <= gqa::mq_max_queries(geo == Geometry::kSliding);
}

gqa_status_t check_common(const CallShape& c, const void* q, const void* out,
                          const int32_t* seq_lens, gqa_out_dtype_t out_dtype) {
    if (c.B < 0 || c.B > GQA_MAX_BATCH || c.window < 0) return GQA_ERR_INVALID_ARGUMENT;
    if (out_dtype != GQA_OUT_BF16 && out_dtype != GQA_OUT_F32) return GQA_ERR_INVALID_ARGUMENT;
    if (c.geo == Geometry::kNone) return GQA_ERR_UNSUPPORTED;
    if (c.B == 0) return GQA_OK;
    if (!q || !out || !seq_lens) return GQA_ERR_INVALID_ARGUMENT;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(seq_lens, 4))
        return GQA_ERR_INVALID_ARGUMENT;
    return GQA_OK;
}

// Resolves the workspace (caller's or library-owned) and the device's SM count.
gqa_status_t prepare(const CallShape& c, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream, void** ws_out, WorkspaceLayout* lay, int* grid) {
    const int G = heads_per_kv(c.geo);
    *lay = layout_for(c.B, c.KVH, G * c.T, c.D);   // partials hold T * g query rows
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
    DeviceState& ds = g_dev[dev];
    std::lock_guard<std::mutex> lock(ds.mu);
    if (ds.sm_count == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return GQA_ERR_CUDA;
        ds.sm_count = n;
    }
    *grid = ds.sm_count < kMaxCtas ? ds.sm_count : kMaxCtas;
    if (workspace) {
        if (workspace_bytes < lay->total || !aligned(workspace, 256)) return GQA_ERR_WORKSPACE;
        *ws_out = workspace;
        return GQA_OK;
    }
    if (ds.ws_bytes < lay->total) {
        if (ds.ws) {
            cudaFree(ds.ws);   // synchronises the device: no call still uses it
            ds.ws = nullptr;
            ds.ws_bytes = 0;
        }
        void* p = nullptr;
        if (cudaMalloc(&p, lay->total) != cudaSuccess) return GQA_ERR_CUDA;
        if (cudaMemsetAsync(p, 0, lay->total, stream) != cudaSuccess) {
            cudaFree(p);
            return GQA_ERR_CUDA;
        }
        ds.ws = p;
        ds.ws_bytes = lay->total;
    }
    *ws_out = ds.ws;
    return GQA_OK;
}

gqa_status_t run(const CallShape& c, bool paged, const void* q, const void* k, const void* v,
                 const int32_t* block_table, const int32_t* seq_lens, uint64_t rows,
                 uint64_t outer, int capacity, int ring, int num_pages, int max_pages, void* out,
                 gqa_out_dtype_t out_dtype, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream, const void* w_k = nullptr, bool multi_query = false) {
    if (!gqa::tensor_map_encoder()) return GQA_ERR_CUDA;
    void* ws = nullptr;
    WorkspaceLayout lay;
    int grid = 0;
    gqa_status_t st = prepare(c, workspace, workspace_bytes, stream, &ws, &lay, &grid);
    if (st != GQA_OK) return st;

    gqa::LaunchArgs a;
    std::memset(&a, 0, sizeof a);
    a.k = k;
    a.v = v;
    a.rows = rows;
    a.outer = outer;
    uint8_t* w = static_cast<uint8_t*>(ws);
    a.p.q = static_cast<const __nv_bfloat16*>(q);
    a.p.seq_lens = seq_lens;
    a.p.block_table = block_table;
    a.p.out = out;
    a.p.ws_acc = reinterpret_cast<float*>(w + lay.acc_off);
    a.p.ws_ml = reinterpret_cast<float*>(w + lay.ml_off);
    a.p.ws_segs = reinterpret_cast<int4*>(w + kSegsOff);
    a.p.ws_flags = reinterpret_cast<uint32_t*>(w + kFlagsOff);
    a.p.ws_claim = reinterpret_cast<uint32_t*>(w + kClaimOff);
    a.p.ws_seg_count = reinterpret_cast<uint32_t*>(w + kSegCountOff);
    a.p.ws_done = reinterpret_cast<uint32_t*>(w + kDoneOff);
    a.p.dyn_slot_base = kMaxCtas + c.B * c.KVH;
    a.p.max_dyn = gqa::kMaxDynUnits;
    a.p.B = c.B;
    a.p.H = c.H;
    a.p.KVH = c.KVH;
    a.p.capacity = capacity;
    a.p.ring = ring;
    a.p.window = c.window;
    a.p.num_pages = num_pages;
    a.p.max_pages = max_pages;
    a.p.out_f32 = out_dtype == GQA_OUT_F32 ? 1 : 0;
    a.p.T = c.T;
    a.p.test_flags = g_test_mode.load(std::memory_order_relaxed);
    a.grid = grid;
    a.stream = stream;
    if (w_k) {
        // single K=V cache: keys derived in the kernel with the global layers' rotary
        // frequencies theta^(-2i/D), i < 64, theta = 1e6
        a.p.w_k = static_cast<const __nv_bfloat16*>(w_k);
        for (int i = 0; i < 64; ++i)
            a.p.rope_freq[i] = std::pow(kGlobalRopeTheta, -2.0 * i / static_cast<double>(c.D));
        a.p.keqv_operand = reinterpret_cast<__nv_bfloat16*>(w + lay.operand_off);
        const cudaError_t e = keqv_long_history(c.B, capacity, c.KVH, grid)
                                  ? gqa::launch_keqv_tc(a, paged)
                                  : gqa::launch_global_keqv(a, paged);
        return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
    }
    // One new token per sequence is a single-token decode: the mma.sync kernel streams
    // it faster than the tcgen05 multi-query kernel (N = 16 mma for g <= 8 rows).
    if (multi_query && c.T > 1)
        return gqa::launch_mq(a, c.geo == Geometry::kSliding, paged) == cudaSuccess ? GQA_OK
                                                                                   : GQA_ERR_CUDA;
    const cudaError_t e = c.geo == Geometry::kSliding ? gqa::launch_sliding(a, paged)
                                                      : gqa::launch_global(a, paged);
    return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t gqa_workspace_size(int B, int max_seq, int H, int KVH, int D, int window) {
    const Geometry geo = geometry_of(H, KVH, D);
    if (geo == Geometry::kNone || B < 0 || B > GQA_MAX_BATCH || max_seq < 1 ||
        max_seq > GQA_MAX_SEQ || window < 0)
        return 0;
    return layout_for(B, KVH, heads_per_kv(geo), D).total;
}

gqa_status_t gqa_workspace_init(void* workspace, size_t workspace_bytes, gqa_stream_t stream) {
    if (!workspace || workspace_bytes == 0) return GQA_ERR_INVALID_ARGUMENT;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? GQA_OK
               : GQA_ERR_CUDA;
}

gqa_status_t gqa_decode(const void* q, const void* k, const void* v, const int32_t* seq_lens,
                        int B, int S, int H, int KVH, int D, int window, void* out,
                        gqa_out_dtype_t out_dtype, void* workspace, size_t workspace_bytes,
                        gqa_stream_t stream) {
    const CallShape c{geometry_of(H, KVH, D), B, H, KVH, D, window};
    if (S < 1 || S > GQA_MAX_SEQ) return GQA_ERR_INVALID_ARGUMENT;
    gqa_status_t st = check_common(c, q, out, seq_lens, out_dtype);
    if (st != GQA_OK || B == 0) return st;
    if (!k || !v || !aligned(k, 16) || !aligned(v, 16)) return GQA_ERR_INVALID_ARGUMENT;
    return run(c, false, q, k, v, nullptr, seq_lens, static_cast<uint64_t>(S),
               static_cast<uint64_t>(B), S, 0, 0, 0, out, out_dtype, workspace, workspace_bytes,
               reinterpret_cast<cudaStream_t>(stream));
}

gqa_status_t gqa_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* block_table, const int32_t* seq_lens, int B, int P,
                              int max_pages, int page_size, int H, int KVH, int D, int window,
                              void* out, gqa_out_dtype_t out_dtype, void* workspace,
                              size_t workspace_bytes, gqa_stream_t stream) {
    const CallShape c{geometry_of(H, KVH, D), B, H, KVH, D, window};
    if (page_size != GQA_PAGE_SIZE || P < 1 || max_pages < 1 ||
        static_cast<int64_t>(max_pages) * GQA_PAGE_SIZE > GQA_MAX_SEQ)
        return GQA_ERR_INVALID_ARGUMENT;
    gqa_status_t st = check_common(c, q, out, seq_lens, out_dtype);
    if (st != GQA_OK || B == 0) return st;
    if (!k_pages || !v_pages || !block_table || !aligned(k_pages, 16) || !aligned(v_pages, 16) ||
        !aligned(block_table, 4))
        return GQA_ERR_INVALID_ARGUMENT;
    return run(c, true, q, k_pages, v_pages, block_table, seq_lens, GQA_PAGE_SIZE,
               static_cast<uint64_t>(P), max_pages * GQA_PAGE_SIZE, 0, P, max_pages, out,
               out_dtype, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

gqa_status_t gqa_decode_ring(const void* q, const void* k, const void* v, const int32_t* seq_lens,
                             int B, int C, int H, int KVH, int D, int window, void* out,
                             gqa_out_dtype_t out_dtype, void* workspace, size_t workspace_bytes,
                             gqa_stream_t stream) {
    const CallShape c{geometry_of(H, KVH, D), B, H, KVH, D, window};
    if (C < 1 || C > GQA_MAX_SEQ || window < 1 || window > C) return GQA_ERR_INVALID_ARGUMENT;
    gqa_status_t st = check_common(c, q, out, seq_lens, out_dtype);
    if (st != GQA_OK || B == 0) return st;
    if (!k || !v || !aligned(k, 16) || !aligned(v, 16)) return GQA_ERR_INVALID_ARGUMENT;
    // lengths are clamped to the longest context, not to the ring
    return run(c, false, q, k, v, nullptr, seq_lens, static_cast<uint64_t>(C),
               static_cast<uint64_t>(B), GQA_MAX_SEQ, C, 0, 0, out, out_dtype, workspace,
               workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

gqa_status_t gqa_device_status(void* workspace, uint32_t* flags, gqa_stream_t stream) {
    if (!flags) return GQA_ERR_INVALID_ARGUMENT;
    *flags = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!workspace) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
            return GQA_ERR_CUDA;
        std::lock_guard<std::mutex> lock(g_dev[dev].mu);
        workspace = g_dev[dev].ws;
        if (!workspace) return cudaStreamSynchronize(s) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return GQA_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, static_cast<uint8_t*>(workspace) + kFlagsOff, sizeof word,
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return GQA_ERR_CUDA;
    if (word != 0) {
        if (cudaMemsetAsync(workspace, 0, kHeaderBytes, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return GQA_ERR_CUDA;
    }
    *flags = word;
    return GQA_OK;
}

gqa_status_t gqa_decode_keqv(const void* q, const void* v, const void* w_k,
                             const int32_t* seq_lens, int B, int S, int H, int KVH, int D,
                             void* out, gqa_out_dtype_t out_dtype, void* workspace,
                             size_t workspace_bytes, gqa_stream_t stream) {
    const CallShape c{geometry_of(H, KVH, D), B, H, KVH, D, 0};
    if (S < 1 || S > GQA_MAX_SEQ) return GQA_ERR_INVALID_ARGUMENT;
    if (c.geo == Geometry::kSliding) return GQA_ERR_UNSUPPORTED;   // values = keys on global layers only
    gqa_status_t st = check_common(c, q, out, seq_lens, out_dtype);
    if (st != GQA_OK || B == 0) return st;
    if (!v || !w_k || !aligned(v, 16) || !aligned(w_k, 2)) return GQA_ERR_INVALID_ARGUMENT;
    return run(c, false, q, v, v, nullptr, seq_lens, static_cast<uint64_t>(S),
               static_cast<uint64_t>(B), S, 0, 0, 0, out, out_dtype, workspace, workspace_bytes,
               reinterpret_cast<cudaStream_t>(stream), w_k);
}

gqa_status_t gqa_decode_keqv_paged(const void* q, const void* v_pages, const void* w_k,
                                   const int32_t* block_table, const int32_t* seq_lens, int B,
                                   int P, int max_pages, int page_size, int H, int KVH, int D,
                                   void* out, gqa_out_dtype_t out_dtype, void* workspace,
                                   size_t workspace_bytes, gqa_stream_t stream) {
    const CallShape c{geometry_of(H, KVH, D), B, H, KVH, D, 0};
    if (page_size != GQA_PAGE_SIZE || P < 1 || max_pages < 1 ||
        static_cast<int64_t>(max_pages) * GQA_PAGE_SIZE > GQA_MAX_SEQ)
        return GQA_ERR_INVALID_ARGUMENT;
    if (c.geo == Geometry::kSliding) return GQA_ERR_UNSUPPORTED;
    gqa_status_t st = check_common(c, q, out, seq_lens, out_dtype);
    if (st != GQA_OK || B == 0) return st;
    if (!v_pages || !w_k || !block_table || !aligned(v_pages, 16) || !aligned(w_k, 2) ||
        !aligned(block_table, 4))
        return GQA_ERR_INVALID_ARGUMENT;
    return run(c, true, q, v_pages, v_pages, block_table, seq_lens, GQA_PAGE_SIZE,
               static_cast<uint64_t>(P), max_pages * GQA_PAGE_SIZE, 0, P, max_pages, out,
               out_dtype, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), w_k);
}

size_t gqa_workspace_size_mq(int B, int T, int H, int KVH, int D) {
    const Geometry geo = geometry_of(H, KVH, D);
    if (geo == Geometry::kNone || B < 0 || B > GQA_MAX_BATCH || !queries_ok(geo, T)) return 0;
    return layout_for(B, KVH, heads_per_kv(geo) * T, D).total;
}

gqa_status_t gqa_decode_mq(const void* q, const void* k, const void* v, const int32_t* seq_lens,
                           int B, int T, int S, int H, int KVH, int D, int window, void* out,
                           gqa_out_dtype_t out_dtype, void* workspace, size_t workspace_bytes,
                           gqa_stream_t stream) {
    CallShape c{geometry_of(H, KVH, D), B, H, KVH, D, window};
    c.T = T;
    if (S < 1 || S > GQA_MAX_SEQ) return GQA_ERR_INVALID_ARGUMENT;
    if (c.geo != Geometry::kNone && !queries_ok(c.geo, T)) return GQA_ERR_INVALID_ARGUMENT;
    gqa_status_t st = check_common(c, q, out, seq_lens, out_dtype);
    if (st != GQA_OK || B == 0) return st;
    if (!k || !v || !aligned(k, 16) || !aligned(v, 16)) return GQA_ERR_INVALID_ARGUMENT;
    return run(c, false, q, k, v, nullptr, seq_lens, static_cast<uint64_t>(S),
               static_cast<uint64_t>(B), S, 0, 0, 0, out, out_dtype, workspace, workspace_bytes,
               reinterpret_cast<cudaStream_t>(stream), nullptr, true);
}

gqa_status_t gqa_decode_mq_paged(const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* block_table, const int32_t* seq_lens, int B,
                                 int T, int P, int max_pages, int page_size, int H, int KVH,
                                 int D, int window, void* out, gqa_out_dtype_t out_dtype,
                                 void* workspace, size_t workspace_bytes, gqa_stream_t stream) {
    CallShape c{geometry_of(H, KVH, D), B, H, KVH, D, window};
    c.T = T;
    if (page_size != GQA_PAGE_SIZE || P < 1 || max_pages < 1 ||
        static_cast<int64_t>(max_pages) * GQA_PAGE_SIZE > GQA_MAX_SEQ)
        return GQA_ERR_INVALID_ARGUMENT;
    if (c.geo != Geometry::kNone && !queries_ok(c.geo, T)) return GQA_ERR_INVALID_ARGUMENT;
    gqa_status_t st = check_common(c, q, out, seq_lens, out_dtype);
    if (st != GQA_OK || B == 0) return st;
    if (!k_pages || !v_pages || !block_table || !aligned(k_pages, 16) || !aligned(v_pages, 16) ||
        !aligned(block_table, 4))
        return GQA_ERR_INVALID_ARGUMENT;
    return run(c, true, q, k_pages, v_pages, block_table, seq_lens, GQA_PAGE_SIZE,
               static_cast<uint64_t>(P), max_pages * GQA_PAGE_SIZE, 0, P, max_pages, out,
               out_dtype, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
               nullptr, true);
}

gqa_status_t gqa_check_inputs_host(const int32_t* seq_lens, int B, int capacity, int window,
                                   const int32_t* block_table, int max_pages, int P,
                                   int* first_bad) {
    if (first_bad) *first_bad = -1;
    if (B < 0 || B > GQA_MAX_BATCH || capacity < 1 || window < 0 || (B > 0 && !seq_lens))
        return GQA_ERR_INVALID_ARGUMENT;
    if (block_table && (max_pages < 1 || P < 1)) return GQA_ERR_INVALID_ARGUMENT;
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b];
        bool bad = L < 0 || L > capacity;
        if (!bad && block_table && L > 0) {
            const int lo = (window > 0 && L > window) ? L - window : 0;
            const int32_t* row = block_table + static_cast<size_t>(b) * max_pages;
            for (int pg = lo / GQA_PAGE_SIZE; pg <= (L - 1) / GQA_PAGE_SIZE && !bad; ++pg)
                bad = pg >= max_pages || row[pg] < 0 || row[pg] >= P;
        }
        if (bad) {
            if (first_bad) *first_bad = b;
            return GQA_ERR_INVALID_ARGUMENT;
        }
    }
    return GQA_OK;
}

gqa_kernel_t gqa_decode_keqv_kernel(int B, int capacity, int H, int KVH, int D) {
    if (geometry_of(H, KVH, D) != Geometry::kGlobal || B < 1 || B > GQA_MAX_BATCH ||
        capacity < 1 || capacity > GQA_MAX_SEQ)
        return GQA_KERNEL_NONE;
    const int grid = device_grid();
    if (grid == 0) return GQA_KERNEL_NONE;
    return keqv_long_history(B, capacity, KVH, grid) ? GQA_KERNEL_TCGEN05 : GQA_KERNEL_SPLIT_DECODE;
}

uint32_t gqa_set_test_mode(uint32_t flags) {
    return g_test_mode.exchange(flags & (GQA_TEST_SINGLE_PIECE | GQA_TEST_STALL));
}

uint32_t gqa_get_test_mode(void) { return g_test_mode.load(); }

const char* gqa_status_string(gqa_status_t status) {
    switch (status) {
        case GQA_OK: return "GQA_OK";
        case GQA_ERR_INVALID_ARGUMENT: return "GQA_ERR_INVALID_ARGUMENT";
        case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED";
        case GQA_ERR_WORKSPACE: return "GQA_ERR_WORKSPACE";
        case GQA_ERR_CUDA: return "GQA_ERR_CUDA";
    }
    return "GQA_ERR_UNKNOWN";
}

}  // extern "C"
