// gqa_decode_noalloc: the contiguous-cache decode attention call for callers
// that cannot allocate device memory (see include/gqa_decode.h).
//
// Its scratch -- status word, claim counter, per-segment partial lists and the
// split-softmax partials -- lives in one file-scope device array of fixed size
// instead of a workspace the caller passes or the library allocates.  The
// array's device address is looked up once per device with
// cudaGetSymbolAddress (host code must never hand the symbol itself to a
// kernel: on the host it is only a stand-in).  The kernels are the same ones
// gqa_decode launches.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "gqa_decode.h"
#include "launch.h"

namespace {

// The fixed scratch.  Every GPU that loads this library holds it until exit.
__device__ __align__(256) uint8_t g_noalloc_scratch[GQA_NOALLOC_SCRATCH_BYTES];

// Layout of the fixed scratch for one call (offsets in bytes):
//   [0, 4)         status word        (kept across calls; gqa_noalloc_status reads
//                                      and clears it)
//   [64, 68)       claim counter      } cleared before every call
//   [128, 132)     producers finished }
//   [256, 16640)   partials stored per segment, 4096 x uint32: at a fixed place, so
//                  that calls of any shape find them zero (every completed call
//                  leaves them so; gqa_noalloc_status zeroes them after a call that
//                  raised a status bit)
//   [16640, ...)   B*KVH partial lists (int4)
//   [ml, ...)      slots x G x 2 floats;  [acc, ...) slots x G x D floats
// with slots = grid + B*KVH + dyn: static unit j of the kernel keeps its piece
// of segment u at slot j + u (j < grid), dynamic chunk k at slot grid + B*KVH + k
// (k < dyn).  dyn is min(kDynChunksPerCta grid, kMaxDynUnits) when that fits the
// array, else what does fit (down to 0: the kernel then splits the work into
// static units only); the kernel is told the bound and never exceeds it.
constexpr size_t kClaimOff = 64;
constexpr size_t kDoneOff = 128;
constexpr size_t kCountersBytes = 128;   // the claim and producer counters' lines
constexpr size_t kSegCountOff = 256;
constexpr size_t kSegsOff = kSegCountOff + static_cast<size_t>(GQA_MAX_BATCH) * 16 * 4;

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct FixedLayout {
    size_t ml_off, acc_off, total;
    int dyn_slot_base, max_dyn;
};

FixedLayout layout_with(int grid, int B, int KVH, int G, int D, int dyn) {
    const size_t slots = static_cast<size_t>(grid) + static_cast<size_t>(B) * KVH + dyn;
    FixedLayout f;
    f.ml_off = round256(kSegsOff + static_cast<size_t>(B) * KVH * 16);
    f.acc_off = round256(f.ml_off + slots * G * 2 * sizeof(float));
    f.total = round256(f.acc_off + slots * G * D * sizeof(float));
    f.dyn_slot_base = grid + B * KVH;
    f.max_dyn = dyn;
    return f;
}

// The layout with as many dynamic slots (up to the kernel's own bound) as the
// array holds; total > GQA_NOALLOC_SCRATCH_BYTES when not even dyn = 0 fits.
FixedLayout fixed_layout(int grid, int B, int KVH, int G, int D) {
    const int want = gqa::kDynChunksPerCta * grid < gqa::kMaxDynUnits
                         ? gqa::kDynChunksPerCta * grid
                         : gqa::kMaxDynUnits;
    const FixedLayout none = layout_with(grid, B, KVH, G, D, 0);
    if (none.total > GQA_NOALLOC_SCRATCH_BYTES) return none;
    // each slot takes G (D + 2) floats; 512 bytes cover the two 256-byte roundings
    const size_t per_slot = static_cast<size_t>(G) * (D + 2) * sizeof(float);
    const size_t spare = GQA_NOALLOC_SCRATCH_BYTES - none.total;
    const size_t fit = spare >= 512 ? (spare - 512) / per_slot : 0;
    const int dyn = fit < static_cast<size_t>(want) ? static_cast<int>(fit) : want;
    return layout_with(grid, B, KVH, G, D, dyn);
}

constexpr int kMaxDevices = 64;

struct DeviceScratch {
    std::mutex mu;
    bool ready = false;
    uint8_t* ptr = nullptr;   // device address of g_noalloc_scratch on this device
    int sm_count = 0;
};

DeviceScratch g_scratch[kMaxDevices];

// Once per device, with that device current: the array's device address and
// the SM count.
gqa_status_t device_scratch(uint8_t** ptr, int* grid) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
    DeviceScratch& ds = g_scratch[dev];
    std::lock_guard<std::mutex> lock(ds.mu);
    if (!ds.ready) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return GQA_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return GQA_ERR_CUDA;
        ds.ptr = static_cast<uint8_t*>(p);
        ds.sm_count = n < gqa::kMaxCtas ? n : gqa::kMaxCtas;
        ds.ready = true;
    }
    *ptr = ds.ptr;
    *grid = ds.sm_count;
    return GQA_OK;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" gqa_status_t gqa_decode_noalloc(const void* q, const void* k, const void* v,
                                           const int32_t* seq_lens, int B, int S, int H, int KVH,
                                           int D, int window, void* out, gqa_out_dtype_t out_dtype,
                                           gqa_stream_t stream) {
    // argument checks: the same rules as gqa_decode
    const bool sliding = (H == 32 && KVH == 16 && D == 256);
    const bool global = (H == 32 && KVH == 4 && D == 512);
    if (S < 1 || S > GQA_MAX_SEQ || B < 0 || B > GQA_MAX_BATCH || window < 0)
        return GQA_ERR_INVALID_ARGUMENT;
    if (out_dtype != GQA_OUT_BF16 && out_dtype != GQA_OUT_F32) return GQA_ERR_INVALID_ARGUMENT;
    if (!sliding && !global) return GQA_ERR_UNSUPPORTED;
    if (B == 0) return GQA_OK;
    if (!q || !k || !v || !seq_lens || !out) return GQA_ERR_INVALID_ARGUMENT;
    if (!aligned_to(q, 16) || !aligned_to(k, 16) || !aligned_to(v, 16) || !aligned_to(out, 16) ||
        !aligned_to(seq_lens, 4))
        return GQA_ERR_INVALID_ARGUMENT;
    if (!gqa::tensor_map_encoder()) return GQA_ERR_CUDA;

    uint8_t* ws = nullptr;
    int grid = 0;
    gqa_status_t st = device_scratch(&ws, &grid);
    if (st != GQA_OK) return st;
    const int G = H / KVH;
    const FixedLayout lay = fixed_layout(grid, B, KVH, G, D);
    if (lay.total > GQA_NOALLOC_SCRATCH_BYTES) return GQA_ERR_WORKSPACE;   // call too large

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the claim and producer counters must start at zero (the status word keeps earlier
    // calls' bits)
    if (cudaMemsetAsync(ws + kClaimOff, 0, kCountersBytes, s) != cudaSuccess) return GQA_ERR_CUDA;

    gqa::LaunchArgs a;
    std::memset(&a, 0, sizeof a);
    a.k = k;
    a.v = v;
    a.rows = static_cast<uint64_t>(S);
    a.outer = static_cast<uint64_t>(B);
    a.p.q = static_cast<const __nv_bfloat16*>(q);
    a.p.seq_lens = seq_lens;
    a.p.block_table = nullptr;
    a.p.out = out;
    a.p.ws_acc = reinterpret_cast<float*>(ws + lay.acc_off);
    a.p.ws_ml = reinterpret_cast<float*>(ws + lay.ml_off);
    a.p.ws_segs = reinterpret_cast<int4*>(ws + kSegsOff);
    a.p.ws_flags = reinterpret_cast<uint32_t*>(ws);
    a.p.ws_claim = reinterpret_cast<uint32_t*>(ws + kClaimOff);
    a.p.ws_seg_count = reinterpret_cast<uint32_t*>(ws + kSegCountOff);
    a.p.ws_done = reinterpret_cast<uint32_t*>(ws + kDoneOff);
    a.p.dyn_slot_base = lay.dyn_slot_base;
    a.p.max_dyn = lay.max_dyn;
    a.p.B = B;
    a.p.H = H;
    a.p.KVH = KVH;
    a.p.capacity = S;
    a.p.ring = 0;
    a.p.window = window;
    a.p.num_pages = 0;
    a.p.max_pages = 0;
    a.p.out_f32 = out_dtype == GQA_OUT_F32 ? 1 : 0;
    a.p.T = 1;
    a.p.test_flags = gqa_get_test_mode();
    a.grid = grid;
    a.stream = s;
    const cudaError_t e = sliding ? gqa::launch_sliding(a, false) : gqa::launch_global(a, false);
    return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

extern "C" gqa_status_t gqa_noalloc_status(uint32_t* flags, gqa_stream_t stream) {
    if (!flags) return GQA_ERR_INVALID_ARGUMENT;
    *flags = 0;
    uint8_t* ws = nullptr;
    int grid = 0;
    gqa_status_t st = device_scratch(&ws, &grid);
    if (st != GQA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GQA_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return GQA_ERR_CUDA;
    // after a raised bit (perhaps a call that timed out half-way) the word and every
    // counter start again from zero
    if (word != 0 &&
        (cudaMemsetAsync(ws, 0, kSegsOff, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess))
        return GQA_ERR_CUDA;
    *flags = word;
    return GQA_OK;
}
