// Shared launch helper for the per-geometry kernel translation units.
#pragma once

#include <mutex>

#include "kernels/combine_kernel.cuh"
#include "launch.h"

namespace gqa {

// Tensor map of a K or V cache for the TMA boxes of policy Pol (one KV head's
// rows; see gqa_decode_kernel).
//   128-byte swizzled (read with ldmatrix): 4-D view
//     (64 elements, row, 64-element chunk of the KVH*D row (stride 128 B), outer),
//     box (64, 16, D/64, 1) -> shared [D/64][16 rows][128 B] with 16-byte units
//     permuted by row, so 8 consecutive rows of one chunk hit distinct banks.
//   plain: 4-D view (D elements, kv head, row, outer), box (D, 1, rows, 1)
//     -> shared [rows][D].
template <class Pol>
bool encode_kv_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t outer, int KVH,
                   bool paged) {
    constexpr int D = Pol::D;
    const uint64_t row_bytes = static_cast<uint64_t>(KVH) * D * 2;
    const cuuint32_t box_rows = paged ? kPageRows : Pol::kBoxRows;
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4];
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (Pol::kSwizzle128) {
        dims[0] = 64; dims[1] = rows; dims[2] = static_cast<cuuint64_t>(KVH) * (D / 64); dims[3] = outer;
        strides[0] = row_bytes; strides[1] = 128; strides[2] = row_bytes * rows;
        box[0] = 64; box[1] = box_rows; box[2] = D / 64; box[3] = 1;
    } else {
        static_assert(Pol::kSwizzle128 || D <= 256, "a plain box row is at most 256 elements");
        dims[0] = D; dims[1] = static_cast<cuuint64_t>(KVH); dims[2] = rows; dims[3] = outer;
        strides[0] = static_cast<cuuint64_t>(D) * 2; strides[1] = row_bytes; strides[2] = row_bytes * rows;
        box[0] = D; box[1] = 1; box[2] = box_rows; box[3] = 1;
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return false;
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  Pol::kSwizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches the main kernel and, unless the policy merges split segments in the
// main kernel, the combine kernel right behind it.  Both opt in to programmatic
// dependent launch: each may start while the kernel before it in the stream
// drains, and waits (griddepcontrol.wait) before touching global memory that
// kernel writes.
template <class Pol, bool kPaged>
cudaError_t launch_decode(const LaunchArgs& a) {
    constexpr size_t kSmem = sizeof(KernelSmem<Pol>) + 1024;   // + alignment slack
    constexpr int kMaxDevices = 64;
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_err[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(gqa_decode_kernel<Pol, kPaged>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmem));
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];

    CUtensorMap tm_k, tm_v;
    if (!encode_kv_map<Pol>(&tm_k, a.k, a.rows, a.outer, a.p.KVH, kPaged) ||
        !encode_kv_map<Pol>(&tm_v, a.v, a.rows, a.outer, a.p.KVH, kPaged))
        return cudaErrorInvalidValue;

    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.grid));
    cfg.blockDim = dim3(block_threads<Pol>());
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = a.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gqa_decode_kernel<Pol, kPaged>, tm_k, tm_v, a.p);
    if (e != cudaSuccess || Pol::kMergeInKernel) return e;

    const int segments = a.p.B * a.p.KVH;
    constexpr int kChunksPerSeg = (Pol::G * Pol::D / 4 + kCombineThreads - 1) / kCombineThreads;
    const int items = segments * kChunksPerSeg;
    const int cgrid = items < kCombineBlocksPerSm * a.grid ? items : kCombineBlocksPerSm * a.grid;
    cudaLaunchConfig_t ccfg = {};
    ccfg.gridDim = dim3(static_cast<unsigned>(cgrid));
    ccfg.blockDim = dim3(kCombineThreads);
    ccfg.dynamicSmemBytes = 0;
    ccfg.stream = a.stream;
    ccfg.attrs = pdl;
    ccfg.numAttrs = 1;
    return cudaLaunchKernelEx(&ccfg, gqa_combine_kernel<Pol::G, Pol::D>, a.p, segments);
}

}  // namespace gqa
