// Multi-query decode kernels (tcgen05): both geometries, contiguous and paged caches.
#include "kernels/decode_mq_kernel.cuh"
#include "launch_common.cuh"

namespace gqa {

namespace {

// K or V cache for the multi-query kernel: 4-D view (64 elements, row, 64-element
// chunk of the KVH*D row (stride 128 B), outer), 128-byte swizzle; box (64, box_rows,
// 1, 1): on a contiguous cache 128 rows (one 16 KB stage of one chunk) or 16 rows (the
// attended rows of a sequence's last tile, box by box), on a paged pool 16 rows (one
// page of one chunk, 2 KB).
bool encode_mq_kv_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t outer, int KVH,
                      int D, int box_rows) {
    const uint64_t row_bytes = static_cast<uint64_t>(KVH) * D * 2;
    cuuint64_t dims[4] = {64, rows, static_cast<cuuint64_t>(KVH) * (D / 64), outer};
    cuuint64_t strides[3] = {row_bytes, 128, row_bytes * rows};
    cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return false;
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [B, T, H, D]: 4-D view (D, H, T, B), box (64, G, T, 1), 128-byte swizzle: one load
// brings the 64-element column block c of the T * G query rows of a KV head, row
// t * G + g at byte 128 (t * G + g) of a 1024-byte-aligned destination.
bool encode_mq_q_map(CUtensorMap* map, const void* q, int B, int T, int H, int D, int G) {
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                             static_cast<cuuint64_t>(T) * H * D * 2};
    cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(T), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return false;
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The K=V scores' B operand [B, KVH, 16, 512]: for KV head kvh of sequence b, row r < 8
// holds query head kvh * 8 + r, row 8 + r the same head's lo part.  On the unrotated
// dims (d mod 256 >= 64) the rows carry q * w_k split into bf16 hi (row r) and lo
// (row 8 + r), the product being exact in fp32; on the rotated dims the hi row carries
// q itself (the weight is in the derived keys) and the lo row zero.
__global__ void __launch_bounds__(256) gqa_keqv_operand_kernel(const DecodeParams p) {
    ptx::grid_dependency_wait();   // q may come from the kernel before this one
    ptx::allow_dependent_launch();
    const int u = blockIdx.x;      // segment b * KVH + kvh
    const int b = u / p.KVH, kvh = u - b * p.KVH;
    constexpr int G = 8, D = 512;
    for (int e = threadIdx.x; e < 2 * G * D; e += blockDim.x) {
        const int r = e / D, d = e - (e / D) * D;
        const int h = kvh * G + (r & (G - 1));
        const float qv = __bfloat162float(p.q[(static_cast<size_t>(b) * p.H + h) * D + d]);
        __nv_bfloat16 o;
        if ((d & (D / 2 - 1)) < 64) {
            o = r < G ? __float2bfloat16_rn(qv) : __float2bfloat16_rn(0.0f);
        } else {
            const float x = qv * __bfloat162float(p.w_k[d]);
            const __nv_bfloat16 hi = __float2bfloat16_rn(x);
            o = r < G ? hi : __float2bfloat16_rn(x - __bfloat162float(hi));
        }
        p.keqv_operand[static_cast<size_t>(u) * 2 * G * D + e] = o;
    }
}

// The K=V operand [B, KVH, 16, 512]: 4-D view (512, 16, KVH, B), box (64, 16, 1, 1).
bool encode_keqv_operand_map(CUtensorMap* map, const void* base, int B, int KVH) {
    cuuint64_t dims[4] = {512, 16, static_cast<cuuint64_t>(KVH), static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {1024, 16 * 1024, static_cast<cuuint64_t>(KVH) * 16 * 1024};
    cuuint32_t box[4] = {64, 16, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return false;
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class Cfg, bool kPaged>
cudaError_t launch_mq_impl(const LaunchArgs& a) {
    constexpr size_t kSmem = sizeof(MqSmem<Cfg>) + 1024;   // + alignment slack
    static_assert(kSmem <= 232448, "227 KB of shared memory per CTA");
    constexpr int kMaxDevices = 64;
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_err[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(gqa_mq_kernel<Cfg, kPaged>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmem));
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];

    const int T = a.p.T > 1 ? a.p.T : 1;
    CUtensorMap tm_k, tm_v, tm_q, tm_k16, tm_v16;
    const int rows_per_box = kPaged ? kPageRows : kMqTile;
    if (!encode_mq_kv_map(&tm_k, a.k, a.rows, a.outer, a.p.KVH, Cfg::D, rows_per_box) ||
        !encode_mq_kv_map(&tm_v, a.v, a.rows, a.outer, a.p.KVH, Cfg::D, rows_per_box) ||
        !encode_mq_kv_map(&tm_k16, a.k, a.rows, a.outer, a.p.KVH, Cfg::D, kPageRows) ||
        !encode_mq_kv_map(&tm_v16, a.v, a.rows, a.outer, a.p.KVH, Cfg::D, kPageRows))
        return cudaErrorInvalidValue;
    if (Cfg::KEQV ? !encode_keqv_operand_map(&tm_q, a.p.keqv_operand, a.p.B, a.p.KVH)
                  : !encode_mq_q_map(&tm_q, a.p.q, a.p.B, T, a.p.H, Cfg::D, Cfg::G))
        return cudaErrorInvalidValue;

    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;

    if (Cfg::KEQV) {
        cudaLaunchConfig_t ocfg = {};
        ocfg.gridDim = dim3(static_cast<unsigned>(a.p.B * a.p.KVH));
        ocfg.blockDim = dim3(256);
        ocfg.stream = a.stream;
        ocfg.attrs = pdl;
        ocfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&ocfg, gqa_keqv_operand_kernel, a.p);
        if (e != cudaSuccess) return e;
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.grid));
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = a.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gqa_mq_kernel<Cfg, kPaged>, tm_k, tm_v, tm_q, tm_k16, tm_v16, a.p);
    if (e != cudaSuccess) return e;

    const int segments = a.p.B * a.p.KVH;
    const int chunks_per_seg = (T * Cfg::G * Cfg::D / 4 + kCombineThreads - 1) / kCombineThreads;
    const int items = segments * chunks_per_seg;
    const int cgrid = items < kCombineBlocksPerSm * a.grid ? items : kCombineBlocksPerSm * a.grid;
    cudaLaunchConfig_t ccfg = {};
    ccfg.gridDim = dim3(static_cast<unsigned>(cgrid));
    ccfg.blockDim = dim3(kCombineThreads);
    ccfg.dynamicSmemBytes = 0;
    ccfg.stream = a.stream;
    ccfg.attrs = pdl;
    ccfg.numAttrs = 1;
    return cudaLaunchKernelEx(&ccfg, gqa_combine_kernel<Cfg::G, Cfg::D>, a.p, segments);
}

}  // namespace

cudaError_t launch_mq(const LaunchArgs& a, bool sliding, bool paged) {
    if (sliding)
        return paged ? launch_mq_impl<MqSliding, true>(a) : launch_mq_impl<MqSliding, false>(a);
    if (a.p.T <= MqGlobal2::MAXT)
        return paged ? launch_mq_impl<MqGlobal2, true>(a) : launch_mq_impl<MqGlobal2, false>(a);
    return paged ? launch_mq_impl<MqGlobal, true>(a) : launch_mq_impl<MqGlobal, false>(a);
}

cudaError_t launch_keqv_tc(const LaunchArgs& a, bool paged) {
    return paged ? launch_mq_impl<MqKeqV, true>(a) : launch_mq_impl<MqKeqV, false>(a);
}

int mq_max_queries(bool sliding) { return sliding ? MqSliding::MAXT : MqGlobal::MAXT; }

size_t smem_bytes_mq(bool sliding) {
    return (sliding ? sizeof(MqSmem<MqSliding>) : sizeof(MqSmem<MqGlobal>)) + 1024;
}

}  // namespace gqa
