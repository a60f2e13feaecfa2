// gqa_prepare_decode / gqa_prepare_decode_paged: the decode-step producer ahead of
// the attention core (include/gqa_decode.h).
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "gqa_decode.h"
#include "kernels/prepare_kernel.cuh"

namespace {

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Rotary pairs and base of each geometry (Model Spec, `attn.rope` rows).
bool rope_of(int H, int KVH, int D, int* n_rot, double* theta) {
    if (H == 32 && KVH == 16 && D == 256) {   // slidingDecodeGQA layers
        *n_rot = 128;
        *theta = 1.0e4;
        return true;
    }
    if (H == 32 && KVH == 4 && D == 512) {    // decodeGQA layers
        *n_rot = 64;
        *theta = 1.0e6;
        return true;
    }
    return false;
}

template <int D, bool kPaged>
cudaError_t launch(const gqa::PrepareParams& p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    const int vecs = p.H + 2 * p.KVH;   // head vectors per sequence, one per warp
    cfg.gridDim = dim3(static_cast<unsigned>(p.B),
                       static_cast<unsigned>((vecs + gqa::kPrepareThreads / 32 - 1) /
                                             (gqa::kPrepareThreads / 32)));
    cfg.blockDim = dim3(gqa::kPrepareThreads);
    cfg.stream = stream;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gqa::gqa_prepare_kernel<D, kPaged>, p);
}

gqa_status_t run(gqa::PrepareParams& p, int D, bool paged, cudaStream_t stream) {
    double theta = 0.0;
    if (!rope_of(p.H, p.KVH, D, &p.n_rot, &theta)) return GQA_ERR_UNSUPPORTED;
    for (int i = 0; i < p.n_rot; ++i) p.freq[i] = std::pow(theta, -2.0 * i / static_cast<double>(D));
    cudaError_t e;
    if (D == 256)
        e = paged ? launch<256, true>(p, stream) : launch<256, false>(p, stream);
    else
        e = paged ? launch<512, true>(p, stream) : launch<512, false>(p, stream);
    return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

// Shared argument checks; returns GQA_OK to proceed (B > 0).
gqa_status_t check(const void* q_raw, const void* k_raw, const void* v_raw, const void* w_q,
                   const void* w_k, const int32_t* seq_lens, int B, int H, int KVH, int D,
                   const void* q_out, const void* k_cache, const void* v_cache) {
    int n_rot = 0;
    double theta = 0.0;
    if (B < 0 || B > GQA_MAX_BATCH) return GQA_ERR_INVALID_ARGUMENT;
    if (!rope_of(H, KVH, D, &n_rot, &theta)) return GQA_ERR_UNSUPPORTED;
    if (B == 0) return GQA_OK;
    const bool keqv = v_raw == nullptr;
    if (keqv && D != 512) return GQA_ERR_UNSUPPORTED;   // values = keys on global layers only
    if (!q_raw || !k_raw || !w_q || !w_k || !seq_lens || !q_out || !v_cache ||
        (!keqv && !k_cache))
        return GQA_ERR_INVALID_ARGUMENT;
    const void* vec[] = {q_raw, k_raw, v_raw, q_out, k_cache, v_cache};
    for (const void* x : vec)
        if (x && !aligned_to(x, 16)) return GQA_ERR_INVALID_ARGUMENT;
    if (!aligned_to(w_q, 4) || !aligned_to(w_k, 4) || !aligned_to(seq_lens, 4))
        return GQA_ERR_INVALID_ARGUMENT;
    return GQA_OK;
}

}  // namespace

extern "C" gqa_status_t gqa_prepare_decode(const void* q_raw, const void* k_raw, const void* v_raw,
                                           const void* w_q, const void* w_k,
                                           const int32_t* seq_lens, int B, int H, int KVH, int D,
                                           void* q_out, void* k_cache, void* v_cache, int rows,
                                           int ring, gqa_stream_t stream) {
    gqa_status_t st = check(q_raw, k_raw, v_raw, w_q, w_k, seq_lens, B, H, KVH, D, q_out,
                            k_cache, v_cache);
    if (st != GQA_OK || B == 0) return st;
    if (rows < 1 || rows > GQA_MAX_SEQ || (ring != 0 && ring != 1)) return GQA_ERR_INVALID_ARGUMENT;
    gqa::PrepareParams p;
    std::memset(&p, 0, sizeof p);
    p.q_raw = static_cast<const __nv_bfloat16*>(q_raw);
    p.k_raw = static_cast<const __nv_bfloat16*>(k_raw);
    p.v_raw = static_cast<const __nv_bfloat16*>(v_raw);
    p.w_q = static_cast<const __nv_bfloat16*>(w_q);
    p.w_k = static_cast<const __nv_bfloat16*>(w_k);
    p.seq_lens = seq_lens;
    p.q_out = static_cast<__nv_bfloat16*>(q_out);
    p.k_cache = static_cast<__nv_bfloat16*>(k_cache);
    p.v_cache = static_cast<__nv_bfloat16*>(v_cache);
    p.B = B;
    p.H = H;
    p.KVH = KVH;
    p.rows = rows;
    p.ring = ring;
    return run(p, D, false, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" gqa_status_t gqa_prepare_decode_paged(const void* q_raw, const void* k_raw,
                                                 const void* v_raw, const void* w_q,
                                                 const void* w_k, const int32_t* block_table,
                                                 const int32_t* seq_lens, int B, int P,
                                                 int max_pages, int page_size, int H, int KVH,
                                                 int D, void* q_out, void* k_pages, void* v_pages,
                                                 gqa_stream_t stream) {
    gqa_status_t st = check(q_raw, k_raw, v_raw, w_q, w_k, seq_lens, B, H, KVH, D, q_out,
                            k_pages, v_pages);
    if (st != GQA_OK || B == 0) return st;
    if (page_size != GQA_PAGE_SIZE || P < 1 || max_pages < 1 || !block_table ||
        !aligned_to(block_table, 4) ||
        static_cast<int64_t>(max_pages) * GQA_PAGE_SIZE > GQA_MAX_SEQ)
        return GQA_ERR_INVALID_ARGUMENT;
    gqa::PrepareParams p;
    std::memset(&p, 0, sizeof p);
    p.q_raw = static_cast<const __nv_bfloat16*>(q_raw);
    p.k_raw = static_cast<const __nv_bfloat16*>(k_raw);
    p.v_raw = static_cast<const __nv_bfloat16*>(v_raw);
    p.w_q = static_cast<const __nv_bfloat16*>(w_q);
    p.w_k = static_cast<const __nv_bfloat16*>(w_k);
    p.seq_lens = seq_lens;
    p.q_out = static_cast<__nv_bfloat16*>(q_out);
    p.k_cache = static_cast<__nv_bfloat16*>(k_pages);
    p.v_cache = static_cast<__nv_bfloat16*>(v_pages);
    p.block_table = block_table;
    p.B = B;
    p.H = H;
    p.KVH = KVH;
    p.max_pages = max_pages;
    p.num_pages = P;
    return run(p, D, true, reinterpret_cast<cudaStream_t>(stream));
}
