// Internal interface between the C-ABI host code and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "kernels/decode_kernel.cuh"

namespace gqa {

// Grid size bound used to size workspaces independently of the device.
constexpr int kMaxCtas = 1024;
static_assert(kMaxCtas >= 1, "grid bound");

struct LaunchArgs {
    const void* k;          // K cache / page pool
    const void* v;          // V cache / page pool
    uint64_t rows;          // positions per sequence (contiguous) or slots per page (paged)
    uint64_t outer;         // sequences (contiguous) or pages (paged)
    DecodeParams p;
    int grid;
    cudaStream_t stream;
};

// cuTensorMapEncodeTiled from the driver (resolved once); null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Kernel launchers, one translation unit per geometry.  Each sets its kernels'
// shared-memory limit on first use on a device and launches one persistent grid.
cudaError_t launch_sliding(const LaunchArgs& a, bool paged);
cudaError_t launch_global(const LaunchArgs& a, bool paged);
// decodeGQA over a single K=V cache: a.k and a.v are both the value cache.
cudaError_t launch_global_keqv(const LaunchArgs& a, bool paged);

// Multi-query decode (tcgen05): a.p.T query tokens per sequence, q [B, T, H, D],
// out [B, T, H, D]; at most mq_max_queries(sliding) tokens.
cudaError_t launch_mq(const LaunchArgs& a, bool sliding, bool paged);
int mq_max_queries(bool sliding);
// decodeGQA over a single K=V cache on the tcgen05 kernel (a.k == a.v: the value
// cache; a.p.keqv_operand: workspace room for the scores' operand).
cudaError_t launch_keqv_tc(const LaunchArgs& a, bool paged);
size_t smem_bytes_mq(bool sliding);

// Bytes of dynamic shared memory each geometry's kernel requests.
size_t smem_bytes_sliding();
size_t smem_bytes_global();
size_t smem_bytes_global_keqv();

}  // namespace gqa
