// decodeGQA kernels over a single K=V cache (H=32, KVH=4, D=512), contiguous and
// paged caches.
#include "kernels/policy_mma_keqv.cuh"
#include "launch_common.cuh"

namespace gqa {

cudaError_t launch_global_keqv(const LaunchArgs& a, bool paged) {
    return paged ? launch_decode<MmaKeqV, true>(a) : launch_decode<MmaKeqV, false>(a);
}

size_t smem_bytes_global_keqv() { return sizeof(KernelSmem<MmaKeqV>) + 1024; }

}  // namespace gqa
