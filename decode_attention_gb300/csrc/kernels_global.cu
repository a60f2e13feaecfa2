// decodeGQA kernels (H=32, KVH=4, D=512), contiguous and paged caches.
#include "kernels/policy_mma.cuh"
#include "launch_common.cuh"

namespace gqa {

cudaError_t launch_global(const LaunchArgs& a, bool paged) {
    return paged ? launch_decode<GlobalMma, true>(a) : launch_decode<GlobalMma, false>(a);
}

size_t smem_bytes_global() { return sizeof(KernelSmem<GlobalMma>) + 1024; }

}  // namespace gqa
