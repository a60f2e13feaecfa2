// slidingDecodeGQA kernels (H=32, KVH=16, D=256), contiguous and paged caches.
#include "kernels/policy_sliding_core.cuh"
#include "launch_common.cuh"

namespace gqa {

cudaError_t launch_sliding(const LaunchArgs& a, bool paged) {
    return paged ? launch_decode<SlidingCore, true>(a) : launch_decode<SlidingCore, false>(a);
}

size_t smem_bytes_sliding() { return sizeof(KernelSmem<SlidingCore>) + 1024; }

}  // namespace gqa
