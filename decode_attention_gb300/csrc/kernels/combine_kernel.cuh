// Log-sum-exp combine of split-softmax partials (second kernel of a call).
//
// A segment u = (b, kvh) whose attended positions were processed in more than
// one piece has, per piece j, the running max m_j (log2 units), the normaliser
// l_j = sum exp2(s - m_j) and the unnormalised acc_j = sum exp2(s - m_j) v in the
// workspace.  The softmax over the whole range (gemma-4-31B Model Spec,
// "Compute-graph nodes", attn.core rows) is recovered exactly by
//     M = max_j m_j,  o = (sum_j exp2(m_j - M) acc_j) / (sum_j exp2(m_j - M) l_j),
// evaluated here as a running merge over the pieces in the fixed order of
// SegmentParts (static units, then dynamic chunks).
//
// Work items are (segment, 512-element chunk of its G*D outputs); one thread
// owns 4 consecutive outputs of one head and issues the loads of all pieces
// before it merges them.  The kernel is launched right behind the main kernel
// with programmatic dependent launch and waits for it to complete before
// reading the partials; it also resets the dynamic-chunk claim counter.
#pragma once

#include "decode_kernel.cuh"

namespace gqa {

constexpr int kCombineThreads = 128;    // float4 outputs per work item
constexpr int kCombineBatch = 16;       // pieces whose loads are in flight together

template <int G, int D>
__global__ void __launch_bounds__(kCombineThreads)
    gqa_combine_kernel(const DecodeParams p, int num_segments) {
    constexpr int kF4PerSeg = G * D / 4;
    constexpr int kChunksPerSeg = (kF4PerSeg + kCombineThreads - 1) / kCombineThreads;
    __shared__ int4 seg_s[kCombineThreads];

    ptx::grid_dependency_wait();   // the main kernel has finished; its writes are visible
    ptx::allow_dependent_launch();
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.ws_claim = 0u;

    const int tid = threadIdx.x;
    const int items = num_segments * kChunksPerSeg;
    // items of this block: blockIdx.x + k * gridDim.x, k = 0, 1, ...
    for (int k0 = 0; blockIdx.x + k0 * gridDim.x < items; k0 += kCombineThreads) {
        // fetch the partial lists of the next (up to) 128 items in one round trip
        const int it = blockIdx.x + (k0 + tid) * gridDim.x;
        if (it < items) seg_s[tid] = p.ws_segs[it / kChunksPerSeg];
        __syncthreads();
        for (int k = 0; k < kCombineThreads; ++k) {
            const int item = blockIdx.x + (k0 + k) * gridDim.x;
            if (item >= items) break;
            const int4 e = seg_s[k];   // first_s, ns_parts, dk0, nd_parts
            const int nparts = e.y + e.w;
            if (nparts <= 1) continue;   // written directly by the main kernel (or empty)
            const int u = item / kChunksPerSeg;
            const int f4 = (item - u * kChunksPerSeg) * kCombineThreads + tid;
            if (f4 >= kF4PerSeg) continue;
            const int h = (f4 * 4) / D;
            float M = -INFINITY, den = 0.0f;
            float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j0 = 0; j0 < nparts; j0 += kCombineBatch) {
                float mj[kCombineBatch], lj[kCombineBatch];
                float4 aj[kCombineBatch];
#pragma unroll
                for (int q = 0; q < kCombineBatch; ++q) {
                    const int j = j0 + q;
                    mj[q] = -INFINITY;
                    lj[q] = 0.0f;
                    aj[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (j < nparts) {
                        const size_t sl = j < e.y
                                              ? static_cast<size_t>(e.x + j) + u
                                              : static_cast<size_t>(p.dyn_slot_base) + e.z + (j - e.y);
                        const float2 ml = __ldg(reinterpret_cast<const float2*>(p.ws_ml) + sl * G + h);
                        mj[q] = ml.x;
                        lj[q] = ml.y;
                        aj[q] = __ldg(reinterpret_cast<const float4*>(p.ws_acc + sl * G * D) + f4);
                    }
                }
#pragma unroll
                for (int q = 0; q < kCombineBatch; ++q) {
                    if (j0 + q >= nparts) break;
                    const float Mn = fmaxf(M, mj[q]);
                    const float sc = exp2f(M - Mn);   // 0 on the first piece (M = -inf)
                    const float w = exp2f(mj[q] - Mn);
                    den = den * sc + w * lj[q];
                    num.x = num.x * sc + w * aj[q].x;
                    num.y = num.y * sc + w * aj[q].y;
                    num.z = num.z * sc + w * aj[q].z;
                    num.w = num.w * sc + w * aj[q].w;
                    M = Mn;
                }
            }
            const float inv = 1.0f / den;
            // output rows of segment u start at (b H + kvh G) D = u G D (H = KVH G)
            store_out4(p, static_cast<size_t>(u) * G * D + static_cast<size_t>(f4) * 4,
                       make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv));
        }
        __syncthreads();   // seg_s is refilled for the next group of items
    }
}

}  // namespace gqa
