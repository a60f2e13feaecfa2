// Log-sum-exp combine of split-softmax partials (second kernel of a call).
//
// A segment u = (b, kvh) whose attended positions were processed in more than
// one piece has, per piece j and query row r, the running max m_j (log2 units),
// the normaliser l_j = sum exp2(s - m_j) and the unnormalised acc_j =
// sum exp2(s - m_j) v in the workspace.  A segment has R = T * G query rows, row
// r = t * G + h being query token t and head h of the KV head's group.  A piece in
// which a row saw no key has m_j = -inf and l_j = 0 (weight 0); a row that saw no
// key in any piece (a query before the start of its sequence) is the empty sum, 0.
// The softmax over the whole range (gemma-4-31B Model Spec, "Compute-graph
// nodes", attn.core rows) is recovered exactly by
//     M = max_j m_j,  o = (sum_j exp2(m_j - M) acc_j) / (sum_j exp2(m_j - M) l_j),
// evaluated here as a running merge over the pieces in the fixed order of
// SegmentParts (static units, then dynamic chunks).
//
// Work items are (segment, 512-element chunk of its R*D outputs); one thread
// owns 4 consecutive outputs of one query row and issues the loads of all pieces
// before it merges them.  The kernel is launched right behind the main kernel
// with programmatic dependent launch and waits for it to complete before
// reading the partials; it also resets the dynamic-chunk claim counter.
#pragma once

#include "decode_kernel.cuh"

namespace gqa {

constexpr int kCombineThreads = 128;    // float4 outputs per work item
constexpr int kCombineBatch = 16;       // pieces whose loads are in flight together
// Blocks per SM of a combine launch: each block merges its items one after the
// other, one round trip of loads each, so more blocks shorten the kernel (4 per SM
// left sliding T = 8 with ~13 items per block, ~15 us)
constexpr int kCombineBlocksPerSm = 16;

template <int G, int D>
__global__ void __launch_bounds__(kCombineThreads)
    gqa_combine_kernel(const DecodeParams p, int num_segments) {
    const int T = p.T > 1 ? p.T : 1;
    const int R = T * G;   // query rows per segment
    const int kF4PerSeg = R * D / 4;
    const int kChunksPerSeg = (kF4PerSeg + kCombineThreads - 1) / kCombineThreads;
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
            const int h = (f4 * 4) / D;   // query row t * G + head
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
                        const float2 ml = __ldg(reinterpret_cast<const float2*>(p.ws_ml) + sl * R + h);
                        mj[q] = ml.x;
                        lj[q] = ml.y;
                        aj[q] = __ldg(reinterpret_cast<const float4*>(p.ws_acc + sl * R * D) + f4);
                    }
                }
#pragma unroll
                for (int q = 0; q < kCombineBatch; ++q) {
                    if (j0 + q >= nparts) break;
                    const float Mn = fmaxf(M, mj[q]);
                    // 0 on the first piece (M = -inf); a piece that saw no key weighs 0
                    const float sc = M == -INFINITY ? 0.0f : exp2f(M - Mn);
                    const float w = mj[q] == -INFINITY ? 0.0f : exp2f(mj[q] - Mn);
                    den = den * sc + w * lj[q];
                    num.x = num.x * sc + w * aj[q].x;
                    num.y = num.y * sc + w * aj[q].y;
                    num.z = num.z * sc + w * aj[q].z;
                    num.w = num.w * sc + w * aj[q].w;
                    M = Mn;
                }
            }
            // no key in any piece: the empty sum (a NaN normaliser from a bad page stays NaN)
            const float inv = den == 0.0f ? 0.0f : 1.0f / den;
            // row t * G + g of segment u = (b, kvh) is output row (b T + t) H + kvh G + g
            // of [B, T, H, D] (for T = 1: u G + g)
            const int KVH = p.KVH;
            const int b = u / KVH, kvh = u - b * KVH, t = h / G, g = h - t * G;
            const size_t row = (static_cast<size_t>(b) * T + t) * p.H + kvh * G + g;
            store_out4(p, row * D + (f4 * 4 - h * D),
                       make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv));
        }
        __syncthreads();   // seg_s is refilled for the next group of items
    }
}

}  // namespace gqa
