// Shared launch helper for the per-geometry kernel translation units.
#pragma once

#include <mutex>

#include "kernels/combine_kernel.cuh"
#include "launch.h"

namespace gqa {

// Launches the main kernel and, right behind it, the combine kernel.  Both opt
// in to programmatic dependent launch: each may start while the kernel before it
// in the stream drains, and waits (griddepcontrol.wait) before touching global
// memory that kernel writes.
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

    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.grid));
    cfg.blockDim = dim3((Pol::NC + 1) * 32);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = a.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gqa_decode_kernel<Pol, kPaged>, a.tm_k, a.tm_v, a.p);
    if (e != cudaSuccess) return e;

    const int segments = a.p.B * a.p.KVH;
    constexpr int kChunksPerSeg = (Pol::G * Pol::D / 4 + kCombineThreads - 1) / kCombineThreads;
    const int items = segments * kChunksPerSeg;
    const int cgrid = items < 4 * a.grid ? items : 4 * a.grid;
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
