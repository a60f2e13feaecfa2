// Shared launch helper for the per-geometry kernel translation units.
#pragma once

#include <mutex>

#include "launch.h"

namespace gqa {

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

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.grid));
    cfg.blockDim = dim3((Pol::NC + 1) * 32);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = a.stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, gqa_decode_kernel<Pol, kPaged>, a.tm_k, a.tm_v, a.p);
}

}  // namespace gqa
