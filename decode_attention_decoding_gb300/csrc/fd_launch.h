// fd_launch.h -- host-side launch wrappers, one per kernel translation unit.
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fd_kernels.cuh"

namespace fd {

struct SplitLaunch {
    int grid;              // split CTAs
    size_t smem_bytes;     // dynamic shared memory per CTA
    size_t smem_optin;     // the device's opt-in maximum (set once per kernel)
    cudaStream_t stream;
};

// Split kernel with CUDA-core consumers; K/V tensor maps without swizzle.
// Returns cudaErrorInvalidValue for an unsupported group size.
cudaError_t launch_split_contig(int group, const SplitParams &p, const CUtensorMap &tmk,
                                const CUtensorMap &tmv, const SplitLaunch &cfg);
cudaError_t launch_split_paged(int group, const SplitParams &p, const CUtensorMap &tmk,
                               const CUtensorMap &tmv, const SplitLaunch &cfg);
// Split kernel with tensor-core consumers (group 2, 4 or 8); K/V tensor maps
// with 64-dim boxes and the 128-byte swizzle.
cudaError_t launch_split_contig_mma(int group, const SplitParams &p, const CUtensorMap &tmk,
                                    const CUtensorMap &tmv, const SplitLaunch &cfg);
cudaError_t launch_split_paged_mma(int group, const SplitParams &p, const CUtensorMap &tmk,
                                   const CUtensorMap &tmv, const SplitLaunch &cfg);

// Shared by the two split translation units.
template <int G, bool PAGED, bool MMA>
cudaError_t launch_split_t(const SplitParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           const SplitLaunch &c)
{
    // Raise the kernel's dynamic shared-memory limit to the device's opt-in
    // maximum, once per device (so later calls may be captured in a graph).
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(split_kernel<G, PAGED, MMA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)c.smem_optin);
        if (e != cudaSuccess)
            return e;
        configured.fetch_or(bit, std::memory_order_release);
    }
    // Programmatic dependent launch: the kernel's prologue may overlap the
    // previous kernel in the stream; it waits for it before reading inputs.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)c.grid);
    cfg.blockDim = dim3(kSplitThreads);
    cfg.dynamicSmemBytes = c.smem_bytes;
    cfg.stream = c.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_kernel<G, PAGED, MMA>, p, tmk, tmv);
}

}  // namespace fd
