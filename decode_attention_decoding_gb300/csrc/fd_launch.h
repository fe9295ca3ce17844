// fd_launch.h -- host-side launch wrappers, one per kernel translation unit.
#pragma once

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

// Returns cudaErrorInvalidValue for an unsupported group size.
cudaError_t launch_split_contig(int group, const SplitParams &p, const CUtensorMap &tmk,
                                const CUtensorMap &tmv, const SplitLaunch &cfg);
cudaError_t launch_split_paged(int group, const SplitParams &p, const CUtensorMap &tmk,
                               const CUtensorMap &tmv, const SplitLaunch &cfg);
cudaError_t launch_merge(int group, const MergeParams &p, int grid, cudaStream_t stream);

// Shared by the two split translation units.
template <int G, bool PAGED>
cudaError_t launch_split_t(const SplitParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           const SplitLaunch &c)
{
    // cudaFuncSetAttribute is idempotent and cheap; it raises the kernel's
    // dynamic shared-memory limit to the device's opt-in maximum.
    cudaError_t e = cudaFuncSetAttribute(split_kernel<G, PAGED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)c.smem_optin);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)c.grid);
    cfg.blockDim = dim3(kSplitThreads);
    cfg.dynamicSmemBytes = c.smem_bytes;
    cfg.stream = c.stream;
    return cudaLaunchKernelEx(&cfg, split_kernel<G, PAGED>, p, tmk, tmv);
}

}  // namespace fd
