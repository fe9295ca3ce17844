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

// Split kernel with CUDA-core consumers on bf16 inputs; K/V tensor maps
// without swizzle (used by the no-workspace entry point).  Returns
// cudaErrorInvalidValue for an unsupported group size.
cudaError_t launch_split_contig(int group, const SplitParams &p, const CUtensorMap &tmk,
                                const CUtensorMap &tmv, const SplitLaunch &cfg);

// Any variant: layout (paged), consumers (mma: tensor cores for group 2, 4
// or 8, with swizzled K/V maps), input element type (f16: IEEE fp16, else
// bf16).  One translation unit per (layout, element type) defines it.
cudaError_t launch_split_contig_bf16(bool mma, int group, const SplitParams &p, const CUtensorMap &tmk,
                                     const CUtensorMap &tmv, const SplitLaunch &cfg);
cudaError_t launch_split_contig_f16(bool mma, int group, const SplitParams &p, const CUtensorMap &tmk,
                                    const CUtensorMap &tmv, const SplitLaunch &cfg);
cudaError_t launch_split_paged_bf16(bool mma, int group, const SplitParams &p, const CUtensorMap &tmk,
                                    const CUtensorMap &tmv, const SplitLaunch &cfg);
cudaError_t launch_split_paged_f16(bool mma, int group, const SplitParams &p, const CUtensorMap &tmk,
                                   const CUtensorMap &tmv, const SplitLaunch &cfg);

// LSE merge of the split partials; grid = number of segments (requests x kv
// heads).  Launched as a programmatic dependent of the split kernel.
cudaError_t launch_merge(int group, const MergeParams &p, int grid, cudaStream_t stream);

// Shared by the split translation units.
template <int G, bool PAGED, bool MMA, bool F16>
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
        e = cudaFuncSetAttribute(split_kernel<G, PAGED, MMA, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    return cudaLaunchKernelEx(&cfg, split_kernel<G, PAGED, MMA, F16>, p, tmk, tmv);
}

template <bool PAGED, bool F16>
cudaError_t launch_split_group(bool mma, int group, const SplitParams &p, const CUtensorMap &tmk,
                               const CUtensorMap &tmv, const SplitLaunch &c)
{
    if (mma) {
        switch (group) {
        case 2: return launch_split_t<2, PAGED, true, F16>(p, tmk, tmv, c);
        case 4: return launch_split_t<4, PAGED, true, F16>(p, tmk, tmv, c);
        case 8: return launch_split_t<8, PAGED, true, F16>(p, tmk, tmv, c);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (group) {
    case 1: return launch_split_t<1, PAGED, false, F16>(p, tmk, tmv, c);
    case 2: return launch_split_t<2, PAGED, false, F16>(p, tmk, tmv, c);
    case 4: return launch_split_t<4, PAGED, false, F16>(p, tmk, tmv, c);
    case 8: return launch_split_t<8, PAGED, false, F16>(p, tmk, tmv, c);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fd
