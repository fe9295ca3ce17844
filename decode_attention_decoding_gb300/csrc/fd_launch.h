// fd_launch.h -- host-side launch wrappers, one per kernel translation unit.
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fd.h"
#include "fd_kernels.cuh"

namespace fd {

struct SplitLaunch {
    int grid;              // split CTAs
    size_t smem_bytes;     // dynamic shared memory per CTA
    size_t smem_optin;     // the device's opt-in maximum (set once per kernel)
    cudaStream_t stream;
    int late_trigger;      // the merge lets the next kernel launch only after its wait (MergeParams)
    // Non-null: do not launch; store how many CTAs of the kernel fit on one
    // SM with this shared memory (cudaOccupancyMaxActiveBlocksPerMultiprocessor).
    int *blocks_per_sm = nullptr;
};

// Device properties a launch plan needs.
struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;
};

// Calls with fewer (estimated) KV tiles per split CTA than this count as
// short: they keep less K/V in flight per CTA and kv heads are not fused for
// them (fd_api.cu).
constexpr double kFuseMinTilesPerCta = 24.0;

// The split Schedule's cost of a segment start, in tiles (fd_sched.h): a CTA
// that touches one more segment takes this many fewer tiles.
constexpr int kSegCostTiles = 2;

// The tcgen05 score consumers (kConsTc5) are the default for paired E4M3
// heads of up to this many query columns per kv head (fd_api.cu).
constexpr int kTc5DefaultColumns = 4;

// Shared-memory plan of the split kernel (fd_api.cu): pipeline stages, the
// offsets of every region in sp, the L2 prefetch before the dependency wait
// (sp->prefetch_tiles), and the byte size and merge trigger in launch, for
// the call's consumers (kCons*), column group, row dims d, K/V element size,
// batch, and the estimated tiles and K/V bytes per split CTA.
// FD_ERR_UNSUPPORTED if two stages do not fit.
fd_status plan_smem(const DeviceInfo &dev, int cons, int group, int d, int elem_bytes, int batch,
                    double tiles_per_cta, double kv_bytes_per_cta, SplitParams *sp, SplitLaunch *launch);

// K and V tensor maps of a call (fd_api.cu): rows are (token, kv head)
// pairs of d elements of type kv (kKv*), loaded box_rows tokens at a time.
// The tensor-core consumers (mma) take 128-byte swizzled boxes, as one 4-D
// box per load when the driver accepts the view (sets sp->box4d and
// sp->box_rows_log2); the CUDA-core consumers take whole rows.  Returns
// FD_ERR_CUDA if the driver rejects the maps.
fd_status encode_kv_maps(CUtensorMap *tmk, CUtensorMap *tmv, const void *k, const void *v, int hkv,
                         long long rows, int box_rows, bool mma, int kv, int d, SplitParams *sp);

// LSE merge of the split partials; grid = number of segments (requests x kv
// heads).  Launched as a programmatic dependent of the split kernel.
// Returns cudaErrorInvalidValue for an unsupported group size or head_dim.
cudaError_t launch_merge(int group, int head_dim, const MergeParams &p, int grid, cudaStream_t stream);

// Merge of n caller-supplied partial sets (fd_merge_partials); head_dim 64,
// 128 or 256 (cudaErrorInvalidValue otherwise).
cudaError_t launch_merge_parts(int head_dim, const MergePartsParams &p, cudaStream_t stream);

// Shared by the split translation units.
template <int G, bool PAGED, int CONS, int KV, int D, bool CPA = false>
cudaError_t launch_split_t(const SplitParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           const SplitLaunch &c)
{
    // Raise the kernel's dynamic shared-memory limit to the device's opt-in
    // maximum, once per device (so later calls may be captured in a graph);
    // again if a launch is refused (the device's context was reset since).
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = 1ull << (dev & 63);
    auto configure = [&]() -> cudaError_t {
        const cudaError_t r = cudaFuncSetAttribute(split_kernel<G, PAGED, CONS, KV, D, CPA>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem_optin);
        if (r == cudaSuccess)
            configured.fetch_or(bit, std::memory_order_release);
        return r;
    };
    if (!(configured.load(std::memory_order_acquire) & bit) && (e = configure()) != cudaSuccess)
        return e;
    if (c.blocks_per_sm)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(c.blocks_per_sm, split_kernel<G, PAGED, CONS, KV, D, CPA>,
                                                             split_threads(CONS, CPA), c.smem_bytes);
    // Programmatic dependent launch: the kernel's prologue may overlap the
    // previous kernel in the stream; it waits for it before reading inputs.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)c.grid);
    cfg.blockDim = dim3(split_threads(CONS, CPA));
    cfg.dynamicSmemBytes = c.smem_bytes;
    cfg.stream = c.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, split_kernel<G, PAGED, CONS, KV, D, CPA>, p, tmk, tmv);
    if (e == cudaErrorInvalidValue) {   // a refused launch leaves no sticky error: clear it and retry once
        (void)cudaGetLastError();
        if ((e = configure()) != cudaSuccess)
            return e;
        e = cudaLaunchKernelEx(&cfg, split_kernel<G, PAGED, CONS, KV, D, CPA>, p, tmk, tmv);
    }
    return e;
}

// One split-kernel variant per (layout, K/V element type, row dims D):
// consumers on CUDA cores (group 1 to 8), on tensor cores (group 2 to 16,
// swizzled K/V maps, rows of at least 128 bytes), or on tensor cores with two
// fused kv heads per row (group = columns per head, 1 to 16; D = 2 x head_dim),
// or with scores in TMEM (kConsTc5: FP8, D = 256, group 1 to 8).
// cp_async: paged with pages under 8 tokens on the tensor cores (the CPA
// instances, 384 threads; tensor-core groups only).
// Returns cudaErrorInvalidValue for an unsupported combination.
template <bool PAGED, int KV, int D>
cudaError_t launch_split_variant(int cons, int group, bool cp_async, const SplitParams &p,
                                 const CUtensorMap &tmk, const CUtensorMap &tmv, const SplitLaunch &c)
{
    if (cp_async) {   // pages under 8 tokens on the tensor cores: rows copied with cp.async
        if (cons != kConsMma)
            return cudaErrorInvalidValue;
        if constexpr (PAGED && Shape<D, KV>::kParts >= 1) {
            switch (group) {
            case 2: return launch_split_t<2, PAGED, kConsMma, KV, D, true>(p, tmk, tmv, c);
            case 4: return launch_split_t<4, PAGED, kConsMma, KV, D, true>(p, tmk, tmv, c);
            case 8: return launch_split_t<8, PAGED, kConsMma, KV, D, true>(p, tmk, tmv, c);
            case 16: return launch_split_t<16, PAGED, kConsMma, KV, D, true>(p, tmk, tmv, c);
            default: return cudaErrorInvalidValue;
            }
        }
        return cudaErrorInvalidValue;
    }
    if (cons == kConsMma) {
        if constexpr (Shape<D, KV>::kParts >= 1) {
            switch (group) {
            case 2: return launch_split_t<2, PAGED, kConsMma, KV, D>(p, tmk, tmv, c);
            case 4: return launch_split_t<4, PAGED, kConsMma, KV, D>(p, tmk, tmv, c);
            case 8: return launch_split_t<8, PAGED, kConsMma, KV, D>(p, tmk, tmv, c);
            case 16: return launch_split_t<16, PAGED, kConsMma, KV, D>(p, tmk, tmv, c);
            default: return cudaErrorInvalidValue;
            }
        }
        return cudaErrorInvalidValue;
    }
    if (cons == kConsTc5) {   // scores in TMEM: two fused FP8 heads of 128 dims, up to 8 columns each
        if constexpr (kv_is_fp8(KV) && D == 256) {
            switch (group) {
            case 1: return launch_split_t<1, PAGED, kConsTc5, KV, D>(p, tmk, tmv, c);
            case 2: return launch_split_t<2, PAGED, kConsTc5, KV, D>(p, tmk, tmv, c);
            case 4: return launch_split_t<4, PAGED, kConsTc5, KV, D>(p, tmk, tmv, c);
            case 8: return launch_split_t<8, PAGED, kConsTc5, KV, D>(p, tmk, tmv, c);
            default: return cudaErrorInvalidValue;
            }
        }
        return cudaErrorInvalidValue;
    }
    if (cons == kConsMmaPair) {
        if constexpr (Shape<D, KV>::kParts >= 1 && D >= 128) {
            switch (group) {
            case 1: return launch_split_t<1, PAGED, kConsMmaPair, KV, D>(p, tmk, tmv, c);
            case 2: return launch_split_t<2, PAGED, kConsMmaPair, KV, D>(p, tmk, tmv, c);
            case 4: return launch_split_t<4, PAGED, kConsMmaPair, KV, D>(p, tmk, tmv, c);
            case 8: return launch_split_t<8, PAGED, kConsMmaPair, KV, D>(p, tmk, tmv, c);
            case 16: return launch_split_t<16, PAGED, kConsMmaPair, KV, D>(p, tmk, tmv, c);
            default: return cudaErrorInvalidValue;
            }
        }
        return cudaErrorInvalidValue;
    }
    switch (group) {
    case 1: return launch_split_t<1, PAGED, kConsCudaCores, KV, D>(p, tmk, tmv, c);
    case 2: return launch_split_t<2, PAGED, kConsCudaCores, KV, D>(p, tmk, tmv, c);
    case 4: return launch_split_t<4, PAGED, kConsCudaCores, KV, D>(p, tmk, tmv, c);
    case 8: return launch_split_t<8, PAGED, kConsCudaCores, KV, D>(p, tmk, tmv, c);
    default: return cudaErrorInvalidValue;
    }
}

// Each variant is compiled in its own translation unit (fd_split_inst.cu,
// built once per combination), so they compile in parallel.
#define FD_SPLIT_VARIANTS_KV(X, P, KV) X(P, KV, 64) X(P, KV, 128) X(P, KV, 256)
#define FD_SPLIT_VARIANTS_P(X, P)                                                          \
    FD_SPLIT_VARIANTS_KV(X, P, kKvBf16) FD_SPLIT_VARIANTS_KV(X, P, kKvF16)                   \
    FD_SPLIT_VARIANTS_KV(X, P, kKvE4m3) FD_SPLIT_VARIANTS_KV(X, P, kKvE5m2)
#define FD_SPLIT_VARIANTS(X) FD_SPLIT_VARIANTS_P(X, false) FD_SPLIT_VARIANTS_P(X, true)
#define FD_EXTERN_SPLIT(P, KV, D)                                                                \
    extern template cudaError_t launch_split_variant<P, KV, D>(int, int, bool, const SplitParams &, \
                                                              const CUtensorMap &,             \
                                                              const CUtensorMap &, const SplitLaunch &);
FD_SPLIT_VARIANTS(FD_EXTERN_SPLIT)
#undef FD_EXTERN_SPLIT

// Split launch for a call: layout, K/V element type (kKv*) and head_dim pick
// the variant.  Returns cudaErrorInvalidValue for an unsupported head_dim.
inline cudaError_t launch_split(bool paged, int kv, int head_dim, int cons, int group, bool cp_async,
                                const SplitParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                const SplitLaunch &c)
{
#define FD_PICK_SPLIT(P, KV, D)                                                 \
    if (paged == P && kv == KV && head_dim == D)                              \
        return launch_split_variant<P, KV, D>(cons, group, cp_async, p, tmk, tmv, c);
    FD_SPLIT_VARIANTS(FD_PICK_SPLIT)
#undef FD_PICK_SPLIT
    return cudaErrorInvalidValue;
}

}  // namespace fd
