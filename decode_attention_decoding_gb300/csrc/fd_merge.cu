// LSE merge kernel instances, launched with programmatic dependent launch so
// their launch overlaps the split kernel's tail.
#include "fd_launch.h"

namespace fd {

// grid = number of segments (requests x kv heads); one CTA per (segment, query head).
template <int G, int D>
static cudaError_t launch_merge_t(const MergeParams &p, int grid, cudaStream_t stream)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, (unsigned)p.n_cols);   // (segment, query column of its head)
    cfg.blockDim = dim3(D);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_kernel<G, D>, p);
}

template <int D>
static cudaError_t launch_merge_d(int group, const MergeParams &p, int grid, cudaStream_t stream)
{
    switch (group) {
    case 1: return launch_merge_t<1, D>(p, grid, stream);
    case 2: return launch_merge_t<2, D>(p, grid, stream);
    case 4: return launch_merge_t<4, D>(p, grid, stream);
    case 8: return launch_merge_t<8, D>(p, grid, stream);
    case 16: return launch_merge_t<16, D>(p, grid, stream);
    case 32: return launch_merge_t<32, D>(p, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_merge(int group, int head_dim, const MergeParams &p, int grid, cudaStream_t stream)
{
    switch (head_dim) {
    case 64: return launch_merge_d<64>(group, p, grid, stream);
    case 128: return launch_merge_d<128>(group, p, grid, stream);
    case 256: return launch_merge_d<256>(group, p, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

// Merge of caller-supplied partial sets: one warp per query row.
cudaError_t launch_merge_parts(int head_dim, const MergePartsParams &p, cudaStream_t stream)
{
    if (p.rows == 0)
        return cudaSuccess;
    const dim3 grid((unsigned)((p.rows + kMergePartsWarps - 1) / kMergePartsWarps)), block(kMergePartsWarps * 32);
    switch (head_dim) {
    case 64: merge_parts_kernel<64><<<grid, block, 0, stream>>>(p); break;
    case 128: merge_parts_kernel<128><<<grid, block, 0, stream>>>(p); break;
    case 256: merge_parts_kernel<256><<<grid, block, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace fd
