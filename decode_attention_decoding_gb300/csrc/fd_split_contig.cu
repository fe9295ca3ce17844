// Split kernel instances: contiguous KV layout [B, S_max, Hkv, D], bf16.
#include "fd_launch.h"

namespace fd {

cudaError_t launch_split_contig_bf16(bool mma, int group, const SplitParams &p, const CUtensorMap &tmk,
                                     const CUtensorMap &tmv, const SplitLaunch &cfg)
{
    return launch_split_group<false, false>(mma, group, p, tmk, tmv, cfg);
}

cudaError_t launch_split_contig(int group, const SplitParams &p, const CUtensorMap &tmk,
                                const CUtensorMap &tmv, const SplitLaunch &cfg)
{
    return launch_split_group<false, false>(false, group, p, tmk, tmv, cfg);
}

}  // namespace fd
