// Split kernel instances: contiguous KV layout [B, S_max, Hkv, D], fp16.
#include "fd_launch.h"

namespace fd {

cudaError_t launch_split_contig_f16(bool mma, int group, const SplitParams &p, const CUtensorMap &tmk,
                                    const CUtensorMap &tmv, const SplitLaunch &cfg)
{
    return launch_split_group<false, true>(mma, group, p, tmk, tmv, cfg);
}

}  // namespace fd
