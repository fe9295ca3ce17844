// Split kernel instances: paged KV layout [num_pages, P, Hkv, D], bf16.
#include "fd_launch.h"

namespace fd {

cudaError_t launch_split_paged_bf16(bool mma, int group, const SplitParams &p, const CUtensorMap &tmk,
                                    const CUtensorMap &tmv, const SplitLaunch &cfg)
{
    return launch_split_group<true, false>(mma, group, p, tmk, tmv, cfg);
}

}  // namespace fd
