// Split kernel instances for the paged KV layout [num_pages, P, Hkv, D].
#include "fd_launch.h"

namespace fd {

cudaError_t launch_split_paged(int group, const SplitParams &p, const CUtensorMap &tmk,
                               const CUtensorMap &tmv, const SplitLaunch &cfg)
{
    switch (group) {
    case 1: return launch_split_t<1, true, false>(p, tmk, tmv, cfg);
    case 2: return launch_split_t<2, true, false>(p, tmk, tmv, cfg);
    case 4: return launch_split_t<4, true, false>(p, tmk, tmv, cfg);
    case 8: return launch_split_t<8, true, false>(p, tmk, tmv, cfg);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_split_paged_mma(int group, const SplitParams &p, const CUtensorMap &tmk,
                                   const CUtensorMap &tmv, const SplitLaunch &cfg)
{
    switch (group) {
    case 2: return launch_split_t<2, true, true>(p, tmk, tmv, cfg);
    case 4: return launch_split_t<4, true, true>(p, tmk, tmv, cfg);
    case 8: return launch_split_t<8, true, true>(p, tmk, tmv, cfg);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fd
