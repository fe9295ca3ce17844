// Split kernel instances for the contiguous KV layout [B, S_max, Hkv, D].
#include "fd_launch.h"

namespace fd {

cudaError_t launch_split_contig(int group, const SplitParams &p, const CUtensorMap &tmk,
                                const CUtensorMap &tmv, const SplitLaunch &cfg)
{
    switch (group) {
    case 1: return launch_split_t<1, false, false>(p, tmk, tmv, cfg);
    case 2: return launch_split_t<2, false, false>(p, tmk, tmv, cfg);
    case 4: return launch_split_t<4, false, false>(p, tmk, tmv, cfg);
    case 8: return launch_split_t<8, false, false>(p, tmk, tmv, cfg);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_split_contig_mma(int group, const SplitParams &p, const CUtensorMap &tmk,
                                    const CUtensorMap &tmv, const SplitLaunch &cfg)
{
    switch (group) {
    case 2: return launch_split_t<2, false, true>(p, tmk, tmv, cfg);
    case 4: return launch_split_t<4, false, true>(p, tmk, tmv, cfg);
    case 8: return launch_split_t<8, false, true>(p, tmk, tmv, cfg);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fd
