// One split-kernel variant: compiled once per (layout, K/V element type,
// head_dim) with FD_INST_PAGED, FD_INST_KV (0 bf16, 1 fp16, 2 FP8 E4M3,
// 3 FP8 E5M2) and FD_INST_D defined on the command line.
#include "fd_launch.h"

#if !defined(FD_INST_PAGED) || !defined(FD_INST_KV) || !defined(FD_INST_D)
#error "define FD_INST_PAGED, FD_INST_KV and FD_INST_D"
#endif

namespace fd {

template cudaError_t launch_split_variant<FD_INST_PAGED, FD_INST_KV, FD_INST_D>(
    int, int, bool, const SplitParams &, const CUtensorMap &, const CUtensorMap &, const SplitLaunch &);

}  // namespace fd
