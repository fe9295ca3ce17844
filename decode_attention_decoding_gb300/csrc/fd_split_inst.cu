// One split-kernel variant: compiled once per (layout, element type,
// head_dim) with FD_INST_PAGED, FD_INST_F16 and FD_INST_D defined on the
// command line (the build compiles this file twelve times).
#include "fd_launch.h"

#if !defined(FD_INST_PAGED) || !defined(FD_INST_F16) || !defined(FD_INST_D)
#error "define FD_INST_PAGED, FD_INST_F16 and FD_INST_D"
#endif

namespace fd {

template cudaError_t launch_split_variant<FD_INST_PAGED, FD_INST_F16, FD_INST_D>(
    bool, int, const SplitParams &, const CUtensorMap &, const CUtensorMap &, const SplitLaunch &);

}  // namespace fd
