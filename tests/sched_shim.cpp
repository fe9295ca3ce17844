// Exposes the split schedule of fd_sched.h to the host tests (compiled by g++).
#include "fd_sched.h"

extern "C" {
void shim_schedule_range(const int *prefix, const int *nonempty, int batch, int hkv, int w, int P, int c, int *b,
                         int *e)
{
    const fd::Schedule s{prefix, nonempty, batch, hkv, w, P};
    s.range(c, b, e);
}
int shim_schedule_cta_of_tile(const int *prefix, const int *nonempty, int batch, int hkv, int w, int P, int t)
{
    const fd::Schedule s{prefix, nonempty, batch, hkv, w, P};
    return s.cta_at(s.pos_of_tile(t));
}
int shim_request_of_tile(const int *prefix, int batch, int t) { return fd::request_of_tile(prefix, batch, t); }
size_t shim_workspace_total(int batch, int hkv, int group, int d) { return fd::workspace_layout(batch, hkv, group, d).total; }
int shim_slots(int batch, int hkv) { return fd::workspace_layout(batch, hkv, 1, 128).slots; }
int shim_tile_tokens() { return fd::kTileTokens; }
int shim_max_ctas() { return fd::kMaxCtas; }
}
