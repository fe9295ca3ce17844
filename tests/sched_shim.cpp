// Exposes the split schedule of fd_sched.h to the host tests (compiled by g++).
#include "fd_sched.h"

extern "C" {
void shim_cta_tile_range(int T, int P, int c, int *b, int *e) { fd::cta_tile_range(T, P, c, b, e); }
int shim_cta_of_tile(int T, int P, int t) { return fd::cta_of_tile(T, P, t); }
int shim_request_of_tile(const int *prefix, int batch, int t) { return fd::request_of_tile(prefix, batch, t); }
size_t shim_workspace_total(int batch, int hkv, int group, int d) { return fd::workspace_layout(batch, hkv, group, d).total; }
int shim_slots(int batch, int hkv) { return fd::workspace_layout(batch, hkv, 1, 128).slots; }
int shim_tile_tokens() { return fd::kTileTokens; }
int shim_max_ctas() { return fd::kMaxCtas; }
}
