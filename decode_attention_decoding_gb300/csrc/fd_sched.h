// fd_sched.h -- how the KV tiles of one decode call are divided among CTAs.
//
// Work is a list of tiles of BN tokens.  Request b with length L_b has
// n_b = ceil(L_b / BN) tiles per kv head; a "segment" u = b * Hkv + h is the
// n_b tiles of (request b, kv head h).  Tiles are numbered request by
// request, kv head by kv head, token by token, so
//
//     prefix[b]      = Hkv * sum_{b' < b} n_b'        (first tile of request b)
//     segment u      = tiles [prefix[b] + h n_b, prefix[b] + (h + 1) n_b)
//     T = prefix[B]  = total number of tiles.
//
// The P split CTAs each take one contiguous run of tiles of (nearly) equal
// length: CTA c gets floor(T/P) tiles, plus one if c < T mod P.  A CTA that
// covers a whole segment writes that segment's final output; otherwise it
// writes a partial (normalised output + log-sum-exp) for every segment it
// touches, into slot u + c.  That slot is unique: CTAs and segments are both
// visited in increasing order, so two CTAs c < c' that share a slot would
// need u > u' while c' only sees segments >= the last one of c.  There are
// at most B*Hkv + P - 1 slots.  The merge step finds the CTAs of segment u
// from its first and last tile with cta_of_tile().
//
// Shared by the host (tests, sizing) and the kernels.
#pragma once

#include <cstddef>

#if defined(__CUDACC__)
#define FD_HD __host__ __device__ __forceinline__
#else
#define FD_HD inline
#endif

namespace fd {

constexpr int kTileTokens = 64;   // BN: tokens per KV tile
constexpr int kMaxCtas = 1024;    // upper bound on split CTAs (sizes the workspace)
constexpr int kMaxBatch = 4096;   // requests per call (the tile prefix lives in shared memory)

FD_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Tiles [begin, end) of CTA c out of P sharing T tiles.
FD_HD void cta_tile_range(int T, int P, int c, int *begin, int *end)
{
    const int base = T / P, rem = T % P;
    *begin = c * base + (c < rem ? c : rem);
    *end = *begin + base + (c < rem ? 1 : 0);
}

// The CTA that owns tile t (0 <= t < T).
FD_HD int cta_of_tile(int T, int P, int t)
{
    const int base = T / P, rem = T % P;
    const int cut = rem * (base + 1);
    if (t < cut)
        return t / (base + 1);
    return rem + (t - cut) / base;   // base > 0 whenever t >= cut and t < T
}

// Index of the request whose tiles contain tile t: the last b with
// prefix[b] <= t among prefix[0..batch] (prefix is non-decreasing and
// prefix[batch] > t).  Requests with no tiles are skipped automatically.
FD_HD int request_of_tile(const int *prefix, int batch, int t)
{
    int lo = 0, hi = batch;   // invariant: prefix[lo] <= t < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= t)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Workspace layout (byte offsets from the workspace base).
struct WorkspaceLayout {
    size_t err_off;      // uint32 sticky error word
    size_t prefix_off;   // int32 [batch + 1]
    size_t lse_off;      // fp32 [slots][group]
    size_t o_off;        // fp32 [slots][group][head_dim]
    size_t total;
    int slots;
};

FD_HD size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

FD_HD WorkspaceLayout workspace_layout(int batch, int num_kv_heads, int group, int head_dim)
{
    WorkspaceLayout w;
    w.slots = batch * num_kv_heads + kMaxCtas;
    w.err_off = 0;
    w.prefix_off = 256;
    w.lse_off = align_up(w.prefix_off + sizeof(int) * (size_t)(batch + 1), 256);
    w.o_off = align_up(w.lse_off + sizeof(float) * (size_t)w.slots * group, 256);
    w.total = align_up(w.o_off + sizeof(float) * (size_t)w.slots * group * head_dim, 256);
    return w;
}

}  // namespace fd
