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
// cost, where a tile costs 1 and every segment start costs W more: a CTA
// flushes every segment it touches (a CTA-wide combine and the output
// writes), and on GB300 a CTA's time grew by one to two tiles' worth for
// each segment it touched.  Tile t sits at cost position
//
//     pos(t) = t + W * S(t),   S(t) = segments that start at tiles <= t,
//
// which grows with t; with C = T + W * (non-empty segments) and the first
// P' = min(P, C) CTAs, CTA c owns the tiles with c <= pos(t) * P' / C < c + 1
// (Schedule::cta_at), a contiguous run (Schedule::range).  Since P' <= C,
// consecutive tiles of a segment (positions +1 apart) fall to the same CTA
// or the next one: the CTAs of a segment are consecutive, and each of them
// owns some of its tiles.  W = 0 gives runs of equal length.  A CTA that covers a
// whole segment writes that segment's final output; otherwise it writes a
// partial (normalised output + log-sum-exp) for every segment it touches,
// into slot u + c.  That slot is unique: CTAs and segments are both visited
// in increasing order, so two CTAs c < c' that share a slot would need u > u'
// while c' only sees segments >= the last one of c.  There are at most
// B*Hkv + P - 1 slots.  The merge step finds the CTAs of segment u from its
// first and last tile.
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

// The division of a call's tiles among P CTAs.  prefix[b] = Hkv * (tiles of
// requests < b) and nonempty[b] = requests < b with at least one tile, for
// b = 0 .. batch; hkv: the launch's kv heads; w: the cost of a segment start,
// in tiles.
struct Schedule {
    const int *prefix;
    const int *nonempty;
    int batch, hkv, w, P;

    FD_HD int tiles() const { return prefix[batch]; }
    // total cost C
    FD_HD long long cost() const { return (long long)prefix[batch] + (long long)w * hkv * nonempty[batch]; }
    // cost position of the first tile of segment (b, h); its tiles follow at +1 each
    FD_HD long long seg_pos(int b, int h) const
    {
        const int nb = (prefix[b + 1] - prefix[b]) / hkv;
        return (long long)prefix[b] + (long long)h * nb + (long long)w * ((long long)hkv * nonempty[b] + h + 1);
    }
    // CTAs that take tiles: P' = min(P, C), so that no CTA of a segment is skipped
    FD_HD int ctas() const
    {
        const long long C = cost();
        return C < P ? (int)C : P;
    }
    FD_HD int cta_at(long long pos) const { return (int)(pos * ctas() / cost()); }
    // cost position of tile t (0 <= t < tiles())
    FD_HD long long pos_of_tile(int t) const
    {
        const int b = request_of_tile(prefix, batch, t);
        const int nb = (prefix[b + 1] - prefix[b]) / hkv;
        const int h = (t - prefix[b]) / nb;
        return seg_pos(b, h) + (t - prefix[b] - h * nb);
    }
    // The first tile whose cost position is >= x (tiles() if none).
    FD_HD int tile_at(long long x) const
    {
        if (x >= cost())
            return tiles();
        // A_r = cost at the end of request r; the first r with A_r > x holds the tile
        int lo = 0, hi = batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            const long long a = (long long)prefix[mid + 1] + (long long)w * hkv * nonempty[mid + 1];
            if (a > x)
                hi = mid;
            else
                lo = mid + 1;
        }
        const int r = lo;
        const int nb = (prefix[r + 1] - prefix[r]) / hkv;
        // within r, head h's tiles sit at relative positions h (nb + w) + w + j, j < nb
        const long long q = x - ((long long)prefix[r] + (long long)w * hkv * nonempty[r]) - w;
        if (q <= 0)
            return prefix[r];
        long long h = q / (nb + w), j = q - h * (nb + w);
        if (j >= nb) {   // in the gap before head h + 1
            ++h;
            j = 0;
        }
        return prefix[r] + (int)(h * nb + j);
    }
    // Tiles [begin, end) of CTA c: the cost positions [ceil(c C / P'), ceil((c + 1) C / P'));
    // CTAs c >= P' take none.
    FD_HD void range(int c, int *begin, int *end) const
    {
        const long long C = cost();
        const long long Pe = ctas();
        if (Pe == 0 || c >= Pe) {
            *begin = *end = tiles();
            return;
        }
        *begin = tile_at((C * c + Pe - 1) / Pe);
        *end = tile_at((C * (c + 1) + Pe - 1) / Pe);
    }
};

// Workspace layout (byte offsets from the workspace base).
struct WorkspaceLayout {
    size_t err_off;      // uint32 sticky error word
    size_t prefix_off;   // int32 [batch + 1] tile prefix, then int32 [batch + 1] non-empty requests
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
    w.lse_off = align_up(w.prefix_off + 2 * sizeof(int) * (size_t)(batch + 1), 256);
    w.o_off = align_up(w.lse_off + sizeof(float) * (size_t)w.slots * group, 256);
    w.total = align_up(w.o_off + sizeof(float) * (size_t)w.slots * group * head_dim, 256);
    return w;
}

}  // namespace fd
