// fd_kernels.cuh -- split-KV decode attention kernels (sm_103a).
//
// Split kernel ("pass 1" of 纯手搓 flash decoding sm120, section 1/2; the
// Flash-Decoding section of the FlashAttention handbook page): a persistent
// grid of P CTAs, each taking a contiguous run of 64-token KV tiles (see
// fd_sched.h).  Per CTA:
//   * warp 8 is the producer: it walks the CTA's tiles and, for each, waits
//     for a free shared-memory stage, writes the tile's metadata, and issues
//     TMA loads of the K and V tiles (paged: one load per page, addressed
//     through the block table) that complete on the stage's "full" mbarrier;
//   * warps 0..7 are consumers, of one of four kinds (kCons*):
//       - CUDA cores (shown here): warp w reads rows 8w..8w+7 of every tile,
//         32/(D/8) rows at a time (a row spans D/8 lanes; each lane holds 8 of
//         the D head dimensions, one 16-byte shared load, or 8 bytes of FP8
//         codes).  For every query column of the kv head (its GQA group, times
//         the new tokens of the step) it forms the score q.k in fp32 (packed
//         fp32x2 FMAs, a shuffle reduction over the row's lanes), keeps an
//         online softmax in the log2 domain (running max m, running sum l,
//         fp32 accumulator rescaled by 2^(m_old - m_new) every tile, as in the
//         handbook's FlashAttention section), and accumulates p * V;
//       - tensor cores, a warp pair sharing the columns (split_consumer_mma);
//       - tensor cores on two fused kv heads, one per warp of a pair;
//       - for FP8 caches on two fused kv heads: the scores from tcgen05 MMAs
//         into tensor memory, issued by a tenth warp (split_score_issuer), and
//         P.V on warp MMAs, four consumer warps per tile.
//     Each consumer warp then releases the stage on its "empty" mbarrier --
//     there is no CTA-wide barrier per tile.
//   * At the last tile of a segment (request, kv head) within the CTA, the
//     consumer warps merge their states through shared memory and write
//     either the final O and natural-log LSE (the CTA saw the whole segment)
//     or a normalised partial O and its LSE (lse = m ln2 + ln l).
// Merge kernel ("pass 2", section 2 of the sm120 article): one CTA per
// (segment, query column) combines that column's partials:
// LSE = max + ln sum exp(lse_i - max), O = sum O_i exp(lse_i - LSE).
#pragma once

#include "fd_device.cuh"
#include "fd_sched.h"

namespace fd {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
// Producer warps: one issues TMA loads; copying small pages with cp.async
// (the split kernel's CPA instances) takes four.  Twelve warps still put at
// most 3 on each SM sub-partition, so the consumers keep 168 registers a
// thread; the other instances keep the smaller block, which leaves registers
// for the merge CTAs that launch early beside it.
constexpr int kProducerWarps = 4;
constexpr int kSplitThreads = kConsumerThreads + 32;                       // one producer warp
constexpr int kSplitThreadsCpAsync = kConsumerThreads + 32 * kProducerWarps;
constexpr int kPairs = kConsumerWarps / 2;
// The TMEM-score instances (kConsTc5) add one warp that issues the
// tensor-core score MMAs.
constexpr int kSplitThreadsTc5 = kConsumerThreads + 64;
// Their TMEM: kTc5Buffers score buffers of kTc5Cols fp32 columns each
// (one per tile in flight; columns 16 k + 8 hh + c: FP8 query part k of
// column c of paired head hh; up to kTc5MaxParts parts).
constexpr int kTc5Buffers = 4;
constexpr int kTc5MaxParts = 4;
constexpr int kTc5Cols = 64;
constexpr int kTc5TmemCols = kTc5Buffers * kTc5Cols;
// Their shared region (SplitParams::off_tc, 1024-byte aligned): the query
// operand (up to 48 rows of 128 E4M3 codes, swizzled), each consumer warp's weights
// (32 tokens x 8 columns of fp16, high parts then low parts), the score
// multipliers of each buffer (2 heads x 8 columns), the score-ready and
// buffer-free barriers, and the TMEM address.
constexpr int kTc5QBytes = 16 * kTc5MaxParts * 128;
constexpr int kTc5PBytes = 2 * 32 * 8 * 2;   // per consumer warp
constexpr int kTc5OffP = kTc5QBytes;
constexpr int kTc5OffMul = kTc5OffP + kConsumerWarps * kTc5PBytes;
constexpr int kTc5OffBar = kTc5OffMul + kTc5Buffers * 16 * 4;
constexpr int kTc5OffSlot = kTc5OffBar + 2 * kTc5Buffers * 8;
constexpr int kTc5Bytes = kTc5OffSlot + 16;
constexpr int kPartBytes = kTileTokens * 128;           // 64 rows x 128 bytes: one swizzled part
constexpr int kMaxStages = 16;
constexpr int kMetaInts = 8;
constexpr int kRowsPerWarp = kTileTokens / kConsumerWarps;   // 8
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kNegInf = -__builtin_huge_valf();

// Sizes that follow from the head dimension D (64, 128 or 256) and the K/V
// element type KV (16-bit, or 8-bit FP8 codes).
template <int D, int KV>
struct Shape {
    static_assert(D == 64 || D == 128 || D == 256, "head_dim 64, 128 or 256");
    static constexpr int kElemBytes = kv_is_fp8(KV) ? 1 : 2;
    static constexpr int kRowBytes = D * kElemBytes;          // one K or V row
    static constexpr int kTileBytes = kTileTokens * kRowBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;        // K tile + V tile
    static constexpr int kParts = kRowBytes / 128;            // 128-byte swizzled parts of a row
    static constexpr int kPartElems = 128 / kElemBytes;       // elements of one part
    static constexpr int kLanesPerRow = D / 8;                // CUDA cores: 8 elements per lane
    static constexpr int kLaneBytes = 8 * kElemBytes;
    static constexpr int kRowsPerStep = 32 / kLanesPerRow;    // rows a warp reads at once
    static constexpr int kKSteps = D / 16;                    // tensor cores: k-steps of q.K^T
    static constexpr int kDimTilesPerWarp = D / 32;           // P.V dim tiles per warp of a pair
};

// Consumer kinds of the split kernel.
enum : int {
    kConsCudaCores = 0,   // CUDA cores, any group
    kConsMma = 1,         // tensor cores: a warp pair shares the columns, splits the dims
    kConsMmaPair = 2,     // tensor cores on two fused kv heads: each warp of a pair takes one
    // two fused kv heads of an FP8 cache: scores by tcgen05 MMAs into TMEM,
    // P.V by warp MMAs; four warps per tile, two tiles in flight
    kConsTc5 = 3
};

// Threads of a split CTA: the consumer warps and one producer warp; four
// producer warps for the cp.async copies (CPA); one more warp issuing the
// score MMAs for the TMEM-score consumers.
__host__ __device__ constexpr int split_threads(int cons, bool cpa)
{
    return cpa ? kSplitThreadsCpAsync : (cons == kConsTc5 ? kSplitThreadsTc5 : kSplitThreads);
}

// Floats of the shared reduction region (partial O, m, and the weight sums)
// for one segment: one state per warp on CUDA cores, one per warp pair (with
// two weight sums) on tensor cores; with paired heads a pair holds both
// heads' columns, d/2 dims each (the TMEM-score consumers: four states of
// both heads' columns, the same size).
__host__ __device__ constexpr int reduction_floats(int cons, int group, int d)
{
    return (cons == kConsMmaPair || cons == kConsTc5) ? kPairs * 2 * group * (d / 2 + 3)
           : cons == kConsMma   ? kPairs * group * (d + 3)
                                : kConsumerWarps * group * (d + 2);
}

// Full-barrier arrivals per tile when the producers use cp.async: one
// (asynchronous) per producer lane, plus the first producer's lane 0 after it
// writes the tile's metadata.
constexpr int kCpAsyncArrivals = 32 * kProducerWarps + 1;

// Per-tile metadata flags, written by the producer into shared memory.
enum : int { kFirstInCta = 1, kLastInCta = 2, kOwnSegment = 4 };

// Query columns of one kv head (group x new tokens): up to two n8 tiles on
// the tensor-core consumers, one on CUDA cores; a launch head of two paired
// kv heads has twice as many column slots.
constexpr int kMaxColumns = 16;
constexpr int kMaxColumnsCudaCores = 8;
constexpr int kMaxColumnSlots = 2 * kMaxColumns;

struct SplitParams {
    const uint16_t *q;            // [B, Hq, D] bf16 or fp16 bits
    const int32_t *seq_lens;      // [B] device, or null (every length = cap)
    const int32_t *block_table;   // [B, max_blocks] (paged only)
    float *o;                     // [B, Hq, D]
    float *lse;                   // [B, Hq] or null
    float *ws_o;                  // [slots, G, D]
    float *ws_lse;                // [slots, G]
    int32_t *ws_prefix;           // [B + 1] tile prefix, then [B + 1] non-empty requests
    unsigned int *ws_err;
    int batch, hq, hkv;
    int cap;                      // largest valid length
    int s_max;                    // contiguous: token rows per request
    int page_size, max_blocks, num_pages;
    float scale_log2;             // scale * log2(e)
    int num_stages;
    uint32_t off_red, off_prefix, off_bar, off_meta, off_misc;
    uint32_t off_tc;              // the TMEM-score instances' region (kTc5Bytes)
    unsigned long long timeout_ns;
    unsigned int flags;
    // Tensor-core path only: 1 when the K/V tensor maps are 4-D views
    // {128-byte part, rows, parts, Hkv} so one box carries every swizzled
    // part of box_rows rows; 0 for 3-D maps with one box per part.
    int box4d;
    int box_rows_log2;   // log2 of the rows in one box: 6 (64) or log2(page size)
    int page_log2;       // paged, page size under 64: log2 of the page size
    // Paged with pages of 1 or 2 tokens (CUDA-core consumers): 1 when the K/V
    // maps are 2-D {head_dim, num_pages * P * Hkv rows} with one-row boxes and
    // a tile's rows are gathered four per load (row of token o of page e for
    // kv head h: (e * P + o) * Hkv + h); 0 for one box per page.
    int gather4;
    // Paged with pages under 8 tokens on the tensor-core consumers (the CPA
    // instances): the pools [num_pages, P, Hkv, D] the producers copy rows from.
    const uint8_t *k_pool, *v_pool;
    // Query columns of a launch head (see col_info): the caller's q is
    // [B, q_len, Hq, dh], and a launch head is fuse_f adjacent kv heads of
    // the caller read as one row of D elements (fused heads, tensor-core path
    // only; fuse_f = 1 otherwise).  Column n is (part, new token i, query
    // head g), given by col_code[n]; a negative code marks a padding column
    // (zero query, never written).  n_cols: the column slots of a head.
    int q_len, g_real, n_cols, fuse_f;
    int fuse_dh;       // dh when a fused row's parts share each column's dims, else 0
    int col_code[kMaxColumnSlots];   // new token i | part << 4 | head g << 8, or -1 (host-computed)
    int q_f16;        // FP8 caches: 1 when q is fp16, 0 when bf16
    float v_scale;    // multiplies O (an FP8 cache's V dequantisation scale; 1 otherwise)
    int prefetch_tiles;   // first tiles of a CTA prefetched into L2 before the dependency wait (0: none)
    int seg_cost;         // the Schedule's cost of a segment start, in tiles
    // A token range (the partial entry points): the layout holds cache
    // positions kv_begin, kv_begin + 1, .. of each request at its rows 0, 1,
    // .., and the call covers positions [kv_begin, min(L_b, kv_end)).
    // range_on = 0: the whole cache, from position 0.
    int range_on, kv_begin, kv_end;
};

struct MergeParams {
    float *o;
    float *lse;
    const float *ws_o;
    const float *ws_lse;
    const int32_t *ws_prefix;
    int batch, hq, hkv, num_ctas;
    int q_len, g_real, n_cols, fuse_f, fuse_dh;   // as in SplitParams
    int col_code[kMaxColumnSlots];
    const int32_t *seq_lens;   // as in SplitParams (small batches: segment geometry)
    int cap;
    int range_on, kv_begin, kv_end;   // as in SplitParams
    // 1: let the next kernel in the stream launch only once this grid's wait
    // has returned (the split grid is complete) rather than at once.
    int late_trigger;
    int seg_cost;      // as in SplitParams
};

constexpr int kMergeDirectBatch = 32;   // batches this small: segment geometry from the lengths
constexpr int kMergeDirectParts = 16;   // segments split this few ways: one load round trip

// Where launch column n of launch head h of request b reads q and writes O:
// part (which fused kv head), new token i (causal limit), the caller's query
// row, and the first of the D dims that belong to it (0 without fusion).
struct ColInfo {
    int i;
    int dim0;
    size_t row;
    bool valid;
};

// The host lays the columns out as (part, new token i, query head g) and
// passes each column's (i, part, g) in col_code, so no division runs here.
template <class P>
__device__ __forceinline__ ColInfo col_info(const P &p, int b, int h, int n)
{
    ColInfo c;
    const int raw = p.col_code[n];
    c.valid = raw >= 0;
    const int code = c.valid ? raw : 0;
    c.i = code & 15;
    const int part = (code >> 4) & 15, g = code >> 8;
    c.row = ((size_t)b * p.q_len + c.i) * p.hq + (size_t)(h * p.fuse_f + part) * p.g_real + g;
    c.dim0 = part * p.fuse_dh;
    return c;
}

// Store output element d (of D) of query row `row`: unfused rows hold D
// values; a fused head's query rows hold only their own fuse_dh dims.
template <int D>
__device__ __forceinline__ void store_o(float *o, size_t row, int d, int fuse_dh, int part, float v)
{
    if (!fuse_dh)
        o[row * D + d] = v;
    else if (d >= part && d < part + fuse_dh)
        o[row * fuse_dh + (d - part)] = v;
}

// Request b's lengths as the kernels use them.  L: its length L_b, from the
// device array (every request at capacity when there is none).  n: the
// tokens of the call's range that the layout holds, min(L_b, kv_end) -
// kv_begin (L_b for a whole-cache call); they sit at layout rows 0 .. n - 1.
// A negative L_b, or an n above the layout's capacity cap, is clamped (to 0,
// to cap) and recorded in *report when it is given.
struct ReqLen {
    int L;   // L_b (whole cache: at most cap)
    int n;   // tokens of the range, 0 .. cap
};

template <class P>
__device__ __forceinline__ ReqLen req_len_of(const P &p, int L, unsigned int *report)
{
    const int off = p.range_on ? p.kv_begin : 0;
    bool bad = L < 0;
    L = max(L, 0);
    int n = p.range_on ? max(min(L, p.kv_end) - off, 0) : L;
    if (n > p.cap) {
        bad = true;
        n = p.cap;
        if (!p.range_on)
            L = p.cap;
    }
    if (bad && report)
        atomicOr(report, kErrLength);
    return ReqLen{L, n};
}

template <class P>
__device__ __forceinline__ ReqLen req_len(const P &p, int b, unsigned int *report)
{
    return req_len_of(p, p.seq_lens ? p.seq_lens[b] : (p.range_on ? p.kv_begin : 0) + p.cap, report);
}

// Every lane waits (so each acquires the barrier's phase); the outcome is
// made warp-uniform so a wait that runs out exactly at the limit cannot split
// the warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          const volatile int *abort_flag)
{
    const bool ok = mbar_wait_bounded(bar, parity, timeout_ns, abort_flag);
    return __all_sync(0xffffffffu, ok);
}

// Barrier among the consumer warps only, on an mbarrier with kConsumerWarps
// arrivals per phase, so that it can give up (bounded) instead of hanging if
// another warp has left.
__device__ __forceinline__ bool consumer_sync(uint32_t cbar, uint32_t &cph, uint64_t timeout_ns,
                                              const volatile int *abort_flag, int lane)
{
    __syncwarp();
    if (lane == 0)
        mbar_arrive(cbar);
    const bool ok = warp_wait(cbar, cph, timeout_ns, abort_flag);
    cph ^= 1u;
    return ok;
}

// prefix[b] = Hkv * (tiles of requests < b), prefix[B] = total tiles, and
// right after it nonempty[b] = prefix[B + 1 + b] = requests < b with at least
// one tile (the Schedule's two arrays).  All NTHREADS threads of the block
// take part.  scan_tmp: 2 * NTHREADS / 32 ints.
// HINT: a plan for L2 prefetches only, made before the kernels ahead in the
// stream have completed: the lengths are read around L1 (no stale line stays
// there), nothing is reported and the workspace is not written.
template <int NTHREADS, bool HINT = false>
__device__ __forceinline__ void build_prefix(const SplitParams &p, int *prefix, int *scan_tmp)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nthreads = NTHREADS, kWarps = nthreads / 32;
    const int B = p.batch;
    int *nonempty = prefix + B + 1;
    const int per = ceil_div(B, nthreads);
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    unsigned int *report = blockIdx.x == 0 && !HINT ? p.ws_err : nullptr;
    auto tiles_of = [&](int b, unsigned int *rep) -> int {
        if constexpr (HINT) {
            const int L = p.seq_lens ? __ldcg(p.seq_lens + b) : (p.range_on ? p.kv_begin : 0) + p.cap;
            return ceil_div(req_len_of(p, L, nullptr).n, kTileTokens);
        } else {
            return ceil_div(req_len(p, b, rep).n, kTileTokens);
        }
    };
    int local = 0, local_ne = 0;
    for (int b = b0; b < b1; ++b) {
        const int n = tiles_of(b, report);
        local += n;
        local_ne += n > 0;
    }
    int x = local, y = local_ne;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int xo = __shfl_up_sync(0xffffffffu, x, off), yo = __shfl_up_sync(0xffffffffu, y, off);
        if (lane >= off) {
            x += xo;
            y += yo;
        }
    }
    if (lane == 31) {
        scan_tmp[warp] = x;
        scan_tmp[kWarps + warp] = y;
    }
    __syncthreads();
    if (warp == 0) {
        int wx = lane < kWarps ? scan_tmp[lane] : 0, wy = lane < kWarps ? scan_tmp[kWarps + lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int xo = __shfl_up_sync(0xffffffffu, wx, off), yo = __shfl_up_sync(0xffffffffu, wy, off);
            if (lane >= off) {
                wx += xo;
                wy += yo;
            }
        }
        if (lane < kWarps) {
            scan_tmp[lane] = wx;
            scan_tmp[kWarps + lane] = wy;
        }
    }
    __syncthreads();
    int run = x - local + (warp > 0 ? scan_tmp[warp - 1] : 0);
    int run_ne = y - local_ne + (warp > 0 ? scan_tmp[kWarps + warp - 1] : 0);
    for (int b = b0; b < b1; ++b) {
        prefix[b] = run * p.hkv;
        nonempty[b] = run_ne;
        const int n = tiles_of(b, nullptr);
        run += n;
        run_ne += n > 0;
    }
    if (tid == nthreads - 1) {
        prefix[B] = run * p.hkv;
        nonempty[B] = run_ne;
    }
    __syncthreads();
    if (blockIdx.x == 0 && !HINT)
        for (int b = tid; b <= 2 * B + 1; b += nthreads)
            p.ws_prefix[b] = prefix[b];
}

// ------------------------------------------------------------------ producer

// Byte address of 16-byte chunk `chunk` (0 .. row bytes / 16 - 1) of `row`
// in a swizzled tile made of boxes of 2^rl rows, each box laid out
// [128-byte part][row][128 B].  With rl = 6 (one 64-row box per part) the
// tile is PARTS parts of 8 KB.
template <int PARTS>
__device__ __forceinline__ uint32_t sw128_addr(uint32_t tile, int row, int chunk, int rl)
{
    const int rb = row >> rl, rr = row & ((1 << rl) - 1);
    return tile + ((((rb * PARTS) + (chunk >> 3)) << rl) + rr) * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

template <bool PAGED, bool SW128, int D, int KV>
__device__ __forceinline__ void split_producer(const SplitParams &p, const CUtensorMap *tmk,
                                               const CUtensorMap *tmv, uint32_t stage0,
                                               const int *prefix, int *meta, uint32_t full0,
                                               uint32_t empty0, volatile int *abort_flag,
                                               int t_begin, int t_end, int lane)
{
    // The whole warp walks the tiles; lane 0 arms the barriers and the TMA
    // loads of a tile are spread over lanes (one box per lane, or one page
    // per lane for small pages) so they issue together.
    if (lane == 0) {
        tma_prefetch_desc(tmk);
        tma_prefetch_desc(tmv);
    }
    const uint64_t policy = l2_policy_evict_first();
    const int NS = p.num_stages;
    const bool starve = (p.flags & 1u) && blockIdx.x == 0;
    using HD = Shape<D, KV>;
    // Boxes per (tile or page): K and V, each whole (plain or 4-D swizzled)
    // or as one box per 128-byte swizzled part.
    const int box_log2 = (SW128 && !p.box4d) ? 1 + (HD::kParts == 4 ? 2 : HD::kParts - 1) : 1;
    const int kBoxes = 1 << box_log2;
    const int page_log2 = p.page_log2;   // pages under 64 tokens are powers of two

    int t = t_begin;
    int b = request_of_tile(prefix, p.batch, t);
    int nb = (prefix[b + 1] - prefix[b]) / p.hkv;
    int h = (t - prefix[b]) / nb;
    int j = (t - prefix[b]) - h * nb;
    // L: the request's tokens in the layout; Lc: its length counted from the
    // layout's row 0 (the causal limits of several new tokens)
    const int off = p.range_on ? p.kv_begin : 0;
    ReqLen rq = req_len(p, b, nullptr);
    int L = rq.n, Lc = rq.L - off;

    // Paged: block-table entries in a ring of four 32-entry windows (one
    // entry per lane per window).  The current window is e0; e1..e3 are the
    // next three, loaded ahead so table reads stay far off the issue path.
    int win_b = -1, win_base = 0;
    int e0 = 0, e1 = 0, e2 = 0, e3 = 0;
    auto table_load = [&](int bb, int idx) -> int {
        return idx < p.max_blocks ? __ldg(p.block_table + (size_t)bb * p.max_blocks + idx) : 0;
    };
    // Warp-collective: make the current window hold page index pg.
    auto ensure_window = [&](int pg) {
        if (b != win_b || pg < win_base || pg >= win_base + 128) {
            win_b = b;
            win_base = pg & ~31;
            e0 = table_load(b, win_base + lane);
            e1 = table_load(b, win_base + 32 + lane);
            e2 = table_load(b, win_base + 64 + lane);
            e3 = table_load(b, win_base + 96 + lane);
        }
        while (pg >= win_base + 32) {   // advance one window, prefetch the fourth ahead
            e0 = e1;
            e1 = e2;
            e2 = e3;
            win_base += 32;
            e3 = table_load(b, win_base + 96 + lane);
        }
    };
    // Warp-collective: entry of page pg_lane (each lane its own, inside the window).
    auto window_entry = [&](int pg_lane) -> int {
        int e = __shfl_sync(0xffffffffu, e0, (pg_lane - win_base) & 31);
        if (e < 0 || e >= p.num_pages) {
            atomicOr(p.ws_err, kErrPage);
            e = 0;
        }
        return e;
    };
    // Warp-collective: entry of page pg_lane anywhere in the window's 128
    // entries (each lane its own).
    auto window_entry_any = [&](int pg_lane) -> int {
        const int idx = pg_lane - win_base;
        const int src = idx & 31;
        const int a = __shfl_sync(0xffffffffu, e0, src), bq = __shfl_sync(0xffffffffu, e1, src);
        const int c = __shfl_sync(0xffffffffu, e2, src), d = __shfl_sync(0xffffffffu, e3, src);
        int e = idx < 32 ? a : (idx < 64 ? bq : (idx < 96 ? c : d));
        if (idx < 0 || idx >= 128 || e < 0 || e >= p.num_pages) {
            atomicOr(p.ws_err, kErrPage);
            e = 0;
        }
        return e;
    };
    // Box `box` (0..kBoxes-1) of the tile's K/V for the rows starting at tile
    // row r0 (a page's first row, or 0).
    auto load_box = [&](int box, uint32_t kdst, uint32_t vdst, uint32_t full, int r0, int row) {
        if (SW128 && p.box4d) {   // box 0: K, box 1: V; all parts in one box
            tma_load_4d(((box & 1) ? vdst : kdst) + r0 * HD::kRowBytes, (box & 1) ? tmv : tmk, full, 0, row,
                        0, h, policy);
        } else if constexpr (SW128) {   // one box per 128-byte part
            const int part = box & (HD::kParts - 1);
            const bool is_v = box >= HD::kParts;
            const uint32_t dst = (is_v ? vdst : kdst) + part * kPartBytes + r0 * 128;
            tma_load_3d(dst, is_v ? tmv : tmk, full, part * HD::kPartElems, h, row, policy);
        } else {
            const uint32_t dst = ((box & 1) ? vdst : kdst) + r0 * HD::kRowBytes;
            tma_load_3d(dst, (box & 1) ? tmv : tmk, full, 0, h, row, policy);
        }
    };

    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    for (; t < t_end; ++t) {
        if (!warp_wait(empty0 + 8 * s, ph ^ 1u, p.timeout_ns, abort_flag)) {
            if (lane == 0) {
                atomicOr(p.ws_err, kErrTimeout);
                *abort_flag = 1;
            }
            break;
        }
        const int seg_first = prefix[b] + h * nb;
        const int token0 = j * kTileTokens;
        const int nvalid = min(kTileTokens, L - token0);
        int flags = 0;
        if (j == 0 || t == t_begin)
            flags |= kFirstInCta;
        if (j == nb - 1 || t == t_end - 1)
            flags |= kLastInCta;
        if (seg_first >= t_begin && seg_first + nb <= t_end)
            flags |= kOwnSegment;

        const uint32_t full = full0 + 8 * s;
        const uint32_t kdst = stage0 + s * HD::kStageBytes;
        const uint32_t vdst = kdst + HD::kTileBytes;
        const uint32_t extra = (starve && issued == 0) ? 256u : 0u;
        const int P = p.page_size;
        const bool small_pages = PAGED && P < kTileTokens;
        const bool gather = !SW128 && PAGED && p.gather4 != 0;
        // pages of this tile that hold valid tokens (paged, P < 64)
        const int need = small_pages ? min(kTileTokens >> page_log2, (nvalid + P - 1) >> page_log2) : 1;
        if (lane == 0) {
            int *m = meta + s * kMetaInts;
            m[0] = b;
            m[1] = h;
            m[2] = Lc - token0;   // tokens of the request from this tile on (causal limits)
            m[3] = nvalid;
            m[4] = flags;
            m[5] = b * p.hkv + h;
            const uint32_t bytes = gather ? 2u * (uint32_t)(((nvalid + 3) >> 2) * 4 * HD::kRowBytes)
                                   : small_pages ? 2u * need * P * HD::kRowBytes
                                                 : (uint32_t)(2 * HD::kTileBytes);
            mbar_arrive_expect_tx(full, bytes + extra);
        }
        __syncwarp();
        if constexpr (!PAGED) {
            if (lane < kBoxes)
                load_box(lane, kdst, vdst, full, 0, b * p.s_max + token0);
        } else if (P >= kTileTokens) {
            ensure_window(token0 / P);
            const int phys = window_entry(token0 / P);
            if (lane < kBoxes)
                load_box(lane, kdst, vdst, full, 0, phys * P + (token0 % P));
        } else if (gather) {
            if constexpr (!SW128) {
                // Four rows per load: lane l < 16 gathers K rows 4l .. 4l + 3 of
                // the tile, lane 16 + l the same V rows.  Rows past the request's
                // end repeat its last token (never read by the consumers).  The
                // tile's pages (at most 64) lie in the window's 128 entries.
                ensure_window(token0 >> page_log2);
                const int grp = lane & 15;
                int rowc[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int tok = token0 + min(4 * grp + k, nvalid - 1);
                    const int e = window_entry_any(tok >> page_log2);
                    rowc[k] = (e * P + (tok & (P - 1))) * p.hkv + h;
                }
                if (grp < ((nvalid + 3) >> 2))
                    tma_gather4_2d((lane < 16 ? kdst : vdst) + 4 * grp * HD::kRowBytes, lane < 16 ? tmk : tmv,
                                   full, 0, rowc[0], rowc[1], rowc[2], rowc[3], policy);
            }
        } else {
            // One (page, box) pair per lane, so a tile's boxes issue together.
            const int pg0 = token0 >> page_log2;
            const int items = need << box_log2;
            for (int i0 = 0; i0 < items; i0 += 32) {
                ensure_window(pg0 + (i0 >> box_log2));
                const int item = i0 + lane;
                const int k = item >> box_log2;
                const int phys = window_entry(pg0 + (item < items ? k : (i0 >> box_log2)));
                if (item < items)
                    load_box(item & (kBoxes - 1), kdst, vdst, full, k * P, phys * P);
            }
        }
        __syncwarp();
        ++issued;
        if (++s == NS) {
            s = 0;
            ph ^= 1u;
        }
        if (t + 1 < t_end && ++j == nb) {
            j = 0;
            if (++h == p.hkv) {
                h = 0;
                do {
                    ++b;
                } while (b < p.batch && prefix[b + 1] == prefix[b]);
                nb = (prefix[b + 1] - prefix[b]) / p.hkv;
                rq = req_len(p, b, nullptr);
                L = rq.n;
                Lc = rq.L - off;
            }
        }
    }
    // Before leaving, wait (bounded) for every load still in flight so no
    // asynchronous copy outlives the CTA's shared memory.
    if (lane == 0) {
        for (int k = issued > NS ? issued - NS : 0; k < issued; ++k)
            mbar_wait_bounded(full0 + 8 * (k % NS), (uint32_t)((k / NS) & 1), p.timeout_ns, nullptr);
    }
}

// L2 prefetch of tiles [t_begin, t_end) of this CTA, issued by the producer
// warp before the kernel waits for the kernels ahead of it in the stream:
// the same boxes split_producer loads, one (tile, page, box) item per lane.
// The plan (prefix) and the block-table entries are read before that wait
// and may be stale; a prefetch only fills L2, which is where device memory
// is kept coherent, so a stale plan wastes bandwidth and never changes a
// result.  Table entries are read around L1 and entries outside the pool are
// skipped.  Pages of 1 or 2 tokens gathered row by row are not prefetched.
template <bool PAGED, bool SW128, int D, int KV>
__device__ __forceinline__ void split_prefetch(const SplitParams &p, const CUtensorMap *tmk,
                                               const CUtensorMap *tmv, const int *prefix, int t_begin,
                                               int t_end, int lane)
{
    using HD = Shape<D, KV>;
    if (PAGED && p.gather4)
        return;
    const int box_log2 = (SW128 && !p.box4d) ? 1 + (HD::kParts == 4 ? 2 : HD::kParts - 1) : 1;
    const int P = p.page_size;
    const bool small_pages = PAGED && P < kTileTokens;
    const int pages_log2 = small_pages ? 6 - p.page_log2 : 0;   // pages per tile (log2)
    const int per_tile_log2 = pages_log2 + box_log2;
    const int items = (t_end - t_begin) << per_tile_log2;
    for (int i = lane; i < items; i += 32) {
        const int t = t_begin + (i >> per_tile_log2);
        const int box = i & ((1 << box_log2) - 1), pg = (i >> box_log2) & ((1 << pages_log2) - 1);
        const int b = request_of_tile(prefix, p.batch, t);
        const int nb = (prefix[b + 1] - prefix[b]) / p.hkv;
        const int h = (t - prefix[b]) / nb, j = (t - prefix[b]) - h * nb;
        const int token0 = j * kTileTokens;
        int row;
        if constexpr (PAGED) {
            const int tok = token0 + (pg << p.page_log2);
            const int idx = small_pages ? tok >> p.page_log2 : tok / P;
            if (idx >= p.max_blocks)
                continue;
            const int e = __ldcg(p.block_table + (size_t)b * p.max_blocks + idx);
            if (e < 0 || e >= p.num_pages)
                continue;
            row = e * P + (small_pages ? 0 : token0 % P);
        } else {
            row = b * p.s_max + token0;
        }
        const bool is_v = SW128 && !p.box4d ? box >= HD::kParts : (box & 1) != 0;
        const CUtensorMap *map = is_v ? tmv : tmk;
        if (SW128 && p.box4d)
            tma_prefetch_4d(map, 0, row, 0, h);
        else if (SW128)
            tma_prefetch_3d(map, (box & (HD::kParts - 1)) * HD::kPartElems, h, row);
        else
            tma_prefetch_3d(map, 0, h, row);
    }
}

// Producer for pages under 8 tokens on the tensor-core consumers: no TMA.
// All kProducerWarps warps walk the CTA's tiles in the order split_producer
// does; warp pw copies tile rows 16 pw .. 16 pw + 15 that hold valid tokens
// with per-thread 16-byte cp.async, straight into the 128-byte swizzled
// layout the consumers read (TMA page boxes of fewer than 8 rows cannot land
// on the swizzle's 1 KB boundaries).  For each row, lanes 0-15 copy its K
// chunks and lanes 16-31 its V chunks.  The full barrier of a stage expects
// kCpAsyncArrivals arrivals: one per producer lane once its copies have
// landed, and warp 0's lane 0 after it writes the tile's metadata.
template <int D, int KV>
__device__ __forceinline__ void split_producer_cpa(const SplitParams &p, uint32_t stage0, const int *prefix,
                                                   int *meta, uint32_t full0, uint32_t empty0,
                                                   volatile int *abort_flag, int t_begin, int t_end, int lane,
                                                   int pw)
{
    using HD = Shape<D, KV>;
    constexpr int kChunks = HD::kRowBytes / 16;
    constexpr int kRowsPerProducer = kTileTokens / kProducerWarps;   // 16
    const uint64_t policy = l2_policy_evict_first();
    const int NS = p.num_stages;
    const int P = p.page_size, page_log2 = p.page_log2;   // P = 1, 2 or 4
    const bool lead = pw == 0 && lane == 0;
    const bool starve = (p.flags & 1u) && blockIdx.x == 0;   // test hook: the first tile never completes
    const int r_begin = pw * kRowsPerProducer;

    int t = t_begin;
    int b = request_of_tile(prefix, p.batch, t);
    int nb = (prefix[b + 1] - prefix[b]) / p.hkv;
    int h = (t - prefix[b]) / nb;
    int j = (t - prefix[b]) - h * nb;
    // L: the request's tokens in the layout; Lc: its length counted from the
    // layout's row 0 (the causal limits of several new tokens)
    const int off = p.range_on ? p.kv_begin : 0;
    ReqLen rq = req_len(p, b, nullptr);
    int L = rq.n, Lc = rq.L - off;

    // Block-table entries of request b, pages win_base .. win_base + 127: lane
    // l holds entry win_base + l + 32 k in e[k].  The window advances 32
    // entries at a time and loads the fourth block ahead, so a tile's (at most
    // 64) pages, which start in block 0, are read from blocks 0-2 only.
    int win_b = -1, win_base = 0;
    int e[4] = {0, 0, 0, 0};
    auto table_load = [&](int idx) -> int {
        return idx < p.max_blocks ? __ldg(p.block_table + (size_t)b * p.max_blocks + idx) : 0;
    };

    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    for (; t < t_end; ++t) {
        if (!warp_wait(empty0 + 8 * s, ph ^ 1u, p.timeout_ns, abort_flag)) {
            if (lead) {
                atomicOr(p.ws_err, kErrTimeout);
                *abort_flag = 1;
            }
            break;
        }
        const int seg_first = prefix[b] + h * nb;
        const int token0 = j * kTileTokens;
        const int nvalid = min(kTileTokens, L - token0);
        const uint32_t full = full0 + 8 * s;
        const uint32_t kdst = stage0 + s * HD::kStageBytes;
        const uint32_t vdst = kdst + HD::kTileBytes;
        if (lead) {
            int flags = 0;
            if (j == 0 || t == t_begin)
                flags |= kFirstInCta;
            if (j == nb - 1 || t == t_end - 1)
                flags |= kLastInCta;
            if (seg_first >= t_begin && seg_first + nb <= t_end)
                flags |= kOwnSegment;
            int *m = meta + s * kMetaInts;
            m[0] = b;
            m[1] = h;
            m[2] = Lc - token0;
            m[3] = nvalid;
            m[4] = flags;
            m[5] = b * p.hkv + h;
            if (!(starve && issued == 0))
                mbar_arrive(full);
        }

        const int pg0 = token0 >> page_log2;
        if (b != win_b || pg0 < win_base || pg0 >= win_base + 128) {
            win_b = b;
            win_base = pg0 & ~31;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                e[k] = table_load(win_base + 32 * k + lane);
        }
        while (pg0 >= win_base + 32) {
            e[0] = e[1];
            e[1] = e[2];
            e[2] = e[3];
            win_base += 32;
            e[3] = table_load(win_base + 96 + lane);
        }
        // lane l: the pool row of tile row r_begin + (l & 15) (rows past the
        // request's end stand in for its last row; never copied)
        uint32_t prow;
        {
            const int tok = token0 + min(r_begin + (lane & 15), nvalid - 1);
            const int idx = (tok >> page_log2) - win_base;   // 0 .. 94
            const int src = idx & 31;
            const int x0 = __shfl_sync(0xffffffffu, e[0], src), x1 = __shfl_sync(0xffffffffu, e[1], src);
            const int x2 = __shfl_sync(0xffffffffu, e[2], src);
            int pe = idx < 32 ? x0 : (idx < 64 ? x1 : x2);
            if (idx < 0 || idx >= 96 || pe < 0 || pe >= p.num_pages) {
                atomicOr(p.ws_err, kErrPage);
                pe = 0;
            }
            prow = (uint32_t)(((size_t)pe * P + (tok & (P - 1))) * p.hkv + h);   // < 2^32: checked on the host
        }
        const uint8_t *pool = lane < 16 ? p.k_pool : p.v_pool;
        const uint32_t dst0 = lane < 16 ? kdst : vdst;
        const int r_end = min(nvalid, r_begin + kRowsPerProducer);
#pragma unroll 8
        for (int r = r_begin; r < r_end; ++r) {
            const uint32_t row = __shfl_sync(0xffffffffu, prow, r - r_begin);
            const uint8_t *src = pool + (size_t)row * HD::kRowBytes;
#pragma unroll
            for (int c = lane & 15; c < kChunks; c += 16)
                cp_async_16(sw128_addr<HD::kParts>(dst0, r, c, 6), src + c * 16, policy);
        }
        cp_async_mbar_arrive_noinc(full);

        ++issued;
        if (++s == NS) {
            s = 0;
            ph ^= 1u;
        }
        if (t + 1 < t_end && ++j == nb) {
            j = 0;
            if (++h == p.hkv) {
                h = 0;
                do {
                    ++b;
                } while (b < p.batch && prefix[b + 1] == prefix[b]);
                nb = (prefix[b + 1] - prefix[b]) / p.hkv;
                rq = req_len(p, b, nullptr);
                L = rq.n;
                Lc = rq.L - off;
            }
        }
    }
    // Before leaving: this lane's own copies, then (bounded) every stage still
    // in flight, so no copy outlives the CTA's shared memory.
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (lead) {
        for (int k = issued > NS ? issued - NS : 0; k < issued; ++k)
            mbar_wait_bounded(full0 + 8 * (k % NS), (uint32_t)((k / NS) & 1), p.timeout_ns, nullptr);
    }
}

// ------------------------------------------------------------------ consumer

// Combine NSTATE partial softmax states (m, l, acc[G][D]) published in shared
// memory and write the segment's result: final O/LSE when the CTA saw the
// whole segment, otherwise a normalised partial and its LSE.  O is divided by
// the sum of the weights that multiplied V (red_l); the LSE uses the sum of
// the exact fp32 weights (red_lt), which differs only when P was rounded to a
// 16-bit type for the tensor-core product.
template <int G, int NSTATE, int D>
__device__ __forceinline__ void combine_and_write(const SplitParams &p, const float *red_acc,
                                                  const float *red_m, const float *red_l,
                                                  const float *red_lt, int ctid, int b, int h, int u,
                                                  bool own)
{
    const int slot = u + (int)blockIdx.x;
    for (int idx = ctid; idx < G * D; idx += kConsumerThreads) {
        const int g = idx / D, d = idx % D;
        if (p.col_code[g] < 0)
            continue;   // padding column
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < NSTATE; ++w)
            M = fmaxf(M, red_m[w * G + g]);
        float lsum = 0.f, ltrue = 0.f, o = 0.f;
#pragma unroll
        for (int w = 0; w < NSTATE; ++w) {
            const float mw = red_m[w * G + g];
            const float wt = (mw == kNegInf) ? 0.f : exp2_approx(mw - M);
            lsum += wt * red_l[w * G + g];
            ltrue += wt * red_lt[w * G + g];
            o += wt * red_acc[(w * G + g) * D + d];
        }
        const float out = lsum > 0.f ? (o / lsum) * p.v_scale : 0.f;
        const float lse_v = ltrue > 0.f ? (M + log2f(ltrue)) * kLn2 : kNegInf;
        if (own) {
            const ColInfo c = col_info(p, b, h, g);
            store_o<D>(p.o, c.row, d, p.fuse_dh, c.dim0, out);
            if (d == 0 && p.lse)
                p.lse[c.row] = lse_v;
        } else {
            p.ws_o[((size_t)slot * G + g) * D + d] = out;
            if (d == 0)
                p.ws_lse[(size_t)slot * G + g] = lse_v;
        }
    }
}

// Eight consecutive K or V elements of a shared-memory row, widened to fp32:
// one 16-byte load of 16-bit values, or one 8-byte load of FP8 codes.
template <int KV>
__device__ __forceinline__ void load_row8(uint32_t addr, float2 (&x)[4])
{
    if constexpr (kv_is_fp8(KV)) {
        const uint2 w = lds64(addr);
        x[0] = fp8x2_to_float2<KV>(lo16(w.x));
        x[1] = fp8x2_to_float2<KV>(hi16(w.x));
        x[2] = fp8x2_to_float2<KV>(lo16(w.y));
        x[3] = fp8x2_to_float2<KV>(hi16(w.y));
    } else {
        const uint4 w = lds128(addr);
        x[0] = x2_to_float2<KV == kKvF16>(w.x);
        x[1] = x2_to_float2<KV == kKvF16>(w.y);
        x[2] = x2_to_float2<KV == kKvF16>(w.z);
        x[3] = x2_to_float2<KV == kKvF16>(w.w);
    }
}

// The query's element type: that of a 16-bit cache, chosen at run time for
// an FP8 cache.
template <int KV>
__device__ __forceinline__ bool q_is_f16(const SplitParams &p)
{
    if constexpr (kv_is_fp8(KV))
        return p.q_f16 != 0;
    else
        return KV == kKvF16;
}

template <int G, int KV, int D>
__device__ __forceinline__ void split_consumer(const SplitParams &p, uint8_t *smem, uint32_t stage0,
                                               const int *meta, uint32_t full0, uint32_t empty0,
                                               uint32_t cbar, volatile int *abort_flag, int t_begin,
                                               int t_end, int cw, int lane)
{
    using HD = Shape<D, KV>;
    constexpr int LPR = HD::kLanesPerRow, RPS = HD::kRowsPerStep;
    // Eight columns split the warps in two halves (warps 0-3 take columns 0-3,
    // warps 4-7 columns 4-7), each half covering every row of the tile, 16 per
    // warp: a thread then holds the q, O and softmax state of 4 columns, as
    // for G = 4, where 8 columns would spill.  Each K/V row is read from
    // shared memory by two warps.
    constexpr int CS = G == 8 ? 2 : 1;            // column sets
    constexpr int GW = G / CS;                    // columns of this warp
    constexpr int WR = kConsumerWarps / CS;       // warps over the rows of a tile (states per column)
    constexpr int RPW = kTileTokens / WR;         // rows of this warp
    constexpr int RPG = RPW / RPS;                // row steps of this warp
    const int cbase = (cw / WR) * GW;             // first column of this warp
    const int row0 = (cw % WR) * RPW;             // first row of this warp
    const int slot = cw % WR;                     // its state slot in the reduction
    const int NS = p.num_stages;
    const bool qf16 = q_is_f16<KV>(p);
    const int sub = lane / LPR, li = lane % LPR;   // row slot within a warp step, lane within the row
    float *red_acc = reinterpret_cast<float *>(smem + p.off_red);   // [warps][G][D]
    float *red_m = red_acc + kConsumerWarps * G * D;                 // [warps][G]
    float *red_l = red_m + kConsumerWarps * G;                       // [warps][G]
    const int ctid = cw * 32 + lane;
    // rows per online update (fewer live scores for large G)
    constexpr int kSub0 = GW >= 8 ? 1 : (GW >= 4 ? 2 : RPG);
    constexpr int kSub = kSub0 < RPG ? kSub0 : RPG;
    // causal lag of each column: new token i sees q_len - 1 - i fewer tokens
    int lag[GW];
#pragma unroll
    for (int g = 0; g < GW; ++g)
        lag[g] = p.q_len - 1 - col_info(p, 0, 0, cbase + g).i;

    float2 qf[GW][4];
    float2 acc[GW][4];
    float m[GW], l[GW];
#pragma unroll
    for (int g = 0; g < GW; ++g) {
        m[g] = kNegInf;
        l[g] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            acc[g][c] = make_float2(0.f, 0.f);
            qf[g][c] = make_float2(0.f, 0.f);
        }
    }

    int s = 0;
    uint32_t ph = 0, cph = 0;
    auto give_up = [&]() {
        if (lane == 0) {
            atomicOr(p.ws_err, kErrTimeout);
            *abort_flag = 1;
        }
    };
    for (int t = t_begin; t < t_end; ++t) {
        if (!warp_wait(full0 + 8 * s, ph, p.timeout_ns, abort_flag)) {
            if (lane == 0) {
                atomicOr(p.ws_err, kErrTimeout);
                *abort_flag = 1;
            }
            return;
        }
        const int *mt = meta + s * kMetaInts;
        const int b = mt[0], h = mt[1], rem = mt[2], nvalid = mt[3], flags = mt[4], u = mt[5];

        if (flags & kFirstInCta) {
            const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
            for (int g = 0; g < GW; ++g) {
                const ColInfo c = col_info(p, b, h, cbase + g);
                uint4 raw = make_uint4(0u, 0u, 0u, 0u);
                if (c.valid)
                    raw = ldg128_nc(p.q + c.row * D + li * 8);
                const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    qf[g][c] = mul2(qf16 ? f16x2_to_float2(rw[c]) : bf16x2_to_float2(rw[c]), c2);
            }
        }

        const uint32_t kbase = stage0 + s * HD::kStageBytes + li * HD::kLaneBytes;
        const uint32_t vbase = kbase + HD::kTileBytes;

        // Rows of this lane group, kSub at a time.
#pragma unroll
        for (int r0 = 0; r0 < RPG; r0 += kSub) {
            // Scores (log2 units).
            float sc[kSub][GW];
#pragma unroll
            for (int r = 0; r < kSub; ++r) {
                const int row = row0 + RPS * (r0 + r) + sub;
                float2 kx[4];
                load_row8<KV>(kbase + row * HD::kRowBytes, kx);
#pragma unroll
                for (int g = 0; g < GW; ++g) {
                    float2 a = mul2(qf[g][0], kx[0]);
                    a = fma2(qf[g][1], kx[1], a);
                    a = fma2(qf[g][2], kx[2], a);
                    a = fma2(qf[g][3], kx[3], a);
                    sc[r][g] = a.x + a.y;
                }
            }
#pragma unroll
            for (int r = 0; r < kSub; ++r)
#pragma unroll
                for (int g = 0; g < GW; ++g) {
                    float x = sc[r][g];
#pragma unroll
                    for (int off = LPR / 2; off; off >>= 1)
                        x += __shfl_xor_sync(0xffffffffu, x, off);
                    sc[r][g] = x;
                }

            // Online softmax update (rows past the column's causal end, or past
            // the request's end, carry no weight).
            float pr[kSub][GW];
#pragma unroll
            for (int g = 0; g < GW; ++g) {
                const int lim = min(nvalid, rem - lag[g]);   // the column's causal end in this tile
                float tile_max = kNegInf;
#pragma unroll
                for (int r = 0; r < kSub; ++r) {
                    const int row = row0 + RPS * (r0 + r) + sub;
                    if (row < lim)
                        tile_max = fmaxf(tile_max, sc[r][g]);
                }
                const float m_new = fmaxf(m[g], tile_max);
                const float alpha = (m[g] == kNegInf) ? 0.f : exp2_approx(m[g] - m_new);
                float psum = 0.f;
#pragma unroll
                for (int r = 0; r < kSub; ++r) {
                    const int row = row0 + RPS * (r0 + r) + sub;
                    pr[r][g] = (row < lim) ? exp2_approx(sc[r][g] - m_new) : 0.f;
                    psum += pr[r][g];
                }
                l[g] = l[g] * alpha + psum;
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    acc[g][c] = mul2(acc[g][c], a2);
                m[g] = m_new;
            }

            // acc += p * V
#pragma unroll
            for (int r = 0; r < kSub; ++r) {
                const int row = row0 + RPS * (r0 + r) + sub;
                if (row < nvalid) {
                    float2 vx[4];
                    load_row8<KV>(vbase + row * HD::kRowBytes, vx);
#pragma unroll
                    for (int g = 0; g < GW; ++g) {
                        const float2 p2 = make_float2(pr[r][g], pr[r][g]);
                        acc[g][0] = fma2(p2, vx[0], acc[g][0]);
                        acc[g][1] = fma2(p2, vx[1], acc[g][1]);
                        acc[g][2] = fma2(p2, vx[2], acc[g][2]);
                        acc[g][3] = fma2(p2, vx[3], acc[g][3]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty0 + 8 * s);

        if (flags & kLastInCta) {
            // 1. merge the states of the warp's lane groups (rows of one step)
#pragma unroll
            for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
                for (int g = 0; g < GW; ++g) {
                    const float mo = __shfl_xor_sync(0xffffffffu, m[g], off);
                    const float lo = __shfl_xor_sync(0xffffffffu, l[g], off);
                    const float mn = fmaxf(m[g], mo);
                    const float a_self = (m[g] == kNegInf) ? 0.f : exp2_approx(m[g] - mn);
                    const float a_other = (mo == kNegInf) ? 0.f : exp2_approx(mo - mn);
                    l[g] = l[g] * a_self + lo * a_other;
                    const float2 s2 = make_float2(a_self, a_self), o2 = make_float2(a_other, a_other);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float2 other;
                        other.x = __shfl_xor_sync(0xffffffffu, acc[g][c].x, off);
                        other.y = __shfl_xor_sync(0xffffffffu, acc[g][c].y, off);
                        acc[g][c] = fma2(acc[g][c], s2, mul2(other, o2));
                    }
                    m[g] = mn;
                }
            }
            // 2. publish the warp state (its columns, in its slot)
            if (sub == 0) {
#pragma unroll
                for (int g = 0; g < GW; ++g) {
                    float4 *dst = reinterpret_cast<float4 *>(red_acc + (slot * G + cbase + g) * D + li * 8);
                    dst[0] = make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
                    dst[1] = make_float4(acc[g][2].x, acc[g][2].y, acc[g][3].x, acc[g][3].y);
                }
            }
            if (lane == 0) {
#pragma unroll
                for (int g = 0; g < GW; ++g) {
                    red_m[slot * G + cbase + g] = m[g];
                    red_l[slot * G + cbase + g] = l[g];
                }
            }
            if (!consumer_sync(cbar, cph, p.timeout_ns, abort_flag, lane)) {
                give_up();
                return;
            }
            // 3. combine the warps and write the segment's result
            combine_and_write<G, WR, D>(p, red_acc, red_m, red_l, red_l, ctid, b, h, u,
                                        (flags & kOwnSegment) != 0);
            if (!consumer_sync(cbar, cph, p.timeout_ns, abort_flag, lane)) {
                give_up();
                return;
            }
            // 4. fresh state for the next segment
#pragma unroll
            for (int g = 0; g < GW; ++g) {
                m[g] = kNegInf;
                l[g] = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    acc[g][c] = make_float2(0.f, 0.f);
            }
        }
        if (++s == NS) {
            s = 0;
            ph ^= 1u;
        }
    }
}


// ------------------------------------------------------------------ tensor-core consumer
//
// GQA groups (and several new tokens) make q.K^T a small dense contraction:
// for a 16-token slice of a tile, S^T[16 x 8] = K[16 x D] . Q^T[D x 8] with the
// kv head's query columns as the 8 columns (padded with zero columns), and
// O^T[D x 8] += V^T[D x 16] . P^T[16 x 8].  Both are warp-level m16n8k16 MMAs
// (bf16, or fp16 for fp16 and FP8 caches) with fp32 accumulation.  The tile
// arrives with the 128-byte TMA swizzle, so the ldmatrix row reads are free
// of bank conflicts.  For the second product P is taken as a rounded part
// plus its rounded remainder, both of the MMA type (two MMAs), and the
// running sum l adds up exactly the weights that multiply V (a second sum of
// the exact weights gives the LSE).
//
// Warps 2i and 2i+1 take tokens 16i..16i+15 of every tile.  Sharing the
// columns, both form the scores (so each holds the softmax state), and for
// P.V warp 2i covers the first half of the row's dims and warp 2i+1 the
// second.  On two paired kv heads, warp 2i + j owns head j outright: its
// columns, its half of the row for q.K^T and for P.V.


// FP8 caches on the tensor cores.  K and V stay FP8 codes in shared memory
// and are converted to fp16 pairs in registers (exactly), so the products run
// as fp16 MMAs:
//   * K: an ldmatrix of b16 units over a 16-byte chunk gives each lane four
//     consecutive codes, dims 4 qd .. 4 qd + 3 of the chunk.  The MMA's k
//     order is free as long as A and B agree, so k-step positions 2 qd, 2qd+1
//     take dims 4 qd, 4 qd + 1 and positions 2 qd + 8, + 9 take 4 qd + 2, + 3;
//     the query's B fragment is loaded in the same order.
//   * V^T: an ldmatrix.trans of b16 units gives each lane, for tokens 2 qd
//     and 2 qd + 1, the codes of dims 2 grp and 2 grp + 1; one byte permute
//     pairs the two tokens per dim.  So output row grp of a 16-dim tile is dim
//     2 grp and row grp + 8 is dim 2 grp + 1.
//   * q: fp16 has a narrower range than bf16, so each query head is scaled by
//     a power of two that puts its largest |element| in [2^14, 2^15) before
//     the conversion (exact for every element that stays an fp16 normal), and
//     the score is multiplied back by the same power of two.

template <int G, int KV, int D, bool PAIR>
__device__ __forceinline__ void split_consumer_mma(const SplitParams &p, uint8_t *smem, uint32_t stage0,
                                                   const int *meta, uint32_t full0, uint32_t empty0,
                                                   uint32_t cbar, volatile int *abort_flag, int t_begin,
                                                   int t_end, int cw, int lane)
{
    static_assert(G >= 1 && G <= 16, "one or two n8 tiles of query columns");
    using HD = Shape<D, KV>;
    // How the two warps of a pair (the same 16 tokens) share the work:
    //   PAIR:   the row holds two kv heads of D/2 dims; warp dhalf owns head
    //           dhalf entirely (its G columns, its D/2 dims for q.K^T and P.V);
    //   CSPLIT: over 8 columns of one head; warp dhalf owns columns
    //           8 dhalf .. 8 dhalf + 7 over all D dims (each warp one n8 tile);
    //   else:   both warps take all G columns and split the D dims of P.V.
    // A paired head of over 8 columns takes two n8 tiles in its warp: each K
    // and V fragment feeds both.
    constexpr bool CSPLIT = !PAIR && G > 8;
    constexpr int GW = CSPLIT ? G / 2 : G;       // columns of this warp
    constexpr int NT = GW > 8 ? 2 : 1;           // n8 tiles of columns per warp
    constexpr int DW = PAIR ? D / 2 : D;         // dims of one column's q row
    constexpr int KS = DW / 16;                  // k-steps of q.K^T
    constexpr int DT = CSPLIT ? D / 16 : HD::kDimTilesPerWarp;   // 16-dim tiles of P.V per warp
    constexpr int GT = PAIR ? 2 * G : G;         // columns of the launch head
    constexpr int DR = PAIR ? D / 2 : D;         // dims kept per column in the reduction
    constexpr bool FP8 = kv_is_fp8(KV);
    constexpr bool MMA_F16 = KV != kKvBf16;   // fp16 MMAs for fp16 and FP8 caches
    // P.V takes each weight as hi + lo, both of the MMA type, in two MMAs:
    // hi is the weight rounded (8 significant bits in bf16, 11 in fp16), lo
    // its rounded remainder, so the pair carries 16 or 22 bits.  fp16 weights
    // are scaled by 2^15 first (a weight is at most 1), which keeps weights
    // down to ~2^-39 clear of fp16's underflow; l and O share the scale,
    // which cancels in O = acc / l.
    constexpr float kPScale = MMA_F16 ? 32768.f : 1.f;
    static_assert(HD::kParts >= 1, "tensor-core rows span at least one 128-byte part");
    const int NS = p.num_stages;
    const int pair = cw >> 1, dhalf = cw & 1;
    const int grp = lane >> 2, qd = lane & 3;   // mma fragment coordinates
    const int tok0 = pair * 16;
    const int rl = p.box_rows_log2;
    float *red_acc = reinterpret_cast<float *>(smem + p.off_red);   // [pairs][GT][DR]
    float *red_m = red_acc + kPairs * GT * DR;                       // [pairs][GT]
    float *red_l = red_m + kPairs * GT;                              // [2 pairs][GT]: l, then lt
    const int ctid = cw * 32 + lane;
    const int cbase = PAIR ? dhalf * G : (CSPLIT ? dhalf * GW : 0);  // this warp's first column
    const int dtb = CSPLIT ? 0 : dhalf * DT;                         // its first 16-dim tile of P.V
    const int koff = PAIR ? dhalf * (HD::kRowBytes / 32) : 0;        // its first 16-byte chunk of K

    uint32_t qb[NT][KS][2];    // Q^T B-fragments, one pair per 16-dim k-step
    float smul[NT][2];         // score multipliers of columns 2 qd, 2 qd + 1 (log2 units)
    float acc[NT][DT][4];      // O^T fragments of this warp's D/32 dim tiles
    // columns 2 qd and 2 qd + 1 of each tile, this lane's tokens only: l sums
    // the 16-bit rounded weights that multiply V, lt the exact fp32 weights
    // (for the LSE)
    float m[NT][2], l[NT][2], lt[NT][2];
    int lag[NT][2];            // causal lag of those columns
    auto reset = [&]() {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                m[nt][j] = kNegInf;
                l[nt][j] = 0.f;
                lt[nt][j] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < DT; ++i)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    acc[nt][i][c] = 0.f;
        }
    };
    auto give_up = [&]() {
        if (lane == 0) {
            atomicOr(p.ws_err, kErrTimeout);
            *abort_flag = 1;
        }
    };
    reset();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
            qb[nt][ks][0] = qb[nt][ks][1] = 0u;
        smul[nt][0] = smul[nt][1] = p.scale_log2;
        lag[nt][0] = p.q_len - 1 - col_info(p, 0, 0, cbase + nt * 8 + 2 * qd).i;
        lag[nt][1] = p.q_len - 1 - col_info(p, 0, 0, cbase + nt * 8 + 2 * qd + 1).i;
    }

    int s = 0;
    uint32_t ph = 0, cph = 0;
    for (int t = t_begin; t < t_end; ++t) {
        if (!warp_wait(full0 + 8 * s, ph, p.timeout_ns, abort_flag)) {
            give_up();
            return;
        }
        const int *mt = meta + s * kMetaInts;
        const int b = mt[0], h = mt[1], rem = mt[2], nvalid = mt[3], flags = mt[4], u = mt[5];

        if (flags & kFirstInCta) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // A fused head's query reads its own fuse_dh dims; zeros elsewhere.
                // Padding columns keep a zero query.
                const int qdim = PAIR ? DW : (p.fuse_dh ? p.fuse_dh : D);
                const int lc = nt * 8 + grp;   // this lane's column within the warp's columns
                const ColInfo col = col_info(p, b, h, cbase + (lc < GW ? lc : 0));
                const int part = col.dim0;
                const bool colv = col.valid && lc < GW;
                const uint16_t *qrow = p.q + col.row * qdim;
                if constexpr (!FP8) {
                    // B[k = d][n = column]: lane holds column grp, dims 16 ks + 2 qd (+1) and (+8, +9).
                    const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qrow);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int d0 = ks * 16 - part;   // first dim of this k-step in the q row
                        const bool in = colv && d0 >= 0 && d0 < qdim;
                        qb[nt][ks][0] = in ? __ldg(q32 + d0 / 2 + qd) : 0u;
                        qb[nt][ks][1] = in ? __ldg(q32 + d0 / 2 + 4 + qd) : 0u;
                    }
                } else {
                    // lane holds column grp, dims 16 ks + 4 qd .. + 3 (see above)
                    const bool qf16 = p.q_f16 != 0;
                    float qv[KS][4];
                    float amax = 0.f;
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int d0 = ks * 16 - part;
                        const bool in = colv && d0 >= 0 && d0 < qdim;
                        uint2 w = make_uint2(0u, 0u);
                        if (in)
                            w = __ldg(reinterpret_cast<const uint2 *>(qrow + d0 + 4 * qd));
                        const float2 lo = qf16 ? f16x2_to_float2(w.x) : bf16x2_to_float2(w.x);
                        const float2 hi = qf16 ? f16x2_to_float2(w.y) : bf16x2_to_float2(w.y);
                        qv[ks][0] = lo.x;
                        qv[ks][1] = lo.y;
                        qv[ks][2] = hi.x;
                        qv[ks][3] = hi.y;
                        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(lo.x), fabsf(lo.y)), fmaxf(fabsf(hi.x), fabsf(hi.y))));
                    }
                    // the column's max over its four lanes (same grp)
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                    // power of two sh with amax * 2^-sh in [2^14, 2^15); zero columns keep sh = 0
                    int sh = 0;
                    if (amax > 0.f) {
                        const int e = ((__float_as_int(amax) >> 23) & 255) - 127;   // floor(log2 amax), normals
                        sh = min(max(e - 14, -120), 126);
                    }
                    const float down = __int_as_float((127 - sh) << 23);   // 2^-sh
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        qb[nt][ks][0] = pack_f16x2(qv[ks][0] * down, qv[ks][1] * down);
                        qb[nt][ks][1] = pack_f16x2(qv[ks][2] * down, qv[ks][3] * down);
                    }
                    // this lane's score columns are 2 qd and 2 qd + 1 (held by lanes 4 column)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int shj = __shfl_sync(0xffffffffu, sh, (2 * qd + j) * 4);
                        smul[nt][j] = p.scale_log2 * __int_as_float((127 + shj) << 23);
                    }
                }
            }
        }

        const uint32_t ktile = stage0 + s * HD::kStageBytes;
        const uint32_t vtile = ktile + HD::kTileBytes;

        // S^T = K . Q^T for tokens tok0 .. tok0 + 15 (fragment rows grp and grp + 8).
        // Even and odd k-steps accumulate separately: two dependent MMA chains
        // of KS/2 instead of one of KS (the chain's latency bounds the tile).
        float sc[NT][4], sc2[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                sc[nt][i] = sc2[nt][i] = 0.f;
        {
            const int row = tok0 + (lane & 7) + (((lane >> 3) & 1) << 3);
            if constexpr (!FP8) {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(sw128_addr<HD::kParts>(ktile, row, koff + 2 * ks + (lane >> 4), rl), a0, a1, a2,
                                a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_16816<MMA_F16>((ks & 1) ? sc2[nt] : sc[nt], a0, a1, a2, a3, qb[nt][ks][0],
                                           qb[nt][ks][1]);
                }
            } else {
                // one ldmatrix covers two 16-dim chunks: k-steps 2 kk and 2 kk + 1
#pragma unroll
                for (int kk = 0; kk < KS / 2; ++kk) {
                    uint32_t r0, r1, r2, r3;
                    ldmatrix_x4(sw128_addr<HD::kParts>(ktile, row, koff + 2 * kk + (lane >> 4), rl), r0, r1, r2,
                                r3);
                    const uint32_t e0 = fp8x2_to_f16x2<KV>(lo16(r0)), e1 = fp8x2_to_f16x2<KV>(lo16(r1));
                    const uint32_t e2 = fp8x2_to_f16x2<KV>(hi16(r0)), e3 = fp8x2_to_f16x2<KV>(hi16(r1));
                    const uint32_t o0 = fp8x2_to_f16x2<KV>(lo16(r2)), o1 = fp8x2_to_f16x2<KV>(lo16(r3));
                    const uint32_t o2 = fp8x2_to_f16x2<KV>(hi16(r2)), o3 = fp8x2_to_f16x2<KV>(hi16(r3));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_16816<true>(sc[nt], e0, e1, e2, e3, qb[nt][2 * kk][0], qb[nt][2 * kk][1]);
                        mma_16816<true>(sc2[nt], o0, o1, o2, o3, qb[nt][2 * kk + 1][0], qb[nt][2 * kk + 1][1]);
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    sc[nt][i] += sc2[nt][i];
        }

        // Per n8 tile: mask, online softmax over this warp's 16 tokens, P.
        float alpha[NT][2];
        uint32_t pb0[NT], pb1[NT];
        uint32_t pe0[NT], pe1[NT];   // the remainders' B operands
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            // sc[0]: (token grp, column 2qd), sc[1]: (grp, 2qd+1), sc[2]: (grp+8, 2qd), sc[3]: (grp+8, 2qd+1);
            // a token counts for a column if it is inside the column's causal end
            // (the request's end when there is one new token)
            float x[4];
            if (p.q_len == 1) {
                const bool v0 = tok0 + grp < nvalid, v1 = tok0 + grp + 8 < nvalid;
                x[0] = v0 ? sc[nt][0] * smul[nt][0] : kNegInf;
                x[1] = v0 ? sc[nt][1] * smul[nt][1] : kNegInf;
                x[2] = v1 ? sc[nt][2] * smul[nt][0] : kNegInf;
                x[3] = v1 ? sc[nt][3] * smul[nt][1] : kNegInf;
            } else {
                const int lim0 = min(nvalid, rem - lag[nt][0]), lim1 = min(nvalid, rem - lag[nt][1]);
                x[0] = tok0 + grp < lim0 ? sc[nt][0] * smul[nt][0] : kNegInf;
                x[1] = tok0 + grp < lim1 ? sc[nt][1] * smul[nt][1] : kNegInf;
                x[2] = tok0 + grp + 8 < lim0 ? sc[nt][2] * smul[nt][0] : kNegInf;
                x[3] = tok0 + grp + 8 < lim1 ? sc[nt][3] * smul[nt][1] : kNegInf;
            }
            float pw[4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float mx = fmaxf(x[j], x[j + 2]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m[nt][j], mx);
                alpha[nt][j] = (m[nt][j] == kNegInf) ? 0.f : exp2_approx(m[nt][j] - m_new);
                pw[j] = (x[j] == kNegInf) ? 0.f : exp2_approx(x[j] - m_new);
                pw[j + 2] = (x[j + 2] == kNegInf) ? 0.f : exp2_approx(x[j + 2] - m_new);
                m[nt][j] = m_new;
            }
            float ps[4];   // the weights in the units of the P.V product
#pragma unroll
            for (int i = 0; i < 4; ++i)
                ps[i] = pw[i] * kPScale;
            const uint32_t p_r0 = pack_x2<MMA_F16>(ps[0], ps[1]);   // token grp, columns 2qd, 2qd+1
            const uint32_t p_r8 = pack_x2<MMA_F16>(ps[2], ps[3]);   // token grp + 8
            {
                float2 r0 = x2_to_float2<MMA_F16>(p_r0), r8 = x2_to_float2<MMA_F16>(p_r8);
                // the remainder of each weight: ps - hi is exact in fp32
                const uint32_t e_r0 = pack_x2<MMA_F16>(ps[0] - r0.x, ps[1] - r0.y);
                const uint32_t e_r8 = pack_x2<MMA_F16>(ps[2] - r8.x, ps[3] - r8.y);
                const float2 f0 = x2_to_float2<MMA_F16>(e_r0), f8 = x2_to_float2<MMA_F16>(e_r8);
                r0 = make_float2(r0.x + f0.x, r0.y + f0.y);
                r8 = make_float2(r8.x + f8.x, r8.y + f8.y);
                pe0[nt] = movmatrix_trans(e_r0);
                pe1[nt] = movmatrix_trans(e_r8);
                l[nt][0] = l[nt][0] * alpha[nt][0] + (r0.x + r8.x);
                l[nt][1] = l[nt][1] * alpha[nt][1] + (r0.y + r8.y);
                lt[nt][0] = lt[nt][0] * alpha[nt][0] + (pw[0] + pw[2]);
                lt[nt][1] = lt[nt][1] * alpha[nt][1] + (pw[1] + pw[3]);
            }
            // P^T as the B operand (k = token, n = column): transpose the 8x8 blocks.
            pb0[nt] = movmatrix_trans(p_r0);
            pb1[nt] = movmatrix_trans(p_r8);
        }

        // Rows past the request's end may hold anything (even NaN), and the
        // tensor core would form 0 * NaN: zero the part of them this warp
        // reads (its half of the dims; every dim under CSPLIT, where both
        // warps of the pair store the same zeros).
        const bool ragged = nvalid < tok0 + 16;
        if (ragged) {
            constexpr int kChunks = HD::kRowBytes / (CSPLIT ? 16 : 32);   // 16-byte chunks this warp reads
            const int c0 = CSPLIT ? 0 : dhalf * kChunks;
            const int first = nvalid > tok0 ? nvalid : tok0;
            for (int idx = lane; idx < (tok0 + 16 - first) * kChunks; idx += 32) {
                const uint32_t a = sw128_addr<HD::kParts>(vtile, first + idx / kChunks,
                                                          c0 + idx % kChunks, rl);
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
            }
            __syncwarp();
        }

        // O^T = alpha O^T + V^T . P^T over this warp's dims (tiles dtb .. dtb + DT - 1).
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < DT; ++i) {
                acc[nt][i][0] *= alpha[nt][0];
                acc[nt][i][1] *= alpha[nt][1];
                acc[nt][i][2] *= alpha[nt][0];
                acc[nt][i][3] *= alpha[nt][1];
            }
        if constexpr (!FP8) {
            const int vrow = tok0 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
            for (int i = 0; i < DT; ++i) {
                const int dt = dtb + i;   // 16-dim tile index
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4_trans(sw128_addr<HD::kParts>(vtile, vrow, 2 * dt + ((lane >> 3) & 1), rl), a0, a1,
                                  a2, a3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_16816<MMA_F16>(acc[nt][i], a0, a1, a2, a3, pb0[nt], pb1[nt]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_16816<MMA_F16>(acc[nt][i], a0, a1, a2, a3, pe0[nt], pe1[nt]);
            }
        } else {
            // matrices (tokens 0-7 | 8-15) x (chunk c | c + 1): two 16-dim tiles per ldmatrix
            const int vrow = tok0 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
            for (int ii = 0; ii < DT / 2; ++ii) {
                const int c = dtb + 2 * ii;   // chunk = 16-dim tile index
                uint32_t r0, r1, r2, r3;
                ldmatrix_x4_trans(sw128_addr<HD::kParts>(vtile, vrow, c + (lane >> 4), rl), r0, r1, r2, r3);
                // bytes (t, 2grp), (t, 2grp+1), (t+1, 2grp), (t+1, 2grp+1) -> dim pairs over tokens
                const uint32_t s0 = prmt(r0, 0u, 0x3120u), s1 = prmt(r1, 0u, 0x3120u);
                const uint32_t s2 = prmt(r2, 0u, 0x3120u), s3 = prmt(r3, 0u, 0x3120u);
                const uint32_t a0 = fp8x2_to_f16x2<KV>(lo16(s0)), a1 = fp8x2_to_f16x2<KV>(hi16(s0));
                const uint32_t a2 = fp8x2_to_f16x2<KV>(lo16(s1)), a3 = fp8x2_to_f16x2<KV>(hi16(s1));
                const uint32_t b0 = fp8x2_to_f16x2<KV>(lo16(s2)), b1 = fp8x2_to_f16x2<KV>(hi16(s2));
                const uint32_t b2 = fp8x2_to_f16x2<KV>(lo16(s3)), b3 = fp8x2_to_f16x2<KV>(hi16(s3));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_16816<true>(acc[nt][2 * ii], a0, a1, a2, a3, pb0[nt], pb1[nt]);
                    mma_16816<true>(acc[nt][2 * ii + 1], b0, b1, b2, b3, pb0[nt], pb1[nt]);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_16816<true>(acc[nt][2 * ii], a0, a1, a2, a3, pe0[nt], pe1[nt]);
                    mma_16816<true>(acc[nt][2 * ii + 1], b0, b1, b2, b3, pe0[nt], pe1[nt]);
                }
            }
        }
        if (ragged)   // order the zeroing stores before the next TMA write to this stage
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty0 + 8 * s);

        if (flags & kLastInCta) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // l over the warp's 16 tokens (lanes sharing qd hold the same columns)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], 4);
                    l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], 8);
                    l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], 16);
                    lt[nt][j] += __shfl_xor_sync(0xffffffffu, lt[nt][j], 4);
                    lt[nt][j] += __shfl_xor_sync(0xffffffffu, lt[nt][j], 8);
                    lt[nt][j] += __shfl_xor_sync(0xffffffffu, lt[nt][j], 16);
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int head = nt * 8 + 2 * qd + j;     // this warp's column
                    const int gcol = cbase + head;            // the launch head's column
                    if (head < GW && p.col_code[gcol] >= 0) {
                        if ((PAIR || CSPLIT || dhalf == 0) && grp == 0) {
                            red_m[pair * GT + gcol] = m[nt][j];
                            red_l[pair * GT + gcol] = l[nt][j];
                            red_l[(kPairs + pair) * GT + gcol] = lt[nt][j];   // exact sums after the pairs' slots
                        }
#pragma unroll
                        for (int i = 0; i < DT; ++i) {
                            // output rows grp and grp + 8 of the tile: dims grp and grp + 8, or for
                            // FP8 caches 2 grp and 2 grp + 1 (see above); paired heads keep their own dims
                            const int d0 = (dtb + i) * 16 - (PAIR ? dhalf * DR : 0);
                            const int dlo = d0 + (FP8 ? 2 * grp : grp), dhi = d0 + (FP8 ? 2 * grp + 1 : grp + 8);
                            red_acc[(pair * GT + gcol) * DR + dlo] = acc[nt][i][j];
                            red_acc[(pair * GT + gcol) * DR + dhi] = acc[nt][i][j + 2];
                        }
                    }
                }
            }
            if (!consumer_sync(cbar, cph, p.timeout_ns, abort_flag, lane)) {
                give_up();
                return;
            }
            combine_and_write<GT, kPairs, DR>(p, red_acc, red_m, red_l, red_l + kPairs * GT, ctid, b, h, u,
                                              (flags & kOwnSegment) != 0);
            if (!consumer_sync(cbar, cph, p.timeout_ns, abort_flag, lane)) {
                give_up();
                return;
            }
            reset();
        }
        if (++s == NS) {
            s = 0;
            ph ^= 1u;
        }
    }
}

// ------------------------------------------------------------------ TMEM scores (E4M3, paired heads)

// The score issuer of the TMEM-score instances: one warp.  For each tile of
// the CTA it forms S = K . Q^T for both kv heads of the fused row with four
// tcgen05 MMAs (M = 128 rows: the tile's 64 tokens of head 0, then those of
// head 1, as the 128-byte parts of the swizzled K tile lie; N = 16 columns
// per query part; K = 128 FP8 dims in four steps of 32) into TMEM buffer
// (tile index mod kTc5Buffers), and signals the buffer's ready barrier.
//
// The query operand holds each column's 16-bit query row as NP parts in the
// cache's FP8 format (A and B of one MMA share a format) of x = q 2^-sh (sh
// per column, so that the column's largest |x| lies in [128, 256)): part 0 =
// FP8(x), and part k+1 = FP8(R r_k) of the remainder r_k = (x scaled by R^k)
// - (parts 0..k so scaled), R = 16 for E4M3 and 8 for E5M2.  Each part keeps
// 4 (E4M3) or 3 (E5M2) more significant bits, so a bf16 query's 8 take 2 or
// 3 parts and an fp16 query's 11 take 3 or 4: x = sum_k part_k R^-k exactly
// for every element within 2^13 of its column's largest (E4M3; E5M2's range
// covers every fp16 and bf16 ratio in use); smaller ones are off by under
// 2^-21 of the largest.  The consumers take S = (sum_k S_k R^-k) 2^sh scale
// log2(e).
template <int KV>
__host__ __device__ constexpr int tc5_query_parts(bool q_f16)
{
    return KV == kKvE4m3 ? (q_f16 ? 3 : 2) : (q_f16 ? 4 : 3);
}

template <int G, int KV>
__device__ __forceinline__ void split_score_issuer(const SplitParams &p, uint8_t *tc, uint32_t stage0,
                                                   const int *meta, uint32_t full0, uint32_t ready0,
                                                   uint32_t free0, uint32_t tmem, volatile int *abort_flag,
                                                   int t_begin, int t_end, int lane)
{
    static_assert(G >= 1 && G <= 8, "up to 8 query columns per kv head");
    static_assert(KV == kKvE4m3 || KV == kKvE5m2, "FP8 caches");
    constexpr int kStage = Shape<256, KV>::kStageBytes;
    constexpr float kRadix = KV == kKvE4m3 ? 16.f : 8.f;   // R: one part's weight over the next
    const bool qf16 = p.q_f16 != 0;
    const int np = tc5_query_parts<KV>(qf16);               // query parts
    const uint32_t idesc = umma_idesc_fp8_f32(128, 16 * np, KV == kKvE4m3 ? 0u : 1u);
    const int NS = p.num_stages;
    const uint32_t qop = smem_addr(tc);
    float *mul_buf = reinterpret_cast<float *>(tc + kTc5OffMul);
    // lane: query column (head hh, column c) = lane / 2, dims 64 (lane % 2) .. + 63
    const int pc = lane >> 1, half = lane & 1;
    const int hh = pc >> 3, c = pc & 7;
    const int gcol = hh * G + c;
    float my_mul = 0.f;   // this column's score multiplier (lanes with half == 0 publish it)

    auto give_up = [&]() {
        if (lane == 0) {
            atomicOr(p.ws_err, kErrTimeout);
            *abort_flag = 1;
        }
    };
    // Query rows of segment (b, h) as the E4M3 operand (row 16 k + 8 hh + c
    // holds part k of column c of head hh; padding columns zero) and this
    // lane's column multiplier.
    auto load_query = [&](int b, int h) {
        const bool colv = c < G && p.col_code[gcol] >= 0;
        float x[64];
        float amax = 0.f;
        if (colv) {
            const ColInfo col = col_info(p, b, h, gcol);
            const uint4 *src = reinterpret_cast<const uint4 *>(p.q + col.row * 128 + half * 64);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint4 w = __ldg(src + k);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = qf16 ? f16x2_to_float2(ws[e]) : bf16x2_to_float2(ws[e]);
                    x[8 * k + 2 * e] = f.x;
                    x[8 * k + 2 * e + 1] = f.y;
                }
            }
#pragma unroll
            for (int k = 0; k < 64; ++k)
                amax = fmaxf(amax, fabsf(x[k]));
        } else {
#pragma unroll
            for (int k = 0; k < 64; ++k)
                x[k] = 0.f;
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        int sh = 0;
        if (amax > 0.f) {
            const int e = ((__float_as_int(amax) >> 23) & 255) - 127;   // floor(log2 amax), normals
            sh = min(max(e - 7, -120), 126);
        }
        const float down = __int_as_float((127 - sh) << 23);   // 2^-sh
        my_mul = p.scale_log2 * __int_as_float((127 + sh) << 23);
#pragma unroll
        for (int k = 0; k < 64; ++k)
            x[k] *= down;
#pragma unroll
        for (int part = 0; part < kTc5MaxParts; ++part) {
            if (part >= np)
                break;
            const int row = 16 * part + 8 * hh + c;
#pragma unroll
            for (int k = 0; k < 4; ++k) {   // 16-dim chunk half * 4 + k of the row
                uint32_t wd[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float *v = x + 16 * k + 4 * e;
                    const uint16_t c01 = KV == kKvE4m3 ? pack_e4m3x2(v[0], v[1]) : pack_e5m2x2(v[0], v[1]);
                    const uint16_t c23 = KV == kKvE4m3 ? pack_e4m3x2(v[2], v[3]) : pack_e5m2x2(v[2], v[3]);
                    const float2 b01 = fp8x2_to_float2<KV>(c01), b23 = fp8x2_to_float2<KV>(c23);
                    // the remainder, scaled for the next part (exact in fp32)
                    v[0] = kRadix * (v[0] - b01.x);
                    v[1] = kRadix * (v[1] - b01.y);
                    v[2] = kRadix * (v[2] - b23.x);
                    v[3] = kRadix * (v[3] - b23.y);
                    wd[e] = (uint32_t)c01 | ((uint32_t)c23 << 16);
                }
                const int chunk = half * 4 + k;
                const uint32_t a = qop + (row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(wd[0]), "r"(wd[1]),
                             "r"(wd[2]), "r"(wd[3])
                             : "memory");
            }
        }
        // the MMAs (async proxy) read what these generic stores wrote
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
    };

    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    for (int t = t_begin; t < t_end; ++t) {
        const int i = t - t_begin;
        if (!warp_wait(full0 + 8 * s, ph, p.timeout_ns, abort_flag)) {
            give_up();
            break;
        }
        const uint32_t ma = smem_addr(meta + s * kMetaInts);   // 8-byte aligned
        const uint2 m01 = lds64(ma), m45 = lds64(ma + 16);
        const bool first = ((int)m45.x & kFirstInCta) != 0;
        const int bi = i % kTc5Buffers;
        if (first) {
            // a new segment: the previous tile's MMAs (the last issued) must
            // have read the query operand before it is rewritten
            if (i > 0 && !warp_wait(ready0 + 8 * ((i - 1) % kTc5Buffers), (uint32_t)(((i - 1) / kTc5Buffers) & 1),
                                    p.timeout_ns, abort_flag)) {
                give_up();
                break;
            }
            load_query((int)m01.x, (int)m01.y);
        }
        // the consumers of the tile kTc5Buffers back have read this buffer
        if (!warp_wait(free0 + 8 * bi, (uint32_t)((i / kTc5Buffers) & 1) ^ 1u, p.timeout_ns, abort_flag)) {
            give_up();
            break;
        }
        tc_fence_after();
        if (lane == 0) {
            const uint32_t ktile = stage0 + s * kStage;
            const uint32_t d = tmem + (uint32_t)(bi * kTc5Cols);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                umma_f8f6f4(d, umma_desc_sw128(ktile + 32 * k), umma_desc_sw128(qop + 32 * k), idesc, k > 0);
            umma_commit(ready0 + 8 * bi);
        }
        if (half == 0)
            mul_buf[bi * 16 + pc] = my_mul;
        __syncwarp();
        if (lane == 0)
            mbar_arrive(ready0 + 8 * bi);   // the second arrival: the multipliers are written
        ++issued;
        if (++s == NS) {
            s = 0;
            ph ^= 1u;
        }
    }
    // Before the TMEM is freed: wait (bounded) for the last MMAs issued.
    if (issued > 0) {
        const int k = issued - 1;
        mbar_wait_bounded(ready0 + 8 * (k % kTc5Buffers), (uint32_t)((k / kTc5Buffers) & 1), p.timeout_ns, nullptr);
    }
    __syncwarp();
}

// The consumers of the TMEM-score instances (FP8, two fused kv heads of 128
// dims, up to 8 columns each).  The eight warps form two groups of four;
// group g takes the CTA's tiles of index g (mod 2), so two tiles are in
// flight.  In a group, warp w reads TMEM lanes 32 (w % 4) .. + 31: the
// scores of 32 tokens of head (w % 4) / 2, one token per lane and its
// head's columns in registers.  Each warp runs its own online softmax over
// its tokens (column maxima by redux), stages its weights in shared memory
// as two fp16 parts (as split_consumer_mma: hi, and the rounded remainder lo,
// both of weights scaled by 2^15), reads them back as the B fragments of P.V,
// and forms O^T += V^T . P^T over its head's 128 dims with warp MMAs on V
// converted to fp16 in registers.  The four states of each head (2 groups x
// 2 token halves) are combined at every segment's last tile in the CTA.
template <int G, int KV>
__device__ __forceinline__ void split_consumer_tc5(const SplitParams &p, uint8_t *smem, uint8_t *tc,
                                                   uint32_t stage0, const int *meta, uint32_t full0,
                                                   uint32_t empty0, uint32_t cbar, uint32_t ready0, uint32_t free0,
                                                   uint32_t tmem, volatile int *abort_flag, int t_begin, int t_end,
                                                   int cw, int lane)
{
    static_assert(G >= 1 && G <= 8, "up to 8 query columns per kv head");
    using HD = Shape<256, KV>;
    constexpr int GT = 2 * G;    // columns of the launch head
    constexpr int DR = 128;      // dims of one head
    constexpr int DT = DR / 16;  // 16-dim tiles of P.V
    constexpr float kPScale = 32768.f;
    const int NS = p.num_stages;
    const int gsel = cw >> 2, quad = cw & 3;
    const int hh = quad >> 1, tokw = (quad & 1) * 32;
    const int grp = lane >> 2, qd = lane & 3;
    const int st = gsel * 2 + (quad & 1);   // this warp's state among the head's four
    float *red_acc = reinterpret_cast<float *>(smem + p.off_red);   // [4 states][GT][DR]
    float *red_m = red_acc + kPairs * GT * DR;                       // [4 states][GT]
    float *red_l = red_m + kPairs * GT;                              // [2][4 states][GT]: l, then lt
    const float *mul_buf = reinterpret_cast<const float *>(tc + kTc5OffMul);
    const uint32_t pbuf = smem_addr(tc + kTc5OffP + cw * kTc5PBytes);
    const uint32_t lane_row = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(hh * 8);
    const int ctid = cw * 32 + lane;
    const int np = tc5_query_parts<KV>(p.q_f16 != 0);   // query parts
    constexpr float kInvRadix = KV == kKvE4m3 ? 0.0625f : 0.125f;   // one part's weight over the previous

    float acc[DT][4];            // O^T fragments: dims 16 i + 2 grp (+1), columns 2 qd (+1)
    float m[G], l[G], lt[G];     // m is the same in every lane; l, lt sum this lane's token
    int lag[G];
    auto reset = [&]() {
#pragma unroll
        for (int c = 0; c < G; ++c) {
            m[c] = kNegInf;
            l[c] = 0.f;
            lt[c] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < DT; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                acc[i][k] = 0.f;
    };
    auto give_up = [&]() {
        if (lane == 0) {
            atomicOr(p.ws_err, kErrTimeout);
            *abort_flag = 1;
        }
    };
    reset();
#pragma unroll
    for (int c = 0; c < G; ++c)
        lag[c] = p.q_len - 1 - col_info(p, 0, 0, hh * G + c).i;

    int s = 0;
    uint32_t ph = 0, cph = 0;
    for (int t = t_begin; t < t_end; ++t) {
        const int i = t - t_begin;
        if (!warp_wait(full0 + 8 * s, ph, p.timeout_ns, abort_flag)) {
            give_up();
            return;
        }
        const uint32_t ma = smem_addr(meta + s * kMetaInts);   // 8-byte aligned
        const uint2 mv0 = lds64(ma), mv1 = lds64(ma + 8), mv2 = lds64(ma + 16);
        const int b = (int)mv0.x, h = (int)mv0.y, rem = (int)mv1.x, nvalid = (int)mv1.y, flags = (int)mv2.x,
                  u = (int)mv2.y;
        bool ragged = false;
        if ((i & 1) == gsel) {
            const int bi = i % kTc5Buffers;
            if (!warp_wait(ready0 + 8 * bi, (uint32_t)((i / kTc5Buffers) & 1), p.timeout_ns, abort_flag)) {
                give_up();
                return;
            }
            tc_fence_after();
            // the query parts' scores of this lane's token (16 columns apart)
            float s0[8], s1[8], s2[8], s3[8];
            const uint32_t tb = lane_row + (uint32_t)(bi * kTc5Cols);
            tmem_ld_x8(tb, s0);
            tmem_ld_x8(tb + 16, s1);
            if (np > 2)
                tmem_ld_x8(tb + 32, s2);
            if (np > 3)
                tmem_ld_x8(tb + 48, s3);
            // the buffer's multipliers, read before it is released: the issuer
            // rewrites them with the buffer's next MMAs
            float mul[G];
            {
                const uint32_t mb = smem_addr(mul_buf) + (uint32_t)(bi * 64 + hh * 32);
                const uint4 m0 = lds128(mb), m1 = lds128(mb + 16);
                const float mm[8] = {__uint_as_float(m0.x), __uint_as_float(m0.y), __uint_as_float(m0.z),
                                     __uint_as_float(m0.w), __uint_as_float(m1.x), __uint_as_float(m1.y),
                                     __uint_as_float(m1.z), __uint_as_float(m1.w)};
#pragma unroll
                for (int c = 0; c < G; ++c)
                    mul[c] = mm[c];
            }
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(free0 + 8 * bi);   // the buffer may take the next MMAs

            // Mask, online softmax over this warp's 32 tokens, weights as hi + lo.
            const int tok = tokw + lane;
            float alpha[G];
            uint32_t phi[4], plo[4];   // columns 2k, 2k + 1 of this lane's token (fp16 pairs)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                phi[k] = plo[k] = 0u;
#pragma unroll
            for (int c = 0; c < G; c += 2) {
                float x[2], pw[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int cc = c + j < G ? c + j : c;
                    const int lim = p.q_len == 1 ? nvalid : min(nvalid, rem - lag[cc]);
                    float sc = np > 3 ? s3[cc] : 0.f;
                    sc = np > 2 ? s2[cc] + sc * kInvRadix : sc;
                    sc = s0[cc] + (s1[cc] + sc * kInvRadix) * kInvRadix;
                    x[j] = tok < lim ? sc * mul[cc] : kNegInf;
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (c + j >= G) {
                        pw[j] = 0.f;
                        continue;
                    }
                    const float m_new = fmaxf(m[c + j], warp_max_f32(x[j]));
                    alpha[c + j] = (m[c + j] == kNegInf) ? 0.f : exp2_approx(m[c + j] - m_new);
                    pw[j] = (x[j] == kNegInf) ? 0.f : exp2_approx(x[j] - m_new);
                    m[c + j] = m_new;
                }
                const uint32_t hi = pack_f16x2(pw[0] * kPScale, pw[1] * kPScale);
                const float2 hv = f16x2_to_float2(hi);
                const uint32_t lo = pack_f16x2(pw[0] * kPScale - hv.x, pw[1] * kPScale - hv.y);
                const float2 lv = f16x2_to_float2(lo);
                phi[c >> 1] = hi;
                plo[c >> 1] = lo;
                l[c] = l[c] * alpha[c] + (hv.x + lv.x);
                lt[c] = lt[c] * alpha[c] + pw[0];
                if (c + 1 < G) {
                    l[c + 1] = l[c + 1] * alpha[c + 1] + (hv.y + lv.y);
                    lt[c + 1] = lt[c + 1] * alpha[c + 1] + pw[1];
                }
            }
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(pbuf + lane * 16), "r"(phi[0]),
                         "r"(phi[1]), "r"(phi[2]), "r"(phi[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(pbuf + 512 + lane * 16), "r"(plo[0]),
                         "r"(plo[1]), "r"(plo[2]), "r"(plo[3])
                         : "memory");
            __syncwarp();
            // P^T B fragments: matrix k of each x4 is tokens 8k .. 8k + 7 of the warp's 32
            uint32_t bh[4], bl[4];
            ldmatrix_x4_trans(pbuf + lane * 16, bh[0], bh[1], bh[2], bh[3]);
            ldmatrix_x4_trans(pbuf + 512 + lane * 16, bl[0], bl[1], bl[2], bl[3]);

            const uint32_t vtile = stage0 + s * HD::kStageBytes + HD::kTileBytes;
            // V rows past the request's end may hold anything (even NaN), and
            // the tensor core would form 0 * NaN: zero this warp's rows of its head.
            ragged = nvalid < tokw + 32;
            if (ragged) {
                const int first = nvalid > tokw ? nvalid : tokw;
                for (int idx = lane; idx < (tokw + 32 - first) * 8; idx += 32) {
                    const uint32_t a = sw128_addr<HD::kParts>(vtile, first + idx / 8, hh * 8 + idx % 8, 6);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
                }
                __syncwarp();
            }

            // O^T = alpha O^T + V^T . P^T over the head's 128 dims
            // alpha of columns 2 qd and 2 qd + 1, by selects (an indexed read
            // of alpha would put it in local memory)
            float a0 = alpha[0], a1 = G > 1 ? alpha[G > 1 ? 1 : 0] : 1.f;
#pragma unroll
            for (int k = 1; 2 * k < G; ++k) {
                const bool mine = qd == k;
                a0 = mine ? alpha[2 * k] : a0;
                a1 = mine ? alpha[2 * k + 1] : a1;
            }
#pragma unroll
            for (int k = 0; k < DT; ++k) {
                acc[k][0] *= a0;
                acc[k][1] *= a1;
                acc[k][2] *= a0;
                acc[k][3] *= a1;
            }
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                // matrices (tokens 0-7 | 8-15 of the k step) x (chunk c | c + 1)
                const int vrow = tokw + 16 * ks + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
                for (int ii = 0; ii < DT / 2; ++ii) {
                    const int c = 2 * ii;
                    uint32_t r0, r1, r2, r3;
                    ldmatrix_x4_trans(sw128_addr<HD::kParts>(vtile, vrow, hh * 8 + c + (lane >> 4), 6), r0, r1, r2,
                                      r3);
                    const uint32_t s0 = prmt(r0, 0u, 0x3120u), s1 = prmt(r1, 0u, 0x3120u);
                    const uint32_t s2 = prmt(r2, 0u, 0x3120u), s3 = prmt(r3, 0u, 0x3120u);
                    const uint32_t x0 = fp8x2_to_f16x2<KV>(lo16(s0)), x1 = fp8x2_to_f16x2<KV>(hi16(s0));
                    const uint32_t x2 = fp8x2_to_f16x2<KV>(lo16(s1)), x3 = fp8x2_to_f16x2<KV>(hi16(s1));
                    const uint32_t y0 = fp8x2_to_f16x2<KV>(lo16(s2)), y1 = fp8x2_to_f16x2<KV>(hi16(s2));
                    const uint32_t y2 = fp8x2_to_f16x2<KV>(lo16(s3)), y3 = fp8x2_to_f16x2<KV>(hi16(s3));
                    mma_16816<true>(acc[c], x0, x1, x2, x3, bh[2 * ks], bh[2 * ks + 1]);
                    mma_16816<true>(acc[c + 1], y0, y1, y2, y3, bh[2 * ks], bh[2 * ks + 1]);
                    mma_16816<true>(acc[c], x0, x1, x2, x3, bl[2 * ks], bl[2 * ks + 1]);
                    mma_16816<true>(acc[c + 1], y0, y1, y2, y3, bl[2 * ks], bl[2 * ks + 1]);
                }
            }
        }
        if (ragged)   // order the zeroing stores before the next TMA write to this stage
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty0 + 8 * s);

        if (flags & kLastInCta) {
#pragma unroll
            for (int c = 0; c < G; ++c)
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    l[c] += __shfl_xor_sync(0xffffffffu, l[c], o);
                    lt[c] += __shfl_xor_sync(0xffffffffu, lt[c], o);
                }
            if (lane == 0) {
#pragma unroll
                for (int c = 0; c < G; ++c) {
                    const int gcol = hh * G + c;
                    red_m[st * GT + gcol] = m[c];
                    red_l[st * GT + gcol] = l[c];
                    red_l[(kPairs + st) * GT + gcol] = lt[c];
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c = 2 * qd + j;   // this lane's columns of the O^T fragments
                if (c < G) {
                    float *dst = red_acc + (st * GT + hh * G + c) * DR + 2 * grp;
#pragma unroll
                    for (int k = 0; k < DT; ++k) {
                        dst[16 * k] = acc[k][j];
                        dst[16 * k + 1] = acc[k][j + 2];
                    }
                }
            }
            if (!consumer_sync(cbar, cph, p.timeout_ns, abort_flag, lane)) {
                give_up();
                return;
            }
            combine_and_write<GT, kPairs, DR>(p, red_acc, red_m, red_l, red_l + kPairs * GT, ctid, b, h, u,
                                              (flags & kOwnSegment) != 0);
            if (!consumer_sync(cbar, cph, p.timeout_ns, abort_flag, lane)) {
                give_up();
                return;
            }
            reset();
        }
        if (++s == NS) {
            s = 0;
            ph ^= 1u;
        }
    }
}

// ------------------------------------------------------------------ kernels

// CPA: paged with pages under 8 tokens on the tensor-core consumers, rows
// copied by kProducerWarps warps with cp.async (split_producer_cpa).
template <int G, bool PAGED, int CONS, int KV, int D, bool CPA>
__global__ void __launch_bounds__(split_threads(CONS, CPA), 1)
    split_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv)
{
    static_assert(!CPA || (PAGED && CONS != kConsCudaCores), "cp.async copies feed paged tensor-core launches");
    static_assert(CONS != kConsTc5 || (kv_is_fp8(KV) && D == 256 && !CPA),
                  "TMEM scores: two fused FP8 kv heads of 128 dims");
    constexpr int kThreads = split_threads(CONS, CPA);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int *prefix = reinterpret_cast<int *>(smem + p.off_prefix);
    int *meta = reinterpret_cast<int *>(smem + p.off_meta);
    int *misc = reinterpret_cast<int *>(smem + p.off_misc);   // [0] abort flag, [1..] scan scratch
    const uint32_t full0 = smem_addr(smem + p.off_bar);
    const uint32_t empty0 = full0 + 8 * p.num_stages;
    const uint32_t cbar = empty0 + 8 * p.num_stages;   // consumer-warp barrier
    const uint32_t stage0 = smem_addr(smem);

    if (tid == 0) {
        for (int s = 0; s < p.num_stages; ++s) {
            mbar_init(full0 + 8 * s, CPA ? kCpAsyncArrivals : 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        mbar_init(cbar, kConsumerWarps);
        if constexpr (CONS == kConsTc5) {
            const uint32_t ready0 = smem_addr(smem + p.off_tc + kTc5OffBar);
            for (int k = 0; k < kTc5Buffers; ++k) {
                mbar_init(ready0 + 8 * k, 2);                        // the MMAs' commit + the issuer
                mbar_init(ready0 + 8 * (kTc5Buffers + k), 4);        // the four warps reading it
            }
        }
        misc[0] = 0;
        mbar_init_fence();
    }
    // Launched as a programmatic dependent of the previous kernel in the
    // stream: everything up to the wait overlaps its tail, and inputs and the
    // workspace are touched only after it has completed -- except for L2
    // prefetches of this CTA's first tiles, planned from the lengths as they
    // read now (split_prefetch), so that the first loads after the wait find
    // their data in L2.
    if constexpr (!CPA) {
        if (p.prefetch_tiles > 0) {
            build_prefix<kThreads, true>(p, prefix, misc + 1);   // ends with __syncthreads
            int pb, pe;
            const Schedule hint{prefix, prefix + p.batch + 1, p.batch, p.hkv, p.seg_cost, (int)gridDim.x};
            hint.range((int)blockIdx.x, &pb, &pe);
            if (warp == kConsumerWarps && pb < pe)
                split_prefetch<PAGED, CONS != kConsCudaCores, D, KV>(p, &tmk, &tmv, prefix, pb,
                                                                     min(pe, pb + p.prefetch_tiles), lane);
        }
    }
    pdl_wait_prior_grid();
    // The merge kernel may launch now; it waits for this grid on its own.  Its
    // early part reads the lengths, which the kernels before this one (now
    // complete) may have written.
    pdl_launch_dependents();
    build_prefix<kThreads>(p, prefix, misc + 1);   // ends with __syncthreads

    int t_begin, t_end;
    const Schedule sched{prefix, prefix + p.batch + 1, p.batch, p.hkv, p.seg_cost, (int)gridDim.x};
    sched.range((int)blockIdx.x, &t_begin, &t_end);
    if (t_begin >= t_end)
        return;
    volatile int *abort_flag = misc;
    if constexpr (CONS == kConsTc5) {
        // The score issuer's warp holds the CTA's TMEM from here to the end;
        // every warp reaches both barriers (the roles return, bounded, on
        // their own), and the issuer has waited for its last MMAs.
        uint8_t *tc = smem + p.off_tc;
        const uint32_t ready0 = smem_addr(tc + kTc5OffBar), free0 = ready0 + 8 * kTc5Buffers;
        const uint32_t slot = smem_addr(tc + kTc5OffSlot);
        const int issuer = kConsumerWarps + 1;
        if (warp == issuer)
            tmem_alloc(slot, kTc5TmemCols);
        tc_fence_before();
        named_bar_sync(1, kThreads);
        tc_fence_after();
        const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tc + kTc5OffSlot);
        if (warp == kConsumerWarps)
            split_producer<PAGED, true, D, KV>(p, &tmk, &tmv, stage0, prefix, meta, full0, empty0, abort_flag,
                                               t_begin, t_end, lane);
        else if (warp == issuer)
            split_score_issuer<G, KV>(p, tc, stage0, meta, full0, ready0, free0, tmem, abort_flag, t_begin, t_end,
                                  lane);
        else
            split_consumer_tc5<G, KV>(p, smem, tc, stage0, meta, full0, empty0, cbar, ready0, free0, tmem,
                                  abort_flag, t_begin, t_end, warp, lane);
        tc_fence_before();
        named_bar_sync(1, kThreads);
        if (warp == issuer) {
            tc_fence_after();
            tmem_dealloc(tmem, kTc5TmemCols);
        }
    } else if (warp >= kConsumerWarps) {
        if constexpr (CPA)
            split_producer_cpa<D, KV>(p, stage0, prefix, meta, full0, empty0, abort_flag, t_begin, t_end, lane,
                                      warp - kConsumerWarps);
        else
            split_producer<PAGED, CONS != kConsCudaCores, D, KV>(p, &tmk, &tmv, stage0, prefix, meta, full0,
                                                                 empty0, abort_flag, t_begin, t_end, lane);
    }
    else if constexpr (CONS != kConsCudaCores)
        split_consumer_mma<G, KV, D, CONS == kConsMmaPair>(p, smem, stage0, meta, full0, empty0, cbar,
                                                           abort_flag, t_begin, t_end, warp, lane);
    else
        split_consumer<G, KV, D>(p, smem, stage0, meta, full0, empty0, cbar, abort_flag, t_begin, t_end,
                                 warp, lane);
}

// One CTA per (segment, query head of its group); thread d owns output dim d.
// After the split grid completes, the merge is a chain of dependent loads, so
// it keeps the chain short: for small batches the segment's tile range comes
// from the lengths before the wait (as the split kernel derives it), and a
// segment split n <= kMergeDirectParts ways is merged with one round trip of
// loads and no block reductions.  Larger cases stage the partials' LSEs and
// merge weights in shared memory.
template <int G, int D>
__global__ void __launch_bounds__(D) merge_kernel(const __grid_constant__ MergeParams p)
{
    __shared__ float s_w[kMaxCtas];
    __shared__ float s_lse;
    // small batches: first tile of request b, its end, total tiles, non-empty
    // requests before b, in all
    __shared__ int s_geo[5];
    const int u = blockIdx.x, g = blockIdx.y;
    const int b = u / p.hkv, h = u - b * p.hkv;
    const int d = threadIdx.x;
    const bool small = p.batch <= kMergeDirectBatch;
    if (small && d < 32) {
        int L = 0;
        if (d < p.batch)
            L = req_len(p, d, nullptr).n;   // clamped as the split kernel clamps
        const int t = ceil_div(L, kTileTokens), e = t > 0;
        int x = t, y = e;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int xo = __shfl_up_sync(0xffffffffu, x, off), yo = __shfl_up_sync(0xffffffffu, y, off);
            if (d >= off) {
                x += xo;
                y += yo;
            }
        }
        if (d == b) {
            s_geo[0] = (x - t) * p.hkv;
            s_geo[1] = x * p.hkv;
            s_geo[3] = y - e;
        }
        if (d == 31) {
            s_geo[2] = x * p.hkv;
            s_geo[4] = y;
        }
    }
    __syncthreads();
    // The next call's split kernel may start its prologue (and its L2
    // prefetch) now, or, for short calls, once the split grid is complete.
    if (!p.late_trigger)
        pdl_launch_dependents();
    pdl_wait_prior_grid();
    if (p.late_trigger)
        pdl_launch_dependents();
    int pb, pe, T, ne_b, ne;
    if (small) {
        pb = s_geo[0];
        pe = s_geo[1];
        T = s_geo[2];
        ne_b = s_geo[3];
        ne = s_geo[4];
    } else {
        pb = p.ws_prefix[b];
        pe = p.ws_prefix[b + 1];
        T = p.ws_prefix[p.batch];
        ne_b = p.ws_prefix[p.batch + 1 + b];
        ne = p.ws_prefix[2 * p.batch + 1];
    }
    const ColInfo col = col_info(p, b, h, g);   // g < n_cols (the grid's y extent)
    if (!col.valid)
        return;   // padding column: nothing to write
    const size_t row = col.row;
    const int part = col.dim0;
    if (pe == pb) {   // empty request: O = 0, LSE = -inf
        store_o<D>(p.o, row, d, p.fuse_dh, part, 0.f);
        if (d == 0 && p.lse)
            p.lse[row] = kNegInf;
        return;
    }
    const int nb = (pe - pb) / p.hkv;
    // the CTAs that own the segment's first and last tiles (the Schedule's
    // cost positions, written out for one segment)
    const long long cost = (long long)T + (long long)p.seg_cost * p.hkv * ne;
    const long long ctas = cost < p.num_ctas ? cost : p.num_ctas;
    const long long pos0 = (long long)pb + (long long)h * nb + (long long)p.seg_cost * ((long long)p.hkv * ne_b + h + 1);
    const int c0 = (int)(pos0 * ctas / cost), c1 = (int)((pos0 + nb - 1) * ctas / cost);
    if (c0 == c1)
        return;   // one CTA saw the whole segment and wrote it
    const int n = c1 - c0 + 1;
    if (n <= kMergeDirectParts) {
        // every thread loads the n partial LSEs (the same addresses) and its own
        // n partial outputs together, then combines them itself
        float lv[kMergeDirectParts], ov[kMergeDirectParts];
        const float *lsrc = p.ws_lse + (size_t)(u + c0) * G + g;
        const float *osrc = p.ws_o + ((size_t)(u + c0) * G + g) * D + d;
#pragma unroll
        for (int i = 0; i < kMergeDirectParts; ++i) {
            lv[i] = i < n ? lsrc[(size_t)i * G] : kNegInf;
            ov[i] = i < n ? osrc[(size_t)i * G * D] : 0.f;
        }
        float M = kNegInf;
#pragma unroll
        for (int i = 0; i < kMergeDirectParts; ++i) {
            if (i >= n)
                break;
            M = fmaxf(M, lv[i]);
        }
        if (M == kNegInf) {   // no partial saw a visible token
            store_o<D>(p.o, row, d, p.fuse_dh, part, 0.f);
            if (d == 0 && p.lse)
                p.lse[row] = kNegInf;
            return;
        }
        float S = 0.f;
#pragma unroll
        for (int i = 0; i < kMergeDirectParts; ++i) {
            if (i >= n)
                break;
            S += expf(lv[i] - M);
        }
        const float lse = M + logf(S);
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < kMergeDirectParts; ++i) {
            if (i >= n)
                break;
            acc += ov[i] * expf(lv[i] - lse);
        }
        store_o<D>(p.o, row, d, p.fuse_dh, part, acc);
        if (d == 0 && p.lse)
            p.lse[row] = lse;
        return;
    }
    float lmax = kNegInf;
    for (int i = d; i < n; i += D) {
        const float v = p.ws_lse[(size_t)(u + c0 + i) * G + g];
        s_w[i] = v;
        lmax = fmaxf(lmax, v);
    }
    // block max, then block sum of exp(lse_i - max): warp shuffles + shared memory
    __shared__ float s_red[D / 32];
#pragma unroll
    for (int off = 16; off; off >>= 1)
        lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, off));
    if ((d & 31) == 0)
        s_red[d >> 5] = lmax;
    __syncthreads();
    float M = s_red[0];
#pragma unroll
    for (int w = 1; w < D / 32; ++w)
        M = fmaxf(M, s_red[w]);
    if (M == kNegInf) {   // no partial saw a visible token (a new token before the cache's start)
        store_o<D>(p.o, row, d, p.fuse_dh, part, 0.f);
        if (d == 0 && p.lse)
            p.lse[row] = kNegInf;
        return;           // M is the same in every thread: the whole block leaves
    }
    __syncthreads();
    float sum = 0.f;
    for (int i = d; i < n; i += D)
        sum += expf(s_w[i] - M);
#pragma unroll
    for (int off = 16; off; off >>= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if ((d & 31) == 0)
        s_red[d >> 5] = sum;
    __syncthreads();
    if (d == 0) {
        float S = 0.f;
#pragma unroll
        for (int w = 0; w < D / 32; ++w)
            S += s_red[w];
        s_lse = M + logf(S);
    }
    __syncthreads();
    const float lse = s_lse;
    for (int i = d; i < n; i += D)
        s_w[i] = expf(s_w[i] - lse);
    __syncthreads();
    // several partial rows in flight per thread: the loop is latency-bound
    float acc = 0.f;
    const float *src = p.ws_o + ((size_t)(u + c0) * G + g) * D + d;
    const size_t stride = (size_t)G * D;
    int i = 0;
    for (; i + 4 <= n; i += 4) {
        const float x0 = src[(size_t)i * stride], x1 = src[(size_t)(i + 1) * stride];
        const float x2 = src[(size_t)(i + 2) * stride], x3 = src[(size_t)(i + 3) * stride];
        acc += x0 * s_w[i] + x1 * s_w[i + 1] + x2 * s_w[i + 2] + x3 * s_w[i + 3];
    }
    for (; i < n; ++i)
        acc += src[(size_t)i * stride] * s_w[i];
    store_o<D>(p.o, row, d, p.fuse_dh, part, acc);
    if (d == 0 && p.lse)
        p.lse[row] = lse;
}

// ------------------------------------------------------------------ merge of caller partials
//
// Sequence sharding: each of n partial sets holds, for every query row, the
// attention over one token range -- a normalised output O_s and its
// natural-log LSE lse_s (the Flash-Decoding section of the FlashAttention
// handbook page; the pass-2 merge of the sm120 article, section 2).  The
// merge is the same as merge_kernel's: M = max_s lse_s, LSE = M + ln sum_s
// exp(lse_s - M), O = sum_s O_s exp(lse_s - LSE); a set with lse_s = -inf saw
// no token and contributes nothing (handbook exercise 2), and a row that no
// set saw gets O = 0, LSE = -inf.

struct MergePartsParams {
    const float *o_parts;     // [n][rows][D]
    const float *lse_parts;   // [n][rows]
    float *o;                 // [rows][D]
    float *lse;               // [rows] or null
    int n, rows;
};

constexpr int kMergePartsWarps = 8;

// One warp per query row: lane l takes sets l, l + 32, .. for the LSE, and
// dims D/32 l .. D/32 (l + 1) - 1 of every set's output row (one coalesced
// row read per set).
template <int D>
__global__ void __launch_bounds__(kMergePartsWarps * 32) merge_parts_kernel(const __grid_constant__ MergePartsParams p)
{
    constexpr int kVec = D / 32;   // 2, 4 or 8 dims per lane
    static_assert(D % 64 == 0, "head_dim 64, 128 or 256");
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kMergePartsWarps + (threadIdx.x >> 5);
    if (row >= p.rows)
        return;   // warp-uniform
    const size_t rows = (size_t)p.rows;
    float M = kNegInf;
    for (int s = lane; s < p.n; s += 32)
        M = fmaxf(M, p.lse_parts[(size_t)s * rows + row]);
#pragma unroll
    for (int off = 16; off; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float *dst = p.o + (size_t)row * D + lane * kVec;
    if (M == kNegInf) {   // no set saw a token of this row
#pragma unroll
        for (int i = 0; i < kVec; ++i)
            dst[i] = 0.f;
        if (lane == 0 && p.lse)
            p.lse[row] = kNegInf;
        return;
    }
    float S = 0.f;
    for (int s = lane; s < p.n; s += 32)
        S += expf(p.lse_parts[(size_t)s * rows + row] - M);   // exp(-inf) = 0 for empty sets
#pragma unroll
    for (int off = 16; off; off >>= 1)
        S += __shfl_xor_sync(0xffffffffu, S, off);
    const float lse = M + logf(S);
    float acc[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i)
        acc[i] = 0.f;
    for (int s0 = 0; s0 < p.n; s0 += 32) {
        const int s = s0 + lane;
        const float w = s < p.n ? expf(p.lse_parts[(size_t)s * rows + row] - lse) : 0.f;
        const int cnt = min(32, p.n - s0);
        for (int i = 0; i < cnt; ++i) {
            const float wi = __shfl_sync(0xffffffffu, w, i);
            if (wi == 0.f)
                continue;   // warp-uniform: an empty set (or a weight below fp32's range)
            const float4 *src =
                reinterpret_cast<const float4 *>(p.o_parts + ((size_t)(s0 + i) * rows + row) * D + lane * kVec);
            if constexpr (kVec == 2) {
                const float2 x = *reinterpret_cast<const float2 *>(src);
                acc[0] += wi * x.x;
                acc[1] += wi * x.y;
            } else {
#pragma unroll
                for (int v = 0; v < kVec / 4; ++v) {
                    const float4 x = src[v];
                    acc[4 * v + 0] += wi * x.x;
                    acc[4 * v + 1] += wi * x.y;
                    acc[4 * v + 2] += wi * x.z;
                    acc[4 * v + 3] += wi * x.w;
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kVec; ++i)
        dst[i] = acc[i];
    if (lane == 0 && p.lse)
        p.lse[row] = lse;
}

}  // namespace fd
