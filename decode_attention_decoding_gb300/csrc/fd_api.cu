// fd_api.cu -- the C ABI of include/fd.h: argument checks, workspace layout,
// split planning, TMA descriptors and the two launches (split, then merge).
//
// Host side of "纯手搓 flash decoding sm120" section 1 (binding and launch
// code), re-planned for GB300: instead of a chunk size bucketed from a fixed
// SM count, the grid is one persistent CTA per SM and the device divides the
// KV tiles of all (request, kv head) pairs evenly among them (fd_sched.h),
// so the plan needs no host copy of the lengths and no per-call allocation.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fd.h"
#include "fd_launch.h"
#include "fd_sched.h"

namespace fd {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// Tensor-map element type and size of a K/V element type (kKv*).
static CUtensorMapDataType kv_map_type(int kv)
{
    return kv == kKvBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                         : (kv == kKvF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8);
}
static int kv_elem_bytes(int kv) { return kv_is_fp8(kv) ? 1 : 2; }

// A rank-3 view {head_dim, Hkv, rows} of a K or V tensor whose rows are
// (token, kv head) pairs of head_dim elements; each load is a box of
// box_rows tokens of one kv head: the whole row, or (swizzled) one 128-byte
// part of it with the 128-byte swizzle that the tensor-core consumers read.
static fd_status encode_kv_map(CUtensorMap *map, const void *base, int hkv, long long rows, int box_rows,
                        bool swizzled, int kv, int d)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return FD_ERR_CUDA;
    const int eb = kv_elem_bytes(kv);
    const cuuint64_t row_bytes = (cuuint64_t)eb * (cuuint64_t)d;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hkv, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {row_bytes, (cuuint64_t)hkv * row_bytes};
    const cuuint32_t box[3] = {(cuuint32_t)(swizzled ? 128 / eb : d), 1u, (cuuint32_t)box_rows};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = fn(map, kv_map_type(kv), 3,
                          const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzled ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FD_OK : FD_ERR_CUDA;
}

// A rank-4 view {128-byte part, rows, parts, Hkv} of the same tensor (a part
// is 64 16-bit elements or 128 FP8 codes), so that one box {part, box_rows,
// parts, 1} carries every 128-byte-swizzled part of box_rows rows of one kv
// head (laid out part by part in shared memory).
static fd_status encode_kv_map_4d(CUtensorMap *map, const void *base, int hkv, long long rows, int box_rows,
                           int kv, int d)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return FD_ERR_CUDA;
    const int eb = kv_elem_bytes(kv);
    const cuuint64_t row_bytes = (cuuint64_t)eb * (cuuint64_t)d;
    const cuuint32_t part = (cuuint32_t)(128 / eb), parts = (cuuint32_t)(row_bytes / 128);
    const cuuint64_t dims[4] = {part, (cuuint64_t)rows, parts, (cuuint64_t)hkv};
    const cuuint64_t strides[3] = {(cuuint64_t)hkv * row_bytes, 128u, row_bytes};
    const cuuint32_t box[4] = {part, (cuuint32_t)box_rows, parts, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = fn(map, kv_map_type(kv), 4,
                          const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FD_OK : FD_ERR_CUDA;
}

// A rank-2 view {d, rows} of a paged K or V pool whose rows are (page, token,
// kv head) triples of d elements, with one-row boxes and no swizzle: the
// CUDA-core consumers gather pages of 1 or 2 tokens four rows per load.
static fd_status encode_kv_rows_2d(CUtensorMap *map, const void *base, long long rows, int kv, int d)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return FD_ERR_CUDA;
    const cuuint64_t row_bytes = (cuuint64_t)kv_elem_bytes(kv) * (cuuint64_t)d;
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)d, 1u};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(map, kv_map_type(kv), 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FD_OK : FD_ERR_CUDA;
}

// K and V maps for a call: the tensor-core consumers prefer 4-D maps (one
// box per tile or page carries every swizzled part) and fall back to 3-D
// maps with one box per 64-dim part if the driver rejects the 4-D view.
fd_status encode_kv_maps(CUtensorMap *tmk, CUtensorMap *tmv, const void *k, const void *v, int hkv,
                         long long rows, int box_rows, bool mma, int kv, int d, SplitParams *sp)
{
    int rl = 0;
    while ((1 << rl) < box_rows)
        ++rl;
    sp->box4d = 0;
    sp->box_rows_log2 = 6;
    if (mma && !(sp->flags & FD_FLAG_NO_4D_BOXES) &&
        encode_kv_map_4d(tmk, k, hkv, rows, box_rows, kv, d) == FD_OK &&
        encode_kv_map_4d(tmv, v, hkv, rows, box_rows, kv, d) == FD_OK) {
        sp->box4d = 1;
        sp->box_rows_log2 = rl;
        return FD_OK;
    }
    fd_status st;
    if ((st = encode_kv_map(tmk, k, hkv, rows, box_rows, mma, kv, d)) != FD_OK ||
        (st = encode_kv_map(tmv, v, hkv, rows, box_rows, mma, kv, d)) != FD_OK)
        return st;
    return FD_OK;
}

constexpr size_t kMergeRoomBytes = 32u * 1024u;   // shared memory left beside a split CTA
constexpr size_t kShortCallInFlightBytes = 96u * 1024u;   // K/V in flight per CTA on short calls
constexpr int kPrefetchStages = 4;   // long calls: tiles prefetched before the dependency wait, in stages
constexpr int kPrefetchTiles = 24;    // at most this many tiles prefetched per CTA
constexpr size_t kShortCallBytes = 1u << 20;   // calls with less K/V per split CTA are short

// Shared-memory plan of the split kernel for the call's consumers, group,
// head_dim, K/V element size and batch; fills the offsets and stage count in
// sp and the byte size in launch.
fd_status plan_smem(const DeviceInfo &dev, int cons, int group, int d, int elem_bytes, int batch,
                    double tiles_per_cta, double kv_bytes_per_cta, SplitParams *sp, SplitLaunch *launch)
{
    const size_t stage_bytes = 2u * kTileTokens * (size_t)elem_bytes * (size_t)d;   // K and V tiles
    const size_t red = align_up((size_t)reduction_floats(cons, group, d) * sizeof(float), 16);
    const size_t prefix = align_up(2 * sizeof(int) * (size_t)(batch + 1), 16);   // tile prefix, non-empty requests
    const size_t misc = 128;   // abort flag, two scans' scratch
    const size_t per_stage_extra = 2 * 8 + kMetaInts * sizeof(int);   // 2 barriers + metadata
    const size_t tc = cons == kConsTc5 ? align_up((size_t)kTc5Bytes, 16) : 0;   // TMEM-score region
    const size_t fixed = 1024 /* alignment slack */ + tc + red + prefix + misc + 8 /* consumer barrier */;
    const size_t avail = (size_t)dev.smem_optin;
    if (avail <= fixed)
        return FD_ERR_UNSUPPORTED;
    int ns = (int)((avail - fixed) / (stage_bytes + per_stage_extra));
    if (ns > kMaxStages)
        ns = kMaxStages;
    // Leave room beside the split CTA for merge CTAs, which are launched early
    // (programmatic dependent launch) and then start the moment the split grid
    // ends -- unless that costs the pipeline its fourth stage.  Measured on
    // GB300: 32 KB free took the 1 GiB MHA call from 161.3 to 157.1 us and the
    // small calls 1.5-1.7% faster; with 64 KB stages (3 -> 2) it cost 4%.
    // The TMEM-score consumers hold each stage longer (the score MMAs, four
    // warps per tile) and keep the stage instead: 5 rather than 4 stages took
    // the FP8 calls 0.5-1% faster.
    {
        const size_t keep = kMergeRoomBytes;
        int ns_keep = ns;
        while (ns_keep > 2 && 1024 + fixed + ns_keep * (stage_bytes + per_stage_extra) + keep > avail)
            --ns_keep;
        if (ns_keep >= 4 && cons != kConsTc5)
            ns = ns_keep;
    }
    // A short call (few tiles per CTA) starts faster with less in flight: every
    // CTA's first tiles arrive sooner when the launch burst is smaller.
    // Measured on GB300 (MHA, 64 MiB, 13.5 tiles per CTA): 16.3 us with 5
    // stages, 15.6 us with 3; long calls keep their stages (3 cost the 1 GiB
    // call 3%).
    if (tiles_per_cta < kFuseMinTilesPerCta) {
        int ns_short = (int)(kShortCallInFlightBytes / stage_bytes);
        ns_short = ns_short < 2 ? 2 : ns_short;
        ns = ns < ns_short ? ns : ns_short;
    }
    if (ns < 2)
        return FD_ERR_UNSUPPORTED;
    sp->num_stages = ns;
    // L2 prefetch before the dependency wait, and when the merge lets the next
    // call launch.  Measured on GB300 (same box, us per call):
    //  * Long calls (over kShortCallBytes of K/V per CTA): the merge lets the
    //    next call launch at once, so its split CTAs take each SM as this
    //    call's CTA leaves it, and they prefetch kPrefetchStages stages' worth
    //    of tiles (at most kPrefetchTiles).  Without -> with 1, 2, 4, 8
    //    stages' worth: ragged GQA-4 (workload 3) 53.6 -> 50.2, 49.3, 48.2,
    //    49.1; MHA 1 GiB 159.0 -> 156.0, 155.5, 155.0, 155.8; paged GQA-4 313.2
    //    -> 310.7, 310.0, 309.3, 313.7; GQA-8 1 GiB 164.8 -> 164.2, 164.2,
    //    164.9, 168.7.
    //  * Short calls: their split CTAs fit two to an SM, so the next call's
    //    CTAs launched beside this call's a whole call early and their
    //    prefetches only competed with it (MHA 64 MiB: 16.7 -> 20.0 us).  The
    //    merge therefore lets the next call launch only once this call's split
    //    grid is complete, and one stage's worth is prefetched: 16.7 -> 15.7
    //    us (two stages 16.1, four 17.1); FP8 ragged GQA-4 35.3 -> 34.7.
    const bool short_call = kv_bytes_per_cta < (double)kShortCallBytes;
    launch->late_trigger = short_call ? 1 : 0;
    int pf = short_call ? ns : kPrefetchStages * ns;
    pf = pf < kPrefetchTiles ? pf : kPrefetchTiles;
    sp->prefetch_tiles = (sp->flags & FD_FLAG_NO_PREFETCH) ? 0 : pf;
    sp->off_tc = (uint32_t)(ns * stage_bytes);   // 1024-byte aligned: stages are multiples of 1 KB
    sp->off_red = (uint32_t)(sp->off_tc + tc);
    sp->off_prefix = (uint32_t)(sp->off_red + red);
    sp->off_bar = (uint32_t)(sp->off_prefix + prefix);
    sp->off_meta = (uint32_t)(sp->off_bar + (2 * ns + 1) * 8);
    sp->off_misc = (uint32_t)(sp->off_meta + ns * kMetaInts * sizeof(int));
    launch->smem_bytes = 1024 + sp->off_misc + misc;
    launch->smem_optin = (size_t)dev.smem_optin;
    return launch->smem_bytes <= avail ? FD_OK : FD_ERR_UNSUPPORTED;
}

}  // namespace fd

namespace {

using namespace fd;

constexpr int kVersion = 10400;   // 1.4.0
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;

// The one piece of state kept across calls: a cache of device properties.
std::mutex g_dev_mu;
DeviceInfo g_dev[64];
bool g_dev_ok[64] = {};

fd_status device_info(DeviceInfo *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return FD_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_ok[dev]) {
        DeviceInfo d;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return FD_ERR_CUDA;
        g_dev[dev] = d;
        g_dev_ok[dev] = true;
    }
    *out = g_dev[dev];
    return FD_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Query columns of a kv head (group x new tokens): the kernels are built for
// 1, 2, 4, 8 or 16 columns and pad the rest.
int pow2_columns(int cols) { return cols <= 1 ? 1 : cols <= 2 ? 2 : cols <= 4 ? 4 : cols <= 8 ? 8 : 16; }

int q_len_of(const fd_options *opts) { return opts && opts->q_len > 0 ? opts->q_len : 1; }

bool supported_head_dim(int d) { return d == 64 || d == 128 || d == 256; }

// fd_options fields in range; FP8 scales must be finite and positive (0 = 1).
bool options_valid(const fd_options *opts)
{
    if (!opts)
        return true;
    auto scale_ok = [](float x) { return x == 0.f || (x > 0.f && x < __builtin_huge_valf()); };
    return opts->num_ctas >= 0 && opts->num_ctas <= kMaxCtas && opts->dtype >= 0 && opts->dtype <= 1 &&
           opts->kv_dtype >= FD_KV_AS_Q && opts->kv_dtype <= FD_KV_FP8_E5M2 && scale_ok(opts->k_scale) &&
           scale_ok(opts->v_scale) && opts->q_len >= 0;
}

// Checks shared by both entry points.  Returns FD_OK or the status to report.
fd_status check_common(const void *q, const float *o, const void *ws, int batch, int hq, int hkv,
                       int head_dim, const fd_options *opts)
{
    if (batch < 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0)
        return FD_ERR_INVALID_ARG;
    if (!q || !o || !ws)
        return FD_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(o, 16) || !aligned(ws, 256))
        return FD_ERR_INVALID_ARG;
    if (!options_valid(opts))
        return FD_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim) || (long long)(hq / hkv) * q_len_of(opts) > kMaxColumns ||
        batch > kMaxBatch)
        return FD_ERR_UNSUPPORTED;
    return FD_OK;
}

// Bytes of one K/V element under these options.
int kv_elem_bytes_of(const fd_options *opts)
{
    const int kvd = opts ? opts->kv_dtype : FD_KV_AS_Q;
    return (kvd == FD_KV_FP8_E4M3 || kvd == FD_KV_FP8_E5M2) ? 1 : 2;
}

// More than 8 query columns per kv head run on the tensor-core consumers only:
// no FD_FLAG_CUDA_CORES, and a row of at least 128 bytes -- directly, or by
// pairing two kv heads (an FP8 head of 64 dims; pairing needs pages of at
// least 8 tokens).  Host-only; FD_OK or FD_ERR_UNSUPPORTED.
fd_status check_columns(int hq, int hkv, int head_dim, int page_size, const fd_options *opts)
{
    if ((long long)(hq / hkv) * q_len_of(opts) <= kMaxColumnsCudaCores)
        return FD_OK;
    const unsigned flags = opts ? opts->flags : 0u;
    if (flags & FD_FLAG_CUDA_CORES)
        return FD_ERR_UNSUPPORTED;
    if (head_dim * kv_elem_bytes_of(opts) >= 128)
        return FD_OK;
    const bool pairable = 2 * head_dim <= 256 && hkv % 2 == 0 && !(flags & FD_FLAG_NO_HEAD_FUSION) &&
                          (page_size == 0 || page_size >= 8);
    return pairable ? FD_OK : FD_ERR_UNSUPPORTED;
}

struct CallPlan {
    SplitParams sp;
    MergeParams mp;
    SplitLaunch launch;
    int group;        // split kernel's columns per warp group (template G)
    int head_dim;     // split kernel's row dims (template D)
    int cons;         // consumer kind (kCons*)
    bool mma;         // tensor-core consumers (either kind)
    int merge_group;  // merge kernel's columns per launch head
    int merge_dim;    // merge kernel's dims per column
    int kv;           // K/V element type (kKv*): bf16, fp16 (q of the same type) or FP8
    bool cp_async;    // paged, pages under 8 tokens, tensor cores: rows copied with cp.async
    bool two_per_sm;  // short call on the default grid: two split CTAs per SM if both fit
};

// Tensor-core consumers serve GQA groups; a row must fill at least one
// 128-byte swizzled part.  Pages of 8 tokens or more arrive by TMA (every
// page box starts on a 1 KB swizzle boundary); smaller pages are copied row
// by row with cp.async into the same swizzled layout.
bool use_mma(int group, int row_bytes, const fd_options *opts)
{
    if (opts && (opts->flags & FD_FLAG_CUDA_CORES))
        return false;
    return group >= 2 && row_bytes >= 128;
}

// Fusion pays where a kv head's TMA rows are short (under 256 bytes: 64
// 16-bit dims or an FP8 row of up to 128 dims, or page boxes under 64
// tokens) and the call is long enough for the
// wider tiles: measured on GB300, it lost up to a quarter of the time on
// calls of under ~24 tiles per CTA (larger tiles, fewer of them per CTA,
// twice the merge width) and gained 10-85% above that on such rows: hence
// the kFuseMinTilesPerCta threshold (fd_launch.h).
//
// Kv heads fused into one launch head, on the tensor-core path only, for
// short rows and at least kFuseMinTilesPerCta (estimated) tiles per CTA
// unless FD_FLAG_FUSE_HEADS forces it:
//   * 2 (paired heads: each warp of a pair takes one of the two heads, up to
//     16 query columns each) when 2 x head_dim <= 256 and Hkv is even --
//     unless the paired row is still under 256 bytes and 4 heads fit: then
//   * 4 (one shared 256-dim row; 4 x columns <= 8, 4 | Hkv);
//   * 1 otherwise.
int fuse_factor(int cols, int hkv, int head_dim, int elem_bytes, int page_size, double tiles_per_cta,
                const fd_options *opts)
{
    if (opts && (opts->flags & (FD_FLAG_CUDA_CORES | FD_FLAG_NO_HEAD_FUSION)))
        return 1;
    if (page_size != 0 && page_size < 8)
        return 1;
    const bool short_rows = head_dim * elem_bytes < 256 || (page_size > 0 && page_size < kTileTokens);
    // over 8 columns need the tensor-core consumers, whose rows span at least
    // 128 bytes: a shorter row (an FP8 head of 64 dims) is paired whenever it can be
    const bool needed = cols > kMaxColumnsCudaCores && head_dim * elem_bytes < 128;
    // One column per kv head of an FP8 cache with 128 dims would run on CUDA
    // cores unfused; paired, it takes the tensor cores, which measured faster
    // on GB300 at any length (MHA over a 32 MiB E4M3 cache: 16.3 -> 14.1 us,
    // at half that length 12.9 -> 12.2 us).
    const bool fp8_single = elem_bytes == 1 && head_dim == 128 && cols == 1;
    const bool forced = (opts && (opts->flags & FD_FLAG_FUSE_HEADS)) || needed || fp8_single;
    if (!forced && (!short_rows || tiles_per_cta < kFuseMinTilesPerCta))
        return 1;
    const bool four = 4 * head_dim <= 256 && 4 * cols <= 8 && hkv % 4 == 0;
    const bool two = 2 * head_dim <= 256 && cols <= kMaxColumns && hkv % 2 == 0;
    if (two && (2 * head_dim * elem_bytes >= 256 || !four))
        return 2;
    return four ? 4 : 1;
}

// The cache positions a call covers: the whole cache (on = false), or the
// range [begin, end) of the partial entry points, whose layout holds
// position begin of each request at its row 0.
struct KvRange {
    bool on;
    int begin, end;
    // tokens of a request of length L that the call covers
    long long tokens(long long L) const
    {
        if (!on)
            return L;
        const long long e = L < end ? L : end;
        return e > begin ? e - begin : 0;
    }
};

// KV tiles of a call (unfused): from the host copy of the lengths when the
// caller passes one, else every request at the capacity `span`.
long long estimate_tiles(const int32_t *seq_lens_host, int batch, int hkv, long long span, const KvRange &r)
{
    long long tiles = 0;
    if (seq_lens_host)
        for (int b = 0; b < batch; ++b)
            tiles += ceil_div(r.tokens(seq_lens_host[b]), (long long)kTileTokens);
    else
        tiles = (long long)batch * ceil_div(span, (long long)kTileTokens);
    return tiles * hkv;
}

// Host copy of the lengths against the layout's capacity: every L_b >= 0 and
// the tokens the call covers at most cap.
bool host_lens_valid(const int32_t *seq_lens_host, int batch, long long cap, const KvRange &r)
{
    if (seq_lens_host)
        for (int b = 0; b < batch; ++b)
            if (seq_lens_host[b] < 0 || r.tokens(seq_lens_host[b]) > cap)
                return false;
    return true;
}

// Workspace for every launch shape a call of this shape may take (fused or
// not), with the launch's column count rounded up as the kernels pad it.
size_t workspace_bytes_needed(int batch, int hq, int hkv, int head_dim, int q_len)
{
    const int cols = (hq / hkv) * q_len;
    size_t need = workspace_layout(batch, hkv, pow2_columns(cols), head_dim).total;
    auto take = [&](size_t t) { need = t > need ? t : need; };
    if (2 * head_dim <= 256 && hkv % 2 == 0)   // paired heads: both heads' columns
        take(workspace_layout(batch, hkv / 2, 2 * pow2_columns(cols), head_dim).total);
    if (4 * head_dim <= 256 && 4 * cols <= 8 && hkv % 4 == 0)   // four heads in one row
        take(workspace_layout(batch, hkv / 4, pow2_columns(4 * cols), 4 * head_dim).total);
    return need;
}

fd_status fill_plan(CallPlan *cp, const DeviceInfo &dev, const void *q, const int32_t *seq_lens_dev,
                    const int32_t *block_table, int batch, int hq, int hkv, int cap, int s_max,
                    int head_dim, int page_size, int max_blocks, int num_pages, float scale, float *o,
                    float *lse, void *workspace, long long est_tiles, const KvRange &range,
                    const fd_options *opts, fd_stream_t stream)
{
    int num_ctas = opts && opts->num_ctas > 0 ? opts->num_ctas : dev.sms;
    if (num_ctas > kMaxCtas)
        return FD_ERR_INVALID_ARG;
    const bool q_f16 = opts && opts->dtype == FD_DTYPE_F16;
    const int kv_dtype = opts ? opts->kv_dtype : FD_KV_AS_Q;
    const int kv = kv_dtype == FD_KV_FP8_E4M3 ? kKvE4m3
                   : kv_dtype == FD_KV_FP8_E5M2 ? kKvE5m2 : (q_f16 ? kKvF16 : kKvBf16);
    const int eb = kv_elem_bytes(kv);
    // Launch shape: F fused kv heads of head_dim dims become one head of
    // F * head_dim dims.  A kv head's query columns (q_len x group) are padded
    // to 1, 2, 4, 8 or 16.  Paired heads (F = 2) keep each head's columns in its
    // own warp of a pair (2 x padded columns in all, head_dim dims each); four
    // fused heads share one set of 4 x columns over 4 x head_dim dims.
    const int real_group = hq / hkv;
    const int q_len = q_len_of(opts);
    const int cols = real_group * q_len;
    const int fuse = fuse_factor(cols, hkv, head_dim, eb, page_size, (double)est_tiles / num_ctas, opts);
    const bool paired = fuse == 2;
    const int group = paired ? pow2_columns(cols) : pow2_columns(fuse * cols);
    const int slots = paired ? 2 * group : group;        // column slots of a launch head
    const int d = fuse * head_dim;
    const int merge_dim = paired ? head_dim : d;
    hkv /= fuse;
    const WorkspaceLayout wl = workspace_layout(batch, hkv, slots, merge_dim);
    uint8_t *ws = static_cast<uint8_t *>(workspace);

    SplitParams &sp = cp->sp;
    std::memset(&sp, 0, sizeof sp);
    sp.q = static_cast<const uint16_t *>(q);
    sp.seq_lens = seq_lens_dev;
    sp.block_table = block_table;
    sp.o = o;
    sp.lse = lse;
    sp.ws_o = reinterpret_cast<float *>(ws + wl.o_off);
    sp.ws_lse = reinterpret_cast<float *>(ws + wl.lse_off);
    sp.ws_prefix = reinterpret_cast<int32_t *>(ws + wl.prefix_off);
    sp.ws_err = reinterpret_cast<unsigned int *>(ws + wl.err_off);
    sp.batch = batch;
    sp.hq = hq;
    sp.hkv = hkv;
    sp.cap = cap;
    sp.s_max = s_max;
    sp.page_size = page_size;
    sp.page_log2 = 0;
    while (page_size > 0 && page_size < kTileTokens && (1 << sp.page_log2) < page_size)
        ++sp.page_log2;
    sp.max_blocks = max_blocks;
    sp.num_pages = num_pages;
    // An FP8 cache's k_scale multiplies every score: fold it into the scale.
    const float k_scale = kv_is_fp8(kv) && opts && opts->k_scale != 0.f ? opts->k_scale : 1.f;
    const float v_scale = kv_is_fp8(kv) && opts && opts->v_scale != 0.f ? opts->v_scale : 1.f;
    sp.scale_log2 = scale * k_scale * 1.4426950408889634f;
    sp.v_scale = v_scale;
    sp.q_f16 = q_f16 ? 1 : 0;
    sp.timeout_ns = opts && opts->wait_timeout_ns ? opts->wait_timeout_ns : kDefaultTimeoutNs;
    sp.flags = opts ? opts->flags : 0u;
    sp.fuse_dh = fuse == 4 ? head_dim : 0;   // only a shared 4-head row splits a column's dims
    sp.fuse_f = fuse;
    sp.q_len = q_len;
    sp.seg_cost = kSegCostTiles;
    sp.range_on = range.on ? 1 : 0;
    sp.kv_begin = range.on ? range.begin : 0;
    sp.kv_end = range.on ? range.end : 0;
    sp.g_real = real_group;
    sp.n_cols = slots;
    // column slot n = (part, new token i, query head g), part-major; each part
    // holds `cols` real columns, in a block of `group` slots when paired
    const int per_part = paired ? group : cols;
    for (int n = 0; n < kMaxColumnSlots; ++n) {
        const int part = n / per_part, c = n % per_part;
        const bool real = n < slots && part < fuse && c < cols;
        sp.col_code[n] = real ? (c / real_group) | (part << 4) | ((c % real_group) << 8) : -1;
    }

    cp->group = group;
    cp->head_dim = d;
    cp->kv = kv;
    cp->cp_async = false;   // the paged entry point sets it for pages under 8 tokens
    cp->merge_group = slots;
    cp->merge_dim = merge_dim;
    cp->mma = paired || use_mma(group, eb * d, opts);
    cp->cons = paired ? kConsMmaPair : (cp->mma ? kConsMma : kConsCudaCores);
    // Scores by tcgen05 MMAs into TMEM.  Their K operand is the tile's 128
    // swizzled rows as 64-row boxes lay them out (head 0's 64 rows, then
    // head 1's): contiguous caches and pages of 64 tokens or more.  Smaller
    // pages interleave the heads page by page.  By default for up to
    // kTc5DefaultColumns columns per kv head: their consumers' softmax work
    // grows with the columns, the warp MMAs' does not (measured on GB300:
    // 1 and 4 columns faster, 8 slower); and for calls of at least
    // kFuseMinTilesPerCta (paired) tiles per CTA, where their fixed costs
    // (TMEM, the score round trip) amortise (MHA over a 32 MiB E4M3 cache,
    // 6.7 tiles per CTA: 14.1 us with warp MMAs, 16.3 with them).
    const bool tc5_shape = paired && kv_is_fp8(kv) && d == 256 && group <= 8 &&
                           (page_size == 0 || page_size >= kTileTokens);
    const bool tc5_default = group <= kTc5DefaultColumns && est_tiles / (2.0 * num_ctas) >= kFuseMinTilesPerCta;
    if (tc5_shape && !(sp.flags & FD_FLAG_NO_TMEM_SCORES) && (tc5_default || (sp.flags & FD_FLAG_TMEM_SCORES)))
        cp->cons = kConsTc5;
    if (fuse > 1 && !use_mma(2, eb * d, opts))
        return FD_ERR_UNSUPPORTED;   // fusion is defined for the tensor-core consumers only
    if (!cp->mma && group > kMaxColumnsCudaCores)
        return FD_ERR_UNSUPPORTED;   // over 8 columns need the tensor-core consumers
    cp->launch.grid = num_ctas;
    cp->launch.stream = reinterpret_cast<cudaStream_t>(stream);
    cp->launch.blocks_per_sm = nullptr;
    const double kv_bytes = (double)est_tiles * 2.0 * kTileTokens * head_dim * eb;   // unfused tiles
    fd_status st = plan_smem(dev, cp->cons, group, d, eb, batch, (double)est_tiles / num_ctas,
                             kv_bytes / num_ctas, &sp, &cp->launch);
    if (st != FD_OK)
        return st;

    MergeParams &mp = cp->mp;
    std::memset(&mp, 0, sizeof mp);
    mp.o = o;
    mp.lse = lse;
    mp.ws_o = sp.ws_o;
    mp.ws_lse = sp.ws_lse;
    mp.ws_prefix = sp.ws_prefix;
    mp.batch = batch;
    mp.hq = hq;
    mp.hkv = hkv;
    mp.num_ctas = num_ctas;
    mp.fuse_dh = sp.fuse_dh;
    mp.fuse_f = sp.fuse_f;
    mp.q_len = sp.q_len;
    mp.g_real = sp.g_real;
    mp.n_cols = sp.n_cols;
    std::memcpy(mp.col_code, sp.col_code, sizeof mp.col_code);
    mp.seq_lens = seq_lens_dev;
    mp.cap = cap;
    mp.late_trigger = cp->launch.late_trigger;
    mp.seg_cost = sp.seg_cost;
    cp->two_per_sm = cp->launch.late_trigger && !(opts && opts->num_ctas > 0) && 2 * num_ctas <= kMaxCtas;
    mp.range_on = sp.range_on;
    mp.kv_begin = sp.kv_begin;
    mp.kv_end = sp.kv_end;
    return FD_OK;
}

// Record a caller's timing event on `stream`.  Inside a stream capture the
// record becomes an event node of the graph (cudaEventRecordExternal), so
// every replay of the graph records it.
bool record_event(cudaEvent_t ev, cudaStream_t stream)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess)
        return false;
    const cudaError_t e = cs == cudaStreamCaptureStatusActive
                              ? cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal)
                              : cudaEventRecord(ev, stream);
    return e == cudaSuccess;
}

fd_status run(CallPlan cp, bool paged, const CUtensorMap &tmk, const CUtensorMap &tmv, const fd_options *opts)
{
    // A short call's CTAs each stream less than the tail of the call lasts:
    // when two split CTAs fit on an SM (shared memory and registers), launch
    // two per SM, so that each CTA's share, and the spread of the last tiles,
    // halves.  Measured on GB300 (MHA 64 MiB, CUDA-core consumers, 76
    // registers): 15.9 us with one CTA per SM, 15.3 with two.
    if (cp.two_per_sm) {
        int fit = 0;
        SplitLaunch q = cp.launch;
        q.blocks_per_sm = &fit;
        if (launch_split(paged, cp.kv, cp.head_dim, cp.cons, cp.group, cp.cp_async, cp.sp, tmk, tmv, q) ==
                cudaSuccess &&
            fit >= 2) {
            cp.launch.grid *= 2;
            cp.mp.num_ctas = cp.launch.grid;
        }
    }
    cudaStream_t stream = cp.launch.stream;
    cudaEvent_t ev0 = opts ? static_cast<cudaEvent_t>(opts->split_start_event) : nullptr;
    cudaEvent_t ev1 = opts ? static_cast<cudaEvent_t>(opts->split_end_event) : nullptr;
    if (ev0 && !record_event(ev0, stream))
        return FD_ERR_CUDA;
    cudaError_t e = launch_split(paged, cp.kv, cp.head_dim, cp.cons, cp.group, cp.cp_async, cp.sp, tmk, tmv,
                                 cp.launch);
    if (e != cudaSuccess)
        return FD_ERR_CUDA;
    if (ev1 && !record_event(ev1, stream))
        return FD_ERR_CUDA;
    e = launch_merge(cp.merge_group, cp.merge_dim, cp.mp, cp.sp.batch * cp.sp.hkv, stream);
    if (e != cudaSuccess)
        return FD_ERR_CUDA;
    return FD_OK;
}

// A partial call's range: 0 <= begin <= end, and the position of the layout's
// last row (begin + capacity) inside int32.
bool range_valid(int begin, int end, long long cap)
{
    return begin >= 0 && end >= begin && (long long)begin + cap < (1ll << 31);
}

fd_status decode_contiguous(const void *q, const void *k, const void *v, const int32_t *seq_lens_dev,
                            const int32_t *seq_lens_host, int batch, int num_q_heads, int num_kv_heads,
                            int head_dim, int s_max, const KvRange &range, float scale, float *o, float *lse,
                            void *workspace, size_t workspace_bytes, const fd_options *opts, fd_stream_t stream)
{
    fd_status st = check_common(q, o, workspace, batch, num_q_heads, num_kv_heads, head_dim, opts);
    if (st != FD_OK)
        return st;
    if (s_max < 0 || !k || !v || !aligned(k, 16) || !aligned(v, 16) || (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    if (!host_lens_valid(seq_lens_host, batch, s_max, range))
        return FD_ERR_INVALID_ARG;
    if (!options_valid(opts))
        return FD_ERR_INVALID_ARG;
    if ((st = check_columns(num_q_heads, num_kv_heads, head_dim, 0, opts)) != FD_OK)
        return st;
    if ((long long)batch * s_max >= (1ll << 31) ||
        (long long)num_kv_heads * batch * ceil_div(s_max, kTileTokens) >= (1ll << 31))
        return FD_ERR_UNSUPPORTED;
    if (workspace_bytes <
        fd_workspace_size_q(batch, num_q_heads, num_kv_heads, head_dim, s_max, 0, q_len_of(opts)))
        return FD_ERR_WORKSPACE_TOO_SMALL;
    if (batch == 0)
        return FD_OK;

    DeviceInfo dev;
    if ((st = device_info(&dev)) != FD_OK)
        return st;
    CallPlan cp;
    st = fill_plan(&cp, dev, q, seq_lens_dev, nullptr, batch, num_q_heads, num_kv_heads, s_max, s_max,
                   head_dim, 0, 0, 0, scale, o, lse, workspace,
                   estimate_tiles(seq_lens_host, batch, num_kv_heads, s_max, range), range, opts, stream);
    if (st != FD_OK)
        return st;
    alignas(64) CUtensorMap tmk, tmv;
    const long long rows = (long long)batch * (s_max > 0 ? s_max : 1);
    if ((st = encode_kv_maps(&tmk, &tmv, k, v, cp.sp.hkv, rows, kTileTokens, cp.mma, cp.kv, cp.head_dim,
                             &cp.sp)) != FD_OK)
        return st;
    return run(cp, false, tmk, tmv, opts);
}

fd_status decode_paged(const void *q, const void *k_pages, const void *v_pages, const int32_t *block_table,
                       int max_blocks_per_seq, const int32_t *seq_lens_dev, const int32_t *seq_lens_host, int batch,
                       int num_q_heads, int num_kv_heads, int head_dim, int page_size, int num_pages,
                       const KvRange &range, float scale, float *o, float *lse, void *workspace,
                       size_t workspace_bytes, const fd_options *opts, fd_stream_t stream)
{
    fd_status st = check_common(q, o, workspace, batch, num_q_heads, num_kv_heads, head_dim, opts);
    if (st != FD_OK)
        return st;
    if (!k_pages || !v_pages || !block_table || !seq_lens_dev || !aligned(k_pages, 16) ||
        !aligned(v_pages, 16) || !aligned(block_table, 4) || (lse && !aligned(lse, 4)) ||
        max_blocks_per_seq <= 0 || page_size <= 0 || num_pages <= 0)
        return FD_ERR_INVALID_ARG;
    if (!((page_size < kTileTokens && kTileTokens % page_size == 0) || page_size % kTileTokens == 0))
        return FD_ERR_UNSUPPORTED;
    if (!options_valid(opts))
        return FD_ERR_INVALID_ARG;
    // A page's TMA box lands at a multiple of its own size in shared memory,
    // and tensor copies need 128-byte aligned destinations: pages under 64
    // tokens must hold at least 128 bytes per kv head (only an FP8 cache with
    // head_dim 64 and one-token pages falls short).
    if (page_size < kTileTokens && page_size * head_dim * kv_elem_bytes_of(opts) < 128)
        return FD_ERR_UNSUPPORTED;
    if ((st = check_columns(num_q_heads, num_kv_heads, head_dim, page_size, opts)) != FD_OK)
        return st;
    const long long cap = (long long)max_blocks_per_seq * page_size;
    if (cap >= (1ll << 31) || (long long)num_pages * page_size >= (1ll << 31) ||
        (long long)num_kv_heads * batch * ((cap + kTileTokens - 1) / kTileTokens) >= (1ll << 31))
        return FD_ERR_UNSUPPORTED;
    if (!host_lens_valid(seq_lens_host, batch, cap, range))
        return FD_ERR_INVALID_ARG;
    if (!options_valid(opts))
        return FD_ERR_INVALID_ARG;
    if (workspace_bytes < fd_workspace_size_q(batch, num_q_heads, num_kv_heads, head_dim, (int)cap,
                                              page_size, q_len_of(opts)))
        return FD_ERR_WORKSPACE_TOO_SMALL;
    if (batch == 0)
        return FD_OK;

    DeviceInfo dev;
    if ((st = device_info(&dev)) != FD_OK)
        return st;
    CallPlan cp;
    st = fill_plan(&cp, dev, q, seq_lens_dev, block_table, batch, num_q_heads, num_kv_heads, (int)cap, 0,
                   head_dim, page_size, max_blocks_per_seq, num_pages, scale, o, lse, workspace,
                   estimate_tiles(seq_lens_host, batch, num_kv_heads, cap, range), range, opts, stream);
    if (st != FD_OK)
        return st;
    alignas(64) CUtensorMap tmk, tmv;
    const long long rows = (long long)num_pages * page_size;
    // Pages under 8 tokens on the tensor-core consumers: the producer copies
    // rows with cp.async into the swizzled layout; no tensor maps.
    cp.cp_async = false;
    if (cp.mma && page_size < 8) {
        if (rows * cp.sp.hkv >= (1ll << 32))   // pool rows must fit the producer's 32-bit row index
            return FD_ERR_UNSUPPORTED;
        std::memset(&tmk, 0, sizeof tmk);
        std::memset(&tmv, 0, sizeof tmv);
        cp.cp_async = true;
        cp.sp.k_pool = static_cast<const uint8_t *>(k_pages);
        cp.sp.v_pool = static_cast<const uint8_t *>(v_pages);
        cp.sp.box4d = 0;
        cp.sp.box_rows_log2 = 6;   // the consumers' layout: one 64-row box per 128-byte part
        return run(cp, true, tmk, tmv, opts);
    }
    // Pages of 1 or 2 tokens (CUDA-core consumers): gather a tile's rows four
    // per load when the (page, token, kv head) row index fits int32; one box
    // per page otherwise, with FD_FLAG_NO_GATHER, or if the driver rejects the
    // view.  The TMA unit's cost per load, not its size, bounds these pages:
    // measured on GB300, gathering ran one-token pages 2.2-2.5x and two-token
    // pages 1.4x faster; four-token pages carry four rows per box already.
    cp.sp.gather4 = 0;
    if (!cp.mma && page_size <= 2 && rows * cp.sp.hkv < (1ll << 31) && !(cp.sp.flags & FD_FLAG_NO_GATHER) &&
        encode_kv_rows_2d(&tmk, k_pages, rows * cp.sp.hkv, cp.kv, cp.head_dim) == FD_OK &&
        encode_kv_rows_2d(&tmv, v_pages, rows * cp.sp.hkv, cp.kv, cp.head_dim) == FD_OK) {
        cp.sp.gather4 = 1;
        return run(cp, true, tmk, tmv, opts);
    }
    const int box = page_size < kTileTokens ? page_size : kTileTokens;
    if ((st = encode_kv_maps(&tmk, &tmv, k_pages, v_pages, cp.sp.hkv, rows, box, cp.mma, cp.kv,
                             cp.head_dim, &cp.sp)) != FD_OK)
        return st;
    return run(cp, true, tmk, tmv, opts);
}

}  // namespace

extern "C" {

size_t fd_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim, int max_kv_len,
                         int page_size)
{
    return fd_workspace_size_q(batch, num_q_heads, num_kv_heads, head_dim, max_kv_len, page_size, 1);
}

size_t fd_workspace_size_q(int batch, int num_q_heads, int num_kv_heads, int head_dim, int max_kv_len,
                           int page_size, int q_len)
{
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_kv_len < 0 ||
        page_size < 0 || num_q_heads % num_kv_heads != 0 || q_len < 1 ||
        (long long)(num_q_heads / num_kv_heads) * q_len > kMaxColumns)
        return 0;
    return workspace_bytes_needed(batch, num_q_heads, num_kv_heads, head_dim, q_len);
}

fd_status fd_workspace_init(void *workspace, size_t workspace_bytes, fd_stream_t stream)
{
    if (!workspace || workspace_bytes < 256 || !aligned(workspace, 256))
        return FD_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? FD_OK
               : FD_ERR_CUDA;
}

fd_status fd_decode(const void *q, const void *k, const void *v, const int32_t *seq_lens_dev,
                    const int32_t *seq_lens_host, int batch, int num_q_heads, int num_kv_heads,
                    int head_dim, int s_max, float scale, float *o, float *lse, void *workspace,
                    size_t workspace_bytes, const fd_options *opts, fd_stream_t stream)
{
    return decode_contiguous(q, k, v, seq_lens_dev, seq_lens_host, batch, num_q_heads, num_kv_heads, head_dim,
                             s_max, KvRange{false, 0, 0}, scale, o, lse, workspace, workspace_bytes, opts, stream);
}

fd_status fd_decode_partial(const void *q, const void *k, const void *v, const int32_t *seq_lens_dev,
                            const int32_t *seq_lens_host, int batch, int num_q_heads, int num_kv_heads,
                            int head_dim, int s_max, int kv_begin, int kv_end, float scale, float *o_part,
                            float *lse_part, void *workspace, size_t workspace_bytes, const fd_options *opts,
                            fd_stream_t stream)
{
    if (!range_valid(kv_begin, kv_end, s_max) || !lse_part)
        return FD_ERR_INVALID_ARG;
    return decode_contiguous(q, k, v, seq_lens_dev, seq_lens_host, batch, num_q_heads, num_kv_heads, head_dim,
                             s_max, KvRange{true, kv_begin, kv_end}, scale, o_part, lse_part, workspace,
                             workspace_bytes, opts, stream);
}

fd_status fd_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                          const int32_t *block_table, int max_blocks_per_seq,
                          const int32_t *seq_lens_dev, const int32_t *seq_lens_host, int batch,
                          int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                          int num_pages, float scale, float *o, float *lse, void *workspace,
                          size_t workspace_bytes, const fd_options *opts, fd_stream_t stream)
{
    return decode_paged(q, k_pages, v_pages, block_table, max_blocks_per_seq, seq_lens_dev, seq_lens_host, batch,
                        num_q_heads, num_kv_heads, head_dim, page_size, num_pages, KvRange{false, 0, 0}, scale, o,
                        lse, workspace, workspace_bytes, opts, stream);
}

fd_status fd_decode_paged_partial(const void *q, const void *k_pages, const void *v_pages,
                                  const int32_t *block_table, int max_blocks_per_seq,
                                  const int32_t *seq_lens_dev, const int32_t *seq_lens_host, int batch,
                                  int num_q_heads, int num_kv_heads, int head_dim, int page_size, int num_pages,
                                  int kv_begin, int kv_end, float scale, float *o_part, float *lse_part,
                                  void *workspace, size_t workspace_bytes, const fd_options *opts,
                                  fd_stream_t stream)
{
    if (max_blocks_per_seq <= 0 || page_size <= 0 ||
        !range_valid(kv_begin, kv_end, (long long)max_blocks_per_seq * page_size) || !lse_part)
        return FD_ERR_INVALID_ARG;
    return decode_paged(q, k_pages, v_pages, block_table, max_blocks_per_seq, seq_lens_dev, seq_lens_host, batch,
                        num_q_heads, num_kv_heads, head_dim, page_size, num_pages, KvRange{true, kv_begin, kv_end},
                        scale, o_part, lse_part, workspace, workspace_bytes, opts, stream);
}

fd_status fd_merge_partials(const float *o_parts, const float *lse_parts, int num_parts, int rows, int head_dim,
                            float *o, float *lse, fd_stream_t stream)
{
    if (num_parts < 1 || rows < 0 || !o_parts || !lse_parts || !o || !aligned(o_parts, 16) ||
        !aligned(lse_parts, 4) || !aligned(o, 16) || (lse && !aligned(lse, 4)))
        return FD_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim))
        return FD_ERR_UNSUPPORTED;
    MergePartsParams mp;
    mp.o_parts = o_parts;
    mp.lse_parts = lse_parts;
    mp.o = o;
    mp.lse = lse;
    mp.n = num_parts;
    mp.rows = rows;
    return launch_merge_parts(head_dim, mp, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FD_OK
                                                                                                   : FD_ERR_CUDA;
}

fd_status fd_get_device_error(void *workspace, fd_stream_t stream)
{
    if (!workspace || !aligned(workspace, 256))
        return FD_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return FD_ERR_CUDA;
    if (word != 0 && (cudaMemsetAsync(workspace, 0, sizeof word, s) != cudaSuccess ||
                      cudaStreamSynchronize(s) != cudaSuccess))
        return FD_ERR_CUDA;
    if (word & kErrTimeout)
        return FD_ERR_TIMEOUT;
    if (word & (kErrLength | kErrPage))
        return FD_ERR_DEVICE_INPUT;
    return FD_OK;
}

const char *fd_status_string(fd_status status)
{
    switch (status) {
    case FD_OK: return "FD_OK";
    case FD_ERR_INVALID_ARG: return "FD_ERR_INVALID_ARG";
    case FD_ERR_UNSUPPORTED: return "FD_ERR_UNSUPPORTED";
    case FD_ERR_WORKSPACE_TOO_SMALL: return "FD_ERR_WORKSPACE_TOO_SMALL";
    case FD_ERR_CUDA: return "FD_ERR_CUDA";
    case FD_ERR_TIMEOUT: return "FD_ERR_TIMEOUT";
    case FD_ERR_DEVICE_INPUT: return "FD_ERR_DEVICE_INPUT";
    }
    return "FD_ERR_UNKNOWN";
}

int fd_version(void) { return kVersion; }

}  // extern "C"
