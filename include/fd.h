/*
 * fd.h -- split-KV ("Flash-Decoding") single-query decode attention for
 * NVIDIA GB300 (sm_103a).  C ABI: plain pointers and sizes, no C++ or torch
 * types.  Link against libfd.so.
 *
 * What one call computes, for every request b < batch and query head
 * h < num_q_heads, over the first L_b = seq_lens[b] tokens of the KV cache:
 *
 *     s_t   = scale * sum_d q[b,h,d] * K_b[t, g, d]          g = h / (Hq/Hkv)
 *     O     = sum_t softmax(s)_t * V_b[t, g, :]              (fp32)
 *     LSE   = ln sum_t exp(s_t)                              (fp32, natural log)
 *
 * Sources (the pages this library follows):
 *   - "纯手搓 flash decoding sm120" (wingedge777.com), section 1 (flash
 *     decoding: split the KV sequence into chunks, one CTA per chunk writes a
 *     partial output and its log-sum-exp) and section 2 (the pass-2 merge by
 *     log-sum-exp; lse = m ln2 + ln d in the log2 domain).
 *   - "FlashAttention 与推理算子" (anrans.github.io ai-infra-handbooks):
 *     the online-softmax update of the FlashAttention section, the
 *     PagedAttention section (token t of a request lives in physical block
 *     block_table[t / page_size], slot t % page_size), the Flash-Decoding
 *     section (merge of normalised split outputs), and exercise 3 (one CTA
 *     serves every query head of a GQA group, so K/V are read once).
 *
 * Conventions shared by every entry point:
 *   - Ownership: the caller owns every buffer.  The library allocates no
 *     memory, keeps no per-call state, and never synchronises the stream
 *     (except fd_get_device_error, which says so).
 *   - Streams: all device work is ordered on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  Calls with distinct workspaces may run
 *     concurrently on different streams; calls sharing a workspace must be
 *     ordered.
 *   - Errors: arguments are checked on the host before any launch; a bad
 *     argument returns a status and launches nothing.  Values that live only
 *     on the device (lengths, block-table entries) are checked by the kernels,
 *     which clamp them into range, never read out of bounds, and record the
 *     problem in the workspace header; fd_get_device_error reports it.
 *   - Alignment: q, k, v, k_pages, v_pages and o must be 16-byte aligned, and
 *     the workspace 256-byte aligned; otherwise FD_ERR_INVALID_ARG.
 *   - Supported shapes: head_dim 64, 128 or 256; G = Hq/Hkv and the new query
 *     tokens per request q_len (fd_options.q_len) with G * q_len <= 16;
 *     batch <= 4096.  Other shapes return FD_ERR_UNSUPPORTED.  Over 8 query
 *     columns (G * q_len > 8) run on the tensor-core consumers only, so they
 *     also return FD_ERR_UNSUPPORTED with FD_FLAG_CUDA_CORES, and for an FP8
 *     cache with head_dim 64 when the kv heads cannot be paired (odd Hkv,
 *     FD_FLAG_NO_HEAD_FUSION, or pages under 8 tokens).
 *   - Several new tokens (q_len > 1, e.g. checking draft tokens): the cache
 *     of length L already holds them, q is [batch, q_len, Hq, head_dim], and
 *     new token i (0-based) attends causally to positions 0 .. L - q_len + i.
 *     O is [batch, q_len, Hq, head_dim] and LSE [batch, q_len, Hq]; a row that
 *     sees no position (L < q_len - i) gets O = 0 and LSE = -inf.
 *   - Precision: q, K and V are bf16 (default) or IEEE fp16
 *     (fd_options.dtype); K and V may instead be an FP8 cache
 *     (fd_options.kv_dtype: OCP E4M3 or E5M2 codes, one byte per element, with
 *     per-tensor dequantisation scales k_scale and v_scale).  Scores, softmax
 *     and accumulation are fp32; outputs are fp32.
 */
#ifndef FD_H
#define FD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st *fd_stream_t;

typedef enum fd_status {
    FD_OK = 0,
    FD_ERR_INVALID_ARG = 1,         /* null pointer, bad size, misalignment, length > capacity */
    FD_ERR_UNSUPPORTED = 2,         /* valid but not implemented: head_dim, group size, page size, batch */
    FD_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < fd_workspace_size(...) */
    FD_ERR_CUDA = 4,                /* a CUDA runtime or driver call failed (launch, tensor map) */
    FD_ERR_TIMEOUT = 5,             /* a kernel's bounded wait ran out (reported by fd_get_device_error) */
    FD_ERR_DEVICE_INPUT = 6         /* a device-side length or block-table entry was out of range */
} fd_status;

/* Element type of q, K and V. */
typedef enum fd_dtype {
    FD_DTYPE_BF16 = 0,   /* bfloat16 (default) */
    FD_DTYPE_F16 = 1     /* IEEE binary16 */
} fd_dtype;

/* Element type of the K/V cache.  An FP8 cache holds one code per element,
 * [.., head_dim] bytes per (token, kv head) row, and represents
 * K = k_scale * decode(code) and V = v_scale * decode(code). */
typedef enum fd_kv_dtype {
    FD_KV_AS_Q = 0,       /* the type of q (fd_options.dtype) */
    FD_KV_FP8_E4M3 = 1,   /* OCP FP8 E4M3 ("fn": no infinities, max 448) */
    FD_KV_FP8_E5M2 = 2    /* OCP FP8 E5M2 */
} fd_kv_dtype;

/* Optional knobs; pass NULL for the defaults. */
typedef struct fd_options {
    /* Number of persistent split CTAs that share the KV tiles (1..1024).
     * 0 = one per SM of the current device.  Results do not depend on it
     * beyond fp32 summation order. */
    int num_ctas;
    /* FD_FLAG_* bits; 0 for normal use. */
    unsigned int flags;
    /* Limit for every wait inside the kernels, in nanoseconds; 0 = 2 s.
     * When a wait runs out the kernel stops, records FD_ERR_TIMEOUT in the
     * workspace header and returns instead of hanging. */
    unsigned long long wait_timeout_ns;
    /* Optional cudaEvent_t handles recorded on `stream` immediately before
     * and after the split kernel (for timing the kernel alone); NULL = none.
     * During a stream capture they become event-record nodes of the graph
     * (cudaEventRecordExternal), recorded by every replay. */
    void *split_start_event;
    void *split_end_event;
    /* Element type of q, K and V (fd_dtype); 0 = bf16. */
    int dtype;
    /* Element type of K and V (fd_kv_dtype); 0 = that of q. */
    int kv_dtype;
    /* Dequantisation scales of an FP8 cache; 0 means 1.  k_scale multiplies
     * every K element (it enters the scores), v_scale every V element (it
     * multiplies O).  Ignored for 16-bit caches. */
    float k_scale;
    float v_scale;
    /* New query tokens per request (0 means 1); see the note on q_len above. */
    int q_len;
} fd_options;

/* ---- User flags (fd_options.flags) ---- */

/* Use the CUDA-core consumers for every group size.  By default GQA groups
 * (Hq/Hkv x q_len >= 2 query columns per kv head, rows of at least 128 bytes
 * or kv heads paired to reach them) run q.K^T and P.V on the tensor cores
 * (bf16 or fp16 MMA, fp32 accumulation; for P.V each softmax weight is
 * taken as a rounded part plus its rounded remainder in two MMAs, 16 or 22
 * significant bits), with any page size; this flag selects the all-fp32
 * CUDA-core arithmetic instead (up to 8 query columns per kv head). */
#define FD_FLAG_CUDA_CORES 0x2u

/* Tensor-core consumers: load each 64-dim part of a K/V tile as its own TMA
 * box (3-D tensor maps) instead of one box carrying every part (4-D maps).
 * Results are identical; for comparisons only. */
#define FD_FLAG_NO_4D_BOXES 0x4u

/* Do not fuse kv heads.  By default, when the tensor-core consumers apply
 * (contiguous KV, or pages of at least 8 tokens, and no FD_FLAG_CUDA_CORES),
 * a kv head's rows are short (under 256 bytes: head_dim 64, or an FP8 cache
 * with head_dim up to 128, or pages under 64 tokens) and the call has at
 * least 24 KV tiles of 64 tokens per split CTA (counted from seq_lens_host
 * when given, else from the capacity) -- or, whatever the call's length, the
 * cache is FP8 with head_dim 128 and one query column per kv head -- F
 * adjacent kv heads are read as one head of F * head_dim dims: [.., Hkv, D] and [.., Hkv/F, F*D] are the same
 * bytes, so each TMA row is F times longer.
 *   F = 4 when 4 * head_dim <= 256, 4 * G * q_len <= 8 and 4 divides Hkv: the
 *         four query groups share one tensor-core tile, with zeros for the
 *         dims of the other heads;
 *   F = 2 otherwise, when 2 * head_dim <= 256 and 2 divides Hkv: each warp of
 *         a pair takes one of the two heads.
 * Over 8 query columns with an FP8 head_dim of 64 always pair.  Every query
 * head still attends only to its own kv head.  This flag keeps one kv head
 * per segment. */
#define FD_FLAG_NO_HEAD_FUSION 0x8u

/* Do not gather pages of 1 or 2 tokens four rows per TMA load
 * (tile::gather4); load one box per page instead.  Results are identical; for
 * comparisons only. */
#define FD_FLAG_NO_GATHER 0x20u

/* Fuse kv heads whenever the shape and consumers allow it (the F rule
 * above), whatever the row length and the call's size.  FD_FLAG_NO_HEAD_FUSION
 * wins if both are set. */
#define FD_FLAG_FUSE_HEADS 0x10u

/* Do not prefetch.  By default, in calls of at least 24 KV tiles per split
 * CTA, each split CTA asks L2 for its first KV tiles while it waits for the
 * kernels ahead of it in the stream to complete (a plan made from the
 * lengths and block table as they read at that moment; a stale plan only
 * costs bandwidth).  Results are identical; for comparisons only. */
#define FD_FLAG_NO_PREFETCH 0x40u

/* Scores on the tcgen05 tensor cores.  For an FP8 cache (E4M3 or E5M2) whose
 * kv heads are paired (head_dim 128; contiguous, or pages of at least 64
 * tokens) the scores are by default formed with tcgen05 MMAs straight from
 * the FP8 K tile into tensor memory, against the query split into parts of
 * the same FP8 format (exact: two to four parts for a bf16 or fp16 query),
 * when a kv head has at most 4 query columns and the call has at least 24
 * paired KV tiles per split CTA; warp MMAs on K converted to fp16 in
 * registers otherwise.  Measured on GB300 (E4M3), the tcgen05 scores took
 * the 1 GiB MHA call 6% and the ragged GQA-4 call 3% faster, and the GQA-8
 * call 2% slower.  This flag takes the tcgen05 scores for up to 8 columns
 * and any length too; FD_FLAG_NO_TMEM_SCORES never (it wins if both are
 * set).  Results agree to fp32 rounding. */
#define FD_FLAG_TMEM_SCORES 0x80u
#define FD_FLAG_NO_TMEM_SCORES 0x100u

/* ---- Test hooks (fd_options.flags): for the library's own tests only ---- */

/* CTA 0 announces more bytes for its first tile than it loads, so its
 * consumers' wait can never complete and must run out (the bounded-wait
 * test).  Never set it in production; the outputs of such a call are
 * undefined. */
#define FD_FLAG_TEST_STARVE_FIRST_TILE 0x1u

/*
 * Bytes of workspace that fd_decode / fd_decode_paged (and their partial
 * forms) need for this shape.  The pages allocate their split partials per
 * call; this sizing call has no counterpart there: it lets the caller own one
 * workspace for every call of a shape.
 * Pure host function (no CUDA call).  The size does not depend on the
 * lengths: it holds a 256-byte header, the per-request tile prefix and one
 * fp32 partial (Hq/Hkv rows of head_dim outputs plus their log-sum-exp) per
 * (request, kv head) plus one per possible split CTA -- sized for whichever
 * launch shape the call takes, with or without fused kv heads (see
 * FD_FLAG_NO_HEAD_FUSION).  max_kv_len and page_size are validated but do
 * not change the size.
 * Returns 0 for invalid arguments and for more than 16 query columns per kv
 * head (Hq/Hkv x q_len), which no call accepts.
 */
size_t fd_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                         int max_kv_len, int page_size);

/* fd_workspace_size for calls with q_len new query tokens per request
 * (fd_options.q_len); q_len = 1 gives fd_workspace_size.  Returns 0 for
 * invalid arguments. */
size_t fd_workspace_size_q(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                           int max_kv_len, int page_size, int q_len);

/*
 * Zero-fill a workspace (its sticky device-error word must start at zero).
 * Call once after allocating a workspace, before its first use.
 * Stream-ordered, asynchronous.  No counterpart on the pages (workspace
 * ownership is this library's).
 */
fd_status fd_workspace_init(void *workspace, size_t workspace_bytes, fd_stream_t stream);

/*
 * Decode attention over a contiguous KV cache.  Arithmetic: "纯手搓 flash
 * decoding sm120", sections 1-2 (split the sequence, partial O and LSE per
 * split, pass-2 merge by LSE) with the online softmax of the handbook's
 * FlashAttention section; layout [seq, head, dim] per request as in that
 * article's problem statement.
 *   q            [batch, num_q_heads, head_dim] bf16 or fp16, device.
 *   k, v         [batch, s_max, num_kv_heads, head_dim] device, row-major, of
 *                q's type or FP8 codes (fd_options.kv_dtype).
 *                Positions t >= seq_lens[b] of request b are never used
 *                (they may hold anything, including NaN).
 *   seq_lens_dev [batch] int32, device: L_b in [0, s_max].  NULL means every
 *                request has length s_max.  A device value above s_max is
 *                clamped to s_max and reported as FD_ERR_DEVICE_INPUT.
 *   seq_lens_host [batch] int32, host copy of the lengths, or NULL.  Only used
 *                to validate lengths on the host (FD_ERR_INVALID_ARG if any is
 *                outside [0, s_max]); the kernels read seq_lens_dev.
 *   scale        multiplies q.k (callers usually pass 1/sqrt(head_dim)).
 *   o            [batch, num_q_heads, head_dim] fp32, device, written.
 *   lse          [batch, num_q_heads] fp32, device, written, natural log; may
 *                be NULL.  A request with L_b = 0 gets O = 0 and LSE = -inf.
 *   workspace    device scratch of at least fd_workspace_size(batch,
 *                num_q_heads, num_kv_heads, head_dim, s_max, 0) bytes,
 *                initialised once with fd_workspace_init.
 *   opts         NULL or options (see fd_options).
 */
fd_status fd_decode(const void *q, const void *k, const void *v,
                    const int32_t *seq_lens_dev, const int32_t *seq_lens_host,
                    int batch, int num_q_heads, int num_kv_heads, int head_dim, int s_max,
                    float scale, float *o, float *lse,
                    void *workspace, size_t workspace_bytes,
                    const fd_options *opts, fd_stream_t stream);

/*
 * Decode attention over a paged KV cache.  Indirection: the PagedAttention
 * section of "FlashAttention 与推理算子" (token t of a request in physical
 * block block_table[t / page_size], slot t % page_size); arithmetic as for
 * fd_decode.
 *   k_pages, v_pages [num_pages, page_size, num_kv_heads, head_dim] device, of
 *                q's type or FP8 codes (fd_options.kv_dtype).
 *   block_table  [batch, max_blocks_per_seq] int32, device, row-major: token t
 *                of request b is in page block_table[b][t / page_size], slot
 *                t % page_size.  Only the first ceil(L_b / page_size) entries of
 *                a row are read; the rest may hold anything (e.g. -1).  An entry
 *                outside [0, num_pages) is replaced by page 0 and reported as
 *                FD_ERR_DEVICE_INPUT.
 *   page_size    a divisor of 64 (1, 2, 4, ..., 32) or a multiple of 64; a
 *                page under 64 tokens must hold at least 128 bytes per kv head
 *                (an FP8 cache with head_dim 64 needs pages of 2 or more).
 *                Other sizes return FD_ERR_UNSUPPORTED.  Pages under 8 tokens
 *                on the tensor-core consumers (GQA groups) are copied row by
 *                row and need num_pages * page_size * num_kv_heads < 2^32
 *                (FD_ERR_UNSUPPORTED otherwise; any pool that fits a GB300
 *                does).
 *   seq_lens_dev [batch] int32, device, L_b in [0, max_blocks_per_seq * page_size];
 *                must not be NULL.
 *   Other arguments as for fd_decode.
 */
fd_status fd_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                          const int32_t *block_table, int max_blocks_per_seq,
                          const int32_t *seq_lens_dev, const int32_t *seq_lens_host,
                          int batch, int num_q_heads, int num_kv_heads, int head_dim,
                          int page_size, int num_pages, float scale,
                          float *o, float *lse,
                          void *workspace, size_t workspace_bytes,
                          const fd_options *opts, fd_stream_t stream);

/*
 * Sequence sharding: attention over one range of cache positions, and the
 * merge of such partial results.  Sources: the handbook's Flash-Decoding
 * section (split-K decode: each split keeps its normalised output and
 * softmax statistics, and the splits are combined by them; exercise 2: a
 * split that saw no token is skipped) and the pass-2 merge by log-sum-exp of
 * "纯手搓 flash decoding sm120", section 2 (written out at
 * fd_merge_partials).  A rank that holds cache positions [kv_begin, kv_end) of
 * every request computes its partial with fd_decode_partial (or the paged
 * form); the ranks exchange the partials (n sets of [rows, head_dim] outputs
 * and [rows] LSEs, e.g. one all-gather) and fd_merge_partials combines them
 * into the result fd_decode would give on the whole cache.
 */

/*
 * fd_decode over the cache positions [kv_begin, min(L_b, kv_end)) of every
 * request.  k and v hold the range: row t' of request b
 * ([batch, s_max, num_kv_heads, head_dim]) is cache position kv_begin + t'.
 * seq_lens are the requests' whole lengths L_b (device; NULL = every request
 * has kv_begin + s_max tokens), so several new tokens (fd_options.q_len) keep
 * their causal limits at the whole sequence's positions.  The range of
 * request b holds n_b = min(L_b, kv_end) - kv_begin tokens (0 if negative),
 * and n_b <= s_max is required (seq_lens_host: FD_ERR_INVALID_ARG; a device
 * value: clamped and reported as FD_ERR_DEVICE_INPUT).
 *   kv_begin, kv_end  0 <= kv_begin <= kv_end (INT32_MAX: to the end), and
 *                kv_begin + s_max < 2^31; else FD_ERR_INVALID_ARG.
 *   o_part       [batch, (q_len,) num_q_heads, head_dim] fp32: the output
 *                normalised over the range.
 *   lse_part     [batch, (q_len,) num_q_heads] fp32, natural log, required
 *                (NULL: FD_ERR_INVALID_ARG).  A row that sees no position of
 *                the range gets O = 0 and LSE = -inf.
 * Workspace and every other argument as for fd_decode (the workspace size
 * of the shape with max_kv_len = s_max).
 */
fd_status fd_decode_partial(const void *q, const void *k, const void *v,
                            const int32_t *seq_lens_dev, const int32_t *seq_lens_host,
                            int batch, int num_q_heads, int num_kv_heads, int head_dim, int s_max,
                            int kv_begin, int kv_end, float scale, float *o_part, float *lse_part,
                            void *workspace, size_t workspace_bytes,
                            const fd_options *opts, fd_stream_t stream);

/*
 * fd_decode_paged over the cache positions [kv_begin, min(L_b, kv_end)):
 * block_table row b maps the range's own tokens, token t' = position
 * kv_begin + t' in page block_table[b][t' / page_size], slot t' % page_size,
 * and n_b <= max_blocks_per_seq * page_size is required.  seq_lens_dev is
 * required; everything else as for fd_decode_partial and fd_decode_paged.
 */
fd_status fd_decode_paged_partial(const void *q, const void *k_pages, const void *v_pages,
                                  const int32_t *block_table, int max_blocks_per_seq,
                                  const int32_t *seq_lens_dev, const int32_t *seq_lens_host,
                                  int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                  int page_size, int num_pages, int kv_begin, int kv_end, float scale,
                                  float *o_part, float *lse_part, void *workspace, size_t workspace_bytes,
                                  const fd_options *opts, fd_stream_t stream);

/*
 * Merge num_parts partial sets into one result, for every one of `rows`
 * query rows (batch x q_len x num_q_heads):
 *     M = max_s lse_s,  LSE = M + ln sum_s exp(lse_s - M),
 *     O = sum_s O_s exp(lse_s - LSE);
 * a set with lse_s = -inf is skipped, and a row that no set saw gets O = 0,
 * LSE = -inf.
 *   o_parts      [num_parts, rows, head_dim] fp32, device, 16-byte aligned.
 *   lse_parts    [num_parts, rows] fp32, device (natural log).
 *   o            [rows, head_dim] fp32, device, 16-byte aligned, written.
 *   lse          [rows] fp32, device, written, or NULL.
 * num_parts >= 1 and rows >= 0 (FD_ERR_INVALID_ARG otherwise); head_dim 64,
 * 128 or 256 (FD_ERR_UNSUPPORTED otherwise).  No workspace; stream-ordered.
 */
fd_status fd_merge_partials(const float *o_parts, const float *lse_parts, int num_parts, int rows,
                            int head_dim, float *o, float *lse, fd_stream_t stream);

/* Bytes of the fixed device scratch array used by fd_decode_noalloc. */
#define FD_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Bits of the status word fd_decode_noalloc writes to *device_status. */
#define FD_DEVICE_STATUS_TIMEOUT 0x1u     /* a bounded wait ran out */
#define FD_DEVICE_STATUS_BAD_LENGTH 0x2u  /* a device length was outside [0, s_max] and was clamped */

/*
 * fd_decode without a workspace, for callers that cannot allocate device
 * memory where they run attention: code inside a host framework or plugin
 * that forbids device allocation at that point, latency-critical paths that
 * must not risk an allocation stalling or failing, and applications whose
 * device memory all belongs to their own pool.  The sources this library
 * follows have no counterpart to this call; it exists only for such callers.
 *
 * It computes what fd_decode computes for a contiguous, unfused call (the
 * same split kernel -- CUDA-core consumers for Hq = Hkv, tensor-core
 * consumers for GQA groups -- and the same merge, one split CTA per SM), with
 * the split partials and the tile prefix held in a fixed device array of FD_NOALLOC_SCRATCH_BYTES (8 MiB) that is
 * part of this library: every GPU that loads the library reserves it until
 * the process exits.  Nothing is allocated -- no cudaMalloc, cudaFree or
 * allocating library routine -- and no workspace is passed.  The caller still
 * passes the inputs and the outputs.
 *   q, k, v, seq_lens_dev, batch, num_q_heads, num_kv_heads, head_dim, s_max,
 *   scale, o, lse: as for fd_decode (lse may be NULL).
 *   device_status: NULL, or a device uint32 that receives this call's
 *   FD_DEVICE_STATUS_* bits (0 when all went well), stream-ordered.
 * Limits: bf16 inputs, head_dim 128 and Hq/Hkv in {1, 2, 4, 8} only (other
 * shapes return FD_ERR_UNSUPPORTED); the scratch must hold 256 bytes + 4 (batch + 1) bytes + (batch *
 * num_kv_heads + number of SMs) partials of (Hq/Hkv) * (head_dim + 1) * 4
 * bytes, each region rounded up to 256 bytes; a larger shape returns
 * FD_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 * The first call on each device resolves the array's device address
 * (cudaGetSymbolAddress) and caches it with the device's current context;
 * make that first call before any stream capture.  A call that finds a
 * different context (the device was reset with cudaDeviceReset) resolves the
 * address again, so make the first call after a reset before any capture
 * too.
 * Every call on a device shares the one array, which keeps the previous
 * call's contents; each call clears the part that must start at zero (the
 * status word) itself.  Calls whose kernels can overlap on the GPU (for
 * example on two unordered streams) race on the array: order them.
 */
fd_status fd_decode_noalloc(const void *q, const void *k, const void *v,
                            const int32_t *seq_lens_dev, int batch, int num_q_heads,
                            int num_kv_heads, int head_dim, int s_max, float scale, float *o,
                            float *lse, unsigned int *device_status, fd_stream_t stream);

/*
 * Read and clear the sticky device-error word of a workspace: FD_OK,
 * FD_ERR_TIMEOUT or FD_ERR_DEVICE_INPUT (timeout wins if both happened).
 * After FD_ERR_TIMEOUT the outputs of the failed call are undefined; the
 * workspace can be reused as it is.
 * SYNCHRONISES `stream` (it copies one word to the host).
 */
fd_status fd_get_device_error(void *workspace, fd_stream_t stream);
/* (No counterpart on the pages: their kernels have no bounded waits and no
 * device-side input checks to report.) */

/* Human-readable name of a status; never NULL.  No counterpart on the pages. */
const char *fd_status_string(fd_status status);

/* Library version, major*10000 + minor*100 + patch.  No counterpart on the pages. */
int fd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FD_H */
