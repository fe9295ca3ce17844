// fd_noalloc.cu -- fd_decode_noalloc: contiguous decode attention whose
// split/merge scratch lives in a fixed device array inside this library, so
// the call needs no workspace and performs no allocation of any kind.
//
// Who needs it: callers that cannot call cudaMalloc or any allocator at the
// point where they run attention -- for example code running inside a
// framework hook or plugin that forbids device allocation, a real-time path
// that must not risk the latency or failure of an allocation, or a host
// application that owns all device memory through its own pool and cannot
// hand a pointer from it to this library.  They pass only inputs and
// outputs.
//
// The scratch array (kNoallocScratchBytes) is reserved on every GPU that
// loads this library and stays reserved until the process exits.  Every call
// on a device uses the same array, and the array keeps whatever the previous
// call left in it; the call clears the one word that must start at zero (the
// device-error word) before its kernels run.  Two calls whose kernels
// overlap on the GPU (different streams, no ordering between them) race on
// the array and give undefined results.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fd.h"
#include "fd_launch.h"
#include "fd_sched.h"

namespace {

using namespace fd;

constexpr size_t kNoallocScratchBytes = FD_NOALLOC_SCRATCH_BYTES;
constexpr int kD = 128;   // the one head_dim this entry point serves

// The scratch: device-error word, tile prefix, partial LSEs and partial outputs.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct NoallocDevice {
    unsigned char *scratch = nullptr;   // device address of g_noalloc_scratch
    DeviceInfo info;
    unsigned long long ctx_id = 0;      // the context the address belongs to (0: unknown)
};

std::mutex g_mu;
NoallocDevice g_devs[64];
bool g_ready[64] = {};

// The current CUDA context's id, which the driver never reuses within a
// process (a context created after cudaDeviceReset gets a new one); 0 when
// there is no current context or the driver lacks the query.
unsigned long long current_context_id()
{
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static const GetCurrentFn get_current = []() -> GetCurrentFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                           cudaSuccess && q == cudaDriverEntryPointSuccess
                   ? reinterpret_cast<GetCurrentFn>(p)
                   : nullptr;
    }();
    static const GetIdFn get_id = []() -> GetIdFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                       q == cudaDriverEntryPointSuccess
                   ? reinterpret_cast<GetIdFn>(p)
                   : nullptr;
    }();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Once per device and context, with that device current: resolve the
// array's device address (in host code its name is only a host-side
// stand-in) and the properties the launch needs.  The address belongs to
// the context that was current when it was resolved, so it is resolved again
// when the device's context has changed (after cudaDeviceReset), and on
// every call if the driver cannot tell contexts apart.
fd_status noalloc_setup(NoallocDevice *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return FD_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    const unsigned long long ctx = current_context_id();
    if (!g_ready[dev] || ctx == 0 || ctx != g_devs[dev].ctx_id) {
        NoallocDevice d;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return FD_ERR_CUDA;   // (this call also makes the device's primary context current)
        d.scratch = static_cast<unsigned char *>(p);
        d.ctx_id = current_context_id();
        if (cudaDeviceGetAttribute(&d.info.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.info.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return FD_ERR_CUDA;
        g_devs[dev] = d;
        g_ready[dev] = true;
    }
    *out = g_devs[dev];
    return FD_OK;
}

// Scratch layout for `slots` partials of `group` rows: the same regions as a
// caller-provided workspace, but sized for the actual number of split CTAs.
struct NoallocLayout {
    size_t prefix_off, lse_off, o_off, total;
};

NoallocLayout noalloc_layout(int batch, int slots, int group)
{
    NoallocLayout l;
    l.prefix_off = 256;
    l.lse_off = align_up(l.prefix_off + 2 * sizeof(int) * (size_t)(batch + 1), 256);   // prefix, non-empty counts
    l.o_off = align_up(l.lse_off + sizeof(float) * (size_t)slots * group, 256);
    l.total = align_up(l.o_off + sizeof(float) * (size_t)slots * group * kD, 256);
    return l;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" fd_status fd_decode_noalloc(const void *q, const void *k, const void *v,
                                       const int32_t *seq_lens_dev, int batch, int num_q_heads,
                                       int num_kv_heads, int head_dim, int s_max, float scale, float *o,
                                       float *lse, unsigned int *device_status, fd_stream_t stream)
{
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        s_max < 0 || !q || !k || !v || !o || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(o) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
        (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)))
        return FD_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    if (head_dim != kD || !(group == 1 || group == 2 || group == 4 || group == 8) ||
        batch > kMaxBatch || (long long)batch * s_max >= (1ll << 31) ||
        (long long)num_kv_heads * batch * ceil_div(s_max, kTileTokens) >= (1ll << 31))
        return FD_ERR_UNSUPPORTED;
    if (batch == 0)
        return FD_OK;

    NoallocDevice dev;
    fd_status st = noalloc_setup(&dev);
    if (st != FD_OK)
        return st;
    const int num_ctas = dev.info.sms;
    const NoallocLayout wl = noalloc_layout(batch, batch * num_kv_heads + num_ctas, group);
    if (wl.total > kNoallocScratchBytes)
        return FD_ERR_WORKSPACE_TOO_SMALL;   // shape needs more scratch than the fixed array holds

    // Split-kernel parameters, pointing into the fixed array.
    SplitParams sp;
    std::memset(&sp, 0, sizeof sp);
    sp.q = static_cast<const uint16_t *>(q);
    sp.seq_lens = seq_lens_dev;
    sp.o = o;
    sp.lse = lse;
    sp.ws_err = reinterpret_cast<unsigned int *>(dev.scratch);
    sp.ws_prefix = reinterpret_cast<int32_t *>(dev.scratch + wl.prefix_off);
    sp.ws_lse = reinterpret_cast<float *>(dev.scratch + wl.lse_off);
    sp.ws_o = reinterpret_cast<float *>(dev.scratch + wl.o_off);
    sp.batch = batch;
    sp.hq = num_q_heads;
    sp.hkv = num_kv_heads;
    sp.cap = s_max;
    sp.s_max = s_max;
    sp.scale_log2 = scale * 1.4426950408889634f;
    sp.v_scale = 1.f;
    sp.q_len = 1;   // one query token per request, no fused heads
    sp.g_real = group;
    sp.n_cols = group;
    sp.fuse_f = 1;
    for (int n = 0; n < kMaxColumnSlots; ++n)
        sp.col_code[n] = n < group ? n << 8 : -1;   // token 0, part 0, query head n
    sp.timeout_ns = 2000000000ull;
    sp.seg_cost = kSegCostTiles;

    // Consumers as fd_decode picks them for an unfused call: CUDA cores for
    // one query head per kv head, tensor cores for GQA groups.
    const int cons = group >= 2 ? kConsMma : kConsCudaCores;

    // Shared-memory plan: the workspace entry points' rule, with the tiles per
    // CTA estimated from the capacity (as fd_decode does without host lengths).
    SplitLaunch launch;
    launch.grid = num_ctas;
    launch.stream = reinterpret_cast<cudaStream_t>(stream);
    const double est_tiles = (double)batch * num_kv_heads * ceil_div(s_max, kTileTokens);
    if ((st = plan_smem(dev.info, cons, group, kD, 2, batch, est_tiles / num_ctas,
                        est_tiles * 2.0 * kTileTokens * kD * 2 / num_ctas, &sp, &launch)) != FD_OK)
        return st;

    MergeParams mp;
    std::memset(&mp, 0, sizeof mp);   // no fused heads; every field defined
    mp.o = o;
    mp.lse = lse;
    mp.ws_o = sp.ws_o;
    mp.ws_lse = sp.ws_lse;
    mp.ws_prefix = sp.ws_prefix;
    mp.batch = batch;
    mp.hq = num_q_heads;
    mp.hkv = num_kv_heads;
    mp.num_ctas = num_ctas;
    mp.seq_lens = seq_lens_dev;
    mp.cap = s_max;
    mp.q_len = 1;
    mp.g_real = group;
    mp.n_cols = group;
    mp.fuse_f = 1;
    mp.late_trigger = launch.late_trigger;
    mp.seg_cost = sp.seg_cost;
    for (int n = 0; n < kMaxColumnSlots; ++n)
        mp.col_code[n] = n < group ? n << 8 : -1;

    alignas(64) CUtensorMap tmk, tmv;
    const long long rows = (long long)batch * (s_max > 0 ? s_max : 1);
    if ((st = encode_kv_maps(&tmk, &tmv, k, v, num_kv_heads, rows, kTileTokens, cons != kConsCudaCores, kKvBf16,
                             kD, &sp)) != FD_OK)
        return st;

    // The status word is the only part of the scratch that must start at zero.
    if (cudaMemsetAsync(sp.ws_err, 0, sizeof(unsigned int), launch.stream) != cudaSuccess)
        return FD_ERR_CUDA;
    if (launch_split_variant<false, kKvBf16, kD>(cons, group, false, sp, tmk, tmv, launch) != cudaSuccess)
        return FD_ERR_CUDA;
    if (launch_merge(group, kD, mp, batch * num_kv_heads, launch.stream) != cudaSuccess)
        return FD_ERR_CUDA;
    if (device_status &&
        cudaMemcpyAsync(device_status, sp.ws_err, sizeof(unsigned int), cudaMemcpyDeviceToDevice,
                        launch.stream) != cudaSuccess)
        return FD_ERR_CUDA;
    return FD_OK;
}
