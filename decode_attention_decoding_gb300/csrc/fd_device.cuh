// fd_device.cuh -- device primitives for the decode-attention kernels (sm_103a).
//
// Thin inline-PTX wrappers: shared-memory mbarriers (init, arrive with a
// transaction count, bounded parity wait), TMA tile loads into shared memory,
// the global timer, named barriers, programmatic-dependent-launch control,
// packed fp32x2 arithmetic and bf16 unpacking.  Nothing here knows about
// attention.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fd {

// Bits of the sticky device-error word at the start of the workspace.
enum : unsigned int {
    kErrTimeout = 1u,      // a bounded wait ran out
    kErrLength = 2u,       // a device length was outside [0, capacity]
    kErrPage = 4u,         // a block-table entry was outside [0, num_pages)
};

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One arrival that also raises the expected transaction byte count.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until the phase with the given parity has completed, for at most
// timeout_ns.  If `abort_flag` (shared memory) becomes non-zero the wait
// gives up early.  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                                  const volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (abort_flag && *abort_flag)
            return false;
        if (global_timer_ns() - t0 > timeout_ns)
            return false;
    }
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void *desc)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(desc)) : "memory");
}

// 3-D tiled bulk tensor load global -> shared, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *desc, uint32_t bar, int c0, int c1,
                                            int c2, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

// 16-byte asynchronous copy global -> shared (L2 only), with an L2 policy.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint64_t policy)
{
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "l"(policy)
                 : "memory");
}

// One arrive on `bar` once every cp.async this thread issued before has
// landed; the barrier's expected count already includes it (no increment).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Four rows of a 2-D tensor map (rows r0..r3, columns from c0, one box
// {columns, 1} each) gathered into four consecutive box-sized slots at dst,
// completing on `bar`.
__device__ __forceinline__ void tma_gather4_2d(uint32_t dst, const void *desc, uint32_t bar, int c0, int r0,
                                               int r1, int r2, int r3, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar),
        "l"(policy)
        : "memory");
}

// 4-D tiled bulk tensor load global -> shared, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *desc, uint32_t bar, int c0, int c1,
                                            int c2, int c3, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
        : "memory");
}

// Prefetch one box of a tiled tensor into L2 (3-D / 4-D coordinates).  A
// hint: nothing lands in shared memory and nothing signals completion; the
// unit skips elements outside the tensor.
__device__ __forceinline__ void tma_prefetch_3d(const void *desc, int c0, int c1, int c2)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(desc)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_4d(const void *desc, int c0, int c1, int c2, int c3)
{
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(desc)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// L2 policy for data read exactly once (the KV cache stream).
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- sync

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: allow the next kernel in the stream to
// start launching; it waits for this grid's completion on its own.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Block until the preceding grid in the stream has completed and its memory
// operations are visible.
__device__ __forceinline__ void pdl_wait_prior_grid()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- math

__device__ __forceinline__ float exp2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pair arithmetic (one instruction for two lanes of work).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Two bf16 values packed in a 32-bit word (element 0 in the low half) to fp32.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Two IEEE fp16 values packed in a 32-bit word (element 0 low) to fp32.
__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w)
{
    float2 r;
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(w));
    return r;
}

// Packed 16-bit pair to fp32 for the input element type (bf16 or fp16).
template <bool F16>
__device__ __forceinline__ float2 x2_to_float2(uint32_t w)
{
    if constexpr (F16)
        return f16x2_to_float2(w);
    else
        return bf16x2_to_float2(w);
}

// Element types of the K/V cache.  bf16 and fp16 caches come with a query of
// the same type; an FP8 cache (OCP E4M3 or E5M2 codes) with a bf16 or fp16
// query chosen at run time.
enum : int { kKvBf16 = 0, kKvF16 = 1, kKvE4m3 = 2, kKvE5m2 = 3 };

__host__ __device__ constexpr bool kv_is_fp8(int kv) { return kv >= kKvE4m3; }

// Two FP8 codes (element 0 in the low byte) to two fp16 values (element 0 in
// the low half).  Every E4M3 and E5M2 value is an fp16 value, so the
// conversion is exact.
template <int KV>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint16_t w)
{
    uint32_t r;
    if constexpr (KV == kKvE4m3)
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(w));
    else
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(r) : "h"(w));
    return r;
}

// Low and high 16-bit halves of a word.
__device__ __forceinline__ uint16_t lo16(uint32_t w) { return (uint16_t)(w & 0xFFFFu); }
__device__ __forceinline__ uint16_t hi16(uint32_t w) { return (uint16_t)(w >> 16); }

// Byte permute: result byte i = byte sel_i of {b, a} (a holds bytes 0..3).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Two FP8 codes to fp32.
template <int KV>
__device__ __forceinline__ float2 fp8x2_to_float2(uint16_t w)
{
    return f16x2_to_float2(fp8x2_to_f16x2<KV>(w));
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 ldg128_nc(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

}  // namespace fd

// ---------------------------------------------------------------- warp MMA

namespace fd {

// Four 8x8 b16 matrices from shared memory; lane i supplies the row address
// of matrix i / 8.  Result register r holds matrix r in the mma fragment
// layout (lane l: row l / 4, elements 2 (l % 4) and 2 (l % 4) + 1).
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// As ldmatrix_x4, each matrix transposed.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Transpose one 8x8 b16 matrix held in the fragment layout across the warp.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D = A (16x16 bf16, row) * B (16x8 bf16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two fp32 values rounded to bf16 (nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 values rounded to fp16 (nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// D = A (16x16 fp16, row) * B (16x8 fp16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The 16-bit MMA for the input element type.
template <bool F16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1)
{
    if constexpr (F16)
        mma_f16_16816(d, a0, a1, a2, a3, b0, b1);
    else
        mma_bf16_16816(d, a0, a1, a2, a3, b0, b1);
}

template <bool F16>
__device__ __forceinline__ uint32_t pack_x2(float lo, float hi)
{
    if constexpr (F16)
        return pack_f16x2(lo, hi);
    else
        return pack_bf16x2(lo, hi);
}

}  // namespace fd

// ---------------------------------------------------------------- tcgen05 / TMEM

namespace fd {

// Tensor memory (TMEM): 512 columns x 128 lanes of 32-bit cells per SM.  An
// address is lane << 16 | column.  Allocation is per CTA, by one whole warp,
// in a power of two of at least 32 columns; the address lands in shared
// memory at `slot`.  The same warp frees it before the CTA exits.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order tcgen05 operations around a thread synchronisation (a barrier or an
// mbarrier wait): `before` ahead of the signalling side, `after` behind the
// waiting side.
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout that TMA writes with 128-byte swizzling: rows of 128 bytes,
// eight-row groups 1024 bytes apart, the 16-byte chunk c of row r stored at
// chunk c ^ (r & 7).  The operand starts at `addr` (its group 1024-byte
// aligned; a K step inside the 128-byte row adds its byte offset to addr).
// Fields: start address >> 4 (bits 0-13), leading byte offset >> 4 (16-29;
// unused here, set to 1), stride byte offset >> 4 (32-45: 1024 B between
// row groups), the descriptor version 1 (46-47), base offset 0 (49-51), and
// the swizzle mode 2 = 128-byte (61-63).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t addr)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of a dense kind::f8f6f4 MMA with A and B of one FP8
// format (fmt 0 = E4M3, 1 = E5M2; both K-major) and an fp32 accumulator: D
// format 1 = F32 (bits 4-5), A and B formats (7-9, 10-12), N >> 3 (17-22),
// M >> 4 (24-28).
__host__ __device__ constexpr uint32_t umma_idesc_fp8_f32(int m, int n, uint32_t fmt)
{
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D[tmem] (+)= A . B^T for one K step of 32 FP8 elements, issued by one thread.
__device__ __forceinline__ void umma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// One arrival on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Eight consecutive 32-bit columns of this thread's TMEM lane (warp w of a
// warpgroup reaches lanes 32 (w % 4) .. 32 (w % 4) + 31; thread i its lane
// base + i).  The registers are valid after tmem_wait_ld.
__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Maximum of v over the 32 lanes of the warp, in every lane.
__device__ __forceinline__ float warp_max_f32(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// Two fp32 values rounded to E4M3 (nearest even, saturating at +-448), `lo`
// in the low byte.
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 values rounded to E5M2 (nearest even, saturating at +-57344),
// `lo` in the low byte.
__device__ __forceinline__ uint16_t pack_e5m2x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace fd
