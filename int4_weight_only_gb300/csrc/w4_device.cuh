// w4_device.cuh - inline-PTX building blocks shared by the libw4 kernels
// (sm_103a): mbarriers with bounded waits, TMA tile loads, ldmatrix,
// mma.sync, bf16x2 nibble conversion, named barriers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "../../include/w4.h"

namespace w4 {

// A bounded wait gives up after a limit of SM clock cycles, records
// W4_ERR_DEVICE_TIMEOUT and returns false.  The default is about one second
// at the GB300's clocks.
constexpr long long kWaitLimitCycles = 2000000000LL;

// The library's device status block (one per device): the error flag that
// kernels set, the fault-injection switch of the failure tests
// (w4_set_fault_injection), then the wait limit (w4_set_wait_limit; 0 = the
// default).  Kernels receive the flag's address and read the limit from the
// same block when a wait starts to take long.  Drains of copies already
// issued always wait up to the default, so nothing is left in flight when a
// CTA exits.
struct DeviceStatus {
    int err;
    int inject;
    long long wait_limit;
};

// Fault-injection switches (read once per CTA by the grouped decode kernel
// only): a wait that nothing will ever complete, so the failure path runs
// without any fault.
constexpr int kInjectNoList = 1;     // the consumers never publish the group list
constexpr int kInjectNoRelease = 2;  // the consumers never free a ring slot

__device__ __forceinline__ int fault_injection_of(const int* err) {
    return reinterpret_cast<const volatile DeviceStatus*>(err)->inject;
}

__device__ __forceinline__ long long wait_limit_of(const int* err) {
    const long long v = reinterpret_cast<const volatile DeviceStatus*>(err)->wait_limit;
    return v > 0 ? v : kWaitLimitCycles;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false when
// `*abort` is set by another thread of the CTA or when the wait exceeds
// kWaitLimitCycles; in the latter case it raises `*abort` and the device
// error flag.  Every thread of the CTA therefore leaves its loops in bounded
// time once any wait has failed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    const long long lim = wait_limit_of(err);
    while (true) {
        if (*abort) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > lim) {
            *abort = 1;
            atomicCAS(err, 0, W4_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}

// Same, but ignores `abort`: used to drain copies already in flight before a
// CTA exits.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, int* err) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimitCycles) {
            atomicCAS(err, 0, W4_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
    return true;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes.  c0 is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map,
                                            int c0, int c1, uint64_t* bar,
                                            uint64_t cache_policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)),
           "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(cache_policy)
        : "memory");
}

// 1D bulk copy global -> shared (16-byte aligned, size a multiple of 16),
// completion signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
           "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- barriers
// Named barrier `id` over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns the AND of `pred` over its threads.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(nthreads) : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- warp MMA
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}

// Same, without a memory clobber: for reads of shared memory whose ordering
// is already fixed by a preceding mbarrier wait.
__device__ __forceinline__ void ldmatrix_x4_nc(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                               uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D = A * B + C, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1, const float* c) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1),
          "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// D = A * B + C, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float* d, uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1, const float* c) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1),
          "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// (x & mask) | bits, one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t mask, uint32_t bits) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(mask), "r"(bits));
    return r;
}

// Acquire load / release store of a flag at GPU scope.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.s32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// a - b on bf16 pairs (exact for the small integers it is used on).
__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Eight 4-bit codes c0..c7 of v (c_i in bits 4i..4i+3) -> four bf16x2 words
// (128 + c0, 128 + c1), (128 + c2, 128 + c3), (128 + c4, 128 + c5),
// (128 + c6, 128 + c7), exact: bf16 128.0 (0x4300) has seven mantissa bits
// of spacing 1, so a code OR-ed into the low four gives 128 + c.  A byte
// permute puts the two codes of one byte (from v and from v >> 4) into the
// two halves, one LOP3 masks them and adds the exponent.
__device__ __forceinline__ void nibbles_to_bf16x2_pairs(uint32_t v, uint32_t* o) {
    const uint32_t vh = v >> 4, m = 0x000F000Fu, e = 0x43004300u;
    o[0] = and_or(__byte_perm(v, vh, 0x4400), m, e);
    o[1] = and_or(__byte_perm(v, vh, 0x5511), m, e);
    o[2] = and_or(__byte_perm(v, vh, 0x6622), m, e);
    o[3] = and_or(__byte_perm(v, vh, 0x7733), m, e);
}

// Eight codes c0..c7 of v -> four fp16x2 words, exact:
//   (1024 + c0, 1024 + c4), (1024 + 16 c1, 1024 + 16 c5),
//   (1024 + c2, 1024 + c6), (1024 + 16 c3, 1024 + 16 c7).
// fp16 1024.0 (0x6400) has ten mantissa bits of spacing 1, so both nibbles
// of a byte can be OR-ed in place; only one shift (by 8) is needed.
__device__ __forceinline__ void nibbles_to_f16x2_biased(uint32_t v, uint32_t* o) {
    const uint32_t e = 0x64006400u;
    const uint32_t w = v >> 8;
    o[0] = and_or(v, 0x000F000Fu, e);
    o[1] = and_or(v, 0x00F000F0u, e);
    o[2] = and_or(w, 0x000F000Fu, e);
    o[3] = and_or(w, 0x00F000F0u, e);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------------- integer
// d = c + sum_i a.u8[i] * b.s8[i]
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float ld_cg_f32(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ int ld_cg_s32(const int* p) {
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// L2-coherent loads (skip L1) for partial sums other CTAs wrote.
// Atomic add with acquire-release semantics at GPU scope (returns the old
// value): a split-K ticket.  Taken by one thread after a CTA barrier, it
// publishes the CTA's earlier stores and, for the last arriver, makes the
// other CTAs' stores visible to the loads that follow the next barrier.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;"
                 : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// ---------------------------------------------------------------- INT8 activations
// The per-token dynamic INT8 rule ("Jetson Orin AGX INT4 推理优化实践",
// section "从 FP 线性层到 INT4 DP4A 的数学推导"), shared by the activation
// quantizer and the SwiGLU epilogue that emits INT8 activations.
// q = clip(rint(fp32(v / s)), -127, 127) as a byte (s > 0), bit-identical to
// the IEEE quotient without dividing in the common case.  |v| <= 127.x s, and
// t = v * rcp(s) (product and reciprocal each correctly rounded) differs from
// v / s by at most three roundings, under 2^-22 |v/s| <= 2^-15, as does
// fp32(v / s); so both round to the same integer unless t lies within 2^-14
// of a half-integer.  Only then (or when t is not finite, for a subnormal s)
// is the quotient computed.
__device__ __forceinline__ uint32_t quant_s8(float v, float s, float rs) {
    float t = v * rs;
    if (!(fabsf(fabsf(t - truncf(t)) - 0.5f) > 0x1p-14f)) t = __fdiv_rn(v, s);
    return (uint32_t)(uint8_t)(int8_t)(int)fminf(fmaxf(rintf(t), -127.f), 127.f);
}

// Eight values to eight INT8 bytes, as quant_s8 each; all zero when s = 0.
// One branch for the eight (the quotient is rarely needed), so that the
// eight products, tests and conversions are independent instructions.
__device__ __forceinline__ uint2 quant_s8x8(const float f[8], float s, float rs) {
    if (s == 0.f) return make_uint2(0u, 0u);
    float t[8];
    bool near = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        t[j] = f[j] * rs;
        near |= !(fabsf(fabsf(t[j] - truncf(t[j])) - 0.5f) > 0x1p-14f);
    }
    if (near) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (!(fabsf(fabsf(t[j] - truncf(t[j])) - 0.5f) > 0x1p-14f)) t[j] = __fdiv_rn(f[j], s);
    }
    uint32_t b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        b[j] = (uint32_t)(uint8_t)(int8_t)(int)fminf(fmaxf(rintf(t[j]), -127.f), 127.f);
    return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                      b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

// 16-byte L2-coherent load (skips L1) of words another CTA wrote.
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_cg(const float* p) { return ld_cg_f32(p); }
__device__ __forceinline__ int32_t ld_cg(const int32_t* p) { return ld_cg_s32(p); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

}  // namespace w4

// ---------------------------------------------------------------- tcgen05
namespace w4 {

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole warp: allocate `ncols` TMEM columns; the base address is written to
// shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst)), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16, issued by one thread.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 / 32 consecutive columns of this warp's 32 TMEM lanes (one lane per
// thread).  The load and its tcgen05.wait::ld are one asm statement: the
// load writes its registers asynchronously, so with a separate wait the
// compiler could schedule register-only uses of the outputs (adds,
// conversions) between the two, reading them before they land.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr) : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr) : "memory");
}

// Shared-memory matrix descriptor (sm_100 format) for a K-major operand in
// the 128-byte swizzled layout: rows of 128 bytes, groups of 8 rows 1024
// bytes apart.  Fields: start address >> 4 [0,14), leading byte offset >> 4
// [16,30) (unused for this layout), stride byte offset >> 4 [32,46),
// version 1 [46,48), base offset 0 [49,52), layout type 2 = SWIZZLE_128B
// [61,64).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                       // D format: f32
         | (1u << 7)                       // A format: bf16
         | (1u << 10)                      // B format: bf16
         | ((uint32_t)(N >> 3) << 17)      // N / 8
         | ((uint32_t)(M >> 4) << 24);     // M / 16
}

// ---------------------------------------------------------------- CTA pairs
// (thread-block clusters of 2 running one tcgen05 MMA with cta_group::2)

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in
// the peer CTA).  Default semantics (release, CTA scope): the data this
// announces is this CTA's own shared memory, read by its own SM's half of a
// pair MMA, and a cluster-scope release would also wait for unrelated loads
// in flight (measured: ~1200 cycles per arrival in the dequantizing warps).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];"
                 :: "r"(cluster_addr) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster with release semantics
// at cluster scope: this CTA's earlier stores into that CTA's shared memory
// (st_shared_cluster) are visible to whoever completes the wait.
__device__ __forceinline__ void mbar_arrive_release_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 :: "r"(cluster_addr) : "memory");
}

// Store to shared memory of a CTA of the cluster (address from mapa_shared).
__device__ __forceinline__ void st_shared_cluster(uint32_t cluster_addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(cluster_addr), "f"(v) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// mbar_wait for barriers that receive arrivals from the peer CTA.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, int* err) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const long long t0 = clock64();
    const long long lim = wait_limit_of(err);
    while (true) {
        if (*abort) return false;
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (clock64() - t0 > lim) {
            *abort = 1;
            atomicCAS(err, 0, W4_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}

// All threads of both CTAs of the cluster (non-.aligned forms: callers may
// arrive from diverged lanes).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\t"
                 "barrier.cluster.wait.acquire;" ::: "memory");
}

// 2D tiled load into this CTA's shared memory whose completion is counted
// on an mbarrier of either CTA of the pair (`bar_cluster`: shared::cluster
// address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, int c0,
                                                 int c1, uint32_t bar_cluster,
                                                 uint64_t cache_policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)),
           "r"(c0), "r"(c1), "r"(bar_cluster), "l"(cache_policy)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst)), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

// D[tmem of both CTAs] (+)= A[smem of both CTAs] * B[smem of both CTAs],
// kind::f16, M = 256 split 128/128 over the pair, N split N/2 + N/2; issued
// by one thread of the even CTA.
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive once on the mbarrier at `bar`'s offset in every CTA of `cta_mask`
// when the pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        :: "r"(smem_u32(bar)), "h"(cta_mask) : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace w4
