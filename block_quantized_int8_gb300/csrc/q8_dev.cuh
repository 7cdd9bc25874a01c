// q8_dev.cuh -- device helpers for libq8 (sm_103a): inline-PTX wrappers for
// streaming loads, mbarriers, bulk async copies, warp MMA and code conversion.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "q8.h"

namespace q8 {

// ---------------------------------------------------------------------------
// global loads
// ---------------------------------------------------------------------------
// Weight codes and scales are read exactly once per call: read-only path, no
// L1 allocation, and ask L2 to fetch whole 256-byte lines (rows are streamed
// front to back, so the rest of the line is used by the neighbouring lanes and
// the next iteration).
__device__ __forceinline__ uint2 ldg_stream_u2(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ldg_stream_u4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ float4 ldg_stream_f4(const void *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}
// A 2-byte read-only load that allocates in L1 (neighbouring scales of the
// same row are read by the following k-tiles).
__device__ __forceinline__ uint32_t ldg_nc_u16(const void *p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_stream_u16(const void *p) {
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// time, for bounded waits
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Longest any wait in this library may spin before it gives up (ns).  The
// waits are for copies of a few KB from L2/HBM, normally a few microseconds.
constexpr uint64_t kWaitLimitNs = 200ull * 1000ull * 1000ull;  // 0.2 s

// ---------------------------------------------------------------------------
// mbarrier (CTA scope) and bulk async copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// After giving up on a wait: keep this thread -- so its CTA and the CTA's
// shared memory -- alive for a bounded time, so that bulk copies already
// issued into that shared memory land before it is released.
constexpr uint64_t kDrainNs = 2ull * 1000ull * 1000ull;  // 2 ms
__device__ __forceinline__ void drain_after_timeout() {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < kDrainNs) __nanosleep(1000);
}

// Wait for phase `parity` of `bar` to complete; false if limit_ns passed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}
// Programmatic dependent launch: let the next kernel in the stream start
// launching (its CTAs take SM slots as ours exit), and wait until the
// kernels before this one have completed and their writes are visible (a
// no-op when this kernel was not launched as a dependent).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Zero, computed from every lane's v: an instruction that cannot issue
// before the loads that produced v have returned their data in all lanes of
// the warp.  A warp that hands a shared-memory stage back to an async-proxy
// writer (a bulk or tensor copy) right after reading it must make the release
// depend on its loaded values this way: a release that only followed the
// load instructions in program order let the next copy overwrite the stage
// before the loads had read it (measured: codes of the stage's next fill
// turned up in the product).  `zero` must be 0 at run time but unknown to the
// compiler (a kernel argument): masking with a literal 0 is folded away.
__device__ __forceinline__ uint32_t warp_loaded_zero(uint32_t v, uint32_t zero) {
    return __reduce_or_sync(0xFFFFFFFFu, v & zero);
}

// 1-D bulk copy global -> shared, completing `bytes` on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// code conversion
// ---------------------------------------------------------------------------
// Four int8 codes (one 32-bit word) -> two bf16x2 words, exactly.
// bf16 holds integers 0..255 exactly, but its 7 fraction bits give unit
// spacing only on [128, 256): so write 128 + (c & 0x7f) there (0x43 is the
// high byte of 128.0 in bf16) and subtract 128 (c >= 0) or 256 (c < 0, the
// sign bit of c lands on the exponent LSB and turns 0x4300 into 0x4380):
//   c >= 0: (128 + c) - 128 = c;   c < 0: (128 + c + 128) - 256 = c.
// lo = codes 0,1 ; hi = codes 2,3 (element 0 in the low half).
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ void codes4_to_bf16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t plo = __byte_perm(w, 0x43434343u, 0x4140);   // [43 c1 43 c0]
    const uint32_t phi = __byte_perm(w, 0x43434343u, 0x4342);   // [43 c3 43 c2]
    const uint32_t alo = plo & 0xFF7FFF7Fu;                      // 128 + (c & 0x7f)
    const uint32_t ahi = phi & 0xFF7FFF7Fu;
    const uint32_t blo = (plo & 0x00800080u) | 0x43004300u;     // 128 or 256
    const uint32_t bhi = (phi & 0x00800080u) | 0x43004300u;
    lo = bf16x2_sub(alo, blo);
    hi = bf16x2_sub(ahi, bhi);
}

// Four int8 codes -> two f16x2 words, exactly.  binary16 has 10 fraction
// bits, so 0x6400 | u is 1024 + u for a byte u = c ^ 0x80 = c + 128, and one
// packed subtraction of 1152 (0x6480) leaves c.
__device__ __forceinline__ void codes4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t plo = __byte_perm(u, 0x64646464u, 0x4140);   // [64 u1 64 u0]
    const uint32_t phi = __byte_perm(u, 0x64646464u, 0x4342);   // [64 u3 64 u2]
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(plo), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(phi), "r"(0x64806480u));
}

// D = A B on int8: A 16 x 32 (row), B 32 x 8 (column), int32 out.
// Fragments: a0 / a1 rows g / g + 8 at k = 4t..4t+3, a2 / a3 the same rows at
// k = 16 + 4t..; b0 / b1 column g at k = 4t.. and 16 + 4t..; d0 d1 row g,
// columns 2t, 2t + 1, d2 d3 row g + 8.
__device__ __forceinline__ void mma_s8_16832(int &d0, int &d1, int &d2, int &d3, uint32_t a0, uint32_t a1,
                                             uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0));
}

// Two floats -> f16x2 (a in the low half), round to nearest even.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// Four int8 codes -> four floats, exactly: 0x4B000000 | u is 2^23 + u for a
// byte u, and u = c ^ 0x80 = c + 128.
__device__ __forceinline__ void codes4_to_f32(uint32_t w, float &f0, float &f1, float &f2, float &f3) {
    const uint32_t u = w ^ 0x80808080u;
    const float bias = 8388736.0f;  // 2^23 + 128
    f0 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - bias;
    f1 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - bias;
    f2 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - bias;
    f3 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - bias;
}

// bf16 pair (low, high) -> floats
__device__ __forceinline__ float bf16lo_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// bf16 bits b that binary16 holds exactly: zero, or |b| in [2^-17, 65504]
// (biased exponent >= 110 and magnitude bits <= 0x477F = 65280, the largest
// bf16 not above 65504); NaN and infinity fail the second test.  Integer
// compares only (measured: the same test on floats made the pipeline
// kernel's x preparation several times slower).
__device__ __forceinline__ bool bf16_fits_f16(uint32_t b) {
    const uint32_t m = b & 0x7FFFu;
    return m == 0u || m - 0x3700u <= 0x477Fu - 0x3700u;
}

// binary16 bits -> float (exact)
__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
    float f;
    asm("{\n\t.reg .b16 t;\n\tmov.b16 t, %1;\n\tcvt.f32.f16 %0, t;\n\t}" : "=f"(f) : "h"((unsigned short)h));
    return f;
}

// ---------------------------------------------------------------------------
// warp MMA: D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16_16816(float &d0, float &d1, float &d2, float &d3,
                                               uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, binary16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float &d0, float &d1, float &d2, float &d3,
                                              uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace q8
