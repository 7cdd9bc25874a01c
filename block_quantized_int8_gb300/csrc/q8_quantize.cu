// q8_quantize.cu -- Q8_0 quantizer kernel (binary32 weights -> int8 codes +
// binary16 block scales).
//
// Method: "MODEL-BASELINE-RESULTS" (fak), ACT 3 item 1 (32-wide blocks,
// d = maxabs/127, int8 codes), ACT 4 "Correctness" (round half away from zero,
// never add-0.5-and-truncate), ACT 5 item 3 (exact on zeros, denormals and
// exact halves).  The scale is stored in binary16 (the page's 1.06 B/weight).
//
// GPU realisation of the exact rounding: the code of |w| against the stored
// scale s is the unique k with (k - 1/2)*s <= |w| < (k + 1/2)*s (ties go up,
// i.e. away from zero).  A binary32 estimate t = |w| * (1/s) is within a tiny
// fraction of the true quotient, so round(t) is off by at most one; the two
// products (k +- 1/2)*s are exact in binary32 (9-bit times 11-bit
// significands) and one compare in each direction fixes the estimate.
//
// Compatibility mode (Q8_QUANT_FL32): the code is the binary32 quotient
// w / d32 (IEEE division, d32 = amax/127 before the binary16 rounding of the
// stored scale) rounded half away from zero -- ACT 4's q8round applied to a
// float32 value: truncate, recover the fraction exactly, step away from zero
// when it is at least one half.
//
// Layout: 8 lanes own one block (a float4 each); a warp covers four blocks,
// 512 contiguous bytes per load, and issues the loads of four such runs
// before it converts any (one load per thread in flight was measured at
// 3.2 TB/s).  Bandwidth-bound: 4 B read + 1.0625 B written
// per weight.
#include <cuda_fp16.h>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

__device__ __forceinline__ int32_t code_of(float v, float sf, float rcp) {
    const float a = fabsf(v);
    float k = fminf(floorf(__fadd_rn(__fmul_rn(a, rcp), 0.5f)), 128.0f);
    if (__fmul_rn(__fadd_rn(k, 0.5f), sf) <= a) {
        k = __fadd_rn(k, 1.0f);
    } else if (k > 0.0f && __fmul_rn(__fsub_rn(k, 0.5f), sf) > a) {
        k = __fsub_rn(k, 1.0f);
    }
    const int32_t ki = static_cast<int32_t>(fminf(k, 127.0f));
    return v < 0.0f ? -ki : ki;
}

__device__ __forceinline__ int32_t code_fl32(float v, float d) {
    const float t = __fdiv_rn(v, d);
    const float k0 = truncf(t);
    float k = fabsf(k0);
    if (fabsf(__fsub_rn(t, k0)) >= 0.5f) k = __fadd_rn(k, 1.0f);  // t - trunc(t) is exact
    const int32_t ki = static_cast<int32_t>(fminf(k, 127.0f));
    return t < 0.0f ? -ki : ki;
}

constexpr int kUnroll = 4;  // float4 loads in flight per thread

template <bool FL32>
__global__ void __launch_bounds__(256)
quantize_kernel(const float *__restrict__ w, int64_t nblocks, uint32_t *__restrict__ q,
                uint16_t *__restrict__ s, uint32_t *__restrict__ status) {
    const int lane = threadIdx.x & 31;
    const int64_t total = nblocks * 8;  // float4 slots
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t wstride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    // a warp takes kUnroll runs of 32 float4 (4 blocks each) per iteration and
    // issues all their loads first, so that enough bytes are in flight
    for (int64_t base = warp0 * 32 * kUnroll; base < total; base += wstride * 32 * kUnroll) {
        float4 vs[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + 32 * u + lane;
            vs[u] = i < total ? ldg_stream_f4(w + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + 32 * u + lane;
            const bool valid = i < total;
            const float4 v = vs[u];
            uint32_t bad = (isfinite(v.x) && isfinite(v.y) && isfinite(v.z) && isfinite(v.w)) ? 0u : 1u;
            float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                bad |= __shfl_xor_sync(0xffffffffu, bad, off);
            }
            const float d = __fdiv_rn(amax, 127.0f);
            const __half h = __float2half_rn(d);
            const float sf = __half2float(h);
            uint32_t flags = bad ? Q8_DEV_NONFINITE : (isinf(sf) ? Q8_DEV_SCALE_OVF : 0u);
            uint32_t packed = 0;
            uint16_t sbits = __half_as_ushort(h);
            if (flags) {
                sbits = 0;
            } else if (sf != 0.0f) {
                uint32_t c0, c1, c2, c3;
                if constexpr (FL32) {
                    c0 = static_cast<uint32_t>(code_fl32(v.x, d)) & 0xFFu;
                    c1 = static_cast<uint32_t>(code_fl32(v.y, d)) & 0xFFu;
                    c2 = static_cast<uint32_t>(code_fl32(v.z, d)) & 0xFFu;
                    c3 = static_cast<uint32_t>(code_fl32(v.w, d)) & 0xFFu;
                } else {
                    const float rcp = __frcp_rn(sf);
                    c0 = static_cast<uint32_t>(code_of(v.x, sf, rcp)) & 0xFFu;
                    c1 = static_cast<uint32_t>(code_of(v.y, sf, rcp)) & 0xFFu;
                    c2 = static_cast<uint32_t>(code_of(v.z, sf, rcp)) & 0xFFu;
                    c3 = static_cast<uint32_t>(code_of(v.w, sf, rcp)) & 0xFFu;
                }
                packed = c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
            }
            if (valid) {
                q[i] = packed;
                if ((lane & 7) == 0) {
                    s[i >> 3] = sbits;
                    if (flags && status) atomicOr(status, flags);
                }
            }
        }
    }
}

q8_status launch_quantize(const float *w, int64_t rows, int64_t K, int8_t *q, uint16_t *s,
                          uint32_t *dev_status, cudaStream_t stream, int mode) {
    const int64_t nblocks = rows * (K / 32);
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    const int threads = 256;
    const int64_t warps_needed = (nblocks * 8 + 32 * kUnroll - 1) / (32 * kUnroll);
    int64_t grid = (warps_needed + (threads / 32) - 1) / (threads / 32);
    const int64_t cap = static_cast<int64_t>(di->sm_count) * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    if (mode == Q8_QUANT_FL32)
        quantize_kernel<true><<<static_cast<unsigned>(grid), threads, 0, stream>>>(
            w, nblocks, reinterpret_cast<uint32_t *>(q), s, dev_status);
    else
        quantize_kernel<false><<<static_cast<unsigned>(grid), threads, 0, stream>>>(
            w, nblocks, reinterpret_cast<uint32_t *>(q), s, dev_status);
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

}  // namespace q8
