// q8_chain.cu -- a dependent chain of skinny matmuls, run on the device.
//
// Step i multiplies its input x_i by its Q8_0 weights into y_i (fp32); the
// next step's input x_{i+1} (bf16) is made from y_i on the device by a small
// kernel: the RMS normalisation (no learnable weight, eps = 1e-6) of the
// first K_{i+1} values of each row, or of SwiGLU(a, b) = silu(a) * b over
// a = y[0, K_{i+1}) and b = y[K_{i+1}, 2 K_{i+1}).  "Frigg" README: the model
// card (RMSNorm without weights, eps 1e-6; SwiGLU MLP of width 4,096; the
// two 16-layer modules run L L L H L L L H per token) and Finding 3 (a
// decode step is a long chain of small dependent launches: launch-bound
// before it is bandwidth-bound, hence one graph whose launches overlap).
//
// Every kernel of the chain is a programmatic dependent of the one before
// it.  A matmul loads its first weight stages while the normalisation
// before it runs and reads x only after that kernel has completed; a
// normalisation lets the next matmul launch at once and reads y only after
// its matmul has completed.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kGlueThreads = 256;   // the general kernel (any K)
constexpr int kFastThreads = 1024;  // the register kernel: K <= 8 * 1024

struct GlueParams {
    const float *y;
    uint16_t *x;
    int64_t ldy;
    int64_t ldx;
    int32_t K;       // values per row of x
    int32_t swiglu;  // 1: x = norm(silu(y[0:K)) * y[K:2K)); 0: x = norm(y[0:K))
};

__device__ __forceinline__ float glue_value(const float *yr, int K, int k, int swiglu) {
    const float a = yr[k];
    if (!swiglu) return a;
    return a / (1.0f + expf(-a)) * yr[K + k];
}

// One CTA per row of x.  The sum of squares is reduced in a fixed order (each
// thread's strided sum, the warps' shuffle trees, then the 8 warp sums in
// warp order), so the bits do not depend on timing.
__global__ void __launch_bounds__(kGlueThreads) glue_kernel(const __grid_constant__ GlueParams p) {
    // the next matmul reads only weights before its own wait
    pdl_launch_dependents();
    // y is the previous kernel's output
    pdl_wait_prior();
    __shared__ float warp_ss[kGlueThreads / 32];
    const int m = blockIdx.x;
    const float *yr = p.y + m * p.ldy;
    float ss = 0.f;
    for (int k = threadIdx.x; k < p.K; k += kGlueThreads) {
        const float v = glue_value(yr, p.K, k, p.swiglu);
        ss = fmaf(v, v, ss);
    }
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < kGlueThreads / 32; ++w) tot += warp_ss[w];
    // 1 / sqrt(mean + eps) with IEEE division and square root
    const float r = 1.0f / sqrtf(tot / static_cast<float>(p.K) + 1e-6f);
    uint16_t *xr = p.x + m * p.ldx;
    for (int k = threadIdx.x; k < p.K; k += kGlueThreads)
        xr[k] = __bfloat16_as_ushort(__float2bfloat16_rn(glue_value(yr, p.K, k, p.swiglu) * r));
}

// K <= G * 1024: thread t holds the values k = t + 1024 j (j < G) in
// registers, loaded all at once (so their latencies overlap) and read from
// y only once; its sum of squares in j order, then the warps' shuffle trees
// and the 32 warp sums in warp order.
template <int G>
__global__ void __launch_bounds__(kFastThreads) glue_regs_kernel(const __grid_constant__ GlueParams p) {
    pdl_launch_dependents();
    pdl_wait_prior();
    __shared__ float warp_ss[kFastThreads / 32];
    const int m = blockIdx.x;
    const float *yr = p.y + m * p.ldy;
    float a[G], b[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const int k = threadIdx.x + kFastThreads * j;
        a[j] = k < p.K ? yr[k] : 0.f;
        b[j] = (p.swiglu && k < p.K) ? yr[p.K + k] : 0.f;
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < G; ++j) {
        if (p.swiglu) a[j] = a[j] / (1.0f + expf(-a[j])) * b[j];
        ss = fmaf(a[j], a[j], ss);
    }
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < kFastThreads / 32; ++w) tot += warp_ss[w];
    const float r = 1.0f / sqrtf(tot / static_cast<float>(p.K) + 1e-6f);
    uint16_t *xr = p.x + m * p.ldx;
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const int k = threadIdx.x + kFastThreads * j;
        if (k < p.K) xr[k] = __bfloat16_as_ushort(__float2bfloat16_rn(a[j] * r));
    }
}

q8_status launch_glue(const GlueParams &g, int M, cudaStream_t stream) {
    cudaError_t e;
    if (g.K <= kFastThreads)
        e = launch_kernel(glue_regs_kernel<1>, dim3(M), dim3(kFastThreads), 0, stream, true, g);
    else if (g.K <= 2 * kFastThreads)
        e = launch_kernel(glue_regs_kernel<2>, dim3(M), dim3(kFastThreads), 0, stream, true, g);
    else if (g.K <= 4 * kFastThreads)
        e = launch_kernel(glue_regs_kernel<4>, dim3(M), dim3(kFastThreads), 0, stream, true, g);
    else if (g.K <= 8 * kFastThreads)
        e = launch_kernel(glue_regs_kernel<8>, dim3(M), dim3(kFastThreads), 0, stream, true, g);
    else
        e = launch_kernel(glue_kernel, dim3(M), dim3(kGlueThreads), 0, stream, true, g);
    return e == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

q8_linear_desc desc_of(const q8_chain_step &st) {
    q8_linear_desc d{};
    d.q = st.q;
    d.s = st.s;
    d.x = st.x;
    d.y = st.y;
    d.N = st.N;
    d.K = st.K;
    d.ldx = st.ldx;
    d.ldy = st.ldy;
    return d;
}

// The workspace region of each step: one region per distinct (N, K), so
// that every region always holds the same layout (its counters stay zero
// from one step to the next and nothing needs clearing); 256-byte aligned.
// Returns the total.
size_t chain_regions(const q8_chain_step *steps, int count, int M, size_t *off) {
    size_t total = 0;
    for (int i = 0; i < count; ++i) {
        int j = 0;
        while (j < i && !(steps[j].N == steps[i].N && steps[j].K == steps[i].K)) ++j;
        if (j < i) {
            if (off) off[i] = off[j];
            continue;
        }
        const q8_linear_desc d = desc_of(steps[i]);
        SplitPlan plans[1];
        size_t sched_off;
        const size_t need = skinny_workspace(&d, 1, M, plans, &sched_off);
        if (off) off[i] = total;
        total += (need + 255) / 256 * 256;
    }
    return total;
}

}  // namespace

size_t chain_workspace(const q8_chain_step *steps, int count, int M) { return chain_regions(steps, count, M, nullptr); }

q8_status check_chain(const q8_chain_step *steps, int count, int M) {
    if (!steps || count < 1 || count > Q8_MAX_CHAIN) return Q8_ERR_ARG;
    if (M < 1 || M > Q8_SKINNY_MAX_M) return Q8_ERR_SHAPE;
    for (int i = 0; i < count; ++i) {
        const q8_chain_step &st = steps[i];
        const q8_linear_desc d = desc_of(st);
        const q8_status s = check_skinny_args(d, M);
        if (s != Q8_OK) return s;
        if (st.N < 1) return Q8_ERR_SHAPE;
        if (i + 1 == count) {
            if (st.next != Q8_CHAIN_END) return Q8_ERR_ARG;
            continue;
        }
        const int64_t kn = steps[i + 1].K;
        if (st.next == Q8_CHAIN_RMSNORM) {
            if (kn > st.N) return Q8_ERR_SHAPE;
        } else if (st.next == Q8_CHAIN_SWIGLU_RMSNORM) {
            if (2 * kn > st.N) return Q8_ERR_SHAPE;
        } else {
            return Q8_ERR_ARG;
        }
    }
    return Q8_OK;
}

q8_status launch_chain(const q8_chain_step *steps, int count, int M, void *ws, size_t ws_bytes,
                       uint32_t *dev_status, cudaStream_t stream) {
    static thread_local size_t off[Q8_MAX_CHAIN];
    const size_t total = chain_regions(steps, count, M, off);
    if (total > ws_bytes) return Q8_ERR_WORKSPACE;
    for (int i = 0; i < count; ++i) {
        const q8_linear_desc d = desc_of(steps[i]);
        uint8_t *region = ws ? static_cast<uint8_t *>(ws) + off[i] : nullptr;
        q8_status st = launch_skinny(&d, 1, M, Q8_VARIANT_AUTO, region, ws_bytes - off[i], dev_status, stream, true);
        if (st != Q8_OK) return st;
        if (i + 1 == count) break;
        GlueParams g;
        g.y = steps[i].y;
        g.ldy = steps[i].ldy;
        g.x = steps[i + 1].x;
        g.ldx = steps[i + 1].ldx;
        g.K = static_cast<int32_t>(steps[i + 1].K);
        g.swiglu = steps[i].next == Q8_CHAIN_SWIGLU_RMSNORM ? 1 : 0;
        st = launch_glue(g, M, stream);
        if (st != Q8_OK) return st;
    }
    return Q8_OK;
}

}  // namespace q8
