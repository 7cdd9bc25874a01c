// q8_pipe.cu -- Q8_0 W8A16 matmul for 2 <= M <= 8 activation rows over one or
// several matrices in one persistent launch (K <= 4096).
//
// Y[m][n] = sum_k s[n][k/32] * q[n][k] * x[m][k]; "Frigg" README, Finding 8
// (a batched W8A16 kernel reads each weight once for the whole batch of rows)
// and Finding 3 (one launch for the many small matrices of a decode step).
//
// Design (bulk-copy fed, tensor cores through warp mma):
//  * A stage is RT = 16 weight rows (8 when K > 1984) with their full K.  Lane
//    0 of warp 0 copies each row with one cp.async.bulk into a shared-memory
//    row padded to K + 16 bytes, and the RT*K/16 scale bytes (contiguous in
//    global memory) with one more; kStages stages in flight per CTA, two CTAs
//    per SM, byte-balanced contiguous stage ranges per CTA (as q8_gemv.cu).
//  * The 8 warps split K: warp w owns blocks [w*bpw, (w+1)*bpw).  Its part of
//    x stays in registers in the mma B-fragment layout, reloaded only when
//    the matrix changes.
//  * Per 32-code block a warp runs two mma.sync.m16n8k16 (bf16 in, fp32 out)
//    with the weights as the 16-row A operand (lane (g, t) holds bytes
//    [8t, 8t+8) of rows g and g+8; the 16-byte row skew makes these reads
//    bank-conflict free) and x^T as B (columns = activation rows, zero past
//    M).  Codes become bf16 exactly (|q| <= 127); each block's fp32 result is
//    scaled by its binary16 scale.
//  * With 8-row stages each warp copies its share into registers and releases
//    the slot before any arithmetic.  The 8 partial sums of a row are added in
//    warp order 0..7 by whichever warp finishes the stage last (shared-memory
//    counter over a small ring; nobody waits), so results are deterministic
//    and independent of batching.
// Every wait is bounded (Q8_DEV_TIMEOUT on expiry).
#include <algorithm>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;
constexpr int kCodeCap = 33280;          // RT * (K + 16): 16 rows of K <= 2064 or 8 rows of K <= 4144
constexpr int kScaleCap = 2064;          // RT * K / 16 + alignment offset
constexpr int kSlotBytes = kCodeCap + kScaleCap;
constexpr int kPipeMaxK = 4096;          // x fragments: at most 16 blocks per warp
constexpr int kMaxBpw = 16;
constexpr int kMaxGrid = 1024;
// Partial-sum ring: a warp can run at most kStages stages ahead of the last
// warp's combine, so kStages + 2 entries are never reused too early.
constexpr int kRed = kStages + 2;

struct PDesc {
    const int8_t *q;
    const uint16_t *s;
    const uint16_t *x;
    float *y;
    int64_t ldx;
    int64_t ldy;
    int32_t N;
    int32_t K;
    int32_t nb;
    int32_t RT;          // rows per stage (16 or 8)
    int32_t RS;          // shared-memory row stride, K + 16
    int32_t bpw;         // blocks per warp = ceil(nb / 8)
    int32_t stage_begin;
    int32_t stages;
};

struct PParams {
    PDesc d[Q8_MAX_BATCH];
    uint32_t *status;
    int32_t count;
    int32_t M;
    int32_t cta_begin[kMaxGrid + 1];
};

struct PSmem {
    alignas(128) uint8_t slot[kStages][kSlotBytes];
    float red[kRed][kWarps][32][4];  // per-warp partial D fragments, ring over stages
    uint32_t cnt[kRed];
    uint64_t full[kStages];
    uint64_t empty[kStages];
};

__device__ __forceinline__ bool test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ int find_pdesc(const PParams &p, int stage) {
    int d = 0;
    while (d + 1 < p.count && stage >= p.d[d + 1].stage_begin) ++d;
    return d;
}

// One warp's part of a stage in registers: BPW blocks (the last ones masked
// by kb < kb1) of rows g and g+8, with their scales.
// TWO: the stage has 16 rows (a second row group g+8); with 8-row stages the
// upper half of the A operand is zero and needs no registers.
template <int BPW, bool TWO>
struct PFrag {
    uint2 cg[BPW];
    uint32_t sg[BPW];
    uint2 ch[TWO ? BPW : 1];
    uint32_t sh[TWO ? BPW : 1];
};

template <int BPW, bool TWO>
__device__ __forceinline__ void load_frag(PFrag<BPW, TWO> &f, const uint8_t *codes, const uint16_t *scales, int RS,
                                          int nb, int kb0, int kb1, int g, int t) {
#pragma unroll
    for (int j = 0; j < BPW; ++j) {
        const int kb = kb0 + j;
        f.cg[j] = make_uint2(0u, 0u);
        f.sg[j] = 0u;
        if constexpr (TWO) {
            f.ch[j] = f.cg[j];
            f.sh[j] = 0u;
        }
        if (kb < kb1) {
            f.cg[j] = *reinterpret_cast<const uint2 *>(codes + g * RS + kb * 32 + 8 * t);
            f.sg[j] = scales[g * nb + kb];
            if constexpr (TWO) {
                f.ch[j] = *reinterpret_cast<const uint2 *>(codes + (g + 8) * RS + kb * 32 + 8 * t);
                f.sh[j] = scales[(g + 8) * nb + kb];
            }
        }
    }
}

template <int BPW, bool TWO>
__device__ __forceinline__ void mma_frag(const PFrag<BPW, TWO> &f, const uint4 (&xr)[kMaxBpw], float (&acc)[4]) {
#pragma unroll
    for (int j = 0; j < BPW; ++j) {
        uint32_t g01, g23, g45, g67, h01 = 0u, h23 = 0u, h45 = 0u, h67 = 0u;
        codes4_to_bf16x2(f.cg[j].x, g01, g23);
        codes4_to_bf16x2(f.cg[j].y, g45, g67);
        if constexpr (TWO) {
            codes4_to_bf16x2(f.ch[j].x, h01, h23);
            codes4_to_bf16x2(f.ch[j].y, h45, h67);
        }
        float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
        mma_bf16_16816(d0, d1, d2, d3, g01, h01, g23, h23, xr[j].x, xr[j].y);
        mma_bf16_16816(d0, d1, d2, d3, g45, h45, g67, h67, xr[j].z, xr[j].w);
        const float sg = f16_bits_to_f32(f.sg[j]);
        acc[0] = fmaf(sg, d0, acc[0]);
        acc[1] = fmaf(sg, d1, acc[1]);
        if constexpr (TWO) {
            const float sh = f16_bits_to_f32(f.sh[j]);
            acc[2] = fmaf(sh, d2, acc[2]);
            acc[3] = fmaf(sh, d3, acc[3]);
        }
    }
}

// 8-row stages (TWO false): copy this warp's share of the stage into
// registers, hand the slot back to the producer (the release orders every
// lane's reads before any refill), then do the arithmetic.  16-row stages
// hold twice the registers, so they compute block by block straight from
// shared memory and release the slot afterwards.
template <int BPW, bool TWO>
__device__ __forceinline__ void stage_mma(const uint8_t *codes, const uint16_t *scales, int RS, int nb, int kb0,
                                          int kb1, int g, int t, const uint4 (&xr)[kMaxBpw],
                                          uint64_t *empty_bar, int lane, float (&acc)[4]) {
    if constexpr (TWO) {
#pragma unroll
        for (int j = 0; j < BPW; ++j) {
            const int kb = kb0 + j;
            if (kb < kb1) {
                PFrag<1, true> f;
                f.cg[0] = *reinterpret_cast<const uint2 *>(codes + g * RS + kb * 32 + 8 * t);
                f.ch[0] = *reinterpret_cast<const uint2 *>(codes + (g + 8) * RS + kb * 32 + 8 * t);
                f.sg[0] = scales[g * nb + kb];
                f.sh[0] = scales[(g + 8) * nb + kb];
                const uint4 xj[kMaxBpw] = {xr[j]};
                mma_frag<1, true>(f, xj, acc);
            }
        }
        __syncwarp();
        if (lane == 0)
            asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_addr(empty_bar)) : "memory");
    } else {
        PFrag<BPW, TWO> f;
        load_frag<BPW, TWO>(f, codes, scales, RS, nb, kb0, kb1, g, t);
        __syncwarp();
        if (lane == 0)
            asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_addr(empty_bar)) : "memory");
        mma_frag<BPW, TWO>(f, xr, acc);
    }
}

__global__ void __launch_bounds__(kThreads, 2) pipe_kernel(const __grid_constant__ PParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    PSmem &sm = *reinterpret_cast<PSmem *>(smem_raw);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int begin = p.cta_begin[blockIdx.x];
    const int end = p.cta_begin[blockIdx.x + 1];
    const int M = p.M;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kWarps);
        }
        for (int i = 0; i < kRed; ++i) sm.cnt[i] = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    if (end <= begin) return;

    // ---- producer (lane 0 of warp 0, between its own stages) ------------------
    const int nstages = end - begin;
    int pi = 0;
    int pd = find_pdesc(p, begin);
    bool prod_ok = true;
    auto produce = [&](int upto) {
        while (prod_ok && pi < nstages && pi <= upto) {
            const int slot = pi % kStages;
            if (pi >= kStages) {
                const uint32_t par = ((pi / kStages) - 1) & 1;
                if (pi <= upto - (kStages - 1)) {
                    if (!mbar_wait_bounded(&sm.empty[slot], par)) {
                        prod_ok = false;
                        if (p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
                        return;
                    }
                } else if (!test_wait(&sm.empty[slot], par)) {
                    return;
                }
            }
            const int i = begin + pi;
            while (i >= p.d[pd].stage_begin + p.d[pd].stages) ++pd;
            const PDesc &D = p.d[pd];
            const int r0 = (i - D.stage_begin) * D.RT;
            const int rows = min(D.RT, D.N - r0);
            uint8_t *dst = sm.slot[slot];
            // scales: same offset mod 16 as in global memory; unaligned head
            // and tail by plain copies, published by the arrive below
            const uint32_t sbytes = static_cast<uint32_t>(rows) * static_cast<uint32_t>(D.nb) * 2u;
            const int64_t sstart = static_cast<int64_t>(r0) * D.nb * 2;
            const uint32_t a = static_cast<uint32_t>(sstart & 15);
            const uint8_t *gs = reinterpret_cast<const uint8_t *>(D.s) + sstart;
            uint8_t *sdst = dst + kCodeCap + a;
            const uint32_t head = min(sbytes, a ? 16u - a : 0u);
            const uint32_t body = (sbytes - head) & ~15u;
            for (uint32_t b = 0; b < head; b += 2)
                *reinterpret_cast<uint16_t *>(sdst + b) = *reinterpret_cast<const uint16_t *>(gs + b);
            for (uint32_t b = head + body; b < sbytes; b += 2)
                *reinterpret_cast<uint16_t *>(sdst + b) = *reinterpret_cast<const uint16_t *>(gs + b);
            mbar_arrive_expect_tx(&sm.full[slot], static_cast<uint32_t>(rows) * static_cast<uint32_t>(D.K) + body);
            for (int r = 0; r < rows; ++r)
                bulk_g2s(dst + r * D.RS, D.q + static_cast<int64_t>(r0 + r) * D.K, static_cast<uint32_t>(D.K),
                         &sm.full[slot]);
            if (body) bulk_g2s(sdst + head, gs + head, body, &sm.full[slot]);
            ++pi;
        }
    };

    // ---- consumers --------------------------------------------------------------
    int d = find_pdesc(p, begin);
    int cur_d = -1;
    uint4 xr[kMaxBpw];
    int kb0 = 0, kb1 = 0;
    for (int i = begin, k = 0; i < end; ++i, ++k) {
        if (warp == 0 && lane == 0) produce(k + kStages - 1);
        __syncwarp();
        while (i >= p.d[d].stage_begin + p.d[d].stages) ++d;
        const PDesc &D = p.d[d];
        if (d != cur_d) {
            // this warp's x fragments: x[m = g][block kb][8t .. 8t+8), zero past M
            cur_d = d;
            kb0 = warp * D.bpw;
            kb1 = min(D.nb, kb0 + D.bpw);
#pragma unroll
            for (int j = 0; j < kMaxBpw; ++j) {
                const int kb = kb0 + j;
                xr[j] = make_uint4(0u, 0u, 0u, 0u);
                if (g < M && kb < kb1) xr[j] = __ldg(reinterpret_cast<const uint4 *>(D.x + g * D.ldx + kb * 32 + 8 * t));
            }
        }
        const int slot = k % kStages;
        if (!mbar_wait_bounded(&sm.full[slot], (k / kStages) & 1)) {
            if (lane == 0 && p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
            return;
        }
        const int r0 = (i - D.stage_begin) * D.RT;
        const int rows = min(D.RT, D.N - r0);
        const uint8_t *codes = sm.slot[slot];
        const uint16_t *scales = reinterpret_cast<const uint16_t *>(
            sm.slot[slot] + kCodeCap + ((static_cast<int64_t>(r0) * D.nb * 2) & 15));
        const bool two = D.RT == 16;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int bpw = D.bpw;
        uint64_t *eb = &sm.empty[slot];
        // 16-row stages have K <= 2048 (bpw <= 8); 8-row stages have K > 1984 (bpw >= 8)
        if (two) {
            if (bpw <= 2) stage_mma<2, true>(codes, scales, D.RS, D.nb, kb0, kb1, g, t, xr, eb, lane, acc);
            else if (bpw <= 4) stage_mma<4, true>(codes, scales, D.RS, D.nb, kb0, kb1, g, t, xr, eb, lane, acc);
            else if (bpw <= 6) stage_mma<6, true>(codes, scales, D.RS, D.nb, kb0, kb1, g, t, xr, eb, lane, acc);
            else stage_mma<8, true>(codes, scales, D.RS, D.nb, kb0, kb1, g, t, xr, eb, lane, acc);
        } else {
            if (bpw <= 8) stage_mma<8, false>(codes, scales, D.RS, D.nb, kb0, kb1, g, t, xr, eb, lane, acc);
            else if (bpw <= 12) stage_mma<12, false>(codes, scales, D.RS, D.nb, kb0, kb1, g, t, xr, eb, lane, acc);
            else stage_mma<16, false>(codes, scales, D.RS, D.nb, kb0, kb1, g, t, xr, eb, lane, acc);
        }
        const int rs = k % kRed;

        // publish this warp's partials; the last warp adds all 8 in warp order
        *reinterpret_cast<float4 *>(&sm.red[rs][warp][lane][0]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __threadfence_block();
        __syncwarp();
        uint32_t prev = 0;
        if (lane == 0) prev = atomicAdd(&sm.cnt[rs], 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == kWarps - 1) {
            __threadfence_block();
            float4 v = *reinterpret_cast<const float4 *>(&sm.red[rs][0][lane][0]);
#pragma unroll
            for (int w = 1; w < kWarps; ++w) {
                const float4 u = *reinterpret_cast<const float4 *>(&sm.red[rs][w][lane][0]);
                v.x += u.x;
                v.y += u.y;
                v.z += u.z;
                v.w += u.w;
            }
            const int m0 = 2 * t;
            const int ng = r0 + g;
            const int nh = r0 + g + 8;
            if (g < rows) {
                if (m0 < M) D.y[m0 * D.ldy + ng] = v.x;
                if (m0 + 1 < M) D.y[(m0 + 1) * D.ldy + ng] = v.y;
            }
            if (two && g + 8 < rows) {
                if (m0 < M) D.y[m0 * D.ldy + nh] = v.z;
                if (m0 + 1 < M) D.y[(m0 + 1) * D.ldy + nh] = v.w;
            }
            if (lane == 0) sm.cnt[rs] = 0u;
        }
    }
}

int g_configured_dev = -1;
int g_occ = 0;

}  // namespace

bool pipe_supported(const q8_linear_desc *descs, int count, int M) {
    if (M < 1 || M > 8) return false;
    for (int i = 0; i < count; ++i) {
        const int64_t K = descs[i].K;
        if (K > kPipeMaxK) return false;
        const int RT = (16 * (K + 16) <= kCodeCap) ? 16 : 8;
        if (RT * (K + 16) > kCodeCap || RT * (K / 32) * 2 + 16 > kScaleCap) return false;
    }
    return true;
}

q8_status launch_pipe(const q8_linear_desc *descs, int count, int M, uint32_t *dev_status, cudaStream_t stream) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (g_configured_dev != di->device) {
        if (cudaFuncSetAttribute(pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sizeof(PSmem))) != cudaSuccess)
            return Q8_ERR_CUDA;
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, pipe_kernel, kThreads, sizeof(PSmem)) != cudaSuccess)
            return Q8_ERR_CUDA;
        g_occ = std::max(o, 1);
        g_configured_dev = di->device;
    }
    static thread_local PParams p;
    double total_bytes = 0.0;
    int stages = 0;
    for (int i = 0; i < count; ++i) {
        PDesc &D = p.d[i];
        const int K = static_cast<int>(descs[i].K);
        D.q = descs[i].q;
        D.s = descs[i].s;
        D.x = descs[i].x;
        D.y = descs[i].y;
        D.ldx = descs[i].ldx;
        D.ldy = descs[i].ldy;
        D.N = static_cast<int32_t>(descs[i].N);
        D.K = K;
        D.nb = K / 32;
        D.RT = (16 * (K + 16) <= kCodeCap) ? 16 : 8;
        D.RS = K + 16;
        D.bpw = (D.nb + kWarps - 1) / kWarps;
        D.stage_begin = stages;
        D.stages = (D.N + D.RT - 1) / D.RT;
        stages += D.stages;
        total_bytes += static_cast<double>(D.N) * K * 1.0625;
    }
    p.status = dev_status;
    p.count = count;
    p.M = M;
    if (stages == 0) return Q8_OK;
    const int grid = std::min(std::min(stages, di->sm_count * g_occ), kMaxGrid);
    int c = 0;
    double acc = 0.0;
    p.cta_begin[0] = 0;
    for (int i = 0; i < count && c < grid - 1; ++i) {
        const PDesc &D = p.d[i];
        const double full = static_cast<double>(D.RT) * D.K * 1.0625;
        for (int st = 0; st < D.stages && c < grid - 1; ++st) {
            const int rows = std::min(D.RT, D.N - st * D.RT);
            acc += full * rows / D.RT;
            while (c < grid - 1 && acc >= total_bytes * (c + 1) / grid) p.cta_begin[++c] = D.stage_begin + st + 1;
        }
    }
    while (c < grid) p.cta_begin[++c] = stages;
    pipe_kernel<<<grid, kThreads, sizeof(PSmem), stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

}  // namespace q8
