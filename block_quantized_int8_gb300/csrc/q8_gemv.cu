// q8_gemv.cu -- Q8_0 W8A16 matrix-vector product (M = 1) over one or several
// matrices in one persistent launch.
//
// y[n] = sum_k s[n][k/32] * q[n][k] * x[k].  "Frigg" README, "The machine"
// (at batch 1 every decode matmul is this GEMV shape and it is bound by
// memory bandwidth) and Finding 3 (a decode step of many small matrices is
// launch-bound first: hence one launch for the whole list).
//
// Design (warp-specialised, bulk-copy fed):
//  * A "stage" is RT consecutive weight rows with their full K.  Rows of the
//    row-major codes q[N][K] and scales s[N][K/32] are contiguous, so a stage
//    is ONE bulk async copy of RT*K code bytes plus one of RT*K/16 scale bytes.
//  * Each CTA owns a contiguous, byte-balanced range of the stages of all
//    matrices (the host cuts the list so every CTA streams the same bytes).
//  * Lane 0 of warp 0 also produces: it keeps kStages copies in flight
//    (cp.async.bulk -> shared memory, completion on a "full" mbarrier) and
//    refills a slot once every warp has released it ("empty" mbarrier).  A
//    CTA is 8 warps, so two CTAs fit on an SM without capping registers
//    (a ninth warp would put five warps on one SM sub-partition).
//  * All 8 warps consume; each copies its share of a stage into registers and
//    releases the slot before doing any arithmetic.  A row is split into P = pow2(ceil(K/2048))
//    K-slices; each warp always owns the same slice (w % P), so its part of x
//    stays in registers as fp32 (at most 64 values per lane), reloaded only
//    when the matrix changes.  Lanes read 16-byte chunks of the row from
//    shared memory (consecutive lanes, consecutive chunks: no bank
//    conflicts), turn codes into floats exactly (2^23 + byte trick) and use
//    packed fma.rn.f32x2 for the dot product; each half block's sum is scaled
//    by its binary16 scale in fp32; a warp shuffle tree sums the lanes.
//  * With P > 1 the slices of a row are added in slice order by whichever warp
//    finishes the row last (shared-memory counter; nobody waits), so results
//    are deterministic and independent of how matrices are batched.
// Every wait is bounded (Q8_DEV_TIMEOUT on expiry); no barrier spans warps
// that might have given up.
#include <algorithm>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = kConsumerWarps * 32;
constexpr int kStages = 3;
constexpr int kUnits = 16;                     // (row, slice) units per stage = RT * P
constexpr int kCodeBytes = 32768;              // RT * K <= 32 KB per stage
constexpr int kScaleBytes = kCodeBytes / 16 + 16;  // RT * K / 16, plus up to 14 bytes of alignment offset
constexpr int kStageBytes = kCodeBytes + kScaleBytes;
constexpr int kMaxK = 8 * 2048;                // P <= 8 with 2048-wide slices
constexpr int kMaxGrid = 1024;
constexpr int kJMax = 4;                       // 16-code chunks per lane per slice (2048 k)

struct GDesc {
    const int8_t *q;
    const uint16_t *s;
    const uint16_t *x;
    float *y;
    int32_t N;
    int32_t K;
    int32_t nb;          // K / 32
    int32_t P;           // slices per row (power of two <= 8)
    int32_t RT;          // rows per stage = min(16 / P, 24576 / K)
    int32_t bps;         // blocks per slice
    int32_t stage_begin; // first global stage index of this matrix
    int32_t stages;      // ceil(N / RT)
};

struct GParams {
    GDesc d[Q8_MAX_BATCH];
    uint32_t *status;
    int32_t count;
    int32_t total_stages;
    int32_t cta_begin[kMaxGrid + 1];  // CTA c owns stages [cta_begin[c], cta_begin[c+1])
};

struct Smem {
    alignas(128) uint8_t stage[kStages][kStageBytes];
    float red[2 * kStages][kUnits][8];   // per-stage slice sums (P > 1), ring of 2*kStages
    uint32_t cnt[2 * kStages][kUnits];
    uint64_t full[kStages];
    uint64_t empty[kStages];
};

__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
    return (static_cast<unsigned long long>(__float_as_uint(b)) << 32) | __float_as_uint(a);
}
__device__ __forceinline__ unsigned long long fma_f32x2(unsigned long long a, unsigned long long b,
                                                        unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long add_f32x2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Four codes of word w times four activations (two packed pairs) added to acc.
// Codes become exact floats: 0x4B000000 | (c ^ 0x80) is 2^23 + 128 + c.
__device__ __forceinline__ unsigned long long dot4(uint32_t w, unsigned long long x01, unsigned long long x23,
                                                   unsigned long long acc) {
    const uint32_t u = w ^ 0x80808080u;
    const unsigned long long m01 = (static_cast<unsigned long long>(__byte_perm(u, 0x4B000000u, 0x7651)) << 32) |
                                   __byte_perm(u, 0x4B000000u, 0x7650);
    const unsigned long long m23 = (static_cast<unsigned long long>(__byte_perm(u, 0x4B000000u, 0x7653)) << 32) |
                                   __byte_perm(u, 0x4B000000u, 0x7652);
    const unsigned long long nb2 = 0xCB000080CB000080ull;  // (-(2^23 + 128), -(2^23 + 128))
    acc = fma_f32x2(add_f32x2(m01, nb2), x01, acc);
    acc = fma_f32x2(add_f32x2(m23, nb2), x23, acc);
    return acc;
}


// One lane's share of a stage for rows A and B: NJ chunks of 16 codes and
// their half-block scales, pulled from shared memory into registers so the
// slot can be handed back to the producer before any arithmetic.
template <int NJ>
struct RowPair {
    uint4 wA[NJ], wB[NJ];
    uint32_t h[NJ];  // binary16 scale bits: row A low half, row B high half
};

// FULL: both rows exist and every lane has NJ chunks (the common case), so
// the loads need no predicates and no zero fill.
template <int NJ, bool FULL>
__device__ __forceinline__ void load_rows(RowPair<NJ> &rp, const uint8_t *cA, const uint8_t *cB,
                                          const uint16_t *sA, const uint16_t *sB, bool vA, bool vB, int lane,
                                          int chunks_slice) {
    if constexpr (FULL) {
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int c = lane + 32 * j;
            rp.wA[j] = *reinterpret_cast<const uint4 *>(cA + 16 * c);
            rp.wB[j] = *reinterpret_cast<const uint4 *>(cB + 16 * c);
            rp.h[j] = static_cast<uint32_t>(sA[c >> 1]) | (static_cast<uint32_t>(sB[c >> 1]) << 16);
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int c = lane + 32 * j;
        const bool in = c < chunks_slice;
        rp.wA[j] = make_uint4(0u, 0u, 0u, 0u);
        rp.wB[j] = rp.wA[j];
        rp.h[j] = 0u;
        if (in && vA) {
            rp.wA[j] = *reinterpret_cast<const uint4 *>(cA + 16 * c);
            rp.h[j] = sA[c >> 1];
        }
        if (in && vB) {
            rp.wB[j] = *reinterpret_cast<const uint4 *>(cB + 16 * c);
            rp.h[j] |= static_cast<uint32_t>(sB[c >> 1]) << 16;
        }
    }
}

// Dot products of the lane's chunks with its x chunks, each half block's sum
// scaled by its binary16 scale.  NJ is a compile-time constant so both rows'
// chunks form one straight-line block the scheduler can interleave; two packed
// accumulators per chunk keep the fma.rn.f32x2 dependency chains short.
template <int NJ, int KJ>
__device__ __forceinline__ void dot_rows(const RowPair<NJ> &rp, const unsigned long long (&xr)[KJ][8],
                                         float &accA, float &accB) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        unsigned long long a0 = dot4(rp.wA[j].x, xr[j][0], xr[j][1], 0ull);
        unsigned long long a1 = dot4(rp.wA[j].y, xr[j][2], xr[j][3], 0ull);
        unsigned long long b0 = dot4(rp.wB[j].x, xr[j][0], xr[j][1], 0ull);
        unsigned long long b1 = dot4(rp.wB[j].y, xr[j][2], xr[j][3], 0ull);
        a0 = dot4(rp.wA[j].z, xr[j][4], xr[j][5], a0);
        a1 = dot4(rp.wA[j].w, xr[j][6], xr[j][7], a1);
        b0 = dot4(rp.wB[j].z, xr[j][4], xr[j][5], b0);
        b1 = dot4(rp.wB[j].w, xr[j][6], xr[j][7], b1);
        const unsigned long long a = add_f32x2(a0, a1);
        const unsigned long long b = add_f32x2(b0, b1);
        accA = fmaf(f16_bits_to_f32(rp.h[j] & 0xFFFFu), __uint_as_float(static_cast<uint32_t>(a)) +
                                                           __uint_as_float(static_cast<uint32_t>(a >> 32)), accA);
        accB = fmaf(f16_bits_to_f32(rp.h[j] >> 16), __uint_as_float(static_cast<uint32_t>(b)) +
                                                       __uint_as_float(static_cast<uint32_t>(b >> 32)), accB);
    }
}

// Load this warp's part of the stage, release the slot, then compute.
template <int NJ, int KJ, bool FULL>
__device__ __forceinline__ void stage_rows(const uint8_t *cA, const uint8_t *cB, const uint16_t *sA,
                                           const uint16_t *sB, bool vA, bool vB, int lane, int chunks_slice,
                                           const unsigned long long (&xr)[KJ][8], uint64_t *empty_bar,
                                           float &accA, float &accB) {
    RowPair<NJ> rp;
    load_rows<NJ, FULL>(rp, cA, cB, sA, sB, vA, vB, lane, chunks_slice);
    // the arrive has release semantics: every lane's shared-memory reads above
    // are ordered before the producer may overwrite the slot
    __syncwarp();
    if (lane == 0) {
        asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_addr(empty_bar)) : "memory");
    }
    dot_rows<NJ, KJ>(rp, xr, accA, accB);
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ int find_gdesc(const GParams &p, int stage) {
    int d = 0;
    while (d + 1 < p.count && stage >= p.d[d + 1].stage_begin) ++d;
    return d;
}

// The work of one CTA over stages [begin, end); KJ is the number of 16-code
// chunks per lane in a warp's K slice (4: slices up to 2048 wide).
// `ring` counts the stages this CTA has already passed through its ring of
// kStages slots; slot and mbarrier phase follow from it.
template <int KJ>
__device__ __forceinline__ void cta_work(const GParams &p, Smem &sm, int begin, int end, int warp, int lane,
                                         int ring) {
    // Lane 0 of warp 0 is also the producer.  Before warp 0 consumes stage k it
    // tops the ring up: stages up to k + kStages - 1 are issued as soon as their
    // slot is free (non-blocking check); stage k itself is issued even if that
    // means waiting for the slowest warp to release its slot, so no consumer can
    // wait on a copy that nobody will start.
    const int nstages = end - begin;
    int pi = 0;                       // stages issued so far (producer lane only)
    int pd = find_gdesc(p, begin);    // descriptor of the next stage to issue
    bool prod_ok = true;
    auto produce = [&](int upto) {
        while (prod_ok && pi < nstages && pi <= upto) {
            const int q = ring + pi;  // ring position of the stage to issue
            const int slot = q % kStages;
            if (q >= kStages) {
                const uint32_t par = ((q / kStages) - 1) & 1;
                const bool must = pi <= upto - (kStages - 1);
                if (must) {
                    if (!mbar_wait_bounded(&sm.empty[slot], par)) {
                        prod_ok = false;
                        if (p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
                        return;
                    }
                } else if (!mbar_test_wait(&sm.empty[slot], par)) {
                    return;
                }
            }
            const int i = begin + pi;
            while (i >= p.d[pd].stage_begin + p.d[pd].stages) ++pd;
            const GDesc &D = p.d[pd];
            const int r0 = (i - D.stage_begin) * D.RT;
            const int rows = min(D.RT, D.N - r0);
            const uint32_t cbytes = static_cast<uint32_t>(rows) * static_cast<uint32_t>(D.K);
            // scales: bulk copies need 16-byte aligned source AND destination, so
            // the stage keeps them at the same address offset mod 16 as in global
            // memory; the unaligned head and tail (< 16 bytes each) go by plain
            // copies, published by the arrive below
            const uint32_t sbytes = static_cast<uint32_t>(rows) * static_cast<uint32_t>(D.nb) * 2u;
            const int64_t sstart = static_cast<int64_t>(r0) * D.nb * 2;
            const uint32_t a = static_cast<uint32_t>(sstart & 15);
            const uint8_t *gs = reinterpret_cast<const uint8_t *>(D.s) + sstart;
            uint8_t *dst = sm.stage[slot];
            uint8_t *sdst = dst + kCodeBytes + a;
            const uint32_t head = min(sbytes, a ? 16u - a : 0u);
            const uint32_t body = (sbytes - head) & ~15u;
            for (uint32_t b = 0; b < head; b += 2)
                *reinterpret_cast<uint16_t *>(sdst + b) = *reinterpret_cast<const uint16_t *>(gs + b);
            for (uint32_t b = head + body; b < sbytes; b += 2)
                *reinterpret_cast<uint16_t *>(sdst + b) = *reinterpret_cast<const uint16_t *>(gs + b);
            mbar_arrive_expect_tx(&sm.full[slot], cbytes + body);
            bulk_g2s(dst, D.q + static_cast<int64_t>(r0) * D.K, cbytes, &sm.full[slot]);
            if (body) bulk_g2s(sdst + head, gs + head, body, &sm.full[slot]);
            ++pi;
        }
    };

    // ---------------------------------------------------------------- consumers
    int d = find_gdesc(p, begin);
    int cur_d = -1;
    unsigned long long xr[KJ][8];  // this lane's x chunks as packed fp32 pairs
    int slice = 0, nj = 0, k0 = 0, chunks_slice = 0;
    for (int i = begin, k = 0; i < end; ++i, ++k) {
        if (warp == 0 && lane == 0) produce(k + kStages - 1);
        __syncwarp();
        while (i >= p.d[d].stage_begin + p.d[d].stages) ++d;
        const GDesc &D = p.d[d];
        if (d != cur_d) {
            // (re)load this warp's slice of x into registers as fp32 pairs
            cur_d = d;
            slice = warp & (D.P - 1);
            const int kb0 = slice * D.bps;
            const int kb1 = min(D.nb, kb0 + D.bps);
            chunks_slice = (kb1 - kb0) * 2;  // 16-code chunks in the slice
            k0 = kb0 * 32;
            nj = (chunks_slice + 31) / 32;
#pragma unroll
            for (int j = 0; j < KJ; ++j) {
                const int c = lane + 32 * j;
                uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
                if (c < chunks_slice) {
                    const uint4 *xp = reinterpret_cast<const uint4 *>(D.x + k0 + 16 * c);
                    a = __ldg(xp);
                    b = __ldg(xp + 1);
                }
                const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) xr[j][e] = f2_pack(bf16lo_f32(v[e]), bf16hi_f32(v[e]));
            }
        }
        const int slot = (ring + k) % kStages;
        if (!mbar_wait_bounded(&sm.full[slot], ((ring + k) / kStages) & 1)) {
            if (lane == 0 && p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
            return;
        }
        const uint8_t *codes = sm.stage[slot];
        const int r0 = (i - D.stage_begin) * D.RT;
        const uint16_t *scales = reinterpret_cast<const uint16_t *>(
            sm.stage[slot] + kCodeBytes + ((static_cast<int64_t>(r0) * D.nb * 2) & 15));
        const int rows = min(D.RT, D.N - r0);
        // this warp's two units of the stage: rows rA and rB, both of slice `slice`
        const int rA = warp / D.P;
        const int rB = (warp + kConsumerWarps) / D.P;
        const bool vA = rA < rows, vB = rB < rows;
        const uint8_t *cA = codes + rA * D.K + k0;
        const uint8_t *cB = codes + rB * D.K + k0;
        const uint16_t *sA = scales + rA * D.nb + (k0 >> 5);
        const uint16_t *sB = scales + rB * D.nb + (k0 >> 5);
        float accA = 0.f, accB = 0.f;
        if (vA && vB && chunks_slice == 32 * nj) {
            switch (nj) {
                case 1: stage_rows<1, KJ, true>(cA, cB, sA, sB, vA, vB, lane, chunks_slice, xr, &sm.empty[slot], accA, accB); break;
                case 2: stage_rows<2, KJ, true>(cA, cB, sA, sB, vA, vB, lane, chunks_slice, xr, &sm.empty[slot], accA, accB); break;
                case 3: if constexpr (KJ >= 3) stage_rows<3, KJ, true>(cA, cB, sA, sB, vA, vB, lane, chunks_slice, xr, &sm.empty[slot], accA, accB); break;
                default: if constexpr (KJ >= 4) stage_rows<4, KJ, true>(cA, cB, sA, sB, vA, vB, lane, chunks_slice, xr, &sm.empty[slot], accA, accB); break;
            }
        } else {
            switch (nj) {
                case 1: stage_rows<1, KJ, false>(cA, cB, sA, sB, vA, vB, lane, chunks_slice, xr, &sm.empty[slot], accA, accB); break;
                case 2: stage_rows<2, KJ, false>(cA, cB, sA, sB, vA, vB, lane, chunks_slice, xr, &sm.empty[slot], accA, accB); break;
                case 3: if constexpr (KJ >= 3) stage_rows<3, KJ, false>(cA, cB, sA, sB, vA, vB, lane, chunks_slice, xr, &sm.empty[slot], accA, accB); break;
                default: if constexpr (KJ >= 4) stage_rows<4, KJ, false>(cA, cB, sA, sB, vA, vB, lane, chunks_slice, xr, &sm.empty[slot], accA, accB); break;
            }
        }
        // reduce both rows at once: after the first exchange lanes 0-15 carry
        // row A and lanes 16-31 row B, then a 4-step tree within each half
        {
            const bool hi = (lane & 16) != 0;
            const float keep = hi ? accB : accA;
            const float give = hi ? accA : accB;
            float v = keep + __shfl_xor_sync(0xffffffffu, give, 16);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            const int row = hi ? rB : rA;
            const bool valid = hi ? vB : vA;
            if ((lane & 15) == 0 && valid) {
                if (D.P == 1) {
                    D.y[r0 + row] = v;
                } else {
                    const int rs = (ring + k) % (2 * kStages);
                    sm.red[rs][row][slice] = v;
                    __threadfence_block();
                    const uint32_t prev = atomicAdd(&sm.cnt[rs][row], 1u);
                    if (prev == static_cast<uint32_t>(D.P - 1)) {
                        __threadfence_block();
                        float t = sm.red[rs][row][0];
                        for (int sl = 1; sl < D.P; ++sl) t += sm.red[rs][row][sl];
                        D.y[r0 + row] = t;
                        sm.cnt[rs][row] = 0u;
                    }
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const __grid_constant__ GParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int begin = p.cta_begin[blockIdx.x];
    const int end = p.cta_begin[blockIdx.x + 1];

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kConsumerWarps);
        }
        fence_mbar_init();
    }
    for (int i = tid; i < 2 * kStages * kUnits; i += kThreads) (&sm.cnt[0][0])[i] = 0u;
    __syncthreads();
    if (end > begin) cta_work<kJMax>(p, sm, begin, end, warp, lane, 0);
}

int g_configured_dev = -1;
int g_occ = 0;

}  // namespace

bool gemv_supported(const q8_linear_desc *descs, int count) {
    for (int i = 0; i < count; ++i)
        if (descs[i].K > kMaxK) return false;
    return true;
}

q8_status launch_gemv(const q8_linear_desc *descs, int count, uint32_t *dev_status, cudaStream_t stream) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (g_configured_dev != di->device) {
        if (cudaFuncSetAttribute(gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sizeof(Smem))) != cudaSuccess)
            return Q8_ERR_CUDA;
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, gemv_kernel, kThreads, sizeof(Smem)) != cudaSuccess)
            return Q8_ERR_CUDA;
        g_occ = std::max(o, 1);
        g_configured_dev = di->device;
    }
    static thread_local GParams p;  // large: keep it off the stack
    double total_bytes = 0.0;
    int stages = 0;
    for (int i = 0; i < count; ++i) {
        GDesc &D = p.d[i];
        const int K = static_cast<int>(descs[i].K);
        int P = 1;
        while (P * 2048 < K) P *= 2;
        D.q = descs[i].q;
        D.s = descs[i].s;
        D.x = descs[i].x;
        D.y = descs[i].y;
        D.N = static_cast<int32_t>(descs[i].N);
        D.K = K;
        D.nb = K / 32;
        D.P = P;
        D.RT = std::min(kUnits / P, kCodeBytes / K);
        D.bps = (D.nb + P - 1) / P;
        D.stage_begin = stages;
        D.stages = (D.N + D.RT - 1) / D.RT;
        stages += D.stages;
        total_bytes += static_cast<double>(D.N) * K * 1.0625;
    }
    p.status = dev_status;
    p.count = count;
    p.total_stages = stages;
    if (stages == 0) return Q8_OK;
    const int grid = std::min(std::min(stages, di->sm_count * g_occ), kMaxGrid);
    // cut the stage list into `grid` ranges of (nearly) equal bytes
    int c = 0;
    double acc = 0.0;
    p.cta_begin[0] = 0;
    for (int i = 0; i < count && c < grid - 1; ++i) {
        const GDesc &D = p.d[i];
        const double full = static_cast<double>(D.RT) * D.K * 1.0625;
        for (int st = 0; st < D.stages && c < grid - 1; ++st) {
            const int rows = std::min(D.RT, D.N - st * D.RT);
            acc += full * rows / D.RT;
            while (c < grid - 1 && acc >= total_bytes * (c + 1) / grid) p.cta_begin[++c] = D.stage_begin + st + 1;
        }
    }
    while (c < grid) p.cta_begin[++c] = stages;
    const int launch = grid;
    gemv_kernel<<<launch, kThreads, sizeof(Smem), stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

}  // namespace q8
