// q8_gemm_tc.cu -- prefill-shaped Q8_0 W8A16 GEMM (M > 32) on the 5th
// generation tensor cores (tcgen05, TMEM accumulators).
//
// Y[m][n] = sum_k x[m][k] * bf16(s[n][k/32] * q[n][k]), fp32 accumulation,
// bf16 output.  "MODEL-BASELINE-RESULTS" (fak), ACT 4 (a batched prefill GEMM
// reads each weight once for all tokens, which makes the op compute-bound) and
// "Parity lane" item 2; the weight tile is dequantised to bf16 in shared
// memory so the tensor cores see a plain bf16 x bf16 product.
//
// One CTA (one per SM) computes BMP x 128 rows (m) by BN columns (n) of Y over
// all of K, in k-tiles of 64, through a ring of up to 8 shared-memory stages
// (x tiles, raw code tile, dequantised weight tile):
//   warp 0, lane 0  TMA producer: for each k-tile the BMP x tiles (bf16,
//                   128 rows x 128 bytes each, 128-byte swizzle = the tensor
//                   core's K-major layout) and the raw code tile (int8, BN
//                   rows x 64 bytes) via cp.async.bulk.tensor, once the MMAs
//                   of the stage's previous k-tile are done.
//   warps 4-11      dequantisers: code tile x block scale (scales loaded once
//                   per CTA) -> bf16(s*q) in the swizzled K-major layout of
//                   the stage's weight tile, fence.proxy.async, arrive; then
//                   the epilogue: tcgen05.ld of their 32 TMEM lanes (warp % 4)
//                   and half of the columns each, fp32 -> bf16, store Y.
//   warp 1, lane 0  MMA issuer: per k-tile and m-tile, 4 x tcgen05.mma.kind::f16
//                   (M=128, N=BN, K=16) into fp32 TMEM accumulators; the BMP
//                   m-tiles share the dequantised weight tile, so each weight
//                   is converted once per BMP x 128 rows of x.  One
//                   tcgen05.commit per k-tile frees the stage; a last one
//                   signals acc_full.
// The host picks (BMP, BN) = (2, 128), (1, 128) or (1, 64) to fill the SMs.
// All waits are bounded; on expiry the CTA reports Q8_DEV_TIMEOUT, stops
// issuing work, lets its copies and MMAs drain (bounded) and frees its TMEM.
#include <cuda.h>

#include <algorithm>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kBM = 128;          // rows of x / Y per m-tile (MMA M)
constexpr int kBK = 64;           // k per stage (128 bytes of bf16)
constexpr int kMaxStages = 8;
constexpr int kThreads = 384;           // warps 0-1 roles, 2-3 idle, 4-11 dequantise + epilogue
constexpr int kDeqThreads = 256;
constexpr int kMaxScaleBytes = 48 * 1024;  // 128 rows * (K/32) * 2 -> K <= 6144
constexpr int kSmemMax = 232448;           // dynamic shared memory of one CTA per SM
constexpr int kXTile = kBM * 128;          // one m-tile of x per stage

// Shared memory: [stages: BMP x tiles, weight tile, code tile][scales][ctl],
// tiles on 1024-byte boundaries.
struct GemmCtl {
    uint64_t full_tma[kMaxStages];   // x and codes landed (TMA bytes)
    uint64_t full_w[kMaxStages];     // weight tile dequantised (8 warps)
    uint64_t empty[kMaxStages];      // MMAs reading the stage done (commit)
    uint64_t scales_full;
    uint64_t acc_full;
    uint32_t tmem_base;
    int32_t abort_flag;
};

template <int BMP, int BN>
struct GemmSmem {
    static constexpr int kW = BN * 128;
    static constexpr int kStage = BMP * kXTile + kW + BN * 64;
    uint8_t *base;
    int ST;
    __device__ __forceinline__ uint8_t *x(int s, int i) const { return base + s * kStage + i * kXTile; }
    __device__ __forceinline__ uint8_t *w(int s) const { return base + s * kStage + BMP * kXTile; }
    __device__ __forceinline__ uint8_t *codes(int s) const { return base + s * kStage + BMP * kXTile + kW; }
    __device__ __forceinline__ uint8_t *scales() const { return base + ST * kStage; }
};

struct GemmParams {
    CUtensorMap tm_x;      // bf16 [M][ldx], box {64, 128}, 128-byte swizzle
    CUtensorMap tm_q;      // int8 [N][K],   box {64, BN}, no swizzle
    const uint16_t *s;     // binary16 scales [N][K/32]
    uint16_t *y;           // bf16 [M][ldy]
    uint32_t *status;
    int32_t M, N, K, nb;
    int32_t ST;            // ring stages
    int32_t ctl_off;       // byte offset of the control block from the aligned base
    int64_t ldy;
};

// ---- tcgen05 / TMA wrappers ---------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), leading offset unused for this layout.
__device__ __forceinline__ uint64_t sw128_desc(const void *tile) {
    const uint64_t addr = smem_addr(tile);
    uint64_t d = 0;
    d |= (addr & 0x3FFFFull) >> 4;          // start address
    d |= static_cast<uint64_t>(1) << 16;    // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;  // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;    // descriptor version (sm_100 family)
    d |= static_cast<uint64_t>(2) << 61;    // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: D f32, A bf16, B bf16, both K-major,
// N = BN, M = kBM.
template <int BN>
constexpr uint32_t idesc_for() {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
           (static_cast<uint32_t>(kBM >> 4) << 24);
}

template <int BN>
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(tmem_d), "l"(da), "l"(db), "r"(idesc_for<BN>()), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// A bounded wait that also gives up at once when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(GemmCtl &sm, uint64_t *bar, uint32_t parity, uint32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int32_t *>(&sm.abort_flag)) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicExch(&sm.abort_flag, 1);
            if (status) atomicOr(status, Q8_DEV_TIMEOUT);
            return false;
        }
    }
}

template <int BMP, int BN>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    // the tiles need 1024-byte alignment (128-byte swizzle atoms)
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const GemmSmem<BMP, BN> L{base, p.ST};
    GemmCtl &sm = *reinterpret_cast<GemmCtl *>(base + p.ctl_off);
    constexpr int kTmemCols = BMP * BN;
    const int ST = p.ST;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int n0 = blockIdx.x * BN;
    const int m0 = blockIdx.y * (BMP * kBM);
    const int KT = (p.K + kBK - 1) / kBK;
    const int rows_n = min(BN, p.N - n0);

    if (tid == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&sm.full_tma[i], 1);
            mbar_init(&sm.full_w[i], kDeqThreads / 64);  // the 4 warps of one group
            mbar_init(&sm.empty[i], 1);
        }
        mbar_init(&sm.scales_full, 1);
        mbar_init(&sm.acc_full, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_addr(&sm.tmem_base)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0 && lane == 0) {
        // -------------------------------------------------------- TMA producer
        // scales of this CTA's rows, all K: contiguous in global memory
        const uint32_t sbytes = static_cast<uint32_t>(rows_n) * static_cast<uint32_t>(p.nb) * 2u;
        const uint32_t sb16 = sbytes & ~15u;
        const uint8_t *ssrc = reinterpret_cast<const uint8_t *>(p.s + static_cast<int64_t>(n0) * p.nb);
        for (uint32_t b = sb16; b < sbytes; b += 2)
            *reinterpret_cast<uint16_t *>(L.scales() + b) = *reinterpret_cast<const uint16_t *>(ssrc + b);
        mbar_arrive_expect_tx(&sm.scales_full, sb16);
        if (sb16) bulk_g2s(L.scales(), ssrc, sb16, &sm.scales_full);
        // an m-tile wholly past M is not loaded (its rows are never stored)
        const int mtiles = min(BMP, (p.M - m0 + kBM - 1) / kBM);
        for (int kt = 0; kt < KT; ++kt) {
            const int st = kt % ST;
            if (kt >= ST && !wait_or_abort(sm, &sm.empty[st], ((kt / ST) - 1) & 1, p.status)) break;
            mbar_arrive_expect_tx(&sm.full_tma[st], mtiles * kXTile + BN * 64);
            for (int i = 0; i < mtiles; ++i) tma_load_2d(L.x(st, i), &p.tm_x, kt * kBK, m0 + i * kBM, &sm.full_tma[st]);
            tma_load_2d(L.codes(st), &p.tm_q, kt * kBK, n0, &sm.full_tma[st]);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        // full_w implies full_tma: the dequantisers waited for the stage's
        // TMA bytes (x included) before they arrived
        for (int kt = 0; kt < KT; ++kt) {
            const int st = kt % ST;
            if (!wait_or_abort(sm, &sm.full_w[st], (kt / ST) & 1, p.status)) break;
            tc_fence_after();
            const uint64_t db = sw128_desc(L.w(st));
#pragma unroll
            for (int i = 0; i < BMP; ++i) {
                const uint64_t da = sw128_desc(L.x(st, i));
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    // advance 16 elements (32 bytes) along K inside the swizzled rows
                    umma_bf16<BN>(tmem + static_cast<uint32_t>(i * BN), da + static_cast<uint64_t>(kk * 2),
                                  db + static_cast<uint64_t>(kk * 2), (kt > 0 || kk > 0) ? 1u : 0u);
                }
            }
            umma_commit(&sm.empty[st]);
        }
        umma_commit(&sm.acc_full);
    } else if (warp >= 4) {
        // ------------------------------------------------ dequantise, epilogue
        // two groups of 4 warps take alternate k-tiles (more independent work
        // per warp, and the groups overlap)
        const int grp = (warp - 4) >> 2;
        const int t = tid - 128 - 128 * grp;  // 0..127
        bool ok = wait_or_abort(sm, &sm.scales_full, 0, p.status);
        const uint16_t *sc = reinterpret_cast<const uint16_t *>(L.scales());
        for (int kt = grp; ok && kt < KT; kt += 2) {
            const int st = kt % ST;
            // the stage (and its weight tile) is free again: the producer
            // waited for the MMAs of k-tile kt - ST before refilling it
            if (!wait_or_abort(sm, &sm.full_tma[st], (kt / ST) & 1, p.status)) {
                ok = false;
                break;
            }
            // BN rows x 4 chunks of 16 codes; task j -> row j/4, chunk j%4
#pragma unroll
            for (int i = 0; i < BN * 4 / (kDeqThreads / 2); ++i) {
                const int j = t + (kDeqThreads / 2) * i;
                const int row = j >> 2;
                const int c = j & 3;  // 16-code chunk within the 64-code k-tile
                const int kb = kt * 2 + (c >> 1);  // block index along K
                const uint4 w = *reinterpret_cast<const uint4 *>(L.codes(st) + row * 64 + c * 16);
                const float s = (row < rows_n && kb < p.nb) ? f16_bits_to_f32(sc[row * p.nb + kb]) : 0.f;
                const uint32_t words[4] = {w.x, w.y, w.z, w.w};
                uint32_t out[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float f0, f1, f2, f3;
                    codes4_to_f32(words[e], f0, f1, f2, f3);
                    out[2 * e] = pack_bf16x2(f0 * s, f1 * s);
                    out[2 * e + 1] = pack_bf16x2(f2 * s, f3 * s);
                }
                // logical 16-byte chunks 2c and 2c+1 of the row, swizzled by row % 8
                uint8_t *wrow = L.w(st) + row * 128;
                *reinterpret_cast<uint4 *>(wrow + (((2 * c) ^ (row & 7)) << 4)) =
                    make_uint4(out[0], out[1], out[2], out[3]);
                *reinterpret_cast<uint4 *>(wrow + (((2 * c + 1) ^ (row & 7)) << 4)) =
                    make_uint4(out[4], out[5], out[6], out[7]);
            }
            fence_proxy_async_smem();  // generic writes -> visible to the tensor core
            __syncwarp();
            if (lane == 0)
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(&sm.full_w[st])) : "memory");
        }
        // epilogue: TMEM lanes 32*(warp%4) .. +31 hold rows 32*(warp%4) + lane
        // of each m-tile; warps 4-7 drain columns [0, BN/2), warps 8-11 the rest
        if (ok && wait_or_abort(sm, &sm.acc_full, 0, p.status)) {
            tc_fence_after();
            const int cbeg = warp < 8 ? 0 : BN / 2;
#pragma unroll 1
            for (int i = 0; i < BMP; ++i) {
                const int m = m0 + i * kBM + 32 * (warp & 3) + lane;
#pragma unroll 1
                for (int c0 = cbeg; c0 < cbeg + BN / 2; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) +
                                  static_cast<uint32_t>(i * BN + c0), v);
                    if (m < p.M) {
                        uint16_t *yrow = p.y + static_cast<int64_t>(m) * p.ldy + n0 + c0;
                        if (n0 + c0 + 32 <= p.N) {
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                const uint4 o = make_uint4(
                                    pack_bf16x2(__uint_as_float(v[8 * q4 + 0]), __uint_as_float(v[8 * q4 + 1])),
                                    pack_bf16x2(__uint_as_float(v[8 * q4 + 2]), __uint_as_float(v[8 * q4 + 3])),
                                    pack_bf16x2(__uint_as_float(v[8 * q4 + 4]), __uint_as_float(v[8 * q4 + 5])),
                                    pack_bf16x2(__uint_as_float(v[8 * q4 + 6]), __uint_as_float(v[8 * q4 + 7])));
                                *reinterpret_cast<uint4 *>(yrow + 8 * q4) = o;
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                if (n0 + c0 + e < p.N) {
                                    const uint32_t h = pack_bf16x2(__uint_as_float(v[e]), 0.f);
                                    yrow[e] = static_cast<uint16_t>(h & 0xFFFFu);
                                }
                            }
                        }
                    }
                }
            }
        }
    }

    // ------------------------------------------------------------- teardown
    // If a role gave up, let in-flight copies and MMAs land (bounded) first.
    if (tid == 0 && *reinterpret_cast<volatile int32_t *>(&sm.abort_flag)) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) {
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// cuTensorMapEncodeTiled, taken from the driver through the runtime at first
// use, so the library itself does not link against libcuda.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

bool encode_maps(GemmParams &p, const int8_t *q, const uint16_t *x, int64_t N, int64_t K, int64_t M,
                 int64_t ldx, int BN) {
    const EncodeTiledFn cuTensorMapEncodeTiled = encode_tiled();
    if (!cuTensorMapEncodeTiled) return false;
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
        const cuuint32_t box[2] = {kBK, kBM};
        const cuuint32_t estr[2] = {1, 1};
        if (cuTensorMapEncodeTiled(&p.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims,
                                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
        const cuuint32_t box[2] = {kBK, static_cast<cuuint32_t>(BN)};
        const cuuint32_t estr[2] = {1, 1};
        if (cuTensorMapEncodeTiled(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t *>(q), dims, strides,
                                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

int g_configured_dev = -1;

template <int BMP, int BN>
bool configure() {
    return cudaFuncSetAttribute(gemm_tc_kernel<BMP, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax) ==
           cudaSuccess;
}

// Shared memory of a (BMP, BN) launch with ST TMA stages, or 0 if even two do
// not fit; sets ST and the control block offset.
template <int BMP, int BN>
size_t smem_for(int64_t nb, int &ST, int &ctl_off) {
    using L = GemmSmem<BMP, BN>;
    const int scale_bytes = static_cast<int>((static_cast<int64_t>(BN) * nb * 2 + 1023) / 1024 * 1024);
    const int fixed = 1024 + scale_bytes + static_cast<int>(sizeof(GemmCtl));
    ST = std::min(kMaxStages, (kSmemMax - fixed) / L::kStage);
    if (ST < 2) return 0;
    ctl_off = ST * L::kStage + scale_bytes;
    return static_cast<size_t>(1024 + ctl_off + sizeof(GemmCtl));
}

template <int BMP, int BN>
q8_status run(GemmParams &p, const int8_t *q, const uint16_t *x, int64_t N, int64_t K, int64_t M, int64_t ldx,
              cudaStream_t stream) {
    int ST = 0, ctl_off = 0;
    const size_t smem = smem_for<BMP, BN>(p.nb, ST, ctl_off);
    if (smem == 0) return Q8_ERR_UNSUPPORTED;
    if (!encode_maps(p, q, x, N, K, M, ldx, BN)) return Q8_ERR_CUDA;
    p.ST = ST;
    p.ctl_off = ctl_off;
    const dim3 grid(static_cast<unsigned>((N + BN - 1) / BN), static_cast<unsigned>((M + BMP * kBM - 1) / (BMP * kBM)));
    gemm_tc_kernel<BMP, BN><<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

}  // namespace

q8_status launch_gemm_tc(const int8_t *q, const uint16_t *s, int64_t N, int64_t K, const uint16_t *x, int64_t ldx,
                         int32_t M, uint16_t *y, int64_t ldy, int32_t tile, uint32_t *dev_status,
                         cudaStream_t stream) {
    const int64_t nb = K / 32;
    if (static_cast<int64_t>(kBM) * nb * 2 > kMaxScaleBytes) return Q8_ERR_UNSUPPORTED;  // K > 6144
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (g_configured_dev != di->device) {
        if (!configure<2, 128>() || !configure<1, 128>() || !configure<1, 64>()) return Q8_ERR_CUDA;
        g_configured_dev = di->device;
    }
    GemmParams p;
    p.s = s;
    p.y = y;
    p.status = dev_status;
    p.M = M;
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.nb = static_cast<int32_t>(nb);
    p.ldy = ldy;
    // tile shape: two m-tiles per weight tile if that still gives most SMs a
    // CTA, else one; 64-wide n-tiles for short N
    if (tile == Q8_GEMM_TILE_AUTO) {
        auto ctas = [&](int bmp, int bn) { return ((N + bn - 1) / bn) * ((M + bmp * kBM - 1) / (bmp * kBM)); };
        const int64_t want = static_cast<int64_t>(di->sm_count) * 4 / 5;
        if (ctas(2, 128) >= want)
            tile = Q8_GEMM_TILE_256x128;
        else if (ctas(1, 128) >= want || ctas(1, 128) >= ctas(1, 64))
            tile = Q8_GEMM_TILE_128x128;
        else
            tile = Q8_GEMM_TILE_128x64;
    }
    if (tile == Q8_GEMM_TILE_256x128) return run<2, 128>(p, q, x, N, K, M, ldx, stream);
    if (tile == Q8_GEMM_TILE_128x128) return run<1, 128>(p, q, x, N, K, M, ldx, stream);
    return run<1, 64>(p, q, x, N, K, M, ldx, stream);
}

}  // namespace q8
