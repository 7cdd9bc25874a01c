// q8_tile.cu -- Q8_0 W8A16 matmul for 9 <= M <= 32 activation rows over one or
// several matrices in one persistent launch (K a multiple of 256).
//
// Y[m][n] = sum_k s[n][k/32] * q[n][k] * x[m][k]; "Frigg" README, Finding 8
// (a batched W8A16 kernel reads each weight once for the whole batch of rows)
// and Finding 3 (one launch for the many small matrices of a decode step).
//
// Design (TMA fed, tensor cores through warp mma):
//  * An item is 128 consecutive weight rows of one matrix; CTAs own
//    contiguous, byte-balanced ranges of items.  Each of the 8 warps owns a
//    16-row tile of the item over all of K, so a row's sum never leaves its
//    warp (no cross-warp reduction, no workspace).
//  * K is streamed in chunks of 256 through a 2-slot ring per CTA (two CTAs
//    per SM).  A stage is one chunk of one item: the codes (128 rows x 256
//    bytes as two 128-byte-wide boxes), the x chunk (M rows x 256 bf16 as
//    four boxes) and the block scales (128 rows x 8), all by
//    cp.async.bulk.tensor; codes and x land in the 128-byte swizzled layout,
//    so the lanes' fragment reads (rows g and g+8, or x rows 8j+g) fall on
//    distinct banks.  No producer warp: thread 0 issues the first stages and
//    the warp that releases a slot last issues the next one into it.
//  * Per 32-code block the warp converts its codes to bf16 exactly (a sign
//    split, |q| <= 127) and runs two mma.sync.m16n8k16 per 8 activation rows
//    (weights as A, x^T as B), then scales the fp32 result by the binary16
//    block scales of its two rows.  Products are exact; fp32 sums in k order.
// Every wait is bounded (Q8_DEV_TIMEOUT on expiry).
#include <cuda.h>

#include <algorithm>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 128;              // weight rows per item
constexpr int kChunk = 256;             // K per stage
constexpr int kSlots = 2;
constexpr int kMaxGrid = 320;              // >= SMs x 2 on GB300 (the parameter block is near its limit)
constexpr int kCodeBox = kRows * 128;   // one 128-byte-wide box of codes

struct TMaps {
    CUtensorMap q;      // int8 [N][K], box {128, 128}, 128-byte swizzle
    CUtensorMap x;      // bf16 [M][ldx], box {64, MP}, 128-byte swizzle
    CUtensorMap s;      // binary16 [N][K/32], box {8, 128}
};

struct TDesc {
    float *y;
    int64_t ldy;
    int32_t N;
    int32_t KC;          // chunks per item, K / 256
    int32_t item_begin;  // first global item of this matrix
    int32_t items;       // ceil(N / 128)
};

struct TParams {
    TMaps m[Q8_MAX_BATCH];
    TDesc d[Q8_MAX_BATCH];
    uint32_t *status;
    int32_t count;
    int32_t M;
    int32_t cta_begin[kMaxGrid + 1];
};
static_assert(sizeof(TParams) <= 32764, "kernel parameters exceed the 32764-byte limit");

template <int MP>
struct TLayout {
    static constexpr int kXBox = MP * 128;                       // one 64-element-wide box of x
    static constexpr int kScales = kCodeBox * 2 + 4 * kXBox;      // offset of the scales
    static constexpr int kStage = kScales + kRows * 16;
    static constexpr int kSmem = 1024 + kSlots * kStage + 64;
};

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *tm, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ int find_tdesc(const TParams &p, int item) {
    int d = 0;
    while (d + 1 < p.count && item >= p.d[d + 1].item_begin) ++d;
    return d;
}

// Position (descriptor, item, chunk) in a CTA's sequence of stages.
struct Pos {
    int d, item, chunk;
    __device__ __forceinline__ void next(const TParams &p) {
        if (++chunk == p.d[d].KC) {
            chunk = 0;
            ++item;
            while (d + 1 < p.count && item >= p.d[d + 1].item_begin) ++d;
        }
    }
};

template <int MT>
__global__ void __launch_bounds__(kThreads, 2) tile_kernel(const __grid_constant__ TParams p) {
    constexpr int MP = MT * 8;
    using L = TLayout<MP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(base + kSlots * L::kStage);
    uint32_t *rel = reinterpret_cast<uint32_t *>(full + kSlots);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int M = p.M;
    const int ib = p.cta_begin[blockIdx.x];
    const int ie = p.cta_begin[blockIdx.x + 1];

    if (tid == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&full[i], 1);
            rel[i] = 0u;
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (ie <= ib) return;

    // total stages of this CTA
    int nstages = 0;
    {
        int d = find_tdesc(p, ib);
        for (int it = ib; it < ie; ++it) {
            while (d + 1 < p.count && it >= p.d[d + 1].item_begin) ++d;
            nstages += p.d[d].KC;
        }
    }

    auto issue = [&](int k, Pos pos) {
        const int slot = k % kSlots;
        const TDesc &D = p.d[pos.d];
        const TMaps &T = p.m[pos.d];
        uint8_t *st = base + slot * L::kStage;
        const int row0 = (pos.item - D.item_begin) * kRows;
        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(L::kStage));
        tma_2d(st, &T.q, pos.chunk * kChunk, row0, &full[slot]);
        tma_2d(st + kCodeBox, &T.q, pos.chunk * kChunk + 128, row0, &full[slot]);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            tma_2d(st + 2 * kCodeBox + j * L::kXBox, &T.x, pos.chunk * kChunk + 64 * j, 0, &full[slot]);
        tma_2d(st + L::kScales, &T.s, pos.chunk * (kChunk / 32), row0, &full[slot]);
    };
    Pos pos{find_tdesc(p, ib), ib, 0};
    if (tid == 0) {
        Pos q = pos;
        for (int k = 0; k < min(kSlots, nstages); ++k) {
            issue(k, q);
            q.next(p);
        }
    }

    // per-lane swizzled offsets: codes block b' (0..3) within a 128-byte box
    // for rows with (row & 7) == g; x 32-element half kbb (0..1) of a box
    uint32_t offq[4], offx[2];
#pragma unroll
    for (int b = 0; b < 4; ++b) offq[b] = ((((2 * b + (t >> 1)) ^ g)) << 4) + 8 * (t & 1);
#pragma unroll
    for (int h = 0; h < 2; ++h) offx[h] = (((4 * h + t) ^ g)) << 4;
    const int ra = 16 * warp + g;  // item-local rows of this lane: ra, ra + 8

    float acc[MT][4];
#pragma unroll
    for (int j = 0; j < MT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

    for (int k = 0; k < nstages; ++k) {
        const int slot = k % kSlots;
        if (!mbar_wait_bounded(&full[slot], (k / kSlots) & 1)) {
            if (lane == 0 && p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
            return;
        }
        const uint8_t *st = base + slot * L::kStage;
        const uint16_t *sc = reinterpret_cast<const uint16_t *>(st + L::kScales);
#pragma unroll
        for (int bl = 0; bl < kChunk / 32; ++bl) {
            const uint8_t *cbox = st + (bl >> 2) * kCodeBox;
            const uint2 wa = *reinterpret_cast<const uint2 *>(cbox + ra * 128 + offq[bl & 3]);
            const uint2 wb = *reinterpret_cast<const uint2 *>(cbox + (ra + 8) * 128 + offq[bl & 3]);
            const float s_a = f16_bits_to_f32(sc[ra * 8 + bl]);
            const float s_b = f16_bits_to_f32(sc[(ra + 8) * 8 + bl]);
            uint32_t a01, a23, a45, a67, b01, b23, b45, b67;
            codes4_to_bf16x2(wa.x, a01, a23);
            codes4_to_bf16x2(wa.y, a45, a67);
            codes4_to_bf16x2(wb.x, b01, b23);
            codes4_to_bf16x2(wb.y, b45, b67);
            const uint8_t *xbox = st + 2 * kCodeBox + (bl >> 1) * L::kXBox;
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                const uint4 xj = *reinterpret_cast<const uint4 *>(xbox + (8 * j + g) * 128 + offx[bl & 1]);
                float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
                mma_bf16_16816(d0, d1, d2, d3, a01, b01, a23, b23, xj.x, xj.y);
                mma_bf16_16816(d0, d1, d2, d3, a45, b45, a67, b67, xj.z, xj.w);
                acc[j][0] = fmaf(s_a, d0, acc[j][0]);
                acc[j][1] = fmaf(s_a, d1, acc[j][1]);
                acc[j][2] = fmaf(s_b, d2, acc[j][2]);
                acc[j][3] = fmaf(s_b, d3, acc[j][3]);
            }
        }
        // release the slot: reads ordered (fence, counter, fence) before the
        // refill that the last of the 8 warps issues
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const uint32_t done = atomicAdd(&rel[slot], 1u);
            if (done == kWarps - 1) {
                __threadfence_block();
                rel[slot] = 0u;
                fence_proxy_async_smem();
                if (k + kSlots < nstages) {
                    Pos q = pos;
                    for (int s = 0; s < kSlots; ++s) q.next(p);
                    issue(k + kSlots, q);
                }
            }
        }
        __syncwarp();
        // the item's last chunk: store y and start the next item
        const TDesc &D = p.d[pos.d];
        if (pos.chunk == D.KC - 1) {
            const int row0 = (pos.item - D.item_begin) * kRows;
            const int na = row0 + ra, nbr = row0 + ra + 8;
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                const int m0 = 8 * j + 2 * t;
                if (na < D.N) {
                    if (m0 < M) D.y[m0 * D.ldy + na] = acc[j][0];
                    if (m0 + 1 < M) D.y[(m0 + 1) * D.ldy + na] = acc[j][1];
                }
                if (nbr < D.N) {
                    if (m0 < M) D.y[m0 * D.ldy + nbr] = acc[j][2];
                    if (m0 + 1 < M) D.y[(m0 + 1) * D.ldy + nbr] = acc[j][3];
                }
                acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
            }
        }
        pos.next(p);
    }
}

int g_configured_dev = -1;
int g_occ = 0;

template <int MT>
bool configure(int &occ) {
    if (cudaFuncSetAttribute(tile_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, TLayout<MT * 8>::kSmem) !=
        cudaSuccess)
        return false;
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, tile_kernel<MT>, kThreads, TLayout<MT * 8>::kSmem) !=
        cudaSuccess)
        return false;
    occ = std::min(occ, std::max(o, 1));
    return true;
}

template <int MT>
q8_status run(TParams &p, const DeviceInfo *di, int items, double total_bytes, cudaStream_t stream) {
    const int grid = std::min(std::min(items, di->sm_count * g_occ), kMaxGrid);
    // cut the item list into `grid` ranges of (nearly) equal bytes
    int c = 0;
    double acc = 0.0;
    p.cta_begin[0] = 0;
    for (int i = 0; i < p.count && c < grid - 1; ++i) {
        const TDesc &D = p.d[i];
        const double per_row = static_cast<double>(D.KC) * kChunk * 1.0625;
        for (int it = 0; it < D.items && c < grid - 1; ++it) {
            acc += per_row * std::min(kRows, D.N - it * kRows);
            while (c < grid - 1 && acc >= total_bytes * (c + 1) / grid) p.cta_begin[++c] = D.item_begin + it + 1;
        }
    }
    while (c < grid) p.cta_begin[++c] = items;
    tile_kernel<MT><<<grid, kThreads, TLayout<MT * 8>::kSmem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

}  // namespace

bool tile_supported(const q8_linear_desc *descs, int count, int M) {
    if (M < 9 || M > 32 || count > Q8_MAX_BATCH) return false;
    for (int i = 0; i < count; ++i)
        if (descs[i].K % kChunk != 0) return false;
    return true;
}

q8_status launch_tile(const q8_linear_desc *descs, int count, int M, uint32_t *dev_status, cudaStream_t stream) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (g_configured_dev != di->device) {
        int o = 1 << 30;
        if (!configure<2>(o) || !configure<4>(o)) return Q8_ERR_CUDA;
        g_occ = o;
        g_configured_dev = di->device;
    }
    static thread_local TParams p;
    const int MP = M <= 16 ? 16 : 32;
    int items = 0;
    double total_bytes = 0.0;
    for (int i = 0; i < count; ++i) {
        TDesc &D = p.d[i];
        TMaps &T = p.m[i];
        const q8_linear_desc &d = descs[i];
        const int64_t nb = d.K / 32;
        if (!encode_2d(&T.q, 1, d.q, static_cast<uint64_t>(d.K), static_cast<uint64_t>(d.N),
                       static_cast<uint64_t>(d.K), 128, kRows, true) ||
            !encode_2d(&T.x, 2, d.x, static_cast<uint64_t>(d.K), static_cast<uint64_t>(M),
                       static_cast<uint64_t>(d.ldx) * 2, 64, static_cast<uint32_t>(MP), true) ||
            !encode_2d(&T.s, 2, d.s, static_cast<uint64_t>(nb), static_cast<uint64_t>(d.N),
                       static_cast<uint64_t>(nb) * 2, 8, kRows, false))
            return Q8_ERR_CUDA;
        D.y = d.y;
        D.ldy = d.ldy;
        D.N = static_cast<int32_t>(d.N);
        D.KC = static_cast<int32_t>(d.K / kChunk);
        D.item_begin = items;
        D.items = static_cast<int32_t>((d.N + kRows - 1) / kRows);
        items += D.items;
        total_bytes += static_cast<double>(d.N) * d.K * 1.0625;
    }
    p.status = dev_status;
    p.count = count;
    p.M = M;
    if (items == 0) return Q8_OK;
    return M <= 16 ? run<2>(p, di, items, total_bytes, stream) : run<4>(p, di, items, total_bytes, stream);
}

}  // namespace q8
