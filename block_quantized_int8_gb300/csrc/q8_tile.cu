// q8_tile.cu -- Q8_0 W8A16 matmul for 2 <= M <= 32 activation rows over one or
// several matrices in one persistent launch (any K >= 256, a multiple of
// 32).  Serves M = 9..32, and M = 2..8 where q8_pipe.cu does not (K = 1536
// and K not a multiple of 256 up to 4096 go there: whole-row stages are as
// fast in batches and faster for a lone matrix).
//
// Y[m][n] = sum_k s[n][k/32] * q[n][k] * x[m][k]; "Frigg" README, Finding 8
// (a batched W8A16 kernel reads each weight once for the whole batch of rows)
// and Finding 3 (one launch for the many small matrices of a decode step).
//
// Design (TMA fed, tensor cores through warp mma):
//  * K is cut into chunks of 256.  A stage is one chunk of 128 weight rows
//    (32 KB of codes), with the x chunk and the block scales that go with
//    it, each loaded by one cp.async.bulk.tensor (codes and x in the
//    128-byte swizzled layout, so the lanes' fragment reads fall on distinct
//    banks).  The 8 warps own 16 rows each.  No producer warp: thread 0
//    issues the first stages and the warp that releases a slot last issues
//    the next one, through a 2-slot ring (two CTAs per SM).
//  * Per 32-code block a warp converts its codes exactly (|q| <= 127), runs
//    two mma.sync.m16n8k16 per 8 activation rows (weights as A, x^T as B)
//    and adds the result times the binary16 block scale of each row to an
//    fp32 accumulator.  Products are exact.  For M <= 16 the operands are
//    binary16 (codes in three operations per pair) wherever binary16 holds
//    the chunk's x exactly, bf16 (codes by a sign split, four operations per
//    pair) elsewhere: a small kernel launched first copies each distinct x
//    into the workspace, chunk by chunk, as binary16 when every value of the
//    chunk (all M rows) converts exactly, as the unchanged bf16 bits
//    otherwise, with one flag word per chunk saying which, and the tile
//    kernel reads x from that copy.  For M > 16 they are bf16, x read in
//    place.
//  * Work units: the chunks of a matrix fall into C classes of consecutive
//    chunks (up to 4 of at least 2 chunks each, 4 for M > 16); an item is one class
//    of one block of 128 rows.  A class's blocks are summed in chunk order,
//    and a row block's classes are added in class order, so the result
//    depends on the matrix and M only: the same bits alone or in any batch,
//    for any grid.  CTAs own contiguous, byte-balanced ranges of items (four
//    per row block instead of one keeps the ranges even); a CTA that holds
//    a row block from its first class adds the classes as it goes; where a
//    row block is shared between CTAs, each writes its partial (the running
//    sum through its last class, or single classes) to the workspace and the
//    last to arrive on the row block's ticket adds them in class order.
//    For M > 16 the running class sum does not fit the registers (128 per
//    thread at two CTAs per SM): each thread keeps it in its own slot of the
//    workspace (16 KB per CTA, L2-resident), read and written once per class.
//  * K not a multiple of 256: the last chunk is partial.  Its codes come
//    as two 2-D boxes of [N][K] (TMA writes zeros past K), x from a copy
//    padded with zeros (M <= 16) or four 2-D boxes of the caller's x (zeros
//    past K), so the blocks past K add exact zeros.  Such a matrix's scale
//    rows are not 16-byte aligned, so no TMA box reads them: each lane loads
//    its rows' 8 scales of a stage from global memory one stage ahead.
//  * Batch-invariant mode (any 1 <= M <= 32): bf16 operands from the
//    caller's x and one class, so every row's arithmetic is the same for
//    every M (a warp MMA computes each output from its own row only).
// Every wait is bounded (Q8_DEV_TIMEOUT on expiry).
#include <cuda.h>

#include <algorithm>
#include <vector>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kChunk = 256;             // K per chunk
constexpr int kRows = 128;              // weight rows per stage and per item
constexpr int kSlots = 2;
constexpr int kMaxGrid = 320;           // >= SMs x 2 on GB300 (the parameter block is near its limit)
constexpr int kMaxClasses = 4;
constexpr int kCodeBytes = kRows * kChunk;  // codes of a stage
constexpr int kXBytes = 16384;              // x of a stage: MP rows x 256 bf16, MP <= 32
constexpr int kScaleBytes = kRows * 16;     // block scales of a stage: 128 rows x 8
constexpr int kStage = kCodeBytes + kXBytes + kScaleBytes;  // a multiple of 1024
// W8A8: per chunk of 256, x row m's codes are 9 blocks of 32 (the 9th zero,
// which spreads the rows over the shared-memory banks) and its scales 9
// binary16; a chunk's MP rows are contiguous, so a stage's x is two bulk
// copies (codes at the start of the x region, scales at kW8ScaleOff)
constexpr int kW8Blocks = 9;
constexpr int kW8Row = kW8Blocks * 32;
constexpr int kW8ScaleOff = 32 * kW8Row;
static_assert(kW8ScaleOff + 32 * kW8Blocks * 2 <= kXBytes, "W8A8 x of a stage exceeds its region");
enum TileMode { kModeDefault = 0, kModeInvariant = 1, kModeW8A8 = 2 };
// K not a multiple of 256: per warp two buffers with the block scales of its
// 16 rows for one stage, each row the two 16-byte aligned segments that hold
// its 8 scales (a slot of 16 halves)
constexpr int kScSlot = 16;
constexpr int kScBuf = 16 * kScSlot;
constexpr int kScBytes = kWarps * 2 * kScBuf * 2;
// shared memory of tile_kernel: alignment slack, ring, barriers and counters,
// and with matrices whose K is not a multiple of 256 the scale buffers
constexpr int smem_bytes(bool ragged) { return 1024 + kSlots * kStage + 128 + (ragged ? kScBytes : 0); }
static_assert(kStage % 1024 == 0, "stages must keep the 1024-byte alignment of the swizzled boxes");
// M <= 16 reads x from the workspace copy (binary16 where exact); M > 16 reads
// the caller's bf16 x (measured: with four 8-row tiles per block the binary16
// conversion of the codes gains nothing, and the second operand path costs
// registers)
constexpr bool tile_uses_x_copy(int MT) { return MT < 4; }
// classes of a matrix with KC chunks at M rows: the most, up to 4, that
// divide KC into classes of at least two chunks for M <= 16, four for M > 16
// (measured: shorter classes cost more at their ends than they balance --
// at M > 16 the running sum also goes through the workspace at each end)
int classes_for(int64_t KC, int MT) {
    const int64_t min_chunks = MT == 4 ? 4 : 2;
    for (int c = kMaxClasses; c > 1; --c)
        if (KC % c == 0 && KC / c >= min_chunks) return c;
    return 1;
}

struct TMaps {
    CUtensorMap q;      // int8 [N][K] as {128, N, K/128}, box {128, 128, 2}, 128-byte swizzle
    CUtensorMap x;      // 16-bit [M][ld] as {64, M, K/64}, box {64, MP, 4}, 128-byte swizzle
    CUtensorMap s;      // binary16 [N][K/32], box {8, 128}
};

struct TDesc {
    float *y;
    const uint32_t *xflag;  // per chunk: 0 = x copy is binary16, 1 = bf16; W8A8: the x codes
    const uint16_t *s;      // block scales [N][nb], read in place when nb % 8 != 0
    int64_t ldy;
    int32_t nb;             // blocks per row, K / 32 (nb % 8 != 0: the last chunk is partial)
    int32_t N;
    int32_t KC;          // chunks per row, K / 256
    int32_t item_begin;  // first global item of this matrix
    int32_t items;       // row blocks x C
    int32_t C;           // classes: class c holds chunks [c KC / C, (c + 1) KC / C)
    int16_t cls[kMaxClasses + 1];  // the class bounds c KC / C
};

// A row block whose items are shared between CTAs: its partials and ticket
// live in the workspace under a split id; `sharers` CTAs contribute, and the
// one holding class 0 writes its running sum through class `pe`.
struct TParams {
    TMaps m[Q8_MAX_BATCH];
    TDesc d[Q8_MAX_BATCH];
    uint32_t *status;
    uint32_t *tickets;   // [split id][8 warps], zero between launches
    float4 *parts;       // [split id][class][8 warps][32 lanes][MT]
    float4 *fold;        // MT = 4 with classes: [CTA][8 warps][32 lanes][4], the running class sums
    int32_t count;
    int32_t M;
    int32_t early_signal;  // the grid fills every CTA slot: signal dependents at start
    int32_t mode;          // TileMode: batch-invariant (bf16 operands from the caller's x, one
                           // class) or W8A8 (x quantized to Q8_0, integer block dots)
    const uint8_t *w8_codes;   // W8A8: the codes of every distinct x, one after another ...
    const uint8_t *w8_scales;  // ... and their scales in the same order (18 bytes per 288 of codes)
    int32_t cta_begin[kMaxGrid + 1];
    int16_t first_sid[kMaxGrid];  // split id of a CTA's first row block, -1 if whole
    int16_t last_sid[kMaxGrid];   // split id of a CTA's last row block, -1 if whole
    uint8_t sharers[kMaxGrid];
    int8_t pe[kMaxGrid];
};
static_assert(sizeof(TParams) <= 32764, "kernel parameters exceed the 32764-byte limit");

__host__ __device__ __forceinline__ int class_lo(int KC, int C, int c) { return (c * KC) / C; }

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *tm, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_3d(void *dst, const CUtensorMap *tm, int c0, int c1, int c2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2),
           "r"(smem_addr(bar))
        : "memory");
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned); the
// bytes past src_bytes (0..16) are written as zeros and not read
__device__ __forceinline__ void cp_async_16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(smem_addr(dst)), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// all but the most recent group of this thread's copies have landed
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ int find_tdesc(const TParams &p, int item) {
    int d = 0;
    while (d + 1 < p.count && item >= p.d[d + 1].item_begin) ++d;
    return d;
}

// Position in a CTA's sequence of stages: descriptor, item, the chunk of
// this stage and the end of the item's class.
struct Pos {
    int d, item, c, row0, chunk, cend;  // descriptor, item, its class and first row, chunk, class end
    __device__ __forceinline__ void init(const TParams &p, int it) {
        d = find_tdesc(p, it);
        item = it;
        const TDesc &D = p.d[d];
        c = (it - D.item_begin) % D.C;
        row0 = (it - D.item_begin) / D.C * kRows;
        chunk = D.cls[c];
        cend = D.cls[c + 1];
    }
    __device__ __forceinline__ void next(const TParams &p) {
        if (++chunk == cend) {
            ++item;
            if (d + 1 < p.count && item >= p.d[d + 1].item_begin) {
                while (d + 1 < p.count && item >= p.d[d + 1].item_begin) ++d;
                c = 0;
                row0 = 0;
            } else if (++c == p.d[d].C) {
                c = 0;
                row0 += kRows;
            }
            chunk = p.d[d].cls[c];
            cend = p.d[d].cls[c + 1];
        }
    }
};

// One chunk (8 blocks of 32) of a warp's 16-row tile into the accumulators a.
//   cb: the chunk's first code box (128 K-bytes x 128 rows, swizzled), rb = 128 x 128
//   xb: the chunk's first x box (64 K x MP rows, swizzled)
//   sa, sb: the block scales of rows ra and ra + 8 (shared memory)
//   F16: x of the chunk is binary16 (else bf16)
template <int MT, bool F16>
__device__ __forceinline__ void chunk_mma(float (&a)[MT][4], const uint8_t *cb, int rb, const uint8_t *xb,
                                          const uint16_t *sa, const uint16_t *sb, int ra, const uint32_t (&offq)[4],
                                          const uint32_t (&offx)[2], int g) {
    constexpr int MP = MT * 8;
#pragma unroll
    for (int bl = 0; bl < kChunk / 32; ++bl) {
        const uint8_t *cbox = cb + (bl >> 2) * rb;
        const uint2 wa = *reinterpret_cast<const uint2 *>(cbox + ra * 128 + offq[bl & 3]);
        const uint2 wb = *reinterpret_cast<const uint2 *>(cbox + (ra + 8) * 128 + offq[bl & 3]);
        const float s_a = f16_bits_to_f32(sa[bl]);
        const float s_b = f16_bits_to_f32(sb[bl]);
        uint32_t a01, a23, a45, a67, b01, b23, b45, b67;
        if constexpr (F16) {
            codes4_to_f16x2(wa.x, a01, a23);
            codes4_to_f16x2(wa.y, a45, a67);
            codes4_to_f16x2(wb.x, b01, b23);
            codes4_to_f16x2(wb.y, b45, b67);
        } else {
            codes4_to_bf16x2(wa.x, a01, a23);
            codes4_to_bf16x2(wa.y, a45, a67);
            codes4_to_bf16x2(wb.x, b01, b23);
            codes4_to_bf16x2(wb.y, b45, b67);
        }
        const uint8_t *xbox = xb + (bl >> 1) * (MP * 128);
#pragma unroll
        for (int j = 0; j < MT; ++j) {
            const uint4 xj = *reinterpret_cast<const uint4 *>(xbox + (8 * j + g) * 128 + offx[bl & 1]);
            float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
            if constexpr (F16) {
                mma_f16_16816(d0, d1, d2, d3, a01, b01, a23, b23, xj.x, xj.y);
                mma_f16_16816(d0, d1, d2, d3, a45, b45, a67, b67, xj.z, xj.w);
            } else {
                mma_bf16_16816(d0, d1, d2, d3, a01, b01, a23, b23, xj.x, xj.y);
                mma_bf16_16816(d0, d1, d2, d3, a45, b45, a67, b67, xj.z, xj.w);
            }
            a[j][0] = fmaf(s_a, d0, a[j][0]);
            a[j][1] = fmaf(s_a, d1, a[j][1]);
            a[j][2] = fmaf(s_b, d2, a[j][2]);
            a[j][3] = fmaf(s_b, d3, a[j][3]);
        }
    }
}

// W8A8: one chunk of a warp's 16-row tile against Q8_0 x.  Lane (g, t)
// holds bytes 8t..8t+7 of each 32-code block of its weight rows and of x row
// 8j + g; both operands use them as k = 4t..4t+3 and 16+4t..16+4t+3, so one
// int8 MMA gives the exact block dot, scaled by s_w s_x (exact in fp32).
//   xq: the chunk's x codes [MP][9 x 32]; xs: its scales [MP][9]
template <int MT>
__device__ __forceinline__ void chunk_mma_w8a8(float (&a)[MT][4], const uint8_t *cb, int rb, const uint8_t *xq,
                                               const uint16_t *xs, const uint16_t *sa, const uint16_t *sb, int ra,
                                               const uint32_t (&offq)[4], int g, int t) {
#pragma unroll
    for (int bl = 0; bl < kChunk / 32; ++bl) {
        const uint8_t *cbox = cb + (bl >> 2) * rb;
        const uint2 wa = *reinterpret_cast<const uint2 *>(cbox + ra * 128 + offq[bl & 3]);
        const uint2 wb = *reinterpret_cast<const uint2 *>(cbox + (ra + 8) * 128 + offq[bl & 3]);
        const float s_a = f16_bits_to_f32(sa[bl]);
        const float s_b = f16_bits_to_f32(sb[bl]);
#pragma unroll
        for (int j = 0; j < MT; ++j) {
            const uint2 xa = *reinterpret_cast<const uint2 *>(xq + (8 * j + g) * kW8Row + bl * 32 + 8 * t);
            int d0, d1, d2, d3;
            mma_s8_16832(d0, d1, d2, d3, wa.x, wb.x, wa.y, wb.y, xa.x, xa.y);
            const float x0 = f16_bits_to_f32(xs[(8 * j + 2 * t) * kW8Blocks + bl]);
            const float x1 = f16_bits_to_f32(xs[(8 * j + 2 * t + 1) * kW8Blocks + bl]);
            a[j][0] = fmaf(s_a * x0, static_cast<float>(d0), a[j][0]);
            a[j][1] = fmaf(s_a * x1, static_cast<float>(d1), a[j][1]);
            a[j][2] = fmaf(s_b * x0, static_cast<float>(d2), a[j][2]);
            a[j][3] = fmaf(s_b * x1, static_cast<float>(d3), a[j][3]);
        }
    }
}

template <int MT>
__device__ __forceinline__ void store_tile(const TDesc &D, int row0, int ra, int t, int M, const float (&v)[MT][4]) {
    const int na = row0 + ra, nbr = row0 + ra + 8;
#pragma unroll
    for (int j = 0; j < MT; ++j) {
        const int m0 = 8 * j + 2 * t;
        if (na < D.N) {
            if (m0 < M) D.y[m0 * D.ldy + na] = v[j][0];
            if (m0 + 1 < M) D.y[(m0 + 1) * D.ldy + na] = v[j][1];
        }
        if (nbr < D.N) {
            if (m0 < M) D.y[m0 * D.ldy + nbr] = v[j][2];
            if (m0 + 1 < M) D.y[(m0 + 1) * D.ldy + nbr] = v[j][3];
        }
    }
}


// The partial of warp `warp` for class c of split row block `sid`:
// [split id][class][warp][lane][MT] float4.
template <int MT>
__device__ __forceinline__ float4 *part_slot(const TParams &p, int sid, int c, int warp) {
    return p.parts + ((static_cast<size_t>(sid) * kMaxClasses + c) * kWarps + warp) * 32 * MT;
}

template <int MT>
__device__ __forceinline__ void put_part(float4 *slot, int lane, const float (&v)[MT][4]) {
#pragma unroll
    for (int j = 0; j < MT; ++j) slot[lane * MT + j] = make_float4(v[j][0], v[j][1], v[j][2], v[j][3]);
}

// Last of the sharers of split row block sid for this warp's rows: add the
// partials in class order (the running sum through class pe, then the single
// classes after it) and store the rows.  The tickets go back to zero.
template <int MT>
__device__ __forceinline__ void finish_split(const TParams &p, const TDesc &D, int sid, int warp, int lane,
                                             int row0, int ra, int t) {
    __threadfence();
    __syncwarp();
    uint32_t prev = 0;
    if (lane == 0) prev = atomicAdd(&p.tickets[sid * kWarps + warp], 1u);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev + 1 != p.sharers[sid]) return;
    __threadfence();
    const int pe = p.pe[sid];
    float v[MT][4];
    {
        const float4 *s0 = part_slot<MT>(p, sid, pe, warp);
#pragma unroll
        for (int j = 0; j < MT; ++j) {
            const float4 u = __ldcg(s0 + lane * MT + j);
            v[j][0] = u.x;
            v[j][1] = u.y;
            v[j][2] = u.z;
            v[j][3] = u.w;
        }
    }
    for (int c = pe + 1; c < D.C; ++c) {
        const float4 *sc = part_slot<MT>(p, sid, c, warp);
#pragma unroll
        for (int j = 0; j < MT; ++j) {
            const float4 u = __ldcg(sc + lane * MT + j);
            v[j][0] += u.x;
            v[j][1] += u.y;
            v[j][2] += u.z;
            v[j][3] += u.w;
        }
    }
    store_tile<MT>(D, row0, ra, t, p.M, v);
    __syncwarp();
    if (lane == 0) p.tickets[sid * kWarps + warp] = 0u;
}

// RAGGED: some matrix of the launch has K % 256 != 0 (the launches without
// one run without its code and shared memory)
template <int MT, bool RAGGED>
__global__ void __launch_bounds__(kThreads, 2) tile_kernel(const __grid_constant__ TParams p) {
    constexpr int MP = MT * 8;
    constexpr bool kCopy = tile_uses_x_copy(MT);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(base + kSlots * kStage);
    uint32_t *rel = reinterpret_cast<uint32_t *>(full + kSlots);  // per slot: warps done with it
    uint16_t *scb = reinterpret_cast<uint16_t *>(base + kSlots * kStage + 128);  // the warps' scale buffers
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
    // a grid that fills every CTA slot signals a chained launch after it at
    // once (its CTAs can only take the slots ours free); a smaller one late
    if (p.early_signal && tid == 0) pdl_launch_dependents();
    if (ie <= ib) return;
    // MT = 4: this thread's running class sum (16 floats) in the workspace
    float4 *fold_slot = MT == 4 && p.fold != nullptr
                            ? p.fold + ((static_cast<size_t>(blockIdx.x) * kWarps + warp) * 32 + lane) * MT
                            : nullptr;

    // total stages of this CTA: the chunks of each item's class
    int nstages = 0;
    {
        int d = find_tdesc(p, ib);
        for (int it = ib; it < ie; ++it) {
            while (d + 1 < p.count && it >= p.d[d + 1].item_begin) ++d;
            const TDesc &D = p.d[d];
            const int c = (it - D.item_begin) % D.C;
            nstages += D.cls[c + 1] - D.cls[c];
        }
    }

    // stage k at position pos: all bytes announced on the slot's barrier,
    // then the weight boxes and (unless deferred) the x box
    // x bytes of a stage: the TMA box, or for W8A8 the chunk's codes and scales
    const uint32_t xbytes = p.mode == kModeW8A8 ? MP * (kW8Row + 2 * kW8Blocks) : MP * 512;
    auto issue_x = [&](int k, const Pos &pos) {
        const int slot = k % kSlots;
        uint8_t *dst = base + slot * kStage + kCodeBytes;
        if (p.mode == kModeW8A8) {
            const TDesc &D = p.d[pos.d];
            const uint8_t *xq = reinterpret_cast<const uint8_t *>(D.xflag);
            const uint8_t *xs = p.w8_scales + (xq - p.w8_codes) / 16;
            bulk_g2s(dst, xq + static_cast<size_t>(pos.chunk) * MP * kW8Row, MP * kW8Row, &full[slot]);
            bulk_g2s(dst + kW8ScaleOff, xs + static_cast<size_t>(pos.chunk) * MP * kW8Blocks * 2, MP * kW8Blocks * 2,
                     &full[slot]);
        } else if (RAGGED && !kCopy && (p.d[pos.d].nb & 7) != 0) {
            // the caller's x, K not a multiple of 256: four 2-D boxes of 64
            // columns in the 3-D box's layout (zeros past K)
            for (int i = 0; i < 4; ++i)
                tma_2d(dst + i * (MP * 128), &p.m[pos.d].x, kChunk * pos.chunk + 64 * i, 0, &full[slot]);
        } else {
            tma_3d(dst, &p.m[pos.d].x, 0, 0, 4 * pos.chunk, &full[slot]);
        }
    };
    auto issue = [&](int k, const Pos &pos, bool with_x) {
        const int slot = k % kSlots;
        const TMaps &T = p.m[pos.d];
        uint8_t *st = base + slot * kStage;
        const int row0 = pos.row0;
        if (RAGGED && (p.d[pos.d].nb & 7) != 0) {
            // K not a multiple of 256: the codes as two 2-D boxes of 128
            // K-bytes (zeros past K), the scales by the consumers
            mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(kCodeBytes) + xbytes);
            tma_2d(st, &T.q, kChunk * pos.chunk, row0, &full[slot]);
            tma_2d(st + kRows * 128, &T.q, kChunk * pos.chunk + 128, row0, &full[slot]);
        } else {
            mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(kCodeBytes + kScaleBytes) + xbytes);
            tma_3d(st, &T.q, 0, row0, 2 * pos.chunk, &full[slot]);
            tma_2d(st + kCodeBytes + kXBytes, &T.s, 8 * pos.chunk, row0, &full[slot]);
        }
        if (with_x) issue_x(k, pos);
    };
    Pos pos;
    pos.init(p, ib);
    // the first stages' weights go out at once; their x only after the
    // kernels before this one (when launched as their dependent) completed
    if (tid == 0) {
        Pos q = pos;
        for (int k = 0; k < min(kSlots, nstages); ++k) {
            issue(k, q, false);
            q.next(p);
        }
    }
    pdl_wait_prior();
    if (tid == 0) {
        Pos q = pos;
        for (int k = 0; k < min(kSlots, nstages); ++k) {
            issue_x(k, q);
            q.next(p);
        }
    }

    // per-lane swizzled offsets: codes block b' (0..3) within a 128-byte box
    // for rows with (row & 7) == g; x 32-element half (0..1) of a box
    uint32_t offq[4], offx[2];
#pragma unroll
    for (int b = 0; b < 4; ++b) offq[b] = ((((2 * b + (t >> 1)) ^ g)) << 4) + 8 * (t & 1);
#pragma unroll
    for (int h = 0; h < 2; ++h) offx[h] = (((4 * h + t) ^ g)) << 4;

    const int ra = 16 * warp + g;  // item-local rows of this lane: ra, ra + 8
    float acc[MT][4], fold[MT][4];
#pragma unroll
    for (int j = 0; j < MT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = fold[j][e] = 0.f;
    // x flags of a matrix (bit j: chunk xbase + j reads bf16 x, else
    // binary16), loaded when the matrix or the 32-chunk window changes;
    // written by the x copy kernel, which completed before the wait above;
    // read through L2
    uint32_t xmask = 0u;
    int xd = -1, xbase = 0;
    // K not a multiple of 256: the block scales of the warp's 16 rows for a
    // stage are gathered by cp.async into the warp's two buffers, one stage
    // ahead: lane l copies the 16-byte aligned segment l % 2 of the two that
    // hold row l / 2's 8 scales, which then start at half o % 8 of its slot
    // (o: the first scale's index in the array).  Zeros past K and past N
    // (the copies' zero fill), so the blocks past K add exact zeros whatever
    // the scales beyond the row hold.
    uint16_t *wsc = scb + warp * (2 * kScBuf);
    auto gather_scales = [&](const Pos &q, uint16_t *buf) {
        const TDesc &E = p.d[q.d];
        const int r = lane >> 1, sg = lane & 1;
        const int n = q.row0 + 16 * warp + r;
        const int left = min(8, E.nb - 8 * q.chunk);  // scales of this chunk inside the row
        const int64_t o = static_cast<int64_t>(min(n, E.N - 1)) * E.nb + 8 * q.chunk;
        const int64_t seg = (o & ~static_cast<int64_t>(7)) + 8 * sg;  // the segment's first half
        const int64_t v = n < E.N ? o + left - seg : 0;  // halves of it to copy (clamped to 0..8)
        const uint32_t bytes = v <= 0 ? 0u : (v >= 8 ? 16u : static_cast<uint32_t>(2 * v));
        cp_async_16(buf + r * kScSlot + 8 * sg, bytes ? E.s + seg : E.s, bytes);
    };
    if constexpr (RAGGED) {
        if ((p.d[pos.d].nb & 7) != 0) gather_scales(pos, wsc);
        cp_async_commit();
    }

    for (int k = 0; k < nstages; ++k) {
        // every stage of this CTA is issued: a chained launch after this one
        // may start once all CTAs are this far
        if (!p.early_signal && k == max(0, nstages - kSlots) && tid == 0) pdl_launch_dependents();
        const int slot = k % kSlots;
        const TDesc &D = p.d[pos.d];
        const int c = pos.c;
        if (kCopy && p.mode == kModeDefault && (pos.d != xd || (pos.chunk & ~31) != xbase)) {
            xd = pos.d;
            xbase = pos.chunk & ~31;
            const int ch = xbase + lane;
            xmask = __ballot_sync(0xffffffffu, ch < D.KC && __ldcg(D.xflag + ch) != 0u);
        }
        const uint32_t xbf = kCopy && p.mode == kModeDefault ? (xmask >> (pos.chunk & 31)) & 1u : 1u;
        const bool ragged = RAGGED && (D.nb & 7) != 0;
        if constexpr (RAGGED) {
            // the next stage's scales into the other buffer (one group per
            // stage, empty if none), then this stage's group is complete
            if (k + 1 < nstages) {
                Pos q = pos;
                q.next(p);
                if ((p.d[q.d].nb & 7) != 0) gather_scales(q, wsc + ((k + 1) & 1) * kScBuf);
            }
            cp_async_commit();
            if (ragged) {
                cp_async_wait_1();
                __syncwarp();
            }
        }
        if (!mbar_wait_bounded(&full[slot], (k / kSlots) & 1)) {
            if (lane == 0 && p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
            if constexpr (RAGGED) cp_async_wait_all();
            drain_after_timeout();
            return;
        }
        {
            const uint8_t *st = base + slot * kStage;
            const uint8_t *xb = st + kCodeBytes;
            const uint16_t *sa = reinterpret_cast<const uint16_t *>(st + kCodeBytes + kXBytes) + ra * 8;
            const uint16_t *sb = sa + 64;
            if (ragged) {
                const uint16_t *buf = wsc + (k & 1) * kScBuf;
                const int na = min(pos.row0 + ra, D.N - 1), nbr = min(pos.row0 + ra + 8, D.N - 1);
                const int64_t c8 = 8 * pos.chunk;
                sa = buf + g * kScSlot + static_cast<int>((static_cast<int64_t>(na) * D.nb + c8) & 7);
                sb = buf + (g + 8) * kScSlot + static_cast<int>((static_cast<int64_t>(nbr) * D.nb + c8) & 7);
            }
            if (p.mode == kModeW8A8)
                chunk_mma_w8a8<MT>(acc, st, kRows * 128, xb,
                                   reinterpret_cast<const uint16_t *>(xb + kW8ScaleOff), sa, sb, ra, offq, g, t);
            else if (kCopy && xbf == 0u)
                chunk_mma<MT, kCopy>(acc, st, kRows * 128, xb, sa, sb, ra, offq, offx, g);
            else
                chunk_mma<MT, false>(acc, st, kRows * 128, xb, sa, sb, ra, offq, offx, g);
        }
        if (pos.chunk + 1 == pos.cend) {
            // the item's last stage.  A CTA that ran class 0 of the row block
            // adds the classes as they come; otherwise, or where the row
            // block goes on in another CTA, the partial goes to the
            // workspace and the row block's last sharer adds them up
            const int row0 = pos.row0;
            const bool prefix = pos.item - c >= ib;
            const bool last_here = c == D.C - 1 || pos.item == ie - 1;
            if constexpr (MT == 4) {
                if (D.C == 1) {
                    store_tile<MT>(D, row0, ra, t, M, acc);  // one class: the item is the row block
                } else if (prefix) {
                    // the same steps as below, the running sum in the
                    // workspace, added into acc in place (acc is cleared after)
                    if (c > 0) {
#pragma unroll
                        for (int j = 0; j < MT; ++j) {
                            const float4 u = fold_slot[j];
                            acc[j][0] += u.x;
                            acc[j][1] += u.y;
                            acc[j][2] += u.z;
                            acc[j][3] += u.w;
                        }
                    }
                    if (c == D.C - 1) {
                        store_tile<MT>(D, row0, ra, t, M, acc);
                    } else if (last_here && p.last_sid[blockIdx.x] >= 0) {
                        const int sid = p.last_sid[blockIdx.x];
                        put_part<MT>(part_slot<MT>(p, sid, c, warp), lane, acc);
                        finish_split<MT>(p, D, sid, warp, lane, row0, ra, t);
                    } else {
#pragma unroll
                        for (int j = 0; j < MT; ++j)
                            fold_slot[j] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
                    }
                } else if (p.first_sid[blockIdx.x] >= 0) {
                    const int sid = p.first_sid[blockIdx.x];
                    put_part<MT>(part_slot<MT>(p, sid, c, warp), lane, acc);
                    if (last_here) finish_split<MT>(p, D, sid, warp, lane, row0, ra, t);
                }
            } else if (prefix) {
#pragma unroll
                for (int j = 0; j < MT; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) fold[j][e] = c == 0 ? acc[j][e] : fold[j][e] + acc[j][e];
                if (c == D.C - 1) {
                    store_tile<MT>(D, row0, ra, t, M, fold);
                } else if (last_here && p.last_sid[blockIdx.x] >= 0) {
                    const int sid = p.last_sid[blockIdx.x];
                    put_part<MT>(part_slot<MT>(p, sid, c, warp), lane, fold);
                    finish_split<MT>(p, D, sid, warp, lane, row0, ra, t);
                }
            } else if (p.first_sid[blockIdx.x] >= 0) {
                const int sid = p.first_sid[blockIdx.x];
                put_part<MT>(part_slot<MT>(p, sid, c, warp), lane, acc);
                if (last_here) finish_split<MT>(p, D, sid, warp, lane, row0, ra, t);
            }
#pragma unroll
            for (int j = 0; j < MT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
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
                    for (int s2 = 0; s2 < kSlots; ++s2) q.next(p);
                    issue(k + kSlots, q, true);
                }
            }
        }
        __syncwarp();
        pos.next(p);
    }
    // (every scale gather was waited for by its stage; none may outlive the CTA)
    if constexpr (RAGGED) cp_async_wait_all();
}

// ---- the x copy ------------------------------------------------------------------
struct XJob {
    const uint16_t *x;    // bf16 bits [M][ldx]
    uint16_t *xo;         // copy [M][K], binary16 or bf16 bits per chunk
    uint32_t *flag;       // [K / 256]: 0 = binary16, 1 = bf16
    float *xf;            // W8A8: x as binary32 in the chunk-major block order of xq
    int8_t *xq;           // W8A8: codes [K / 256][MP][9 x 32], then scales [K / 256][MP][9]
    int64_t ldx;
    int64_t K;            // K rounded up to a multiple of 256: the copy's row length
    int64_t kx;           // columns of x (the copy is zero from there to K)
    int32_t chunk_begin;  // first CTA of this x
};

struct XParams {
    XJob j[Q8_MAX_BATCH];
    int32_t count;
    int32_t M;
};

// One CTA per chunk of 256 columns of one x, all M <= 32 rows: thread t
// holds the 8 values at columns 8 (t % 32) .. 8 (t % 32) + 7 of rows t / 32,
// t / 32 + 8, t / 32 + 16 and t / 32 + 24 (zeros past the columns of x).
// The chunk goes out as binary16 if binary16 holds every one of its values
// exactly, else bit for bit as bf16.
__global__ void __launch_bounds__(kThreads) x_copy_kernel(const __grid_constant__ XParams p) {
    // the tile kernel may start launching at once: it reads weights only
    // until this kernel has completed
    pdl_launch_dependents();
    int j = 0;
    while (j + 1 < p.count && static_cast<int>(blockIdx.x) >= p.j[j + 1].chunk_begin) ++j;
    const XJob &J = p.j[j];
    const int c = static_cast<int>(blockIdx.x) - J.chunk_begin;
    const int64_t col = static_cast<int64_t>(c) * kChunk + 8 * (threadIdx.x & 31);
    const int r0 = static_cast<int>(threadIdx.x >> 5);
    // x may be written by the kernels before this one
    pdl_wait_prior();
    uint4 v[4];
    bool inexact = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + 8 * i;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (r < p.M && col < J.kx) {
            v[i] = __ldcg(reinterpret_cast<const uint4 *>(J.x + r * J.ldx + col));
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                inexact |= !bf16_fits_f16(w[e] & 0xFFFFu) || !bf16_fits_f16(w[e] >> 16);
        }
    }
    const bool keep = __syncthreads_or(inexact) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + 8 * i;
        if (r < p.M) {
            uint4 o = v[i];
            if (!keep) {
                o.x = f32x2_to_f16x2(bf16lo_f32(v[i].x), bf16hi_f32(v[i].x));
                o.y = f32x2_to_f16x2(bf16lo_f32(v[i].y), bf16hi_f32(v[i].y));
                o.z = f32x2_to_f16x2(bf16lo_f32(v[i].z), bf16hi_f32(v[i].z));
                o.w = f32x2_to_f16x2(bf16lo_f32(v[i].w), bf16hi_f32(v[i].w));
            }
            *reinterpret_cast<uint4 *>(J.xo + r * J.K + col) = o;
        }
    }
    if (threadIdx.x == 0) J.flag[c] = keep ? 1u : 0u;
}

// W8A8: x as binary32 blocks in the order the quantizer turns into the
// stage layout -- for chunk c, row m < MP, block b < 9: x[m][256 c + 32 b ..]
// (zero past M and in the ninth block).  One CTA per chunk of one x.
__global__ void __launch_bounds__(kThreads) w8a8_widen_kernel(const __grid_constant__ XParams p, int MP) {
    int j = 0;
    while (j + 1 < p.count && static_cast<int>(blockIdx.x) >= p.j[j + 1].chunk_begin) ++j;
    const XJob &J = p.j[j];
    const int c = static_cast<int>(blockIdx.x) - J.chunk_begin;
    pdl_wait_prior();
    float *out = J.xf + static_cast<size_t>(c) * MP * kW8Row;
    for (int i = threadIdx.x; i < MP * kW8Row; i += kThreads) {
        const int m = i / kW8Row, e = i - m * kW8Row;
        float v = 0.f;
        if (m < p.M && e < kChunk) v = __uint_as_float(static_cast<uint32_t>(J.x[m * J.ldx + c * kChunk + e]) << 16);
        out[i] = v;
    }
}


int g_configured_dev = -1;
// resident CTAs per SM of tile_kernel<1>, <2>, <4>, without and with RAGGED
int g_occ[2][3] = {{0, 0, 0}, {0, 0, 0}};
constexpr int occ_index(int MT) { return MT == 1 ? 0 : (MT == 2 ? 1 : 2); }

template <int MT, bool RAGGED>
bool configure() {
    if (cudaFuncSetAttribute(tile_kernel<MT, RAGGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes(RAGGED)) != cudaSuccess)
        return false;
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, tile_kernel<MT, RAGGED>, kThreads, smem_bytes(RAGGED)) !=
        cudaSuccess)
        return false;
    g_occ[RAGGED ? 1 : 0][occ_index(MT)] = std::max(o, 1);
    return true;
}


// Cuts the item list into `grid` ranges of (nearly) equal bytes and marks
// the row blocks that two or more ranges share: a split id each, the number
// of CTAs that share it and the last class of the one that holds class 0.
template <int MT, bool RAGGED>
q8_status run(TParams &p, const DeviceInfo *di, int items, double total_bytes, int max_sids, cudaStream_t stream,
              bool chained) {
    const int occ = g_occ[RAGGED ? 1 : 0][occ_index(MT)];
    const int grid = std::min(std::min(items, di->sm_count * occ), kMaxGrid);
    int c = 0;
    double acc = 0.0;
    p.cta_begin[0] = 0;
    for (int i = 0; i < p.count && c < grid - 1; ++i) {
        const TDesc &D = p.d[i];
        for (int it = 0; it < D.items && c < grid - 1; ++it) {
            const int rb = it / D.C, cl = it % D.C;
            const int rows = std::min(kRows, D.N - rb * kRows);
            const int chunks = class_lo(D.KC, D.C, cl + 1) - class_lo(D.KC, D.C, cl);
            acc += static_cast<double>(rows) * chunks * kChunk * 1.0625;
            while (c < grid - 1 && acc >= total_bytes * (c + 1) / grid) p.cta_begin[++c] = D.item_begin + it + 1;
        }
    }
    while (c < grid) p.cta_begin[++c] = items;

    // row block of a global item: its first item, and the matrix's classes
    int d = 0;
    const auto block_of = [&](int item, int &first, int &C) {
        d = 0;
        while (d + 1 < p.count && item >= p.d[d + 1].item_begin) ++d;
        C = p.d[d].C;
        first = item - (item - p.d[d].item_begin) % C;
    };
    int nsid = 0, cur_key = -1;
    const auto sid_of = [&](int key) {
        if (key != cur_key) {
            cur_key = key;
            p.sharers[nsid] = 0;
            p.pe[nsid] = -1;
            ++nsid;
        }
        return nsid - 1;
    };
    for (int i = 0; i < grid; ++i) {
        p.first_sid[i] = p.last_sid[i] = -1;
        const int b = p.cta_begin[i], e = p.cta_begin[i + 1];
        if (e <= b) continue;
        int kf, cf, kl, cl;
        block_of(b, kf, cf);
        block_of(e - 1, kl, cl);
        if (kf == kl) {
            if (b == kf && e == kf + cf) continue;  // the whole row block
            if (nsid >= max_sids && kf != cur_key) return Q8_ERR_WORKSPACE;
            const int s = sid_of(kf);
            p.first_sid[i] = p.last_sid[i] = static_cast<int16_t>(s);
            ++p.sharers[s];
            if (b == kf) p.pe[s] = static_cast<int8_t>(e - 1 - kf);
            continue;
        }
        if (b > kf) {  // enters its first row block after class 0
            if (nsid >= max_sids && kf != cur_key) return Q8_ERR_WORKSPACE;
            const int s = sid_of(kf);
            p.first_sid[i] = static_cast<int16_t>(s);
            ++p.sharers[s];
        }
        if (e < kl + cl) {  // leaves its last row block before its last class
            if (nsid >= max_sids && kl != cur_key) return Q8_ERR_WORKSPACE;
            const int s = sid_of(kl);
            p.last_sid[i] = static_cast<int16_t>(s);
            ++p.sharers[s];
            p.pe[s] = static_cast<int8_t>(e - 1 - kl);
        }
    }
    p.early_signal = grid >= di->sm_count * occ ? 1 : 0;
    return launch_kernel(tile_kernel<MT, RAGGED>, dim3(grid), dim3(kThreads), smem_bytes(RAGGED), stream, chained,
                         p) ==
                   cudaSuccess
               ? Q8_OK
               : Q8_ERR_CUDA;
}

size_t up256(int64_t b) { return static_cast<size_t>((b + 255) / 256 * 256); }

int mt_for(int M) { return M <= 8 ? 1 : (M <= 16 ? 2 : 4); }

// Split row blocks a call may have: at most one per CTA boundary and one per
// row block.
int64_t max_splits(const q8_linear_desc *descs, int count, int M) {
    (void)M;
    int64_t rbs = 0;
    for (int i = 0; i < count; ++i) rbs += (descs[i].N + kRows - 1) / kRows;
    return std::min<int64_t>(kMaxGrid, rbs);
}

// workspace of one matrix's x: the binary16 copy and its flags (M <= 16),
// or for W8A8 the binary32 blocks, then the codes and scales of x
// (K not a multiple of 256: the copy's rows are padded to whole chunks)
size_t tile_x_region(int64_t K, int M, bool w8a8) {
    const int64_t KC = (K + kChunk - 1) / kChunk, MP = 8 * mt_for(M);
    if (w8a8) return up256(KC * MP * kW8Row * 4) + up256(KC * MP * (kW8Row + 2 * kW8Blocks));
    if (!tile_uses_x_copy(mt_for(M))) return 0;
    return up256(static_cast<int64_t>(M) * KC * kChunk * 2) + up256(KC * 4);
}

}  // namespace

bool tile_k_supported(int64_t K) { return K >= kChunk && K % 32 == 0; }
bool tile_k_whole_chunks(int64_t K) { return K > 0 && K % kChunk == 0; }

// M > 16 with classes: the running class sums of the CTAs, one slot per
// thread, for at most min(items, kMaxGrid) CTAs
int64_t fold_ctas(const q8_linear_desc *descs, int count, int M) {
    if (mt_for(M) != 4) return 0;
    int64_t items = 0;
    bool classes = false;
    for (int i = 0; i < count; ++i) {
        const int C = classes_for((descs[i].K + kChunk - 1) / kChunk, 4);
        classes = classes || C > 1;
        items += (descs[i].N + kRows - 1) / kRows * C;
    }
    return classes ? std::min<int64_t>(items, kMaxGrid) : 0;
}

size_t fold_bytes(int64_t ctas) { return static_cast<size_t>(ctas) * kWarps * 32 * 4 * 16; }

size_t tile_workspace(const q8_linear_desc *descs, int count, int M, size_t *ticket_off, size_t *ticket_bytes,
                      bool w8a8) {
    const int MT = mt_for(M);
    size_t bytes = 0;
    for (int i = 0; i < count; ++i) bytes += tile_x_region(descs[i].K, M, w8a8);
    const int64_t ms = max_splits(descs, count, M);
    if (ticket_off) *ticket_off = bytes;
    if (ticket_bytes) *ticket_bytes = up256(ms * kWarps * 4);
    if (ms > 0) bytes += up256(ms * kWarps * 4) + static_cast<size_t>(ms) * kMaxClasses * kWarps * 32 * MT * 16;
    // (then the fold slots, 256-byte aligned: the sizes above are multiples of 256)
    return bytes + fold_bytes(fold_ctas(descs, count, M));
}

q8_status launch_tile(const q8_linear_desc *descs, int count, int M, uint8_t *xws, uint32_t *dev_status,
                      cudaStream_t stream, bool chained, int mode) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    const bool invariant = mode == kModeInvariant, w8 = mode == kModeW8A8;
    if (M < (mode != kModeDefault ? 1 : 2) || M > 32 || count > Q8_MAX_BATCH) return Q8_ERR_UNSUPPORTED;
    for (int i = 0; i < count; ++i)
        if (mode == kModeDefault ? !tile_k_supported(descs[i].K) : !tile_k_whole_chunks(descs[i].K))
            return Q8_ERR_UNSUPPORTED;
    if (g_configured_dev != di->device) {
        if (!configure<1, false>() || !configure<2, false>() || !configure<4, false>() || !configure<1, true>() ||
            !configure<2, true>() || !configure<4, true>())
            return Q8_ERR_CUDA;
        g_configured_dev = di->device;
    }
    static thread_local TParams p;
    static thread_local XParams xp;
    const int MT = mt_for(M);
    const int MP = 8 * MT;
    // the batch-invariant arithmetic reads the caller's x and keeps one
    // class per row block (no shared row blocks): no workspace
    const bool copy = mode == kModeDefault && tile_uses_x_copy(MT);
    size_t ticket_off = 0, ticket_bytes = 0;
    const size_t need = invariant ? 0 : tile_workspace(descs, count, M, &ticket_off, &ticket_bytes, w8);
    if (need > 0 && xws == nullptr) return Q8_ERR_WORKSPACE;
    const int64_t ms = invariant ? 0 : max_splits(descs, count, M);
    p.tickets = ms > 0 ? reinterpret_cast<uint32_t *>(xws + ticket_off) : nullptr;
    p.parts = ms > 0 ? reinterpret_cast<float4 *>(xws + ticket_off + ticket_bytes) : nullptr;
    const int64_t fc = invariant ? 0 : fold_ctas(descs, count, M);
    p.fold = fc > 0 ? reinterpret_cast<float4 *>(xws + need - fold_bytes(fc)) : nullptr;

    // x copies: matrix i owns the workspace region after those of 0 .. i-1;
    // a matrix whose x (pointer, row stride, K) an earlier one already has
    // reads that one's copy
    int xcopy[Q8_MAX_BATCH];
    int chunks = 0;
    xp.count = 0;
    xp.M = M;
    size_t off = 0;
    // W8A8: the binary32 blocks, the codes and the scales of every distinct x
    // each in one array (x after x), so one quantizer launch serves them all
    int64_t w8_rows = 0, w8_before = 0;
    for (int i = 0; i < count && w8; ++i) {
        bool seen = false;
        for (int j = 0; j < i && !seen; ++j)
            seen = descs[j].x == descs[i].x && descs[j].ldx == descs[i].ldx && descs[j].K == descs[i].K;
        if (!seen) w8_rows += (descs[i].K + kChunk - 1) / kChunk * MP;
    }
    float *w8_xf = reinterpret_cast<float *>(xws);
    int8_t *w8_q = w8 ? reinterpret_cast<int8_t *>(xws + up256(w8_rows * kW8Row * 4)) : nullptr;
    uint16_t *w8_s = w8 ? reinterpret_cast<uint16_t *>(w8_q + w8_rows * kW8Row) : nullptr;
    for (int i = 0; i < count && (copy || w8); ++i) {
        const q8_linear_desc &d = descs[i];
        const size_t region = off;
        off += tile_x_region(d.K, M, w8);
        xcopy[i] = -1;
        for (int j = 0; j < i && xcopy[i] < 0; ++j)
            if (descs[j].x == d.x && descs[j].ldx == d.ldx && descs[j].K == d.K) xcopy[i] = xcopy[j];
        if (xcopy[i] >= 0) continue;
        const int64_t KC = (d.K + kChunk - 1) / kChunk;
        XJob &J = xp.j[xp.count];
        J.x = d.x;
        J.xo = reinterpret_cast<uint16_t *>(xws + region);
        J.flag = reinterpret_cast<uint32_t *>(xws + region + up256(static_cast<int64_t>(M) * KC * kChunk * 2));
        J.xf = w8_xf + w8_before * kW8Row;
        J.xq = w8 ? w8_q + w8_before * kW8Row : nullptr;
        if (w8) w8_before += KC * MP;
        J.ldx = d.ldx;
        J.K = KC * kChunk;
        J.kx = d.K;
        J.chunk_begin = chunks;
        chunks += static_cast<int>(KC);
        xcopy[i] = xp.count++;
    }
    int items = 0;
    double total_bytes = 0.0;
    for (int i = 0; i < count; ++i) {
        TDesc &D = p.d[i];
        TMaps &T = p.m[i];
        const q8_linear_desc &d = descs[i];
        // x as the kernel reads it: the copy [M][K rounded up to 256], or the
        // caller's [M][ldx]
        const bool whole = tile_k_whole_chunks(d.K);
        const int64_t KC = (d.K + kChunk - 1) / kChunk;
        const void *xsrc = copy ? static_cast<const void *>(xp.j[xcopy[i]].xo) : static_cast<const void *>(d.x);
        const int64_t xld = copy ? KC * kChunk : d.ldx;
        const uint64_t qdims[3] = {128, static_cast<uint64_t>(d.N), static_cast<uint64_t>(d.K / 128)};
        const uint64_t qstr[2] = {static_cast<uint64_t>(d.K), 128};
        const uint32_t qbox[3] = {128, kRows, 2};
        const uint64_t xdims[3] = {64, static_cast<uint64_t>(M), static_cast<uint64_t>(KC * 4)};
        const uint64_t xstr[2] = {static_cast<uint64_t>(xld) * 2, 128};
        const uint32_t xbox[3] = {64, static_cast<uint32_t>(MP), 4};
        const int64_t nb = d.K / 32;
        bool ok;
        if (whole) {
            ok = encode_tmap(&T.q, 1, d.q, 3, qdims, qstr, qbox, true) &&
                 encode_tmap(&T.x, 2, xsrc, 3, xdims, xstr, xbox, true) &&
                 encode_2d(&T.s, 2, d.s, static_cast<uint64_t>(nb), static_cast<uint64_t>(d.N),
                           static_cast<uint64_t>(nb) * 2, 8, kRows, false);
        } else {
            // codes [N][K] in boxes of 128 K-bytes x 128 rows; x the padded
            // copy (3-D, as above) or the caller's [M][K] in boxes of 64
            // columns x MP rows; no scale map (rows not 16-byte aligned)
            ok = encode_2d(&T.q, 1, d.q, static_cast<uint64_t>(d.K), static_cast<uint64_t>(d.N),
                           static_cast<uint64_t>(d.K), 128, kRows, true) &&
                 (copy ? encode_tmap(&T.x, 2, xsrc, 3, xdims, xstr, xbox, true)
                       : encode_2d(&T.x, 2, d.x, static_cast<uint64_t>(d.K), static_cast<uint64_t>(M),
                                   static_cast<uint64_t>(d.ldx) * 2, 64, static_cast<uint32_t>(MP), true));
        }
        if (!ok) return Q8_ERR_CUDA;
        D.y = d.y;
        D.s = d.s;
        D.nb = static_cast<int32_t>(nb);
        D.xflag = copy ? xp.j[xcopy[i]].flag
                  : w8 ? reinterpret_cast<const uint32_t *>(xp.j[xcopy[i]].xq)
                       : nullptr;
        D.ldy = d.ldy;
        D.N = static_cast<int32_t>(d.N);
        D.KC = static_cast<int32_t>(KC);
        D.C = invariant ? 1 : classes_for(KC, MT);
        for (int c = 0; c <= kMaxClasses; ++c)
            D.cls[c] = static_cast<int16_t>(c <= D.C ? class_lo(static_cast<int>(KC), D.C, c) : KC);
        D.item_begin = items;
        D.items = static_cast<int32_t>((d.N + kRows - 1) / kRows) * D.C;
        items += D.items;
        // (the same measure as the cut in run(): a partial last chunk counts
        // whole, as it costs a whole chunk's boxes and MMAs)
        total_bytes += static_cast<double>(d.N) * KC * kChunk * 1.0625;
    }
    p.status = dev_status;
    p.count = count;
    p.M = M;
    p.mode = mode;
    p.w8_codes = reinterpret_cast<const uint8_t *>(w8_q);
    p.w8_scales = reinterpret_cast<const uint8_t *>(w8_s);
    bool ragged = false;
    for (int i = 0; i < count; ++i) ragged = ragged || !tile_k_whole_chunks(descs[i].K);
    if (items == 0) return Q8_OK;
    // the x copy (waits for the kernels before it when chained), then the
    // tiles as its dependent: their first weight stages load while it runs
    if (copy && launch_kernel(x_copy_kernel, dim3(chunks), dim3(kThreads), 0, stream, chained, xp) != cudaSuccess)
        return Q8_ERR_CUDA;
    if (w8) {
        // x to binary32 blocks, then the Q8_0 quantizer over them (codes and
        // scales land in the stage layout); the tile kernel follows in order
        w8a8_widen_kernel<<<chunks, kThreads, 0, stream>>>(xp, MP);
        if (cudaGetLastError() != cudaSuccess) return Q8_ERR_CUDA;
        const q8_status st = launch_quantize(w8_xf, w8_rows, kW8Row, w8_q, w8_s, dev_status, stream);
        if (st != Q8_OK) return st;
    }
    const bool dep = copy || chained;
    const int msi = static_cast<int>(ms);
    if (ragged) {
        if (MT == 1) return run<1, true>(p, di, items, total_bytes, msi, stream, dep);
        return MT == 2 ? run<2, true>(p, di, items, total_bytes, msi, stream, dep)
                       : run<4, true>(p, di, items, total_bytes, msi, stream, dep);
    }
    if (MT == 1) return run<1, false>(p, di, items, total_bytes, msi, stream, dep);
    return MT == 2 ? run<2, false>(p, di, items, total_bytes, msi, stream, dep)
                   : run<4, false>(p, di, items, total_bytes, msi, stream, dep);
}

}  // namespace q8
