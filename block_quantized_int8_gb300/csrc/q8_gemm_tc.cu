// q8_gemm_tc.cu -- prefill-shaped Q8_0 W8A16 GEMM (M > 32) on the 5th
// generation tensor cores (tcgen05, tensor-memory accumulators).
//
// Y[m][n] = sum_k x[m][k] * bf16(s[n][k/32] * q[n][k]), fp32 accumulation,
// bf16 output.  "MODEL-BASELINE-RESULTS" (fak), ACT 4 (a batched prefill GEMM
// reads each weight once for all tokens, which makes the op compute-bound) and
// "Parity lane" item 2.
//
// The product is computed transposed, D = W' X^T: the dequantised weights are
// the tensor core's A operand (M = 128 weight rows) and the activations its
// B operand (N = BT = 256, 128 or 64 rows of x, "tokens").  One CTA (one per
// SM) computes a 128 x BT tile of Y^T over a range of k-tiles of 64, with
// three rings in shared memory, each stage freed as soon as its last reader
// is done:
//   x ring      the x tile of a k-tile: bf16, BT rows x 128 bytes, 128-byte
//               swizzle (the K-major layout the tensor core reads).
//   code ring   the codes of two k-tiles: int8, 128 rows x 128 bytes.
//   A ring      the dequantised weights of a k-tile: bf16(s q), 128 rows x
//               128 bytes, in the same swizzled K-major layout.
// Roles:
//   warp 0, lane 0  TMA producer of the x ring.  CTAs of neighbouring weight
//                   tiles need the same x tiles: groups of C of them (a
//                   thread-block cluster) take turns, CTA i % C loading
//                   k-tile i into all C rings by multicast.
//   warp 2, lane 0  TMA producer of the code ring.
//   warp 1          MMA issuer (lane 0): per k-tile 4 x tcgen05.mma.kind::f16
//                   (M = 128, N = BT, K = 16), both operands from shared
//                   memory, fp32 accumulators in tensor memory; stages freed
//                   in pairs by one commit per ring (none for a stage no
//                   later k-tile uses); a last commit signals the epilogue.
//   16 converters   warp 3 and the warps 4..23 of schedulers 0, 2 and 3;
//                   all of them work on every k-tile (a short latency per
//                   stage), both k-tiles of a code stage per pass, each on 32
//                   weight rows and 16 of the 64 codes of a row, turning
//                   codes into bf16(s q) (the product is exact in fp32, one
//                   rounding) and storing them into the A stages.  A code
//                   stage goes back to its producer as soon as every
//                   converter's loads of it have returned (the release
//                   depends on the loaded values), not when they are used.
//   The warps of scheduler 1 convert nothing: the MMA thread shares that
//   scheduler, and warps busy with the conversion arithmetic beside it hold
//   the tensor pipe well below its rate (measured; also with the weights in
//   tensor memory, where rows 32..63 can only be written from scheduler 1),
//   so scheduler 1 is left to the MMA issue.  After the main loop the 16
//   warps 4..19 run the epilogue: tcgen05.ld of the accumulators (a thread
//   holds one weight row), bf16, transposed through shared memory into Y's
//   row-major order, one TMA store.
//
// Split K (short N, long K: too few tiles for the SMs): the S CTAs of one
// tile form a thread-block cluster and take consecutive ranges of k-tiles.
// Each writes its fp32 partial tile, in 16-column units, into the shared
// memory of the unit's owner (distributed shared memory); after a cluster
// barrier each owner adds the S partials in cluster-rank order -- a fixed
// order, so the result is the same on every run -- and stores its units.
//
// All mbarrier waits are bounded; on expiry the CTA reports Q8_DEV_TIMEOUT,
// stops issuing work, still passes every cluster barrier, lets its copies
// and MMAs drain (bounded) and frees its tensor memory.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kWRows = 128;              // weight rows per tile (MMA M)
constexpr int kBK = 64;                  // k per k-tile (one 128-byte bf16 row of x)
constexpr int kRing = 8;                 // most stages of any ring
constexpr int kEpiWarps = 16;            // warps 4..19: the epilogue
constexpr int kConverters = 16;          // warp 3 and the warps 4..23 off the MMA warp's scheduler
constexpr int kThreads = 32 * 24;        // warps 0-2 roles, 3 converter, 4..23 converters / epilogue
constexpr int kCodeTile = 2 * kWRows * kBK;  // codes of two k-tiles of all 128 rows: [128 rows][128 bytes]
constexpr int kATile = kWRows * kBK * 2;     // bf16 weights of one k-tile: [128 rows][128 bytes]
constexpr int kCS = 2;                   // code ring stages (two k-tiles each)
constexpr int kMmaSched = 1;             // the scheduler of the MMA warp (warp 1): no converters there
constexpr int kSmemMax = 232448;         // dynamic shared memory of one CTA per SM
constexpr int kUnit = 16;                // columns (tokens) per split-K reduction unit
constexpr int kMaxSplits = 8;

// k-tile i uses x stage i % XS and A stage i % AS.  One barrier per stage
// says it is ready (the x bytes landed; the 12 converter warps stored
// their parts); stages are freed in pairs (k-tiles 2j
// and 2j + 1) by one MMA commit per ring, so the MMA thread waits twice per
// k-tile and commits twice per two.
struct GemmCtl {
    uint64_t x_full[kRing];     // x tile landed (TMA bytes)
    uint64_t a_full[kRing];     // A stage stored (12 converter warps)
    uint64_t x_free[kRing / 2]; // MMAs of x stages 2j, 2j + 1 done (commits of every CTA sharing the x tiles)
    uint64_t a_free[kRing / 2]; // MMAs of A stages 2j, 2j + 1 done (commits of every CTA sharing the A tiles)
    uint64_t c_full[kRing];     // code tile landed (TMA bytes)
    uint64_t c_empty[kRing];    // code tile read by every converter warp
    uint64_t acc_full;          // all MMAs done
    uint32_t tmem_base;
    int32_t abort_flag;
};

// Shared memory: [x ring][A ring][code ring][ctl], tiles on 1024-byte
// boundaries.  Both rings have an even number of stages (freed in pairs):
// at BT = 256, 4 x stages of 32 KB and 4 A stages of 16 KB; narrower tiles
// take more of each, up to 8.
template <int BT>
struct Layout {
    static constexpr int kX = BT * 128;  // x tile bytes
    static constexpr int kAvail = kSmemMax - 1024 - static_cast<int>(sizeof(GemmCtl)) - kCS * kCodeTile;
    static constexpr int kPair = kX + kATile;  // one x stage and one A stage
    static constexpr int kS0 = (kAvail / kPair < kRing ? kAvail / kPair : kRing) & ~1;
    static constexpr int kXS = kS0;
    // spare room goes to more A stages (the conversion's latency is the longer)
    static constexpr int kAS0 = ((kAvail - kXS * kX) / kATile) & ~1;
    static constexpr int kAS = kAS0 < kRing ? kAS0 : kRing;
    static constexpr int kA = kXS * kX;                     // offset of the A ring
    static constexpr int kCodes = kA + kAS * kATile;        // offset of the code ring
    static constexpr int kCtl = kCodes + kCS * kCodeTile;
    static constexpr int kSmem = 1024 + kCtl + static_cast<int>(sizeof(GemmCtl));
    static constexpr int kTmemCols = BT;                    // the accumulators
    static_assert(kXS >= 2 && kAS >= 2, "rings too small");
    static_assert(kSmem <= kSmemMax, "shared memory");
};

struct GemmParams {
    CUtensorMap tm_x;  // bf16 [M][ldx], box {64, BT}, 128-byte swizzle
    CUtensorMap tm_q;  // int8 [N][K], box {128, 128} (two k-tiles), 128-byte swizzle
    CUtensorMap tm_y;  // bf16 [M][ldy], box {128, BT} (S == 1) or {128, 16} (S > 1)
    const uint16_t *s; // binary16 scales [N][K/32]
    uint32_t *status;
    int32_t M, N, K, nb, KT;  // KT: k-tiles, ceil(K / 64)
    int32_t S;                // K splits (the cluster's size along z)
    int32_t C;                // CTAs sharing each x tile by multicast (the cluster's size along x)
    uint32_t zero;            // 0 (a value the compiler cannot see: see warp_loaded_zero)
};

// ---- tcgen05 / TMA wrappers ---------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}
// The same box into the same shared-memory offset of every CTA in ctamask
// (each CTA's barrier at bar's offset receives the bytes that land in it).
__device__ __forceinline__ void tma_load_2d_mc(void *dst, const CUtensorMap *tm, int c0, int c1, uint64_t *bar,
                                               uint16_t ctamask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster "
        "[%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_addr(bar)),
           "h"(ctamask)
        : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *tm, const void *src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_addr(src)) : "memory");
}
__device__ __forceinline__ void bulk_commit_and_drain() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), leading byte offset unused.
__device__ __forceinline__ uint64_t sw128_desc(const void *tile) {
    const uint64_t addr = smem_addr(tile);
    uint64_t d = 0;
    d |= (addr & 0x3FFFFull) >> 4;                 // start address
    d |= static_cast<uint64_t>(1) << 16;           // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;   // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;           // descriptor version (sm_100 family)
    d |= static_cast<uint64_t>(2) << 61;           // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: D f32, A bf16, B bf16, both K-major,
// M = 128, N = BT.
template <int BT>
constexpr uint32_t idesc_for() {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BT >> 3) << 17) |
           (static_cast<uint32_t>(kWRows >> 4) << 24);
}

// D[tmem_d] (+)= A[desc] * B[desc]^T
template <int BT>
__device__ __forceinline__ void umma_ss(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(tmem_d), "l"(da), "l"(db), "r"(idesc_for<BT>()), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_addr(bar)) : "memory");
}
// Arrive on the barrier at bar's offset in every CTA of ctamask once the
// MMAs issued so far are done.
__device__ __forceinline__ void umma_commit_mc(uint64_t *bar, uint16_t ctamask) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 :: "r"(smem_addr(bar)), "h"(ctamask) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Four int8 codes (one word, code 0 in the low byte) times the block scale
// (s2 = the scale in both halves) -> bf16(s q) for codes 0,1 (lo) and 2,3
// (hi).  0x4B000000 | u is 2^23 + u for the byte u = q + 128, so subtracting
// 2^23 + 128 gives q exactly; s q is exact in fp32 (8-bit by 11-bit
// significands); the conversion rounds once, to nearest even.  Packed
// f32x2 arithmetic: 11 instructions per 4 codes.
__device__ __forceinline__ void codes4_scaled_bf16(uint32_t w, unsigned long long s2, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const unsigned long long bias = 0xCB000080CB000080ull;  // -(2^23 + 128) in both halves
    const unsigned long long m01 = static_cast<unsigned long long>(__byte_perm(u, 0x4B000000u, 0x7650)) |
                                   static_cast<unsigned long long>(__byte_perm(u, 0x4B000000u, 0x7651)) << 32;
    const unsigned long long m23 = static_cast<unsigned long long>(__byte_perm(u, 0x4B000000u, 0x7652)) |
                                   static_cast<unsigned long long>(__byte_perm(u, 0x4B000000u, 0x7653)) << 32;
    unsigned long long a, b;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(a) : "l"(m01), "l"(bias));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(b) : "l"(m23), "l"(bias));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(a) : "l"(a), "l"(s2));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(b) : "l"(b), "l"(s2));
    lo = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(a)), __uint_as_float(static_cast<uint32_t>(a >> 32)));
    hi = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(b)), __uint_as_float(static_cast<uint32_t>(b >> 32)));
}
__device__ __forceinline__ uint16_t bf16_rn(float v) {
    return static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
}

// thread-block cluster helpers
__device__ __forceinline__ uint32_t cluster_ctaid_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctaid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_ctaid_z() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctaid.z;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
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

// Reduction units of a split tile: NU = BT / 16 units of 16 columns, owned by
// the S cluster ranks in contiguous runs (rank o owns [o NU / S, (o+1) NU / S)).
__host__ __device__ __forceinline__ int unit_lo(int NU, int S, int o) { return o * NU / S; }

template <int BT>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    // tiles need 1024-byte alignment (swizzle atoms)
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    using L = Layout<BT>;
    constexpr int XS = L::kXS, AS = L::kAS;
    GemmCtl &sm = *reinterpret_cast<GemmCtl *>(base + L::kCtl);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int n0 = blockIdx.x * kWRows;
    const int m0 = blockIdx.y * BT;
    const int S = p.S;
    const int z = static_cast<int>(blockIdx.z);
    // K splits in whole groups of 4 k-tiles (the 3-D code view's box starts
    // at an even k-tile; ranges stay coarse)
    const int KQ = (p.KT + 3) / 4;
    const int kt0 = 4 * (z * KQ / S);
    const int nk = min(p.KT, 4 * ((z + 1) * KQ / S)) - kt0;
    const int C = p.C;
    // position in the cluster: cx along the CTAs that share x tiles, cz
    // along the K splits of one tile
    const int cx = C > 1 ? static_cast<int>(cluster_ctaid_x()) : 0;
    const int cz = S > 1 ? static_cast<int>(cluster_ctaid_z()) : 0;
    const uint16_t xmask = static_cast<uint16_t>(((1u << C) - 1u) << (C * cz));
    auto x_tile = [&](int xs) { return base + xs * L::kX; };
    auto a_tile = [&](int as) { return base + L::kA + as * kATile; };
    auto code_tile = [&](int cs) { return base + L::kCodes + cs * kCodeTile; };
    // k-tile i (>= ring size R) may reuse its stage once the MMAs of k-tile
    // i - R are done: the pair barrier of (i - R) / 2, in its round
    auto wait_pair = [&](uint64_t *bars, int R, int i) {
        const int pr = (i - R) >> 1;
        return wait_or_abort(sm, &bars[pr % (R / 2)], (pr / (R / 2)) & 1, p.status);
    };

    if (tid == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&sm.x_full[i], 1);
            mbar_init(&sm.a_full[i], kConverters);
            mbar_init(&sm.c_full[i], 1);
            mbar_init(&sm.c_empty[i], kConverters);       // every converter, once per stage (both k-tiles)
            if (i < kRing / 2) {
                mbar_init(&sm.x_free[i], C);  // the MMAs of every CTA that shares the x tiles
                mbar_init(&sm.a_free[i], 1);
            }
        }
        mbar_init(&sm.acc_full, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_addr(&sm.tmem_base)), "r"(L::kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    // peers multicast into this CTA's rings and arrive on its barriers: all
    // barriers of the cluster are initialised before anyone starts
    if (C * S > 1) cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;       // accumulators: columns [0, BT)
    bool ok = true;

    if (warp == 0 && lane == 0) {
        // -------------------------------------------------- TMA producer: x
        for (int i = 0; i < nk; ++i) {
            const int xs = i % XS;
            if (i >= XS && !wait_pair(sm.x_free, XS, i)) break;
            mbar_arrive_expect_tx(&sm.x_full[xs], L::kX);
            if (C == 1)
                tma_load_2d(x_tile(xs), &p.tm_x, (kt0 + i) * kBK, m0, &sm.x_full[xs]);
            else if (i % C == cx)
                // the group's CTAs take turns: k-tile i comes from CTA i % C,
                // into every CTA of the group (a TMA box costs the same time
                // whatever its size, so each SM issues 1 / C of the boxes)
                tma_load_2d_mc(x_tile(xs), &p.tm_x, (kt0 + i) * kBK, m0, &sm.x_full[xs], xmask);
        }
    } else if (warp == 2 && lane == 0) {
        // ---------------------------------------------- TMA producer: codes
        // one box of 128-byte rows per pair of k-tiles
        for (int j = 0; 2 * j < nk; ++j) {
            const int cs = j % kCS;
            if (j >= kCS && !wait_or_abort(sm, &sm.c_empty[cs], ((j / kCS) - 1) & 1, p.status)) break;
            mbar_arrive_expect_tx(&sm.c_full[cs], kCodeTile);
            tma_load_2d(code_tile(cs), &p.tm_q, (kt0 + 2 * j) * kBK, n0, &sm.c_full[cs]);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        // the whole warp walks the stages (waits by every lane keep it
        // converged); lane 0 issues the MMAs and the commits.  Descriptors
        // of stage 0; stage s starts s tiles later (the start address field
        // counts 16-byte units).
        const uint64_t db0 = sw128_desc(x_tile(0));
        const uint64_t da0 = sw128_desc(a_tile(0));
        bool go = true;
        for (int i0 = 0; go && i0 < nk; i0 += 2) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = i0 + h;
                if (i >= nk) break;
                const int xs = i % XS, as = i % AS;
                const bool ready = wait_or_abort(sm, &sm.x_full[xs], (i / XS) & 1, p.status) &&
                                   wait_or_abort(sm, &sm.a_full[as], (i / AS) & 1, p.status);
                if (!__all_sync(0xFFFFFFFFu, ready)) {
                    go = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        // 16 bf16 = 32 bytes per step along K in both operands
                        umma_ss<BT>(tmem, da0 + static_cast<uint64_t>(as * (kATile >> 4) + 2 * kk),
                                    db0 + static_cast<uint64_t>(xs * (L::kX >> 4) + 2 * kk),
                                    (i > 0 || kk > 0) ? 1u : 0u);
                }
                __syncwarp();
            }
            if (!go) break;
            // stages of k-tiles i0 and i0 + 1 are free once these MMAs are
            // done (every sharer of a tile may refill it); a stage no later
            // k-tile uses gets no commit, so no arrival from a peer can come
            // after the main loops
            if (lane == 0) {
                const int pr = i0 >> 1;
                if (i0 + XS < nk) {
                    if (C == 1)
                        umma_commit(&sm.x_free[pr % (XS / 2)]);
                    else
                        umma_commit_mc(&sm.x_free[pr % (XS / 2)], xmask);
                }
                if (i0 + AS < nk) umma_commit(&sm.a_free[pr % (AS / 2)]);
            }
            __syncwarp();
        }
        if (lane == 0) umma_commit(&sm.acc_full);
        __syncwarp();
    } else if (warp >= 3) {
        if ((warp & 3) != kMmaSched) {
            // --------------------------------------------------- converters
            // every k-tile is converted by all 16 converter warps (short
            // latency: the A ring is only 4 deep at BT = 256), both k-tiles of
            // a code stage in one pass (twice the independent work per
            // wait): converter c owns weight rows 32 (c % 4) .. +31 and the
            // 16 codes 16 (c / 4) .. +15 of each row's 64 in a k-tile, i.e.
            // one 16-byte unit of the code row, two 16-byte chunks of the A
            // row and one block scale per k-tile
            const int wi = warp - 4;
            const int c = warp == 3 ? 0 : 1 + wi - (wi + 3 - kMmaSched) / 4;
            const int h = c >> 2;
            const int r = 32 * (c & 3) + lane;           // weight row in the tile
            const uint16_t *srow = p.s + static_cast<int64_t>(min(n0 + r, p.N - 1)) * p.nb;
            const bool row_ok = n0 + r < p.N;
            // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r & 7)
            const int sw = r & 7;
            auto scale_of = [&](int i) -> uint32_t {
                const int kb = 2 * (kt0 + i) + (h >> 1);  // codes 16 h .. 16 h + 15 lie in one block
                return (row_ok && i < nk && kb < p.nb) ? ldg_nc_u16(srow + kb) : 0u;
            };
            // 8 codes -> 4 bf16x2 words -> 16-byte chunk j of the A row
            auto put = [&](uint8_t *arow, int j, uint32_t w0, uint32_t w1, unsigned long long sc) {
                uint32_t o0, o1, o2, o3;
                codes4_scaled_bf16(w0, sc, o0, o1);
                codes4_scaled_bf16(w1, sc, o2, o3);
                *reinterpret_cast<uint4 *>(arow + ((j ^ sw) << 4)) = make_uint4(o0, o1, o2, o3);
            };
            uint32_t sa = scale_of(0), sb = scale_of(1);
            for (int m = 0; 2 * m < nk; ++m) {
                const int i0 = 2 * m;
                const bool two = i0 + 1 < nk;
                const int cs = m % kCS, as = i0 % AS;   // the pair's A stages as, as + 1 (AS is even)
                // (one pair barrier frees both A stages)
                bool good = wait_or_abort(sm, &sm.c_full[cs], (m / kCS) & 1, p.status) &&
                            (i0 < AS || wait_pair(sm.a_free, AS, i0));
                if (!__all_sync(0xFFFFFFFFu, good)) {
                    ok = false;
                    break;
                }
                // my 16 codes of each k-tile: 16-byte units h and 4 + h of
                // the 128-byte code row, swizzled
                const uint8_t *crow = code_tile(cs) + r * 128;
                const uint4 ca = *reinterpret_cast<const uint4 *>(crow + ((h ^ sw) << 4));
                const uint4 cb = *reinterpret_cast<const uint4 *>(crow + (((4 + h) ^ sw) << 4));
                // the codes are in registers: hand the stage back to its
                // producer once the loads have returned (see warp_loaded_zero)
                {
                    const uint32_t dep = warp_loaded_zero(ca.x | ca.y | ca.z | ca.w | cb.x | cb.y | cb.z | cb.w, p.zero);
                    if (lane == 0)
                        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];"
                                     :: "r"(smem_addr(&sm.c_empty[cs]) + dep) : "memory");
                }
                const unsigned long long sca =
                    static_cast<unsigned long long>(__float_as_uint(f16_bits_to_f32(sa))) * 0x100000001ull;
                const unsigned long long scb =
                    static_cast<unsigned long long>(__float_as_uint(f16_bits_to_f32(sb))) * 0x100000001ull;
                sa = scale_of(i0 + 2);
                sb = scale_of(i0 + 3);
                uint8_t *arow = a_tile(as) + r * 128;
                put(arow, 2 * h, ca.x, ca.y, sca);
                put(arow, 2 * h + 1, ca.z, ca.w, sca);
                if (two) {
                    arow += kATile;
                    put(arow, 2 * h, cb.x, cb.y, scb);
                    put(arow, 2 * h + 1, cb.z, cb.w, scb);
                }
                // generic stores -> visible to the tensor core (async proxy)
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(&sm.a_full[as])) : "memory");
                    if (two)
                        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];"
                                     :: "r"(smem_addr(&sm.a_full[as + 1])) : "memory");
                }
            }
        }
        ok = __all_sync(0xFFFFFFFFu, ok && wait_or_abort(sm, &sm.acc_full, 0, p.status));
        tc_fence_after();
    }
    __syncwarp();  // lanes of the role warps reconverge before the warp-wide steps below

    // ------------------------------------------------------------- epilogue
    // warps 4..: warp (qd, part) drains TMEM lanes 32 qd .. +31 (weight rows)
    // and columns [part BT / 4, (part + 1) BT / 4) (tokens)
    const bool epi = warp >= 4 && warp < 4 + kEpiWarps;
    const int qd = warp & 3;
    const int part = (warp - 4) >> 2;
    const int r = 32 * qd + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
    if (S == 1) {
        if (epi && ok) {
            // the whole tile, bf16, [BT tokens][128 rows] in the (now idle) ring
            uint16_t *out = reinterpret_cast<uint16_t *>(base);
            constexpr int kCols = BT / 4;  // 16, 32 or 64 columns per warp
#pragma unroll 1
            for (int c0 = part * kCols; c0 < (part + 1) * kCols; c0 += 32) {
                // up to 32 columns per round trip to tensor memory
                uint32_t v[2][16];
                tmem_ld16_async(tmem + lane_off + static_cast<uint32_t>(c0), v[0]);
                if (kCols > 16) tmem_ld16_async(tmem + lane_off + static_cast<uint32_t>(c0 + 16), v[1]);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) out[(c0 + j) * kWRows + r] = bf16_rn(__uint_as_float(v[0][j]));
                if (kCols > 16) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) out[(c0 + 16 + j) * kWRows + r] = bf16_rn(__uint_as_float(v[1][j]));
                }
            }
            fence_proxy_async_smem();
        }
        if (epi) named_bar_sync(1, kEpiWarps * 32);
        // (a CTA past N or M only fills out a cluster: nothing to store)
        if (warp == 4 && lane == 0 && n0 < p.N && m0 < p.M && !*reinterpret_cast<volatile int32_t *>(&sm.abort_flag)) {
            tma_store_2d(&p.tm_y, base, n0, m0);
            bulk_commit_and_drain();
        }
    } else {
        // split K: every CTA of the cluster is past its main loop before any
        // writes into another's ring
        constexpr int NU = BT / kUnit;
        const int umax = (NU + S - 1) / S;
        cluster_sync_all();
        if (epi && ok) {
            // my partial, unit by unit, into the owner's slot for my rank:
            // slot [src][unit][4 column groups][128 rows] float4
#pragma unroll 1
            for (int u0 = part * (NU / 4); u0 < (part + 1) * (NU / 4); u0 += 2) {
                // two units per round trip to tensor memory
                const int nu = min(2, (part + 1) * (NU / 4) - u0);
                uint32_t v[2][16];
                tmem_ld16_async(tmem + lane_off + static_cast<uint32_t>(u0 * kUnit), v[0]);
                if (nu > 1) tmem_ld16_async(tmem + lane_off + static_cast<uint32_t>((u0 + 1) * kUnit), v[1]);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    if (k >= nu) break;
                    const int u = u0 + k;
                    int o = 0;
                    while (o + 1 < S && unit_lo(NU, S, o + 1) <= u) ++o;
                    const int ul = u - unit_lo(NU, S, o);
                    const uint32_t slot =
                        smem_addr(base) + static_cast<uint32_t>(((cz * umax + ul) * 4 * kWRows) * 16);
                    // the owner: same tile (same cx), split o
                    const uint32_t remote = map_rank(slot, static_cast<uint32_t>(cx + C * o));
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        st_cluster_v4(remote + static_cast<uint32_t>((g * kWRows + r) * 16), v[k][4 * g],
                                      v[k][4 * g + 1], v[k][4 * g + 2], v[k][4 * g + 3]);
                }
            }
        }
        cluster_sync_all();
        // my units: add the S partials in rank order, bf16, store
        const int ub = unit_lo(NU, S, cz);
        const int U = unit_lo(NU, S, cz + 1) - ub;
        uint16_t *out = reinterpret_cast<uint16_t *>(base + S * umax * 4 * kWRows * 16);
        if (epi && !*reinterpret_cast<volatile int32_t *>(&sm.abort_flag)) {
            const float4 *slots = reinterpret_cast<const float4 *>(base);
            const int t = tid - 128;
#pragma unroll 1
            for (int idx = t; idx < U * 4 * kWRows; idx += kEpiWarps * 32) {
                const int ul = idx / (4 * kWRows);
                const int g = (idx / kWRows) & 3;
                const int rr = idx % kWRows;
                float4 a = slots[(0 * umax + ul) * 4 * kWRows + g * kWRows + rr];
                for (int src = 1; src < S; ++src) {
                    const float4 b = slots[(src * umax + ul) * 4 * kWRows + g * kWRows + rr];
                    a.x += b.x;
                    a.y += b.y;
                    a.z += b.z;
                    a.w += b.w;
                }
                const int tok = ul * kUnit + 4 * g;
                out[(tok + 0) * kWRows + rr] = bf16_rn(a.x);
                out[(tok + 1) * kWRows + rr] = bf16_rn(a.y);
                out[(tok + 2) * kWRows + rr] = bf16_rn(a.z);
                out[(tok + 3) * kWRows + rr] = bf16_rn(a.w);
            }
            fence_proxy_async_smem();
        }
        if (epi) named_bar_sync(1, kEpiWarps * 32);
        if (warp == 4 && lane == 0 && n0 < p.N && !*reinterpret_cast<volatile int32_t *>(&sm.abort_flag)) {
            for (int ul = 0; ul < U; ++ul) {
                const int row = m0 + (ub + ul) * kUnit;
                if (row < p.M) tma_store_2d(&p.tm_y, out + ul * kUnit * kWRows, n0, row);
            }
            bulk_commit_and_drain();
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
    // no CTA leaves while a peer may still arrive on its barriers or write
    // into its shared memory
    if (C * S > 1) cluster_sync_all();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(L::kTmemCols) : "memory");
    }
}

// ---- host side ---------------------------------------------------------------
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

bool encode(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
            uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_configured_dev = -1;
constexpr int kMaxCluster = 16;
constexpr int kMaxMulticast = 8;
// co-resident clusters of shape (C, 1, S), per tile width; -1: not asked yet
int g_max_clusters[3][kMaxMulticast + 1][kMaxSplits + 1];

template <int BT>
size_t smem_for() {
    return static_cast<size_t>(Layout<BT>::kSmem);
}

// The reduction slots and output units of a split tile fit the idle rings.
template <int BT>
bool split_fits(int S) {
    const int NU = BT / kUnit;
    const int umax = (NU + S - 1) / S;
    return S * umax * 4 * kWRows * 16 + umax * kUnit * kWRows * 2 <= Layout<BT>::kCtl;
}

template <int BT>
bool configure() {
    if (cudaFuncSetAttribute(gemm_tc_kernel<BT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_for<BT>())) != cudaSuccess)
        return false;
    return cudaFuncSetAttribute(gemm_tc_kernel<BT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
           cudaSuccess;
}

cudaLaunchAttribute cluster_attr(int C, int S) {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = static_cast<unsigned>(C);
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = static_cast<unsigned>(S);
    return a;
}

int bt_of(int tile) { return tile == Q8_GEMM_TILE_256x128 ? 256 : (tile == Q8_GEMM_TILE_128x128 ? 128 : 64); }
int bi_of(int bt) { return bt == 256 ? 0 : (bt == 128 ? 1 : 2); }

template <int BT>
int query_clusters(int C, int S) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C), 1, static_cast<unsigned>(S));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_for<BT>();
    cudaLaunchAttribute attr[1] = {cluster_attr(C, S)};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, gemm_tc_kernel<BT>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        nc = 0;
    }
    return nc;
}

// CTAs of one launch that can run at once with clusters of (C, 1, S).
int64_t cta_slots(int bt, int C, int S, int sm_count) {
    if (C * S == 1) return sm_count;
    int &nc = g_max_clusters[bi_of(bt)][C][S];
    if (nc < 0) nc = bt == 256 ? query_clusters<256>(C, S) : bt == 128 ? query_clusters<128>(C, S)
                                                                        : query_clusters<64>(C, S);
    return static_cast<int64_t>(nc) * C * S;
}

bool shape_ok(int bt, int C, int S, int KT, int sm_count) {
    if (S < 1 || S > kMaxSplits || S > (KT + 3) / 4 || C > kMaxMulticast || C * S > kMaxCluster) return false;
    if (S > 1 && (bt == 256 ? !split_fits<256>(S) : bt == 128 ? !split_fits<128>(S) : !split_fits<64>(S)))
        return false;
    return cta_slots(bt, C, S, sm_count) > 0;
}

// Modelled time of a launch (clocks): waves of CTAs, each running its
// k-tiles at the slowest of the tensor rate of its tile width, the
// dequantisers' rate (kConvClk per k-tile of 128 weight rows, measured),
// its SM's TMA issue (~390 clocks per box, whatever its size: 1 / C x
// boxes and 1/2 code box per k-tile) and its share of L2 (~12 KB/clock for
// all CTAs at once), plus a fixed start and, when split, the exchange of
// partial tiles.
constexpr double kConvClk = 1400.0;
double model_time(int bt, int C, int S, int64_t N, int64_t M, int KT, int sm_count) {
    const int64_t ctas = ((N + kWRows * C - 1) / (kWRows * C)) * C * ((M + bt - 1) / bt) * S;
    const int64_t slots = cta_slots(bt, C, S, sm_count);
    if (slots <= 0) return 1e30;
    const int64_t waves = (ctas + slots - 1) / slots;
    const double conc = static_cast<double>(std::min(ctas, slots));
    const double bytes = bt * 128.0 + kWRows * kBK;        // delivered into the SM per k-tile
    const double boxes = 1.0 / C + 0.5;                    // issued by the SM per k-tile, ~390 clocks each
    const double kt_clk = std::max(std::max(2.0 * bt, kConvClk), std::max(boxes * 390.0, conc * bytes / 12000.0));
    const double per_cta = 4.0 * std::ceil(std::ceil(KT / 4.0) / S) * kt_clk + 3000.0 +
                           (S > 1 ? bt * kWRows * 4.0 * (S - 1) / S / 24.0 + 2000.0 : 0.0);
    return static_cast<double>(waves) * per_cta;
}

template <int BT>
q8_status run(GemmParams &p, const int8_t *q, const uint16_t *x, const uint16_t *y, int64_t ldx, int64_t ldy,
              int C, int S, cudaStream_t stream) {
    if (!encode(&p.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.M),
                static_cast<uint64_t>(ldx) * 2, kBK, BT, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.N),
                static_cast<uint64_t>(p.K), 2 * kBK, kWRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(&p.tm_y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, y, static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.M),
                static_cast<uint64_t>(ldy) * 2, kWRows, S == 1 ? BT : kUnit, CU_TENSOR_MAP_SWIZZLE_NONE))
        return Q8_ERR_CUDA;
    p.S = S;
    p.C = C;
    // weight tiles rounded up to whole multicast groups (the extra CTAs
    // load their share of x and store nothing)
    const unsigned gx = static_cast<unsigned>((p.N + kWRows * C - 1) / (kWRows * C) * C);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, static_cast<unsigned>((p.M + BT - 1) / BT), static_cast<unsigned>(S));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_for<BT>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {cluster_attr(C, S)};
    cfg.attrs = attr;
    cfg.numAttrs = C * S > 1 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BT>, p) == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

}  // namespace

q8_status launch_gemm_tc(const int8_t *q, const uint16_t *s, int64_t N, int64_t K, const uint16_t *x, int64_t ldx,
                         int32_t M, uint16_t *y, int64_t ldy, int32_t tile, int32_t splits, uint32_t *dev_status,
                         cudaStream_t stream) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (g_configured_dev != di->device) {
        if (!configure<256>() || !configure<128>() || !configure<64>()) return Q8_ERR_CUDA;
        for (auto &a : g_max_clusters)
            for (auto &b : a)
                for (int &c : b) c = -1;
        g_configured_dev = di->device;
    }
    GemmParams p;
    p.s = s;
    p.zero = 0;
    p.status = dev_status;
    p.M = M;
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.nb = static_cast<int32_t>(K / 32);
    p.KT = static_cast<int32_t>((K + kBK - 1) / kBK);
    // the (tile, split, multicast group) with the smallest modelled time
    // among those this device can co-schedule; the multicast group does not
    // change the arithmetic, the tile and split are the caller's if given
    int bt = 0, S = 0, C = 0;
    double best = 1e300;
    // Q8_GEMM_MULTICAST = 1, 2, 4 or 8 asks for that multicast group
    // (measurement); ignored where no allowed shape has it
    int force_c = 0;
    if (const char *e = std::getenv("Q8_GEMM_MULTICAST")) force_c = std::atoi(e);
    for (int pass = 0; pass < 2 && bt == 0; ++pass, force_c = 0)
    for (int t = Q8_GEMM_TILE_256x128; t <= Q8_GEMM_TILE_64x128; ++t) {
        if (tile != Q8_GEMM_TILE_AUTO && t != tile) continue;
        for (int sp = 1; sp <= kMaxSplits; ++sp) {
            if (splits != 0 && sp != splits) continue;
            for (int c = 1; c <= kMaxMulticast; c *= 2) {
                if (force_c > 0 && c != force_c) continue;
                if (!shape_ok(bt_of(t), c, sp, p.KT, di->sm_count)) continue;
                const double tm = model_time(bt_of(t), c, sp, N, M, p.KT, di->sm_count);
                if (tm < best * 0.999) {
                    best = tm;
                    bt = bt_of(t);
                    S = sp;
                    C = c;
                }
            }
        }
    }
    if (bt == 0) return Q8_ERR_UNSUPPORTED;
    if (bt == 256) return run<256>(p, q, x, y, ldx, ldy, C, S, stream);
    if (bt == 128) return run<128>(p, q, x, y, ldx, ldy, C, S, stream);
    return run<64>(p, q, x, y, ldx, ldy, C, S, stream);
}

}  // namespace q8
