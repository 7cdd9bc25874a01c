// q8_gguf.cu -- repack between GGUF's interleaved Q8_0 blocks and the planar
// layout of this library.
//
// A GGUF Q8_0 tensor (the model file format the "aubier" README's engine
// loads, "Layout", and the serverAppConfigs log's models ship in) stores each
// block of 32 weights as 34 bytes:
// the binary16 scale d, then the 32 int8 codes; blocks follow each other
// along the row and rows follow each other, so a [rows][K] tensor is one run
// of rows * K / 32 blocks.  The planar layout keeps the same blocks as codes
// [rows][K] (32 bytes per block, contiguous) and scales [rows][K/32] (2 bytes
// per block), so block g maps to codes[32 g .. 32 g + 32) and scales[g]
// whatever the row length.  Pure data movement, bit for bit; HBM-bound at
// 34 bytes in and 34 bytes out per block.
//
// Ingest: one thread per block.  A block starts at byte 34 g of a 16-byte
// aligned buffer, so at an even offset o (0..14) inside its 16-byte chunk;
// the thread loads the 48 bytes from the chunk start (three 16-byte loads,
// the warp's windows overlap and share cache lines) and funnel-shifts the
// scale and the eight code words out, then stores the codes as two 16-byte
// words.  Blocks whose 48-byte window would pass the end of the buffer use
// 2-byte loads instead.
#include <algorithm>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kThreads = 256;
constexpr int64_t kBlockBytes = 34;

// Scale and codes of the block at even byte offset O of the 48-byte window w.
template <int O>
__device__ __forceinline__ void extract(const uint32_t (&w)[12], uint32_t &d, uint32_t (&c)[8]) {
    static_assert(O % 2 == 0 && O >= 0 && O <= 14, "blocks start at even offsets");
    constexpr int sw = O / 4, sb = (O % 4) * 8;
    d = (w[sw] >> sb) & 0xFFFFu;
    constexpr int a = (O + 2) / 4, r = ((O + 2) % 4) * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if constexpr (r == 0)
            c[i] = w[a + i];
        else
            c[i] = __funnelshift_r(w[a + i], w[a + i + 1], r);
    }
}

__global__ void __launch_bounds__(kThreads) gguf_ingest_kernel(const uint8_t *__restrict__ blocks, int64_t nblocks,
                                                               int8_t *__restrict__ q, uint16_t *__restrict__ s) {
    const int64_t end = nblocks * kBlockBytes;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; g < nblocks;
         g += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int64_t at = g * kBlockBytes;
        const int o = static_cast<int>(at & 15);
        const int64_t chunk = at - o;
        uint32_t d, c[8];
        if (chunk + 48 <= end) {
            const uint4 *p = reinterpret_cast<const uint4 *>(blocks + chunk);
            uint32_t w[12];
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const uint4 v = __ldg(p + i);
                w[4 * i] = v.x;
                w[4 * i + 1] = v.y;
                w[4 * i + 2] = v.z;
                w[4 * i + 3] = v.w;
            }
            switch (o >> 1) {
                case 0: extract<0>(w, d, c); break;
                case 1: extract<2>(w, d, c); break;
                case 2: extract<4>(w, d, c); break;
                case 3: extract<6>(w, d, c); break;
                case 4: extract<8>(w, d, c); break;
                case 5: extract<10>(w, d, c); break;
                case 6: extract<12>(w, d, c); break;
                default: extract<14>(w, d, c); break;
            }
        } else {
            // the last blocks: exactly their own 34 bytes, 2 at a time
            const uint16_t *h = reinterpret_cast<const uint16_t *>(blocks + at);
            d = __ldg(h);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                c[i] = static_cast<uint32_t>(__ldg(h + 1 + 2 * i)) |
                       (static_cast<uint32_t>(__ldg(h + 2 + 2 * i)) << 16);
        }
        uint4 *qo = reinterpret_cast<uint4 *>(q + 32 * g);
        qo[0] = make_uint4(c[0], c[1], c[2], c[3]);
        qo[1] = make_uint4(c[4], c[5], c[6], c[7]);
        s[g] = static_cast<uint16_t>(d);
    }
}

// Export: a warp takes 32 consecutive blocks (1088 bytes, a multiple of 16,
// so 16-byte aligned in the output), each lane writes its block into a
// shared-memory copy of that run, then the warp stores the run with 16-byte
// stores.  A last run of fewer than 32 blocks uses 2-byte stores.
__global__ void __launch_bounds__(kThreads) gguf_export_kernel(const int8_t *__restrict__ q,
                                                               const uint16_t *__restrict__ s, int64_t nblocks,
                                                               uint8_t *__restrict__ blocks) {
    __shared__ __align__(16) uint16_t run[kThreads / 32][32 * kBlockBytes / 2];
    const int lane = threadIdx.x & 31;
    uint16_t *r = run[threadIdx.x >> 5];
    const int64_t nruns = (nblocks + 31) / 32;
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5); c < nruns;
         c += wstride) {
        const int64_t g = 32 * c + lane;
        uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        uint16_t d = 0;
        if (g < nblocks) {
            const uint4 *qi = reinterpret_cast<const uint4 *>(q + 32 * g);
            const uint4 a = __ldg(qi), b = __ldg(qi + 1);
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
            w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
            d = __ldg(s + g);
        }
        if (32 * c + 32 <= nblocks) {
            uint16_t *h = r + lane * (kBlockBytes / 2);
            h[0] = d;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                h[1 + 2 * i] = static_cast<uint16_t>(w[i] & 0xFFFFu);
                h[2 + 2 * i] = static_cast<uint16_t>(w[i] >> 16);
            }
            __syncwarp();
            const uint4 *src = reinterpret_cast<const uint4 *>(r);
            uint4 *dst = reinterpret_cast<uint4 *>(blocks + 32 * c * kBlockBytes);
            for (int i = lane; i < 32 * kBlockBytes / 16; i += 32) dst[i] = src[i];
            __syncwarp();
        } else if (g < nblocks) {
            uint16_t *h = reinterpret_cast<uint16_t *>(blocks + g * kBlockBytes);
            h[0] = d;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                h[1 + 2 * i] = static_cast<uint16_t>(w[i] & 0xFFFFu);
                h[2 + 2 * i] = static_cast<uint16_t>(w[i] >> 16);
            }
        }
    }
}

int grid_for(int64_t nblocks, const DeviceInfo *di) {
    const int64_t want = (nblocks + kThreads - 1) / kThreads;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(di->sm_count) * 8)));
}

}  // namespace

q8_status launch_gguf_ingest(const void *blocks, int64_t nblocks, int8_t *q, uint16_t *s, cudaStream_t stream) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (nblocks == 0) return Q8_OK;
    gguf_ingest_kernel<<<grid_for(nblocks, di), kThreads, 0, stream>>>(static_cast<const uint8_t *>(blocks), nblocks,
                                                                       q, s);
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

q8_status launch_gguf_export(const int8_t *q, const uint16_t *s, int64_t nblocks, void *blocks, cudaStream_t stream) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (nblocks == 0) return Q8_OK;
    const int64_t nruns = (nblocks + 31) / 32;
    const int grid = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>((nruns + kThreads / 32 - 1) / (kThreads / 32), static_cast<int64_t>(di->sm_count) * 8)));
    gguf_export_kernel<<<grid, kThreads, 0, stream>>>(q, s, nblocks, static_cast<uint8_t *>(blocks));
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

}  // namespace q8
