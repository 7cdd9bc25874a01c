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
// Both directions move whole runs of 32 blocks (1088 bytes, a multiple of 16)
// between global memory and a per-warp copy in shared memory with 16-byte
// accesses; each lane handles one block of the run at 2-byte granularity.
#include <algorithm>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kThreads = 256;
constexpr int64_t kBlockBytes = 34;

// Ingest: a warp takes 32 consecutive blocks (1088 bytes, 16-byte aligned),
// loads the run with 16-byte loads into shared memory and each lane takes
// its block out of it (scale and eight code words, 2-byte aligned), then
// stores the codes as two 16-byte words.  A last run of fewer than 32 blocks
// goes lane by lane with 2-byte loads.
__global__ void __launch_bounds__(kThreads) gguf_ingest_kernel(const uint8_t *__restrict__ blocks, int64_t nblocks,
                                                               int8_t *__restrict__ q, uint16_t *__restrict__ s) {
    __shared__ __align__(16) uint16_t run[kThreads / 32][32 * kBlockBytes / 2];
    const int lane = threadIdx.x & 31;
    uint16_t *r = run[threadIdx.x >> 5];
    const int64_t nruns = (nblocks + 31) / 32;
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5); c < nruns;
         c += wstride) {
        const int64_t g = 32 * c + lane;
        uint32_t d = 0, w[8];
        if (32 * c + 32 <= nblocks) {
            const uint4 *src = reinterpret_cast<const uint4 *>(blocks + 32 * c * kBlockBytes);
            uint4 *dst = reinterpret_cast<uint4 *>(r);
            for (int i = lane; i < 32 * kBlockBytes / 16; i += 32) dst[i] = __ldg(src + i);
            __syncwarp();
            const uint16_t *h = r + lane * (kBlockBytes / 2);
            d = h[0];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                w[i] = static_cast<uint32_t>(h[1 + 2 * i]) | (static_cast<uint32_t>(h[2 + 2 * i]) << 16);
            __syncwarp();
        } else if (g < nblocks) {
            const uint16_t *h = reinterpret_cast<const uint16_t *>(blocks + g * kBlockBytes);
            d = __ldg(h);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                w[i] = static_cast<uint32_t>(__ldg(h + 1 + 2 * i)) | (static_cast<uint32_t>(__ldg(h + 2 + 2 * i)) << 16);
        }
        if (g < nblocks) {
            uint4 *qo = reinterpret_cast<uint4 *>(q + 32 * g);
            qo[0] = make_uint4(w[0], w[1], w[2], w[3]);
            qo[1] = make_uint4(w[4], w[5], w[6], w[7]);
            s[g] = static_cast<uint16_t>(d);
        }
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

// One warp per run of 32 blocks, up to 8 CTAs per SM.
int grid_for(int64_t nblocks, const DeviceInfo *di) {
    const int64_t nruns = (nblocks + 31) / 32;
    return static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>((nruns + kThreads / 32 - 1) / (kThreads / 32), static_cast<int64_t>(di->sm_count) * 8)));
}

}  // namespace

q8_status launch_gguf_ingest(const void *blocks, int64_t nblocks, int8_t *q, uint16_t *s, cudaStream_t stream) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (nblocks == 0) return Q8_OK;
    gguf_ingest_kernel<<<grid_for(nblocks, di), kThreads, 0, stream>>>(static_cast<const uint8_t *>(blocks), nblocks, q, s);
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

q8_status launch_gguf_export(const int8_t *q, const uint16_t *s, int64_t nblocks, void *blocks, cudaStream_t stream) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (nblocks == 0) return Q8_OK;
    gguf_export_kernel<<<grid_for(nblocks, di), kThreads, 0, stream>>>(q, s, nblocks, static_cast<uint8_t *>(blocks));
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

}  // namespace q8
