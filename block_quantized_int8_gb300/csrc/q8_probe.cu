// q8_probe.cu -- the streaming-read ceiling the decode kernels are compared
// with: "Frigg" README, "The machine" measures a device-to-device copy, a
// fused read and the GEMV side by side; this is the read.  Each thread keeps
// four 16-byte non-allocating loads in flight, folds what it read into one
// word (so the loads cannot be dropped) and each CTA writes one word.
#include <algorithm>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeUnroll = 4;

__global__ void __launch_bounds__(kProbeThreads) stream_read_kernel(const uint4 *__restrict__ src, int64_t n16,
                                                                    uint32_t *__restrict__ out) {
    uint32_t acc = 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kProbeThreads * kProbeUnroll;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * kProbeThreads * kProbeUnroll + threadIdx.x; base < n16;
         base += stride) {
        uint4 v[kProbeUnroll];
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) {
            const int64_t i = base + static_cast<int64_t>(u) * kProbeThreads;
            if (i < n16) {
                asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                             : "l"(src + i));
            } else {
                v[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    acc = __reduce_xor_sync(0xffffffffu, acc);
    if ((threadIdx.x & 31) == 0) atomicXor(out + blockIdx.x, acc);
}

}  // namespace

int stream_read_grid(const DeviceInfo *di) { return di->sm_count * 8; }

q8_status launch_stream_read(const void *src, size_t bytes, uint32_t *out, cudaStream_t stream) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    const int64_t n16 = static_cast<int64_t>(bytes / 16);
    if (n16 == 0) return Q8_OK;
    const int64_t want = (n16 + kProbeThreads * kProbeUnroll - 1) / (kProbeThreads * kProbeUnroll);
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, stream_read_grid(di))));
    stream_read_kernel<<<grid, kProbeThreads, 0, stream>>>(static_cast<const uint4 *>(src), n16, out);
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

}  // namespace q8
