// q8_noalloc.cu -- q8_gemm_skinny for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the matmul:
// code running under an allocator that forbids new device allocations (a
// memory pool fixed at start-up, a real-time loop that must not block in the
// driver), or plugin hosts that hand over only input and output buffers.  For
// them this file provides q8_gemm_skinny_noalloc: the same computation as
// q8_gemm_skinny, with the split-K scratch (tickets and partial sums) taken
// from one file-scope device array instead of a caller workspace.
//
// The array is part of the library image: every GPU that loads libq8 holds
// kNoAllocScratchBytes of it until the process exits.  All calls on a device
// share it, so calls whose kernels overlap on the GPU (different streams
// without ordering) race on it; calls ordered on one stream are fine.  The
// array keeps the last call's contents; each call clears the ticket words it
// needs before its kernel runs (partial sums are always written before they
// are read).
#include <mutex>

#include "q8_internal.h"

namespace q8 {

namespace {

constexpr size_t kNoAllocScratchBytes = Q8_NOALLOC_SCRATCH_BYTES;  // 4 MiB

// Device-side scratch.  In host code this name is only a stand-in for the
// device symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices];

// Device address of the scratch on device `dev`, which must be current.  The
// first successful lookup on a device is kept for later calls; a failed one
// (for example one made during a stream capture) is not kept, so the next
// call tries again.  The lookup may load the library's device code, which is
// why the first call on a device belongs outside any stream capture.
void *scratch_address(int dev) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) == cudaSuccess) g_addr[dev] = p;
    }
    return g_addr[dev];
}

}  // namespace

}  // namespace q8

using namespace q8;

extern "C" q8_status q8_gemm_skinny_noalloc(const int8_t *q, const uint16_t *s, int64_t N, int64_t K,
                                            const uint16_t *x, int64_t ldx, int32_t M, float *y, int64_t ldy,
                                            uint32_t *dev_status, q8_stream_t stream) {
    // same argument rules as q8_gemm_skinny, plus the scratch limit, all
    // checked on the host before any CUDA call
    q8_linear_desc d{};
    d.q = q;
    d.s = s;
    d.x = x;
    d.y = y;
    d.N = N;
    d.K = K;
    d.ldx = ldx;
    d.ldy = ldy;
    q8_status st = check_skinny_args(d, M);
    if (st != Q8_OK) return st;
    if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3u)) return Q8_ERR_ALIGN;
    if (N == 0 || M == 0) return Q8_OK;
    const size_t need = q8_workspace_size(N, K, M);
    if (need > kNoAllocScratchBytes) return Q8_ERR_WORKSPACE;

    // the device check comes before anything is queued: a call that fails
    // it enqueues nothing
    const DeviceInfo *di = nullptr;
    st = check_arch(&di);
    if (st != Q8_OK) return st;
    if (di->device < 0 || di->device >= kMaxDevices) return Q8_ERR_CUDA;
    void *ws = scratch_address(di->device);
    if (ws == nullptr) return Q8_ERR_CUDA;

    if (need > 0) {
        // clear the words the kernels count with: the ticket words (first in
        // the layout), the GEMV's pool counter block and the tile kernel's
        // tickets of shared row blocks
        SplitPlan pl;
        size_t sched_off, tile_off;
        (void)skinny_workspace(&d, 1, M, &pl, &sched_off, &tile_off);
        if (tile_off != SIZE_MAX) {
            size_t toff = 0, tbytes = 0;
            (void)tile_workspace(&d, 1, M, &toff, &tbytes);
            if (tbytes > 0 && cudaMemsetAsync(static_cast<unsigned char *>(ws) + tile_off + toff, 0, tbytes,
                                              reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
                return Q8_ERR_CUDA;
        }
        const size_t ticket_bytes = pl.part_off - pl.ticket_off;
        if (ticket_bytes > 0 &&
            cudaMemsetAsync(static_cast<unsigned char *>(ws) + pl.ticket_off, 0, ticket_bytes,
                            reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
            return Q8_ERR_CUDA;
        if (sched_off != SIZE_MAX &&
            cudaMemsetAsync(static_cast<unsigned char *>(ws) + sched_off, 0, 256,
                            reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
            return Q8_ERR_CUDA;
    }
    return q8_gemm_skinny(q, s, N, K, x, ldx, M, y, ldy, ws, kNoAllocScratchBytes, dev_status, stream);
}
