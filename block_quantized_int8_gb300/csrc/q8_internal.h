// q8_internal.h -- host-side declarations shared by the libq8 translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "q8.h"

namespace q8 {

struct DeviceInfo {
    int device;
    int sm_count;
    int cc_major;
    int cc_minor;
};

// Cached properties of the current device; nullptr if a CUDA call failed.
const DeviceInfo *device_info();
// The current device's properties, if it is compute capability 10.3:
// Q8_ERR_CUDA if they cannot be read, Q8_ERR_ARCH for another device.
q8_status check_arch(const DeviceInfo **out);

// ---- quantizer --------------------------------------------------------------
// mode: Q8_QUANT_EXACT (codes from the stored scale) or Q8_QUANT_FL32.
q8_status launch_quantize(const float *w, int64_t rows, int64_t K, int8_t *q, uint16_t *s,
                          uint32_t *dev_status, cudaStream_t stream, int mode = Q8_QUANT_EXACT);

// ---- skinny matmul (M <= 32) -------------------------------------------------
constexpr int kSkinnyWarps = 8;
constexpr int kSkinnyThreads = kSkinnyWarps * 32;
constexpr int kTileRows = kSkinnyWarps * 16;  // rows of W per work item

// Blocks of K held in one x staging buffer, by M class.
inline int ksb_for_m(int M) { return M <= 8 ? 64 : (M <= 16 ? 32 : 16); }

// Per-matrix split of K and the offsets of its partial sums in the workspace.
struct SplitPlan {
    int32_t tiles;      // ceil(N / kTileRows)
    int32_t S;          // K splits
    int32_t bps;        // blocks per split
    size_t part_off;    // byte offset of float partials [S][M][N] (if S > 1)
    size_t ticket_off;  // byte offset of uint32 tickets [tiles] (if S > 1)
};

// Plans every descriptor and returns the workspace bytes needed.
// invariant: the split depends on K alone (the batch-invariant variant).
size_t plan_skinny(const q8_linear_desc *descs, int count, int M, SplitPlan *plans, bool invariant = false);

// Workspace of a skinny call: the general kernel's plan of every matrix, then
// (when some matrix is served by the GEMV) a 256-byte block whose first word
// is the GEMV's pool counter, at *sched_off (SIZE_MAX if none), then (when
// some matrix is served by the tile kernel) the tile kernel's workspace
// (tile_workspace of those matrices) at *tile_off (SIZE_MAX if none).
// The workspace of the W8A8 variant (tile kernel for K % 256 == 0, general
// kernel otherwise); gen_x_off / gen_plan_off: where the general kernel's
// quantized activations and split partials start.
size_t w8a8_workspace(const q8_linear_desc *all, int all_count, int M, size_t *gen_x_off = nullptr,
                      size_t *gen_plan_off = nullptr);
size_t skinny_workspace(const q8_linear_desc *descs, int count, int M, SplitPlan *plans, size_t *sched_off,
                        size_t *tile_off = nullptr);

// Dependent matmul chains (q8_chain.cu): the host check of a chain, its
// workspace (the largest of its steps') and its launches.
q8_status check_chain(const q8_chain_step *steps, int count, int M);
size_t chain_workspace(const q8_chain_step *steps, int count, int M);
q8_status launch_chain(const q8_chain_step *steps, int count, int M, void *ws, size_t ws_bytes,
                       uint32_t *dev_status, cudaStream_t stream);

// M = 1 bulk-copy pipeline (q8_gemv.cu): matrices with K <= 12288.
bool gemv_k_supported(int64_t K);
// sched: a zeroed device word the launch uses as its pool counter and leaves
// zero again (null: every CTA keeps its whole static range).
// chained: launched as a programmatic dependent of the previous kernel in the
// stream; the first weight stages are read before that kernel completes,
// x, y and the counter only after.
q8_status launch_gemv(const q8_linear_desc *descs, int count, uint32_t *sched, uint32_t *dev_status,
                      cudaStream_t stream, bool chained = false);

// 1 <= M <= 8 bulk-copy pipeline with warp MMA (q8_pipe.cu): K <= 4096.
bool pipe_k_supported(int64_t K);
q8_status launch_pipe(const q8_linear_desc *descs, int count, int M, uint32_t *dev_status, cudaStream_t stream,
                      bool chained = false);

// 2 <= M <= 32 chunked tile kernel (q8_tile.cu).  The default arithmetic
// takes any K >= 256 (a multiple of 32: the last chunk of 256 may be
// partial); the batch-invariant and W8A8 modes take whole chunks only.
bool tile_k_supported(int64_t K);
bool tile_k_whole_chunks(int64_t K);
// workspace bytes of the tile kernel for these matrices: each one's x copy
// and per-chunk flags (M <= 16), in call order, then the tickets and
// partials of the row blocks that CTAs share; the tickets (zero between
// launches) are [*ticket_off, *ticket_off + *ticket_bytes)
size_t tile_workspace(const q8_linear_desc *descs, int count, int M, size_t *ticket_off = nullptr,
                      size_t *ticket_bytes = nullptr, bool w8a8 = false);
// mode 0: the default arithmetic; 1: batch-invariant (bf16 operands, one
// class, no x copy, any 1 <= M <= 32, no workspace); 2: W8A8 (x quantized
// to Q8_0 in the workspace, int8 block dots, any 1 <= M <= 32)
q8_status launch_tile(const q8_linear_desc *descs, int count, int M, uint8_t *xws, uint32_t *dev_status,
                      cudaStream_t stream, bool chained = false, int mode = 0);

// GGUF Q8_0 block repack (q8_gguf.cu): nblocks blocks of 34 bytes (binary16
// scale, 32 int8 codes) <-> planar codes (32 bytes per block) and scales.
q8_status launch_gguf_ingest(const void *blocks, int64_t nblocks, int8_t *q, uint16_t *s, cudaStream_t stream);
q8_status launch_gguf_export(const int8_t *q, const uint16_t *s, int64_t nblocks, void *blocks, cudaStream_t stream);

// Streaming-read ceiling (q8_probe.cu): reads bytes (a multiple of 16) from a
// 16-byte aligned buffer; each CTA XORs what it read into out[blockIdx.x]
// (out holds stream_read_grid() words).
int stream_read_grid(const DeviceInfo *di);
q8_status launch_stream_read(const void *src, size_t bytes, uint32_t *out, cudaStream_t stream);

// Bounded wait on an mbarrier nothing arrives on (q8_selftest.cu).
q8_status launch_selftest_wait_timeout(uint64_t limit_ns, uint32_t *status, uint64_t *elapsed_ns,
                                       cudaStream_t stream);

// 2-D TMA tensor map over a row-major [outer][inner] array of 1- or 2-byte
// elements (q8_tmap.cu; cached by parameters).  false if encoding fails.
bool encode_2d(CUtensorMap *map, int elem_bytes, const void *base, uint64_t inner, uint64_t outer,
               uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128);
// Rank-2 or rank-3 map: dims[0] innermost, stride_bytes[i] the byte stride of
// dims[i + 1], box[] the box extent per dimension.
bool encode_tmap(CUtensorMap *map, int elem_bytes, const void *base, int rank, const uint64_t *dims,
                 const uint64_t *stride_bytes, const uint32_t *box, bool swizzle128);

// kernel<<<grid, block, smem, stream>>>(p); chained: launched as a
// programmatic dependent of the previous kernel in the stream (it may start
// as that kernel's CTAs exit; it must wait with griddepcontrol.wait before
// reading anything that kernel may write).
template <typename P>
inline cudaError_t launch_kernel(void (*kernel)(P), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 bool chained, const P &p) {
    if (!chained) {
        kernel<<<grid, block, smem, stream>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

q8_status launch_skinny(const q8_linear_desc *descs, int count, int M, int variant,
                        void *ws, size_t ws_bytes, uint32_t *dev_status, cudaStream_t stream,
                        bool chained = false);

// Host-only argument check of one skinny matmul, as q8_gemm_skinny does it.
q8_status check_skinny_args(const q8_linear_desc &d, int32_t M);

// ---- prefill GEMM (M > 32) ----------------------------------------------------
q8_status launch_gemm_tc(const int8_t *q, const uint16_t *s, int64_t N, int64_t K,
                         const uint16_t *x, int64_t ldx, int32_t M, uint16_t *y, int64_t ldy, int32_t tile,
                         int32_t splits, uint32_t *dev_status, cudaStream_t stream);

}  // namespace q8
