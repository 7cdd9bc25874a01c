/*
 * q8.h -- C ABI of libq8: the Q8_0 W8A16 decode matmul on GB300 (sm_103a).
 *
 * Format (from "MODEL-BASELINE-RESULTS" (fak), ACT 3 item 1 and ACT 4
 * "Correctness"): a weight matrix W[N][K] is cut along K into blocks of 32.
 * Each block stores one scale d = maxabs/127, kept as IEEE binary16 (the page's
 * ~1.06 bytes per weight is 32 one-byte codes plus a two-byte scale), and 32
 * int8 codes q = round-half-away-from-zero(w/d), so that w ~= d*q.  The
 * matmul is W8A16 ("Frigg" README, Finding 8): int8 weights times bf16
 * activations, each weight read from memory once per call, fp32 accumulation.
 *
 * Storage is planar and row-major:
 *   codes   int8      q[N][K]        (row n at q + n*K)
 *   scales  binary16  s[N][K/32]     (raw bits in uint16_t)
 *   x       bfloat16  x[M][ldx]      (raw bits in uint16_t)
 *   y       float     y[M][ldy]      (bf16 bits for q8_gemm)
 * so that y[m][n] = sum_k s[n][k/32] * q[n][k] * x[m][k].
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or synchronises; work is enqueued on `stream`
 *    (NULL = the legacy default stream) and may still be running on return.
 *  - Arguments are checked on the host before any CUDA call; a failed check
 *    returns an error status and enqueues nothing.  Launch failures return
 *    Q8_ERR_CUDA (the CUDA error is left for cudaGetLastError()).
 *  - `dev_status` (nullable) is a device word the kernels OR bits into
 *    (Q8_DEV_*) when they meet bad data or give up waiting; read it after
 *    your own synchronisation.  The kernels never trap.
 *  - Alignment: q, s and x must be 16-byte aligned, ldx a multiple of 8;
 *    y must be 4-byte aligned (2-byte for bf16 output).  K must be a
 *    positive multiple of 32.  N == 0 or M == 0 is a no-op.
 *  - Results are bitwise reproducible from run to run and under CUDA-graph
 *    replay for the same arguments (split-K partial sums are combined in a
 *    fixed order, never with floating-point atomics).
 */
#ifndef Q8_H_
#define Q8_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *q8_stream_t;

typedef enum q8_status {
    Q8_OK = 0,
    Q8_ERR_ARG = 1,        /* null pointer or bad count */
    Q8_ERR_ALIGN = 2,      /* pointer or leading dimension misaligned */
    Q8_ERR_SHAPE = 3,      /* K not a positive multiple of 32, M out of range, ld too small */
    Q8_ERR_WORKSPACE = 4,  /* workspace missing or smaller than the *_workspace_size() result */
    Q8_ERR_ARCH = 5,       /* current device is not compute capability 10.3 */
    Q8_ERR_CUDA = 6,       /* a CUDA runtime call failed */
    Q8_ERR_UNSUPPORTED = 7 /* valid request this build does not implement */
} q8_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define Q8_DEV_NONFINITE 0x1u /* quantizer: a block held NaN/Inf; stored as zero codes, zero scale */
#define Q8_DEV_SCALE_OVF 0x2u /* quantizer: amax/127 overflowed binary16; block stored as zeros */
#define Q8_DEV_TIMEOUT   0x4u /* a bounded wait gave up; outputs of that call are not valid */

#define Q8_BLOCK 32          /* weights per block along K */
#define Q8_SKINNY_MAX_M 32   /* largest M for q8_gemv / q8_gemm_skinny / q8_linear_batch */
#define Q8_MAX_BATCH 64      /* most descriptors per q8_linear_batch call */

/* Kernel variants for the M <= 32 path (the _ex entry points). */
#define Q8_VARIANT_AUTO 0    /* M = 1: CUDA-core GEMV; M = 2..8: the warp-MMA pipeline (K = 1536, and K % 256 != 0 up to 4096), else TMA-fed warp-MMA tiles; M > 8: the tiles (K >= 256; smaller K the general kernel) */
#define Q8_VARIANT_SIMT 1    /* CUDA-core FFMA: codes dequantised in registers, one FMA per weight per row */
#define Q8_VARIANT_MMA  2    /* warp mma.sync bf16 on exact bf16 codes, block scale applied in fp32 */
/* Batch-invariant: row m of Y is the same, bit for bit, for every M in
 * 1..32 that includes that row (a decode row equals the same row computed
 * in a batch).  Source: "Frigg" README, Finding 4 (a matmul over one row
 * is not bit-identical to the same matmul over a batch holding it, so a
 * decode row could not be compared with a batch row).  Every row takes the
 * same arithmetic whatever M is: bf16 operands, exact products, per-block
 * fp32 results times the block scale added in block order, one sum per row
 * over all of K (a warp MMA computes each output from its own row only) --
 * in the TMA-fed tile kernel for K % 256 == 0 (no workspace), in the
 * general kernel for other K (any multiple of 32), with K split into
 * ceil(K / 512) ranges -- a split from K alone -- whose partial sums are
 * added in range order (workspace: q8_linear_batch_workspace_size_ex).
 * Slower than AUTO where AUTO splits K or uses binary16 operands. */
#define Q8_VARIANT_BATCH_INVARIANT 3
/* W8A8: each activation row is quantized to Q8_0 by the weights' rule (the
 * A1 quantizer of its binary32 values), then y = sum over blocks of
 * s_w * s_x * (exact int8 block dot), one warp int8 MMA per block and 8
 * rows.  Source: "MODEL-BASELINE-RESULTS" (fak), ACT 3 items 1 and 3
 * (weights and activations in Q8_0 blocks, integer block dots).  Accuracy
 * against the W8A8 definition as for the other variants (2e-3 * sum |w' x'|
 * + 1e-6, x' the dequantised activations); against the bf16 activations it
 * adds the activations' quantization error.  Any K (a multiple of 32):
 * K % 256 == 0 runs in the tile kernel, other K in the general kernel (x
 * quantized to rows of Q8_0 codes and scales, the same block dot and
 * scaling); workspace: q8_linear_batch_workspace_size_ex(..., Q8_VARIANT_W8A8)
 * bytes (per distinct x its binary32 copy, codes and scales, plus the
 * kernels' split-K areas). */
#define Q8_VARIANT_W8A8 4

/*
 * q8_quantize_rows -- Q8_0-quantize binary32 weights w[rows][K] along K.
 * Source: "MODEL-BASELINE-RESULTS" (fak), ACT 3 item 1 (blocks of 32,
 * d = maxabs/127), ACT 4 "Correctness" (round half away from zero; 0.49999997
 * gives 0), ACT 5 item 3 (exact on zeros, denormals, exact halves).
 * Per block: amax = max|w| (binary32), d = amax/127 (binary32, round to
 * nearest even), s = binary16(d) (nearest even, subnormals kept), then
 * q = clamp(round-half-away(w/s), -127, 127) with the quotient taken exactly
 * against the stored s; s == 0 gives q = 0.  A block holding NaN/Inf, or whose
 * s overflows, is stored as zeros and sets Q8_DEV_NONFINITE / Q8_DEV_SCALE_OVF.
 *   w  : float [rows][K], 16-byte aligned     (in)
 *   q  : int8  [rows][K], 16-byte aligned     (out)
 *   s  : binary16 bits [rows][K/32], 16-byte aligned (out)
 * The result is bit-identical to the definition above (no tolerance).
 */
q8_status q8_quantize_rows(const float *w, int64_t rows, int64_t K,
                           int8_t *q, uint16_t *s,
                           uint32_t *dev_status, q8_stream_t stream);

/*
 * q8_stream_read -- the streaming-read ceiling the decode kernels are
 * measured against ("Frigg" README, "The machine": copy, read and GEMV
 * bandwidth side by side).  Reads `bytes` (a multiple of 16) from the
 * 16-byte aligned device buffer `src` with 16-byte non-allocating loads and
 * XORs what it read into out[0 .. q8_stream_read_out_words()) (device
 * words, zeroed by the caller, one per CTA), so the loads are not elided.
 */
q8_status q8_stream_read(const void *src, size_t bytes, uint32_t *out, q8_stream_t stream);
size_t q8_stream_read_out_words(void);

/*
 * q8_selftest_wait_timeout -- exercise the kernels' failure path without a
 * fault: one thread waits, with the same bounded mbarrier wait the kernels
 * use, on a barrier that nothing ever arrives on, gives up after limit_ns
 * (1 .. 1e9), ORs Q8_DEV_TIMEOUT into *dev_status and writes the time it
 * waited (ns) to *dev_elapsed_ns (both device pointers, nullable).  The
 * context stays usable.  Q8_ERR_ARG for a limit out of range.
 */
q8_status q8_selftest_wait_timeout(uint64_t limit_ns, uint32_t *dev_status, uint64_t *dev_elapsed_ns,
                                   q8_stream_t stream);

/* Code rules of q8_quantize_rows_ex. */
#define Q8_QUANT_EXACT 0  /* as q8_quantize_rows: exact quotient by the stored binary16 scale */
#define Q8_QUANT_FL32 1   /* compatibility: binary32 quotient w / d (d = amax/127 in binary32) */

/*
 * q8_quantize_rows_ex -- q8_quantize_rows with a choice of code rule.
 * Q8_QUANT_FL32 rounds (half away from zero, clamp +-127) the binary32
 * quotient w / d, IEEE division by the binary32 scale d = amax/127 before its
 * rounding to the stored binary16 s -- the float32 value that
 * "MODEL-BASELINE-RESULTS" (fak), ACT 4 "Correctness", rounds with q8round.
 * Scales, flags and the zero-scale rule are those of Q8_QUANT_EXACT; codes
 * can differ by one where s != d.  Bit-identical to that definition.
 * An unknown mode returns Q8_ERR_ARG.
 */
q8_status q8_quantize_rows_ex(const float *w, int64_t rows, int64_t K,
                              int8_t *q, uint16_t *s, int32_t mode,
                              uint32_t *dev_status, q8_stream_t stream);

/*
 * q8_gguf_to_planar -- repack a GGUF Q8_0 tensor into this library's layout.
 * Source: the GGUF model files of the "aubier" README ("Layout": the engine's
 * GGUF loader) and the serverAppConfigs log; the block is the Q8_0 block of
 * "MODEL-BASELINE-RESULTS" (fak), ACT 3 item 1.
 *   blocks : rows * K/32 blocks of 34 bytes, consecutive (a [rows][K] tensor
 *            in GGUF order): binary16 scale d, then 32 int8 codes;
 *            16-byte aligned                                       (in)
 *   q      : int8 [rows][K], 16-byte aligned                       (out)
 *   s      : binary16 bits [rows][K/32], 16-byte aligned           (out)
 * Block g (row g / (K/32), block g % (K/32)) becomes q[32g .. 32g+32) and
 * s[g], bit for bit.  K must be a positive multiple of 32.
 */
q8_status q8_gguf_to_planar(const void *blocks, int64_t rows, int64_t K,
                            int8_t *q, uint16_t *s, q8_stream_t stream);

/* q8_planar_to_gguf -- the inverse of q8_gguf_to_planar (same alignment). */
q8_status q8_planar_to_gguf(const int8_t *q, const uint16_t *s, int64_t rows, int64_t K,
                            void *blocks, q8_stream_t stream);

/*
 * q8_gemv -- y[n] = sum_k s[n][k/32]*q[n][k]*x[k] for one activation row (M = 1).
 * Source: "Frigg" README, "The machine" (at batch 1 every decode GEMM is this
 * GEMV shape) and Finding 8 (W8A16: read each weight once).
 *   q, s : Q8_0 weights [N][K], [N][K/32]      (in)
 *   x    : bf16 bits [K]                        (in)
 *   y    : float [N]                            (out)
 *   ws   : workspace of q8_workspace_size(N, K, 1) bytes (may be NULL if that
 *          is 0).  Zero it once after allocation; the kernels leave it zeroed
 *          again, so it can be reused across calls and graph replays, but not
 *          by two calls that run at the same time.
 * Accuracy: |y - y_ref| <= 2e-3 * sum_k |s*q*x| + 1e-6 per output, where y_ref
 * is the exact dequantise-then-dot value.
 */
q8_status q8_gemv(const int8_t *q, const uint16_t *s, int64_t N, int64_t K,
                  const uint16_t *x, float *y,
                  void *ws, size_t ws_bytes,
                  uint32_t *dev_status, q8_stream_t stream);

/*
 * q8_gemm_skinny -- Y[M][N] = X[M][K] * W^T for 1 <= M <= 32 decode rows.
 * Source: "Frigg" README, Finding 8 (a batched W8A16 kernel reads each weight
 * matrix once for the whole batch; split-K through a partials buffer rather
 * than atomics so that replays are bit-identical).
 *   x : bf16 bits [M][ldx], ldx >= K and a multiple of 8   (in)
 *   y : float [M][ldy], ldy >= N                            (out)
 *   ws: q8_workspace_size(N, K, M) bytes, zeroed once (see q8_gemv).
 * Accuracy as q8_gemv.
 */
q8_status q8_gemm_skinny(const int8_t *q, const uint16_t *s, int64_t N, int64_t K,
                         const uint16_t *x, int64_t ldx, int32_t M,
                         float *y, int64_t ldy,
                         void *ws, size_t ws_bytes,
                         uint32_t *dev_status, q8_stream_t stream);

/* One matrix of a q8_linear_batch call: y = x * W^T with W = (q, s). */
typedef struct q8_linear_desc {
    const int8_t *q;     /* int8 [N][K] */
    const uint16_t *s;   /* binary16 bits [N][K/32] */
    const uint16_t *x;   /* bf16 bits [M][ldx] */
    float *y;            /* float [M][ldy] */
    int64_t N, K, ldx, ldy;
} q8_linear_desc;

/*
 * q8_linear_batch -- several independent skinny matmuls (same M, any shapes)
 * in one persistent launch per kernel family that walks a static list of
 * (matrix, row tile, K split) work items; each matrix is routed on its own K
 * and M, so a call whose matrices all share a family is one launch.  Source: "Frigg" README, Finding 3 and Finding 8 (a
 * decode step of many small matmuls is launch-bound before it is
 * bandwidth-bound).
 *   descs : HOST array of `count` descriptors, 1 <= count <= Q8_MAX_BATCH;
 *           copied into the launch, may be reused on return.
 *   ws    : q8_linear_batch_workspace_size(descs, count, M) bytes, zeroed once.
 *           At M = 1 it ends with a 256-byte block whose first word the GEMV
 *           uses as a work counter (it hands its last stages to whichever CTA
 *           is free first) and leaves zero; after a Q8_DEV_TIMEOUT zero the
 *           workspace again.  One workspace may serve later calls of other
 *           shapes (at the same address, in stream order): where the words
 *           a call counts with may hold an earlier call's partial sums or x
 *           copies (or on the first use of an address), the library clears
 *           them first with one cudaMemsetAsync per range in the call's
 *           stream; M = 1 calls and repeated calls of the same shapes clear
 *           nothing.
 * Each output equals, bit for bit, what q8_gemm_skinny returns for that matrix.
 * Outputs must not overlap each other or any input.
 */
q8_status q8_linear_batch(const q8_linear_desc *descs, int32_t count, int32_t M,
                          void *ws, size_t ws_bytes,
                          uint32_t *dev_status, q8_stream_t stream);

/*
 * q8_linear_batch_chained -- as q8_linear_batch, for a stream of calls whose
 * weights no earlier work in the stream writes (a decode loop over fixed
 * model weights).  The launch may start while the previous kernel in the
 * stream is finishing (programmatic dependent launch): it reads the first
 * stages of weights (q, s) before that kernel completes, and x, y and ws only
 * after it has completed and its writes are visible.  So the previous work
 * may produce x, but must not write any q or s of this call.  Same results,
 * bit for bit, as q8_linear_batch.  Every kernel family of the call is
 * launched this way; the bulk-copy kernels (M <= 8 GEMV and pipeline) and the
 * TMA tile kernel issue their first weight stages before the wait, the
 * general kernel waits first.
 */
q8_status q8_linear_batch_chained(const q8_linear_desc *descs, int32_t count, int32_t M,
                                  void *ws, size_t ws_bytes,
                                  uint32_t *dev_status, q8_stream_t stream);

/* As q8_linear_batch / q8_gemm_skinny with an explicit kernel variant
 * (Q8_VARIANT_*), for side-by-side measurement.  Variants agree within the
 * accuracy bound, not bit for bit. */
q8_status q8_linear_batch_ex(const q8_linear_desc *descs, int32_t count, int32_t M,
                             int32_t variant, void *ws, size_t ws_bytes,
                             uint32_t *dev_status, q8_stream_t stream);

/* Workspace bytes for the calls above; depends only on the shapes, not on
 * the device.  0 means none is needed.  It holds the split-K partial sums and
 * tickets, at M = 1 the GEMV's counter block, and for every matrix that the
 * tile kernel serves with binary16 operands (9 <= M <= 16 with K >= 256, or
 * 2 <= M <= 8 with K % 256 == 0 and K != 1536 or K > 4096) a copy of its x,
 * M * Kp * 2 bytes rounded up to 256 (Kp = K rounded up to a multiple of
 * 256; zero past K), plus a 256-byte-rounded flag word per 256 columns of
 * Kp: each 256-column chunk of x (all M rows) is copied as binary16 where
 * binary16 holds all its values exactly, else as bf16, and the matmul
 * takes the matching operand type.
 * After the copies come, for M <= 16, the tickets (one 32-byte group each,
 * 256-byte rounded) and fp32 partials (16 KB x ceil(M / 8) each) of up to
 * min(320, total 128-row blocks of those matrices) row blocks whose work is
 * shared between CTAs.  The copies and partials need no zeroing; the words
 * the kernels count with are left zero. */
size_t q8_workspace_size(int64_t N, int64_t K, int32_t M);
size_t q8_linear_batch_workspace_size(const q8_linear_desc *descs, int32_t count, int32_t M);
/* The workspace of q8_linear_batch_ex with `variant` (the W8A8 variant needs
 * its own; the batch-invariant one the general kernel's partial sums of its
 * matrices with K % 256 != 0, none if there are none; the others as above). */
size_t q8_linear_batch_workspace_size_ex(const q8_linear_desc *descs, int32_t count, int32_t M, int32_t variant);

/*
 * q8_linear_chain -- a chain of dependent skinny matmuls, each step's input
 * made on the device from the output of the step before it.  Source:
 * "Frigg" README, the model card (RMSNorm without learnable weights, eps
 * 1e-6; a SwiGLU MLP; two 16-layer modules run L L L H L L L H per token)
 * and Finding 3 (a decode step is a long chain of small dependent launches,
 * launch-bound before it is bandwidth-bound).
 *   Step i computes y_i[M][N_i] = x_i[M][K_i] * dequant(q_i, s_i)^T (fp32,
 *   as q8_linear_batch, routed on its own K and M with the automatic
 *   variant), then, unless it is the last step, writes the next step's
 *   input x_{i+1}[M][K_{i+1}] (bf16, round to nearest even) from y_i:
 *     Q8_CHAIN_RMSNORM:        v = y_i[m][0 .. K_{i+1})  (needs N_i >= K_{i+1})
 *     Q8_CHAIN_SWIGLU_RMSNORM: v[k] = silu(y_i[m][k]) * y_i[m][K_{i+1} + k],
 *                              silu(a) = a / (1 + e^-a)  (needs N_i >= 2 K_{i+1})
 *   and x_{i+1}[m][k] = v[k] / sqrt(mean over k of v[k]^2 + 1e-6), in fp32
 *   (the sum of squares in a fixed order).  The last step has Q8_CHAIN_END.
 *   Every kernel of the chain is launched as a programmatic dependent of the
 *   one before it (as q8_linear_batch_chained): a matmul loads its first
 *   weight stages before the normalisation ahead of it completes, so no
 *   work earlier in the stream may write any q or s of the chain.
 *   steps : HOST array of `count` steps, 1 <= count <= Q8_MAX_CHAIN, checked
 *           on the host before anything is enqueued.  Step 0's x is the
 *           caller's; every later x is written by the chain.  x and y follow
 *           q8_linear_desc's alignment rules; no x or y may overlap a q, s
 *           or another step's x or y that the chain still reads.
 *   ws    : DEVICE workspace of q8_linear_chain_workspace_size() bytes,
 *           256-byte aligned, zeroed once: one region per distinct (N, K) of
 *           the steps, shared by the steps of that shape (they run one after
 *           another).
 * Returns Q8_ERR_ARG for a bad `next` code or count, Q8_ERR_SHAPE when a
 * step's K does not fit the previous step's N.
 */
#define Q8_MAX_CHAIN 4096
#define Q8_CHAIN_END 0
#define Q8_CHAIN_RMSNORM 1
#define Q8_CHAIN_SWIGLU_RMSNORM 2
typedef struct q8_chain_step {
    const int8_t *q;     /* int8 [N][K] */
    const uint16_t *s;   /* binary16 bits [N][K/32] */
    uint16_t *x;         /* bf16 bits [M][ldx]: this step's input */
    float *y;            /* float [M][ldy]: this step's output */
    int64_t N, K, ldx, ldy;
    int32_t next;        /* Q8_CHAIN_*: how the next step's x is made from y */
    int32_t reserved;    /* 0 */
} q8_chain_step;
q8_status q8_linear_chain(const q8_chain_step *steps, int32_t count, int32_t M, void *ws, size_t ws_bytes,
                          uint32_t *dev_status, q8_stream_t stream);
/* Workspace bytes for q8_linear_chain (0 if the chain fails its checks or
 * needs none). */
size_t q8_linear_chain_workspace_size(const q8_chain_step *steps, int32_t count, int32_t M);

/*
 * q8_gemm -- prefill-shaped Y[M][N] = X[M][K] * W^T for M > 32 on the 5th
 * generation tensor cores (tcgen05): each weight is dequantised to bf16
 * (bf16(s*q): the product is exact in binary32, then one round to nearest
 * even) into shared memory and multiplied in bf16 with fp32 accumulation in
 * tensor memory; y is bf16 (round to nearest even).  Any M, N and K (K a
 * positive multiple of 32).
 * Source: "MODEL-BASELINE-RESULTS" (fak), ACT 4 (batched prefill GEMM that
 * reads each weight once for all tokens) and "Parity lane" item 2.
 *   x : bf16 bits [M][ldx]; y : bf16 bits [M][ldy]; ldx, ldy multiples of 8;
 *   x and y 16-byte aligned.
 * Accuracy: |y - y_ref| <= 2e-3 * sum_k |s*q*x| + 1e-6 + half a bf16 ulp of y_ref
 * on the tested workloads (the bf16 weights round each weight by up to 2^-9
 * relative).  Needs no workspace: when K is split over several CTAs (short N,
 * long K), the partial sums meet in the CTAs' shared memory.
 */
q8_status q8_gemm(const int8_t *q, const uint16_t *s, int64_t N, int64_t K,
                  const uint16_t *x, int64_t ldx, int32_t M,
                  uint16_t *y, int64_t ldy,
                  uint32_t *dev_status, q8_stream_t stream);

/* Tile shapes of q8_gemm_ex: one CTA per SM computes a tile of (rows of x)
 * x (weight rows). */
#define Q8_GEMM_TILE_AUTO     0   /* the tile and split with the shortest modelled time */
#define Q8_GEMM_TILE_256x128  1
#define Q8_GEMM_TILE_128x128  2
#define Q8_GEMM_TILE_64x128   3
#define Q8_GEMM_MAX_SPLITS    8   /* most CTAs that share one tile's K range */

/*
 * q8_gemm_ex -- q8_gemm with an explicit tile shape (Q8_GEMM_TILE_*) and K
 * split (1 .. Q8_GEMM_MAX_SPLITS, 0 = automatic).  With split S the S CTAs
 * of a tile (one thread-block cluster) sum consecutive ranges of K (whole
 * groups of 256) and their S partial sums are added in range order, so each
 * output is the same bit for bit for every tile shape with the same S, and
 * from run to run.  CTAs that work on the same rows of x (neighbouring weight tiles)
 * share each x tile through a TMA multicast in groups of 1, 2, 4 or 8 (one
 * thread-block cluster); the group is chosen with the tile and split, and
 * the environment variable Q8_GEMM_MULTICAST (1, 2, 4 or 8) asks for one
 * for measurement (ignored where no allowed shape has it) -- it never
 * changes the results.  Unknown `tile` or `splits`
 * out of range: Q8_ERR_ARG; a shape this device cannot co-schedule (or more
 * splits than groups of 256 in K): Q8_ERR_UNSUPPORTED.
 */
q8_status q8_gemm_ex(const int8_t *q, const uint16_t *s, int64_t N, int64_t K,
                     const uint16_t *x, int64_t ldx, int32_t M,
                     uint16_t *y, int64_t ldy, int32_t tile, int32_t splits,
                     uint32_t *dev_status, q8_stream_t stream);

/*
 * q8_gemm_w8a8 -- the W8A8 product (Q8_VARIANT_W8A8's arithmetic) for any
 * M, e.g. a prefill of M = 512: each activation row is quantized to Q8_0 by
 * the weights' rule, and y[m][n] (fp32) = sum over blocks of
 * s_w[n][b] * s_x[m][b] * (exact int8 block dot).  Source: "MODEL-BASELINE-
 * RESULTS" (fak), ACT 3 items 1 and 3 (weights and activations in Q8_0
 * blocks, integer block dots).  x is cut into slices of 32 rows, run as
 * the matrices of q8_linear_batch launches (up to Q8_MAX_BATCH slices each,
 * sharing the weights, which the slices then read mostly from L2), with the
 * int8 warp MMA (mma.sync m16n8k32.s8): the 5th-generation tensor cores'
 * int8 kind is not accepted for sm_103a by this toolchain.  Accuracy as for
 * the W8A8 variant.  Any K (a multiple of 32).
 *   x: bf16 [M][ldx]; y: float [M][ldy] (ldy >= N when M > 1); alignment as
 *   for q8_linear_batch.  ws: q8_gemm_w8a8_workspace_size(N, K, M) bytes,
 *   256-byte aligned, zeroed once (per slice: the quantized activations).
 */
q8_status q8_gemm_w8a8(const int8_t *q, const uint16_t *s, int64_t N, int64_t K,
                       const uint16_t *x, int64_t ldx, int32_t M, float *y, int64_t ldy,
                       void *ws, size_t ws_bytes, uint32_t *dev_status, q8_stream_t stream);
size_t q8_gemm_w8a8_workspace_size(int64_t N, int64_t K, int32_t M);

/*
 * q8_gemm_skinny_noalloc -- q8_gemm_skinny for callers that cannot allocate
 * device memory when they run the matmul (a fixed memory pool, a loop that
 * must not enter the allocator, a host that passes only inputs and outputs).
 * The source pages have no counterpart to this entry point; it exists for
 * library users.
 *   Arguments, layouts, accuracy and errors: as q8_gemm_skinny, with no
 *   workspace argument.  The split-K scratch is a device array built into the
 *   library of Q8_NOALLOC_SCRATCH_BYTES (4 MiB), held by every GPU that loads
 *   the library until the process exits.  A shape whose scratch need
 *   (q8_workspace_size(N, K, M)) exceeds it returns Q8_ERR_WORKSPACE before
 *   any CUDA call.  Nothing is allocated or freed.
 *   The first call on a device looks the array's device address up (with
 *   that device current) and keeps it for later calls: make that first call
 *   outside any stream capture (a lookup that fails is not kept, and the
 *   next call tries again).  cudaDeviceReset() makes the kept address stale:
 *   after resetting a device, do not call this entry point on it again in
 *   the same process.
 *   All calls on a device share the array: calls whose kernels may overlap on
 *   the GPU (unordered streams) race on it; calls ordered on one stream do
 *   not.  Each call clears the ticket words it needs before its kernel runs.
 */
#define Q8_NOALLOC_SCRATCH_BYTES (4u << 20)
q8_status q8_gemm_skinny_noalloc(const int8_t *q, const uint16_t *s, int64_t N, int64_t K,
                                 const uint16_t *x, int64_t ldx, int32_t M,
                                 float *y, int64_t ldy,
                                 uint32_t *dev_status, q8_stream_t stream);

/* Human-readable name of a status code (static string). */
const char *q8_status_str(q8_status st);

/* ABI version of this header (bumped on any signature change). */
int32_t q8_abi_version(void);
#define Q8_ABI_VERSION 2

#ifdef __cplusplus
}
#endif
#endif /* Q8_H_ */
