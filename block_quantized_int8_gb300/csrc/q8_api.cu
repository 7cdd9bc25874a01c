// q8_api.cu -- the C ABI of libq8: argument checks (host only, before any
// CUDA call), device checks, and dispatch to the kernels.
#include <mutex>

#include <algorithm>

#include "q8_internal.h"

namespace q8 {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::once_flag g_once[kMaxDevices];
int g_ok[kMaxDevices];

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
}  // namespace

const DeviceInfo *device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::call_once(g_once[dev], [dev]() {
        DeviceInfo &d = g_info[dev];
        d.device = dev;
        g_ok[dev] = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
                    cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
                    cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess;
    });
    return g_ok[dev] ? &g_info[dev] : nullptr;
}

q8_status check_arch(const DeviceInfo **out) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (di->cc_major != 10 || di->cc_minor != 3) return Q8_ERR_ARCH;
    *out = di;
    return Q8_OK;
}

static q8_status check_weights(const int8_t *q, const uint16_t *s, int64_t N, int64_t K) {
    if (N < 0 || K <= 0 || (K % 32) != 0 || N > INT32_MAX || K > INT32_MAX) return Q8_ERR_SHAPE;
    if (N == 0) return Q8_OK;
    if (!q || !s) return Q8_ERR_ARG;
    if (!aligned(q, 16) || !aligned(s, 16)) return Q8_ERR_ALIGN;
    return Q8_OK;
}

static q8_status check_desc(const q8_linear_desc &d, int32_t M) {
    q8_status st = check_weights(d.q, d.s, d.N, d.K);
    if (st != Q8_OK) return st;
    if (d.N == 0) return Q8_OK;
    if (!d.x || !d.y) return Q8_ERR_ARG;
    if (d.ldx < d.K || (M > 1 && d.ldy < d.N) || d.ldy < 1) return Q8_ERR_SHAPE;
    if (!aligned(d.x, 16) || (d.ldx % 8) != 0 || !aligned(d.y, 4)) return Q8_ERR_ALIGN;
    return Q8_OK;
}

// Host-only argument check of one skinny matmul (no CUDA call).
q8_status check_skinny_args(const q8_linear_desc &d, int32_t M) {
    if (M < 0 || M > Q8_SKINNY_MAX_M) return Q8_ERR_SHAPE;
    return check_desc(d, M);
}

}  // namespace q8

using namespace q8;

extern "C" {

int32_t q8_abi_version(void) { return Q8_ABI_VERSION; }

const char *q8_status_str(q8_status st) {
    switch (st) {
        case Q8_OK: return "ok";
        case Q8_ERR_ARG: return "invalid argument (null pointer or bad count)";
        case Q8_ERR_ALIGN: return "misaligned pointer or leading dimension";
        case Q8_ERR_SHAPE: return "bad shape (K must be a positive multiple of 32; check M and leading dimensions)";
        case Q8_ERR_WORKSPACE: return "workspace missing or too small";
        case Q8_ERR_ARCH: return "current device is not sm_103 (GB300)";
        case Q8_ERR_CUDA: return "CUDA runtime error";
        case Q8_ERR_UNSUPPORTED: return "not supported by this build";
    }
    return "unknown status";
}

q8_status q8_quantize_rows(const float *w, int64_t rows, int64_t K, int8_t *q, uint16_t *s,
                           uint32_t *dev_status, q8_stream_t stream) {
    return q8_quantize_rows_ex(w, rows, K, q, s, Q8_QUANT_EXACT, dev_status, stream);
}

q8_status q8_quantize_rows_ex(const float *w, int64_t rows, int64_t K, int8_t *q, uint16_t *s, int32_t mode,
                              uint32_t *dev_status, q8_stream_t stream) {
    if (mode != Q8_QUANT_EXACT && mode != Q8_QUANT_FL32) return Q8_ERR_ARG;
    if (rows < 0 || K <= 0 || (K % 32) != 0) return Q8_ERR_SHAPE;
    if (rows == 0) return Q8_OK;
    if (!w || !q || !s) return Q8_ERR_ARG;
    if (!aligned(w, 16) || !aligned(q, 16) || !aligned(s, 16)) return Q8_ERR_ALIGN;
    if (dev_status && !aligned(dev_status, 4)) return Q8_ERR_ALIGN;
    const DeviceInfo *di;
    q8_status st = check_arch(&di);
    if (st != Q8_OK) return st;
    return launch_quantize(w, rows, K, q, s, dev_status, reinterpret_cast<cudaStream_t>(stream), mode);
}

q8_status q8_gguf_to_planar(const void *blocks, int64_t rows, int64_t K, int8_t *q, uint16_t *s,
                            q8_stream_t stream) {
    if (rows < 0 || K <= 0 || (K % 32) != 0) return Q8_ERR_SHAPE;
    if (rows == 0) return Q8_OK;
    if (!blocks || !q || !s) return Q8_ERR_ARG;
    if (!aligned(blocks, 16) || !aligned(q, 16) || !aligned(s, 16)) return Q8_ERR_ALIGN;
    if (rows > INT64_MAX / K) return Q8_ERR_SHAPE;
    const DeviceInfo *di;
    q8_status st = check_arch(&di);
    if (st != Q8_OK) return st;
    return launch_gguf_ingest(blocks, rows * (K / 32), q, s, reinterpret_cast<cudaStream_t>(stream));
}

q8_status q8_planar_to_gguf(const int8_t *q, const uint16_t *s, int64_t rows, int64_t K, void *blocks,
                            q8_stream_t stream) {
    if (rows < 0 || K <= 0 || (K % 32) != 0) return Q8_ERR_SHAPE;
    if (rows == 0) return Q8_OK;
    if (!blocks || !q || !s) return Q8_ERR_ARG;
    if (!aligned(blocks, 16) || !aligned(q, 16) || !aligned(s, 16)) return Q8_ERR_ALIGN;
    if (rows > INT64_MAX / K) return Q8_ERR_SHAPE;
    const DeviceInfo *di;
    q8_status st = check_arch(&di);
    if (st != Q8_OK) return st;
    return launch_gguf_export(q, s, rows * (K / 32), blocks, reinterpret_cast<cudaStream_t>(stream));
}

q8_status q8_selftest_wait_timeout(uint64_t limit_ns, uint32_t *dev_status, uint64_t *dev_elapsed_ns,
                                   q8_stream_t stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull) return Q8_ERR_ARG;
    if (dev_status && !aligned(dev_status, 4)) return Q8_ERR_ALIGN;
    if (dev_elapsed_ns && !aligned(dev_elapsed_ns, 8)) return Q8_ERR_ALIGN;
    const DeviceInfo *di;
    q8_status st = check_arch(&di);
    if (st != Q8_OK) return st;
    return launch_selftest_wait_timeout(limit_ns, dev_status, dev_elapsed_ns, reinterpret_cast<cudaStream_t>(stream));
}

size_t q8_stream_read_out_words(void) {
    const DeviceInfo *di = device_info();
    return di ? static_cast<size_t>(stream_read_grid(di)) : 0;
}

q8_status q8_stream_read(const void *src, size_t bytes, uint32_t *out, q8_stream_t stream) {
    if (bytes == 0) return Q8_OK;
    if (!src || !out) return Q8_ERR_ARG;
    if (!aligned(src, 16) || (bytes % 16) != 0 || !aligned(out, 4)) return Q8_ERR_ALIGN;
    const DeviceInfo *di;
    q8_status st = check_arch(&di);
    if (st != Q8_OK) return st;
    return launch_stream_read(src, bytes, out, reinterpret_cast<cudaStream_t>(stream));
}

size_t q8_workspace_size(int64_t N, int64_t K, int32_t M) {
    if (N <= 0 || K <= 0 || (K % 32) != 0 || M < 1 || M > Q8_SKINNY_MAX_M) return 0;
    q8_linear_desc d{};
    d.N = N;
    d.K = K;
    SplitPlan pl;
    size_t sched_off;
    return skinny_workspace(&d, 1, M, &pl, &sched_off);
}

size_t q8_linear_batch_workspace_size_ex(const q8_linear_desc *descs, int32_t count, int32_t M, int32_t variant) {
    if (variant != Q8_VARIANT_W8A8 && variant != Q8_VARIANT_BATCH_INVARIANT)
        return q8_linear_batch_workspace_size(descs, count, M);
    if (!descs || count < 1 || count > Q8_MAX_BATCH || M < 1 || M > Q8_SKINNY_MAX_M) return 0;
    q8_linear_desc tmp[Q8_MAX_BATCH];
    int n = 0;
    if (variant == Q8_VARIANT_BATCH_INVARIANT) {
        // the general kernel's partial sums for the matrices off the 256 grid
        for (int i = 0; i < count; ++i)
            if (descs[i].N > 0 && descs[i].K > 0 && descs[i].K % 256) tmp[n++] = descs[i];
        SplitPlan pl[Q8_MAX_BATCH];
        return n > 0 ? plan_skinny(tmp, n, M, pl, true) : 0;
    }
    for (int i = 0; i < count; ++i) {
        if (descs[i].N <= 0 || descs[i].K <= 0 || descs[i].K % 32) continue;
        tmp[n++] = descs[i];
    }
    return n > 0 ? w8a8_workspace(tmp, n, M) : 0;
}

size_t q8_linear_batch_workspace_size(const q8_linear_desc *descs, int32_t count, int32_t M) {
    if (!descs || count < 1 || count > Q8_MAX_BATCH || M < 1 || M > Q8_SKINNY_MAX_M) return 0;
    q8_linear_desc tmp[Q8_MAX_BATCH];
    int n = 0;
    for (int i = 0; i < count; ++i) {
        if (descs[i].N <= 0 || descs[i].K <= 0 || descs[i].K % 32) continue;
        tmp[n++] = descs[i];
    }
    if (n == 0) return 0;
    SplitPlan pl[Q8_MAX_BATCH];
    size_t sched_off;
    return skinny_workspace(tmp, n, M, pl, &sched_off);
}

namespace {

q8_status linear_batch(const q8_linear_desc *descs, int32_t count, int32_t M, int32_t variant, void *ws,
                       size_t ws_bytes, uint32_t *dev_status, q8_stream_t stream, bool chained) {
    if (!descs || count < 0 || count > Q8_MAX_BATCH) return Q8_ERR_ARG;
    if (variant < Q8_VARIANT_AUTO || variant > Q8_VARIANT_W8A8) return Q8_ERR_ARG;
    if (M < 0 || M > Q8_SKINNY_MAX_M) return Q8_ERR_SHAPE;
    if (dev_status && !aligned(dev_status, 4)) return Q8_ERR_ALIGN;
    // drop empty matrices; check the rest
    q8_linear_desc live[Q8_MAX_BATCH];
    int n = 0;
    for (int i = 0; i < count; ++i) {
        q8_status st = check_desc(descs[i], M);
        if (st != Q8_OK) return st;
        if (descs[i].N > 0) live[n++] = descs[i];
    }
    if (M == 0 || n == 0) return Q8_OK;
    const DeviceInfo *di;
    q8_status st = check_arch(&di);
    if (st != Q8_OK) return st;
    return launch_skinny(live, n, M, variant, ws, ws_bytes, dev_status, reinterpret_cast<cudaStream_t>(stream),
                         chained);
}

}  // namespace

q8_status q8_linear_batch_ex(const q8_linear_desc *descs, int32_t count, int32_t M, int32_t variant,
                             void *ws, size_t ws_bytes, uint32_t *dev_status, q8_stream_t stream) {
    return linear_batch(descs, count, M, variant, ws, ws_bytes, dev_status, stream, false);
}

q8_status q8_linear_batch_chained(const q8_linear_desc *descs, int32_t count, int32_t M, void *ws,
                                  size_t ws_bytes, uint32_t *dev_status, q8_stream_t stream) {
    return linear_batch(descs, count, M, Q8_VARIANT_AUTO, ws, ws_bytes, dev_status, stream, true);
}

q8_status q8_linear_chain(const q8_chain_step *steps, int32_t count, int32_t M, void *ws, size_t ws_bytes,
                          uint32_t *dev_status, q8_stream_t stream) {
    q8_status st = check_chain(steps, count, M);
    if (st != Q8_OK) return st;
    if (dev_status && !aligned(dev_status, 4)) return Q8_ERR_ALIGN;
    const size_t need = chain_workspace(steps, count, M);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) return Q8_ERR_WORKSPACE;
    if (need > 0 && !aligned(ws, 256)) return Q8_ERR_ALIGN;
    const DeviceInfo *di;
    st = check_arch(&di);
    if (st != Q8_OK) return st;
    return launch_chain(steps, count, M, ws, ws_bytes, dev_status, reinterpret_cast<cudaStream_t>(stream));
}

size_t q8_linear_chain_workspace_size(const q8_chain_step *steps, int32_t count, int32_t M) {
    if (check_chain(steps, count, M) != Q8_OK) return 0;
    return chain_workspace(steps, count, M);
}

q8_status q8_linear_batch(const q8_linear_desc *descs, int32_t count, int32_t M,
                          void *ws, size_t ws_bytes, uint32_t *dev_status, q8_stream_t stream) {
    return q8_linear_batch_ex(descs, count, M, Q8_VARIANT_AUTO, ws, ws_bytes, dev_status, stream);
}

q8_status q8_gemm_skinny(const int8_t *q, const uint16_t *s, int64_t N, int64_t K,
                         const uint16_t *x, int64_t ldx, int32_t M, float *y, int64_t ldy,
                         void *ws, size_t ws_bytes, uint32_t *dev_status, q8_stream_t stream) {
    q8_linear_desc d;
    d.q = q;
    d.s = s;
    d.x = x;
    d.y = y;
    d.N = N;
    d.K = K;
    d.ldx = ldx;
    d.ldy = ldy;
    return q8_linear_batch_ex(&d, 1, M, Q8_VARIANT_AUTO, ws, ws_bytes, dev_status, stream);
}

extern "C++" {
namespace {

// q8_gemm_w8a8's launches: the full 32-row slices of x in groups of at most
// Q8_MAX_BATCH (one q8_linear_batch launch each, the slices as matrices that
// share the weights), then the remaining rows.
template <typename F>
q8_status for_w8a8_launches(const q8_linear_desc &d, int32_t M, F &&f) {
    q8_linear_desc descs[Q8_MAX_BATCH];
    const int32_t full = M / Q8_SKINNY_MAX_M;
    for (int32_t b = 0; b < full; b += Q8_MAX_BATCH) {
        const int32_t cnt = std::min<int32_t>(Q8_MAX_BATCH, full - b);
        for (int32_t j = 0; j < cnt; ++j) {
            descs[j] = d;
            descs[j].x = d.x + static_cast<int64_t>(b + j) * Q8_SKINNY_MAX_M * d.ldx;
            descs[j].y = d.y + static_cast<int64_t>(b + j) * Q8_SKINNY_MAX_M * d.ldy;
        }
        const q8_status st = f(descs, cnt, Q8_SKINNY_MAX_M);
        if (st != Q8_OK) return st;
    }
    const int32_t rem = M - full * Q8_SKINNY_MAX_M;
    if (rem > 0) {
        descs[0] = d;
        descs[0].x = d.x + static_cast<int64_t>(full) * Q8_SKINNY_MAX_M * d.ldx;
        descs[0].y = d.y + static_cast<int64_t>(full) * Q8_SKINNY_MAX_M * d.ldy;
        return f(descs, 1, rem);
    }
    return Q8_OK;
}

q8_linear_desc w8a8_desc(const int8_t *q, const uint16_t *s, int64_t N, int64_t K, const uint16_t *x, int64_t ldx,
                         float *y, int64_t ldy) {
    q8_linear_desc d;
    d.q = q;
    d.s = s;
    d.x = x;
    d.y = y;
    d.N = N;
    d.K = K;
    d.ldx = ldx;
    d.ldy = ldy;
    return d;
}

}  // namespace
}  // extern "C++"

size_t q8_gemm_w8a8_workspace_size(int64_t N, int64_t K, int32_t M) {
    if (N <= 0 || K <= 0 || K % 32 || M < 1) return 0;
    // placeholder addresses: only the slices' x must differ from one another
    const uintptr_t base = uintptr_t(1) << 40;
    const q8_linear_desc d = w8a8_desc(reinterpret_cast<const int8_t *>(base), reinterpret_cast<const uint16_t *>(base),
                                       N, K, reinterpret_cast<const uint16_t *>(base), K,
                                       reinterpret_cast<float *>(base), N);
    size_t need = 0;
    (void)for_w8a8_launches(d, M, [&](const q8_linear_desc *ds, int cnt, int m) {
        need = std::max(need, w8a8_workspace(ds, cnt, m));
        return Q8_OK;
    });
    return need;
}

q8_status q8_gemm_w8a8(const int8_t *q, const uint16_t *s, int64_t N, int64_t K, const uint16_t *x, int64_t ldx,
                       int32_t M, float *y, int64_t ldy, void *ws, size_t ws_bytes, uint32_t *dev_status,
                       q8_stream_t stream) {
    if (M < 0) return Q8_ERR_SHAPE;
    if (dev_status && !aligned(dev_status, 4)) return Q8_ERR_ALIGN;
    const q8_linear_desc d = w8a8_desc(q, s, N, K, x, ldx, y, ldy);
    q8_status st = check_desc(d, std::min<int32_t>(M, Q8_SKINNY_MAX_M));
    if (st != Q8_OK) return st;
    if (M > 1 && ldy < N) return Q8_ERR_SHAPE;
    if (M == 0 || N == 0) return Q8_OK;
    const size_t need = q8_gemm_w8a8_workspace_size(N, K, M);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) return Q8_ERR_WORKSPACE;
    if (need > 0 && !aligned(ws, 256)) return Q8_ERR_ALIGN;
    const DeviceInfo *di;
    st = check_arch(&di);
    if (st != Q8_OK) return st;
    return for_w8a8_launches(d, M, [&](const q8_linear_desc *ds, int cnt, int m) {
        return launch_skinny(ds, cnt, m, Q8_VARIANT_W8A8, ws, ws_bytes, dev_status,
                             reinterpret_cast<cudaStream_t>(stream), false);
    });
}

q8_status q8_gemv(const int8_t *q, const uint16_t *s, int64_t N, int64_t K, const uint16_t *x, float *y,
                  void *ws, size_t ws_bytes, uint32_t *dev_status, q8_stream_t stream) {
    return q8_gemm_skinny(q, s, N, K, x, K + ((8 - K % 8) % 8), 1, y, N > 0 ? N : 1, ws, ws_bytes,
                          dev_status, stream);
}

q8_status q8_gemm(const int8_t *q, const uint16_t *s, int64_t N, int64_t K, const uint16_t *x, int64_t ldx,
                  int32_t M, uint16_t *y, int64_t ldy, uint32_t *dev_status, q8_stream_t stream) {
    return q8_gemm_ex(q, s, N, K, x, ldx, M, y, ldy, Q8_GEMM_TILE_AUTO, 0, dev_status, stream);
}

q8_status q8_gemm_ex(const int8_t *q, const uint16_t *s, int64_t N, int64_t K, const uint16_t *x, int64_t ldx,
                     int32_t M, uint16_t *y, int64_t ldy, int32_t tile, int32_t splits, uint32_t *dev_status,
                     q8_stream_t stream) {
    if (tile < Q8_GEMM_TILE_AUTO || tile > Q8_GEMM_TILE_64x128) return Q8_ERR_ARG;
    if (splits < 0 || splits > Q8_GEMM_MAX_SPLITS) return Q8_ERR_ARG;
    q8_status st = check_weights(q, s, N, K);
    if (st != Q8_OK) return st;
    if (M < 0) return Q8_ERR_SHAPE;
    if (N == 0 || M == 0) return Q8_OK;
    if (!x || !y) return Q8_ERR_ARG;
    if (ldx < K || ldy < N) return Q8_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(y, 16) || (ldx % 8) || (ldy % 8)) return Q8_ERR_ALIGN;
    if (dev_status && !aligned(dev_status, 4)) return Q8_ERR_ALIGN;
    const DeviceInfo *di;
    st = check_arch(&di);
    if (st != Q8_OK) return st;
    return launch_gemm_tc(q, s, N, K, x, ldx, M, y, ldy, tile, splits, dev_status,
                          reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
