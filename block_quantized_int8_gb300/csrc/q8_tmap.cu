// q8_tmap.cu -- 2-D and 3-D TMA tensor maps for the kernels that load tiles with
// cp.async.bulk.tensor: cuTensorMapEncodeTiled is taken from the driver
// through the runtime at first use (the library does not link libcuda), and
// encoded maps are cached by their parameters so that repeated calls on the
// same tensors skip the encoding.
#include <cuda.h>

#include <mutex>
#include <unordered_map>

#include "q8_internal.h"

namespace q8 {

namespace {

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

struct Key {
    uint64_t base, dims[3], strides[2];
    uint32_t box[3], rank, elem, swz;
    bool operator==(const Key &o) const {
        return base == o.base && rank == o.rank && elem == o.elem && swz == o.swz && dims[0] == o.dims[0] &&
               dims[1] == o.dims[1] && dims[2] == o.dims[2] && strides[0] == o.strides[0] &&
               strides[1] == o.strides[1] && box[0] == o.box[0] && box[1] == o.box[1] && box[2] == o.box[2];
    }
};
struct KeyHash {
    size_t operator()(const Key &k) const {
        uint64_t h = k.base * 0x9E3779B97F4A7C15ull;
        for (uint64_t v : {k.dims[0], k.dims[1], k.dims[2], k.strides[0], k.strides[1],
                           static_cast<uint64_t>(k.box[0]) << 32 | k.box[1],
                           static_cast<uint64_t>(k.box[2]) << 32 | k.rank << 16 | k.elem << 8 | k.swz})
            h = (h ^ v) * 0x100000001B3ull;
        return static_cast<size_t>(h);
    }
};

std::mutex g_mu;
std::unordered_map<Key, CUtensorMap, KeyHash> g_cache;
constexpr size_t kCacheMax = 4096;

}  // namespace

bool encode_tmap(CUtensorMap *map, int elem_bytes, const void *base, int rank, const uint64_t *dims,
                 const uint64_t *stride_bytes, const uint32_t *box, bool swizzle128) {
    if (rank < 2 || rank > 3) return false;
    Key key{};
    key.base = reinterpret_cast<uint64_t>(base);
    key.rank = static_cast<uint32_t>(rank);
    key.elem = static_cast<uint32_t>(elem_bytes);
    key.swz = swizzle128 ? 1u : 0u;
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) key.strides[i] = stride_bytes[i];
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_cache.find(key);
        if (it != g_cache.end()) {
            *map = it->second;
            return true;
        }
    }
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    CUtensorMapDataType dt;
    switch (elem_bytes) {
        case 1: dt = CU_TENSOR_MAP_DATA_TYPE_UINT8; break;
        case 2: dt = CU_TENSOR_MAP_DATA_TYPE_UINT16; break;
        default: return false;
    }
    cuuint64_t d[3], st[2];
    cuuint32_t b[3];
    const cuuint32_t estr[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) st[i] = stride_bytes[i];
    if (fn(map, dt, static_cast<cuuint32_t>(rank), const_cast<void *>(base), d, st, b, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_cache.size() >= kCacheMax) g_cache.clear();
    g_cache.emplace(key, *map);
    return true;
}

bool encode_2d(CUtensorMap *map, int elem_bytes, const void *base, uint64_t inner, uint64_t outer,
               uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
    const uint64_t dims[2] = {inner, outer};
    const uint32_t box[2] = {box_inner, box_outer};
    return encode_tmap(map, elem_bytes, base, 2, dims, &stride_bytes, box, swizzle128);
}

}  // namespace q8
