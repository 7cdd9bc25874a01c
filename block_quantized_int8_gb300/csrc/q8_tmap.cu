// q8_tmap.cu -- 2-D TMA tensor maps for the kernels that load tiles with
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
    uint64_t base, inner, outer, stride;
    uint32_t box_inner, box_outer, elem, swz;
    bool operator==(const Key &o) const {
        return base == o.base && inner == o.inner && outer == o.outer && stride == o.stride &&
               box_inner == o.box_inner && box_outer == o.box_outer && elem == o.elem && swz == o.swz;
    }
};
struct KeyHash {
    size_t operator()(const Key &k) const {
        uint64_t h = k.base * 0x9E3779B97F4A7C15ull;
        for (uint64_t v : {k.inner, k.outer, k.stride, static_cast<uint64_t>(k.box_inner) << 32 | k.box_outer,
                           static_cast<uint64_t>(k.elem) << 8 | k.swz})
            h = (h ^ v) * 0x100000001B3ull;
        return static_cast<size_t>(h);
    }
};

std::mutex g_mu;
std::unordered_map<Key, CUtensorMap, KeyHash> g_cache;
constexpr size_t kCacheMax = 4096;

}  // namespace

bool encode_2d(CUtensorMap *map, int elem_bytes, const void *base, uint64_t inner, uint64_t outer,
               uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
    const Key key{reinterpret_cast<uint64_t>(base), inner, outer, stride_bytes, box_inner, box_outer,
                  static_cast<uint32_t>(elem_bytes), swizzle128 ? 1u : 0u};
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
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_cache.size() >= kCacheMax) g_cache.clear();
    g_cache.emplace(key, *map);
    return true;
}

}  // namespace q8
