// q8_gemm_tc.cu -- prefill-shaped Q8_0 W8A16 GEMM (M > 32) on tcgen05.
#include "q8_internal.h"

namespace q8 {

q8_status launch_gemm_tc(const int8_t *, const uint16_t *, int64_t, int64_t, const uint16_t *, int64_t,
                         int32_t, uint16_t *, int64_t, uint32_t *, cudaStream_t) {
    return Q8_ERR_UNSUPPORTED;
}

}  // namespace q8
