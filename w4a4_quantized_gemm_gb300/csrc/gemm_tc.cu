// tcgen05 W4A4 GEMM (placeholder until the tensor-memory kernel lands).
#include "kernels.h"

namespace w4a4 {

w4a4_status launch_gemm_tc(const uint8_t*, const uint8_t*, const uint16_t*, const uint16_t*, int, int, int, int,
                           uint16_t*, int32_t*, cudaStream_t) {
    set_dispatch("gemm_tc unavailable");
    return W4A4_ERR_UNSUPPORTED_SHAPE;
}

w4a4_status tc_read_and_clear_status() { return W4A4_OK; }

}  // namespace w4a4
