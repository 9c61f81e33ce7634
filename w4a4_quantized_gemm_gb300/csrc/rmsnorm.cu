// RMSNorm glue between the linears of a stacked decoder (unit gain):
//   x[m, k] = fp16( y[m, k] / sqrt(mean_k(y[m, :K]^2) + eps) ),  k < K
// reading the first K columns of each row of Y (row stride ld_y), so that a
// wider linear output (fused q|k|v, gate|up) feeds the next, narrower linear
// ("W4A4 CUDA Kernel for Voice Clone", 3.9: RMSNorm between the layer's
// linears; the page gives no epsilon, 1e-6 is the Qwen3 value).
//
// The arithmetic is fixed so that any implementation of it gives the same
// fp16 bits: each square of an fp16 value is exact in fp32, the sum is
// accumulated in fp64, 1 / sqrt(mean + eps) is taken in fp64 with IEEE
// division and square root, and the product y * inv is rounded once, from
// fp64 to fp16, to nearest even.  Only the order of the fp64 additions may
// differ, which moves the result by a few fp64 ulps.
//
// One warp per row: each lane reads 16 bytes (8 values) per step, coalesced;
// the row is read twice (the second time from L1/L2).
#include "kernels.h"

namespace w4a4 {
namespace {

constexpr int kRowsPerCta = 8;  // one warp per row

__global__ void __launch_bounds__(kRowsPerCta * 32) rmsnorm_f16_kernel(const uint16_t* __restrict__ Y, int M,
                                                                       int ld_y, int K, double eps,
                                                                       uint16_t* __restrict__ X) {
    const int lane = threadIdx.x & 31;
    const int m = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
    if (m >= M) return;
    const uint16_t* yr = Y + (size_t)m * ld_y;
    double ss = 0.0;
    for (int k = lane * 8; k < K; k += 32 * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(yr + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
            ss += double(f.x * f.x) + double(f.y * f.y);  // each square exact in fp32
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const double inv = 1.0 / sqrt(ss / double(K) + eps);
    uint16_t* xr = X + (size_t)m * K;
    for (int k = lane * 8; k < K; k += 32 * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(yr + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
            const uint32_t lo = __half_as_ushort(__double2half(double(f.x) * inv));
            const uint32_t hi = __half_as_ushort(__double2half(double(f.y) * inv));
            out[j] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(xr + k) = make_uint4(out[0], out[1], out[2], out[3]);
    }
}

}  // namespace

void launch_rmsnorm_f16(const uint16_t* Y, int M, int ld_y, int K, double eps, uint16_t* X, cudaStream_t s) {
    const int grid = (M + kRowsPerCta - 1) / kRowsPerCta;
    rmsnorm_f16_kernel<<<grid, kRowsPerCta * 32, 0, s>>>(Y, M, ld_y, K, eps, X);
    set_dispatch("rmsnorm_f16 rows=%d K=%d ld=%d grid=%d", M, K, ld_y, grid);
}

}  // namespace w4a4
