// RMSNorm glue between the linears of a stacked decoder (unit gain):
//   x[m, k] = fp16( y[m, k] / sqrt(mean_k(y[m, :K]^2) + eps) ),  k < K
// reading the first K columns of each row of Y (row stride ld_y), so that a
// wider linear output (fused q|k|v, gate|up) feeds the next, narrower linear
// ("W4A4 CUDA Kernel for Voice Clone", 3.9: RMSNorm between the layer's
// linears; the page gives no epsilon, 1e-6 is the Qwen3 value).
//
// The arithmetic is fixed so that any implementation of it gives the same
// fp16 bits: each square of an fp16 value is exact in fp32, the sum is taken
// to (at least) fp64 accuracy, 1 / sqrt(mean + eps) is taken in fp64 with IEEE
// division and square root, and the product y * inv is rounded once, from its
// fp64 value to fp16, to nearest even.
//
// GB300's fp64 rate is low, so neither pass runs fp64 per element:
//  * the sum is an error-free two-term fp32 accumulation (hi + lo, Knuth's
//    two-sum), combined in fp64 per row: its error is ~2^-44 relative,
//    far below what could move an fp16 result;
//  * the product is formed in fp32; where it lands within 2 fp32 ulps of a
//    midpoint between two fp16 numbers, an exact fp32 residual decides the
//    side (norm.cuh), and only the fp16-subnormal results (and products within
//    2^-44 of a midpoint) are redone in fp64, so the rounding to fp16 is the
//    one the fp64 product gets.
//
// One CTA per row: each thread reads its 16-byte chunks once (coalesced), keeps
// them in registers, and writes the normalised values.
#include "kernels.h"
#include "norm.cuh"

namespace w4a4 {
namespace {

// One CTA of 256 threads per row; thread t holds chunks (c * 256 + t) of 8
// values (c < CH) in registers between the two steps.  The fp64 partial sums
// are combined warp by warp, then over the 8 warps in a fixed order.
template <int CH>
__global__ void __launch_bounds__(256) rmsnorm_f16_kernel(const uint16_t* __restrict__ Y, int ld_y, int K,
                                                          double eps, uint16_t* __restrict__ X) {
    __shared__ double red[8];
    __shared__ double row_inv;
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint16_t* yr = Y + (size_t)blockIdx.x * ld_y;
    uint16_t* xr = X + (size_t)blockIdx.x * K;
    uint4 v[CH];
    float hi = 0.f, lo = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int k = (c * 256 + tid) * 8;
        v[c] = k < K ? *reinterpret_cast<const uint4*>(yr + k) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) add_squares(v[c], hi, lo);
    double ss = double(hi) + double(lo);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
        double t = 0.0;
#pragma unroll
        for (int w = 0; w < 8; ++w) t += red[w];
        row_inv = 1.0 / sqrt(t / double(K) + eps);
    }
    __syncthreads();
    const double inv = row_inv;
    float inva, invb;
    split_inv(inv, inva, invb);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        if ((c * 256 + warp * 32) * 8 < K) {  // warp-uniform: the vote inside stays converged
            const int k = (c * 256 + tid) * 8;
            const uint4 o = scale_to_f16(v[c], inv, inva, invb);
            if (k < K) *reinterpret_cast<uint4*>(xr + k) = o;
        }
    }
}

}  // namespace

void launch_rmsnorm_f16(const uint16_t* Y, int M, int ld_y, int K, double eps, uint16_t* X, cudaStream_t s) {
    const int ch = (K + 2047) / 2048;  // 8-value chunks per thread
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    cfg.attrs = attr;
    cfg.numAttrs = add_pdl_attr(attr, 0);
    cfg.gridDim = dim3(unsigned(M));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    if (ch <= 1)
        cudaLaunchKernelEx(&cfg, rmsnorm_f16_kernel<1>, Y, ld_y, K, eps, X);
    else if (ch <= 2)
        cudaLaunchKernelEx(&cfg, rmsnorm_f16_kernel<2>, Y, ld_y, K, eps, X);
    else if (ch <= 4)
        cudaLaunchKernelEx(&cfg, rmsnorm_f16_kernel<4>, Y, ld_y, K, eps, X);
    else
        cudaLaunchKernelEx(&cfg, rmsnorm_f16_kernel<8>, Y, ld_y, K, eps, X);
    set_dispatch("rmsnorm_f16 rows=%d K=%d ld=%d chunks/thread=%d", M, K, ld_y, ch <= 2 ? ch : (ch <= 4 ? 4 : 8));
}

}  // namespace w4a4
