// Per-(row, 64-column group) activation quantisation, shared by the activation
// kernel and the fused small-M linear so that both give the same codes and
// scales bit for bit ("W4A4 CUDA Kernel for Voice Clone", 3.6: symmetric INT4
// per row and group, scale = absmax / 7).
#pragma once
#include <cuda_fp16.h>

#include "common.cuh"

namespace w4a4 {

// Two integer-valued floats -> E4M3 bytes: lo -> bits 0-7, hi -> bits 8-15.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// A lane and its partner (lane ^ 1) hold the two halves of one row's 64-value
// group: xv is this lane's 32 consecutive fp16 values.  Returns the group's
// scale s = max(absmax / 7, 1e-10) (IEEE division), the group's code sum SA
// (both lanes), and this lane's 32 codes as E4M3 bytes in column order.
// Called by all 32 lanes of the warp together.
//
// Codes are rint(fl(x / s)).  They are computed as rint(x * (1 / s)), which
// gives the same integer except when the product lies within 2^-18 of a
// rounding boundary k + 1/2 (the product is within 2^-20 of x / s, the IEEE
// quotient within 2^-21); those elements are flagged branch-free and redone
// with the IEEE quotient, the warp taking that path only when a lane flagged
// one.  |x| <= absmax and s >= fl(absmax / 7) keep |x / s| <= 7 (1 + 2^-23),
// so codes lie in [-7, 7] and the clamp to [-8, 7] never acts.
__device__ __forceinline__ void quantize_half_group(const uint4 (&xv)[4], float& s_out, float& csum_out,
                                                    uint32_t (&packed)[8]) {
    float x[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
            x[8 * i + 2 * j] = f.x;
            x[8 * i + 2 * j + 1] = f.y;
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const float s = fmaxf(__fdiv_rn(amax, 7.0f), 1e-10f);
    const float inv = __frcp_rn(s);
    float* c = x;  // x[] is overwritten by the codes; the fp16 inputs stay in xv
    bool near_tie = false;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float y = x[i] * inv;
        c[i] = rintf(y);
        near_tie |= fabsf(y - c[i]) >= 0.5f - 3.814697265625e-06f;
    }
    if (__any_sync(0xffffffffu, near_tie)) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t wv = (&xv[i >> 3].x)[(i & 7) >> 1];
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv));
            const float xi = (i & 1) ? f.y : f.x;
            const float y = xi * inv;
            if (fabsf(y - c[i]) >= 0.5f - 3.814697265625e-06f) c[i] = rintf(__fdiv_rn(xi, s));
        }
    }
    float csum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        csum += (c[4 * i] + c[4 * i + 1]) + (c[4 * i + 2] + c[4 * i + 3]);
        packed[i] = cvt_e4m3x2(c[4 * i], c[4 * i + 1]) | (cvt_e4m3x2(c[4 * i + 2], c[4 * i + 3]) << 16);
    }
    csum += __shfl_xor_sync(0xffffffffu, csum, 1);
    s_out = s;
    csum_out = csum;
}

}  // namespace w4a4
