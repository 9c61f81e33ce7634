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

__device__ __forceinline__ float half_at(const uint4 (&xv)[4], int i) {
    const uint32_t wv = (&xv[i >> 3].x)[(i & 7) >> 1];
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv));
    return (i & 1) ? f.y : f.x;
}
// The IEEE quotient, out of line: called only for elements near a rounding tie,
// so the division's instruction sequence stays out of the callers' common path.
static __device__ __noinline__ float ieee_quotient(float a, float b) { return __fdiv_rn(a, b); }

// Element e (0..31) of the 32 fp16 values, with e known only at run time:
// a tree of selects over the 16 words (no indexed register array, which would
// move the values to local memory).
__device__ __forceinline__ float half_at_dyn(const uint4 (&xv)[4], int e) {
    const int w = e >> 1;
    const uint4 q = (w & 8) ? ((w & 4) ? xv[3] : xv[2]) : ((w & 4) ? xv[1] : xv[0]);
    const uint32_t v = (w & 2) ? ((w & 1) ? q.w : q.z) : ((w & 1) ? q.y : q.x);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
    return (e & 1) ? f.y : f.x;
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
    // absmax: the maximum of |x| is exact in fp16, taken as a tree over the 16 pairs
    __half2 m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t a = (&xv[i >> 1].x)[2 * (i & 1)], b = (&xv[i >> 1].x)[2 * (i & 1) + 1];
        m[i] = __hmax2(__habs2(*reinterpret_cast<const __half2*>(&a)), __habs2(*reinterpret_cast<const __half2*>(&b)));
    }
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] = __hmax2(m[i], m[i + w]);
    float amax = fmaxf(__low2float(m[0]), __high2float(m[0]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const float s = fmaxf(__fdiv_rn(amax, 7.0f), 1e-10f);
    const float inv = __frcp_rn(s);
    // codes: rint(y) as (y + 1.5 2^23) - 1.5 2^23, exact round-to-nearest-even for |y| < 2^22
    // (|y| <= 7 (1 + 2^-23) here; a code 0 may come out as +0 or -0), packed as they are made;
    // elements near a tie are marked in tmask (bit e for element e)
    constexpr float kRound = 12582912.f;
    uint32_t tmask = 0;
    float part[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float c[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float y = half_at(xv, 4 * i + j) * inv;
            c[j] = __fadd_rn(__fadd_rn(y, kRound), -kRound);
            if (fabsf(y - c[j]) >= 0.5f - 3.814697265625e-06f) tmask |= 1u << (4 * i + j);
        }
        part[i] = (c[0] + c[1]) + (c[2] + c[3]);
        packed[i] = cvt_e4m3x2(c[0], c[1]) | (cvt_e4m3x2(c[2], c[3]) << 16);
    }
    // code sums are small integers: exact in any order
    float csum = ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
    // (rare) near a tie, the code comes from the IEEE quotient: patch its byte and the sum
    while (tmask != 0u) {
        const int e = __ffs(tmask) - 1;
        tmask &= tmask - 1u;
        const float xi = half_at_dyn(xv, e);
        const float c_old = __fadd_rn(__fadd_rn(xi * inv, kRound), -kRound);
        const float c_new = rintf(ieee_quotient(xi, s));
        csum += c_new - c_old;
        const uint32_t b = cvt_e4m3x2(c_new, 0.f) & 0xFFu, sh = 8u * uint32_t(e & 3);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i == (e >> 2)) packed[i] = (packed[i] & ~(0xFFu << sh)) | (b << sh);
    }
    csum += __shfl_xor_sync(0xffffffffu, csum, 1);
    s_out = s;
    csum_out = csum;
}

}  // namespace w4a4
