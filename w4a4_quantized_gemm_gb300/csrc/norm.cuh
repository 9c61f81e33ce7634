// RMSNorm arithmetic shared by the glue kernel and the fused normalise +
// quantise kernel ("W4A4 CUDA Kernel for Voice Clone", 3.9).  The value is
// defined exactly: squares of fp16 values are exact in fp32, their sum is taken
// to (at least) fp64 accuracy, inv = 1 / sqrt(sum / K + eps) in fp64, and
// fp16(y * inv) is the fp64 product rounded once to fp16.
#pragma once
#include "common.cuh"

namespace w4a4 {

// Two-term (Knuth two-sum) accumulation of the exact fp32 squares of 8 fp16 values.
__device__ __forceinline__ void add_squares(const uint4 v, float& hi, float& lo) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float q = h ? __fmul_rn(f.y, f.y) : __fmul_rn(f.x, f.x);  // exact
            const float s = __fadd_rn(hi, q);                                 // s + e == hi + q exactly
            const float bp = __fsub_rn(s, hi);
            const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(q, bp));
            hi = s;
            lo = __fadd_rn(lo, e);
        }
    }
}

// fp16(y * inv) for 8 values, rounded as the fp64 product would be.  inv is
// split into inva = fp32(inv) and invb = fp32(inv - inva).  The fp32 product
// t = fl(y * inva) is within one fp32 ulp of y * inv, so where t lies more than
// 2 ulps from a midpoint m between fp16 numbers both round alike.  Near a
// midpoint the exact side is read off d = (t - m) + (fma(y, inva, -t) +
// y * invb): t - m and the fma residual are exact, inv - inva - invb is below
// 2^-48 |inv|, and d differs from y * inv - m by less than 2^-44.5 |m|, so
// when |d| > 2^-44 |m| the exact product, and its fp64 rounding, lie strictly
// on d's side of m, and fp16 rounds toward that side.  Only the (vanishingly
// rare) |d| <= 2^-44 |m| and the fp16-subnormal results are redone in fp64.
__device__ __forceinline__ uint4 scale_to_f16(const uint4 v, double inv, float inva, float invb) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float y[8], t[8];
    uint32_t flags = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
        y[2 * j] = f.x;
        y[2 * j + 1] = f.y;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        t[i] = __fmul_rn(y[i], inva);
        // the 13 fp32 mantissa bits below fp16 precision: 0x1000 is a midpoint
        const int low = int(__float_as_uint(t[i]) & 0x1FFFu) - 0x1000;
        const bool near = (fabsf(t[i]) < 6.103515625e-05f && t[i] != 0.f) || (low >= -2 && low <= 2);
        flags |= uint32_t(near) << i;
    }
    uint16_t h[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = __half_as_ushort(__float2half_rn(t[i]));
    if (__any_sync(0xffffffffu, flags != 0)) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (!(flags & (1u << i))) continue;
            bool exact = false;
            if (fabsf(t[i]) >= 6.103515625e-05f) {
                const float m = __uint_as_float((__float_as_uint(t[i]) & ~0x1FFFu) | 0x1000u);
                const float r = __fadd_rn(__fmaf_rn(y[i], inva, -t[i]), __fmul_rn(y[i], invb));
                const float d = __fadd_rn(__fsub_rn(t[i], m), r);
                if (fabsf(d) > 5.684341886080802e-14f * fabsf(m)) {  // 2^-44
                    h[i] = __half_as_ushort(d > 0.f ? __float2half_ru(m) : __float2half_rd(m));
                    exact = true;
                }
            }
            if (!exact) h[i] = __half_as_ushort(__double2half(double(y[i]) * inv));
        }
    }
    return make_uint4(uint32_t(h[0]) | (uint32_t(h[1]) << 16), uint32_t(h[2]) | (uint32_t(h[3]) << 16),
                      uint32_t(h[4]) | (uint32_t(h[5]) << 16), uint32_t(h[6]) | (uint32_t(h[7]) << 16));
}

// The fp32 pieces of inv used by scale_to_f16.
__device__ __forceinline__ void split_inv(double inv, float& inva, float& invb) {
    inva = __double2float_rn(inv);
    invb = __double2float_rn(inv - double(inva));
}

}  // namespace w4a4
