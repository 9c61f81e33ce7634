// Weight-streaming W4A4 GEMM for small M (decode): warp-level FP8 MMA with the
// weights as the 16-row operand ("swap AB"), per-group exact products, fp32
// scaled accumulation, LoRA up and the column affine in the same kernel.
//
// "INT4 Kernel Architecture, in depth" ("Why INT4 kernels exist: the
// roofline", "One token versus a thousand"): at small M the layer is bound by
// the bytes of packed weights, so each weight record is read once with wide
// coalesced loads, expanded in registers, and used against every token of
// the CTA.  "W4A4 CUDA Kernel for Voice Clone", 3.7: per-group integer MMA,
// scaling by act_scale * wgt_scale, LoRA-up into the same accumulator.
//
// Per group g the tensor core computes D = sum_k cA[m,k] * (cW[n,k] + 8)
// exactly (weights are stored offset-binary, see common.cuh), so
//   P = D - 8 SA[m,g],  acc += sW[n,g] * (sA[m,g] * D - 8 SA sA)
// with the per-token constant -8 SA sA hoisted out of the element loop.
#include "kernels.h"

namespace w4a4 {
namespace {

constexpr int kWarps = 8;
constexpr int kTileN = kWarps * 16;  // weight rows per CTA

template <int NT8>
struct SmallMSmem {
    uint8_t q[2][2][NT8 * 8][32];  // [stage][plane][token][32 bytes]
    float2 s[2][NT8 * 8];          // [stage][token] (sA, SA)
    uint16_t y[NT8 * 8][kTileN + 8];
};

template <int NT8, bool DUMP>
__global__ void __launch_bounds__(kWarps * 32) gemm_smallm_kernel(
    const uint8_t* __restrict__ ws, const uint8_t* __restrict__ packed, const uint16_t* __restrict__ colscale,
    const uint16_t* __restrict__ bias, int M, int N, int K, int r, uint16_t* __restrict__ Y,
    int32_t* __restrict__ P) {
    constexpr int TOK = NT8 * 8;
    __shared__ __align__(16) SmallMSmem<NT8> sm;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, q = lane & 3;
    const int G = K / kGroup;
    const ActLayout AL = act_layout(M, K, r);
    const PackedLayout PL = packed_layout(N, K, r);

    const int tok0 = blockIdx.y * TOK;  // first token of this CTA
    const int mt = tok0 / kTileM, rt0 = tok0 % kTileM;
    const int n0 = blockIdx.x * kTileN + warp * 16;
    const bool warp_active = n0 < N;

    const uint8_t* qW = packed + PL.qW;
    const uint16_t* sW = reinterpret_cast<const uint16_t*>(packed + PL.sW);

    auto load_stage = [&](int g, int st) {
        // qA planes: 2 x TOK rows x 32 B contiguous at (mt, g, plane, rt0..)
        const uint8_t* qsrc = ws + AL.qA + (size_t)(mt * G + g) * 2 * (kTileM * 32);
        for (int c = threadIdx.x; c < 2 * TOK * 2; c += kWarps * 32) {
            const int plane = c / (TOK * 2), rem = c % (TOK * 2);
            cp_async16(&sm.q[st][plane][rem >> 1][(rem & 1) * 16],
                       qsrc + (size_t)plane * (kTileM * 32) + (size_t)(rt0 + (rem >> 1)) * 32 + (rem & 1) * 16);
        }
        const uint8_t* ssrc = ws + AL.sS + ((size_t)(mt * G + g) * kTileM + rt0) * 8;
        for (int c = threadIdx.x; c < TOK / 2; c += kWarps * 32)
            cp_async16(reinterpret_cast<uint8_t*>(&sm.s[st][0]) + c * 16, ssrc + c * 16);
    };

    float acc[NT8][4];
#pragma unroll
    for (int t = 0; t < NT8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

    // weight records of rows n0+gid and n0+gid+8, bytes 8q..8q+7
    const uint8_t* recA = qW + (size_t)(n0 + gid) * 32 + 8 * q;
    const uint8_t* recB = recA + 8 * 32;
    const size_t gstride = (size_t)N * 32;
    uint2 wa = make_uint2(0, 0), wb = make_uint2(0, 0);
    float swa = 0.f, swb = 0.f;
    if (warp_active) {
        wa = ldg_nc_v2(recA);
        wb = ldg_nc_v2(recB);
        swa = __half2float(__ushort_as_half(sW[n0 + gid]));
        swb = __half2float(__ushort_as_half(sW[n0 + gid + 8]));
    }

    load_stage(0, 0);
    cp_async_commit();
    for (int g = 0; g < G; ++g) {
        const int st = g & 1;
        if (g + 1 < G) load_stage(g + 1, st ^ 1);
        cp_async_commit();
        // prefetch the next group's weights into registers
        uint2 na = wa, nb = wb;
        float nswa = swa, nswb = swb;
        if (warp_active && g + 1 < G) {
            na = ldg_nc_v2(recA + (g + 1) * gstride);
            nb = ldg_nc_v2(recB + (g + 1) * gstride);
            nswa = __half2float(__ushort_as_half(sW[(size_t)(g + 1) * N + n0 + gid]));
            nswb = __half2float(__ushort_as_half(sW[(size_t)(g + 1) * N + n0 + gid + 8]));
        }
        cp_async_wait<1>();
        __syncthreads();
        if (warp_active) {
            uint32_t a0[4], a1[4];  // k-halves 0 and 1
            a0[0] = expand4(wa.x);
            a0[2] = expand4(wa.x >> 16);
            a0[1] = expand4(wb.x);
            a0[3] = expand4(wb.x >> 16);
            a1[0] = expand4(wa.y);
            a1[2] = expand4(wa.y >> 16);
            a1[1] = expand4(wb.y);
            a1[3] = expand4(wb.y >> 16);
#pragma unroll
            for (int t = 0; t < NT8; ++t) {
                const int row = t * 8 + gid;
                const int sw = swz32(row, 0) * 16;  // row % 8 == (rt0 + row) % 8
                const uint32_t b00 = *reinterpret_cast<const uint32_t*>(&sm.q[st][0][row][sw + 4 * q]);
                const uint32_t b01 = *reinterpret_cast<const uint32_t*>(&sm.q[st][0][row][(sw ^ 16) + 4 * q]);
                const uint32_t b10 = *reinterpret_cast<const uint32_t*>(&sm.q[st][1][row][sw + 4 * q]);
                const uint32_t b11 = *reinterpret_cast<const uint32_t*>(&sm.q[st][1][row][(sw ^ 16) + 4 * q]);
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma_e4m3_16832(d, a0, b00, b01);
                mma_e4m3_16832(d, a1, b10, b11);
                const float2 s0 = sm.s[st][t * 8 + 2 * q], s1 = sm.s[st][t * 8 + 2 * q + 1];
                if constexpr (DUMP) {
                    const int m0 = tok0 + t * 8 + 2 * q;
                    const int na_ = n0 + gid, nb_ = n0 + gid + 8;
                    if (m0 < M) {
                        P[((size_t)m0 * N + na_) * G + g] = int32_t(d[0] - 8.f * s0.y);
                        P[((size_t)m0 * N + nb_) * G + g] = int32_t(d[2] - 8.f * s0.y);
                    }
                    if (m0 + 1 < M) {
                        P[((size_t)(m0 + 1) * N + na_) * G + g] = int32_t(d[1] - 8.f * s1.y);
                        P[((size_t)(m0 + 1) * N + nb_) * G + g] = int32_t(d[3] - 8.f * s1.y);
                    }
                } else {
                    const float c0 = (-8.f * s0.y) * s0.x, c1 = (-8.f * s1.y) * s1.x;
                    acc[t][0] = fmaf(swa, fmaf(s0.x, d[0], c0), acc[t][0]);
                    acc[t][1] = fmaf(swa, fmaf(s1.x, d[1], c1), acc[t][1]);
                    acc[t][2] = fmaf(swb, fmaf(s0.x, d[2], c0), acc[t][2]);
                    acc[t][3] = fmaf(swb, fmaf(s1.x, d[3], c1), acc[t][3]);
                }
            }
        }
        __syncthreads();  // stage st is refilled next iteration
        wa = na; wb = nb; swa = nswa; swb = nswb;
    }
    cp_async_wait<0>();
    if constexpr (DUMP) return;

    if (warp_active) {
        // LoRA up: acc[n, m] += sum_j L_up[j, n] lora[m, j] (fp16 MMA, fp32 accumulate)
        const uint8_t* Lu = packed + PL.Lu;
        const uint8_t* La = ws + AL.La;
        for (int p = 0; p < r / 16; ++p) {
            const uint8_t* la_plane = La + (size_t)(mt * (r / 16) + p) * (kTileM * 32);
            const uint8_t* lu_plane = Lu + (size_t)p * N * 32;
            uint32_t a[4];
            const int na_ = n0 + gid, nb_ = n0 + gid + 8;
            a[0] = __ldg(reinterpret_cast<const uint32_t*>(lu_plane + (size_t)na_ * 32 + swz32(na_, 0) * 16 + 4 * q));
            a[2] = __ldg(reinterpret_cast<const uint32_t*>(lu_plane + (size_t)na_ * 32 + swz32(na_, 1) * 16 + 4 * q));
            a[1] = __ldg(reinterpret_cast<const uint32_t*>(lu_plane + (size_t)nb_ * 32 + swz32(nb_, 0) * 16 + 4 * q));
            a[3] = __ldg(reinterpret_cast<const uint32_t*>(lu_plane + (size_t)nb_ * 32 + swz32(nb_, 1) * 16 + 4 * q));
#pragma unroll
            for (int t = 0; t < NT8; ++t) {
                const int rr = rt0 + t * 8 + gid;
                const uint32_t b0 = __ldg(reinterpret_cast<const uint32_t*>(la_plane + rr * 32 + swz32(rr, 0) * 16 + 4 * q));
                const uint32_t b1 = __ldg(reinterpret_cast<const uint32_t*>(la_plane + rr * 32 + swz32(rr, 1) * 16 + 4 * q));
                mma_f16_16816(acc[t], a, b0, b1);
            }
        }
        // column affine, fp16, staged for coalesced row stores
        const float csa = __half2float(__ushort_as_half(colscale[n0 + gid]));
        const float csb = __half2float(__ushort_as_half(colscale[n0 + gid + 8]));
        const float ba = bias ? __half2float(__ushort_as_half(bias[n0 + gid])) : 0.f;
        const float bb = bias ? __half2float(__ushort_as_half(bias[n0 + gid + 8])) : 0.f;
        const int nl = warp * 16 + gid;
#pragma unroll
        for (int t = 0; t < NT8; ++t) {
            const int m0 = t * 8 + 2 * q;
            sm.y[m0][nl] = __half_as_ushort(__float2half_rn(fmaf(csa, acc[t][0], ba)));
            sm.y[m0 + 1][nl] = __half_as_ushort(__float2half_rn(fmaf(csa, acc[t][1], ba)));
            sm.y[m0][nl + 8] = __half_as_ushort(__float2half_rn(fmaf(csb, acc[t][2], bb)));
            sm.y[m0 + 1][nl + 8] = __half_as_ushort(__float2half_rn(fmaf(csb, acc[t][3], bb)));
        }
    }
    __syncthreads();
    const int nbase = blockIdx.x * kTileN;
    for (int c = threadIdx.x; c < TOK * (kTileN / 8); c += kWarps * 32) {
        const int t = c / (kTileN / 8), ch = c % (kTileN / 8);
        const int m = tok0 + t, n = nbase + ch * 8;
        if (m < M && n < N)
            *reinterpret_cast<uint4*>(Y + (size_t)m * N + n) = *reinterpret_cast<const uint4*>(&sm.y[t][ch * 8]);
    }
}

template <int NT8>
w4a4_status launch_nt(const uint8_t* ws, const uint8_t* packed, const uint16_t* cs, const uint16_t* bias, int M,
                      int N, int K, int r, uint16_t* Y, int32_t* P, cudaStream_t s) {
    dim3 grid((N + kTileN - 1) / kTileN, (M + NT8 * 8 - 1) / (NT8 * 8));
    if (P)
        gemm_smallm_kernel<NT8, true><<<grid, kWarps * 32, 0, s>>>(ws, packed, cs, bias, M, N, K, r, Y, P);
    else
        gemm_smallm_kernel<NT8, false><<<grid, kWarps * 32, 0, s>>>(ws, packed, cs, bias, M, N, K, r, Y, P);
    set_dispatch("gemm_smallm mma.sync.e4m3 tokens/CTA=%d grid=%ux%u%s", NT8 * 8, grid.x, grid.y,
                 P ? " (partials dump)" : "");
    return launch_status();
}

}  // namespace

w4a4_status launch_gemm_smallm(const uint8_t* ws, const uint8_t* packed, const uint16_t* colscale,
                               const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, int32_t* P_dump,
                               cudaStream_t s) {
    if (M <= 8) return launch_nt<1>(ws, packed, colscale, bias, M, N, K, r, Y, P_dump, s);
    if (M <= 16) return launch_nt<2>(ws, packed, colscale, bias, M, N, K, r, Y, P_dump, s);
    if (M <= 32) return launch_nt<4>(ws, packed, colscale, bias, M, N, K, r, Y, P_dump, s);
    return launch_nt<8>(ws, packed, colscale, bias, M, N, K, r, Y, P_dump, s);
}

}  // namespace w4a4
