// Fused activation kernel: per-(row, 64-column group) absmax INT4 quantisation
// of fp16 X, codes written in the GEMM's tile layout, and the LoRA
// down-projection X . L_down from the same read of X ("W4A4 CUDA Kernel for
// Voice Clone", 3.6 fused_quantize_repack_act_kernel and its LoRA-down branch).
//
// Differences from the page's design, for GB300:
//  * One CTA owns whole rows (16 per CTA) and its warps split the K groups, so
//    the LoRA partial sums are reduced inside the CTA in a fixed order: no
//    atomics, deterministic results, and no separate repack kernel (the
//    page's pack_lora_act exists only to wait for atomics).
//  * Codes are stored as FP8 E4M3 bytes, the operand encoding the tcgen05
//    tensor core reads (GB300 has no INT4 tensor-core kind).
#include "kernels.h"

namespace w4a4 {
namespace {

constexpr int kRows = 16;      // rows per CTA (one m16 tile of the LoRA MMA)
constexpr int kWarps = 8;
constexpr int kXsStride = 72;  // halves per staged row (64 + 8 pad: conflict-free ldmatrix)

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

template <int R>  // LoRA rank, multiple of 16 (0 = no LoRA branch)
__global__ void __launch_bounds__(kWarps * 32) quantize_act_kernel(const uint16_t* __restrict__ X,
                                                                   const uint2* __restrict__ Ldp, int M,
                                                                   int K, uint8_t* __restrict__ ws) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                           // [warps][16][72]
    float* red = reinterpret_cast<float*>(smem + kWarps * kRows * kXsStride * 2);  // [warps][16][R]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const ActLayout AL = act_layout(M, K, R);
    const int row0 = blockIdx.x * kRows;
    const int mt = row0 / kTileM;

    // quantisation role: lane owns row (lane/2), columns 32*(lane%2) .. +31 of a group
    const int qrow = lane >> 1, qhalf = lane & 1;
    const int m = row0 + qrow;
    const int rr = m % kTileM;  // row within the 128-row tile
    const bool valid = m < M;

    constexpr int NT = R / 8;  // LoRA n8 tiles
    float acc[NT > 0 ? NT : 1][4];
#pragma unroll
    for (int t = 0; t < (NT > 0 ? NT : 1); ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

    uint16_t* xw = xs + warp * kRows * kXsStride;
    for (int g = warp; g < G; g += kWarps) {
        uint4 xv[4];
        const uint16_t* src = X + (size_t)m * K + (size_t)g * kGroup + qhalf * 32;
#pragma unroll
        for (int i = 0; i < 4; ++i) xv[i] = valid ? ldg_nc_v4(src + 8 * i) : make_uint4(0, 0, 0, 0);
        float x[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                x[8 * i + 2 * j] = __half2float(__ushort_as_half(uint16_t(w[j] & 0xffffu)));
                x[8 * i + 2 * j + 1] = __half2float(__ushort_as_half(uint16_t(w[j] >> 16)));
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        // scale = max(absmax / 7, 1e-10), code = clamp(rint(x / scale), -8, 7), IEEE division
        const float s = fmaxf(__fdiv_rn(amax, 7.0f), 1e-10f);
        uint32_t packed[8];
        int csum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = int(fminf(fmaxf(rintf(__fdiv_rn(x[4 * i + j], s)), -8.0f), 7.0f));
                csum += c;
                word |= e4m3_of_int(c) << (8 * j);
            }
            packed[i] = word;
        }
        csum += __shfl_xor_sync(0xffffffffu, csum, 1);
        // codes -> plane qhalf of (mt, g), row rr, two 16-byte chunks (swizzled)
        uint8_t* plane = ws + AL.qA + ((size_t)(mt * G + g) * 2 + qhalf) * (kTileM * 32);
        *reinterpret_cast<uint4*>(plane + rr * 32 + swz32(rr, 0) * 16) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
        *reinterpret_cast<uint4*>(plane + rr * 32 + swz32(rr, 1) * 16) =
            make_uint4(packed[4], packed[5], packed[6], packed[7]);
        if (qhalf == 0)
            *reinterpret_cast<float2*>(ws + AL.sS + ((size_t)(mt * G + g) * kTileM + rr) * 8) =
                make_float2(s, float(csum));

        if constexpr (R > 0) {
            // stage the fp16 tile for the LoRA-down MMA (A operand via ldmatrix)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4*>(xw + qrow * kXsStride + qhalf * 32 + 8 * i) = xv[i];
            __syncwarp();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t a[4];
                const int lr = (lane & 7) + ((lane >> 3) & 1) * 8, lc = ((lane >> 4) & 1) * 8 + ks * 16;
                ldmatrix_x4(a, xw + lr * kXsStride + lc);
                const uint2* bp = Ldp + ((size_t)(g * 4 + ks) * NT) * 32 + lane;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const uint2 b = __ldg(bp + t * 32);
                    mma_f16_16816(acc[t], a, b.x, b.y);
                }
            }
            __syncwarp();
        }
    }

    if constexpr (R > 0) {
        // fixed-order reduction of the warps' LoRA partials, then fp16 into the tile layout
        const int gid = lane >> 2, tig = lane & 3;
        float* rw = red + warp * kRows * R;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            rw[gid * R + 8 * t + 2 * tig] = acc[t][0];
            rw[gid * R + 8 * t + 2 * tig + 1] = acc[t][1];
            rw[(gid + 8) * R + 8 * t + 2 * tig] = acc[t][2];
            rw[(gid + 8) * R + 8 * t + 2 * tig + 1] = acc[t][3];
        }
        __syncthreads();
        uint16_t* La = reinterpret_cast<uint16_t*>(ws + AL.La);
        for (int idx = threadIdx.x; idx < kRows * R; idx += kWarps * 32) {
            const int row = idx / R, j = idx % R;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) v += red[w * kRows * R + idx];
            const int r2 = (row0 + row) % kTileM;
            const int p = j >> 4, jj = j & 15;
            La[((size_t)(mt * (R / 16) + p) * kTileM + r2) * 16 + swz32(r2, jj >> 3) * 8 + (jj & 7)] =
                __half_as_ushort(__float2half_rn(v));
        }
    }
}

__global__ void unpack_act_kernel(const uint8_t* __restrict__ ws, int M, int K, int r, int8_t* codes,
                                  float* sA, float* SA, float* lora) {
    const ActLayout AL = act_layout(M, K, r);
    const int G = K / kGroup;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < (long long)M * K) {
        const int m = int(i / K), k = int(i % K);
        const int mt = m / kTileM, rr = m % kTileM, g = k / kGroup, kk = k % kGroup;
        const uint8_t* plane = ws + AL.qA + ((size_t)(mt * G + g) * 2 + kk / 32) * (kTileM * 32);
        const int b = kk % 32;
        codes[i] = int8_t(int_of_e4m3(plane[rr * 32 + swz32(rr, b >> 4) * 16 + (b & 15)]));
        if (kk == 0) {
            const float2 v = *reinterpret_cast<const float2*>(ws + AL.sS + ((size_t)(mt * G + g) * kTileM + rr) * 8);
            sA[(size_t)m * G + g] = v.x;
            if (SA) SA[(size_t)m * G + g] = v.y;
        }
    }
    if (lora != nullptr && i < (long long)M * r) {
        const int m = int(i / r), j = int(i % r);
        const int mt = m / kTileM, rr = m % kTileM, p = j >> 4, jj = j & 15;
        const uint16_t h = reinterpret_cast<const uint16_t*>(ws + AL.La)
            [((size_t)(mt * (r / 16) + p) * kTileM + rr) * 16 + swz32(rr, jj >> 3) * 8 + (jj & 7)];
        lora[i] = __half2float(__ushort_as_half(h));
    }
}

template <int R>
w4a4_status launch_q(const uint16_t* X, const uint8_t* packed, int M, int K, uint8_t* ws, cudaStream_t s) {
    const size_t smem = kWarps * kRows * kXsStride * 2 + (size_t)kWarps * kRows * R * 4;
    static bool attr_set = false;  // per process; identical for every device
    if (!attr_set) {
        if (cudaFuncSetAttribute(quantize_act_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem)) != cudaSuccess)
            return W4A4_ERR_CUDA;
        attr_set = true;
    }
    const unsigned grid = unsigned((M + kRows - 1) / kRows);
    quantize_act_kernel<R><<<grid, kWarps * 32, smem, s>>>(X, reinterpret_cast<const uint2*>(packed), M, K, ws);
    set_dispatch("quantize_act rows/CTA=%d grid=%u rank=%d", kRows, grid, R);
    return launch_status();
}

}  // namespace

w4a4_status launch_quantize_act(const uint16_t* X, const uint8_t* packed, int M, int K, int r, uint8_t* ws,
                                cudaStream_t s) {
    switch (r) {
        case 0: return launch_q<0>(X, packed, M, K, ws, s);
        case 16: return launch_q<16>(X, packed, M, K, ws, s);
        case 32: return launch_q<32>(X, packed, M, K, ws, s);
        case 48: return launch_q<48>(X, packed, M, K, ws, s);
        case 64: return launch_q<64>(X, packed, M, K, ws, s);
        case 80: return launch_q<80>(X, packed, M, K, ws, s);
        case 96: return launch_q<96>(X, packed, M, K, ws, s);
        case 112: return launch_q<112>(X, packed, M, K, ws, s);
        case 128: return launch_q<128>(X, packed, M, K, ws, s);
        default: return W4A4_ERR_UNSUPPORTED_SHAPE;
    }
}

void launch_unpack_act(const uint8_t* ws, int M, int K, int r, int8_t* codes, float* sA, float* SA, float* lora,
                       cudaStream_t s) {
    long long n = (long long)M * K;
    if ((long long)M * r > n) n = (long long)M * r;
    unpack_act_kernel<<<unsigned((n + 255) / 256), 256, 0, s>>>(ws, M, K, r, codes, sA, SA, r ? lora : nullptr);
}

}  // namespace w4a4
