// Offline weight packing: INT4 quantisation of W with fp16 per-group scales,
// nibble packing in the order both GEMM kernels read, and the LoRA factors in
// tensor-core-ready layouts.  Runs once per layer ("W4A4 CUDA Kernel for Voice
// Clone", 3.10: weights are repacked once at model load; "INT4 Kernel
// Architecture, in depth", "How the weights are stored").
#include "kernels.h"

namespace w4a4 {
namespace {

// Position of code k (0..63 within a group) in the 32-byte record: word index
// (8*q + 4*h)/4 and nibble j, inverse of the formula in include/w4a4.h.
__host__ __device__ inline void code_slot(int k, int& word, int& nib) {
    int h = k >> 5, kk = k & 31;
    int q = (kk & 15) >> 2;
    int j = ((kk >> 4) << 2) | (kk & 3);
    word = 2 * q + h;
    nib = j;
}

// Record word `lane` (lanes 0..7) of a 64-group whose codes 2l and 2l + 1 lane l
// holds as nibbles u0, u1 (word and nibble order as in include/w4a4.h).
__device__ __forceinline__ uint32_t gather_record_word(uint32_t u0, uint32_t u1, int lane) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        // lane w (< 8) wants nibble j of word w: k = 32 h + (j<4 ? 4q+j : 16+4q+j-4)
        int w = lane & 7, q = w >> 1, h = w & 1;
        int k = 32 * h + (j < 4 ? 4 * q + j : 16 + 4 * q + (j - 4));
        uint32_t v0 = __shfl_sync(0xffffffffu, u0, k >> 1);
        uint32_t v1 = __shfl_sync(0xffffffffu, u1, k >> 1);
        word |= ((k & 1) ? v1 : v0) << (4 * j);
    }
    return word;
}

// One warp per (group g, row n): lane l owns k = 2l, 2l+1 of the group.
// silu_I > 0: the rows of a fused gate|up W (I gate rows, then I up rows) in the
// order of the SiLU(gate) * up epilogue (gate_up_row).
__global__ void __launch_bounds__(256) pack_weights_kernel(const float* __restrict__ W,
                                                           const int8_t* __restrict__ codes,
                                                           const uint16_t* __restrict__ scales, int N,
                                                           int K, int silu_I, uint32_t* __restrict__ qW,
                                                           uint16_t* __restrict__ sW) {
    const int lane = threadIdx.x & 31;
    const long long task = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int G = K / kGroup;
    if (task >= (long long)G * N) return;
    const int g = int(task / N), n = int(task % N);
    const int src = silu_I > 0 ? gate_up_row(n, silu_I) : n;
    const size_t base = (size_t)src * K + (size_t)g * kGroup + 2 * lane;

    int q0, q1;
    uint16_t sbits;
    if (W != nullptr) {
        float w0 = W[base], w1 = W[base + 1];
        float amax = fmaxf(fabsf(w0), fabsf(w1));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        // scale = fp16(max(absmax / 7, 2^-14)); codes against the stored fp16 value
        float s32 = fmaxf(__fdiv_rn(amax, 7.0f), 6.103515625e-05f);
        __half hs = __float2half_rn(s32);
        float s = __half2float(hs);
        q0 = int(fminf(fmaxf(rintf(__fdiv_rn(w0, s)), -8.0f), 7.0f));
        q1 = int(fminf(fmaxf(rintf(__fdiv_rn(w1, s)), -8.0f), 7.0f));
        sbits = __half_as_ushort(hs);
    } else {
        q0 = codes[base];
        q1 = codes[base + 1];
        sbits = scales[(size_t)n * G + g];
    }
    // offset-binary nibbles, gathered by lanes 0..7 (one 32-bit word each)
    const uint32_t word = gather_record_word(uint32_t(q0 + 8) & 15u, uint32_t(q1 + 8) & 15u, lane);
    if (lane < 8) qW[((size_t)g * N + n) * 8 + lane] = word;
    if (lane == 0) sW[(size_t)g * N + n] = sbits;
}

// Asymmetric 4-bit weights, groups of 128 ("INT4 Kernel Architecture, in
// depth", "How the weights are stored"): one warp per (128-group g, row n);
// lane l owns k = 2l, 2l+1 of each 64-half.  scale = max(hi - lo, 1e-8) / 15,
// zero = rint(-lo / scale) (+0 for a zero point of 0), code u = clamp(rint(w /
// scale + zero), 0, 15), all in IEEE binary32.  The codes go into the two
// 64-group records as plain nibbles u; the scale plane holds fp16(scale) in
// the first half's slot and fp16(zero) in the second's.  A zero point outside
// [-1024, 1023] (where 1024 + zero stops being exact in fp16) is flagged.
__device__ int g_pack_asym_zero_range = 0;

__global__ void __launch_bounds__(256) pack_weights_asym_kernel(const float* __restrict__ W, int N, int K,
                                                                uint32_t* __restrict__ qW,
                                                                uint16_t* __restrict__ sW) {
    const int lane = threadIdx.x & 31;
    const long long task = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int GA = K / (2 * kGroup);
    if (task >= (long long)GA * N) return;
    const int g = int(task / N), n = int(task % N);
    const float* wr = W + (size_t)n * K + (size_t)g * 2 * kGroup;
    const float2 a = *reinterpret_cast<const float2*>(wr + 2 * lane);
    const float2 b = *reinterpret_cast<const float2*>(wr + kGroup + 2 * lane);
    float lo = fminf(fminf(a.x, a.y), fminf(b.x, b.y)), hi = fmaxf(fmaxf(a.x, a.y), fmaxf(b.x, b.y));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const float sc = __fdiv_rn(fmaxf(__fsub_rn(hi, lo), 1e-8f), 15.0f);
    const float z = __fadd_rn(rintf(__fdiv_rn(-lo, sc)), 0.0f);
    auto code = [&](float w) { return uint32_t(fminf(fmaxf(rintf(__fadd_rn(__fdiv_rn(w, sc), z)), 0.0f), 15.0f)); };
    const uint32_t w0 = gather_record_word(code(a.x), code(a.y), lane);
    const uint32_t w1 = gather_record_word(code(b.x), code(b.y), lane);
    const size_t g0 = (size_t)2 * g;
    if (lane < 8) {
        qW[(g0 * N + n) * 8 + lane] = w0;
        qW[((g0 + 1) * N + n) * 8 + lane] = w1;
    }
    if (lane == 0) {
        sW[g0 * N + n] = __half_as_ushort(__float2half_rn(sc));
        sW[(g0 + 1) * N + n] = __half_as_ushort(__float2half_rn(z));
        if (z < -1024.0f || z > 1023.0f) atomicExch(&g_pack_asym_zero_range, 1);
    }
}

// L_down -> B-operand fragments of mma.m16n8k16: [K/16][r/8][32][2] words.
__global__ void pack_ldown_kernel(const uint16_t* __restrict__ Ld, int K, int r, uint32_t* __restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total = (long long)(K / 16) * (r / 8) * 64;
    if (i >= total) return;
    const int w = int(i & 1), L = int((i >> 1) & 31);
    const long long st = i >> 6;
    const int t = int(st % (r / 8)), s = int(st / (r / 8));
    const int k = 16 * s + 2 * (L & 3) + 8 * w, j = 8 * t + (L >> 2);
    out[i] = uint32_t(Ld[(size_t)k * r + j]) | (uint32_t(Ld[(size_t)(k + 1) * r + j]) << 16);
}

// L_up [r, N] -> [r/16][N][32 bytes] with the 32-byte swizzle (silu_I > 0:
// column n of the packed weights' order, gate_up_row).
__global__ void pack_lup_kernel(const uint16_t* __restrict__ Lu, int N, int r, int silu_I,
                                uint16_t* __restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)r * N) return;
    const int j = int(i / N), n = int(i % N);
    const int p = j >> 4, jj = j & 15;
    const int chunk = swz32(n, jj >> 3);
    const int src = silu_I > 0 ? gate_up_row(n, silu_I) : n;
    out[((size_t)p * N + n) * 16 + chunk * 8 + (jj & 7)] = Lu[(size_t)j * N + src];
}

// ---- debug: packed buffer -> logical tensors ------------------------------
__global__ void unpack_weights_kernel(const uint8_t* __restrict__ packed, int N, int K, int r,
                                      int8_t* __restrict__ codes, uint16_t* __restrict__ scales,
                                      uint16_t* __restrict__ Ld, uint16_t* __restrict__ Lu) {
    const PackedLayout PL = packed_layout(N, K, r);
    const int G = K / kGroup;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < (long long)N * K) {
        const int n = int(i / K), kk = int(i % K);
        const int g = kk / kGroup;
        int word, nib;
        code_slot(kk % kGroup, word, nib);
        const uint32_t* rec = reinterpret_cast<const uint32_t*>(packed + PL.qW) + ((size_t)g * N + n) * 8;
        codes[i] = int8_t(int((rec[word] >> (4 * nib)) & 15u) - 8);
        if (kk % kGroup == 0)
            scales[(size_t)n * G + g] = reinterpret_cast<const uint16_t*>(packed + PL.sW)[(size_t)g * N + n];
    }
    if (Ld != nullptr && i < (long long)K * r) {
        const int k = int(i / r), j = int(i % r);
        const int s = k / 16, kr = k % 16, w = kr / 8, L2 = (kr % 8) / 2, lo = kr & 1;
        const int t = j / 8, L = (j % 8) * 4 + L2;
        const uint32_t v = reinterpret_cast<const uint32_t*>(packed + PL.Ld)[(((size_t)s * (r / 8) + t) * 32 + L) * 2 + w];
        Ld[i] = uint16_t(lo ? (v >> 16) : (v & 0xffffu));
    }
    if (Lu != nullptr && i < (long long)r * N) {
        const int j = int(i / N), n = int(i % N);
        const int p = j >> 4, jj = j & 15;
        Lu[i] = reinterpret_cast<const uint16_t*>(packed + PL.Lu)[((size_t)p * N + n) * 16 + swz32(n, jj >> 3) * 8 + (jj & 7)];
    }
}

inline unsigned blocks_for(long long n, int per) { return unsigned((n + per - 1) / per); }

}  // namespace

void launch_pack_weights(const float* W, const int8_t* codes, const uint16_t* scales, int N, int K, int r,
                         int silu_I, uint8_t* packed, cudaStream_t s) {
    const PackedLayout PL = packed_layout(N, K, r);
    const long long tasks = (long long)(K / kGroup) * N;
    pack_weights_kernel<<<blocks_for(tasks, 8), 256, 0, s>>>(
        W, codes, scales, N, K, silu_I, reinterpret_cast<uint32_t*>(packed + PL.qW),
        reinterpret_cast<uint16_t*>(packed + PL.sW));
}

w4a4_status launch_pack_weights_asym(const float* W, int N, int K, int r, uint8_t* packed, cudaStream_t s) {
    const PackedLayout PL = packed_layout(N, K, r);
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_pack_asym_zero_range, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return W4A4_ERR_CUDA;
    const long long tasks = (long long)(K / (2 * kGroup)) * N;
    pack_weights_asym_kernel<<<blocks_for(tasks, 8), 256, 0, s>>>(
        W, N, K, reinterpret_cast<uint32_t*>(packed + PL.qW), reinterpret_cast<uint16_t*>(packed + PL.sW));
    if (cudaGetLastError() != cudaSuccess) return W4A4_ERR_CUDA;
    int bad = 0;
    if (cudaMemcpyFromSymbolAsync(&bad, g_pack_asym_zero_range, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return W4A4_ERR_CUDA;
    return bad ? W4A4_ERR_INVALID_ARG : W4A4_OK;
}

void launch_pack_lora(const uint16_t* L_down, const uint16_t* L_up, int N, int K, int r, int silu_I,
                      uint8_t* packed, cudaStream_t s) {
    if (r == 0) return;
    const PackedLayout PL = packed_layout(N, K, r);
    const long long nld = (long long)(K / 16) * (r / 8) * 64;
    pack_ldown_kernel<<<blocks_for(nld, 256), 256, 0, s>>>(L_down, K, r,
                                                           reinterpret_cast<uint32_t*>(packed + PL.Ld));
    pack_lup_kernel<<<blocks_for((long long)r * N, 256), 256, 0, s>>>(L_up, N, r, silu_I,
                                                                      reinterpret_cast<uint16_t*>(packed + PL.Lu));
}

void launch_unpack_weights(const uint8_t* packed, int N, int K, int r, int8_t* codes, uint16_t* scales,
                           uint16_t* L_down, uint16_t* L_up, cudaStream_t s) {
    long long n = (long long)N * K;
    if ((long long)K * r > n) n = (long long)K * r;
    if ((long long)r * N > n) n = (long long)r * N;
    unpack_weights_kernel<<<blocks_for(n, 256), 256, 0, s>>>(packed, N, K, r, codes, scales,
                                                             r ? L_down : nullptr, r ? L_up : nullptr);
}

}  // namespace w4a4
