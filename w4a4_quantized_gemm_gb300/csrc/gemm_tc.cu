// W4A4 GEMM + LoRA up + column affine on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), for M above the small-M range.
//
// Computes, per 128 x 128 output tile ("W4A4 CUDA Kernel for Voice Clone",
// 3.7; "High-Performance Kernel Design for W4A4 ... on Blackwell", 1):
//   acc = lora_act . L_up  +  sum_g sW[n,g] (sA[m,g] D_g - 8 SA[m,g] sA[m,g])
//   D_g = sum_{k in g} E4M3(cA) * E4M3(cW + 8)     (exact, one group per TMEM buffer)
//   Y   = fp16(colscale * acc + bias)
//
// Structure (the warp-specialised persistent design of the Blackwell W4A4
// article, section 3.2, rebuilt for tcgen05): one CTA per SM walks tiles in a
// static round-robin; warps have fixed roles and talk through mbarriers:
//   warp 0      producer: 1-D bulk copies of activation codes, (sA, SA),
//               packed weight nibbles and scales into a STAGES-deep ring, and
//               the tile's LoRA operands;
//   warp 1      MMA issuer (one thread) + tensor-memory owner: per group two
//               kind::f8f6f4 MMAs (K = 32 each) into one of two TMEM buffers,
//               per tile one kind::f16 LoRA-up MMA chain;
//   warps 2-3   nibble -> E4M3 expansion of the weight tile into the
//               32-byte-swizzled B operand, fp16 -> fp32 weight scales;
//   warps 4-11  epilogue: TMEM -> registers, per-group scale-FMA into fp32
//               running sums (two warpgroups, 64 columns each), then the
//               column affine and the fp16 store.
// Every wait is bounded (2 s); on give-up the kernel records
// W4A4_ERR_TIMEOUT in its status word, unwinds every role, waits for its own
// copies and MMAs, frees tensor memory and returns.
#include "kernels.h"
#include "tc_ptx.cuh"

namespace w4a4 {

__device__ int g_tc_status = 0;

namespace {
using namespace tc;

constexpr int BN = 128;  // output columns per tile (MMA N)
constexpr int BM = 128;  // output rows per tile (MMA M, TMEM lanes)
constexpr int STAGES = 5;
constexpr int NUM_THREADS = 384;
constexpr int WARP_PRODUCER = 0, WARP_MMA = 1, WARP_EXPAND0 = 2, NUM_EXPAND_WARPS = 2;
constexpr int WARP_EPI0 = 4, NUM_EPI_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;  // two BN-column buffers used; whole TMEM held (one CTA per SM)
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;

// Shared-memory map (byte offsets from a 1024-aligned base).
constexpr uint32_t kStageA = 2 * BM * 32;  // 2 planes x 128 rows x 32 B
constexpr uint32_t kStageB = 2 * BN * 32;
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * kStageA;
constexpr uint32_t OFF_WP = OFF_B + STAGES * kStageB;
constexpr uint32_t OFF_SS = OFF_WP + STAGES * BN * 32;
constexpr uint32_t OFF_SW16 = OFF_SS + STAGES * BM * 8;
constexpr uint32_t OFF_SWF = OFF_SW16 + STAGES * BN * 2;
constexpr uint32_t OFF_LA = OFF_SWF + STAGES * BN * 4;
constexpr int kNumBars = 3 * STAGES + 7;

__host__ __device__ constexpr uint32_t off_lu(int rp) { return OFF_LA + uint32_t(rp) * BM * 32; }
__host__ __device__ constexpr uint32_t off_bar(int rp) { return (off_lu(rp) + uint32_t(rp) * BN * 32 + 7u) & ~7u; }
// + 1024 for aligning the base, + 8 KB of unused tail slack
__host__ __device__ constexpr uint32_t smem_bytes(int rp) { return off_bar(rp) + kNumBars * 8 + 8 + 1024 + 8192; }
static_assert(smem_bytes(8) <= 227 * 1024, "shared-memory budget exceeded at rank 128");

template <bool DUMP>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const uint8_t* __restrict__ ws, const uint8_t* __restrict__ packed,
                   const uint16_t* __restrict__ colscale, const uint16_t* __restrict__ bias, int M, int N, int K,
                   int r, uint16_t* __restrict__ Y, int32_t* __restrict__ P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const int RP = DUMP ? 0 : r / 16;
    const ActLayout AL = act_layout(M, K, r);
    const PackedLayout PL = packed_layout(N, K, r);
    const int MT = AL.MT, NT = (N + BN - 1) / BN;
    const int tiles = MT * NT;

    const uint32_t LU = off_lu(RP);
    const uint32_t BAR = off_bar(RP);
    auto full = [&](int s) { return base + BAR + 8u * s; };
    auto bready = [&](int s) { return base + BAR + 8u * (STAGES + s); };
    auto empty = [&](int s) { return base + BAR + 8u * (2 * STAGES + s); };
    auto tfull = [&](int b) { return base + BAR + 8u * (3 * STAGES + b); };
    auto tempty = [&](int b) { return base + BAR + 8u * (3 * STAGES + 2 + b); };
    const uint32_t lfull = base + BAR + 8u * (3 * STAGES + 4);
    const uint32_t lempty = base + BAR + 8u * (3 * STAGES + 5);
    const uint32_t mmadone = base + BAR + 8u * (3 * STAGES + 6);
    const uint32_t TSLOT = BAR + 8u * kNumBars;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + TSLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + TSLOT + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(bready(s), NUM_EXPAND_WARPS);
            mbar_init(empty(s), 1 + NUM_EPI_WARPS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), NUM_EPI_WARPS);
        }
        mbar_init(lfull, 1);
        mbar_init(lempty, 1);
        mbar_init(mmadone, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(base + TSLOT, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int no_abort = 0;

    auto fail = [&]() {
        atomicExch(&g_tc_status, int(W4A4_ERR_TIMEOUT));
        *abort_flag = 1;
    };

    if (warp == WARP_PRODUCER) {
        if (lane == 0) {
            uint32_t it = 0, lp = 0, lora_issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int mt = t % MT, n0 = (t / MT) * BN;
                const int rows = min(BN, N - n0);
                if (RP > 0) {
                    if (!wait_parity(lempty, lp ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(lfull, uint32_t(RP) * (BM * 32 + rows * 32));
                    bulk_g2s(base + OFF_LA, ws + AL.La + size_t(mt) * RP * (BM * 32), uint32_t(RP) * BM * 32, lfull);
                    for (int p = 0; p < RP; ++p)
                        bulk_g2s(base + LU + uint32_t(p) * BN * 32, packed + PL.Lu + (size_t(p) * N + n0) * 32,
                                 uint32_t(rows) * 32, lfull);
                    lp ^= 1u;
                    lora_issued = 1;
                }
                for (int g = 0; g < G; ++g) {
                    const int s = int(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_parity(empty(s), ph ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(full(s), kStageA + BM * 8 + uint32_t(rows) * 34);
                    const size_t ag = size_t(mt) * G + g;
                    bulk_g2s(base + OFF_A + s * kStageA, ws + AL.qA + ag * kStageA, kStageA, full(s));
                    bulk_g2s(base + OFF_SS + s * (BM * 8), ws + AL.sS + ag * (BM * 8), BM * 8, full(s));
                    bulk_g2s(base + OFF_WP + s * (BN * 32), packed + PL.qW + (size_t(g) * N + n0) * 32,
                             uint32_t(rows) * 32, full(s));
                    bulk_g2s(base + OFF_SW16 + s * (BN * 2), packed + PL.sW + (size_t(g) * N + n0) * 2,
                             uint32_t(rows) * 2, full(s));
                    ++it;
                }
            }
            if (!ok) fail();
            // drain: the copies of the last STAGES iterations (distinct stages) and the last LoRA load
            for (uint32_t k = (it > STAGES ? it - STAGES : 0u); k < it; ++k)
                wait_parity(full(int(k % STAGES)), (k / STAGES) & 1u, &no_abort, DRAIN_LIMIT_NS);
            if (lora_issued) wait_parity(lfull, lp ^ 1u, &no_abort, DRAIN_LIMIT_NS);
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_m128(BN);
            uint32_t it = 0, jc = 0, lp = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                if (RP > 0) {
                    const uint32_t b = jc & 1u, tph = (jc >> 1) & 1u;
                    if (!wait_parity(tempty(b), tph ^ 1u, abort_flag, WAIT_LIMIT_NS) ||
                        !wait_parity(lfull, lp, abort_flag, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int p = 0; p < RP; ++p)
                        mma_f16(tmem + b * BN, sdesc_sw32(base + OFF_LA + uint32_t(p) * BM * 32),
                                sdesc_sw32(base + LU + uint32_t(p) * BN * 32), IDESC, p > 0 ? 1u : 0u);
                    mma_commit(tfull(b));
                    mma_commit(lempty);
                    ++jc;
                    lp ^= 1u;
                }
                for (int g = 0; g < G; ++g) {
                    const int s = int(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    const uint32_t b = jc & 1u, tph = (jc >> 1) & 1u;
                    if (!wait_parity(full(s), ph, abort_flag, WAIT_LIMIT_NS) ||
                        !wait_parity(bready(s), ph, abort_flag, WAIT_LIMIT_NS) ||
                        !wait_parity(tempty(b), tph ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = base + OFF_A + s * kStageA, b0 = base + OFF_B + s * kStageB;
                    mma_f8(tmem + b * BN, sdesc_sw32(a0), sdesc_sw32(b0), IDESC, 0u);
                    mma_f8(tmem + b * BN, sdesc_sw32(a0 + BM * 32), sdesc_sw32(b0 + BN * 32), IDESC, 1u);
                    mma_commit(empty(s));
                    mma_commit(tfull(b));
                    ++it;
                    ++jc;
                }
            }
            if (!ok) fail();
            mma_commit(mmadone);  // every MMA issued above has completed once this arrives
            wait_parity(mmadone, 0u, &no_abort, DRAIN_LIMIT_NS);
        }
    } else if (warp < WARP_EPI0) {
        // ---- expansion: packed offset-binary nibbles -> E4M3 B operand planes
        const int et = (warp - WARP_EXPAND0) * 32 + lane;
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
            for (int g = 0; g < G; ++g) {
                const int s = int(it % STAGES);
                const uint32_t ph = (it / STAGES) & 1u;
                if (!wait_parity(full(s), ph, abort_flag, WAIT_LIMIT_NS)) {
                    ok = false;
                    break;
                }
                uint8_t* bp = gbase + OFF_B + s * kStageB;
                const uint8_t* wp = gbase + OFF_WP + s * (BN * 32);
                const uint16_t* sw16 = reinterpret_cast<const uint16_t*>(gbase + OFF_SW16 + s * (BN * 2));
                float* swf = reinterpret_cast<float*>(gbase + OFF_SWF + s * (BN * 4));
#pragma unroll
                for (int row = et; row < BN; row += NUM_EXPAND_WARPS * 32) {
                    const uint4 w01 = *reinterpret_cast<const uint4*>(wp + row * 32);
                    const uint4 w23 = *reinterpret_cast<const uint4*>(wp + row * 32 + 16);
                    // words: w01 = (q0h0, q0h1, q1h0, q1h1), w23 = (q2h0, q2h1, q3h0, q3h1)
                    const uint4 p0c0 = make_uint4(expand4(w01.x), expand4(w01.z), expand4(w23.x), expand4(w23.z));
                    const uint4 p0c1 = make_uint4(expand4(w01.x >> 16), expand4(w01.z >> 16), expand4(w23.x >> 16),
                                                  expand4(w23.z >> 16));
                    const uint4 p1c0 = make_uint4(expand4(w01.y), expand4(w01.w), expand4(w23.y), expand4(w23.w));
                    const uint4 p1c1 = make_uint4(expand4(w01.y >> 16), expand4(w01.w >> 16), expand4(w23.y >> 16),
                                                  expand4(w23.w >> 16));
                    *reinterpret_cast<uint4*>(bp + row * 32 + swz32(row, 0) * 16) = p0c0;
                    *reinterpret_cast<uint4*>(bp + row * 32 + swz32(row, 1) * 16) = p0c1;
                    *reinterpret_cast<uint4*>(bp + BN * 32 + row * 32 + swz32(row, 0) * 16) = p1c0;
                    *reinterpret_cast<uint4*>(bp + BN * 32 + row * 32 + swz32(row, 1) * 16) = p1c1;
                    swf[row] = __half2float(__ushort_as_half(sw16[row]));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bready(s));
                ++it;
            }
        }
        if (!ok) fail();
    } else {
        // ---- epilogue
        const int ew = warp - WARP_EPI0;
        const int c0 = (ew >> 2) * 64;  // column half of the tile
        const int lq = warp & 3;        // TMEM lane quarter this warp may access
        const int row = lq * 32 + lane;
        const uint32_t tl = tmem + (uint32_t(lq * 32) << 16) + uint32_t(c0);
        uint32_t it = 0, jc = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
            const int mt = t % MT, n0 = (t / MT) * BN;
            const int m = mt * BM + row;
            float acc[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) acc[c] = 0.f;
            if (RP > 0) {
                const uint32_t b = jc & 1u, tph = (jc >> 1) & 1u;
                if (!wait_parity(tfull(b), tph, abort_flag, WAIT_LIMIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                __syncwarp();
                float v0[32], v1[32];
                tmem_ld32(tl + b * BN, v0);
                tmem_ld32(tl + b * BN + 32, v1);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty(b));
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    acc[c] = v0[c];
                    acc[32 + c] = v1[c];
                }
                ++jc;
            }
            for (int g = 0; g < G; ++g) {
                const int s = int(it % STAGES);
                const uint32_t ph = (it / STAGES) & 1u;
                const uint32_t b = jc & 1u, tph = (jc >> 1) & 1u;
                if (!wait_parity(tfull(b), tph, abort_flag, WAIT_LIMIT_NS) ||
                    !wait_parity(full(s), ph, abort_flag, WAIT_LIMIT_NS) ||
                    !wait_parity(bready(s), ph, abort_flag, WAIT_LIMIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                __syncwarp();
                float v[64];
                {
                    float v0[32], v1[32];
                    tmem_ld32(tl + b * BN, v0);
                    tmem_ld32(tl + b * BN + 32, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        v[c] = v0[c];
                        v[32 + c] = v1[c];
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty(b));
                const float2 sv = reinterpret_cast<const float2*>(gbase + OFF_SS + s * (BM * 8))[row];
                if constexpr (DUMP) {
                    if (m < M) {
#pragma unroll
                        for (int c = 0; c < 64; ++c) {
                            const int n = n0 + c0 + c;
                            if (n < N) P[(size_t(m) * N + n) * G + g] = int32_t(v[c] - 8.f * sv.y);
                        }
                    }
                } else {
                    const float cm = (-8.f * sv.y) * sv.x;
                    const float2 sa2 = make_float2(sv.x, sv.x), cm2 = make_float2(cm, cm);
                    const float4* swf = reinterpret_cast<const float4*>(gbase + OFF_SWF + s * (BN * 4) + c0 * 4);
#pragma unroll
                    for (int c4 = 0; c4 < 16; ++c4) {
                        const float4 w = swf[c4];
                        const float2 t0 = ffma2(sa2, make_float2(v[4 * c4], v[4 * c4 + 1]), cm2);
                        const float2 t1 = ffma2(sa2, make_float2(v[4 * c4 + 2], v[4 * c4 + 3]), cm2);
                        const float2 a0 = ffma2(make_float2(w.x, w.y), t0, make_float2(acc[4 * c4], acc[4 * c4 + 1]));
                        const float2 a1 =
                            ffma2(make_float2(w.z, w.w), t1, make_float2(acc[4 * c4 + 2], acc[4 * c4 + 3]));
                        acc[4 * c4] = a0.x;
                        acc[4 * c4 + 1] = a0.y;
                        acc[4 * c4 + 2] = a1.x;
                        acc[4 * c4 + 3] = a1.y;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty(s));
                ++it;
                ++jc;
            }
            if (!ok) break;
            if constexpr (!DUMP) {
                if (m < M) {
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const int n = n0 + c0 + ch * 8;
                        if (n < N) {
                            const uint4 csv = __ldg(reinterpret_cast<const uint4*>(colscale + n));
                            const uint4 bsv =
                                bias ? __ldg(reinterpret_cast<const uint4*>(bias + n)) : make_uint4(0, 0, 0, 0);
                            const uint32_t cw[4] = {csv.x, csv.y, csv.z, csv.w};
                            const uint32_t bw[4] = {bsv.x, bsv.y, bsv.z, bsv.w};
                            uint32_t out[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float2 cs2 = __half22float2(*reinterpret_cast<const __half2*>(&cw[j]));
                                const float2 b2 = __half22float2(*reinterpret_cast<const __half2*>(&bw[j]));
                                const float y0 = fmaf(cs2.x, acc[ch * 8 + 2 * j], b2.x);
                                const float y1 = fmaf(cs2.y, acc[ch * 8 + 2 * j + 1], b2.y);
                                const __half2 h = __floats2half2_rn(y0, y1);
                                out[j] = *reinterpret_cast<const uint32_t*>(&h);
                            }
                            *reinterpret_cast<uint4*>(Y + size_t(m) * N + n) =
                                make_uint4(out[0], out[1], out[2], out[3]);
                        }
                    }
                }
            }
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == WARP_MMA) tmem_dealloc(tmem, TMEM_COLS);
}

template <bool DUMP>
w4a4_status launch_impl(const uint8_t* ws, const uint8_t* packed, const uint16_t* cs, const uint16_t* bias, int M,
                        int N, int K, int r, uint16_t* Y, int32_t* P, cudaStream_t s) {
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(gemm_tc_kernel<DUMP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem_bytes(8))) != cudaSuccess)
            return W4A4_ERR_CUDA;
        attr_done[dev] = 1;
    }
    const int rp = DUMP ? 0 : r / 16;
    const int MT = (M + BM - 1) / BM, NT = (N + BN - 1) / BN;
    const int tiles = MT * NT;
    const int grid = tiles < device_sm_count() ? tiles : device_sm_count();
    gemm_tc_kernel<DUMP><<<grid, NUM_THREADS, smem_bytes(rp), s>>>(ws, packed, cs, bias, M, N, K, r, Y, P);
    set_dispatch("gemm_tc tcgen05.f8f6f4 tile=%dx%d stages=%d tiles=%d grid=%d%s", BM, BN, STAGES, tiles, grid,
                 DUMP ? " (partials dump)" : "");
    return launch_status();
}

}  // namespace

w4a4_status launch_gemm_tc(const uint8_t* ws, const uint8_t* packed, const uint16_t* colscale, const uint16_t* bias,
                           int M, int N, int K, int r, uint16_t* Y, int32_t* P_dump, cudaStream_t s) {
    if (P_dump) return launch_impl<true>(ws, packed, colscale, bias, M, N, K, r, Y, P_dump, s);
    return launch_impl<false>(ws, packed, colscale, bias, M, N, K, r, Y, nullptr, s);
}

w4a4_status tc_read_and_clear_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int));
        return W4A4_ERR_TIMEOUT;
    }
    return W4A4_OK;
}

}  // namespace w4a4
