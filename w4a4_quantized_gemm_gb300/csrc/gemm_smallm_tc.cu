// Weight-streaming W4A4 GEMM for small M on the 5th-generation tensor cores:
// the weights are the MMA's 128-row operand and the tokens its N (16, 32 or
// 64), so one tcgen05 MMA covers 128 weight rows x all tokens x 32 k with the
// products landing in tensor memory ("INT4 Kernel Architecture, in depth",
// "One token versus a thousand": swap the operands so that the small
// dimension is N; "W4A4 CUDA Kernel for Voice Clone", 3.7: exact per-group
// products, scaled per group, LoRA up into the same accumulator).
//
// Per group g, D[n, m] = 2^-9 sum_k (cW[n,k] + 8) * cA[m,k] exactly in its own
// tensor-memory buffer (the weight bytes are the offset codes themselves, which
// E4M3 reads as u * 2^-9), and the epilogue adds sW[n,g] (2^9 sA[m,g] D - 8 SA sA)
// to fp32 sums held in registers (one thread per weight row, one column pair
// per two tokens).
//
// CTA: 128 weight rows x one token block x a K slice; K is split over a
// cluster of KS CTAs as in the warp-MMA small-M kernel.  Roles (10 warps):
//   warps 0-3  expand the weight nibbles of their 32 rows into the E4M3 A
//              operand (32-byte swizzled K-major planes);
//   warp 4     producer: 1-D bulk copies of each group's weight records,
//              weight scales, the token block's codes and (sA, SA), in an
//              S-deep ring; on rank 0 the LoRA planes;
//   warp 5     tensor-memory owner and MMA issuer (one thread): on rank 0 a
//              kind::f16 LoRA-up chain, then per group two kind::f8f6f4 MMAs;
//   warps 6-9  epilogue, one tensor-memory lane quarter each (warp w: rows
//              32 (w % 4) ...), running one group behind the expansion, so the
//              two overlap; then the exchange, the affine and the store.
// The partial sums are exchanged in blocks of 4 tokens: block b belongs to
// cluster rank b % KS, the other ranks push their fp32 sums there with
// st.async, and the owner adds them in rank order before the affine and the
// store.  Every wait is bounded (2 s; W4A4_ERR_TIMEOUT in the status word); on
// give-up every role unwinds, the MMA issuer waits for its MMAs, tensor
// memory is freed, and the cluster barriers (reached by every thread on every
// path) keep peers' shared memory alive.
#include "kernels.h"
#include "tc_ptx.cuh"

namespace w4a4 {
namespace {
using namespace tc;

constexpr int kRows = 128;  // weight rows per CTA (MMA M, tensor-memory lanes)
constexpr int kThreads = 320;
constexpr int WARP_PROD = 4, WARP_MMA = 5, WARP_EPI0 = 6;
constexpr int kMaxKS = 8;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kSuspendNs = 20000;

__device__ int g_smtc_status = 0;

// Byte offsets of the shared-memory sections (all multiples of 16; the E4M3
// planes and the LoRA planes, read by the tensor core, at multiples of 1024).
struct TcPlan {
    uint32_t wexp, lu, la, wraw, aq, sa, sw, red, bar, total;
    uint32_t tmem_cols;
};
// Stages: 4, or 3 for 64 tokens, so that (stages + 1) x tokens tensor-memory
// columns round up to at most 256 and two CTAs' allocations fit one SM.
__host__ __device__ constexpr int stages_for(int tokn) { return tokn >= 64 ? 3 : 4; }

__host__ __device__ inline TcPlan tc_plan(int tokn, int r, int ks) {
    TcPlan p;
    const int kS = stages_for(tokn);
    uint32_t o = 0;
    p.wexp = o, o += kS * 2 * kRows * 32;             // [stage][plane][128 rows][32 B]
    p.lu = o, o += uint32_t(r / 16) * kRows * 32;     // [plane][128 rows][32 B]
    p.la = o, o += uint32_t(r / 16) * tokn * 32;      // [plane][tokn][32 B]
    o = (o + 1023u) & ~1023u;
    p.aq = o, o += kS * 2 * tokn * 32;                // [stage][plane][tokn][32 B]
    p.wraw = o, o += kS * kRows * 32;                 // [stage][128 rows][32 B]
    p.sa = o, o += kS * tokn * 8;                     // [stage][tokn] (sA, SA) -> (sA[], cc[]) in place
    p.sw = o, o += kS * kRows * 2;                    // [stage][128] fp16
    const int blocks = tokn / 4, own = (blocks + ks - 1) / ks;
    p.red = o, o += uint32_t(ks > 1 ? ks - 1 : 0) * kRows * own * 16;  // [sender][row][owned block] float4
    p.bar = o, o += 256;                              // full, expd, tfull, sfree [stages]; lfull, tlora, mmadone, red_full
    p.total = o;
    const uint32_t need = uint32_t((kS + 1) * tokn);
    p.tmem_cols = need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : 256;
    return p;
}

// DUMP: the debug variant, which also writes every group's exact integer product to
// P and stores no Y (colscale and bias are not read).
template <int TOKN, bool DUMP>
__global__ void __launch_bounds__(kThreads, TOKN >= 64 ? 1 : 2) gemm_smallm_tc_kernel(
    const uint8_t* __restrict__ ws, const uint8_t* __restrict__ packed, const uint16_t* __restrict__ colscale,
    const uint16_t* __restrict__ bias, int M, int N, int K, int r, uint16_t* __restrict__ Y,
    int32_t* __restrict__ P, int KS, int silu_I) {
    constexpr int BLK = TOKN / 4;  // 4-token blocks
    constexpr int kS = stages_for(TOKN);
    extern __shared__ uint8_t smdyn[];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag, never_abort;
    const TcPlan PLN = tc_plan(TOKN, r, KS);
    // the tensor core's operands want 1024-byte aligned planes: align the dynamic region by hand
    const uint32_t raw = smem_u32(smdyn);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smraw = smdyn + (sbase - raw);
    const uint32_t bar0 = sbase + PLN.bar;
    auto full = [&](int s) { return bar0 + 8u * s; };              // copies landed
    auto expd = [&](int s) { return bar0 + 8u * (kS + s); };       // A operand expanded (4 warps)
    auto tfull = [&](int s) { return bar0 + 8u * (2 * kS + s); };  // MMAs of the stage done
    auto sfree = [&](int s) { return bar0 + 8u * (3 * kS + s); };  // epilogue done with stage + buffer
    const uint32_t lfull = bar0 + 8u * (4 * kS), tlora = lfull + 8u, mmadone = lfull + 16u, red_full = lfull + 24u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const ActLayout AL = act_layout(M, K, r);
    const PackedLayout PL = packed_layout(N, K, r);
    const int kr = KS > 1 ? int(cluster_ctarank()) : 0;
    const int ntile = blockIdx.x / KS;
    const int g_begin = (G * kr) / KS, n_groups = (G * (kr + 1)) / KS - g_begin;
    const int tok0 = blockIdx.y * TOKN;
    const int mt = tok0 / kTileM, rt0 = tok0 % kTileM;
    const int nbase = ntile * kRows;
    const int rows_valid = min(kRows, N - nbase);  // a multiple of 16
    const int RP = (kr == 0) ? r / 16 : 0;         // the LoRA term is added by rank 0 only
    volatile int* abort = &abort_flag;
    constexpr uint32_t IDESC = idesc_m128(TOKN);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        never_abort = 0;
        for (int s = 0; s < kS; ++s) {
            mbar_init(full(s), 1);
            mbar_init(expd(s), 4);
            mbar_init(tfull(s), 1);
            mbar_init(sfree(s), 4);
        }
        mbar_init(lfull, 1);
        mbar_init(tlora, 1);
        mbar_init(mmadone, 1);
        mbar_init(red_full, 1);
        fence_mbar_init();
        if (KS > 1) {
            int owned = 0;
            for (int b = 0; b < BLK; ++b) owned += (b % KS == kr);
            mbar_expect_tx(red_full, uint32_t((KS - 1) * kRows * owned * 16));
        }
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(&tmem_slot), PLN.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (KS > 1) cluster_arrive_release();
    // The setup above touches only this CTA's shared and tensor memory and overlaps
    // the previous kernel; so does warming L2 with this CTA's share of the weight
    // records and scales (a prefetch only fills the cache; the copies come after the wait).
    if (warp == WARP_PROD && lane == 0) {
        for (int i = 0; i < n_groups; ++i) {
            prefetch_l2(packed + PL.qW + ((size_t)(g_begin + i) * N + nbase) * 32, uint32_t(rows_valid) * 32);
            prefetch_l2(packed + PL.sW + ((size_t)(g_begin + i) * N + nbase) * 2, uint32_t(rows_valid) * 2);
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    bool ok = true;

    if (warp == WARP_PROD) {
        if (lane == 0) {
            if (RP > 0) {
                mbar_expect_tx(lfull, uint32_t(RP) * (rows_valid * 32 + TOKN * 32));
                for (int p = 0; p < RP; ++p) {
                    bulk_g2s(sbase + PLN.lu + p * (kRows * 32), packed + PL.Lu + ((size_t)p * N + nbase) * 32,
                             rows_valid * 32, lfull);
                    bulk_g2s(sbase + PLN.la + p * (TOKN * 32),
                             ws + AL.La + ((size_t)(mt * (r / 16) + p) * kTileM + rt0) * 32, TOKN * 32, lfull);
                }
            }
            for (int i = 0; i < n_groups && ok; ++i) {
                const int s = i % kS;
                const uint32_t ph = uint32_t(i / kS) & 1u;
                if (i >= kS && !wait_parity_suspend(sfree(s), ph ^ 1u, abort, kWaitNs, kSuspendNs)) {
                    ok = false;
                    break;
                }
                const int g = g_begin + i;
                const uint32_t bytes = uint32_t(rows_valid) * 34 + 2u * TOKN * 32 + TOKN * 8;
                mbar_expect_tx(full(s), bytes);
                bulk_g2s(sbase + PLN.wraw + s * (kRows * 32), packed + PL.qW + ((size_t)g * N + nbase) * 32,
                         rows_valid * 32, full(s));
                bulk_g2s(sbase + PLN.sw + s * (kRows * 2), packed + PL.sW + ((size_t)g * N + nbase) * 2,
                         rows_valid * 2, full(s));
                const uint8_t* qa = ws + AL.qA + (size_t)(mt * G + g) * 2 * (kTileM * 32) + (size_t)rt0 * 32;
                bulk_g2s(sbase + PLN.aq + s * (2 * TOKN * 32), qa, TOKN * 32, full(s));
                bulk_g2s(sbase + PLN.aq + s * (2 * TOKN * 32) + TOKN * 32, qa + kTileM * 32, TOKN * 32, full(s));
                bulk_g2s(sbase + PLN.sa + s * (TOKN * 8), ws + AL.sS + ((size_t)(mt * G + g) * kTileM + rt0) * 8,
                         TOKN * 8, full(s));
            }
            if (!ok) {
                atomicExch(&g_smtc_status, int(W4A4_ERR_TIMEOUT));
                *abort = 1;
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            if (RP > 0) {
                if (!wait_parity_suspend(lfull, 0u, abort, kWaitNs, kSuspendNs)) {
                    ok = false;
                } else {
                    tc_fence_after();
                    for (int p = 0; p < RP; ++p)
                        mma_f16(tmem + uint32_t(kS * TOKN), sdesc_sw32(sbase + PLN.lu + p * (kRows * 32)),
                                sdesc_sw32(sbase + PLN.la + p * (TOKN * 32)), IDESC, p > 0 ? 1u : 0u);
                    mma_commit(tlora);
                }
            }
            for (int i = 0; i < n_groups && ok; ++i) {
                const int s = i % kS;
                const uint32_t ph = uint32_t(i / kS) & 1u;
                if (!wait_parity_suspend(expd(s), ph, abort, kWaitNs, kSuspendNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + uint32_t(s * TOKN);
                const uint32_t a0 = sbase + PLN.wexp + s * (2 * kRows * 32);
                const uint32_t b0 = sbase + PLN.aq + s * (2 * TOKN * 32);
                mma_f8(d, sdesc_sw32(a0), sdesc_sw32(b0), IDESC, 0u);
                mma_f8(d, sdesc_sw32(a0 + kRows * 32), sdesc_sw32(b0 + TOKN * 32), IDESC, 1u);
                mma_commit(tfull(s));
            }
            if (!ok) {
                atomicExch(&g_smtc_status, int(W4A4_ERR_TIMEOUT));
                *abort = 1;
            }
            mma_commit(mmadone);  // every MMA issued above has completed once this arrives
            wait_parity_suspend(mmadone, 0u, &never_abort, kWaitNs, kSuspendNs);
        }
        __syncwarp();
    }

    // ---- warps 0-3: expansion; warps 6-9: epilogue, one group behind
    const bool is_epi = warp >= WARP_EPI0;
    const int row = is_epi ? (warp & 3) * 32 + lane : warp * 32 + lane;  // weight row = tensor-memory lane
    uint64_t acc[TOKN / 2];                                                // running sums, token pairs
#pragma unroll
    for (int c = 0; c < TOKN / 2; ++c) acc[c] = 0ull;
    if (warp < 4) {
        for (int i = 0; i < n_groups && ok; ++i) {
            const int s = i % kS;
            const uint32_t ph = uint32_t(i / kS) & 1u;
            if (!warp_wait_parity_suspend(full(s), ph, abort, kWaitNs, kSuspendNs)) {
                ok = false;
                break;
            }
            // nibbles -> E4M3: row `row`, k-plane p, 16-byte chunk c at row * 32 + swz32(row, c) * 16
            const uint8_t* wr = smraw + PLN.wraw + s * (kRows * 32) + row * 32;
            const uint4 w01 = *reinterpret_cast<const uint4*>(wr);
            const uint4 w23 = *reinterpret_cast<const uint4*>(wr + 16);
            uint4 p0c0, p0c1, p1c0, p1c1;  // (the bytes are the codes + 8, as E4M3 values scaled by 2^-9)
            expand8(w01.x, p0c0.x, p0c1.x);
            expand8(w01.z, p0c0.y, p0c1.y);
            expand8(w23.x, p0c0.z, p0c1.z);
            expand8(w23.z, p0c0.w, p0c1.w);
            expand8(w01.y, p1c0.x, p1c1.x);
            expand8(w01.w, p1c0.y, p1c1.y);
            expand8(w23.y, p1c0.z, p1c1.z);
            expand8(w23.w, p1c0.w, p1c1.w);
            uint8_t* ep = smraw + PLN.wexp + s * (2 * kRows * 32);
            *reinterpret_cast<uint4*>(ep + row * 32 + swz32(row, 0) * 16) = p0c0;
            *reinterpret_cast<uint4*>(ep + row * 32 + swz32(row, 1) * 16) = p0c1;
            *reinterpret_cast<uint4*>(ep + kRows * 32 + row * 32 + swz32(row, 0) * 16) = p1c0;
            *reinterpret_cast<uint4*>(ep + kRows * 32 + row * 32 + swz32(row, 1) * 16) = p1c1;
            if (warp == 0) {
                // (sA, SA) pairs -> 2^9 sA[] (undoing the 2^-9 of the expanded weights) and
                // cc[] = -8 SA sA, in place (the pairs' 8 bytes per token)
                float* sp = reinterpret_cast<float*>(smraw + PLN.sa + s * (TOKN * 8));
                float v0[TOKN / 32 + 1], v1[TOKN / 32 + 1];
#pragma unroll
                for (int u = 0; u * 32 < TOKN; ++u) {
                    const int m = u * 32 + lane;
                    if (m < TOKN) {
                        v0[u] = sp[2 * m];
                        v1[u] = sp[2 * m + 1];
                    }
                }
                __syncwarp();
#pragma unroll
                for (int u = 0; u * 32 < TOKN; ++u) {
                    const int m = u * 32 + lane;
                    if (m < TOKN) {
                        sp[m] = v0[u] * kExpand8Scale;
                        sp[TOKN + m] = (-8.f * v1[u]) * v0[u];
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(expd(s));
        }
        if (!ok && lane == 0) {
            atomicExch(&g_smtc_status, int(W4A4_ERR_TIMEOUT));
            *abort = 1;
        }
    } else if (is_epi) {
        const uint32_t tl = tmem + (uint32_t((warp & 3) * 32) << 16);
        if (RP > 0) {
            const bool w_ok = warp_wait_parity_suspend(tlora, 0u, abort, kWaitNs, kSuspendNs);
            if (w_ok) {
                tc_fence_after();
                float l[TOKN];
                if constexpr (TOKN == 16) {
                    tmem_ld16(tl + uint32_t(kS * TOKN), l);
                } else {
#pragma unroll
                    for (int c = 0; c < TOKN / 32; ++c) tmem_ld32_at(tl + uint32_t(kS * TOKN + 32 * c), l + 32 * c);
                }
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < TOKN / 2; ++c) acc[c] = f2_pack(l[2 * c], l[2 * c + 1]);
            } else {
                ok = false;
            }
        }
        for (int e = 0; e < n_groups && ok; ++e) {
            const int s = e % kS;
            const uint32_t ph = uint32_t(e / kS) & 1u;
            if (!warp_wait_parity_suspend(tfull(s), ph, abort, kWaitNs, kSuspendNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // (the expansion barrier of this stage, already complete: orders warp 0's rewrite of the
            // stage's (sA, SA) into (sA, cc) before the reads below)
            if (!warp_wait_parity_suspend(expd(s), ph, abort, kWaitNs, kSuspendNs)) {
                ok = false;
                break;
            }
            float d[TOKN];
            if constexpr (TOKN == 16) {
                tmem_ld16(tl + uint32_t(s * TOKN), d);
            } else {
#pragma unroll
                for (int c = 0; c < TOKN / 32; ++c) tmem_ld32_at(tl + uint32_t(s * TOKN + 32 * c), d + 32 * c);
            }
            tmem_wait_ld();
            if (DUMP && nbase + row < N) {
                // partials dump: P = 2^9 D - 8 SA, exact in fp32 (|2^9 D| < 2^13), SA read from the workspace
                const int g = g_begin + e, n = nbase + row;
                const float* ssg = reinterpret_cast<const float*>(ws + AL.sS + ((size_t)(mt * G + g) * kTileM + rt0) * 8);
#pragma unroll
                for (int c = 0; c < TOKN; ++c)
                    if (tok0 + c < M) P[((size_t)(tok0 + c) * N + n) * G + g] = int32_t(d[c] * kExpand8Scale - 8.f * ssg[2 * c + 1]);
            }
            const float sw = __half2float(__ushort_as_half(
                reinterpret_cast<const uint16_t*>(smraw + PLN.sw + s * (kRows * 2))[row]));
            const uint64_t sw2 = f2_pack(sw, sw);
            const uint64_t* sa2 = reinterpret_cast<const uint64_t*>(smraw + PLN.sa + s * (TOKN * 8));
            const uint64_t* cc2 = sa2 + TOKN / 2;
#pragma unroll
            for (int c = 0; c < TOKN / 2; ++c)
                acc[c] = ffma2_b64(sw2, ffma2_b64(sa2[c], f2_pack(d[2 * c], d[2 * c + 1]), cc2[c]), acc[c]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sfree(s));
        }
        if (!ok && lane == 0) {
            atomicExch(&g_smtc_status, int(W4A4_ERR_TIMEOUT));
            *abort = 1;
        }
    }
    // ---- all roles done with the ring and tensor memory
    tc_fence_before();
    const bool aborted = __syncthreads_or(*abort);
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, PLN.tmem_cols);
    }
    if (aborted && threadIdx.x == 0) {
        // let the copies already requested land before this CTA's shared memory goes away
        for (int i = max(0, n_groups - kS); i < n_groups; ++i)
            wait_parity_suspend(full(i % kS), uint32_t(i / kS) & 1u, &never_abort, kWaitNs, kSuspendNs);
        if (RP > 0) wait_parity_suspend(lfull, 0u, &never_abort, kWaitNs, kSuspendNs);
    }

    // ---- exchange: 4-token block b belongs to rank b % KS
    float* red = reinterpret_cast<float*>(smraw + PLN.red);
    const int own = (BLK + KS - 1) / KS;
    if (KS > 1) {
        cluster_wait_acquire();  // every rank's barriers are initialised
        if (is_epi) {
#pragma unroll
            for (int b = 0; b < BLK; ++b) {
                const int o = b % KS;
                if (o == kr) continue;
                const int sidx = kr < o ? kr : kr - 1, ob = b / KS;
                const uint32_t dst = mapa_shared(sbase + PLN.red + uint32_t((sidx * kRows + row) * own + ob) * 16,
                                                 uint32_t(o));
                const float2 p0 = f2_unpack(acc[2 * b]), p1 = f2_unpack(acc[2 * b + 1]);
                st_async_v4(dst, make_float4(p0.x, p0.y, p1.x, p1.y), mapa_shared(red_full, uint32_t(o)));
            }
            int owned = 0;
            for (int b = 0; b < BLK; ++b) owned += (b % KS == kr);
            if (owned > 0) {
                const bool r_ok = warp_wait_parity_suspend(red_full, 0u, abort, kWaitNs, kSuspendNs);
                if (!r_ok) {
                    if (lane == 0) {
                        atomicExch(&g_smtc_status, int(W4A4_ERR_TIMEOUT));
                        *abort = 1;
                    }
                } else {
#pragma unroll
                    for (int b = 0; b < BLK; ++b) {
                        if (b % KS != kr) continue;
                        const int ob = b / KS;
                        float2 p0 = f2_unpack(acc[2 * b]), p1 = f2_unpack(acc[2 * b + 1]);
                        for (int rk = 0; rk < KS; ++rk) {
                            if (rk == kr) continue;
                            const int sidx = rk < kr ? rk : rk - 1;
                            const float4 v = *reinterpret_cast<const float4*>(red + ((sidx * kRows + row) * own + ob) * 4);
                            p0.x += v.x, p0.y += v.y, p1.x += v.z, p1.y += v.w;
                        }
                        acc[2 * b] = f2_pack(p0.x, p0.y);
                        acc[2 * b + 1] = f2_pack(p1.x, p1.y);
                    }
                }
            }
        }
        cluster_arrive_release();  // this rank's part of the exchange is done
    }

    // ---- affine of the owned token blocks, staged as rows [token][128 + 8] over the weight planes
    uint16_t* ys = reinterpret_cast<uint16_t*>(smraw + PLN.wexp);
    constexpr int LDY = kRows + 8;
    constexpr bool store = !DUMP;
    if (is_epi && !*abort && store && silu_I > 0) {
        // fused gate|up weights (gate_up_row order): lanes 0..15 of the warp on lane quarter q
        // hold the gates of outputs j = 64 t + 16 q + lane, lanes 16..31 the matching ups;
        // h = silu(g) u is staged as [token][64 + 8] at column 16 q + lane
        const int q = warp & 3;
        const int j = (nbase >> 1) + 16 * q + (lane & 15);
        const bool gate = lane < 16, valid = j < silu_I;
        const int src = gate ? j : silu_I + j;
        const float cs = valid ? __half2float(__ushort_as_half(colscale[src])) : 0.f;
        const float bs = (bias && valid) ? __half2float(__ushort_as_half(bias[src])) : 0.f;
#pragma unroll
        for (int b = 0; b < BLK; ++b) {
            if (b % KS != kr) continue;
            const float2 p0 = f2_unpack(acc[2 * b]), p1 = f2_unpack(acc[2 * b + 1]);
            const float v[4] = {p0.x, p0.y, p1.x, p1.y};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float y = fmaf(cs, v[i], bs);
                const float u = __shfl_down_sync(0xffffffffu, y, 16);
                if (gate)  // silu(y) u, fast exponential and divide (relative error ~1e-6)
                    ys[(4 * b + i) * LDY + 16 * q + lane] =
                        __half_as_ushort(__float2half_rn(__fdividef(y, 1.0f + __expf(-y)) * u));
            }
        }
    } else if (is_epi && !*abort && store) {
        const int n = nbase + row;
        const float cs = n < N ? __half2float(__ushort_as_half(colscale[n])) : 0.f;
        const float bs = (bias && n < N) ? __half2float(__ushort_as_half(bias[n])) : 0.f;
#pragma unroll
        for (int b = 0; b < BLK; ++b) {
            if (b % KS != kr) continue;
            const float2 p0 = f2_unpack(acc[2 * b]), p1 = f2_unpack(acc[2 * b + 1]);
            ys[(4 * b + 0) * LDY + row] = __half_as_ushort(__float2half_rn(fmaf(cs, p0.x, bs)));
            ys[(4 * b + 1) * LDY + row] = __half_as_ushort(__float2half_rn(fmaf(cs, p0.y, bs)));
            ys[(4 * b + 2) * LDY + row] = __half_as_ushort(__float2half_rn(fmaf(cs, p1.x, bs)));
            ys[(4 * b + 3) * LDY + row] = __half_as_ushort(__float2half_rn(fmaf(cs, p1.y, bs)));
        }
    }
    __syncthreads();
    if (!*abort && store && silu_I > 0) {
        for (int c = threadIdx.x; c < TOKN * (kRows / 16); c += kThreads) {
            const int t = c / (kRows / 16), ch = c % (kRows / 16);
            const int m = tok0 + t, j = (nbase >> 1) + ch * 8;
            if ((t / 4) % KS != kr) continue;
            if (m < M && j < silu_I)
                *reinterpret_cast<uint4*>(Y + (size_t)m * silu_I + j) =
                    *reinterpret_cast<const uint4*>(&ys[t * LDY + ch * 8]);
        }
    } else if (!*abort && store) {
        for (int c = threadIdx.x; c < TOKN * (kRows / 8); c += kThreads) {
            const int t = c / (kRows / 8), ch = c % (kRows / 8);
            const int m = tok0 + t, n = nbase + ch * 8;
            if ((t / 4) % KS != kr) continue;
            if (m < M && n < N)
                *reinterpret_cast<uint4*>(Y + (size_t)m * N + n) = *reinterpret_cast<const uint4*>(&ys[t * LDY + ch * 8]);
        }
    }
    if (KS > 1) cluster_wait_acquire();  // no rank leaves while a peer may still address its shared memory
}

// Split factor: at most as many CTAs as fit at once (two per SM, one for 64
// tokens, whose registers fill half the register file), at least one group per CTA.
int smtc_split(int M, int N, int K, int TOKN) {
    const int tiles = ((N + kRows - 1) / kRows) * ((M + TOKN - 1) / TOKN);
    const int G = K / kGroup;
    const int per_sm = TOKN >= 64 ? 1 : 2;
    int ks = 1;
    while (ks < kMaxKS && tiles * ks * 2 <= device_sm_count() * per_sm && ks * 2 <= G) ks *= 2;
    return ks;
}

template <int TOKN, bool DUMP>
w4a4_status launch_t(const uint8_t* ws, const uint8_t* packed, const uint16_t* cs, const uint16_t* bias, int M,
                     int N, int K, int r, uint16_t* Y, int32_t* P, int silu_I, cudaStream_t s) {
    const int KS = smtc_split(M, N, K, TOKN);
    const TcPlan plan = tc_plan(TOKN, r, KS);
    const int smem_max = int(tc_plan(TOKN, W4A4_MAX_RANK, kMaxKS).total) + 1024;
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(gemm_smallm_tc_kernel<TOKN, DUMP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) !=
            cudaSuccess)
            return W4A4_ERR_CUDA;
        attr_done[dev] = 1;
    }
    dim3 grid(unsigned(((N + kRows - 1) / kRows) * KS), unsigned((M + TOKN - 1) / TOKN));
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(KS);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = add_pdl_attr(attr, 1);
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.total + 1024;  // (the dynamic region is aligned up to 1024 bytes inside)
    cfg.stream = s;
    if (cudaLaunchKernelEx(&cfg, gemm_smallm_tc_kernel<TOKN, DUMP>, ws, packed, cs, bias, M, N, K, r, Y, P, KS, silu_I) !=
        cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    set_dispatch("gemm_smallm_tc tcgen05.f8f6f4 swap-AB N=%d split-K=%d (cluster) grid=%ux%u%s%s", TOKN, KS, grid.x,
                 grid.y, silu_I ? " silu(gate)*up" : "", DUMP ? " (partials dump)" : "");
    return launch_status();
}

}  // namespace

w4a4_status smtc_read_and_clear_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_smtc_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_smtc_status, &zero, sizeof(int));
        return W4A4_ERR_TIMEOUT;
    }
    return W4A4_OK;
}

w4a4_status launch_gemm_smallm_tc(const uint8_t* ws, const uint8_t* packed, const uint16_t* colscale,
                                  const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, int32_t* P_dump,
                                  int silu_I, cudaStream_t s) {
    if (P_dump) {  // the same token block and split, in the DUMP variant
        if (M <= 16) return launch_t<16, true>(ws, packed, nullptr, nullptr, M, N, K, r, nullptr, P_dump, 0, s);
        if (M <= 32) return launch_t<32, true>(ws, packed, nullptr, nullptr, M, N, K, r, nullptr, P_dump, 0, s);
        return launch_t<64, true>(ws, packed, nullptr, nullptr, M, N, K, r, nullptr, P_dump, 0, s);
    }
    if (M <= 16) return launch_t<16, false>(ws, packed, colscale, bias, M, N, K, r, Y, nullptr, silu_I, s);
    if (M <= 32) return launch_t<32, false>(ws, packed, colscale, bias, M, N, K, r, Y, nullptr, silu_I, s);
    return launch_t<64, false>(ws, packed, colscale, bias, M, N, K, r, Y, nullptr, silu_I, s);
}

}  // namespace w4a4
