// Weight-streaming W4A4 GEMM for small M (decode): warp-level FP8 MMA with the
// weights as the 16-row operand ("swap AB"), per-group exact products, fp32
// scaled accumulation, LoRA up and the column affine in the same kernel.
//
// "INT4 Kernel Architecture, in depth" ("Why INT4 kernels exist: the
// roofline", "One token versus a thousand": split-K for small batches): at
// small M the layer is bound by the bytes of packed weights, so each weight
// record is read once, expanded in registers, and used against every token of
// the CTA.  "W4A4 CUDA Kernel for Voice Clone", 3.7: per-group integer MMA,
// scaling by act_scale * wgt_scale, LoRA-up into the same accumulator.
//
// Per group g the tensor core computes D = sum_k cA[m,k] * (cW[n,k] + 8)
// exactly (weights are stored offset-binary, see common.cuh), so
//   P = D - 8 SA[m,g],  acc += sW[n,g] * (sA[m,g] * D - 8 SA sA)
// with the per-token constant -8 SA sA hoisted out of the element loop.
//
// Layout of the work: a CTA of 8 warps covers 128 weight rows (16 per warp)
// and up to 64 tokens; K is split over a thread-block cluster of KS CTAs (KS
// in {1, 2, 4, 8}) so that the whole machine streams weights.  A CTA requests
// its whole share at the start (up to 16 groups, then 8 more each time 8 are
// consumed): each group's 128 weight records (4 KB, contiguous in the packed
// layout) by one 1-D bulk copy, and the small pieces -- weight scales, the
// token block's codes and scales, the LoRA planes -- by cp.async from every
// thread.  Each group slot has its own mbarrier (the bulk copy's bytes plus
// one cp.async arrival per thread), so the warps start on a group as soon as
// it lands, while the rest stream in.  Warp w's 16 output columns belong to
// cluster rank w % KS: the other ranks push their fp32 partial sums into that
// rank's shared memory with st.async (completing bytes on its mbarrier), and
// the owner adds them in rank order -- a fixed order, no atomics -- before
// the LoRA up, the affine and the store.  Waits are bounded (2 s;
// W4A4_ERR_TIMEOUT in the status word).  Both cluster barriers are split: the
// first (barriers initialised) is arrived at before the weights stream and
// waited on before the first remote store; the last (no rank leaves while a
// peer may address its shared memory) is arrived at after the exchange and
// waited on after the store.
#include "kernels.h"
#include "tc_ptx.cuh"

namespace w4a4 {
namespace {
using namespace tc;

constexpr int kWarps = 8;
constexpr int kTileN = kWarps * 16;  // weight rows per CTA
constexpr int kMaxKS = 8;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kSuspendNs = 20000;  // upper bound of one suspension in a wait

// Status word of this kernel's bounded waits (W4A4_ERR_TIMEOUT once one gave up).
__device__ int g_smallm_status = 0;

// Byte offsets of the shared-memory sections (all multiples of 16).
struct SmallMPlan {
    int ns;  // group slots: two halves of ns / 2, refilled alternately
    uint32_t wq, aq, sw, as, lu, la, red, bar, total;
};
__host__ __device__ inline SmallMPlan smallm_plan(int tok, int r) {
    SmallMPlan p;
    p.ns = tok >= 32 ? 8 : 16;
    uint32_t o = 0;
    p.wq = o, o += uint32_t(p.ns) * kTileN * 32;                 // [slot][128 rows][32 B]
    p.aq = o, o += uint32_t(p.ns) * 2 * tok * 32;                // [slot][plane][tok][32 B]
    p.sw = o, o += uint32_t(p.ns) * kTileN * 2;                  // [slot][128] fp16
    p.as = o, o += uint32_t(p.ns) * tok * 8;                     // [slot][tok] (sA, SA)
    p.lu = o, o += uint32_t(r / 16) * kTileN * 32;               // [plane][128 rows][32 B]
    p.la = o, o += uint32_t(r / 16) * tok * 32;                  // [plane][tok][32 B]
    p.red = o, o += uint32_t(kMaxKS - 1) * 32 * (tok / 8) * 16;  // [sender slot][lane][tok / 8] float4
    p.bar = o, o += 160;                                         // full[ns], aux, red_full
    p.total = o;
    return p;
}
// A rank owns 8 / KS warps and hears from KS - 1 senders: (KS - 1) * (8 / KS)
// <= 7 reduction slots.  The fp16 output tile [tok][128 + 8] is staged over
// the group slots once every group has been consumed (tok * 136 * 2 bytes <=
// ns * 4 KB for both slot counts).

template <int NT8, bool DUMP>
__global__ void __launch_bounds__(kWarps * 32) gemm_smallm_kernel(
    const uint8_t* __restrict__ ws, const uint8_t* __restrict__ packed, const uint16_t* __restrict__ colscale,
    const uint16_t* __restrict__ bias, int M, int N, int K, int r, uint16_t* __restrict__ Y,
    int32_t* __restrict__ P, int KS) {
    constexpr int TOK = NT8 * 8;
    constexpr int NT = kWarps * 32;
    extern __shared__ __align__(128) uint8_t smraw[];
    __shared__ int abort_flag, never_abort;
    const SmallMPlan PLN = smallm_plan(TOK, r);
    const uint32_t sbase = smem_u32(smraw);
    const uint32_t full0 = sbase + PLN.bar;  // full[s] = full0 + 8 s
    const uint32_t aux_full = full0 + 8u * PLN.ns, red_full = aux_full + 8u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, q = lane & 3;
    const int G = K / kGroup;
    const ActLayout AL = act_layout(M, K, r);
    const PackedLayout PL = packed_layout(N, K, r);
    const int kr = KS > 1 ? int(cluster_ctarank()) : 0;
    const int ntile = blockIdx.x / KS;
    const int g_begin = (G * kr) / KS, n_groups = (G * (kr + 1)) / KS - g_begin;
    const int half = PLN.ns / 2;
    const int n_chunks = (n_groups + half - 1) / half;

    const int tok0 = blockIdx.y * TOK;  // first token of this CTA
    const int mt = tok0 / kTileM, rt0 = tok0 % kTileM;
    const int nbase = ntile * kTileN;
    const int rows_valid = min(kTileN, N - nbase);  // a multiple of 16
    const int n0 = nbase + warp * 16;
    const bool warp_active = n0 < N;
    const bool owner = KS == 1 || warp % KS == kr;
    volatile int* abort = &abort_flag;

    const uint8_t* qW = packed + PL.qW;
    const uint8_t* sWg = packed + PL.sW;
    // 16-byte pieces of one group besides the weight records: weight scales,
    // the two code planes of the token block, its (sA, SA) pairs
    const int pc_sw = rows_valid / 8, pc_aq = 4 * TOK, pc_as = TOK / 2;

    // chunk c -- groups g_begin + c * half ... -- into slot half c & 1; every thread takes part
    auto issue_chunk = [&](int c) {
        const int b = c & 1, ng = min(half, n_groups - c * half);
        for (int j = 0; j < ng; ++j) {
            const int g = g_begin + c * half + j, slot = b * half + j;
            const uint32_t bar = full0 + 8u * slot;
            if (threadIdx.x == 0) {
                mbar_expect_tx(bar, uint32_t(rows_valid) * 32);
                bulk_g2s(sbase + PLN.wq + slot * (kTileN * 32), qW + ((size_t)g * N + nbase) * 32, rows_valid * 32,
                         bar);
            }
            const uint8_t* qa = ws + AL.qA + (size_t)(mt * G + g) * 2 * (kTileM * 32) + (size_t)rt0 * 32;
            for (int p = threadIdx.x; p < pc_sw + pc_aq + pc_as; p += NT) {
                if (p < pc_sw) {
                    cp_async16(smraw + PLN.sw + slot * (kTileN * 2) + p * 16, sWg + ((size_t)g * N + nbase) * 2 + p * 16);
                } else if (p < pc_sw + pc_aq) {
                    const int e = p - pc_sw, pl = e / (2 * TOK), o = (e % (2 * TOK)) * 16;
                    cp_async16(smraw + PLN.aq + slot * (2 * TOK * 32) + pl * (TOK * 32) + o,
                               qa + (size_t)pl * (kTileM * 32) + o);
                } else {
                    const int e = p - pc_sw - pc_aq;
                    cp_async16(smraw + PLN.as + slot * (TOK * 8) + e * 16,
                               ws + AL.sS + ((size_t)(mt * G + g) * kTileM + rt0) * 8 + e * 16);
                }
            }
            cp_async_mbar_arrive_noinc(bar);
        }
    };

    if (threadIdx.x == 0) {
        abort_flag = 0;
        never_abort = 0;
        for (int s = 0; s < PLN.ns; ++s) mbar_init(full0 + 8u * s, NT + 1);  // cp.async arrivals + the copy's
        mbar_init(aux_full, NT);
        mbar_init(red_full, 1);
        fence_mbar_init();
        if (KS > 1 && !DUMP)  // bytes this rank receives: its owned warps' fragments from every other rank
            mbar_expect_tx(red_full, uint32_t((KS - 1) * (kWarps / KS) * 32 * NT8 * 16));
    }
    __syncthreads();  // barriers initialised for this CTA's threads
    if (KS > 1 && !DUMP) cluster_arrive_release();  // ... and, once every rank has arrived, for the peers
    // The setup above touches only shared memory and overlaps the previous kernel;
    // so does warming L2 with this CTA's share of the weight records and scales
    // (a prefetch only fills the cache; every copy proper comes after the wait).
    if (threadIdx.x == 0) {
        for (int i = 0; i < n_groups; ++i) {
            prefetch_l2(qW + ((size_t)(g_begin + i) * N + nbase) * 32, uint32_t(rows_valid) * 32);
            prefetch_l2(sWg + ((size_t)(g_begin + i) * N + nbase) * 2, uint32_t(rows_valid) * 2);
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (!DUMP) {
        // LoRA planes first (their barrier then completes with them alone): the
        // token block's activations, and the up-projection rows of the warps this rank owns
        const int own = kWarps / KS, pc_la = 2 * TOK, pc_plane = pc_la + own * 32;
        for (int p = threadIdx.x; p < (r / 16) * pc_plane; p += NT) {
            const int pl = p / pc_plane, e = p % pc_plane;
            if (e < pc_la) {
                cp_async16(smraw + PLN.la + pl * (TOK * 32) + e * 16,
                           ws + AL.La + (size_t)(mt * (r / 16) + pl) * (kTileM * 32) + (size_t)rt0 * 32 + e * 16);
            } else {
                const int w = kr + KS * ((e - pc_la) / 32), o = ((e - pc_la) % 32) * 16;
                if (nbase + w * 16 < N)
                    cp_async16(smraw + PLN.lu + pl * (kTileN * 32) + w * 512 + o,
                               packed + PL.Lu + ((size_t)pl * N + nbase + w * 16) * 32 + o);
            }
        }
        cp_async_mbar_arrive_noinc(aux_full);
    }
    int issued = 0, requested = 0;  // chunks consumed-or-skipped / actually requested (same in every thread)
    for (; issued < 2 && issued < n_chunks; ++issued) issue_chunk(issued);
    requested = issued;

    float csa = 0.f, csb = 0.f, ba = 0.f, bb = 0.f;
    if (!DUMP && owner && warp_active) {
        csa = __half2float(__ushort_as_half(colscale[n0 + gid]));
        csb = __half2float(__ushort_as_half(colscale[n0 + gid + 8]));
        if (bias) {
            ba = __half2float(__ushort_as_half(bias[n0 + gid]));
            bb = __half2float(__ushort_as_half(bias[n0 + gid + 8]));
        }
    }

    // fp32 accumulators as packed pairs: (row a | row b) x (token 2q, 2q + 1) of each 8-token block
    uint64_t acc_a[NT8], acc_b[NT8];
#pragma unroll
    for (int t = 0; t < NT8; ++t) acc_a[t] = acc_b[t] = 0ull;
    const uint64_t m8 = f2_pack(-8.f, -8.f);

    // this lane's weight bytes (rows warp*16 + gid and + 8, bytes 8q..8q+7) and scales in a slot
    const uint8_t* smw = smraw + PLN.wq + (warp * 16 + gid) * 32 + 8 * q;
    const uint16_t* smsw = reinterpret_cast<const uint16_t*>(smraw + PLN.sw) + warp * 16 + gid;
    // ldmatrix row address of this lane within a slot's code planes, token block 0: matrix
    // lane / 8 = (plane, logical 16-byte chunk), row lane % 8 (the chunk's physical place
    // follows the 32-byte swizzle of the token's row; token blocks start at multiples of 8)
    const uint32_t lm_lane = uint32_t((lane >> 4) * (TOK * 32) + (lane & 7) * 32 +
                                      ((((lane >> 3) & 1) ^ ((lane >> 2) & 1)) * 16));
    for (int c = 0; c < n_chunks; ++c) {
        const int b = c & 1, ng = min(half, n_groups - c * half);
        for (int j = 0; j < ng; ++j) {
            const int slot = b * half + j;
            const bool ok = warp_wait_parity_suspend(full0 + 8u * slot, uint32_t(c >> 1) & 1u, abort, kWaitNs,
                                                     kSuspendNs);
            if (!ok) {
                if (lane == 0) {
                    *abort = 1;
                    atomicExch(&g_smallm_status, int(W4A4_ERR_TIMEOUT));
                }
                break;
            }
            if (!warp_active) continue;
            const uint2 wa = *reinterpret_cast<const uint2*>(smw + slot * (kTileN * 32));
            const uint2 wb = *reinterpret_cast<const uint2*>(smw + slot * (kTileN * 32) + 8 * 32);
            const float swa = __half2float(__ushort_as_half(smsw[slot * kTileN]));
            const float swb = __half2float(__ushort_as_half(smsw[slot * kTileN + 8]));
            const uint64_t swa2 = f2_pack(swa, swa), swb2 = f2_pack(swb, swb);
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
                uint32_t bf[4];  // (plane 0 | plane 1) x (k 0-15 | k 16-31) of tokens t*8 .. t*8+7
                ldsm_x4(bf, sbase + PLN.aq + uint32_t(slot * (2 * TOK * 32) + t * 256) + lm_lane);
                // (sA, SA) of tokens t*8 + 2q and + 1
                const float4 s =
                    *reinterpret_cast<const float4*>(smraw + PLN.as + slot * (TOK * 8) + (t * 8 + 2 * q) * 8);
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma_e4m3_16832(d, a0, bf[0], bf[1]);
                mma_e4m3_16832(d, a1, bf[2], bf[3]);
                if constexpr (DUMP) {
                    const int g = g_begin + c * half + j;
                    const int m0 = tok0 + t * 8 + 2 * q;
                    const int na_ = n0 + gid, nb_ = n0 + gid + 8;
                    if (m0 < M) {
                        P[((size_t)m0 * N + na_) * G + g] = int32_t(d[0] - 8.f * s.y);
                        P[((size_t)m0 * N + nb_) * G + g] = int32_t(d[2] - 8.f * s.y);
                    }
                    if (m0 + 1 < M) {
                        P[((size_t)(m0 + 1) * N + na_) * G + g] = int32_t(d[1] - 8.f * s.w);
                        P[((size_t)(m0 + 1) * N + nb_) * G + g] = int32_t(d[3] - 8.f * s.w);
                    }
                } else {
                    // acc += sW * (sA * D + (-8 SA) sA), pairwise over the two tokens
                    const uint64_t sA2 = f2_pack(s.x, s.z);
                    const uint64_t cc = fmul2_b64(fmul2_b64(f2_pack(s.y, s.w), m8), sA2);
                    acc_a[t] = ffma2_b64(swa2, ffma2_b64(sA2, f2_pack(d[0], d[1]), cc), acc_a[t]);
                    acc_b[t] = ffma2_b64(swb2, ffma2_b64(sA2, f2_pack(d[2], d[3]), cc), acc_b[t]);
                }
            }
        }
        if (issued < n_chunks) {  // uniform: refill the half just consumed
            // every warp is done with it; the refill stops, everywhere alike, once a wait gave up
            if (!__syncthreads_or(*abort)) {
                issue_chunk(issued);
                requested = issued + 1;
            }
            ++issued;
        }
    }
    if (__syncthreads_or(*abort)) {
        // let the copies already requested land before this CTA's shared memory goes away
        if (threadIdx.x == 0) {
            for (int c = max(0, requested - 2); c < requested; ++c) {
                const int ng = min(half, n_groups - c * half);
                for (int j = 0; j < ng; ++j)
                    wait_parity_suspend(full0 + 8u * ((c & 1) * half + j), uint32_t(c >> 1) & 1u, &never_abort, kWaitNs, kSuspendNs);
            }
            if (!DUMP) wait_parity_suspend(aux_full, 0u, &never_abort, kWaitNs, kSuspendNs);
        }
    }
    if constexpr (!DUMP) {  // (the partials variant ends with the dump above)

        float acc[NT8][4];
    #pragma unroll
        for (int t = 0; t < NT8; ++t) {
            const float2 pa = f2_unpack(acc_a[t]), pb = f2_unpack(acc_b[t]);
            acc[t][0] = pa.x, acc[t][1] = pa.y, acc[t][2] = pb.x, acc[t][3] = pb.y;
        }
        if (KS > 1) {
            cluster_wait_acquire();  // every rank's barriers are initialised
            const int orank = warp % KS, ow = warp / KS;  // owner rank, owned-warp index there
            if (!owner) {
                // push this warp's partial fragment to the owner of its columns
                const int slot = (kr < orank ? kr : kr - 1) * (kWarps / KS) + ow;
                const uint32_t dst = mapa_shared(sbase + PLN.red + uint32_t(slot * 32 + lane) * (NT8 * 16), uint32_t(orank));
                const uint32_t rbar = mapa_shared(red_full, uint32_t(orank));
    #pragma unroll
                for (int t = 0; t < NT8; ++t)
                    st_async_v4(dst + uint32_t(t) * 16u, make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]), rbar);
            } else {
                const bool ok = warp_wait_parity_suspend(red_full, 0u, abort, kWaitNs, kSuspendNs);
                if (!ok) {
                    if (lane == 0) {
                        *abort = 1;
                        atomicExch(&g_smallm_status, int(W4A4_ERR_TIMEOUT));
                    }
                } else {
                    const float4* red = reinterpret_cast<const float4*>(smraw + PLN.red);
                    for (int rk = 0; rk < KS; ++rk) {
                        if (rk == kr) continue;
                        const int slot = (rk < kr ? rk : rk - 1) * (kWarps / KS) + ow;
    #pragma unroll
                        for (int t = 0; t < NT8; ++t) {
                            const float4 v = red[(slot * 32 + lane) * NT8 + t];
                            acc[t][0] += v.x;
                            acc[t][1] += v.y;
                            acc[t][2] += v.z;
                            acc[t][3] += v.w;
                        }
                    }
                }
            }
            cluster_arrive_release();  // this rank's part of the exchange is done
        }

        // fp16 output tile staged over the group slots, which no warp or copy uses any more
        // (after a timed-out group wait copies may still land there: nothing is staged then)
        uint16_t* ys = reinterpret_cast<uint16_t*>(smraw + PLN.wq);
        constexpr int LDY = kTileN + 8;
        if (owner && warp_active && !*abort) {
            const bool ok = r == 0 || warp_wait_parity_suspend(aux_full, 0u, abort, kWaitNs, kSuspendNs);
            if (!ok && lane == 0) {
                *abort = 1;
                atomicExch(&g_smallm_status, int(W4A4_ERR_TIMEOUT));
            }
            // LoRA up: acc[n, m] += sum_j L_up[j, n] lora[m, j] (fp16 MMA, fp32 accumulate)
            const int na_ = n0 + gid, nb_ = n0 + gid + 8;
            const uint8_t* lu_a = smraw + PLN.lu + (warp * 16 + gid) * 32 + 4 * q;
            const uint8_t* lu_b = lu_a + 8 * 32;
            for (int p = 0; ok && p < r / 16; ++p) {
                uint32_t a[4];
                a[0] = *reinterpret_cast<const uint32_t*>(lu_a + p * (kTileN * 32) + swz32(na_, 0) * 16);
                a[2] = *reinterpret_cast<const uint32_t*>(lu_a + p * (kTileN * 32) + swz32(na_, 1) * 16);
                a[1] = *reinterpret_cast<const uint32_t*>(lu_b + p * (kTileN * 32) + swz32(nb_, 0) * 16);
                a[3] = *reinterpret_cast<const uint32_t*>(lu_b + p * (kTileN * 32) + swz32(nb_, 1) * 16);
                const uint8_t* la = smraw + PLN.la + p * (TOK * 32);
    #pragma unroll
                for (int t = 0; t < NT8; ++t) {
                    const int rr = t * 8 + gid;  // rr % 8 == (rt0 + rr) % 8
                    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(la + rr * 32 + swz32(rr, 0) * 16 + 4 * q);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(la + rr * 32 + swz32(rr, 1) * 16 + 4 * q);
                    mma_f16_16816(acc[t], a, b0, b1);
                }
            }
            // column affine, fp16
            const int nl = warp * 16 + gid;
    #pragma unroll
            for (int t = 0; t < NT8; ++t) {
                const int m0 = t * 8 + 2 * q;
                ys[m0 * LDY + nl] = __half_as_ushort(__float2half_rn(fmaf(csa, acc[t][0], ba)));
                ys[(m0 + 1) * LDY + nl] = __half_as_ushort(__float2half_rn(fmaf(csa, acc[t][1], ba)));
                ys[m0 * LDY + nl + 8] = __half_as_ushort(__float2half_rn(fmaf(csb, acc[t][2], bb)));
                ys[(m0 + 1) * LDY + nl + 8] = __half_as_ushort(__float2half_rn(fmaf(csb, acc[t][3], bb)));
            }
        }
        __syncthreads();
        // store the columns of the warps this rank owns, 16 bytes at a time
        if (!*abort) {
            for (int c = threadIdx.x; c < TOK * (kTileN / 8); c += NT) {
                const int t = c / (kTileN / 8), ch = c % (kTileN / 8);
                const int m = tok0 + t, n = nbase + ch * 8;
                if ((ch >> 1) % KS != kr) continue;  // chunk ch belongs to warp ch / 2
                if (m < M && n < N)
                    *reinterpret_cast<uint4*>(Y + (size_t)m * N + n) = *reinterpret_cast<const uint4*>(&ys[t * LDY + ch * 8]);
            }
        }
        if (r > 0 && threadIdx.x == 0 && !wait_parity_suspend(aux_full, 0u, &never_abort, kWaitNs, kSuspendNs))
            atomicExch(&g_smallm_status, int(W4A4_ERR_TIMEOUT));  // (the LoRA copies land before the CTA leaves)
        if (KS > 1) cluster_wait_acquire();  // no rank leaves while a peer may still address its shared memory
    }
}

// Split factor: up to two CTAs per SM, so that every SM streams weights with
// enough bytes in flight, and at least one group per CTA.
int smallm_split(int M, int N, int K, int TOK) {
    const int tiles = ((N + kTileN - 1) / kTileN) * ((M + TOK - 1) / TOK);
    const int G = K / kGroup;
    int ks = 1;
    while (ks < kMaxKS && tiles * ks * 2 <= 2 * device_sm_count() && ks * 2 <= G) ks *= 2;
    return ks;
}

template <int NT8>
w4a4_status launch_nt(const uint8_t* ws, const uint8_t* packed, const uint16_t* cs, const uint16_t* bias, int M,
                      int N, int K, int r, uint16_t* Y, int32_t* P, cudaStream_t s) {
    const int smem_max = int(smallm_plan(NT8 * 8, W4A4_MAX_RANK).total);  // the attribute covers every rank
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(gemm_smallm_kernel<NT8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_max) != cudaSuccess ||
            cudaFuncSetAttribute(gemm_smallm_kernel<NT8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_max) != cudaSuccess)
            return W4A4_ERR_CUDA;
        attr_done[dev] = 1;
    }
    const int KS = P ? 1 : smallm_split(M, N, K, NT8 * 8);
    dim3 grid(unsigned(((N + kTileN - 1) / kTileN) * KS), unsigned((M + NT8 * 8 - 1) / (NT8 * 8)));
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(KS);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = add_pdl_attr(attr, 1);
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smallm_plan(NT8 * 8, r).total;
    cfg.stream = s;
    cudaError_t e;
    if (P)
        e = cudaLaunchKernelEx(&cfg, gemm_smallm_kernel<NT8, true>, ws, packed, cs, bias, M, N, K, r, Y, P, KS);
    else
        e = cudaLaunchKernelEx(&cfg, gemm_smallm_kernel<NT8, false>, ws, packed, cs, bias, M, N, K, r, Y, P, KS);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    set_dispatch("gemm_smallm mma.sync.e4m3 tokens/CTA=%d split-K=%d (cluster) grid=%ux%u%s", NT8 * 8, KS, grid.x,
                 grid.y, P ? " (partials dump)" : "");
    return launch_status();
}

}  // namespace

w4a4_status smallm_read_and_clear_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_smallm_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_smallm_status, &zero, sizeof(int));
        return W4A4_ERR_TIMEOUT;
    }
    return W4A4_OK;
}

w4a4_status launch_gemm_smallm(const uint8_t* ws, const uint8_t* packed, const uint16_t* colscale,
                               const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, int32_t* P_dump,
                               cudaStream_t s) {
    if (M <= 8) return launch_nt<1>(ws, packed, colscale, bias, M, N, K, r, Y, P_dump, s);
    if (M <= 16) return launch_nt<2>(ws, packed, colscale, bias, M, N, K, r, Y, P_dump, s);
    if (M <= 32) return launch_nt<4>(ws, packed, colscale, bias, M, N, K, r, Y, P_dump, s);
    return launch_nt<8>(ws, packed, colscale, bias, M, N, K, r, Y, P_dump, s);
}

}  // namespace w4a4
