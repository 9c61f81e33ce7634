// The whole W4A4 + LoRA linear for small M in one kernel: activation
// quantisation and LoRA down from fp16 X, the W4A4 GEMM with exact per-group
// products, LoRA up and the column affine ("W4A4 CUDA Kernel for Voice Clone",
// 3.6-3.7: quantise and LoRA-down from one read of X, exact group products
// scaled per group, LoRA up into the same accumulator; "INT4 Kernel
// Architecture, in depth", "One token versus a thousand": at decode sizes the
// call is a weight stream, and split-K keeps every SM busy).
//
// At M <= 32 and K = N = 4096 the weights are 8.9 MB and the rest is a few
// hundred KB, so the call is a weight stream whose length is set by the DRAM
// latency, not by its bytes.  The kernel therefore issues every load it needs
// at once, right after the launch dependency: each CTA (128 weight rows x a
// slice of K groups, the slice split over a cluster of KS CTAs) loads all of
// its weight records (into the registers of the warps that expand them), the
// X slice, the LoRA-down fragments and the weight scales, and computes while
// the weights arrive.
//
// Per group g, D[n, m] = 2^-9 sum_k (cW[n,k] + 8) cA[m,k] exactly (the weight
// bytes are the offset codes, read by E4M3 as u * 2^-9; the weights are the
// MMA's 128-row A operand, held in tensor memory, and the tokens its N), and
// the epilogue adds sW[n,g] (2^9 sA[m,g] D - 8 SA sA) to fp32 sums (one thread
// per weight row, one column pair per two tokens).
//
// Roles (10 warps, two CTAs per SM):
//   warps 0-3  load their 32 weight rows of every group (two 16-byte loads per
//              row and group, all in flight), expand each group's nibbles to
//              bytes in tensor memory, and (warp 0, one thread) issue the
//              group's two kind::f8f6f4 MMAs once the four warps are done;
//   warp 4     bulk copies of the LoRA-down fragments and (on token-block
//              owners) the LoRA-up planes; LoRA down of token rows 0-15
//              (16 tokens: of the first half of the groups);
//   warp 5     tensor-memory owner; bulk copies of the weight scales; LoRA down
//              of token rows 16-31 (16 tokens: the second half of the groups);
//              on owners the sum of the cluster's LoRA-down partials (rank
//              order), fp16, and the kind::f16 LoRA-up MMAs;
//   warps 6-9  stage the X slice (cp.async), quantise it (the same arithmetic
//              as the activation kernel: codes, sA, SA bit for bit) into the
//              B operand, then run the per-group epilogue.
// Token block b (4 tokens) belongs to cluster rank b % KS: the other ranks
// push their LoRA-down partials and, at the end, their fp32 sums of the block
// there (st.async), and the owner adds them in rank order, adds its LoRA-up
// product, applies the affine and stores Y.  Only blocks holding a valid token
// take part.  Cluster barrier phases: (1) every rank's mbarriers are set up,
// (2) every rank is done with its X staging area, which then receives the
// partial sums, (3) every rank is done with the exchange.  Every wait is
// bounded (2 s; W4A4_ERR_TIMEOUT in the status word); on give-up every role
// unwinds, the MMAs issued are waited for, tensor memory is freed, copies in
// flight are waited for, and every thread still passes every barrier.
#include "kernels.h"
#include "quant.cuh"
#include "tc_ptx.cuh"

namespace w4a4 {
namespace {
using namespace tc;

constexpr int kRows = 128;   // weight rows per CTA (MMA M, tensor-memory lanes)
constexpr int kThreads = 320;
constexpr int WARP_LD = 4, WARP_AUX = 5, WARP_Q0 = 6;
constexpr int kMaxKS = 8;
constexpr int kMaxG = 8;     // K groups per CTA
constexpr int kMaxR = 32;    // LoRA rank
constexpr int kXStride = kMaxG * kGroup + 8;  // halves per staged X row (+8: conflict-free ldmatrix)
constexpr uint32_t kTmemCols = 256;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kSuspendNs = 20000;
constexpr uint32_t BAR_EXP = 1, BAR_Q = 2;  // named barriers: expansion warps, quantisation warps

__device__ int g_fused_status = 0;

template <int TOKN>
struct FCfg {
    static constexpr int kT = TOKN == 16 ? 7 : 3;   // product buffers in tensor memory
    static constexpr uint32_t DCOL = kMaxG * 16;     // A operand: 16 columns per group, then the products
    static constexpr uint32_t LCOL = DCOL + kT * TOKN;
    static constexpr int WL = TOKN == 16 ? 2 : 1;    // LoRA-down partial sets per rank (warps 4 and 5)
    static constexpr int BLK = TOKN / 4;
    static_assert(LCOL + TOKN <= kTmemCols, "tensor memory plan");
};

// Byte offsets of the shared-memory sections (multiples of 16; the tensor
// core's operands at multiples of 1024 or of their plane size).
struct FPlan {
    uint32_t lu, la, aq, ldst, xs, sw, sc, lrecv, bar, total;
    int own;  // token blocks per rank
};
__host__ __device__ inline FPlan fplan(int tokn, int r, int ks) {
    FPlan p;
    const int RP = r / 16, NT = r / 8, blk = tokn / 4, wl = tokn == 16 ? 2 : 1;
    p.own = (blk + ks - 1) / ks;
    uint32_t o = 0;
    p.lu = o, o += uint32_t(RP) * kRows * 32;         // [plane][128 rows][32 B]
    p.la = o, o += uint32_t(RP) * tokn * 32;          // [plane][tokn][32 B]
    o = (o + 1023u) & ~1023u;
    p.aq = o, o += uint32_t(kMaxG) * 2 * tokn * 32;   // [group][plane][tokn][32 B]
    p.ldst = o, o += uint32_t(kMaxG) * NT * 1024;     // LoRA-down fragments [group][k step][tile][lane] x 8 B
    p.xs = o;
    const uint32_t xs_bytes = uint32_t(tokn) * kXStride * 2;
    const uint32_t red_bytes = uint32_t(ks > 1 ? ks - 1 : 0) * kRows * p.own * 16;
    o += xs_bytes > red_bytes ? xs_bytes : red_bytes;  // X slice, later the partial sums received
    p.sw = o, o += uint32_t(kMaxG) * kRows * 2;        // [group][128] fp16
    p.sc = o, o += uint32_t(kMaxG) * 3 * tokn * 4;     // [group][2^9 sA | -8 SA sA | SA][tokn]
    p.lrecv = o, o += uint32_t(ks) * wl * p.own * 4 * r * 4;  // [rank][set][owned block][4 rows][r]
    p.bar = o, o += 512;
    p.total = o;
    return p;
}

template <int TOKN, bool DUMP>
__global__ void __launch_bounds__(kThreads, 2) linear_fused_kernel(
    const uint16_t* __restrict__ X, const uint8_t* __restrict__ packed, const uint16_t* __restrict__ colscale,
    const uint16_t* __restrict__ bias, int M, int N, int K, int r, uint16_t* __restrict__ Y, uint8_t* __restrict__ ws,
    int32_t* __restrict__ P, int KS) {
    using C = FCfg<TOKN>;
    constexpr int kT = C::kT;
    extern __shared__ uint8_t smdyn[];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag, never_abort;
    const FPlan PL = fplan(TOKN, r, KS);
    const uint32_t raw = smem_u32(smdyn);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smraw = smdyn + (sbase - raw);
    const uint32_t bar0 = sbase + PL.bar;
    const uint32_t xfull = bar0, ldfull = bar0 + 8, lfull = bar0 + 16, lrecv_full = bar0 + 24, aready = bar0 + 32,
                   tlora = bar0 + 40, mmadone = bar0 + 48, red_full = bar0 + 56;
    auto sfull = [&](int i) { return bar0 + 64u + 8u * i; };             // weight scales of group i landed
    auto tfull = [&](int t) { return bar0 + 128u + 8u * t; };            // product buffer t written
    auto tfree = [&](int t) { return bar0 + 128u + 8u * (kT + t); };     // product buffer t read

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / kGroup, RP = r / 16, NT = r / 8;
    const PackedLayout WLY = packed_layout(N, K, r);
    const ActLayout AL = act_layout(M, K, r);
    const int kr = KS > 1 ? int(cluster_ctarank()) : 0;
    const int ntile = blockIdx.x / KS;
    const int g_begin = (G * kr) / KS, n_groups = (G * (kr + 1)) / KS - g_begin;
    const int nbase = ntile * kRows;
    const int rows_valid = min(kRows, N - nbase);  // a multiple of 16
    const int mvalid = min(M, TOKN);
    const int BLKV = (mvalid + 3) / 4;             // token blocks holding a valid token
    int owned = 0;
    for (int b = kr; b < BLKV; b += KS) ++owned;
    const bool lora_owner = r > 0 && owned > 0;
    volatile int* abort = &abort_flag;
    constexpr uint32_t IDESC = idesc_m128(TOKN);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        never_abort = 0;
        mbar_init(xfull, 128);  // one cp.async arrival per staging thread
        mbar_init(ldfull, 1);
        mbar_init(lfull, 1);
        mbar_init(lrecv_full, 3);  // the expected bytes + this CTA's two LoRA-down warps
        mbar_init(aready, 4);
        mbar_init(tlora, 1);
        mbar_init(mmadone, 1);
        mbar_init(red_full, 1);
        for (int i = 0; i < kMaxG; ++i) mbar_init(sfull(i), 1);
        for (int t = 0; t < kT; ++t) {
            mbar_init(tfull(t), 1);
            mbar_init(tfree(t), 4);
        }
        fence_mbar_init();
        if (KS > 1 && owned > 0) mbar_expect_tx(red_full, uint32_t((KS - 1) * kRows * owned * 16));
        if (lora_owner) mbar_expect_tx(lrecv_full, uint32_t((KS - 1) * C::WL * owned * 4 * r * 4));
    }
    if (warp == WARP_AUX) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (KS > 1) cluster_arrive_release();  // phase 1: this CTA's barriers are set up
    // Overlapping the previous kernel: warm L2 with this CTA's weights, scales and
    // LoRA operands (a prefetch only fills the cache; every load comes after the wait).
    if (warp == WARP_LD && lane == 0) {
        for (int i = 0; i < n_groups; ++i) {
            prefetch_l2(packed + WLY.qW + ((size_t)(g_begin + i) * N + nbase) * 32, uint32_t(rows_valid) * 32);
            prefetch_l2(packed + WLY.sW + ((size_t)(g_begin + i) * N + nbase) * 2, uint32_t(rows_valid) * 2);
        }
        if (r > 0) prefetch_l2(packed + WLY.Ld + (size_t)g_begin * NT * 1024, uint32_t(n_groups * NT * 1024));
        if (lora_owner)
            for (int p = 0; p < RP; ++p)
                prefetch_l2(packed + WLY.Lu + ((size_t)p * N + nbase) * 32, uint32_t(rows_valid) * 32);
    }
    pdl_wait();
    pdl_launch_dependents();

    const bool is_q = warp >= WARP_Q0;
    const int row = (warp & 3) * 32 + lane;  // weight row = tensor-memory lane (warps 0-3 and 6-9)
    uint64_t acc[TOKN / 2];                  // (warps 6-9) running sums, token pairs
#pragma unroll
    for (int c = 0; c < TOKN / 2; ++c) acc[c] = 0ull;

    if (warp < 4) {
        // ---- weight rows -> bytes in tensor memory; warp 0 issues the group MMAs
        uint4 wr[kMaxG][2];
        const bool rv = row < rows_valid;
        const uint8_t* wsrc = packed + WLY.qW + ((size_t)g_begin * N + nbase + row) * 32;
#pragma unroll
        for (int i = 0; i < kMaxG; ++i) {
            if (i < n_groups && rv) {
                wr[i][0] = ldg_stream_v4(wsrc + (size_t)i * N * 32);
                wr[i][1] = ldg_stream_v4(wsrc + (size_t)i * N * 32 + 16);
            } else {
                wr[i][0] = wr[i][1] = make_uint4(0, 0, 0, 0);
            }
        }
        if (KS > 1) {
            cluster_wait_acquire();   // (phase 1)
            cluster_arrive_release();  // phase 2: these warps never touch the X staging area
        }
        const uint32_t tl = tmem + (uint32_t(warp * 32) << 16);
#pragma unroll
        for (int i = 0; i < kMaxG; ++i) {
            if (i >= n_groups) break;
            // word c holds k = 4c .. 4c+3 (byte k % 4); the record's words give k in
            // 16-byte chunks (w0.x, w0.z, w1.x, w1.z: k 0-15 low nibbles, 16-31 high;
            // w0.y, w0.w, w1.y, w1.w: k 32-63 likewise)
            uint32_t a[16];
            expand8(wr[i][0].x, a[0], a[4]);
            expand8(wr[i][0].z, a[1], a[5]);
            expand8(wr[i][1].x, a[2], a[6]);
            expand8(wr[i][1].z, a[3], a[7]);
            expand8(wr[i][0].y, a[8], a[12]);
            expand8(wr[i][0].w, a[9], a[13]);
            expand8(wr[i][1].y, a[10], a[14]);
            expand8(wr[i][1].w, a[11], a[15]);
            tmem_st16_b32(tl + uint32_t(i * 16), a);
            tmem_wait_st();
            tc_fence_before();
            if (named_bar_red_or(BAR_EXP, 128, *abort != 0)) break;  // the same decision in all four warps
            if (warp == 0 && lane == 0) {
                bool ok = true;
                if (i == 0) ok = wait_parity_suspend(aready, 0u, abort, kWaitNs, kSuspendNs);
                const int tb = i % kT;
                if (ok && i >= kT)
                    ok = wait_parity_suspend(tfree(tb), uint32_t((i / kT) - 1) & 1u, abort, kWaitNs, kSuspendNs);
                if (!ok) {
                    atomicExch(&g_fused_status, int(W4A4_ERR_TIMEOUT));
                    *abort = 1;
                } else {
                    tc_fence_after();
                    const uint32_t d = tmem + C::DCOL + uint32_t(tb * TOKN);
                    const uint32_t at = tmem + uint32_t(i * 16);
                    const uint32_t b0 = sbase + PL.aq + uint32_t(i) * (2 * TOKN * 32);
                    mma_f8_tmem_a(d, at, sdesc_sw32(b0), IDESC, 0u);
                    mma_f8_tmem_a(d, at + 8, sdesc_sw32(b0 + TOKN * 32), IDESC, 1u);
                    mma_commit(tfull(tb));
                }
            }
            __syncwarp();
        }
        if (warp == 0 && lane == 0) {
            mma_commit(mmadone);  // every group MMA issued above has completed once this arrives
            wait_parity_suspend(mmadone, 0u, &never_abort, kWaitNs, kSuspendNs);
        }
        __syncwarp();
    } else if (warp == WARP_LD || warp == WARP_AUX) {
        const int w = warp - WARP_LD;
        if (lane == 0) {
            if (warp == WARP_LD) {
                if (r > 0) {
                    const uint32_t lb = uint32_t(n_groups * NT * 1024);
                    mbar_expect_tx(ldfull, lb);
                    bulk_g2s(sbase + PL.ldst, packed + WLY.Ld + (size_t)g_begin * NT * 1024, lb, ldfull);
                }
                if (lora_owner) {
                    mbar_expect_tx(lfull, uint32_t(RP * rows_valid * 32));
                    for (int p = 0; p < RP; ++p)
                        bulk_g2s(sbase + PL.lu + uint32_t(p) * (kRows * 32),
                                 packed + WLY.Lu + ((size_t)p * N + nbase) * 32, uint32_t(rows_valid) * 32, lfull);
                }
            } else {
                for (int i = 0; i < n_groups; ++i) {
                    mbar_expect_tx(sfull(i), uint32_t(rows_valid) * 2);
                    bulk_g2s(sbase + PL.sw + uint32_t(i) * (kRows * 2),
                             packed + WLY.sW + ((size_t)(g_begin + i) * N + nbase) * 2, uint32_t(rows_valid) * 2,
                             sfull(i));
                }
            }
        }
        __syncwarp();
        // ---- LoRA down of this rank's K slice: the staged fp16 X through ldmatrix
        // into mma.m16n8k16 with the staged L_down fragments (fp32 accumulate)
        float la[kMaxR / 8][4];
#pragma unroll
        for (int t = 0; t < kMaxR / 8; ++t) la[t][0] = la[t][1] = la[t][2] = la[t][3] = 0.f;
        const int mt = TOKN == 32 ? w : 0;
        const int i0 = TOKN == 32 ? 0 : (w == 0 ? 0 : (n_groups + 1) / 2);
        const int i1 = TOKN == 32 ? n_groups : (w == 0 ? (n_groups + 1) / 2 : n_groups);
        if (r > 0) {
            const bool ok = warp_wait_parity_suspend(xfull, 0u, abort, kWaitNs, kSuspendNs) &&
                            warp_wait_parity_suspend(ldfull, 0u, abort, kWaitNs, kSuspendNs);
            if (!ok) {
                if (lane == 0) {
                    atomicExch(&g_fused_status, int(W4A4_ERR_TIMEOUT));
                    *abort = 1;
                }
            } else {
                const int lr = (lane & 7) + ((lane >> 3) & 1) * 8, lc = ((lane >> 4) & 1) * 8;
                const uint32_t xa = sbase + PL.xs + uint32_t((mt * 16 + lr) * kXStride + lc) * 2;
                for (int i = i0; i < i1; ++i) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        uint32_t a[4];
                        ldsm_x4(a, xa + uint32_t(i * kGroup + ks * 16) * 2);
                        const uint2* bp =
                            reinterpret_cast<const uint2*>(smraw + PL.ldst) + ((i * 4 + ks) * NT) * 32 + lane;
#pragma unroll
                        for (int t = 0; t < kMaxR / 8; ++t)
                            if (t < NT) {
                                const uint2 b = bp[t * 32];
                                mma_f16_16816(la[t], a, b.x, b.y);
                            }
                    }
                }
            }
        }
        if (KS > 1) cluster_wait_acquire();  // (phase 1: every rank's receive barriers are set up)
        if (r > 0) {
            // lane (gid, tig) holds rows gid and gid + 8 of the m tile, columns 2 tig, 2 tig + 1
            // of each 16 x 8 tile: push each valid row to its block's owner
            const int gid = lane >> 2, tig = lane & 3;
            const int wl = TOKN == 16 ? w : 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int t = mt * 16 + gid + 8 * h, b = t >> 2;
                if (b >= BLKV) continue;
                const int o = b % KS, ob = b / KS;
                const uint32_t off =
                    uint32_t(((((kr * C::WL + wl) * PL.own + ob) * 4 + (t & 3)) * r + 2 * tig) * 4);
#pragma unroll
                for (int tt = 0; tt < kMaxR / 8; ++tt) {
                    if (tt >= NT) break;
                    const uint32_t dst = sbase + PL.lrecv + off + uint32_t(tt * 8 * 4);
                    if (o == kr) {
                        *reinterpret_cast<float2*>(smraw + PL.lrecv + off + tt * 8 * 4) =
                            make_float2(la[tt][2 * h], la[tt][2 * h + 1]);
                    } else {
                        st_async_v2(mapa_shared(dst, uint32_t(o)), la[tt][2 * h], la[tt][2 * h + 1],
                                    mapa_shared(lrecv_full, uint32_t(o)));
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(lrecv_full);  // this warp's own rows are in place
        }
        if (KS > 1) cluster_arrive_release();  // phase 2: done with the X staging area
        if (warp == WARP_AUX && lora_owner) {
            // ---- LoRA-down sums of the owned blocks (rank order), fp16, then LoRA up
            bool ok = warp_wait_parity_suspend(lrecv_full, 0u, abort, kWaitNs, kSuspendNs);
            if (ok) {
                const float* rv = reinterpret_cast<const float*>(smraw + PL.lrecv);
                for (int e = lane; e < owned * 4 * r; e += 32) {
                    const int ob = e / (4 * r), rem = e % (4 * r), rw = rem / r, j = rem % r;
                    float v = 0.f;
                    for (int rk = 0; rk < KS; ++rk)
#pragma unroll
                        for (int s2 = 0; s2 < C::WL; ++s2)
                            v += rv[((((rk * C::WL + s2) * PL.own + ob) * 4 + rw) * r) + j];
                    const int t = 4 * (kr + ob * KS) + rw;  // token
                    const int p = j >> 4, jj = j & 15;
                    const uint16_t hv = __half_as_ushort(__float2half_rn(v));
                    *reinterpret_cast<uint16_t*>(smraw + PL.la + p * (TOKN * 32) + t * 32 + swz32(t, jj >> 3) * 16 +
                                                 (jj & 7) * 2) = hv;
                    if (ws != nullptr && t < M)
                        reinterpret_cast<uint16_t*>(ws + AL.La)[((size_t)p * kTileM + t) * 16 + swz32(t, jj >> 3) * 8 +
                                                                (jj & 7)] = hv;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ok = wait_parity_suspend(lfull, 0u, abort, kWaitNs, kSuspendNs);
                    if (ok) {
                        tc_fence_after();
                        for (int p = 0; p < RP; ++p)
                            mma_f16(tmem + C::LCOL, sdesc_sw32(sbase + PL.lu + uint32_t(p) * (kRows * 32)),
                                    sdesc_sw32(sbase + PL.la + uint32_t(p) * (TOKN * 32)), IDESC, p > 0 ? 1u : 0u);
                        mma_commit(tlora);
                        wait_parity_suspend(tlora, 0u, &never_abort, kWaitNs, kSuspendNs);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            }
            if (!ok && lane == 0) {
                atomicExch(&g_fused_status, int(W4A4_ERR_TIMEOUT));
                *abort = 1;
            }
        }
    } else {
        // ---- warps 6-9: stage and quantise X, then the epilogue
        const int q = warp - WARP_Q0, tq = q * 32 + lane;
        const int cpr = n_groups * 8;  // 16-byte chunks per row of the slice
        const uint16_t* xg = X + (size_t)g_begin * kGroup;
        for (int c = tq; c < TOKN * cpr; c += 128) {
            const int t = c / cpr, ch = c % cpr;
            const bool v = t < M;
            cp_async16_zfill(sbase + PL.xs + uint32_t(t * kXStride + ch * 8) * 2, xg + (size_t)(v ? t : 0) * K + ch * 8,
                             v ? 16u : 0u);
        }
        cp_async_mbar_arrive_noinc(xfull);
        bool ok = warp_wait_parity_suspend(xfull, 0u, abort, kWaitNs, kSuspendNs);
        if (ok) {
            // lane pair (2 u, 2 u + 1) quantises row u of the m tile, one half-group each
            constexpr int WPM = TOKN == 32 ? 2 : 4;  // warps per m tile
            const int mt = q / WPM, qsel = q % WPM;
            const int qrow = lane >> 1, qh = lane & 1;
            const int t = mt * 16 + qrow;
            for (int i = qsel; i < n_groups; i += WPM) {
                const uint8_t* xr = smraw + PL.xs + (size_t)(t * kXStride + i * kGroup + qh * 32) * 2;
                uint4 xv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) xv[j] = *reinterpret_cast<const uint4*>(xr + 16 * j);
                float s, csum;
                uint32_t pk[8];
                quantize_half_group(xv, s, csum, pk);
                uint8_t* plane = smraw + PL.aq + (size_t)(i * 2 + qh) * (TOKN * 32) + t * 32;
                *reinterpret_cast<uint4*>(plane + swz32(t, 0) * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4*>(plane + swz32(t, 1) * 16) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                if (qh == 0) {
                    float* sc = reinterpret_cast<float*>(smraw + PL.sc) + (size_t)i * 3 * TOKN;
                    sc[t] = s * kExpand8Scale;            // 2^9 sA (the products are 2^-9 D)
                    sc[TOKN + t] = (-8.f * csum) * s;     // -8 SA sA
                    sc[2 * TOKN + t] = csum;              // SA
                }
                if (ws != nullptr && t < M) {
                    const int g = g_begin + i;
                    uint8_t* wp = ws + AL.qA + ((size_t)g * 2 + qh) * (kTileM * 32) + t * 32;
                    *reinterpret_cast<uint4*>(wp + swz32(t, 0) * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    *reinterpret_cast<uint4*>(wp + swz32(t, 1) * 16) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    if (qh == 0)
                        *reinterpret_cast<float2*>(ws + AL.sS + ((size_t)g * kTileM + t) * 8) = make_float2(s, csum);
                }
            }
        } else if (lane == 0) {
            atomicExch(&g_fused_status, int(W4A4_ERR_TIMEOUT));
            *abort = 1;
        }
        fence_proxy_async_smem();  // the codes are read by the tensor core
        named_bar_sync(BAR_Q, 128);  // every warp's codes and scales are in place
        if (lane == 0) mbar_arrive(aready);
        if (KS > 1) {
            cluster_wait_acquire();   // (phase 1)
            cluster_arrive_release();  // phase 2: done with the X staging area
        }

        // ---- epilogue: one group at a time as its product lands
        const uint32_t tl = tmem + (uint32_t((warp & 3) * 32) << 16);
        for (int i = 0; i < n_groups && ok; ++i) {
            const int tb = i % kT;
            if (!warp_wait_parity_suspend(tfull(tb), uint32_t(i / kT) & 1u, abort, kWaitNs, kSuspendNs) ||
                !warp_wait_parity_suspend(sfull(i), 0u, abort, kWaitNs, kSuspendNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float d[TOKN];
            if constexpr (TOKN == 16) {
                tmem_ld16(tl + C::DCOL + uint32_t(tb * TOKN), d);
            } else {
                tmem_ld32(tl + C::DCOL + uint32_t(tb * TOKN), d);
            }
            tmem_wait_ld();
            const float* sc = reinterpret_cast<const float*>(smraw + PL.sc) + (size_t)i * 3 * TOKN;
            if (DUMP && nbase + row < N) {
                // partials dump: P = 2^9 D - 8 SA, exact in fp32 (|2^9 D| < 2^13)
                const int g = g_begin + i, n = nbase + row;
#pragma unroll
                for (int c = 0; c < TOKN; ++c)
                    if (c < M) P[((size_t)c * N + n) * G + g] = int32_t(d[c] * kExpand8Scale - 8.f * sc[2 * TOKN + c]);
            }
            const float sw = __half2float(
                __ushort_as_half(reinterpret_cast<const uint16_t*>(smraw + PL.sw + i * (kRows * 2))[row]));
            const uint64_t sw2 = f2_pack(sw, sw);
            const uint64_t* sa2 = reinterpret_cast<const uint64_t*>(sc);
            const uint64_t* cc2 = sa2 + TOKN / 2;
#pragma unroll
            for (int c = 0; c < TOKN / 2; ++c)
                acc[c] = ffma2_b64(sw2, ffma2_b64(sa2[c], f2_pack(d[2 * c], d[2 * c + 1]), cc2[c]), acc[c]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tfree(tb));
        }
        if (ok && lora_owner) {
            // the LoRA-up product of the owned blocks joins this rank's sums before the exchange
            if (!warp_wait_parity_suspend(tlora, 0u, abort, kWaitNs, kSuspendNs)) {
                ok = false;
            } else {
                tc_fence_after();
                float l[TOKN];
                if constexpr (TOKN == 16) {
                    tmem_ld16(tl + C::LCOL, l);
                } else {
                    tmem_ld32(tl + C::LCOL, l);
                }
                tmem_wait_ld();
#pragma unroll
                for (int b = 0; b < C::BLK; ++b) {
                    if (b % KS != kr || b >= BLKV) continue;
                    acc[2 * b] = fadd2_b64(acc[2 * b], f2_pack(l[4 * b], l[4 * b + 1]));
                    acc[2 * b + 1] = fadd2_b64(acc[2 * b + 1], f2_pack(l[4 * b + 2], l[4 * b + 3]));
                }
            }
        }
        if (!ok && lane == 0) {
            atomicExch(&g_fused_status, int(W4A4_ERR_TIMEOUT));
            *abort = 1;
        }
    }

    // ---- all roles are done with tensor memory
    tc_fence_before();
    const bool aborted = __syncthreads_or(*abort);
    if (warp == WARP_AUX) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (aborted && threadIdx.x == 0) {
        // let the copies already requested land before this CTA's shared memory goes away
        wait_parity_suspend(xfull, 0u, &never_abort, kWaitNs, kSuspendNs);
        if (r > 0) wait_parity_suspend(ldfull, 0u, &never_abort, kWaitNs, kSuspendNs);
        if (lora_owner) wait_parity_suspend(lfull, 0u, &never_abort, kWaitNs, kSuspendNs);
        for (int i = 0; i < n_groups; ++i) wait_parity_suspend(sfull(i), 0u, &never_abort, kWaitNs, kSuspendNs);
    }

    // ---- exchange: token block b belongs to rank b % KS
    if (KS > 1) {
        cluster_wait_acquire();  // phase 2: every rank is done with its X staging area (the receive area)
        if (is_q) {
#pragma unroll
            for (int b = 0; b < C::BLK; ++b) {
                const int o = b % KS;
                if (b >= BLKV || o == kr) continue;
                const int sidx = kr < o ? kr : kr - 1, ob = b / KS;
                const uint32_t dst =
                    mapa_shared(sbase + PL.xs + uint32_t((sidx * kRows + row) * PL.own + ob) * 16, uint32_t(o));
                const float2 p0 = f2_unpack(acc[2 * b]), p1 = f2_unpack(acc[2 * b + 1]);
                st_async_v4(dst, make_float4(p0.x, p0.y, p1.x, p1.y), mapa_shared(red_full, uint32_t(o)));
            }
            if (owned > 0) {
                if (!warp_wait_parity_suspend(red_full, 0u, abort, kWaitNs, kSuspendNs)) {
                    if (lane == 0) {
                        atomicExch(&g_fused_status, int(W4A4_ERR_TIMEOUT));
                        *abort = 1;
                    }
                } else {
                    const float* red = reinterpret_cast<const float*>(smraw + PL.xs);
#pragma unroll
                    for (int b = 0; b < C::BLK; ++b) {
                        if (b % KS != kr || b >= BLKV) continue;
                        const int ob = b / KS;
                        float2 p0 = f2_unpack(acc[2 * b]), p1 = f2_unpack(acc[2 * b + 1]);
                        for (int rk = 0; rk < KS; ++rk) {
                            if (rk == kr) continue;
                            const int sidx = rk < kr ? rk : rk - 1;
                            const float4 v = *reinterpret_cast<const float4*>(red + ((sidx * kRows + row) * PL.own + ob) * 4);
                            p0.x += v.x, p0.y += v.y, p1.x += v.z, p1.y += v.w;
                        }
                        acc[2 * b] = f2_pack(p0.x, p0.y);
                        acc[2 * b + 1] = f2_pack(p1.x, p1.y);
                    }
                }
            }
        }
        cluster_arrive_release();  // phase 3: this rank's part of the exchange is done
    }

    // ---- affine of the owned valid blocks, staged as rows [token][128 + 8] over the code planes
    uint16_t* ys = reinterpret_cast<uint16_t*>(smraw + PL.aq);
    constexpr int LDY = kRows + 8;
    if (!DUMP && is_q && !*abort) {
        const int n = nbase + row;
        const float cs = n < N ? __half2float(__ushort_as_half(colscale[n])) : 0.f;
        const float bs = (bias && n < N) ? __half2float(__ushort_as_half(bias[n])) : 0.f;
#pragma unroll
        for (int b = 0; b < C::BLK; ++b) {
            if (b % KS != kr || b >= BLKV) continue;
            const float2 p0 = f2_unpack(acc[2 * b]), p1 = f2_unpack(acc[2 * b + 1]);
            ys[(4 * b + 0) * LDY + row] = __half_as_ushort(__float2half_rn(fmaf(cs, p0.x, bs)));
            ys[(4 * b + 1) * LDY + row] = __half_as_ushort(__float2half_rn(fmaf(cs, p0.y, bs)));
            ys[(4 * b + 2) * LDY + row] = __half_as_ushort(__float2half_rn(fmaf(cs, p1.x, bs)));
            ys[(4 * b + 3) * LDY + row] = __half_as_ushort(__float2half_rn(fmaf(cs, p1.y, bs)));
        }
    }
    __syncthreads();
    if (!DUMP && !*abort) {
        for (int c = threadIdx.x; c < TOKN * (kRows / 8); c += kThreads) {
            const int t = c / (kRows / 8), ch = c % (kRows / 8);
            const int n = nbase + ch * 8;
            if ((t / 4) % KS != kr) continue;
            if (t < M && n < N)
                *reinterpret_cast<uint4*>(Y + (size_t)t * N + n) = *reinterpret_cast<const uint4*>(&ys[t * LDY + ch * 8]);
        }
    }
    if (KS > 1) cluster_wait_acquire();  // phase 3: no rank leaves while a peer may still address its shared memory
}

// Split factor: enough CTAs to cover the SMs twice, and at most kMaxG groups per CTA.
int fused_split(int N, int K) {
    const int tiles = (N + kRows - 1) / kRows;
    const int G = K / kGroup;
    int ks = 1;
    while (ks < kMaxKS && tiles * ks * 2 <= device_sm_count() * 2 && ks * 2 <= G) ks *= 2;
    while (ks < kMaxKS && (G + ks - 1) / ks > kMaxG) ks *= 2;
    return ks;
}

constexpr uint32_t kSmemBudget = 110 * 1024;  // two CTAs per SM

template <int TOKN, bool DUMP>
w4a4_status launch_t(const uint16_t* X, const uint8_t* packed, const uint16_t* cs, const uint16_t* bias, int M, int N,
                     int K, int r, uint16_t* Y, uint8_t* ws, int32_t* P, cudaStream_t s) {
    const int KS = fused_split(N, K);
    const FPlan plan = fplan(TOKN, r, KS);
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(linear_fused_kernel<TOKN, DUMP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(kSmemBudget) + 1024) != cudaSuccess)
            return W4A4_ERR_CUDA;
        attr_done[dev] = 1;
    }
    dim3 grid(unsigned(((N + kRows - 1) / kRows) * KS));
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
    if (cudaLaunchKernelEx(&cfg, linear_fused_kernel<TOKN, DUMP>, X, packed, cs, bias, M, N, K, r, Y, ws, P, KS) !=
        cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    set_dispatch("linear_fused quantize+LoRA+tcgen05.f8f6f4 swap-AB N=%d split-K=%d (cluster) grid=%u%s", TOKN, KS,
                 grid.x, DUMP ? " (partials dump)" : "");
    return launch_status();
}

}  // namespace

bool fused_eligible(int M, int N, int K, int r) {
    if (M < 1 || M > 32 || r > kMaxR || r % 16 != 0 || K % kGroup != 0 || N % 16 != 0) return false;
    const int KS = fused_split(N, K);
    const int G = K / kGroup;
    if ((G + KS - 1) / KS > kMaxG || G < KS) return false;
    return fplan(M <= 16 ? 16 : 32, r, KS).total <= kSmemBudget;
}

w4a4_status fused_read_and_clear_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fused_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_fused_status, &zero, sizeof(int));
        return W4A4_ERR_TIMEOUT;
    }
    return W4A4_OK;
}

w4a4_status launch_linear_fused(const uint16_t* X, const uint8_t* packed, const uint16_t* colscale,
                                const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, uint8_t* ws,
                                int32_t* P_dump, cudaStream_t s) {
    if (P_dump) {
        if (M <= 16) return launch_t<16, true>(X, packed, nullptr, nullptr, M, N, K, r, nullptr, ws, P_dump, s);
        return launch_t<32, true>(X, packed, nullptr, nullptr, M, N, K, r, nullptr, ws, P_dump, s);
    }
    if (M <= 16) return launch_t<16, false>(X, packed, colscale, bias, M, N, K, r, Y, ws, nullptr, s);
    return launch_t<32, false>(X, packed, colscale, bias, M, N, K, r, Y, ws, nullptr, s);
}

}  // namespace w4a4
