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
// latency, not by its bytes.  Each CTA (128 weight rows x a slice of K groups,
// the slice split over a cluster of KS CTAs) therefore starts every transfer
// it needs right after the launch dependency and computes while the weights
// arrive.  The weights and the LoRA-down fragments move by bulk copy (the
// copy engine, not the load/store pipe, which the X staging and the
// quantisation use at the same time) through 4-slot rings.
//
// Per group g, D[n, m] = 2^-9 sum_k (cW[n,k] + 8) cA[m,k] exactly (the weight
// bytes are the offset codes, read by E4M3 as u * 2^-9; the weights are the
// MMA's 128-row A operand, held in tensor memory, and the tokens its N), and
// the epilogue adds sW[n,g] (2^9 sA[m,g] D - 8 SA sA) to fp32 sums (one thread
// per weight row, one column pair per two tokens).
//
// Roles (10 warps, two CTAs per SM):
//   warps 0-3  expand each group's weight nibbles (their 32 rows) to bytes in
//              tensor memory and hand the group to warp 4 (a named barrier
//              per group, arrive only);
//   warp 4     bulk copies of the weights (the ring: slot i % 4 is refilled
//              with group i + 4 once group i is handed over) and, on token-
//              block owners, of the LoRA-up planes; issues the group MMAs
//              (one thread, two kind::f8f6f4 MMAs per group);
//   warp 5     tensor-memory owner; bulk copies of the weight scales and of the
//              LoRA-down fragments (its own ring); the LoRA down of every
//              token row (mma.m16n8k16 from the staged X); on owners the sum of
//              the cluster's LoRA-down partials (rank order), fp16, and the
//              kind::f16 LoRA-up MMAs;
//   warps 6-9  stage the X slice (cp.async), quantise it (the same arithmetic
//              as the activation kernel: codes, sA, SA bit for bit) into the
//              B operand, then run the per-group epilogue.
// Token block b (4 tokens) belongs to cluster rank b % KS: the other ranks
// push their LoRA-down partials and, at the end, their fp32 sums of the block
// there (st.async), and the owner adds them in rank order, adds its LoRA-up
// product, applies the affine and stores Y.  Only blocks holding a valid token
// take part.  Cluster barrier phases: (1) every rank's mbarriers are set up,
// (2) every rank is done with its X staging area, which then receives the
// partial sums, (3) every rank is done with the exchange.  Every mbarrier wait
// is bounded (2 s; W4A4_ERR_TIMEOUT in the status word); on give-up every role
// unwinds but still passes every named and cluster barrier (the expansion
// warps arrive on every group's handoff barrier), the MMAs issued are waited
// for, tensor memory is freed and the copies in flight land before exit.
#include "kernels.h"
#include "quant.cuh"
#include "tc_ptx.cuh"

namespace w4a4 {
namespace {
using namespace tc;

constexpr int kRows = 128;   // weight rows per CTA (MMA M, tensor-memory lanes)
constexpr int kThreads = 320;
constexpr int WARP_MMA = 4, WARP_AUX = 5, WARP_Q0 = 6;
constexpr int kMaxKS = 8;
constexpr int kMaxG = 8;     // K groups per CTA
constexpr int kMaxR = 32;    // LoRA rank
constexpr int kXStride = kMaxG * kGroup + 8;  // halves per staged X row (+8: conflict-free ldmatrix)
constexpr uint32_t kTmemCols = 256;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kSuspendNs = 20000;
// named barriers: 2 + i the handoff of group i (expansion -> MMA warp); 10 the epilogue
// warps' staged Y; 11 every thread, once every role is done with tensor memory
constexpr uint32_t BAR_G0 = 2, BAR_Y = 2 + kMaxG, BAR_END = 3 + kMaxG;
constexpr uint32_t kHandoff = 5 * 32;  // four expansion warps arrive, the MMA warp syncs

__device__ int g_fused_status = 0;

template <int TOKN>
struct FCfg {
    static constexpr int kT = TOKN == 16 ? 7 : 3;   // product buffers in tensor memory
    static constexpr uint32_t DCOL = kMaxG * 16;     // A operand: 16 columns per group, then the products
    static constexpr uint32_t LCOL = DCOL + kT * TOKN;
    static constexpr int BLK = TOKN / 4;
    static constexpr int MT = TOKN / 16;             // m16 tiles of the LoRA down
    static_assert(LCOL + TOKN <= kTmemCols, "tensor memory plan");
};

// Byte offsets of the shared-memory sections (multiples of 16; the tensor
// core's operands at multiples of 1024 or of their plane size).  Only the last
// section, the LoRA-down receive area, depends on the cluster size.
template <int TOKN, int R>
struct FOff {
    static constexpr int RP = R / 16, NT = R / 8;
    static constexpr int RING = TOKN == 16 ? 8 : 4;  // every copy in flight at 16 tokens; 4-slot rings at 32
    static constexpr uint32_t lu = 0;                                        // [plane][128 rows][32 B]
    static constexpr uint32_t la = lu + uint32_t(RP) * kRows * 32;           // [plane][tokn][32 B]
    static constexpr uint32_t aq = (la + uint32_t(RP) * TOKN * 32 + 1023u) & ~1023u;  // [group][plane][tokn][32 B]
    static constexpr uint32_t wraw = aq + uint32_t(kMaxG) * 2 * TOKN * 32;  // weight records [slot][128][32 B]
    static constexpr uint32_t ldr = wraw + uint32_t(RING) * kRows * 32;     // LoRA-down fragments [slot][ks][tile][lane]
    static constexpr uint32_t xs = ldr + uint32_t(RING) * NT * 1024;        // X slice, later the partial sums received
    static constexpr uint32_t sw = xs + uint32_t(TOKN) * kXStride * 2;       // [group][128] fp16
    static constexpr uint32_t sc = sw + uint32_t(kMaxG) * kRows * 2;         // [group][2^9 sA | -8 SA sA | SA][tokn]
    static constexpr uint32_t bar = sc + uint32_t(kMaxG) * 3 * TOKN * 4;
    static constexpr uint32_t lrecv = bar + 512;                             // [rank][owned block][4 rows][R]
    // the partial sums received ((KS - 1) x 128 rows x owned blocks x 16 B) fit the X slice's area
    static_assert((kMaxKS - 1) * kRows * 16 * ((TOKN / 4 + kMaxKS - 1) / kMaxKS) <= TOKN * kXStride * 2 &&
                      3 * kRows * 16 * ((TOKN / 4 + 3) / 4) <= TOKN * kXStride * 2 &&
                      1 * kRows * 16 * ((TOKN / 4 + 1) / 2) <= TOKN * kXStride * 2,
                  "exchange area");
    static uint32_t __host__ __device__ total(int ks) {
        const int own = (TOKN / 4 + ks - 1) / ks;
        return lrecv + uint32_t(ks * own * 4 * R * 4);
    }
};

template <int TOKN, int R, bool DUMP>
__global__ void __launch_bounds__(kThreads, 2) linear_fused_kernel(
    const uint16_t* __restrict__ X, const uint8_t* __restrict__ packed, const uint16_t* __restrict__ colscale,
    const uint16_t* __restrict__ bias, int M, int N, int K, uint16_t* __restrict__ Y, uint8_t* __restrict__ ws,
    int32_t* __restrict__ P, int KS) {
    using C = FCfg<TOKN>;
    using FO = FOff<TOKN, R>;
    constexpr int RP = R / 16, NT = R / 8;
    constexpr int kRing = FO::RING;
    constexpr int r = R;
    constexpr int kT = C::kT;
    extern __shared__ uint8_t smdyn[];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag, never_abort, w_issued, l_issued;
    const uint32_t raw = smem_u32(smdyn);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smraw = smdyn + (sbase - raw);
    const uint32_t bar0 = sbase + FO::bar;
    const uint32_t xfull = bar0, lfull = bar0 + 8, lrecv_full = bar0 + 16, aready = bar0 + 24, tlora = bar0 + 32,
                   mmadone = bar0 + 40, red_full = bar0 + 48;
    auto rfull = [&](int s) { return bar0 + 64u + 8u * s; };             // weight slot s landed
    auto ldfull = [&](int s) { return bar0 + 128u + 8u * s; };           // LoRA-down slot s landed
    auto sfull = [&](int i) { return bar0 + 192u + 8u * i; };            // weight scales of group i landed
    auto tfull = [&](int t) { return bar0 + 256u + 8u * t; };            // product buffer t written
    auto tfree = [&](int t) { return bar0 + 256u + 8u * (kT + t); };     // product buffer t read

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const int own = (C::BLK + KS - 1) / KS;  // token blocks per rank
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
    const uint32_t wbytes = uint32_t(rows_valid) * 32, lbytes = uint32_t(NT) * 1024;
    auto issue_w = [&](int i) {  // weight records of group i into slot i % 4
        mbar_expect_tx(rfull(i % kRing), wbytes);
        bulk_g2s(sbase + FO::wraw + uint32_t(i % kRing) * (kRows * 32),
                 packed + packed_layout(N, K, R).qW + ((size_t)(g_begin + i) * N + nbase) * 32, wbytes, rfull(i % kRing));
    };
    auto issue_l = [&](int i) {  // LoRA-down fragments of group i into slot i % 4
        mbar_expect_tx(ldfull(i % kRing), lbytes);
        bulk_g2s(sbase + FO::ldr + uint32_t(i % kRing) * lbytes, packed + packed_layout(N, K, R).Ld + (size_t)(g_begin + i) * lbytes,
                 lbytes, ldfull(i % kRing));
    };

    if (threadIdx.x == 0) {
        abort_flag = 0;
        never_abort = 0;
        w_issued = 0;
        l_issued = 0;
        mbar_init(xfull, 128);     // one cp.async arrival per staging thread
        mbar_init(lfull, 1);
        mbar_init(lrecv_full, 2);  // the expected bytes + this CTA's own rows
        mbar_init(aready, 8);  // the eight quantising warps
        mbar_init(tlora, 1);
        mbar_init(mmadone, 1);
        mbar_init(red_full, 1);
        for (int s2 = 0; s2 < kRing; ++s2) {
            mbar_init(rfull(s2), 1);
            mbar_init(ldfull(s2), 1);
        }
        for (int i = 0; i < kMaxG; ++i) mbar_init(sfull(i), 1);
        for (int t = 0; t < kT; ++t) {
            mbar_init(tfull(t), 1);
            mbar_init(tfree(t), 4);
        }
        fence_mbar_init();
        if (KS > 1 && owned > 0) mbar_expect_tx(red_full, uint32_t((KS - 1) * kRows * owned * 16));
        if (lora_owner) mbar_expect_tx(lrecv_full, uint32_t((KS - 1) * owned * 4 * r * 4));
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
    if (warp == WARP_MMA && lane == 0) {
        for (int i = 0; i < n_groups; ++i) {
            prefetch_l2(packed + packed_layout(N, K, R).qW + ((size_t)(g_begin + i) * N + nbase) * 32, wbytes);
            prefetch_l2(packed + packed_layout(N, K, R).sW + ((size_t)(g_begin + i) * N + nbase) * 2, uint32_t(rows_valid) * 2);
        }
        if (r > 0) prefetch_l2(packed + packed_layout(N, K, R).Ld + (size_t)g_begin * lbytes, uint32_t(n_groups) * lbytes);
        if (lora_owner)
            for (int p = 0; p < RP; ++p) prefetch_l2(packed + packed_layout(N, K, R).Lu + ((size_t)p * N + nbase) * 32, wbytes);
    }
    pdl_wait();
    pdl_launch_dependents();

    const int row = (warp & 3) * 32 + lane;  // weight row = tensor-memory lane (warps 0-3 and 6-9)

    // Quantisation of the valid token rows, shared by the eight warps 0-3 and 6-9: the
    // (group, token) pairs in group order, 16 per warp pass (a lane pair each, one
    // half-group per lane), passes dealt round-robin (warps 6-9 first).  Rows of the
    // token block beyond M are never read as outputs, so they are left unwritten.
    auto quantise = [&](int qw) -> bool {  // qw: 0..7
        if (!warp_wait_parity_suspend(xfull, 0u, abort, kWaitNs, kSuspendNs)) return false;
        const int T = mvalid * n_groups;
        for (int pass = qw; pass * 16 < T; pass += 8) {
            const int p = pass * 16 + (lane >> 1), qh = lane & 1;
            const bool v = p < T;
            const int i = v ? p / mvalid : 0, t = v ? p % mvalid : 0;
            uint4 xv[4];
            const uint8_t* xr = smraw + FO::xs + (size_t)(t * kXStride + i * kGroup + qh * 32) * 2;
#pragma unroll
            for (int j = 0; j < 4; ++j) xv[j] = *reinterpret_cast<const uint4*>(xr + 16 * j);
            float s, csum;
            uint32_t pk[8];
            quantize_half_group(xv, s, csum, pk);  // (all 32 lanes: shuffles)
            if (!v) continue;
            uint8_t* plane = smraw + FO::aq + (size_t)(i * 2 + qh) * (TOKN * 32) + t * 32;
            *reinterpret_cast<uint4*>(plane + swz32(t, 0) * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(plane + swz32(t, 1) * 16) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            if (qh == 0) {
                float* sc = reinterpret_cast<float*>(smraw + FO::sc) + (size_t)i * 3 * TOKN;
                sc[t] = s * kExpand8Scale;         // 2^9 sA (the products are 2^-9 D)
                sc[TOKN + t] = (-8.f * csum) * s;  // -8 SA sA
                sc[2 * TOKN + t] = csum;           // SA
            }
            if (ws != nullptr) {
                const ActLayout AL = act_layout(M, K, R);
                const int g = g_begin + i;
                uint8_t* wp = ws + AL.qA + ((size_t)g * 2 + qh) * (kTileM * 32) + t * 32;
                *reinterpret_cast<uint4*>(wp + swz32(t, 0) * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4*>(wp + swz32(t, 1) * 16) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                if (qh == 0) *reinterpret_cast<float2*>(ws + AL.sS + ((size_t)g * kTileM + t) * 8) = make_float2(s, csum);
            }
        }
        return true;
    };
    auto quantise_done = [&](bool ok) {
        if (!ok && lane == 0) {
            atomicExch(&g_fused_status, int(W4A4_ERR_TIMEOUT));
            *abort = 1;
        }
        fence_proxy_async_smem();  // the codes are read by the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(aready);
        if (KS > 1) {
            cluster_wait_acquire();   // (phase 1)
            cluster_arrive_release();  // phase 2: done with the X staging area
        }
    };

    if (warp < 4) {
        quantise_done(quantise(4 + warp));
        // ---- weight rows -> bytes in tensor memory, group by group as the slots land
        const uint32_t tl = tmem + (uint32_t(warp * 32) << 16);
        for (int i = 0; i < n_groups; ++i) {
            // every group is handed over, also after a give-up, so the MMA warp's barrier always completes
            bool ok = !*abort &&
                      warp_wait_parity_suspend(rfull(i % kRing), uint32_t(i / kRing) & 1u, abort, kWaitNs, kSuspendNs);
            if (ok) {
                // word c holds k = 4c .. 4c+3 (byte k % 4); the record's words give k in
                // 16-byte chunks (w0.x, w0.z, w1.x, w1.z: k 0-15 low nibbles, 16-31 high;
                // w0.y, w0.w, w1.y, w1.w: k 32-63 likewise)
                const uint8_t* wr = smraw + FO::wraw + uint32_t(i % kRing) * (kRows * 32) + row * 32;
                const uint4 w0 = *reinterpret_cast<const uint4*>(wr);
                const uint4 w1 = *reinterpret_cast<const uint4*>(wr + 16);
                uint32_t a[16];
                expand8(w0.x, a[0], a[4]);
                expand8(w0.z, a[1], a[5]);
                expand8(w1.x, a[2], a[6]);
                expand8(w1.z, a[3], a[7]);
                expand8(w0.y, a[8], a[12]);
                expand8(w0.w, a[9], a[13]);
                expand8(w1.y, a[10], a[14]);
                expand8(w1.w, a[11], a[15]);
                tmem_st16_b32(tl + uint32_t(i * 16), a);
                tmem_wait_st();
            } else if (lane == 0) {
                atomicExch(&g_fused_status, int(W4A4_ERR_TIMEOUT));
                *abort = 1;
            }
            fence_proxy_async_smem();  // the slot's reads are done before the copy engine refills it
            tc_fence_before();
            named_bar_arrive(BAR_G0 + i, kHandoff);
        }
    } else if (warp == WARP_MMA) {
        // ---- weight ring and group MMAs
        if (lane == 0) {
            if (lora_owner) {
                mbar_expect_tx(lfull, uint32_t(RP) * wbytes);
                for (int p = 0; p < RP; ++p)
                    bulk_g2s(sbase + FO::lu + uint32_t(p) * (kRows * 32), packed + packed_layout(N, K, R).Lu + ((size_t)p * N + nbase) * 32,
                             wbytes, lfull);
            }
            const int n0 = min(n_groups, kRing);
            for (int i = 0; i < n0; ++i) issue_w(i);
            w_issued = n0;
        }
        __syncwarp();
        if (KS > 1) {
            cluster_wait_acquire();   // (phase 1)
            cluster_arrive_release();  // phase 2: this warp never touches the X staging area
        }
        for (int i = 0; i < n_groups; ++i) {
            named_bar_sync(BAR_G0 + i, kHandoff);  // group i is in tensor memory, its slot is free
            if (lane == 0 && !*abort) {
                if (i + kRing < n_groups) {
                    issue_w(i + kRing);
                    w_issued = i + kRing + 1;
                }
                const int tb = i % kT;
                bool ok = i > 0 || wait_parity_suspend(aready, 0u, abort, kWaitNs, kSuspendNs);
                if (ok && i >= kT)
                    ok = wait_parity_suspend(tfree(tb), uint32_t((i / kT) - 1) & 1u, abort, kWaitNs, kSuspendNs);
                if (!ok) {
                    atomicExch(&g_fused_status, int(W4A4_ERR_TIMEOUT));
                    *abort = 1;
                } else {
                    tc_fence_after();
                    const uint32_t d = tmem + C::DCOL + uint32_t(tb * TOKN);
                    const uint32_t at = tmem + uint32_t(i * 16);
                    const uint32_t b0 = sbase + FO::aq + uint32_t(i) * (2 * TOKN * 32);
                    mma_f8_tmem_a(d, at, sdesc_sw32(b0), IDESC, 0u);
                    mma_f8_tmem_a(d, at + 8, sdesc_sw32(b0 + TOKN * 32), IDESC, 1u);
                    mma_commit(tfull(tb));
                }
            }
            __syncwarp();
        }
        if (lane == 0) {
            mma_commit(mmadone);  // every group MMA issued above has completed once this arrives
            wait_parity_suspend(mmadone, 0u, &never_abort, kWaitNs, kSuspendNs);
        }
        __syncwarp();
    } else if (warp == WARP_AUX) {
        if (lane == 0) {
            for (int i = 0; i < n_groups; ++i) {
                mbar_expect_tx(sfull(i), uint32_t(rows_valid) * 2);
                bulk_g2s(sbase + FO::sw + uint32_t(i) * (kRows * 2),
                         packed + packed_layout(N, K, R).sW + ((size_t)(g_begin + i) * N + nbase) * 2, uint32_t(rows_valid) * 2, sfull(i));
            }
            if (r > 0) {
                const int n0 = min(n_groups, kRing);
                for (int i = 0; i < n0; ++i) issue_l(i);
                l_issued = n0;
            }
        }
        __syncwarp();
        // ---- LoRA down of this rank's K slice: the staged fp16 X through ldmatrix
        // into mma.m16n8k16 with the LoRA-down fragments (fp32 accumulate)
        float la[C::MT][kMaxR / 8][4];
#pragma unroll
        for (int m = 0; m < C::MT; ++m)
#pragma unroll
            for (int t = 0; t < kMaxR / 8; ++t) la[m][t][0] = la[m][t][1] = la[m][t][2] = la[m][t][3] = 0.f;
        if (r > 0) {
            bool ok = warp_wait_parity_suspend(xfull, 0u, abort, kWaitNs, kSuspendNs);
            const int lr = (lane & 7) + ((lane >> 3) & 1) * 8, lc = ((lane >> 4) & 1) * 8;
            const uint32_t xa = sbase + FO::xs + uint32_t(lr * kXStride + lc) * 2;
            for (int i = 0; i < n_groups && ok; ++i) {
                const int s2 = i % kRing;
                if (!warp_wait_parity_suspend(ldfull(s2), uint32_t(i / kRing) & 1u, abort, kWaitNs, kSuspendNs)) {
                    ok = false;
                    break;
                }
                const uint2* bp = reinterpret_cast<const uint2*>(smraw + FO::ldr + s2 * lbytes) + lane;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint2 b[kMaxR / 8];
#pragma unroll
                    for (int t = 0; t < kMaxR / 8; ++t)
                        if (t < NT) b[t] = bp[(ks * NT + t) * 32];
#pragma unroll
                    for (int m = 0; m < C::MT; ++m) {
                        uint32_t a[4];
                        ldsm_x4(a, xa + uint32_t(m * 16 * kXStride + i * kGroup + ks * 16) * 2);
#pragma unroll
                        for (int t = 0; t < kMaxR / 8; ++t)
                            if (t < NT) mma_f16_16816(la[m][t], a, b[t].x, b[t].y);
                    }
                }
                fence_proxy_async_smem();  // the slot's reads are done before the copy engine refills it
                __syncwarp();
                if (lane == 0 && i + kRing < n_groups) {
                    issue_l(i + kRing);
                    l_issued = i + kRing + 1;
                }
            }
            if (!ok && lane == 0) {
                atomicExch(&g_fused_status, int(W4A4_ERR_TIMEOUT));
                *abort = 1;
            }
        }
        if (KS > 1) cluster_wait_acquire();  // (phase 1: every rank's receive barriers are set up)
        if (r > 0) {
            // lane (gid, tig) holds rows gid and gid + 8 of each m tile, columns 2 tig, 2 tig + 1
            // of each 16 x 8 tile: each valid row goes to its block's owner
            const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
            for (int m = 0; m < C::MT; ++m)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = m * 16 + gid + 8 * h, b = t >> 2;
                    if (b >= BLKV) continue;
                    const int o = b % KS, ob = b / KS;
                    const uint32_t off = uint32_t((((kr * own + ob) * 4 + (t & 3)) * r + 2 * tig) * 4);
#pragma unroll
                    for (int tt = 0; tt < kMaxR / 8; ++tt) {
                        if (tt >= NT) break;
                        if (o == kr) {
                            *reinterpret_cast<float2*>(smraw + FO::lrecv + off + tt * 8 * 4) =
                                make_float2(la[m][tt][2 * h], la[m][tt][2 * h + 1]);
                        } else {
                            st_async_v2(mapa_shared(sbase + FO::lrecv + off + uint32_t(tt * 8 * 4), uint32_t(o)),
                                        la[m][tt][2 * h], la[m][tt][2 * h + 1], mapa_shared(lrecv_full, uint32_t(o)));
                        }
                    }
                }
            __syncwarp();
            if (lane == 0) mbar_arrive(lrecv_full);  // this CTA's own rows are in place
        }
        if (KS > 1) cluster_arrive_release();  // phase 2: done with the X staging area
        if (R > 0 && lora_owner) {
            // ---- LoRA-down sums of the owned blocks (rank order), fp16, then LoRA up
            bool ok = warp_wait_parity_suspend(lrecv_full, 0u, abort, kWaitNs, kSuspendNs);
            if (ok) {
                const float* rv = reinterpret_cast<const float*>(smraw + FO::lrecv);
                constexpr int RR = R > 0 ? R : 1;  // (R = 0 never gets here)
                for (int e = lane; e < owned * 4 * RR; e += 32) {
                    const int ob = e / (4 * RR), rem = e % (4 * RR), rw = rem / RR, j = rem % RR;
                    float v = 0.f;
                    for (int rk = 0; rk < KS; ++rk) v += rv[(((rk * own + ob) * 4 + rw) * r) + j];
                    const int t = 4 * (kr + ob * KS) + rw;  // token
                    const int p = j >> 4, jj = j & 15;
                    const uint16_t hv = __half_as_ushort(__float2half_rn(v));
                    *reinterpret_cast<uint16_t*>(smraw + FO::la + p * (TOKN * 32) + t * 32 + swz32(t, jj >> 3) * 16 +
                                                 (jj & 7) * 2) = hv;
                    if (ws != nullptr && t < M)
                        reinterpret_cast<uint16_t*>(ws + act_layout(M, K, R).La)[((size_t)p * kTileM + t) * 16 + swz32(t, jj >> 3) * 8 +
                                                                (jj & 7)] = hv;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ok = wait_parity_suspend(lfull, 0u, abort, kWaitNs, kSuspendNs);
                    if (ok) {
                        tc_fence_after();
                        for (int p = 0; p < RP; ++p)
                            mma_f16(tmem + C::LCOL, sdesc_sw32(sbase + FO::lu + uint32_t(p) * (kRows * 32)),
                                    sdesc_sw32(sbase + FO::la + uint32_t(p) * (TOKN * 32)), IDESC, p > 0 ? 1u : 0u);
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
            cp_async16_zfill(sbase + FO::xs + uint32_t(t * kXStride + ch * 8) * 2, xg + (size_t)(v ? t : 0) * K + ch * 8,
                             v ? 16u : 0u);
        }
        cp_async_mbar_arrive_noinc(xfull);
        bool ok = quantise(q);
        quantise_done(ok);
        // the epilogue reads every warp's scales: wait for all eight quantising warps
        ok = ok && warp_wait_parity_suspend(aready, 0u, abort, kWaitNs, kSuspendNs);

        // ---- epilogue: one group at a time as its product lands
        uint64_t acc[TOKN / 2];  // running sums, token pairs
#pragma unroll
        for (int c = 0; c < TOKN / 2; ++c) acc[c] = 0ull;
        const uint32_t tl = tmem + (uint32_t((warp & 3) * 32) << 16);
        for (int i = 0; i < n_groups && ok; ++i) {
            const int tb = i % kT;
            if (!warp_wait_parity_suspend(tfull(tb), uint32_t(i / kT) & 1u, abort, kWaitNs, kSuspendNs) ||
                !warp_wait_parity_suspend(sfull(i), 0u, abort, kWaitNs, kSuspendNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float* sc = reinterpret_cast<const float*>(smraw + FO::sc) + (size_t)i * 3 * TOKN;
            const float sw = __half2float(
                __ushort_as_half(reinterpret_cast<const uint16_t*>(smraw + FO::sw + i * (kRows * 2))[row]));
            const uint64_t sw2 = f2_pack(sw, sw);
            const uint64_t* sa2 = reinterpret_cast<const uint64_t*>(sc);
            const uint64_t* cc2 = sa2 + TOKN / 2;
#pragma unroll
            for (int h = 0; h < TOKN / 16; ++h) {  // 16 columns at a time
                float d[16];
                tmem_ld16(tl + C::DCOL + uint32_t(tb * TOKN + 16 * h), d);
                tmem_wait_ld();
                if (DUMP && nbase + row < N) {
                    // partials dump: P = 2^9 D - 8 SA, exact in fp32 (|2^9 D| < 2^13)
                    const int g = g_begin + i, n = nbase + row;
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        if (16 * h + c < M)
                            P[((size_t)(16 * h + c) * N + n) * G + g] =
                                int32_t(d[c] * kExpand8Scale - 8.f * sc[2 * TOKN + 16 * h + c]);
                }
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    acc[8 * h + c] = ffma2_b64(sw2, ffma2_b64(sa2[8 * h + c], f2_pack(d[2 * c], d[2 * c + 1]), cc2[8 * h + c]),
                                               acc[8 * h + c]);
            }
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
        tc_fence_before();
        named_bar_red_or(BAR_END, kThreads, *abort != 0);  // every role is done with tensor memory

        // ---- exchange: token block b belongs to rank b % KS
        if (KS > 1) {
            cluster_wait_acquire();  // phase 2: every rank is done with its X staging area (the receive area)
#pragma unroll
            for (int b = 0; b < C::BLK; ++b) {
                const int o = b % KS;
                if (b >= BLKV || o == kr) continue;
                const int sidx = kr < o ? kr : kr - 1, ob = b / KS;
                const uint32_t dst =
                    mapa_shared(sbase + FO::xs + uint32_t((sidx * kRows + row) * own + ob) * 16, uint32_t(o));
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
                    const float* red = reinterpret_cast<const float*>(smraw + FO::xs);
#pragma unroll
                    for (int b = 0; b < C::BLK; ++b) {
                        if (b % KS != kr || b >= BLKV) continue;
                        const int ob = b / KS;
                        float2 p0 = f2_unpack(acc[2 * b]), p1 = f2_unpack(acc[2 * b + 1]);
                        for (int rk = 0; rk < KS; ++rk) {
                            if (rk == kr) continue;
                            const int sidx = rk < kr ? rk : rk - 1;
                            const float4 v =
                                *reinterpret_cast<const float4*>(red + ((sidx * kRows + row) * own + ob) * 4);
                            p0.x += v.x, p0.y += v.y, p1.x += v.z, p1.y += v.w;
                        }
                        acc[2 * b] = f2_pack(p0.x, p0.y);
                        acc[2 * b + 1] = f2_pack(p1.x, p1.y);
                    }
                }
            }
            cluster_arrive_release();  // phase 3: this rank's part of the exchange is done
        }
        if constexpr (!DUMP) {
            // ---- affine of the owned valid blocks, staged as rows [token][128 + 8] over the code
            // planes (every group MMA has completed), then 16-byte stores by the four warps
            uint16_t* ys = reinterpret_cast<uint16_t*>(smraw + FO::aq);
            constexpr int LDY = kRows + 8;
            if (!*abort) {
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
            named_bar_sync(BAR_Y, 128);
            if (!*abort) {
                for (int c = tq; c < TOKN * (kRows / 8); c += 128) {
                    const int t = c / (kRows / 8), ch = c % (kRows / 8);
                    const int n = nbase + ch * 8;
                    if ((t / 4) % KS != kr) continue;
                    if (t < M && n < N)
                        *reinterpret_cast<uint4*>(Y + (size_t)t * N + n) =
                            *reinterpret_cast<const uint4*>(&ys[t * LDY + ch * 8]);
                }
            }
        }
    }

    if (warp < WARP_Q0) {
        // ---- the other roles: the end barrier, then tensor memory is freed and, after a
        // give-up, the copies already requested land before shared memory goes away
        tc_fence_before();
        const bool aborted = named_bar_red_or(BAR_END, kThreads, *abort != 0);
        if (warp == WARP_AUX) {
            tc_fence_after();
            tmem_dealloc(tmem, kTmemCols);
        }
        if (aborted && threadIdx.x == 0) {
            // (for each ring slot, the last group issued into it)
            wait_parity_suspend(xfull, 0u, &never_abort, kWaitNs, kSuspendNs);
            for (int j = max(0, w_issued - kRing); j < w_issued; ++j)
                wait_parity_suspend(rfull(j % kRing), uint32_t(j / kRing) & 1u, &never_abort, kWaitNs, kSuspendNs);
            for (int j = max(0, l_issued - kRing); j < l_issued; ++j)
                wait_parity_suspend(ldfull(j % kRing), uint32_t(j / kRing) & 1u, &never_abort, kWaitNs, kSuspendNs);
            if (lora_owner) wait_parity_suspend(lfull, 0u, &never_abort, kWaitNs, kSuspendNs);
            for (int i = 0; i < n_groups; ++i) wait_parity_suspend(sfull(i), 0u, &never_abort, kWaitNs, kSuspendNs);
        }
        if (KS > 1) {
            cluster_wait_acquire();   // (phase 2)
            cluster_arrive_release();  // phase 3
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

template <int TOKN, int R, bool DUMP>
w4a4_status launch_t(const uint16_t* X, const uint8_t* packed, const uint16_t* cs, const uint16_t* bias, int M, int N,
                     int K, int r, uint16_t* Y, uint8_t* ws, int32_t* P, cudaStream_t s) {
    const int KS = fused_split(N, K);
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(linear_fused_kernel<TOKN, R, DUMP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    cfg.dynamicSmemBytes = FOff<TOKN, R>::total(KS) + 1024;  // (the dynamic region is aligned up to 1024 bytes inside)
    cfg.stream = s;
    if (cudaLaunchKernelEx(&cfg, linear_fused_kernel<TOKN, R, DUMP>, X, packed, cs, bias, M, N, K, Y, ws, P, KS) !=
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
    const uint32_t total = M <= 16 ? (r == 0 ? FOff<16, 0>::total(KS) : r == 16 ? FOff<16, 16>::total(KS) : FOff<16, 32>::total(KS))
                                   : (r == 0 ? FOff<32, 0>::total(KS) : r == 16 ? FOff<32, 16>::total(KS) : FOff<32, 32>::total(KS));
    return total <= kSmemBudget;
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

template <int TOKN, bool DUMP>
w4a4_status launch_r(const uint16_t* X, const uint8_t* packed, const uint16_t* cs, const uint16_t* bias, int M, int N,
                     int K, int r, uint16_t* Y, uint8_t* ws, int32_t* P, cudaStream_t s) {
    if (r == 0) return launch_t<TOKN, 0, DUMP>(X, packed, cs, bias, M, N, K, r, Y, ws, P, s);
    if (r == 16) return launch_t<TOKN, 16, DUMP>(X, packed, cs, bias, M, N, K, r, Y, ws, P, s);
    return launch_t<TOKN, 32, DUMP>(X, packed, cs, bias, M, N, K, r, Y, ws, P, s);
}

w4a4_status launch_linear_fused(const uint16_t* X, const uint8_t* packed, const uint16_t* colscale,
                                const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, uint8_t* ws,
                                int32_t* P_dump, cudaStream_t s) {
    if (P_dump) {
        if (M <= 16) return launch_r<16, true>(X, packed, nullptr, nullptr, M, N, K, r, nullptr, ws, P_dump, s);
        return launch_r<32, true>(X, packed, nullptr, nullptr, M, N, K, r, nullptr, ws, P_dump, s);
    }
    if (M <= 16) return launch_r<16, false>(X, packed, colscale, bias, M, N, K, r, Y, ws, nullptr, s);
    return launch_r<32, false>(X, packed, colscale, bias, M, N, K, r, Y, ws, nullptr, s);
}

}  // namespace w4a4
