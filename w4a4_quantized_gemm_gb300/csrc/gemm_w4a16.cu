// W4A16 linear for the decode regime: fp16 activations against the same packed
// INT4 weights, LoRA and column affine as the W4A4 layer ("INT4 Kernel
// Architecture, in depth", "W4A16 versus W4A4": the activations stay fp16,
// only the weights are 4-bit and are dequantised in registers; "One token
// versus a thousand": at small M the layer streams its weights).
//
//   Y[m,n] = colscale[n] * ( sum_g sW[n,g] sum_{k in g} X[m,k] c[n,k]
//                            + (X L_down)[m,:] . L_up[:,n] ) + bias[n]
//
// One kernel, no workspace.  The work layout is the small-M W4A4 kernel's: a
// CTA of 8 warps covers 128 weight rows (16 per warp, the weights as the MMA's
// 16-row operand) and up to 64 tokens; K is split over a cluster of KS CTAs;
// each CTA requests its whole share up front (one bulk copy per 4 KB group of
// weight records, cp.async for the scales and the tokens' fp16 values), one
// mbarrier per group slot; partial sums are pushed to the owner rank of each
// warp's columns with st.async and added there in rank order.
//
// Per group the offset-binary nibbles become exact fp16 codes c = u - 8 with a
// mask-and-bias step (nibble | 0x6400 is 1024 + u; minus 1032): nibbles j and
// j + 4 of a 32-bit record word, which hold codes k and k + 16 of the group,
// land in one half2, so each m16n8k16 fp16 MMA takes its k pairs as (k, k+16);
// the tokens' B fragments are paired the same way from shared memory.  The
// group's fp32 sum is scaled by sW (fp16) and added to the fp32 accumulator.
//
// Asymmetric group-128 weights ("How the weights are stored": codes 0..15,
// value (q - zero) scale per 128-group): the same kernel with the nibble's
// bias removed per row, (1024 + q) - (1024 + zero), exact in fp16 for zero
// points in [-1024, 1023]; each 64-channel slot reads its group's scale and
// zero from the two scale-plane slots of the group.
//
// LoRA: each CTA forms its K slice's part of X . L_down (fp16 MMA, fp32
// accumulate) and applies the up-projection to that part before the exchange;
// the map is linear, so the exchange of partial sums also sums the LoRA term.
// The part is split as hi + lo fp16 values (two up MMAs), so nothing is lost
// to an fp16 rounding of a partial sum.
//
// Waits are bounded (2 s; W4A4_ERR_TIMEOUT in the status word), warps suspend
// in the barrier unit rather than poll, and both cluster barriers are split
// (arrive early, wait late).
#include "kernels.h"
#include "tc_ptx.cuh"

namespace w4a4 {
namespace {
using namespace tc;

constexpr int kWarps = 8;
constexpr int kTileN = kWarps * 16;  // weight rows per CTA
constexpr int kMaxKS = 8;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kSuspendNs = 20000;

// Status word of this kernel's bounded waits (W4A4_ERR_TIMEOUT once one gave up).
__device__ int g_w4a16_status = 0;

constexpr int kXs = 64 + 8;  // halves per staged token row of a group (pad: fewer bank conflicts)

// Byte offsets of the shared-memory sections (all multiples of 16).
struct W4A16Plan {
    int ns;  // group slots: two halves of ns / 2, refilled alternately
    uint32_t wq, xs, sw, lu, la, red, bar, total;
};
__host__ __device__ inline W4A16Plan w4a16_plan(int tok, int r, bool asym) {
    W4A16Plan p;
    p.ns = tok <= 8 ? 16 : tok <= 32 ? 8 : 4;  // two CTAs per SM fit for every token count
    uint32_t o = 0;
    p.wq = o, o += uint32_t(p.ns) * kTileN * 32;                 // [slot][128 rows][32 B]
    p.xs = o, o += uint32_t(p.ns) * tok * kXs * 2;               // [slot][tok][72 halves]
    p.sw = o, o += uint32_t(p.ns) * kTileN * (asym ? 4 : 2);     // [slot][128] fp16 (asym: scale, zero)
    p.lu = o, o += uint32_t(r / 16) * kTileN * 32;               // [plane][128 rows][32 B]
    p.la = o, o += 2u * uint32_t(r / 16) * tok * 32;             // [hi|lo][plane][tok][32 B]
    p.red = o, o += uint32_t(kMaxKS - 1) * 32 * (tok / 8) * 16;  // [sender slot][lane][tok / 8] float4
    p.bar = o, o += 160;                                         // full[ns], aux, red_full
    p.total = o;
    return p;
}
// The fp16 output tile [tok][128 + 8] is staged over the weight and token slots
// (contiguous) once every group has been consumed: tok * 136 * 2 bytes <=
// ns * (4 KB + tok * 144 bytes) for every slot count above.

// Nibbles j and j + 4 of w -> exact fp16 values u - (bias - 1024) in the low
// and high half: bias2 = 1032 (offset-binary codes u - 8) or 1024 + zero.
__device__ __forceinline__ uint32_t nib_pair_f16(uint32_t w, int j, __half2 bias2) {
    uint32_t h;
    const uint32_t x = w >> (4 * j);
    asm("lop3.b32 %0, %1, %2, %3, 0xea;\n" : "=r"(h) : "r"(x), "r"(0x000F000Fu), "r"(0x64006400u));  // (x & m) | c
    const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h), bias2);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int NT8, bool ASYM>
__global__ void __launch_bounds__(kWarps * 32) gemm_w4a16_kernel(
    const uint16_t* __restrict__ X, const uint8_t* __restrict__ packed, const uint16_t* __restrict__ colscale,
    const uint16_t* __restrict__ bias, int M, int N, int K, int r, uint16_t* __restrict__ Y, int KS) {
    constexpr int TOK = NT8 * 8;
    constexpr int NT = kWarps * 32;
    extern __shared__ __align__(128) uint8_t smraw[];
    __shared__ int abort_flag, never_abort;
    const W4A16Plan PLN = w4a16_plan(TOK, r, ASYM);
    constexpr uint32_t kSwSlot = kTileN * (ASYM ? 4 : 2);  // scale-plane bytes per slot
    const uint32_t sbase = smem_u32(smraw);
    const uint32_t full0 = sbase + PLN.bar;  // full[s] = full0 + 8 s
    const uint32_t aux_full = full0 + 8u * PLN.ns, red_full = aux_full + 8u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, q = lane & 3;
    const int G = K / kGroup;
    const PackedLayout PL = packed_layout(N, K, r);
    const int kr = KS > 1 ? int(cluster_ctarank()) : 0;
    const int ntile = blockIdx.x / KS;
    const int g_begin = (G * kr) / KS, n_groups = (G * (kr + 1)) / KS - g_begin;
    const int half = PLN.ns / 2;
    const int n_chunks = (n_groups + half - 1) / half;

    const int tok0 = blockIdx.y * TOK;  // first token of this CTA
    const int tok_valid = min(TOK, M - tok0);
    const int nbase = ntile * kTileN;
    const int rows_valid = min(kTileN, N - nbase);  // a multiple of 16
    const int n0 = nbase + warp * 16;
    const bool warp_active = n0 < N;
    const bool owner = KS == 1 || warp % KS == kr;
    volatile int* abort = &abort_flag;

    const uint8_t* qW = packed + PL.qW;
    const uint8_t* sWg = packed + PL.sW;
    // 16-byte pieces of one group besides the weight records: weight scales (asym: the
    // group's scale and zero rows), the tokens' values
    const int pc_sw1 = rows_valid / 8, pc_sw = ASYM ? 2 * pc_sw1 : pc_sw1, pc_x = tok_valid * 8;

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
            for (int p = threadIdx.x; p < pc_sw + pc_x; p += NT) {
                if (p < pc_sw) {
                    const int hz = ASYM ? (p >= pc_sw1) : 0, pp = p - hz * pc_sw1;
                    const int gs = ASYM ? ((g & ~1) | hz) : g;  // asym: the 128-group's scale / zero slot
                    cp_async16(smraw + PLN.sw + slot * kSwSlot + hz * (kTileN * 2) + pp * 16,
                               sWg + ((size_t)gs * N + nbase) * 2 + pp * 16);
                } else {
                    const int e = p - pc_sw, t = e >> 3, c8 = e & 7;
                    cp_async16(smraw + PLN.xs + (slot * TOK + t) * (kXs * 2) + c8 * 16,
                               X + (size_t)(tok0 + t) * K + (size_t)g * kGroup + c8 * 8);
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
        if (KS > 1)  // bytes this rank receives: its owned warps' fragments from every other rank
            mbar_expect_tx(red_full, uint32_t((KS - 1) * (kWarps / KS) * 32 * NT8 * 16));
    }
    // token rows past M are zero in every slot (they are never loaded)
    for (int i = threadIdx.x; i < PLN.ns * TOK * (kXs / 8); i += NT) {
        const int t = (i / (kXs / 8)) % TOK;
        if (t >= tok_valid) *reinterpret_cast<uint4*>(smraw + PLN.xs + i * 16) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();  // barriers initialised for this CTA's threads
    if (KS > 1) cluster_arrive_release();  // ... and, once every rank has arrived, for the peers
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
    // L_up rows of all 128 weight rows (every warp applies the up-projection to its CTA's LoRA part)
    for (int p = threadIdx.x; p < (r / 16) * (rows_valid * 2); p += NT) {
        const int pl = p / (rows_valid * 2), e = p % (rows_valid * 2);
        cp_async16(smraw + PLN.lu + pl * (kTileN * 32) + e * 16, packed + PL.Lu + ((size_t)pl * N + nbase) * 32 + e * 16);
    }
    cp_async_mbar_arrive_noinc(aux_full);
    int issued = 0, requested = 0;
    for (; issued < 2 && issued < n_chunks; ++issued) issue_chunk(issued);
    requested = issued;

    float csa = 0.f, csb = 0.f, ba = 0.f, bb = 0.f;
    if (owner && warp_active) {
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

    // LoRA down over this CTA's K slice: warp w owns the r/8-column tiles w, w + 8, ...
    const uint2* Ldp = reinterpret_cast<const uint2*>(packed + PL.Ld);
    constexpr int MT16 = (TOK + 15) / 16;
    const int rt = r / 8;
    float ld_acc[MT16][2][4];  // [token tile][owned column tile][fragment]
#pragma unroll
    for (int mt = 0; mt < MT16; ++mt)
#pragma unroll
        for (int u = 0; u < 2; ++u) ld_acc[mt][u][0] = ld_acc[mt][u][1] = ld_acc[mt][u][2] = ld_acc[mt][u][3] = 0.f;

    // this lane's weight bytes (rows warp*16 + gid and + 8, bytes 8q..8q+7) and scales in a slot
    const uint8_t* smw = smraw + PLN.wq + (warp * 16 + gid) * 32 + 8 * q;
    const uint16_t* smsw = reinterpret_cast<const uint16_t*>(smraw + PLN.sw) + warp * 16 + gid;
    for (int c = 0; c < n_chunks; ++c) {
        const int b = c & 1, ng = min(half, n_groups - c * half);
        for (int j = 0; j < ng; ++j) {
            const int slot = b * half + j;
            const bool ok = warp_wait_parity_suspend(full0 + 8u * slot, uint32_t(c >> 1) & 1u, abort, kWaitNs,
                                                     kSuspendNs);
            if (!ok) {
                if (lane == 0) {
                    *abort = 1;
                    atomicExch(&g_w4a16_status, int(W4A4_ERR_TIMEOUT));
                }
                break;
            }
            const uint16_t* xsl = reinterpret_cast<const uint16_t*>(smraw + PLN.xs) + slot * TOK * kXs;
            // this group's L_down fragments for the warp's column tiles, in flight during the main MMAs
            const int g = g_begin + c * half + j;
            uint2 ldf[2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    ldf[u][ks] = (r > 0 && warp + 8 * u < rt) ? __ldg(Ldp + ((size_t)(g * 4 + ks) * rt + warp + 8 * u) * 32 + lane)
                                                             : make_uint2(0u, 0u);
            if (warp_active) {
            const uint2 wa = *reinterpret_cast<const uint2*>(smw + slot * (kTileN * 32));
            const uint2 wb = *reinterpret_cast<const uint2*>(smw + slot * (kTileN * 32) + 8 * 32);
            const uint16_t* sws = smsw + slot * (kSwSlot / 2);
            const float swa = __half2float(__ushort_as_half(sws[0]));
            const float swb = __half2float(__ushort_as_half(sws[8]));
            const uint64_t swa2 = f2_pack(swa, swa), swb2 = f2_pack(swb, swb);
            __half2 bias_a = __float2half2_rn(1032.f), bias_b = bias_a;
            if constexpr (ASYM) {  // 1024 + zero of rows a and b (exact for |zero| <= 1024)
                const __half za = __ushort_as_half(sws[kTileN]), zb = __ushort_as_half(sws[kTileN + 8]);
                bias_a = __hadd2(__halves2half2(za, za), __float2half2_rn(1024.f));
                bias_b = __hadd2(__halves2half2(zb, zb), __float2half2_rn(1024.f));
            }
            // word h of this lane's record bytes holds codes k = 32h + 4q + i and 32h + 16 + 4q + i
            // (i = 0..3, nibbles i and i + 4); MMA (h, jp) takes i = jp, jp + 1
            uint32_t af[4][4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t xa = h ? wa.y : wa.x, xb = h ? wb.y : wb.x;
#pragma unroll
                for (int jp = 0; jp < 2; ++jp) {
                    af[2 * h + jp][0] = nib_pair_f16(xa, 2 * jp, bias_a);
                    af[2 * h + jp][2] = nib_pair_f16(xa, 2 * jp + 1, bias_a);
                    af[2 * h + jp][1] = nib_pair_f16(xb, 2 * jp, bias_b);
                    af[2 * h + jp][3] = nib_pair_f16(xb, 2 * jp + 1, bias_b);
                }
            }
#pragma unroll
            for (int t = 0; t < NT8; ++t) {
                const uint16_t* xr = xsl + (t * 8 + gid) * kXs + 4 * q;
                float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int h = i >> 1, jp = (i & 1) * 2;
                    // tokens' values at k0 = 32h + 4q + jp (and + 1) and k0 + 16 (and + 1)
                    const uint32_t lo = *reinterpret_cast<const uint32_t*>(xr + 32 * h + jp);
                    const uint32_t hi = *reinterpret_cast<const uint32_t*>(xr + 32 * h + 16 + jp);
                    const uint32_t b0 = __byte_perm(lo, hi, 0x5410), b1 = __byte_perm(lo, hi, 0x7632);
                    mma_f16_16816(d, af[i], b0, b1);
                }
                acc_a[t] = ffma2_b64(swa2, f2_pack(d[0], d[1]), acc_a[t]);
                acc_b[t] = ffma2_b64(swb2, f2_pack(d[2], d[3]), acc_b[t]);
            }
            }  // warp_active
            if (r > 0) {
                // X . L_down for this group's four 16-wide k blocks and this warp's column tiles
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (warp + 8 * u >= rt) continue;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                        for (int mt = 0; mt < MT16; ++mt) {
                            const uint16_t* r0 = xsl + (mt * 16 + gid) * kXs + ks * 16 + 2 * q;
                            uint32_t a[4];
                            a[0] = *reinterpret_cast<const uint32_t*>(r0);
                            a[2] = *reinterpret_cast<const uint32_t*>(r0 + 8);
                            if (mt * 16 + 8 < TOK) {
                                a[1] = *reinterpret_cast<const uint32_t*>(r0 + 8 * kXs);
                                a[3] = *reinterpret_cast<const uint32_t*>(r0 + 8 * kXs + 8);
                            } else {
                                a[1] = a[3] = 0u;
                            }
                            mma_f16_16816(ld_acc[mt][u], a, ldf[u][ks].x, ldf[u][ks].y);
                        }
                    }
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
    const bool aborted = __syncthreads_or(*abort);
    if (aborted) {
        // let the copies already requested land before this CTA's shared memory goes away
        if (threadIdx.x == 0) {
            for (int c = max(0, requested - 2); c < requested; ++c) {
                const int ng = min(half, n_groups - c * half);
                for (int j = 0; j < ng; ++j)
                    wait_parity_suspend(full0 + 8u * ((c & 1) * half + j), uint32_t(c >> 1) & 1u, &never_abort,
                                        kWaitNs, kSuspendNs);
            }
        }
    }

    // this CTA's LoRA part -> shared memory as hi + lo fp16 planes [plane][tok][32 B] (32-byte swizzle)
    uint8_t* la_hi = smraw + PLN.la;
    uint8_t* la_lo = la_hi + (r / 16) * TOK * 32;
    if (r > 0 && !aborted) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int ct = warp + 8 * u;
            if (ct >= rt) continue;
#pragma unroll
            for (int mt = 0; mt < MT16; ++mt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tk = mt * 16 + gid + (e >> 1) * 8, col = ct * 8 + 2 * q + (e & 1);
                    if (tk >= TOK) continue;
                    const float v = ld_acc[mt][u][e];
                    const __half hv = __float2half_rn(v);
                    const __half lv = __float2half_rn(v - __half2float(hv));
                    const int p = col >> 4, jj = col & 15;
                    const int off = p * (TOK * 32) + tk * 32 + swz32(tk, jj >> 3) * 16 + (jj & 7) * 2;
                    *reinterpret_cast<__half*>(la_hi + off) = hv;
                    *reinterpret_cast<__half*>(la_lo + off) = lv;
                }
            }
        }
    }
    __syncthreads();
    if (r > 0 && warp_active && !aborted) {
        const bool ok = warp_wait_parity_suspend(aux_full, 0u, abort, kWaitNs, kSuspendNs);
        if (!ok && lane == 0) {
            *abort = 1;
            atomicExch(&g_w4a16_status, int(W4A4_ERR_TIMEOUT));
        }
        // LoRA up of this CTA's part: acc[n, m] += sum_j L_up[j, n] part[m, j]
        const int na_ = n0 + gid, nb_ = n0 + gid + 8;
        const uint8_t* lu_a = smraw + PLN.lu + (warp * 16 + gid) * 32 + 4 * q;
        const uint8_t* lu_b = lu_a + 8 * 32;
        for (int p = 0; ok && p < r / 16; ++p) {
            uint32_t a[4];
            a[0] = *reinterpret_cast<const uint32_t*>(lu_a + p * (kTileN * 32) + swz32(na_, 0) * 16);
            a[2] = *reinterpret_cast<const uint32_t*>(lu_a + p * (kTileN * 32) + swz32(na_, 1) * 16);
            a[1] = *reinterpret_cast<const uint32_t*>(lu_b + p * (kTileN * 32) + swz32(nb_, 0) * 16);
            a[3] = *reinterpret_cast<const uint32_t*>(lu_b + p * (kTileN * 32) + swz32(nb_, 1) * 16);
#pragma unroll
            for (int t = 0; t < NT8; ++t) {
                const int rr = t * 8 + gid;
                float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int hl = 0; hl < 2; ++hl) {
                    const uint8_t* la = (hl ? la_lo : la_hi) + p * (TOK * 32);
                    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(la + rr * 32 + swz32(rr, 0) * 16 + 4 * q);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(la + rr * 32 + swz32(rr, 1) * 16 + 4 * q);
                    mma_f16_16816(d, a, b0, b1);
                }
                acc_a[t] = fadd2_b64(acc_a[t], f2_pack(d[0], d[1]));
                acc_b[t] = fadd2_b64(acc_b[t], f2_pack(d[2], d[3]));
            }
        }
    }

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
                    atomicExch(&g_w4a16_status, int(W4A4_ERR_TIMEOUT));
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

    // fp16 output tile staged over the weight and token slots, which no warp or copy uses any more
    uint16_t* ys = reinterpret_cast<uint16_t*>(smraw + PLN.wq);
    constexpr int LDY = kTileN + 8;
    if (owner && warp_active && !*abort) {
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
    if (!*abort) {
        for (int c = threadIdx.x; c < TOK * (kTileN / 8); c += NT) {
            const int t = c / (kTileN / 8), ch = c % (kTileN / 8);
            const int m = tok0 + t, n = nbase + ch * 8;
            if ((ch >> 1) % KS != kr) continue;  // chunk ch belongs to warp ch / 2
            if (m < M && n < N)
                *reinterpret_cast<uint4*>(Y + (size_t)m * N + n) = *reinterpret_cast<const uint4*>(&ys[t * LDY + ch * 8]);
        }
    }
    if (threadIdx.x == 0 && !wait_parity_suspend(aux_full, 0u, &never_abort, kWaitNs, kSuspendNs))
        atomicExch(&g_w4a16_status, int(W4A4_ERR_TIMEOUT));  // (the L_up copies land before the CTA leaves)
    if (KS > 1) cluster_wait_acquire();  // no rank leaves while a peer may still address its shared memory
}

// Split factor: up to two CTAs per SM and at least one group per CTA.
int w4a16_split(int M, int N, int K, int TOK) {
    const int tiles = ((N + kTileN - 1) / kTileN) * ((M + TOK - 1) / TOK);
    const int G = K / kGroup;
    int ks = 1;
    while (ks < kMaxKS && tiles * ks * 2 <= 2 * device_sm_count() && ks * 2 <= G) ks *= 2;
    return ks;
}

template <int NT8, bool ASYM>
w4a4_status launch_nt(const uint16_t* X, const uint8_t* packed, const uint16_t* cs, const uint16_t* bias, int M,
                      int N, int K, int r, uint16_t* Y, cudaStream_t s) {
    const int smem_max = int(w4a16_plan(NT8 * 8, W4A4_MAX_RANK, ASYM).total);  // the attribute covers every rank
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(gemm_w4a16_kernel<NT8, ASYM>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) !=
            cudaSuccess)
            return W4A4_ERR_CUDA;
        attr_done[dev] = 1;
    }
    const int KS = w4a16_split(M, N, K, NT8 * 8);
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
    cfg.dynamicSmemBytes = w4a16_plan(NT8 * 8, r, ASYM).total;
    cfg.stream = s;
    if (cudaLaunchKernelEx(&cfg, gemm_w4a16_kernel<NT8, ASYM>, X, packed, cs, bias, M, N, K, r, Y, KS) != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    set_dispatch("gemm_w4a16%s mma.sync.f16 tokens/CTA=%d split-K=%d (cluster) grid=%ux%u",
                 ASYM ? " (asymmetric g128)" : "", NT8 * 8, KS, grid.x, grid.y);
    return launch_status();
}

}  // namespace

w4a4_status w4a16_read_and_clear_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_w4a16_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_w4a16_status, &zero, sizeof(int));
        return W4A4_ERR_TIMEOUT;
    }
    return W4A4_OK;
}

template <bool ASYM>
w4a4_status launch_w4a16(const uint16_t* X, const uint8_t* packed, const uint16_t* colscale, const uint16_t* bias,
                         int M, int N, int K, int r, uint16_t* Y, cudaStream_t s) {
    if (M <= 8) return launch_nt<1, ASYM>(X, packed, colscale, bias, M, N, K, r, Y, s);
    if (M <= 16) return launch_nt<2, ASYM>(X, packed, colscale, bias, M, N, K, r, Y, s);
    if (M <= 32) return launch_nt<4, ASYM>(X, packed, colscale, bias, M, N, K, r, Y, s);
    return launch_nt<8, ASYM>(X, packed, colscale, bias, M, N, K, r, Y, s);
}

w4a4_status launch_gemm_w4a16(const uint16_t* X, const uint8_t* packed, const uint16_t* colscale,
                              const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, bool asym,
                              cudaStream_t s) {
    return asym ? launch_w4a16<true>(X, packed, colscale, bias, M, N, K, r, Y, s)
                : launch_w4a16<false>(X, packed, colscale, bias, M, N, K, r, Y, s);
}

}  // namespace w4a4
