// Fused activation kernel: per-(row, 64-column group) absmax INT4 quantisation
// of fp16 X, codes written in the GEMM's tile layout, and the LoRA
// down-projection X . L_down from the same read of X ("W4A4 CUDA Kernel for
// Voice Clone", 3.6 fused_quantize_repack_act_kernel and its LoRA-down branch).
//
// GB300 design:
//  * A thread-block cluster of CK CTAs (8 warps each) owns 16 rows; each CTA
//    takes a contiguous range of the K groups, one or two per warp.  Every
//    warp pushes its fp32 LoRA partial tiles (16 rows x 8 columns each) with
//    st.async into the shared memory of the CTA that owns the tile (tile t
//    belongs to cluster rank t % CK), completing bytes on that CTA's
//    mbarrier; the owner adds the 8 x CK partials in a fixed (rank, warp)
//    order and stores fp16.  No atomics, deterministic results, one split
//    cluster barrier (overlapping the main loop) and no separate repack
//    kernel (the page's pack_lora_act exists only to wait for its atomics).
//    With many row blocks (prefill, several waves of CTAs) the cluster splits K
//    less finely: about eight groups per warp, so the cluster set-up, the
//    prologue and the LoRA reduction are paid once for all of them.
//  * Codes are stored as FP8 E4M3 bytes, the operand encoding the tcgen05
//    tensor core reads (GB300 has no INT4 tensor-core kind).
//  * Division x / scale is done as a multiplication by the reciprocal, which
//    gives the same code as the IEEE quotient except when the product lies
//    within 2^-18 of a rounding boundary (k + 1/2); those rare elements are
//    recomputed with the IEEE division, so codes equal rint(fl(x / scale)).
//    The check is branch-free per element; the warp takes the slow path only
//    when one of its lanes flagged such an element.
//  * Fused variant (NORM): the input is the previous linear's output, and the
//    RMSNorm between the two linears ("W4A4 CUDA Kernel for Voice Clone", 3.9)
//    is applied on the way in: every CTA first sums the squares of its 16 rows
//    over its own groups (the rows are L2-resident after the producing GEMM),
//    pushes the partial row sums to every rank of its cluster (st.async onto
//    the peers' mbarriers), and each CTA adds the CK partials in rank order, so
//    all agree on the inverse RMS; then each group's values are normalised to
//    fp16 -- the same bits as the glue kernel writes -- before they are
//    quantised and fed to the LoRA down-projection.
#include <cooperative_groups.h>

#include "kernels.h"
#include "norm.cuh"
#include "quant.cuh"
#include "tc_ptx.cuh"

namespace cg = cooperative_groups;

namespace w4a4 {
namespace {
using namespace tc;

constexpr int kRows = 16;      // rows per cluster (one m16 tile of the LoRA MMA)
constexpr int kWarps = 8;
constexpr int kXsStride = 72;  // halves per staged row (64 + 8 pad: conflict-free ldmatrix)
constexpr int kMaxCluster = 8;
constexpr int kPrefillRowBlocks = 128;  // M >= 2048: the prefill cluster split
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kTileBytes = kRows * 8 * 4;  // one fp32 16 x 8 LoRA partial tile
// staged fp16 tiles, then the LoRA receive area [rank][warp][CK-strided tile][16 x 8] fp32
// (CK * ceil(NT / CK) <= NT + kMaxCluster - 1 tiles per (rank, warp))
__host__ __device__ constexpr int q_smem_bytes(int R) {
    return kWarps * kRows * kXsStride * 2 + (R > 0 ? (R / 8 + kMaxCluster - 1) * kWarps * int(kTileBytes) : 0);
}

// Status word of the kernel's bounded wait (W4A4_ERR_TIMEOUT once it gave up).
__device__ int g_q_status = 0;

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

template <int R, bool NORM>  // LoRA rank, multiple of 16 (0 = no LoRA branch); RMSNorm on the way in
__global__ void __launch_bounds__(kWarps * 32, 2) quantize_act_kernel(const uint16_t* __restrict__ X, int ld_x,
                                                                   const uint2* __restrict__ Ldp, int M,
                                                                   int K, uint8_t* __restrict__ ws) {
    extern __shared__ __align__(16) uint8_t qsm[];
    __shared__ double ssq[kWarps][kRows], row_inv[kRows];
    __shared__ double row_recv[kMaxCluster][kRows];  // (NORM) every rank's partial row sums
    __shared__ __align__(8) uint64_t lora_bar_word, norm_bar_word;
    __shared__ int q_abort;
    uint16_t(*xs)[kRows * kXsStride] = reinterpret_cast<uint16_t(*)[kRows * kXsStride]>(qsm);
    float* recv = reinterpret_cast<float*>(qsm + kWarps * kRows * kXsStride * 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const ActLayout AL = act_layout(M, K, R);
    cg::cluster_group cluster = cg::this_cluster();
    const int CK = int(cluster.num_blocks());
    const int crank = int(cluster.block_rank());
    const int row0 = (blockIdx.x / CK) * kRows;
    const int mt = row0 / kTileM;
    const int g_begin = (G * crank) / CK, g_end = (G * (crank + 1)) / CK;
    constexpr int NT = R / 8;
    // LoRA tiles t with t % CK == crank are this CTA's to finish; receive layout stride
    const int own_tiles = crank < NT ? (NT - crank + CK - 1) / CK : 0;
    const int slot_tiles = (NT + CK - 1) / CK;
    const uint32_t lora_bar = smem_u32(&lora_bar_word), norm_bar = smem_u32(&norm_bar_word);
    if (threadIdx.x == 0) {
        q_abort = 0;
        if (R > 0) {
            mbar_init(lora_bar, 1);
            // this thread's arrival, and the bytes the other ranks' warps will push
            mbar_expect_tx(lora_bar, uint32_t((CK - 1) * kWarps * own_tiles) * kTileBytes);
        }
        if (NORM) {
            mbar_init(norm_bar, 1);
            mbar_expect_tx(norm_bar, uint32_t((CK - 1) * kRows) * 8u);  // the other ranks' row sums
        }
        fence_mbar_init();
    }
    // split cluster barrier: arriving says "my receive barriers are set up"; the wait
    // comes before this CTA's first push into a peer, so its latency overlaps the loads.
    // (The set-up touches only this CTA's shared memory, so it also overlaps the
    // previous kernel.)
    if (CK > 1 && (R > 0 || NORM)) cluster_arrive_release();
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0) {  // the GEMM's stream-K ready flags start every call cleared
        uint32_t* fl = reinterpret_cast<uint32_t*>(ws + AL.flags);
        for (int i = threadIdx.x; i < kStreamKSlots * kStreamKWarps; i += kWarps * 32) fl[i] = 0u;
    }

    // quantisation role: lane owns row (lane/2), columns 32*(lane%2) .. +31 of a group
    const int qrow = lane >> 1, qhalf = lane & 1;
    const int m = row0 + qrow;
    const int rr = m % kTileM;
    const bool valid = m < M;

    float acc[NT > 0 ? NT : 1][4];
#pragma unroll
    for (int t = 0; t < (NT > 0 ? NT : 1); ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

    uint16_t* xw = xs[warp];
    const uint16_t* xrow = X + (size_t)m * ld_x + qhalf * 32;
    double inv = 1.0;
    float inva = 1.f, invb = 0.f;
    if constexpr (NORM) {
        // sum of squares of row qrow over this CTA's groups (this lane's half of each
        // of the warp's groups, then the lane pair, then the 8 warps in order); the
        // cluster's CTAs then add their partial sums in rank order, so every CTA of
        // the cluster holds the same total
        float hi = 0.f, lo = 0.f;
        for (int g0 = g_begin + warp; g0 < g_end; g0 += kWarps) {
            uint4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[i] = valid ? ldg_nc_v4(xrow + (size_t)g0 * kGroup + 8 * i) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int i = 0; i < 4; ++i) add_squares(v[i], hi, lo);
        }
        double ss = double(hi) + double(lo);
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        if (qhalf == 0) ssq[warp][qrow] = ss;
        __syncthreads();
        if (CK > 1) cluster_wait_acquire();  // (every rank's receive barriers are set up)
        if (threadIdx.x < kRows) {
            double t = 0.0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) t += ssq[w][threadIdx.x];
            // this CTA's partial row sum into slot [crank] of every rank of the cluster
            row_recv[crank][threadIdx.x] = t;
            for (int c = 0; c < CK; ++c)
                if (c != crank)
                    st_async_b64(mapa_shared(smem_u32(&row_recv[crank][threadIdx.x]), uint32_t(c)),
                                 __double_as_longlong(t), mapa_shared(norm_bar, uint32_t(c)));
        }
        if (threadIdx.x < kRows) {
            if (CK > 1 && !wait_parity_suspend(norm_bar, 0u, &q_abort, kWaitNs, 20000u)) {
                q_abort = 1;
                atomicExch(&g_q_status, int(W4A4_ERR_TIMEOUT));
            }
            double t = 0.0;
            for (int c = 0; c < CK; ++c) t += row_recv[c][threadIdx.x];  // rank order, the same in every CTA
            row_inv[threadIdx.x] = __drcp_rn(__dsqrt_rn(t / double(K) + W4A4_RMSNORM_EPS));  // = 1.0 / sqrt(.)
        }
        __syncthreads();
        inv = row_inv[qrow];
        split_inv(inv, inva, invb);
    }
    int g = g_begin + warp;
    uint4 xv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        xv[i] = (valid && g < g_end) ? ldg_nc_v4(xrow + (size_t)g * kGroup + 8 * i) : make_uint4(0, 0, 0, 0);
    for (; g < g_end; g += kWarps) {
        // prefetch the warp's next group while this one is processed
        // this group's LoRA-down fragments, in flight while the group is quantised
        // (up to rank 48; larger ranks load them where they are used)
        constexpr bool kPrefetchB = R > 0 && R <= 48;
        constexpr int NTB = kPrefetchB ? NT : 1;
        uint2 b[4][NTB];
        if constexpr (kPrefetchB) {
            const uint2* bp = Ldp + ((size_t)(g * 4) * NT) * 32 + lane;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                for (int t = 0; t < NT; ++t) b[ks][t] = __ldg(bp + (ks * NT + t) * 32);
        }
        uint4 nv[4];
        const int gn = g + kWarps;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            nv[i] = (valid && gn < g_end) ? ldg_nc_v4(xrow + (size_t)gn * kGroup + 8 * i) : make_uint4(0, 0, 0, 0);
        if constexpr (NORM) {
#pragma unroll
            for (int i = 0; i < 4; ++i) xv[i] = scale_to_f16(xv[i], inv, inva, invb);
        }
        float s, csum;
        uint32_t packed[8];
        quantize_half_group(xv, s, csum, packed);
        uint8_t* plane = ws + AL.qA + ((size_t)(mt * G + g) * 2 + qhalf) * (kTileM * 32);
        *reinterpret_cast<uint4*>(plane + rr * 32 + swz32(rr, 0) * 16) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
        *reinterpret_cast<uint4*>(plane + rr * 32 + swz32(rr, 1) * 16) =
            make_uint4(packed[4], packed[5], packed[6], packed[7]);
        if (qhalf == 0)
            *reinterpret_cast<float2*>(ws + AL.sS + ((size_t)(mt * G + g) * kTileM + rr) * 8) = make_float2(s, csum);

        if constexpr (R > 0) {
            // LoRA down: the fp16 tile through ldmatrix into mma.m16n8k16 (fp32 accumulate)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4*>(xw + qrow * kXsStride + qhalf * 32 + 8 * i) = xv[i];
            __syncwarp();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint2 bl[NT];
                if constexpr (!kPrefetchB) {
                    const uint2* bp = Ldp + ((size_t)(g * 4) * NT) * 32 + lane;
#pragma unroll
                    for (int t = 0; t < NT; ++t) bl[t] = __ldg(bp + (ks * NT + t) * 32);
                }
                uint32_t a[4];
                const int lr = (lane & 7) + ((lane >> 3) & 1) * 8, lc = ((lane >> 4) & 1) * 8 + ks * 16;
                ldmatrix_x4(a, xw + lr * kXsStride + lc);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const uint2 bb = kPrefetchB ? b[ks][t % NTB] : bl[t];
                    mma_f16_16816(acc[t], a, bb.x, bb.y);
                }
            }
            __syncwarp();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) xv[i] = nv[i];
    }

    if constexpr (R > 0) {
        // push this warp's partial tiles to their owners: lane (gid, tig) holds rows gid and
        // gid + 8, columns 2 tig and 2 tig + 1 of every 16 x 8 tile
        const int gid = lane >> 2, tig = lane & 3;
        if (CK > 1 && !NORM) cluster_wait_acquire();  // (with the norm, waited for before the row sums)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int o = t % CK, lt = t / CK;
            const uint32_t off =
                ((uint32_t(crank * kWarps + warp) * slot_tiles + lt) * (kRows * 8) + gid * 8 + 2 * tig) * 4;
            if (o == crank) {
                *reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(recv) + off) = make_float2(acc[t][0], acc[t][1]);
                *reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(recv) + off + 8 * 8 * 4) =
                    make_float2(acc[t][2], acc[t][3]);
            } else {
                const uint32_t dst = mapa_shared(smem_u32(recv) + off, uint32_t(o));
                const uint32_t rbar = mapa_shared(lora_bar, uint32_t(o));
                st_async_v2(dst, acc[t][0], acc[t][1], rbar);
                st_async_v2(dst + 8 * 8 * 4, acc[t][2], acc[t][3], rbar);
            }
        }
        __syncthreads();  // this CTA's own partials are in place
        if (own_tiles > 0) {
            if (!wait_parity_suspend(lora_bar, 0u, &q_abort, kWaitNs, 20000u)) {
                q_abort = 1;
                atomicExch(&g_q_status, int(W4A4_ERR_TIMEOUT));
            }
            if (!q_abort) {
                // finish the owned tiles: the 8 x CK partials in (rank, warp) order, fp16 out
                uint16_t* La = reinterpret_cast<uint16_t*>(ws + AL.La);
                for (int e = threadIdx.x; e < own_tiles * kRows * 8; e += kWarps * 32) {
                    const int lt = e / (kRows * 8), rc = e % (kRows * 8), row = rc / 8, col = rc % 8;
                    float v = 0.f;
                    for (int c = 0; c < CK; ++c)
#pragma unroll
                        for (int w = 0; w < kWarps; ++w)
                            v += recv[((c * kWarps + w) * slot_tiles + lt) * (kRows * 8) + rc];
                    const int j = 8 * (lt * CK + crank) + col;
                    const int r2 = (row0 + row) % kTileM;
                    const int p = j >> 4, jj = j & 15;
                    La[((size_t)(mt * (R / 16) + p) * kTileM + r2) * 16 + swz32(r2, jj >> 3) * 8 + (jj & 7)] =
                        __half_as_ushort(__float2half_rn(v));
                }
            }
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

template <int R, bool NORM>
w4a4_status launch_q(const uint16_t* X, int ld_x, const uint8_t* packed, int M, int K, uint8_t* ws,
                     cudaStream_t s) {
    const int G = K / kGroup;
    // split K over a (small) cluster: one group per warp up to clusters of six (at
    // M = 700, K = 2048 and 3072: 4.4 and 4.8 us against 4.9 and 4.9 with two groups
    // per warp), about two groups per warp beyond
    // (with few row blocks -- decode -- the SMs are idle anyway: one group per warp
    // up to the largest cluster)
    // (with many row blocks -- prefill -- one CTA per row block, its warps taking
    // every eighth group: two such CTAs share an SM, and at M = 8192 this is the
    // fastest split for K = 4096 and K = 14336: 36 and 105 us, against 42 / 110
    // with clusters of two)
    const int row_blocks = (M + kRows - 1) / kRows;
    int CK = (G + kWarps - 1) / kWarps;
    if (CK > 6 && row_blocks > 8) CK = (G + 2 * kWarps - 1) / (2 * kWarps);
    if (row_blocks >= kPrefillRowBlocks) CK = 1;
    if (CK > kMaxCluster) CK = kMaxCluster;
    if (CK < 1) CK = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(row_blocks * CK));
    cfg.blockDim = dim3(kWarps * 32);
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    constexpr int smem = q_smem_bytes(R);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(quantize_act_kernel<R, NORM>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return W4A4_ERR_CUDA;
        attr_done[dev] = 1;
    }
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(CK);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = add_pdl_attr(attr, 1);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_act_kernel<R, NORM>, X, ld_x,
                                             reinterpret_cast<const uint2*>(packed), M, K, ws);
    set_dispatch("quantize_act%s rows/cluster=%d cluster=%d grid=%d rank=%d", NORM ? " (RMSNorm fused)" : "", kRows, CK,
                 row_blocks * CK, R);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    return launch_status();
}

template <bool NORM>
w4a4_status launch_qr(const uint16_t* X, int ld_x, const uint8_t* packed, int M, int K, int r, uint8_t* ws,
                      cudaStream_t s) {
    switch (r) {
        case 0: return launch_q<0, NORM>(X, ld_x, packed, M, K, ws, s);
        case 16: return launch_q<16, NORM>(X, ld_x, packed, M, K, ws, s);
        case 32: return launch_q<32, NORM>(X, ld_x, packed, M, K, ws, s);
        case 48: return launch_q<48, NORM>(X, ld_x, packed, M, K, ws, s);
        case 64: return launch_q<64, NORM>(X, ld_x, packed, M, K, ws, s);
        case 80: return launch_q<80, NORM>(X, ld_x, packed, M, K, ws, s);
        case 96: return launch_q<96, NORM>(X, ld_x, packed, M, K, ws, s);
        case 112: return launch_q<112, NORM>(X, ld_x, packed, M, K, ws, s);
        case 128: return launch_q<128, NORM>(X, ld_x, packed, M, K, ws, s);
        default: return W4A4_ERR_UNSUPPORTED_SHAPE;
    }
}

}  // namespace

w4a4_status q_read_and_clear_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_q_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_q_status, &zero, sizeof(int));
        return W4A4_ERR_TIMEOUT;
    }
    return W4A4_OK;
}

w4a4_status launch_quantize_act(const uint16_t* X, const uint8_t* packed, int M, int K, int r, uint8_t* ws,
                                cudaStream_t s) {
    return launch_qr<false>(X, K, packed, M, K, r, ws, s);
}

w4a4_status launch_quantize_act_rmsnorm(const uint16_t* Y, int ld_y, const uint8_t* packed, int M, int K, int r,
                                        uint8_t* ws, cudaStream_t s) {
    return launch_qr<true>(Y, ld_y, packed, M, K, r, ws, s);
}

void launch_unpack_act(const uint8_t* ws, int M, int K, int r, int8_t* codes, float* sA, float* SA, float* lora,
                       cudaStream_t s) {
    long long n = (long long)M * K;
    if ((long long)M * r > n) n = (long long)M * r;
    unpack_act_kernel<<<unsigned((n + 255) / 256), 256, 0, s>>>(ws, M, K, r, codes, sA, SA, r ? lora : nullptr);
}

}  // namespace w4a4
