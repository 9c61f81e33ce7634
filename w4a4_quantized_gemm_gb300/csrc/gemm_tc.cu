// W4A4 GEMM + LoRA up + column affine on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), for M above the small-M range.
//
// Computes, per 128 x 128 output tile ("W4A4 CUDA Kernel for Voice Clone",
// 3.7; "High-Performance Kernel Design for W4A4 ... on Blackwell", 1):
//   acc = lora_act . L_up  +  sum_g sW[n,g] (2^9 sA[m,g] D_g - 8 SA[m,g] sA[m,g])
//   D_g = 2^-9 sum_{k in g} cA * (cW + 8)     (exact, one group per TMEM buffer: the
//         weight bytes are the offset codes, which E4M3 reads as u * 2^-9)
//   Y   = fp16(colscale * acc + bias)
//
// Structure (the warp-specialised persistent design of the Blackwell W4A4
// article, section 3.2, rebuilt for tcgen05): one CTA per SM walks tiles in a
// static round-robin; warps have fixed roles and talk through mbarriers.
// Work moves in jobs of two K groups, so that every role synchronises once per
// two groups.  Tensor memory holds two job buffers (2 x 2 x 128 columns):
//   warps 20,22,23  producers: per job the 1-D bulk copies of activation
//               codes, weight nibbles, and (sA, SA) + weight scales into an
//               S-deep stage ring, one warp each so that the issues overlap;
//               per tile the LoRA operands;
//   warp 21     MMA issuer (one thread) + tensor-memory owner: per tile a
//               kind::f16 LoRA-up chain, per group two kind::f8f6f4 MMAs
//               (M = N = 128, K = 32) into its 128 columns of a job buffer;
//   warps 16-19 nibble -> byte expansion of the weight tiles into the
//               32-byte-swizzled B operand (32 rows each, one warp per SM
//               sub-partition) and the groups' scales as fp32 into a scale
//               ring that outlives the stage;
//   warps 0-15  epilogue, four warps per TMEM lane quarter and 32 columns
//               each: per job the two product slices come out of tensor
//               memory in 16-column chunks and two FMAs per element (packed
//               fp32 pairs) fold each group into the running sums held in
//               registers; at the end of a tile the column affine and the
//               fp16 store.
// The per-group fp32 scaling (two FMAs per output) is the floor of this
// kernel; its instruction count, not the tensor pipe, sets the pace, so the
// epilogue is spread over 16 warps and every fixed per-group cost is paid
// once per job.
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
constexpr int GPJ = 2;   // K groups per job: every role synchronises once per job
constexpr int NUM_THREADS = 768;
constexpr int NUM_EPI_WARPS = 16, WARP_EXP0 = 16, NUM_EXP_WARPS = 4;
constexpr int WARP_PRODUCER = 20, WARP_MMA = 21, WARP_PRODUCER_W = 22, WARP_PRODUCER_S = 23;
constexpr int NUM_PRODUCERS = 3;
constexpr int EPI_COLS = BN / 4;  // columns per epilogue warp
constexpr int EXP_ROWS = BN / NUM_EXP_WARPS;
constexpr int EPI_REGS = 96, OTHER_REGS = 48;
static_assert(NUM_EPI_WARPS * 32 * EPI_REGS + (NUM_THREADS - NUM_EPI_WARPS * 32) * OTHER_REGS <= 65536,
              "register split exceeds the register file");
constexpr int NPB = 2;  // job buffers in tensor memory, GPJ x 128 columns each
constexpr uint32_t TMEM_COLS = 512;
static_assert(NPB * GPJ * BN <= int(TMEM_COLS), "job buffers must fit in tensor memory");
constexpr int SS = 4;  // scale-ring depth (jobs)
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;
// Waiting warps are suspended in the barrier unit until the phase completes (woken at once,
// no issue slots spent), re-checking the abort flag and the clock every SUSPEND_NS at most
constexpr uint32_t SUSPEND_NS = 20000;

// Stage (one job = GPJ groups): activation codes (per group 2 planes x 128 rows
// x 32 B), weight nibbles (per group 128 rows x 32 B), the expanded B operand
// (per group 2 planes x 128 rows x 32 B), (sA, SA) per row and group, fp16
// weight scales.  Operand planes are 256-byte aligned.
constexpr uint32_t kA = 2 * BM * 32, kW = BN * 32, kB = 2 * BN * 32, kS = BM * 8, kSw = BN * 2;
constexpr uint32_t ST_A = 0, ST_W = ST_A + GPJ * kA, ST_B = ST_W + GPJ * kW, ST_S = ST_B + GPJ * kB,
                   ST_SW = ST_S + GPJ * kS;
constexpr uint32_t kStage = ST_SW + GPJ * kSw;
// Scale-ring entry, per group of the job: fp32 sW of the tile's 128 columns,
// then (sA, SA) of its 128 rows.
constexpr uint32_t kScaleG = BN * 4 + BM * 8;
constexpr uint32_t kScale = GPJ * kScaleG;
static_assert(kStage % 256 == 0 && ST_B % 256 == 0 && ST_W % 256 == 0 && kA % 256 == 0 && kB % 256 == 0,
              "operand planes need 256 B alignment");

// Split-K reduction (a cluster of KS CTAs shares a tile): each 32-column
// slice of the tile has an owner rank (slice % KS); the other ranks put their
// fp32 sums for it into the owner's buffer, one 4 KB block per (sender, owned
// slice, lane quarter), 16-byte chunks of the 32 lanes interleaved.
constexpr int MAX_KS = 4;
constexpr uint32_t kRedBlock = 32 * EPI_COLS * 4;
constexpr uint32_t kRed = 64 * 1024;  // max over KS of (KS - 1) * ceil(4 / KS) * 4 blocks
__host__ __device__ constexpr int owned_slices(int KS) { return (4 + KS - 1) / KS; }

// Tile order.  Tile t -> (M tile, N tile): M tiles vary fastest, so the CTAs at
// work at one time share a few weight tiles and sweep all of A -- unless A (the
// activation codes, M x K bytes) is large and larger than the packed weights:
// then N tiles vary fastest, so that A is read from DRAM once and the weights
// (which then fit in L2) are the operand read again (at M = 8192, K = 14336 the
// M-fastest order read 3.5 GB from DRAM for 0.15 GB of operands).
__host__ __device__ inline bool n_fastest(int M, int N, int K) {
    const size_t a = size_t(M) * size_t(K), w = size_t(N) * size_t(K) / 2;
    return a > (size_t(64) << 20) && a > w;
}
__host__ __device__ inline void tile_coords(int t, int MT, int NT, bool nf, int& mt, int& nt) {
    if (nf) {
        mt = t / NT;
        nt = t % NT;
    } else {
        mt = t % MT;
        nt = t / MT;
    }
}
static_assert((2 - 1) * 2 * 4 * kRedBlock <= kRed && (3 - 1) * 2 * 4 * kRedBlock <= kRed &&
                  (4 - 1) * 1 * 4 * kRedBlock <= kRed, "reduction buffer too small");

struct Map {
    uint32_t ST, SC, LA, LU, CB, RED, BAR, SLOT, total;
};
constexpr uint32_t kCB = 128;  // per epilogue warp: its 32 columns' colscale and bias (fp16)
__host__ __device__ constexpr Map smem_map(int S, int rp, bool split) {
    Map m{};
    m.ST = 0;
    m.SC = m.ST + uint32_t(S) * kStage;
    m.LA = m.SC + SS * kScale;
    m.LU = m.LA + uint32_t(rp) * BM * 32;
    m.CB = m.LU + uint32_t(rp) * BN * 32;
    m.RED = m.CB + NUM_EPI_WARPS * kCB;
    m.BAR = m.RED + (split ? kRed : 0u);
    m.SLOT = m.BAR + (3 * S + 2 * SS + 2 * NPB + 6) * 8;
    m.total = m.SLOT + 16 + 1024;  // + base alignment
    return m;
}
static_assert(smem_map(4, 2, false).total <= 227 * 1024, "4 stages must fit at rank 32");
static_assert(smem_map(3, 8, false).total <= 227 * 1024, "3 stages must fit at rank 128");
static_assert(smem_map(3, 2, true).total <= 227 * 1024, "3 stages + the reduction buffer must fit at rank 32");

// DUMP: the debug variant of a schedule, which also writes every group's exact
// integer product to P and stores no Y (colscale and bias are not read).
// MIXED (with SPLIT): tiles below t_split run whole, the rest split over K.
template <int S, bool SPLIT, bool SK, bool DUMP, bool MIXED>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const uint8_t* __restrict__ ws, const uint8_t* __restrict__ packed,
                   const uint16_t* __restrict__ colscale, const uint16_t* __restrict__ bias, int M, int N, int K,
                   int r, uint16_t* __restrict__ Y, int32_t* __restrict__ P, int KS, int silu_I, int t_lo,
                   int t_hi, int t_split) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const int J = (G + GPJ - 1) / GPJ;  // jobs per tile
    // split-K: the KS CTAs of a cluster share a tile, rank kr taking jobs [j0, j1);
    // otherwise every CTA is its own "cluster" of one
    const int kr = SPLIT ? int(cluster_ctarank()) : 0;
    if (!SPLIT) KS = 1;
    if (MIXED) KS = 2;  // (a compile-time split keeps the epilogue within its registers)
    const int cid = int(blockIdx.x) / KS, ncl = int(gridDim.x) / KS;
    const int j0 = kr * J / KS, j1 = (kr + 1) * J / KS;
    const int RPB = r / 16;  // LoRA operand planes held in shared memory
    constexpr bool has_y = !DUMP;
    // Y 32-byte aligned: every 16-column chunk of a row is a 32-byte store (rows are
    // N x 2 bytes, N a multiple of 16); the API guarantees 16 bytes only
    const bool y32 = (reinterpret_cast<uintptr_t>(Y) & 31u) == 0;
    const ActLayout AL = act_layout(M, K, r);
    const PackedLayout PL = packed_layout(N, K, r);
    const int MT = AL.MT, NT = (N + BN - 1) / BN;
    const int tiles = MT * NT;
    const bool nf = n_fastest(M, N, K);
    // Work is walked as segments (tile t, jobs [a, b)).  Round-robin: tiles
    // [t_lo, t_split) are whole, CTA p taking t_lo + p, t_lo + p + gridDim.x, ...;
    // tiles [t_split, t_hi) are split over K, cluster cid taking t_split + cid,
    // t_split + cid + ncl, ... with jobs [j0, j1) on rank kr.  A launch may cover a
    // range of the tiles, and a split-K launch may run its full rounds whole and
    // only the last, thin round split.  Stream-K:
    // the tiles x J jobs, tile-major, are cut into gridDim.x equal runs, CTA p
    // taking run p; a tile cut between CTAs is finished by the CTA holding its
    // first job, which adds the later CTAs' fp32 sums handed over in the workspace.
    // (the host keeps tiles x J below 2^31)
    const int units = tiles * J;
    const int sk_ctas = int(gridDim.x);
    auto sk_start = [&](int p) -> int { return int((long long)p * units / sk_ctas); };
    // (the host passes t_lo <= t_split <= t_hi; only MIXED reads it)
    const int u_begin = SK       ? sk_start(int(blockIdx.x))
                        : !MIXED ? t_lo + cid
                                 : (t_lo + int(blockIdx.x) < t_split ? t_lo + int(blockIdx.x) : t_split + cid);
    const int u_end = SK ? sk_start(int(blockIdx.x) + 1) : t_hi;
    // segment u: tile t, jobs [a, b); split over the cluster or whole
    auto split_seg = [&](int u) -> bool { return SPLIT && (!MIXED || u >= t_split); };
    auto seg_at = [&](int u, int& t, int& a, int& b) {
        if (SK) {
            t = u / J;
            a = u - t * J;
            b = min(J, a + (u_end - u));
        } else {
            t = u;
            a = split_seg(u) ? j0 : 0;
            b = split_seg(u) ? j1 : J;
        }
    };
    auto seg_next = [&](int u, int a, int b) -> int {
        if (SK) return u + (b - a);
        if (!MIXED || u >= t_split) return u + ncl;
        const int nu = u + int(gridDim.x);
        return nu < t_split ? nu : t_split + cid;
    };
    // the LoRA term is added once per tile: by a whole tile's CTA, by split rank 0, or
    // by the stream-K segment holding job 0
    auto lora_planes = [&](int u, int a) -> int { return (SK ? a == 0 : (!split_seg(u) || kr == 0)) ? RPB : 0; };
    const Map mp = smem_map(S, RPB, SPLIT);

    auto full = [&](int s) { return base + mp.BAR + 8u * s; };             // copies landed (producers + tx)
    auto bready = [&](int s) { return base + mp.BAR + 8u * (S + s); };     // B operand expanded
    auto empty = [&](int s) { return base + mp.BAR + 8u * (2 * S + s); };  // MMAs done with the stage
    auto sfull = [&](int q) { return base + mp.BAR + 8u * (3 * S + q); };  // scale entry written
    auto sempty = [&](int q) { return base + mp.BAR + 8u * (3 * S + SS + q); };  // epilogue done with it
    auto tfull = [&](int b) { return base + mp.BAR + 8u * (3 * S + 2 * SS + b); };
    auto tempty = [&](int b) { return base + mp.BAR + 8u * (3 * S + 2 * SS + NPB + b); };
    const uint32_t lfull = base + mp.BAR + 8u * (3 * S + 2 * SS + 2 * NPB);
    const uint32_t lempty = lfull + 8u;
    const uint32_t mmadone = lfull + 16u;
    const uint32_t red_full = lfull + 24u;   // (owner) the senders' blocks for this tile have landed
    const uint32_t red_empty = lfull + 32u;  // (sender) the owners have consumed this CTA's blocks
    const uint32_t own_done = lfull + 40u;   // (owner) this CTA's owner warps have read the blocks
    const int own = SPLIT ? (kr < 4 % KS ? 4 / KS + 1 : 4 / KS) : 4;  // slices owned by this rank
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + mp.SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + mp.SLOT + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), NUM_PRODUCERS);
            mbar_init(bready(s), NUM_EXP_WARPS);
            mbar_init(empty(s), 1);
        }
        for (int q = 0; q < SS; ++q) {
            mbar_init(sfull(q), NUM_EXP_WARPS);
            mbar_init(sempty(q), NUM_EPI_WARPS);
        }
        for (int b = 0; b < NPB; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), NUM_EPI_WARPS);
        }
        mbar_init(lfull, 2);
        mbar_init(lempty, 1);
        mbar_init(mmadone, 1);
        if (SPLIT) {
            mbar_init(red_full, 1);                  // the owner's expect-tx; the senders complete bytes
            mbar_init(red_empty, uint32_t(KS - 1));  // one arrive per owner CTA
            mbar_init(own_done, uint32_t(own * 4));  // one arrive per owner warp
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(base + mp.SLOT, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int no_abort = 0;
    // Everything above touches only this CTA's shared and tensor memory, so it
    // overlaps the previous kernel; so does warming L2 with the weight records of
    // the first jobs (a prefetch only fills the cache, the copies proper come
    // after the wait).  Global data the previous kernel may write is read after it.
    if (warp == WARP_PRODUCER_W && lane == 0 && u_begin < u_end) {
        int t0, a0, b0;
        seg_at(u_begin, t0, a0, b0);
        int mt0, nt0;
        tile_coords(t0, MT, NT, nf, mt0, nt0);
        const int n0 = nt0 * BN, rows = min(BN, N - n0);
        for (int g = a0 * GPJ; g < min(G, (a0 + S) * GPJ); ++g)
            prefetch_l2(packed + PL.qW + (size_t(g) * N + n0) * 32, uint32_t(rows) * 32);
    }
    pdl_wait();
    pdl_launch_dependents();

    auto fail = [&]() {
        atomicExch(&g_tc_status, int(W4A4_ERR_TIMEOUT));
        *abort_flag = 1;
    };

    // Register re-budgeting: each role re-sizes its warpgroup on entry (the
    // four warps of a warpgroup always take the same branch).
    if (warp >= WARP_EXP0) regs_dec<OTHER_REGS>();

    if (warp == WARP_PRODUCER || warp == WARP_PRODUCER_W || warp == WARP_PRODUCER_S) {
        // role 0 = activation codes + LoRA activations, 1 = weight nibbles + L_up,
        // 2 = (sA, SA) and the fp16 weight scales.  Each arrives on the stage's
        // barrier with its own byte count.  Lane 0 issues; the warp walks the loop.
        const int role = warp == WARP_PRODUCER ? 0 : warp == WARP_PRODUCER_W ? 1 : 2;
        uint32_t it = 0, lp = 0, lora_issued = 0;
        bool ok = true;
        int t = 0, a = 0, b = 0;
        for (int u = u_begin; u < u_end && ok; u = seg_next(u, a, b)) {
            seg_at(u, t, a, b);
            const int RP = lora_planes(u, a);
            int mt, nt;
            tile_coords(t, MT, NT, nf, mt, nt);
            const int n0 = nt * BN;
            const int rows = min(BN, N - n0);
            if (RP > 0 && role < 2) {
                if (!warp_wait_parity_suspend(lempty, lp ^ 1u, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    if (role == 0) {
                        mbar_expect_tx(lfull, uint32_t(RP) * BM * 32);
                        bulk_g2s(base + mp.LA, ws + AL.La + size_t(mt) * RP * (BM * 32), uint32_t(RP) * BM * 32,
                                 lfull);
                    } else {
                        mbar_expect_tx(lfull, uint32_t(RP) * rows * 32);
                        for (int p = 0; p < RP; ++p)
                            bulk_g2s(base + mp.LU + uint32_t(p) * BN * 32, packed + PL.Lu + (size_t(p) * N + n0) * 32,
                                     uint32_t(rows) * 32, lfull);
                    }
                }
                __syncwarp();
                lp ^= 1u;
                lora_issued = 1;
            }
            for (int jb = a; jb < b; ++jb) {
                const int g0 = jb * GPJ, ng = min(GPJ, G - g0);
                const int s = int(it % S);
                const uint32_t ph = (it / S) & 1u;
                if (!warp_wait_parity_suspend(empty(s), ph ^ 1u, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t sb = base + mp.ST + uint32_t(s) * kStage;
                    const size_t ag = size_t(mt) * G + g0;
                    if (role == 0) {
                        mbar_expect_tx(full(s), uint32_t(ng) * kA);
                        bulk_g2s(sb + ST_A, ws + AL.qA + ag * kA, uint32_t(ng) * kA, full(s));
                    } else if (role == 1) {
                        mbar_expect_tx(full(s), uint32_t(ng * rows) * 32);
                        for (int j = 0; j < ng; ++j)
                            bulk_g2s(sb + ST_W + uint32_t(j) * kW, packed + PL.qW + (size_t(g0 + j) * N + n0) * 32,
                                     uint32_t(rows) * 32, full(s));
                    } else {
                        mbar_expect_tx(full(s), uint32_t(ng) * kS + uint32_t(ng * rows) * 2);
                        bulk_g2s(sb + ST_S, ws + AL.sS + ag * kS, uint32_t(ng) * kS, full(s));
                        for (int j = 0; j < ng; ++j)
                            bulk_g2s(sb + ST_SW + uint32_t(j) * kSw, packed + PL.sW + (size_t(g0 + j) * N + n0) * 2,
                                     uint32_t(rows) * 2, full(s));
                    }
                }
                __syncwarp();
                ++it;
            }
        }
        if (!ok && lane == 0) fail();
        // drain: the copies of the last S jobs (distinct stages) and the last LoRA load
        if (lane == 0) {
            for (uint32_t k = (it > uint32_t(S) ? it - S : 0u); k < it; ++k)
                wait_parity(full(int(k % S)), (k / S) & 1u, &no_abort, DRAIN_LIMIT_NS);
            if (lora_issued) wait_parity(lfull, lp ^ 1u, &no_abort, DRAIN_LIMIT_NS);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        constexpr uint32_t IDESC = idesc_m128(BN);
        uint32_t it = 0, jc = 0, lp = 0;
        bool ok = true;
        int t = 0, a = 0, b = 0;
        for (int u = u_begin; u < u_end && ok; u = seg_next(u, a, b)) {
            seg_at(u, t, a, b);
            const int RP = lora_planes(u, a);
            if (RP > 0) {
                // the LoRA product takes a job buffer of its own (first 128 columns)
                const uint32_t bf = jc % NPB, tph = (jc / NPB) & 1u;
                if (!warp_wait_parity_suspend(tempty(bf), tph ^ 1u, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS) ||
                    !warp_wait_parity_suspend(lfull, lp, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    for (int p = 0; p < RP; ++p)
                        mma_f16(tmem + bf * (GPJ * BN), sdesc_sw32(base + mp.LA + uint32_t(p) * BM * 32),
                                sdesc_sw32(base + mp.LU + uint32_t(p) * BN * 32), IDESC, p > 0 ? 1u : 0u);
                    mma_commit(tfull(bf));
                    mma_commit(lempty);
                }
                __syncwarp();
                ++jc;
                lp ^= 1u;
            }
            for (int jb = a; jb < b; ++jb) {
                const int ng = min(GPJ, G - jb * GPJ);
                const int s = int(it % S);
                const uint32_t ph = (it / S) & 1u;
                const uint32_t bf = jc % NPB, tph = (jc / NPB) & 1u;
                if (!warp_wait_parity_suspend(full(s), ph, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS) ||
                    !warp_wait_parity_suspend(bready(s), ph, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS) ||
                    !warp_wait_parity_suspend(tempty(bf), tph ^ 1u, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sb = base + mp.ST + uint32_t(s) * kStage;
                    for (int j = 0; j < ng; ++j) {
                        const uint32_t d = tmem + bf * (GPJ * BN) + uint32_t(j) * BN;
                        const uint32_t a0 = sb + ST_A + uint32_t(j) * kA, b0 = sb + ST_B + uint32_t(j) * kB;
                        mma_f8(d, sdesc_sw32(a0), sdesc_sw32(b0), IDESC, 0u);
                        mma_f8(d, sdesc_sw32(a0 + BM * 32), sdesc_sw32(b0 + BN * 32), IDESC, 1u);
                    }
                    mma_commit(tfull(bf));
                    mma_commit(empty(s));
                }
                __syncwarp();
                ++it;
                ++jc;
            }
        }
        if (!ok && lane == 0) fail();
        if (lane == 0) {
            mma_commit(mmadone);  // every MMA issued above has completed once this arrives
            wait_parity(mmadone, 0u, &no_abort, DRAIN_LIMIT_NS);
        }
        __syncwarp();
    } else if (warp >= WARP_EXP0 && warp < WARP_EXP0 + NUM_EXP_WARPS) {
        // ---- expansion: packed offset-binary nibbles -> E4M3 B operand planes, scales -> fp32
        const int e = warp - WARP_EXP0;
        const int row = e * EXP_ROWS + lane;
        static_assert(EXP_ROWS == 32, "one expansion row per lane");
        uint32_t it = 0;
        bool ok = true;
        int t = 0, a = 0, b = 0;
        for (int u = u_begin; u < u_end && ok; u = seg_next(u, a, b)) {
            seg_at(u, t, a, b);
            for (int jb = a; jb < b; ++jb) {
                const int ng = min(GPJ, G - jb * GPJ);
                const int s = int(it % S), q = int(it % SS);
                const uint32_t ph = (it / S) & 1u, sph = (it / SS) & 1u;
                if (!warp_wait_parity_suspend(full(s), ph, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS) ||
                    !warp_wait_parity_suspend(sempty(q), sph ^ 1u, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS)) {
                    ok = false;
                    break;
                }
                uint8_t* sp = gbase + mp.ST + uint32_t(s) * kStage;
                uint8_t* scp = gbase + mp.SC + uint32_t(q) * kScale;
                for (int j = 0; j < ng; ++j) {
                    const uint8_t* wp = sp + ST_W + uint32_t(j) * kW;
                    const uint4 w01 = *reinterpret_cast<const uint4*>(wp + row * 32);
                    const uint4 w23 = *reinterpret_cast<const uint4*>(wp + row * 32 + 16);
                    // words: w01 = (q0h0, q0h1, q1h0, q1h1), w23 = (q2h0, q2h1, q3h0, q3h1)
                    // (the bytes are the codes + 8, as E4M3 values scaled by 2^-9)
                    uint4 p0c0, p0c1, p1c0, p1c1;
                    expand8(w01.x, p0c0.x, p0c1.x);
                    expand8(w01.z, p0c0.y, p0c1.y);
                    expand8(w23.x, p0c0.z, p0c1.z);
                    expand8(w23.z, p0c0.w, p0c1.w);
                    expand8(w01.y, p1c0.x, p1c1.x);
                    expand8(w01.w, p1c0.y, p1c1.y);
                    expand8(w23.y, p1c0.z, p1c1.z);
                    expand8(w23.w, p1c0.w, p1c1.w);
                    uint8_t* bp = sp + ST_B + uint32_t(j) * kB;
                    *reinterpret_cast<uint4*>(bp + row * 32 + swz32(row, 0) * 16) = p0c0;
                    *reinterpret_cast<uint4*>(bp + row * 32 + swz32(row, 1) * 16) = p0c1;
                    *reinterpret_cast<uint4*>(bp + BN * 32 + row * 32 + swz32(row, 0) * 16) = p1c0;
                    *reinterpret_cast<uint4*>(bp + BN * 32 + row * 32 + swz32(row, 1) * 16) = p1c1;
                    uint8_t* sg = scp + uint32_t(j) * kScaleG;
                    reinterpret_cast<float*>(sg)[row] = __half2float(
                        __ushort_as_half(reinterpret_cast<const uint16_t*>(sp + ST_SW + uint32_t(j) * kSw)[row]));
                    // (sA, SA) of this lane's row (rows and weight rows share the index range 0..127)
                    reinterpret_cast<float2*>(sg + BN * 4)[row] =
                        reinterpret_cast<const float2*>(sp + ST_S + uint32_t(j) * kS)[row];
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bready(s));
                    mbar_arrive(sfull(q));
                }
                ++it;
            }
        }
        if (!ok) fail();
    } else if (warp < NUM_EPI_WARPS) {
        // ---- epilogue
        regs_inc<EPI_REGS>();
        const int lq = warp & 3;                // TMEM lane quarter this warp may access
        const int c0 = (warp >> 2) * EPI_COLS;  // column slice of the tile
        const int row = lq * 32 + lane;
        const uint32_t tl = tmem + (uint32_t(lq * 32) << 16) + uint32_t(c0);
        uint32_t it = 0, jc = 0, tc = 0;
        bool ok = true;
        int t = 0, a = 0, b = 0;
        for (int u = u_begin; u < u_end && ok; u = seg_next(u, a, b)) {
            seg_at(u, t, a, b);
            const int RP = lora_planes(u, a);
            int mt, nt;
            tile_coords(t, MT, NT, nf, mt, nt);
            const int n0 = nt * BN;
            const int m = mt * BM + row;
            uint64_t acc[EPI_COLS / 2];  // running sums as packed column pairs
            // this warp's colscale / bias for the tile's store, fetched while the jobs run:
            // 16-byte chunks [cs 0..31 | bias 0..31], or with the SiLU epilogue
            // [cs gate 0..15 | cs up | bias gate | bias up]
            uint8_t* const cbw = gbase + mp.CB + uint32_t(warp) * kCB;
            // (only warps that store this segment: not a stream-K hand-over, not a split-K sender)
            const bool stores = has_y && !(SK && a > 0) && !(split_seg(u) && ((warp >> 2) % KS) != kr);
            if (stores && lane < 8) {
                const uint16_t* src = nullptr;
                if (silu_I > 0) {
                    const int hb = (n0 >> 1) + (c0 >> 1), which = lane >> 1;
                    if (hb < silu_I)
                        src = (which < 2 ? colscale : bias) + ((which & 1) ? silu_I : 0) + hb + (lane & 1) * 8;
                    if (which >= 2 && !bias) src = nullptr;
                } else {
                    const int n = n0 + c0 + (lane & 3) * 8;
                    if (n < N) src = lane < 4 ? colscale : bias;
                    if (src) src += n;
                }
                if (src) cp_async16(cbw + lane * 16, src);
                else *reinterpret_cast<uint4*>(cbw + lane * 16) = make_uint4(0, 0, 0, 0);
            }
            if (stores) cp_async_commit();
            if (RP > 0) {
                const uint32_t bf = jc % NPB, tph = (jc / NPB) & 1u;
                if (!warp_wait_parity_suspend(tfull(bf), tph, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float l[EPI_COLS];
                tmem_ld32(tl + bf * (GPJ * BN), l);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty(bf));
#pragma unroll
                for (int c = 0; c < EPI_COLS / 2; ++c) acc[c] = f2_pack(l[2 * c], l[2 * c + 1]);
                ++jc;
            } else {
#pragma unroll
                for (int c = 0; c < EPI_COLS / 2; ++c) acc[c] = 0ull;
            }
            for (int jb = a; jb < b; ++jb) {
                const int g0 = jb * GPJ;
                const bool two = g0 + 1 < G;
                const int q = int(it % SS);
                const uint32_t sph = (it / SS) & 1u;
                const uint32_t bf = jc % NPB, tph = (jc / NPB) & 1u;
                if (!warp_wait_parity_suspend(tfull(bf), tph, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS) ||
                    !warp_wait_parity_suspend(sfull(q), sph, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* sc0 = gbase + mp.SC + uint32_t(q) * kScale;
                const uint8_t* sc1 = sc0 + kScaleG;
                const float2 sv0 = reinterpret_cast<const float2*>(sc0 + BN * 4)[row];
                const float2 sv1 = two ? reinterpret_cast<const float2*>(sc1 + BN * 4)[row] : make_float2(0.f, 0.f);
                const float cm0 = (-8.f * sv0.y) * sv0.x, cm1 = (-8.f * sv1.y) * sv1.x;
                // (2^9 sA: the tensor memory holds 2^-9 D)
                const float sx0 = sv0.x * kExpand8Scale, sx1 = sv1.x * kExpand8Scale;
                const uint64_t sa0 = f2_pack(sx0, sx0), cc0 = f2_pack(cm0, cm0);
                const uint64_t sa1 = f2_pack(sx1, sx1), cc1 = f2_pack(cm1, cm1);
                const uint32_t tb = tl + bf * (GPJ * BN);
#pragma unroll
                for (int ch = 0; ch < EPI_COLS / 16; ++ch) {
                    float d0[16], d1[16];
                    tmem_ld16(tb + ch * 16, d0);
                    if (two) tmem_ld16(tb + BN + ch * 16, d1);
                    tmem_wait_ld();
                    if (ch == EPI_COLS / 16 - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(tempty(bf));
                    }
                    if (DUMP && m < M) {
                        // partials dump: P = 2^9 (2^-9 D) - 8 SA, exact in fp32 (|D| < 2^13)
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int n = n0 + c0 + ch * 16 + c;
                            if (n < N) {
                                P[(size_t(m) * N + n) * G + g0] = int32_t(d0[c] * kExpand8Scale - 8.f * sv0.y);
                                if (two)
                                    P[(size_t(m) * N + n) * G + g0 + 1] = int32_t(d1[c] * kExpand8Scale - 8.f * sv1.y);
                            }
                        }
                    }
                    {
                        // t = sA D - 8 SA sA, acc += sW t, two columns per instruction
                        uint64_t* a = acc + ch * 8;
                        const ulonglong2* w0 = reinterpret_cast<const ulonglong2*>(sc0 + (c0 + ch * 16) * 4);
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const ulonglong2 w = w0[c4];
                            a[2 * c4] = ffma2_b64(w.x, ffma2_b64(sa0, f2_pack(d0[4 * c4], d0[4 * c4 + 1]), cc0),
                                                  a[2 * c4]);
                            a[2 * c4 + 1] = ffma2_b64(
                                w.y, ffma2_b64(sa0, f2_pack(d0[4 * c4 + 2], d0[4 * c4 + 3]), cc0), a[2 * c4 + 1]);
                        }
                        if (two) {
                            const ulonglong2* w1 = reinterpret_cast<const ulonglong2*>(sc1 + (c0 + ch * 16) * 4);
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) {
                                const ulonglong2 w = w1[c4];
                                a[2 * c4] = ffma2_b64(w.x, ffma2_b64(sa1, f2_pack(d1[4 * c4], d1[4 * c4 + 1]), cc1),
                                                      a[2 * c4]);
                                a[2 * c4 + 1] = ffma2_b64(
                                    w.y, ffma2_b64(sa1, f2_pack(d1[4 * c4 + 2], d1[4 * c4 + 3]), cc1), a[2 * c4 + 1]);
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sempty(q));
                ++it;
                ++jc;
            }
            if (!ok) break;
            if constexpr (SK) {
                // this warp's slice of a CTA's hand-over slot: 8 x (32 lanes x 16 B), coalesced
                uint8_t* const wsw = const_cast<uint8_t*>(ws);
                uint32_t* const flags = reinterpret_cast<uint32_t*>(wsw + AL.flags);
                auto slot_of = [&](int p) {
                    return reinterpret_cast<float4*>(wsw + AL.part + (size_t(p) * kStreamKWarps + warp) * (32 * 32 * 4));
                };
                if (a > 0) {
                    // a later part of a tile: hand the sums to the CTA that finishes it
                    float4* dst = slot_of(int(blockIdx.x));
#pragma unroll
                    for (int c4 = 0; c4 < EPI_COLS / 4; ++c4) {
                        const float2 lo = f2_unpack(acc[2 * c4]), hi = f2_unpack(acc[2 * c4 + 1]);
                        __stcg(dst + c4 * 32 + lane, make_float4(lo.x, lo.y, hi.x, hi.y));
                    }
                    // every lane releases its own chunks; the warp's counter reaches 32 when all have landed
                    red_add_release_gpu(flags + blockIdx.x * kStreamKWarps + warp, 1u);
                    continue;
                }
                if (b < J) {
                    // the tile's first part: add the later CTAs' sums in CTA order
                    const int tile_end = (t + 1) * J;
                    for (int p = int(blockIdx.x) + 1; p < sk_ctas && sk_start(p) < tile_end; ++p) {
                        uint32_t* fl = flags + p * kStreamKWarps + warp;
                        const bool got = __all_sync(0xffffffffu, wait_flag_gpu(fl, 32u, abort_flag, WAIT_LIMIT_NS));
                        if (!got) {
                            ok = false;
                            break;
                        }
                        const float4* src = slot_of(p);
#pragma unroll
                        for (int c4 = 0; c4 < EPI_COLS / 4; ++c4) {
                            const float4 v = __ldcg(src + c4 * 32 + lane);
                            const float2 lo = f2_unpack(acc[2 * c4]), hi = f2_unpack(acc[2 * c4 + 1]);
                            acc[2 * c4] = f2_pack(lo.x + v.x, lo.y + v.y);
                            acc[2 * c4 + 1] = f2_pack(hi.x + v.z, hi.y + v.w);
                        }
                        __syncwarp();
                        if (lane == 0) *fl = 0u;  // cleared for the next call on this workspace
                    }
                    if (!ok) break;
                }
            }
            if (split_seg(u)) {
                const int sl = warp >> 2, owner = sl % KS;
                if (owner != kr) {
                    // send this slice's sums to its owner once it has consumed the previous ones
                    if (!warp_wait_parity_cluster(red_empty, (tc & 1u) ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    const int src = kr < owner ? kr : kr - 1;
                    const uint32_t blk = base + mp.RED +
                                         uint32_t(((src * owned_slices(KS) + sl / KS) * 4 + lq)) * kRedBlock;
                    const uint32_t rblk = mapa_shared(blk, uint32_t(owner));
                    const uint32_t rbar = mapa_shared(red_full, uint32_t(owner));
#pragma unroll
                    for (int c4 = 0; c4 < EPI_COLS / 4; ++c4) {
                        const float2 lo = f2_unpack(acc[2 * c4]), hi = f2_unpack(acc[2 * c4 + 1]);
                        st_async_v4(rblk + uint32_t(c4 * 32 + lane) * 16u, make_float4(lo.x, lo.y, hi.x, hi.y), rbar);
                    }
                    ++tc;
                    continue;  // the owner stores this slice
                }
                // owner: one thread posts the bytes this CTA receives for the tile
                if (sl == kr && lq == 0 && lane == 0)
                    mbar_expect_tx(red_full, uint32_t(own * 4 * (KS - 1)) * kRedBlock);
                if (!warp_wait_parity_suspend(red_full, tc & 1u, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS)) {
                    ok = false;
                    break;
                }
                // add the other ranks' sums in rank order
                for (int src_rank = 0; src_rank < KS; ++src_rank) {
                    if (src_rank == kr) continue;
                    const int src = src_rank < kr ? src_rank : src_rank - 1;
                    const uint8_t* blk =
                        gbase + mp.RED + uint32_t(((src * owned_slices(KS) + sl / KS) * 4 + lq)) * kRedBlock;
#pragma unroll
                    for (int c4 = 0; c4 < EPI_COLS / 4; ++c4) {
                        const float4 v = *reinterpret_cast<const float4*>(blk + (c4 * 32 + lane) * 16);
                        const float2 lo = f2_unpack(acc[2 * c4]), hi = f2_unpack(acc[2 * c4 + 1]);
                        acc[2 * c4] = f2_pack(lo.x + v.x, lo.y + v.y);
                        acc[2 * c4 + 1] = f2_pack(hi.x + v.z, hi.y + v.w);
                    }
                }
                // once every owner warp of this CTA has read its blocks, one thread hands
                // the buffer back to the senders
                __syncwarp();
                if (lane == 0) mbar_arrive(own_done);
                if (sl == kr && lq == 0) {
                    if (!warp_wait_parity_suspend(own_done, tc & 1u, abort_flag, WAIT_LIMIT_NS, SUSPEND_NS)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0)
                        for (int src_rank = 0; src_rank < KS; ++src_rank)
                            if (src_rank != kr) mbar_arrive_remote(mapa_shared(red_empty, uint32_t(src_rank)));
                }
                ++tc;  // (counts the split segments only: both ranks walk the same ones)
            }
            if constexpr (has_y) {
                cp_async_wait<0>();  // this warp's colscale / bias chunks
                __syncwarp();
                if (m < M && silu_I > 0) {
                    // fused gate|up weights: columns 0..15 of this warp's slice are gates, 16..31
                    // the matching ups (gate_up_row); h = silu(gate) * up for 16 outputs
                    const int hb = (n0 >> 1) + (c0 >> 1);
                    if (hb < silu_I) {
                        const uint4* cbv = reinterpret_cast<const uint4*>(cbw);
                        uint16_t* const dst = Y + size_t(m) * silu_I + hb;
                        uint32_t hw[8];
#pragma unroll
                        for (int q8 = 0; q8 < 2; ++q8) {
                            const uint4 csg = cbv[q8], csu = cbv[2 + q8], bg = cbv[4 + q8], bu = cbv[6 + q8];
                            const uint32_t w_cg[4] = {csg.x, csg.y, csg.z, csg.w}, w_cu[4] = {csu.x, csu.y, csu.z, csu.w};
                            const uint32_t w_bg[4] = {bg.x, bg.y, bg.z, bg.w}, w_bu[4] = {bu.x, bu.y, bu.z, bu.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float2 c2g = __half22float2(*reinterpret_cast<const __half2*>(&w_cg[j]));
                                const float2 c2u = __half22float2(*reinterpret_cast<const __half2*>(&w_cu[j]));
                                const float2 b2g = __half22float2(*reinterpret_cast<const __half2*>(&w_bg[j]));
                                const float2 b2u = __half22float2(*reinterpret_cast<const __half2*>(&w_bu[j]));
                                const float2 ag = f2_unpack(acc[q8 * 4 + j]), au = f2_unpack(acc[8 + q8 * 4 + j]);
                                const float g0 = fmaf(c2g.x, ag.x, b2g.x), g1 = fmaf(c2g.y, ag.y, b2g.y);
                                const float u0 = fmaf(c2u.x, au.x, b2u.x), u1 = fmaf(c2u.y, au.y, b2u.y);
                                // silu(g) = g / (1 + e^-g) with the fast exponential and divide
                                // (relative error ~1e-6; e^-g = inf gives -0)
                                const __half2 h = __floats2half2_rn(__fdividef(g0, 1.0f + __expf(-g0)) * u0,
                                                                    __fdividef(g1, 1.0f + __expf(-g1)) * u1);
                                hw[q8 * 4 + j] = *reinterpret_cast<const uint32_t*>(&h);
                            }
                        }
                        if (y32) {  // (rows of H are N/2 x 2 bytes, N a multiple of 32)
                            st_global_v8(dst, hw);
                        } else {
                            reinterpret_cast<uint4*>(dst)[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                            reinterpret_cast<uint4*>(dst)[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                        }
                    }
                } else if (m < M) {
                    // 16 columns (32 bytes) per store: N is a multiple of 16, so a chunk that
                    // starts below N ends within it
                    const uint4* cbv = reinterpret_cast<const uint4*>(cbw);
#pragma unroll
                    for (int c16 = 0; c16 < EPI_COLS / 16; ++c16) {
                        const int n = n0 + c0 + c16 * 16;
                        if (n < N) {
                            uint32_t out[8];
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                const uint4 csv = cbv[c16 * 2 + q];
                                const uint4 bsv = cbv[4 + c16 * 2 + q];
                                const uint32_t cw[4] = {csv.x, csv.y, csv.z, csv.w};
                                const uint32_t bw[4] = {bsv.x, bsv.y, bsv.z, bsv.w};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const float2 cs2 = __half22float2(*reinterpret_cast<const __half2*>(&cw[j]));
                                    const float2 b2 = __half22float2(*reinterpret_cast<const __half2*>(&bw[j]));
                                    const float2 av = f2_unpack(acc[(c16 * 2 + q) * 4 + j]);
                                    const float y0 = fmaf(cs2.x, av.x, b2.x);
                                    const float y1 = fmaf(cs2.y, av.y, b2.y);
                                    const __half2 h = __floats2half2_rn(y0, y1);
                                    out[q * 4 + j] = *reinterpret_cast<const uint32_t*>(&h);
                                }
                            }
                            uint16_t* const dst = Y + size_t(m) * N + n;
                            if (y32) {
                                st_global_v8(dst, out);
                            } else {
                                reinterpret_cast<uint4*>(dst)[0] = make_uint4(out[0], out[1], out[2], out[3]);
                                reinterpret_cast<uint4*>(dst)[1] = make_uint4(out[4], out[5], out[6], out[7]);
                            }
                        }
                    }
                }
            }
        }
        cp_async_wait<0>();  // (a segment left early) nothing lands in shared memory after this
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    if (SPLIT) cluster_sync_all();  // peers may still be using this CTA's shared memory
    tc_fence_after();
    if (warp == WARP_MMA) tmem_dealloc(tmem, TMEM_COLS);
}

// Registers per thread the kernel was compiled for (cached per instantiation).
template <int S, bool SPLIT, bool SK, bool DUMP, bool MIXED>
int launch_regs() {
    static int regs = -1;
    if (regs < 0) {
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, gemm_tc_kernel<S, SPLIT, SK, DUMP, MIXED>) != cudaSuccess) return 0;
        regs = fa.numRegs;
    }
    return regs;
}

template <int S, bool SPLIT, bool SK, bool DUMP, bool MIXED = false>
w4a4_status launch_impl(const uint8_t* ws, const uint8_t* packed, const uint16_t* cs, const uint16_t* bias, int M,
                        int N, int K, int r, uint16_t* Y, int32_t* P, int KS, cudaStream_t s, int sk_ctas = 0,
                        int silu_I = 0, int t_lo = 0, int t_hi = -1, int t_split = -1) {
    auto kern = gemm_tc_kernel<S, SPLIT, SK, DUMP, MIXED>;
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    const int rp = r / 16;
    const uint32_t smem_max = smem_map(S, S == 4 ? 2 : (SPLIT ? 2 : 8), SPLIT).total;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_max)) != cudaSuccess)
            return W4A4_ERR_CUDA;
        attr_done[dev] = 1;
    }
    // the setmaxnreg split needs the launch-time register pool to cover it
    if (launch_regs<S, SPLIT, SK, DUMP, MIXED>() * NUM_THREADS <
        NUM_EPI_WARPS * 32 * EPI_REGS + (NUM_THREADS - NUM_EPI_WARPS * 32) * OTHER_REGS)
        return W4A4_ERR_CUDA;
    const int MT = (M + BM - 1) / BM, NT = (N + BN - 1) / BN;
    const int tiles = MT * NT;
    if (t_hi < 0) t_hi = tiles;
    const int ntl = t_hi - t_lo;  // the tiles of this launch
    const uint32_t smem = smem_map(S, rp, SPLIT).total;
    if (!SPLIT) {
        const int grid = SK ? sk_ctas : (ntl < device_sm_count() ? ntl : device_sm_count());
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        cfg.attrs = attr;
        cfg.numAttrs = add_pdl_attr(attr, 0);
        cfg.gridDim = dim3(unsigned(grid));
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        if (cudaLaunchKernelEx(&cfg, kern, ws, packed, cs, bias, M, N, K, r, Y, P, 1, silu_I, t_lo, t_hi, t_hi) !=
            cudaSuccess) {
            cudaGetLastError();
            return W4A4_ERR_CUDA;
        }
        set_dispatch("gemm_tc tcgen05.f8f6f4 tile=%dx%d groups/job=%d stages=%d tiles=%d grid=%d%s%s%s", BM, BN, GPJ,
                     S, tiles, grid, SK ? " stream-K" : "", silu_I ? " silu(gate)*up" : "",
                     DUMP ? " (partials dump)" : "");
        return launch_status();
    }
    // clusters of KS CTAs, as many as can be resident at once (persistent over tiles)
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(KS);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.gridDim = dim3(unsigned(ntl * KS));
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess || active < 1) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    // t_split > t_lo: the tiles below it run whole, one per CTA and round, on every
    // resident cluster's CTAs; the rest split over K, one per cluster and round
    const bool mixed = MIXED && t_split > t_lo && t_split < t_hi;
    if (!mixed) t_split = t_lo;
    const int split_tiles = t_hi - t_split;
    const int clusters = mixed ? active : (split_tiles < active ? split_tiles : active);
    cfg.gridDim = dim3(unsigned(clusters * KS));
    cfg.numAttrs = add_pdl_attr(attr, 1);
    if (cudaLaunchKernelEx(&cfg, kern, ws, packed, cs, bias, M, N, K, r, Y, P, KS, silu_I, t_lo, t_hi, t_split) !=
        cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    set_dispatch("gemm_tc tcgen05.f8f6f4 tile=%dx%d groups/job=%d stages=%d split-K=%d (cluster) tiles=%d grid=%d%s%s%s",
                 BM, BN, GPJ, S, KS, tiles, clusters * KS, n_fastest(M, N, K) ? " N-tiles-fastest" : "",
                 silu_I ? " silu(gate)*up" : "", DUMP ? " (partials dump)" : "");
    return launch_status();
}

}  // namespace

// Clusters of `ks` split-K CTAs that can be resident at once (cached per device and ks).
static int resident_clusters(int ks) {
    static int cache[64][MAX_KS + 1] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev][ks] == 0) {
        auto kern = gemm_tc_kernel<3, true, false, false, false>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem_map(3, 2, true).total)) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = unsigned(ks);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = smem_map(3, 2, true).total;
        cfg.gridDim = dim3(unsigned(ks * 64));
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = -1;
        }
        cache[dev][ks] = n;
    }
    return cache[dev][ks];
}

// Schedule: the cheapest of round-robin tiles, split-K over clusters, the full
// rounds round-robin followed by the last round split over K (in the same
// launch on clusters of two, or alone in a second launch on clusters sized to
// fill the SMs), and stream-K, in units of one job's time:
//  - round-robin: rounds of tiles x jobs per tile;
//  - split-K: rounds x (jobs / KS + the cluster reduction, about 1.5 jobs);
//  - last round split in the same launch, for a last round of at most one tile
//    per cluster: (rounds - 1) x jobs x 1.04 + jobs / 2 + 1.5 (the factor: the
//    three-stage ring that the reduction buffer leaves room for, measured 4%
//    slower per job on long tiles);
//  - last round split in a second launch, for a last round at most half full:
//    (rounds - 1) x jobs + jobs / KS + 1.5 + about 5 jobs for the second launch
//    (its wait for the first and a tile's fixed costs: measured, a K = 1024
//    tile of 8 jobs lost to it);
//  - stream-K: the longest run of jobs + the hand-over of a tile's sums (about
//    1 job).
// Rank 128 LoRA operands leave no room for the cluster reduction buffer;
// stream-K needs the hand-over area of the workspace.
struct TcSchedule {
    int ks, sk_ctas;       // sk_ctas > 0: stream-K over that many CTAs
    int tail_ks, tail_lo;  // tail_ks > 1: tiles [0, tail_lo) round-robin, then the rest split over tail_ks
    bool tail_inline;      // ... in the same launch (clusters of two), else in a second launch
};
static TcSchedule tc_schedule(int M, int N, int K, int r, bool sk_room) {
    const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int jobs = (K / kGroup + GPJ - 1) / GPJ;
    TcSchedule best_s{1, 0, 1, 0, false};
    if (tiles <= 0) return best_s;
    const int sms = device_sm_count();
    double best = double((tiles + sms - 1) / sms) * jobs;
    for (int ks = 2; r <= 32 && ks <= MAX_KS && ks <= jobs; ++ks) {
        const int cl = resident_clusters(ks);
        if (cl < 1) continue;
        const double cost = double((tiles + cl - 1) / cl) * (double((jobs + ks - 1) / ks) + 1.5);
        if (cost < best) {
            best = cost;
            best_s = TcSchedule{ks, 0, 1, 0, false};
        }
    }
    const int cl2 = r <= 32 && jobs >= 2 ? resident_clusters(2) : 0;
    if (cl2 >= 1 && 2 * cl2 <= sms) {
        const int grid = 2 * cl2, rounds = (tiles + grid - 1) / grid, rem = tiles - (rounds - 1) * grid;
        if (rounds >= 2 && rem <= cl2) {
            const double cost = 1.04 * double(rounds - 1) * jobs + double((jobs + 1) / 2) + 1.5;
            if (cost < best) {
                best = cost;
                best_s = TcSchedule{1, 0, 2, (rounds - 1) * grid, true};
            }
        }
    }
    const int rounds = (tiles + sms - 1) / sms, rem = tiles - (rounds - 1) * sms;
    if (rounds >= 2 && 2 * rem <= sms && r <= 32) {
        for (int ks = 2; ks <= MAX_KS && ks <= jobs && ks * rem <= sms; ++ks) {
            if (resident_clusters(ks) < rem) continue;
            const double cost = double(rounds - 1) * jobs + double((jobs + ks - 1) / ks) + 1.5 + 5.0;
            if (cost < best) {
                best = cost;
                best_s = TcSchedule{1, 0, ks, (rounds - 1) * sms, false};
            }
        }
    }
    if (sk_room && (long long)tiles * jobs < (1ll << 31) / kStreamKSlots) {
        const long long units = (long long)tiles * jobs;
        long long p = sms < kStreamKSlots ? sms : kStreamKSlots;
        if (p > units) p = units;
        const double cost = double((units + p - 1) / p) + 1.0;
        if (cost < best) best_s = TcSchedule{1, int(p), 1, 0, false};
    }
    return best_s;
}

template <bool DUMP>
static w4a4_status dispatch_tc(const uint8_t* ws, const uint8_t* packed, const uint16_t* colscale,
                               const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, int32_t* P, bool sk_room,
                               int silu_I, cudaStream_t s) {
    const TcSchedule sc = tc_schedule(M, N, K, r, sk_room && tc_stream_k_enabled());
    if (sc.sk_ctas > 0) {
        if (r > 32)
            return launch_impl<3, false, true, DUMP>(ws, packed, colscale, bias, M, N, K, r, Y, P, 1, s, sc.sk_ctas,
                                                     silu_I);
        return launch_impl<4, false, true, DUMP>(ws, packed, colscale, bias, M, N, K, r, Y, P, 1, s, sc.sk_ctas,
                                                 silu_I);
    }
    if (sc.tail_ks > 1 && sc.tail_inline) {
        // one launch on clusters of two: the full rounds whole, the last round split over K
        const w4a4_status st = launch_impl<3, true, false, DUMP, true>(ws, packed, colscale, bias, M, N, K, r, Y, P, 2,
                                                                       s, 0, silu_I, 0, -1, sc.tail_lo);
        const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
        set_dispatch("gemm_tc tcgen05.f8f6f4 tile=%dx%d groups/job=%d stages=3 tiles=%d: %d whole, last %d "
                     "split-K=2 in the same launch (cluster)%s%s%s", BM, BN, GPJ, tiles, sc.tail_lo, tiles - sc.tail_lo,
                     n_fastest(M, N, K) ? " N-tiles-fastest" : "", silu_I ? " silu(gate)*up" : "",
                     DUMP ? " (partials dump)" : "");
        return st;
    }
    if (sc.tail_ks > 1) {
        // the full rounds, then the last round's tiles split over K in a launch of their own
        w4a4_status st =
            launch_impl<4, false, false, DUMP>(ws, packed, colscale, bias, M, N, K, r, Y, P, 1, s, 0, silu_I, 0, sc.tail_lo);
        if (st != W4A4_OK) return st;
        st = launch_impl<3, true, false, DUMP>(ws, packed, colscale, bias, M, N, K, r, Y, P, sc.tail_ks, s, 0, silu_I,
                                               sc.tail_lo, -1);
        const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
        set_dispatch("gemm_tc tcgen05.f8f6f4 tile=%dx%d groups/job=%d stages=4 tiles=%d: %d round-robin, last %d "
                     "split-K=%d (cluster)%s%s%s", BM, BN, GPJ, tiles, sc.tail_lo, tiles - sc.tail_lo, sc.tail_ks,
                     n_fastest(M, N, K) ? " N-tiles-fastest" : "", silu_I ? " silu(gate)*up" : "",
                     DUMP ? " (partials dump)" : "");
        return st;
    }
    if (sc.ks > 1)
        return launch_impl<3, true, false, DUMP>(ws, packed, colscale, bias, M, N, K, r, Y, P, sc.ks, s, 0, silu_I);
    if (r > 32)
        return launch_impl<3, false, false, DUMP>(ws, packed, colscale, bias, M, N, K, r, Y, P, 1, s, 0, silu_I);
    return launch_impl<4, false, false, DUMP>(ws, packed, colscale, bias, M, N, K, r, Y, P, 1, s, 0, silu_I);
}

w4a4_status launch_gemm_tc(const uint8_t* ws, const uint8_t* packed, const uint16_t* colscale, const uint16_t* bias,
                           int M, int N, int K, int r, uint16_t* Y, int32_t* P_dump, bool sk_room, int silu_I,
                           cudaStream_t s) {
    // the partials dump runs the schedule the call would run, in its DUMP variant
    if (P_dump) return dispatch_tc<true>(ws, packed, colscale, bias, M, N, K, r, nullptr, P_dump, sk_room, 0, s);
    return dispatch_tc<false>(ws, packed, colscale, bias, M, N, K, r, Y, nullptr, sk_room, silu_I, s);
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
