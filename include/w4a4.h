/*
 * w4a4.h -- C ABI of the GB300 (sm_103a) W4A4 + LoRA quantized linear layer.
 *
 *   Y = colscale (.) ( sum_g sA[m,g] sW[n,g] (qA . qW)_g + (X L_down) L_up ) + bias
 *
 * Sources (page title, section):
 *   [VC]  "W4A4 CUDA Kernel for Voice Clone: From Profiling to 2.6x Faster Than
 *         FP16": 2.1-2.3 (INT4 weights, fp16 per-group-64 scales, LoRA factors),
 *         3.4 (the three kernels of one linear), 3.6 (fused quantize + LoRA down),
 *         3.7 (INT4 GEMM + per-group dequant + LoRA up), 3.10 (weights repacked once
 *         at load).
 *   [INT4] "INT4 Kernel Architecture, in depth": "How the weights are stored"
 *         (nibble packing, reordering for the kernel), "Failure modes" (no silent
 *         fallback; log the kernel chosen), "One token versus a thousand" (shape
 *         dispatch, split-K).
 *   [BW]  "High-Performance Kernel Design for W4A4 Quantized Matrix Multiplication
 *         on Blackwell Architecture", section 1 (scaled low-bit GEMM + low-rank
 *         residual + column-wise affine).
 *
 * Conventions for every entry point
 *   - All data pointers are DEVICE pointers of the current CUDA device, owned by
 *     the caller.  No entry point allocates or frees device memory.  The
 *     library's only device memory of its own is the fixed array that
 *     w4a4_linear_noalloc uses as its workspace (a __device__ variable, part
 *     of the loaded module); besides it, the library keeps a per-device
 *     property cache and the text of the last dispatch decision.
 *   - fp16 tensors are passed as uint16_t bit patterns (IEEE binary16).
 *   - Work is enqueued on `stream` (may be 0); nothing synchronises unless the
 *     function says so.  Argument checks happen on the host before any launch,
 *     and a rejected call launches nothing.
 *   - Every pointer must be 16-byte aligned; shapes must satisfy
 *     K % 64 == 0, K >= 64, N % 16 == 0, N >= 16, r % 16 == 0, 0 <= r <= 128,
 *     M >= 0 (M == 0 is a no-op that returns W4A4_OK).  Anything else returns
 *     an error status: there is no fallback path.
 *   - After each launch, a CUDA launch error is reported as W4A4_ERR_CUDA.
 *
 * Packed weight buffer (layout version W4A4_LAYOUT_VERSION), G = K/64 groups:
 *   offset 0                         Ld   L_down in tensor-core fragment order:
 *       [K/16][r/8][32 lanes][2 x 32-bit], lane L's word w holds the fp16 pair
 *       L_down[16 s + 2 (L % 4) + 8 w + {0,1}][8 t + L / 4] for k-step s, tile t.
 *   offset align256(K*r*2)           qW   [G][N][32 bytes]
 *       One 32-byte record per (group g, output row n) holding the 64 codes
 *       as nibbles in OFFSET-BINARY form (nibble = code + 8, 0..15).  Within a
 *       record, the 32-bit little-endian word at byte 8*q + 4*h (q = 0..3,
 *       h = 0..1) holds, in nibble j (bits 4j..4j+3), the code of
 *           k = 64 g + 32 h + (j < 4 ? 4 q + j : 16 + 4 q + (j - 4)).
 *   next align256                    sW   [G][N] fp16 group scales
 *   next align256                    Lu   L_up as [r/16][N][32 bytes]: row n of
 *       plane p holds L_up[16 p .. 16 p + 15][n] (fp16), its two 16-byte halves
 *       swapped when (n >> 2) & 1 (the 32-byte shared-memory swizzle).
 *   total = w4a4_packed_weights_bytes(N, K, r)
 *
 * Activation workspace (written by w4a4_quantize_act, read by w4a4_linear),
 * MT = ceil(M / 128) tiles of 128 rows:
 *   offset 0                 qA  [MT][G][2][128][32 bytes]: the code of row m,
 *       column k is stored as an FP8 E4M3 byte (every integer in [-8, 7] is exact
 *       in E4M3) in plane (k % 64) / 32, row m % 128, byte k % 32, with the two
 *       16-byte halves of a row swapped when ((m % 128) >> 2) & 1.  Code 0 is
 *       E4M3 zero of either sign (0x00, or 0x80 where x / sA rounds to -0).
 *   next align256            sS  [MT][G][128][2] fp32: (sA, SA) per row and group,
 *       SA = sum of the group's 64 codes (exact integer in fp32).
 *   next align256            La  [MT][r/16][128][32 bytes]: lora_act = X L_down
 *       rounded to fp16, row m, column j in plane j/16, same 32-byte swizzle.
 *   next align256            flags [160][16] uint32: stream-K ready flags of the
 *       tcgen05 GEMM, cleared by w4a4_quantize_act, left cleared by w4a4_linear.
 *   next align256            (M >= 33 only, optional) stream-K hand-over area,
 *       [160 CTAs][16 warps][8][32][4] fp32: partial sums of output tiles that
 *       the GEMM splits between CTAs; written and read by w4a4_linear.
 *   Rows >= roundup(M, 16) of the workspace are never written and never
 *   influence Y.  w4a4_act_workspace_min_bytes(M, K, r) is the size up to and
 *   including the flags (what every call needs); w4a4_act_workspace_bytes adds
 *   the hand-over area.  A workspace without it runs the GEMM on its other
 *   schedules.  Because w4a4_linear writes the flags and the hand-over area,
 *   two calls that may overlap on the GPU must not share a workspace.
 */
#ifndef W4A4_H_
#define W4A4_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W4A4_GROUP 64
#define W4A4_LAYOUT_VERSION 1
#define W4A4_MAX_RANK 128

typedef enum {
    W4A4_OK = 0,
    W4A4_ERR_INVALID_ARG = 1,      /* null pointer where data is needed, negative size */
    W4A4_ERR_UNSUPPORTED_SHAPE = 2,/* K % 64, N % 16, r % 16 or r > 128 violated */
    W4A4_ERR_MISALIGNED = 3,       /* a pointer is not 16-byte aligned */
    W4A4_ERR_WORKSPACE = 4,        /* a buffer size is below the size query's result */
    W4A4_ERR_CUDA = 5,             /* the CUDA runtime reported an error */
    W4A4_ERR_TIMEOUT = 6,          /* a bounded device-side wait gave up */
    W4A4_ERR_NO_DEVICE = 7         /* no usable sm_103 device is current */
} w4a4_status;

/* Kernel selection for w4a4_linear_select / w4a4_debug_group_partials. */
typedef enum {
    W4A4_KERNEL_AUTO = 0,   /* by M: M <= threshold the tcgen05 small-M kernel, else tensor-core tiles */
    W4A4_KERNEL_TC = 1,     /* tcgen05 (TMEM accumulators, bulk-copy pipeline) */
    W4A4_KERNEL_SMALLM = 2, /* weight-streaming kernel (warp-level MMA, split over K) */
    W4A4_KERNEL_SMALLM_TC = 3, /* weight-streaming kernel on tcgen05 (weights as the 128-row operand, tokens
                                  as N; split over K) */
    W4A4_KERNEL_FUSED = 4   /* w4a4_forward only: the whole linear in one kernel for small M (see there) */
} w4a4_kernel;

/* ---- size queries (bytes of caller-allocated device buffers) ---- */
size_t w4a4_packed_weights_bytes(int N, int K, int r);
size_t w4a4_act_workspace_bytes(int M, int K, int r);
size_t w4a4_act_workspace_min_bytes(int M, int K, int r);

/* ---- offline weight packing ([VC] 2.1-2.3, 3.10; [INT4] "How the weights are stored")
 * W      fp32 [N, K] row-major (nn.Linear out x in).
 * L_down fp16 [K, r] row-major, L_up fp16 [r, N] row-major (both NULL when r == 0).
 * Quantises each (row n, group g): sW = fp16(max(absmax/7, 2^-14)) with IEEE
 * division and round-to-nearest-even, qW = clamp(rint(W / sW), -8, 7); writes
 * the packed buffer described above.  Runs once per layer; enqueued on stream. */
w4a4_status w4a4_pack_weights(const float* W, const uint16_t* L_down, const uint16_t* L_up,
                              int N, int K, int r, void* packed, size_t packed_bytes,
                              cudaStream_t stream);

/* Same, from given integer codes int8 [N, K] (values must lie in [-8, 7]) and
 * fp16 scales [N, K/64]: lets callers bring codes of their own quantiser. */
w4a4_status w4a4_pack_weight_codes(const int8_t* codes, const uint16_t* scales,
                                   const uint16_t* L_down, const uint16_t* L_up,
                                   int N, int K, int r, void* packed, size_t packed_bytes,
                                   cudaStream_t stream);

/* ---- fused activation quantisation + LoRA down ([VC] 3.6)
 * X fp16 [M, K] row-major.  Per (row m, group g): sA = max(absmax/7, 1e-10)
 * (fp32, IEEE division), qA = clamp(rint(X / sA), -8, 7), SA = sum of codes;
 * in the same pass lora_act[m, :] = X[m, :] L_down (fp16 inputs, fp32
 * accumulation, deterministic order), stored as fp16.  L_down is read from the
 * packed weight buffer (its first K * r * 2 bytes; packed may be NULL when
 * r == 0); packed_bytes is that buffer's size, and a size below K * r * 2
 * returns W4A4_ERR_WORKSPACE before any launch.  Writes the activation
 * workspace (act_ws_bytes >= w4a4_act_workspace_min_bytes(M, K, r)). */
w4a4_status w4a4_quantize_act(const uint16_t* X, const void* packed, size_t packed_bytes, int M, int K, int r,
                              void* act_ws, size_t act_ws_bytes, cudaStream_t stream);

/* ---- W4A4 GEMM + LoRA up + column affine ([VC] 3.7, [BW] 1)
 * acc[m,n] = sum_g sA[m,g] sW[n,g] P[m,n,g] + sum_j fp16(lora_act[m,j]) L_up[j,n]
 * in fp32, P exact per group; Y[m,n] = fp16_rn(colscale[n] * acc + bias[n]).
 * colscale fp16 [N]; bias fp16 [N] or NULL (zero); Y fp16 [M, N] row-major.
 * The kernel is chosen by M (see w4a4_last_dispatch). */
w4a4_status w4a4_linear(const void* act_ws, size_t act_ws_bytes, const void* packed,
                        size_t packed_bytes, const uint16_t* colscale, const uint16_t* bias,
                        int M, int N, int K, int r, uint16_t* Y, cudaStream_t stream);

/* ---- the whole linear from fp16 activations ([VC] 3.6-3.7; [INT4] "One token
 * versus a thousand": at decode sizes the call is a weight stream)
 * Y = the layer of w4a4_linear applied to X fp16 [M, K] row-major, i.e.
 * w4a4_quantize_act followed by w4a4_linear, in one call.  Arguments as for
 * those two; X must be 16-byte aligned.
 * kernel W4A4_KERNEL_AUTO: for 1 <= M <= 8 and the shapes the fused kernel takes
 * (M <= 32; r <= 32; K / 64 groups split over at most 8 CTAs with at most 8
 * groups each, i.e. K <= 4096 at N >= 1024; the shared-memory plan fits two CTAs
 * per SM), one kernel does everything: quantisation and LoRA down
 * of X (the same codes, scales and SA as w4a4_quantize_act, bit for bit; the
 * LoRA-down sums in another fixed order, so lora_act may differ in its last
 * fp16 bit), the exact per-group products, LoRA up and the affine.  act_ws may
 * then be NULL; if it is given (act_ws_bytes >= w4a4_act_workspace_min_bytes),
 * the kernel also writes the codes, (sA, SA) pairs and lora_act there in the
 * workspace layout.  Otherwise the call runs w4a4_quantize_act and w4a4_linear
 * on act_ws, which is then required.
 * (Above M = 8 the two-call path is faster: each 128-row weight tile repeats the
 * quantisation and LoRA down of the X slice it reads.)
 * kernel W4A4_KERNEL_FUSED: the fused kernel (M <= 32), W4A4_ERR_UNSUPPORTED_SHAPE
 * where it does not apply.  TC, SMALLM, SMALLM_TC: the two-call path with that GEMM.
 * Every argument check runs before anything is launched. */
w4a4_status w4a4_forward(const uint16_t* X, const void* packed, size_t packed_bytes, const uint16_t* colscale,
                         const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, void* act_ws,
                         size_t act_ws_bytes, int kernel, cudaStream_t stream);
/* Whether w4a4_forward's AUTO choice for these sizes is the fused kernel. */
int w4a4_forward_is_fused(int M, int N, int K, int r);

/* ---- fused gate|up linear with the SiLU(gate) * up epilogue ([VC] 1: the
 * decoder MLP's SiLU(gate_proj x) * up_proj x feeding down_proj).
 * w4a4_pack_weights_gate_up packs W fp32 [N, K] whose rows 0..N/2-1 are the
 * gate rows and N/2..N-1 the up rows (N % 32 == 0), like w4a4_pack_weights but
 * with the rows (and the columns of L_up [r, N]) in the order the epilogue
 * pairs them: packed row p of 128-row tile t = p / 128, 32-row slice
 * s = (p % 128) / 32, w = p % 32 holds original row j = 64 t + 16 s + w % 16
 * for w < 16 (a gate) and N/2 + j otherwise (its up).  Same buffer size; the
 * debug unpack returns the rows in that packed order.
 * w4a4_linear_silu_mul computes, with acc as in w4a4_linear (original row
 * indices for colscale and bias, fp16 [N]):
 *   g = colscale[j] acc[m, j] + bias[j],  u = colscale[N/2+j] acc[m, N/2+j] + bias[N/2+j]
 *   H[m, j] = fp16_rn( g / (1 + exp(-g)) * u ),  H fp16 [M, N/2] row-major,
 * in fp32 from the accumulators (no fp16 rounding of g and u).  It runs the
 * tcgen05 tile kernel for every M.  Workspace as for w4a4_linear. */
w4a4_status w4a4_pack_weights_gate_up(const float* W, const uint16_t* L_down, const uint16_t* L_up, int N, int K,
                                      int r, void* packed, size_t packed_bytes, cudaStream_t stream);
w4a4_status w4a4_linear_silu_mul(const void* act_ws, size_t act_ws_bytes, const void* packed, size_t packed_bytes,
                                 const uint16_t* colscale, const uint16_t* bias, int M, int N, int K, int r,
                                 uint16_t* H, cudaStream_t stream);

/* ---- LoRA from the quantisation error ([VC] 2.1-2.2; offline, synchronous)
 * w4a4_pack_weights_svd quantises W fp32 [N, K] like w4a4_pack_weights and
 * derives the LoRA factors from the error instead of taking them: in each of
 * `rounds` rounds, W - LoRA_previous (W in the first) is quantised (the
 * packer's round-to-nearest in place of GPTQ), E = W - Q is formed and its
 * rank-r SVD U S V^T taken (randomized subspace iteration with `power_iters`
 * power steps on a block of 64 or 128 columns, start block drawn
 * from `seed`); the rounds stop once the residual ||E - U S V^T||_F stops
 * falling.  The round with the smallest residual is kept: its codes and
 * scales go into `packed` together with L_down = fp16(V) [K, r] and
 * L_up = fp16((U S)^T) [r, N], which are also written to the device buffers
 * L_down, L_up.  errs (host, may be NULL) receives each round's residual
 * (fp32; -1 for rounds not run).  16 <= r <= 128; scratch: device memory of
 * w4a4_svd_lora_scratch_bytes(N, K, r) bytes.  16 power steps give the
 * residual within ~1e-4 of the exact truncated SVD's on quantisation errors.
 * w4a4_truncated_svd exposes the rank-r SVD alone: A fp32 [N, K] -> U [N, r],
 * S [r], V [K, r] (fp32, device), with the same scratch. */
size_t w4a4_svd_lora_scratch_bytes(int N, int K, int r);
w4a4_status w4a4_pack_weights_svd(const float* W, int N, int K, int r, int rounds, int power_iters,
                                  unsigned long long seed, void* packed, size_t packed_bytes, uint16_t* L_down,
                                  uint16_t* L_up, float* errs, void* scratch, size_t scratch_bytes,
                                  cudaStream_t stream);
w4a4_status w4a4_truncated_svd(const float* A, int N, int K, int r, int power_iters, unsigned long long seed,
                               float* U, float* S, float* V, void* scratch, size_t scratch_bytes,
                               cudaStream_t stream);

/* Same as w4a4_linear with an explicit kernel choice (tests, measurements). */
w4a4_status w4a4_linear_select(const void* act_ws, size_t act_ws_bytes, const void* packed,
                               size_t packed_bytes, const uint16_t* colscale, const uint16_t* bias,
                               int M, int N, int K, int r, uint16_t* Y, int kernel,
                               cudaStream_t stream);

/* ---- allocation-free variant of the whole layer
 * The pages have no counterpart to this entry point.  It serves callers that
 * cannot allocate device memory (code running inside an allocator, a runtime
 * that owns all memory, a plugin interface that only passes in the inputs and
 * outputs): it runs w4a4_quantize_act and w4a4_linear back to back with the
 * activation workspace in a fixed array of W4A4_NOALLOC_WORKSPACE_BYTES that
 * the library keeps in each device's memory from load until process exit.
 * X fp16 [M, K], packed/colscale/bias/Y as for w4a4_linear.  Every argument
 * check of both steps runs before anything is launched; among them, the call
 * returns W4A4_ERR_WORKSPACE when w4a4_act_workspace_min_bytes(M, K, r) exceeds
 * the array (the GEMM's optional stream-K hand-over area is never used through
 * this entry point).  The first call on a device looks up the array's device
 * address (make that first call before any stream capture).  All calls share
 * the array: calls that overlap on the GPU race.  It allocates and frees
 * nothing. */
#define W4A4_NOALLOC_WORKSPACE_BYTES (8u << 20)
w4a4_status w4a4_linear_noalloc(const uint16_t* X, const void* packed, size_t packed_bytes,
                                const uint16_t* colscale, const uint16_t* bias, int M, int N, int K, int r,
                                uint16_t* Y, cudaStream_t stream);

/* RMSNorm glue of a stack of linears (unit gain), "W4A4 CUDA Kernel for Voice
 * Clone", 3.9 (RMSNorm between the linears of a decoder layer; the page gives no
 * epsilon, W4A4_RMSNORM_EPS is the Qwen3 value).  For each row m < M of Y
 * (fp16, row stride ld_y elements) it reads the first K columns and writes
 *   X[m, k] = fp16( Y[m, k] / sqrt( sum_k Y[m, k]^2 / K + eps ) )
 * into X (fp16 [M, K], row-major).  Squares are exact in fp32 and summed in
 * fp64; 1/sqrt(mean + eps) is taken in fp64 and each product y * inv is rounded
 * once, fp64 -> fp16, to nearest even, so the result is the same bits as any
 * implementation of this arithmetic up to the order of the fp64 additions.
 * K % 8 == 0, 8 <= K <= 16384, ld_y >= K, ld_y % 8 == 0, 16-byte aligned pointers;
 * Y and X must not overlap.  M == 0 is a no-op. */
#define W4A4_RMSNORM_EPS 1e-6
w4a4_status w4a4_rmsnorm_f16(const uint16_t* Y, int M, int ld_y, int K, uint16_t* X, cudaStream_t stream);

/* The glue and the next linear's activation step in one kernel: for each row
 * m < M of Y (fp16, row stride ld_y elements), the first K columns are
 * normalised exactly as w4a4_rmsnorm_f16 would write them (the same fp16
 * bits) and then quantised and LoRA-down-projected exactly as
 * w4a4_quantize_act would on those values.  The normalised fp16 values are
 * not written out.  Arguments and limits as for w4a4_quantize_act (with X
 * replaced by Y), plus ld_y >= K and ld_y % 8 == 0. */
w4a4_status w4a4_quantize_act_rmsnorm(const uint16_t* Y, int ld_y, const void* packed, size_t packed_bytes, int M,
                                      int K, int r, void* act_ws, size_t act_ws_bytes, cudaStream_t stream);

/* ---- W4A16 linear ([INT4] "W4A16 versus W4A4": fp16 activations, the
 * weights dequantised in registers), for the decode regime.  Same packed
 * weights, LoRA and affine as w4a4_linear, no activation quantisation:
 *   Y[m,n] = fp16_rn( colscale[n] * ( sum_g sW[n,g] sum_{k in g} X[m,k] c[n,k]
 *                                     + (X L_down)[m,:] . L_up[:,n] ) + bias[n] )
 * with the products accumulated in fp32.  X fp16 [M, K] row-major (16-byte
 * aligned); no workspace.  Any M >= 0 is accepted (the kernel streams the
 * weights once per block of up to 64 rows, so it is meant for small M). */
w4a4_status w4a16_linear(const uint16_t* X, const void* packed, size_t packed_bytes, const uint16_t* colscale,
                         const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, cudaStream_t stream);

/* ---- asymmetric group-128 weights ([INT4] "How the weights are stored": one
 * fp16 scale and one zero point per group of 128 input channels, codes 0..15,
 * value (q - zero) * scale).  K % 128 == 0.  Per row n and group g, in IEEE
 * binary32 (round to nearest even):
 *   scale = max(max w - min w, 1e-8) / 15;  zero = rint(-min w / scale) (+0 if 0);
 *   q = clamp(rint(w / scale + zero), 0, 15);
 * stored: fp16(scale), fp16(zero).  Same buffer size and sections as
 * w4a4_pack_weights (packed_weights_bytes): the codes as plain nibbles q in
 * the same record layout, the scale plane holding fp16(scale) in the slot of
 * the group's first 64 channels and fp16(zero) in the slot of its second
 * (w4a4_debug_unpack_weights then returns q - 8 and those two columns).  The
 * buffer is read by w4a16_linear_asym only.  Synchronises `stream`; returns
 * W4A4_ERR_INVALID_ARG, with the buffer written, when a zero point lies
 * outside [-1024, 1023] (groups far from zero relative to their range). */
w4a4_status w4a16_pack_weights_asym(const float* W, const uint16_t* L_down, const uint16_t* L_up, int N, int K,
                                    int r, void* packed, size_t packed_bytes, cudaStream_t stream);
/* W4A16 linear on those weights:
 *   Y[m,n] = fp16_rn( colscale[n] * ( sum_k X[m,k] (q[n,k] - zero[n,g]) scale[n,g]
 *                                     + (X L_down)[m,:] . L_up[:,n] ) + bias[n] )
 * with the products accumulated in fp32; arguments as for w4a16_linear. */
w4a4_status w4a16_linear_asym(const uint16_t* X, const void* packed, size_t packed_bytes, const uint16_t* colscale,
                              const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, cudaStream_t stream);

/* ---- debug / validation entry points (small shapes; they synchronise `stream`)
 * Unpack the packed weights: codes int8 [N, K], scales fp16 [N, K/64],
 * L_down fp16 [K, r], L_up fp16 [r, N] (the last two may be NULL). */
w4a4_status w4a4_debug_unpack_weights(const void* packed, int N, int K, int r, int8_t* codes,
                                      uint16_t* scales, uint16_t* L_down, uint16_t* L_up,
                                      cudaStream_t stream);
/* Unpack the workspace: codes int8 [M, K], sA fp32 [M, K/64], SA fp32 [M, K/64]
 * (may be NULL), lora_act fp32 [M, r] (may be NULL). */
w4a4_status w4a4_debug_unpack_act(const void* act_ws, int M, int K, int r, int8_t* codes,
                                  float* sA, float* SA, float* lora_act, cudaStream_t stream);
/* Exact per-group partial sums P[m, n, g] (int32 [M, N, K/64]) as produced by
 * the GEMM that w4a4_linear_select(..., kernel) would run on the same
 * arguments: the same kernel instantiation and the same schedule (split-K
 * clusters, stream-K when it is on and act_ws_bytes holds the hand-over area),
 * with its epilogue also writing each group's integer product before scaling.
 * No Y is written, and colscale and bias are not needed.  Argument checks as
 * for w4a4_linear. */
w4a4_status w4a4_debug_group_partials(const void* act_ws, size_t act_ws_bytes, const void* packed,
                                      size_t packed_bytes, int M, int N, int K, int r, int kernel, int32_t* P,
                                      cudaStream_t stream);
/* The same partials from the fused kernel of w4a4_forward (kernel
 * W4A4_KERNEL_FUSED) on X fp16 [M, K]: no Y is written.  act_ws may be NULL or
 * receive the codes, scales and lora_act as in w4a4_forward.
 * W4A4_ERR_UNSUPPORTED_SHAPE where the fused kernel does not apply. */
w4a4_status w4a4_debug_forward_partials(const uint16_t* X, const void* packed, size_t packed_bytes, int M, int N,
                                        int K, int r, void* act_ws, size_t act_ws_bytes, int32_t* P,
                                        cudaStream_t stream);
/* Reads and clears the device status word written by bounded waits
 * (W4A4_OK or W4A4_ERR_TIMEOUT); synchronises the device. */
w4a4_status w4a4_device_status(void);

/* ---- dispatch and diagnostics ([INT4] "Failure modes": log the kernel chosen) */
const char* w4a4_status_string(int status);
const char* w4a4_last_dispatch(void);       /* kernel and launch shape of this thread's last call */
int w4a4_small_m_threshold(void);
/* Whether the tcgen05 GEMM may split tiles between CTAs (stream-K schedule,
 * used when the workspace holds the hand-over area and the schedule's cost
 * model favours it).  Off by default (measured slower than the round-robin and
 * split-K schedules on the decoder-layer shapes); W4A4_STREAM_K=1 turns it on
 * at load. */
int w4a4_stream_k(void);
void w4a4_set_stream_k(int on);
/* AUTO dispatch: M <= threshold -> the small-M kernel, else the tcgen05 tiles.
 * Default 32, or W4A4_SMALL_M at the first query; a negative value means 0
 * (the tiles for every M). */
void w4a4_set_small_m_threshold(int m);
int w4a4_layout_version(void);

#ifdef __cplusplus
}
#endif
#endif /* W4A4_H_ */
