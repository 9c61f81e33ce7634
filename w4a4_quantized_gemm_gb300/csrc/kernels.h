// Internal launchers shared between the C-ABI layer (api.cu) and the kernel
// translation units.  Arguments are validated by the caller.
#pragma once
#include "common.cuh"

namespace w4a4 {

// api.cu: every check of w4a4_linear except those on the activation workspace
// (null and misaligned pointers, shapes, packed_bytes, the current device)
w4a4_status linear_checks_no_ws(const void* packed, size_t packed_bytes, const uint16_t* colscale,
                                const uint16_t* bias, int M, int N, int K, int r, const void* out);

// pack.cu
// silu_I > 0: W is a fused gate|up weight (I gate rows, then I up rows), packed in gate_up_row order
void launch_pack_weights(const float* W, const int8_t* codes, const uint16_t* scales, int N, int K, int r,
                         int silu_I, uint8_t* packed, cudaStream_t s);
// asymmetric group-128 weights; synchronises s; W4A4_ERR_INVALID_ARG when a zero point leaves [-1024, 1023]
w4a4_status launch_pack_weights_asym(const float* W, int N, int K, int r, uint8_t* packed, cudaStream_t s);
void launch_pack_lora(const uint16_t* L_down, const uint16_t* L_up, int N, int K, int r, int silu_I,
                      uint8_t* packed, cudaStream_t s);
void launch_unpack_weights(const uint8_t* packed, int N, int K, int r, int8_t* codes, uint16_t* scales,
                           uint16_t* L_down, uint16_t* L_up, cudaStream_t s);

// quantize.cu
w4a4_status launch_quantize_act(const uint16_t* X, const uint8_t* packed, int M, int K, int r,
                                uint8_t* ws, cudaStream_t s);
void launch_unpack_act(const uint8_t* ws, int M, int K, int r, int8_t* codes, float* sA, float* SA,
                       float* lora, cudaStream_t s);

// gemm_smallm.cu (warp-level MMA, split over K)
w4a4_status launch_gemm_smallm(const uint8_t* ws, const uint8_t* packed, const uint16_t* colscale,
                               const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y,
                               int32_t* P_dump, cudaStream_t s);

// gemm_tc.cu (tcgen05 + TMEM)
// sk_room: the workspace holds the stream-K hand-over area (act_layout().full bytes)
// silu_I > 0: weights packed by w4a4_pack_weights_gate_up; Y receives silu(gate) * up [M, silu_I]
// P_dump != nullptr: the same schedule also writes the exact per-group partials
// (Y == nullptr: no output; colscale and bias are then not read)
w4a4_status launch_gemm_tc(const uint8_t* ws, const uint8_t* packed, const uint16_t* colscale,
                           const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, int32_t* P_dump,
                           bool sk_room, int silu_I, cudaStream_t s);

// rmsnorm.cu (stack glue between linears)
w4a4_status launch_quantize_act_rmsnorm(const uint16_t* Y, int ld_y, const uint8_t* packed, int M, int K, int r,
                                        uint8_t* ws, cudaStream_t s);
// gemm_smallm_tc.cu (tcgen05, weights as the 128-row operand); P_dump != nullptr also
// writes the exact per-group partials (Y == nullptr: no output)
w4a4_status launch_gemm_smallm_tc(const uint8_t* ws, const uint8_t* packed, const uint16_t* colscale,
                                  const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, int32_t* P_dump,
                                  int silu_I, cudaStream_t s);
// linear_fused.cu (the whole linear for small M in one kernel): ws may be nullptr
// (else it also receives codes, (sA, SA) and lora_act); P_dump != nullptr: the
// partials variant (no Y)
bool fused_eligible(int M, int N, int K, int r);
w4a4_status launch_linear_fused(const uint16_t* X, const uint8_t* packed, const uint16_t* colscale,
                                const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, uint8_t* ws,
                                int32_t* P_dump, cudaStream_t s);
w4a4_status launch_gemm_w4a16(const uint16_t* X, const uint8_t* packed, const uint16_t* colscale,
                              const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, bool asym,
                              cudaStream_t s);
// svd_lora.cu (LoRA from the quantisation error; synchronous)
size_t svd_scratch_bytes(int N, int K, int r);
w4a4_status run_truncated_svd(const float* A, int N, int K, int r, int power, unsigned long long seed, float* U,
                              float* S, float* V, uint8_t* scratch, cudaStream_t st);
w4a4_status run_svd_lora(const float* W, int N, int K, int r, int rounds, int power, unsigned long long seed,
                         uint8_t* packed, uint16_t* L_down, uint16_t* L_up, float* errs, uint8_t* scratch,
                         cudaStream_t st);
void launch_rmsnorm_f16(const uint16_t* Y, int M, int ld_y, int K, double eps, uint16_t* X, cudaStream_t s);

}  // namespace w4a4
