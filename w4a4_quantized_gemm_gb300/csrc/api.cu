// C ABI of the W4A4 library: host-side argument checks (before any launch),
// kernel dispatch by M, status mapping and the dispatch log ("INT4 Kernel
// Architecture, in depth", "Failure modes": no silent fallback, log which
// kernel each layer uses).
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "kernels.h"

namespace w4a4 {

namespace {
thread_local char t_dispatch[256] = "none";
int g_small_m_threshold = -1;  // -1: read W4A4_SMALL_M on first use
constexpr int kStreamKDefault = 0;  // stream-K measured slower than split-K / round-robin on every layer shape
constexpr int kDefaultSmallM = 32;  // M <= this -> weight-streaming kernel, else tcgen05 tiles (measured crossover: 32..48)
std::mutex g_mu;
int g_sm_count[64] = {0};

bool log_enabled() {
    static int on = -1;
    if (on < 0) {
        const char* e = std::getenv("W4A4_LOG");
        on = (e && e[0] && e[0] != '0') ? 1 : 0;
    }
    return on == 1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

w4a4_status check_kn(int N, int K, int r) {
    if (N < 0 || K < 0 || r < 0) return W4A4_ERR_INVALID_ARG;
    if (K < kGroup || K % kGroup != 0) return W4A4_ERR_UNSUPPORTED_SHAPE;
    if (N < 16 || N % 16 != 0) return W4A4_ERR_UNSUPPORTED_SHAPE;
    if (r % 16 != 0 || r > W4A4_MAX_RANK) return W4A4_ERR_UNSUPPORTED_SHAPE;
    return W4A4_OK;
}

w4a4_status check_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_NO_DEVICE;
    }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return W4A4_ERR_NO_DEVICE;  // built for sm_103a only
    return W4A4_OK;
}

w4a4_status sync_status(cudaStream_t s) {
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    return W4A4_OK;
}
// Reads and clears the status words of every kernel with bounded waits.
w4a4_status device_status_words() {
    const w4a4_status a = tc_read_and_clear_status();
    const w4a4_status b = smallm_read_and_clear_status();
    const w4a4_status c = w4a16_read_and_clear_status();
    const w4a4_status d = smtc_read_and_clear_status();
    const w4a4_status e = q_read_and_clear_status();
    const w4a4_status f = fused_read_and_clear_status();
    return a != W4A4_OK ? a : b != W4A4_OK ? b : c != W4A4_OK ? c : d != W4A4_OK ? d : e != W4A4_OK ? e : f;
}
}  // namespace

void set_dispatch(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_dispatch, sizeof(t_dispatch), fmt, ap);
    va_end(ap);
    if (log_enabled()) std::fprintf(stderr, "[w4a4] %s\n", t_dispatch);
}

w4a4_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? W4A4_OK : W4A4_ERR_CUDA;
}

unsigned add_pdl_attr(cudaLaunchAttribute* attrs, unsigned n) {
    static const bool on = [] {
        const char* e = std::getenv("W4A4_PDL");
        return !(e && e[0] == '0');
    }();
    if (!on) return n;
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    return n + 1;
}

// Stream-K schedule of the tcgen05 GEMM: W4A4_STREAM_K=1 / 0 sets the initial
// state, w4a4_set_stream_k changes it.
static std::atomic<int> g_stream_k{-1};
bool tc_stream_k_enabled() {
    int v = g_stream_k.load();
    if (v < 0) {
        const char* e = std::getenv("W4A4_STREAM_K");
        v = (e && e[0] == '1') ? 1 : (e && e[0] == '0') ? 0 : kStreamKDefault;
        g_stream_k.store(v);
    }
    return v != 0;
}

int device_sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = n > 0 ? n : 148;
    }
    return g_sm_count[dev];
}

// The checks of w4a4_linear on everything but the activation workspace.
w4a4_status linear_checks_no_ws(const void* packed, size_t packed_bytes, const uint16_t* colscale,
                                const uint16_t* bias, int M, int N, int K, int r, const void* out) {
    if (M < 0) return W4A4_ERR_INVALID_ARG;
    w4a4_status st = check_kn(N, K, r);
    if (st != W4A4_OK) return st;
    if (M == 0) return W4A4_OK;
    if (!packed || !colscale || !out) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(colscale) || (bias && !aligned16(bias)) || !aligned16(out))
        return W4A4_ERR_MISALIGNED;
    if (packed_bytes < packed_layout(N, K, r).total) return W4A4_ERR_WORKSPACE;
    return check_device();
}

}  // namespace w4a4

using namespace w4a4;

extern "C" {

size_t w4a4_packed_weights_bytes(int N, int K, int r) {
    if (check_kn(N, K, r) != W4A4_OK) return 0;
    return packed_layout(N, K, r).total;
}

size_t w4a4_act_workspace_bytes(int M, int K, int r) {
    if (M < 0 || check_kn(16, K, r) != W4A4_OK) return 0;
    return act_layout(M, K, r).full;
}

size_t w4a4_act_workspace_min_bytes(int M, int K, int r) {
    if (M < 0 || check_kn(16, K, r) != W4A4_OK) return 0;
    return act_layout(M, K, r).total;
}

int w4a4_layout_version(void) { return W4A4_LAYOUT_VERSION; }

const char* w4a4_status_string(int status) {
    switch (status) {
        case W4A4_OK: return "ok";
        case W4A4_ERR_INVALID_ARG: return "invalid argument";
        case W4A4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (need K%64==0, N%16==0, r%16==0, r<=128)";
        case W4A4_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case W4A4_ERR_WORKSPACE: return "buffer smaller than the size query";
        case W4A4_ERR_CUDA: return "CUDA runtime error";
        case W4A4_ERR_TIMEOUT: return "bounded device wait timed out";
        case W4A4_ERR_NO_DEVICE: return "no sm_103 device is current";
        default: return "unknown status";
    }
}

const char* w4a4_last_dispatch(void) { return t_dispatch; }

int w4a4_small_m_threshold(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_small_m_threshold < 0) {
        const char* e = std::getenv("W4A4_SMALL_M");
        const int v = e ? std::atoi(e) : kDefaultSmallM;
        g_small_m_threshold = v < 0 ? 0 : v;
    }
    return g_small_m_threshold;
}

void w4a4_set_small_m_threshold(int m) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_small_m_threshold = m < 0 ? 0 : m;
}

int w4a4_stream_k(void) { return tc_stream_k_enabled() ? 1 : 0; }

void w4a4_set_stream_k(int on) { g_stream_k.store(on ? 1 : 0); }

static w4a4_status pack_common(const float* W, const int8_t* codes, const uint16_t* scales, const uint16_t* L_down,
                               const uint16_t* L_up, int N, int K, int r, void* packed, size_t packed_bytes,
                               cudaStream_t stream, int silu_I = 0) {
    w4a4_status st = check_kn(N, K, r);
    if (st != W4A4_OK) return st;
    if (!packed || (!W && !(codes && scales))) return W4A4_ERR_INVALID_ARG;
    if (r > 0 && (!L_down || !L_up)) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(packed) || (W && !aligned16(W)) || (L_down && !aligned16(L_down)) || (L_up && !aligned16(L_up)))
        return W4A4_ERR_MISALIGNED;
    if (packed_bytes < packed_layout(N, K, r).total) return W4A4_ERR_WORKSPACE;
    if ((st = check_device()) != W4A4_OK) return st;
    uint8_t* out = static_cast<uint8_t*>(packed);
    launch_pack_weights(W, codes, scales, N, K, r, silu_I, out, stream);
    if ((st = launch_status()) != W4A4_OK) return st;
    launch_pack_lora(L_down, L_up, N, K, r, silu_I, out, stream);
    set_dispatch("pack_weights%s N=%d K=%d r=%d", silu_I ? " (gate|up order)" : "", N, K, r);
    return launch_status();
}

w4a4_status w4a4_pack_weights(const float* W, const uint16_t* L_down, const uint16_t* L_up, int N, int K, int r,
                              void* packed, size_t packed_bytes, cudaStream_t stream) {
    if (!W) return W4A4_ERR_INVALID_ARG;
    return pack_common(W, nullptr, nullptr, L_down, L_up, N, K, r, packed, packed_bytes, stream);
}

w4a4_status w4a4_pack_weights_gate_up(const float* W, const uint16_t* L_down, const uint16_t* L_up, int N, int K,
                                      int r, void* packed, size_t packed_bytes, cudaStream_t stream) {
    if (!W) return W4A4_ERR_INVALID_ARG;
    if (N % 32 != 0) return W4A4_ERR_UNSUPPORTED_SHAPE;
    return pack_common(W, nullptr, nullptr, L_down, L_up, N, K, r, packed, packed_bytes, stream, N / 2);
}

size_t w4a4_svd_lora_scratch_bytes(int N, int K, int r) {
    if (check_kn(N, K, r) != W4A4_OK || r < 16) return 0;
    return svd_scratch_bytes(N, K, r);
}

w4a4_status w4a4_pack_weights_svd(const float* W, int N, int K, int r, int rounds, int power_iters,
                                  unsigned long long seed, void* packed, size_t packed_bytes, uint16_t* L_down,
                                  uint16_t* L_up, float* errs, void* scratch, size_t scratch_bytes,
                                  cudaStream_t stream) {
    w4a4_status st = check_kn(N, K, r);
    if (st != W4A4_OK) return st;
    if (r < 16) return W4A4_ERR_UNSUPPORTED_SHAPE;
    if (rounds < 1 || rounds > 16 || power_iters < 0 || power_iters > 64) return W4A4_ERR_INVALID_ARG;
    if (!W || !packed || !L_down || !L_up || !scratch) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(packed) || !aligned16(L_down) || !aligned16(L_up) || !aligned16(scratch))
        return W4A4_ERR_MISALIGNED;
    if (packed_bytes < packed_layout(N, K, r).total || scratch_bytes < svd_scratch_bytes(N, K, r))
        return W4A4_ERR_WORKSPACE;
    if ((st = check_device()) != W4A4_OK) return st;
    set_dispatch("pack_weights_svd N=%d K=%d r=%d rounds=%d power=%d", N, K, r, rounds, power_iters);
    return run_svd_lora(W, N, K, r, rounds, power_iters, seed, static_cast<uint8_t*>(packed), L_down, L_up, errs,
                        static_cast<uint8_t*>(scratch), stream);
}

w4a4_status w4a4_truncated_svd(const float* A, int N, int K, int r, int power_iters, unsigned long long seed,
                               float* U, float* S, float* V, void* scratch, size_t scratch_bytes,
                               cudaStream_t stream) {
    w4a4_status st = check_kn(N, K, r);
    if (st != W4A4_OK) return st;
    if (r < 16) return W4A4_ERR_UNSUPPORTED_SHAPE;
    if (power_iters < 0 || power_iters > 64) return W4A4_ERR_INVALID_ARG;
    if (!A || !U || !S || !V || !scratch) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(U) || !aligned16(V) || !aligned16(scratch)) return W4A4_ERR_MISALIGNED;
    if (scratch_bytes < svd_scratch_bytes(N, K, r)) return W4A4_ERR_WORKSPACE;
    if ((st = check_device()) != W4A4_OK) return st;
    set_dispatch("truncated_svd N=%d K=%d r=%d power=%d", N, K, r, power_iters);
    return run_truncated_svd(A, N, K, r, power_iters, seed, U, S, V, static_cast<uint8_t*>(scratch), stream);
}

w4a4_status w4a4_pack_weight_codes(const int8_t* codes, const uint16_t* scales, const uint16_t* L_down,
                                   const uint16_t* L_up, int N, int K, int r, void* packed, size_t packed_bytes,
                                   cudaStream_t stream) {
    if (!codes || !scales) return W4A4_ERR_INVALID_ARG;
    return pack_common(nullptr, codes, scales, L_down, L_up, N, K, r, packed, packed_bytes, stream);
}

// Bytes of the packed buffer the activation kernel reads: its L_down section.
static size_t ldown_bytes(int K, int r) { return size_t(K) * size_t(r) * 2; }

w4a4_status w4a4_quantize_act(const uint16_t* X, const void* packed, size_t packed_bytes, int M, int K, int r,
                              void* act_ws, size_t act_ws_bytes, cudaStream_t stream) {
    if (M < 0) return W4A4_ERR_INVALID_ARG;
    w4a4_status st = check_kn(16, K, r);
    if (st != W4A4_OK) return st;
    if (M == 0) return W4A4_OK;
    if (!X || !act_ws || (r > 0 && !packed)) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(act_ws) || (packed && !aligned16(packed))) return W4A4_ERR_MISALIGNED;
    if (act_ws_bytes < act_layout(M, K, r).total) return W4A4_ERR_WORKSPACE;
    if (r > 0 && packed_bytes < ldown_bytes(K, r)) return W4A4_ERR_WORKSPACE;
    if ((st = check_device()) != W4A4_OK) return st;
    return launch_quantize_act(X, static_cast<const uint8_t*>(packed), M, K, r, static_cast<uint8_t*>(act_ws),
                               stream);
}

w4a4_status w4a4_quantize_act_rmsnorm(const uint16_t* Y, int ld_y, const void* packed, size_t packed_bytes, int M,
                                      int K, int r, void* act_ws, size_t act_ws_bytes, cudaStream_t stream) {
    if (M < 0 || ld_y < K) return W4A4_ERR_INVALID_ARG;
    w4a4_status st = check_kn(16, K, r);
    if (st != W4A4_OK) return st;
    if (ld_y % 8 != 0) return W4A4_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return W4A4_OK;
    if (!Y || !act_ws || (r > 0 && !packed)) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(Y) || !aligned16(act_ws) || (packed && !aligned16(packed))) return W4A4_ERR_MISALIGNED;
    if (act_ws_bytes < act_layout(M, K, r).total) return W4A4_ERR_WORKSPACE;
    if (r > 0 && packed_bytes < ldown_bytes(K, r)) return W4A4_ERR_WORKSPACE;
    if ((st = check_device()) != W4A4_OK) return st;
    return launch_quantize_act_rmsnorm(Y, ld_y, static_cast<const uint8_t*>(packed), M, K, r,
                                       static_cast<uint8_t*>(act_ws), stream);
}

// AUTO: up to the small-M threshold the tcgen05 weight-streaming kernel (it
// beats the warp-MMA one from M = 1 on), above it the tcgen05 tiles (measured
// crossovers on the decoder-layer and K = N = 4096 shapes).  The partials dump
// goes through the same choice.
static int pick_kernel(int M, int kernel) {
    if (kernel == W4A4_KERNEL_TC || kernel == W4A4_KERNEL_SMALLM || kernel == W4A4_KERNEL_SMALLM_TC) return kernel;
    if (M > w4a4_small_m_threshold()) return W4A4_KERNEL_TC;
    return W4A4_KERNEL_SMALLM_TC;
}


static w4a4_status linear_checks(const void* act_ws, size_t act_ws_bytes, const void* packed, size_t packed_bytes,
                                 const uint16_t* colscale, const uint16_t* bias, int M, int N, int K, int r,
                                 const void* out) {
    if (M < 0) return W4A4_ERR_INVALID_ARG;
    w4a4_status st = check_kn(N, K, r);
    if (st != W4A4_OK) return st;
    if (M == 0) return W4A4_OK;
    if (!act_ws) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(act_ws)) return W4A4_ERR_MISALIGNED;
    if (act_ws_bytes < act_layout(M, K, r).total) return W4A4_ERR_WORKSPACE;
    return linear_checks_no_ws(packed, packed_bytes, colscale, bias, M, N, K, r, out);
}

w4a4_status w4a4_linear_select(const void* act_ws, size_t act_ws_bytes, const void* packed, size_t packed_bytes,
                               const uint16_t* colscale, const uint16_t* bias, int M, int N, int K, int r,
                               uint16_t* Y, int kernel, cudaStream_t stream) {
    if (kernel < W4A4_KERNEL_AUTO || kernel > W4A4_KERNEL_SMALLM_TC) return W4A4_ERR_INVALID_ARG;
    w4a4_status st = linear_checks(act_ws, act_ws_bytes, packed, packed_bytes, colscale, bias, M, N, K, r, Y);
    if (st != W4A4_OK || M == 0) return st;
    const uint8_t* ws = static_cast<const uint8_t*>(act_ws);
    const uint8_t* pk = static_cast<const uint8_t*>(packed);
    const int k = pick_kernel(M, kernel);
    if (k == W4A4_KERNEL_TC) {
        const ActLayout AL = act_layout(M, K, r);
        const bool sk_room = AL.full > AL.total && act_ws_bytes >= AL.full;
        return launch_gemm_tc(ws, pk, colscale, bias, M, N, K, r, Y, nullptr, sk_room, 0, stream);
    }
    if (k == W4A4_KERNEL_SMALLM_TC)
        return launch_gemm_smallm_tc(ws, pk, colscale, bias, M, N, K, r, Y, nullptr, 0, stream);
    return launch_gemm_smallm(ws, pk, colscale, bias, M, N, K, r, Y, nullptr, stream);
}

w4a4_status w4a4_linear(const void* act_ws, size_t act_ws_bytes, const void* packed, size_t packed_bytes,
                        const uint16_t* colscale, const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y,
                        cudaStream_t stream) {
    return w4a4_linear_select(act_ws, act_ws_bytes, packed, packed_bytes, colscale, bias, M, N, K, r, Y,
                              W4A4_KERNEL_AUTO, stream);
}

// AUTO takes the fused kernel up to this M.  Every 128-row weight tile's cluster
// repeats the quantisation and LoRA down of the whole X slice it reads, so that
// work grows with M times the tile count: measured at K = N = 4096, r = 32 (a CUDA
// graph of back-to-back calls), the fused call against quantise + GEMM is
// 9.3 vs 11.0 us at M = 1, 9.6 vs 11.5 at M = 4, 11.5 vs 11.4 at M = 16 and
// 14.9 vs 13.0 at M = 32.
constexpr int kFusedMaxM = 8;

int w4a4_forward_is_fused(int M, int N, int K, int r) {
    if (check_kn(N, K, r) != W4A4_OK || M < 1 || M > kFusedMaxM || M > w4a4_small_m_threshold()) return 0;
    return fused_eligible(M, N, K, r) ? 1 : 0;
}

w4a4_status w4a4_forward(const uint16_t* X, const void* packed, size_t packed_bytes, const uint16_t* colscale,
                         const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, void* act_ws,
                         size_t act_ws_bytes, int kernel, cudaStream_t stream) {
    if (kernel < W4A4_KERNEL_AUTO || kernel > W4A4_KERNEL_FUSED) return W4A4_ERR_INVALID_ARG;
    w4a4_status st = linear_checks_no_ws(packed, packed_bytes, colscale, bias, M, N, K, r, Y);
    if (st != W4A4_OK || M == 0) return st;
    if (!X) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(X) || (act_ws && !aligned16(act_ws))) return W4A4_ERR_MISALIGNED;
    const bool fused = kernel == W4A4_KERNEL_FUSED || (kernel == W4A4_KERNEL_AUTO && w4a4_forward_is_fused(M, N, K, r));
    if (fused && !fused_eligible(M, N, K, r)) return W4A4_ERR_UNSUPPORTED_SHAPE;
    const size_t need = act_layout(M, K, r).total;
    if (act_ws ? act_ws_bytes < need : !fused) return act_ws ? W4A4_ERR_WORKSPACE : W4A4_ERR_INVALID_ARG;
    const uint8_t* pk = static_cast<const uint8_t*>(packed);
    if (fused)
        return launch_linear_fused(X, pk, colscale, bias, M, N, K, r, Y, static_cast<uint8_t*>(act_ws), nullptr,
                                   stream);
    st = launch_quantize_act(X, pk, M, K, r, static_cast<uint8_t*>(act_ws), stream);
    if (st != W4A4_OK) return st;
    return w4a4_linear_select(act_ws, act_ws_bytes, packed, packed_bytes, colscale, bias, M, N, K, r, Y, kernel,
                              stream);
}

w4a4_status w4a4_linear_silu_mul(const void* act_ws, size_t act_ws_bytes, const void* packed, size_t packed_bytes,
                                 const uint16_t* colscale, const uint16_t* bias, int M, int N, int K, int r,
                                 uint16_t* H, cudaStream_t stream) {
    if (N % 32 != 0) return W4A4_ERR_UNSUPPORTED_SHAPE;
    w4a4_status st = linear_checks(act_ws, act_ws_bytes, packed, packed_bytes, colscale, bias, M, N, K, r, H);
    if (st != W4A4_OK || M == 0) return st;
    const uint8_t* ws = static_cast<const uint8_t*>(act_ws);
    const uint8_t* pk = static_cast<const uint8_t*>(packed);
    // up to the small-M threshold the tcgen05 weight-streaming kernel, above it the tiles
    if (M <= w4a4_small_m_threshold())
        return launch_gemm_smallm_tc(ws, pk, colscale, bias, M, N, K, r, H, nullptr, N / 2, stream);
    const ActLayout AL = act_layout(M, K, r);
    const bool sk_room = AL.full > AL.total && act_ws_bytes >= AL.full;
    return launch_gemm_tc(ws, pk, colscale, bias, M, N, K, r, H, nullptr, sk_room, N / 2, stream);
}

w4a4_status w4a16_linear(const uint16_t* X, const void* packed, size_t packed_bytes, const uint16_t* colscale,
                         const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, cudaStream_t stream) {
    if (M < 0) return W4A4_ERR_INVALID_ARG;
    w4a4_status st = check_kn(N, K, r);
    if (st != W4A4_OK) return st;
    if (M == 0) return W4A4_OK;
    if (!X || !packed || !colscale || !Y) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(packed) || !aligned16(colscale) || (bias && !aligned16(bias)) || !aligned16(Y))
        return W4A4_ERR_MISALIGNED;
    if (packed_bytes < packed_layout(N, K, r).total) return W4A4_ERR_WORKSPACE;
    if ((st = check_device()) != W4A4_OK) return st;
    return launch_gemm_w4a16(X, static_cast<const uint8_t*>(packed), colscale, bias, M, N, K, r, Y, false, stream);
}

w4a4_status w4a16_pack_weights_asym(const float* W, const uint16_t* L_down, const uint16_t* L_up, int N, int K,
                                    int r, void* packed, size_t packed_bytes, cudaStream_t stream) {
    w4a4_status st = check_kn(N, K, r);
    if (st != W4A4_OK) return st;
    if (K % 128 != 0) return W4A4_ERR_UNSUPPORTED_SHAPE;
    if (!packed || !W || (r > 0 && (!L_down || !L_up))) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(W) || (L_down && !aligned16(L_down)) || (L_up && !aligned16(L_up)))
        return W4A4_ERR_MISALIGNED;
    if (packed_bytes < packed_layout(N, K, r).total) return W4A4_ERR_WORKSPACE;
    if ((st = check_device()) != W4A4_OK) return st;
    uint8_t* out = static_cast<uint8_t*>(packed);
    launch_pack_lora(L_down, L_up, N, K, r, 0, out, stream);
    if ((st = launch_status()) != W4A4_OK) return st;
    set_dispatch("pack_weights_asym N=%d K=%d r=%d group=128", N, K, r);
    return launch_pack_weights_asym(W, N, K, r, out, stream);
}

w4a4_status w4a16_linear_asym(const uint16_t* X, const void* packed, size_t packed_bytes, const uint16_t* colscale,
                              const uint16_t* bias, int M, int N, int K, int r, uint16_t* Y, cudaStream_t stream) {
    if (M < 0) return W4A4_ERR_INVALID_ARG;
    w4a4_status st = check_kn(N, K, r);
    if (st != W4A4_OK) return st;
    if (K % 128 != 0) return W4A4_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return W4A4_OK;
    if (!X || !packed || !colscale || !Y) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(packed) || !aligned16(colscale) || (bias && !aligned16(bias)) || !aligned16(Y))
        return W4A4_ERR_MISALIGNED;
    if (packed_bytes < packed_layout(N, K, r).total) return W4A4_ERR_WORKSPACE;
    if ((st = check_device()) != W4A4_OK) return st;
    return launch_gemm_w4a16(X, static_cast<const uint8_t*>(packed), colscale, bias, M, N, K, r, Y, true, stream);
}

w4a4_status w4a4_rmsnorm_f16(const uint16_t* Y, int M, int ld_y, int K, uint16_t* X, cudaStream_t stream) {
    if (M < 0 || K < 0 || ld_y < K) return W4A4_ERR_INVALID_ARG;
    if (K < 8 || K % 8 != 0 || K > 16384 || ld_y % 8 != 0) return W4A4_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return W4A4_OK;
    if (!Y || !X) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(Y) || !aligned16(X)) return W4A4_ERR_MISALIGNED;
    w4a4_status st = check_device();
    if (st != W4A4_OK) return st;
    launch_rmsnorm_f16(Y, M, ld_y, K, W4A4_RMSNORM_EPS, X, stream);
    return launch_status();
}

w4a4_status w4a4_debug_unpack_weights(const void* packed, int N, int K, int r, int8_t* codes, uint16_t* scales,
                                      uint16_t* L_down, uint16_t* L_up, cudaStream_t stream) {
    w4a4_status st = check_kn(N, K, r);
    if (st != W4A4_OK) return st;
    if (!packed || !codes || !scales) return W4A4_ERR_INVALID_ARG;
    if ((st = check_device()) != W4A4_OK) return st;
    launch_unpack_weights(static_cast<const uint8_t*>(packed), N, K, r, codes, scales, L_down, L_up, stream);
    if ((st = launch_status()) != W4A4_OK) return st;
    return sync_status(stream);
}

w4a4_status w4a4_debug_unpack_act(const void* act_ws, int M, int K, int r, int8_t* codes, float* sA, float* SA,
                                  float* lora_act, cudaStream_t stream) {
    if (M < 0) return W4A4_ERR_INVALID_ARG;
    w4a4_status st = check_kn(16, K, r);
    if (st != W4A4_OK) return st;
    if (M == 0) return W4A4_OK;
    if (!act_ws || !codes || !sA) return W4A4_ERR_INVALID_ARG;
    if ((st = check_device()) != W4A4_OK) return st;
    launch_unpack_act(static_cast<const uint8_t*>(act_ws), M, K, r, codes, sA, SA, lora_act, stream);
    if ((st = launch_status()) != W4A4_OK) return st;
    return sync_status(stream);
}

w4a4_status w4a4_debug_group_partials(const void* act_ws, size_t act_ws_bytes, const void* packed,
                                      size_t packed_bytes, int M, int N, int K, int r, int kernel, int32_t* P,
                                      cudaStream_t stream) {
    if (kernel < W4A4_KERNEL_AUTO || kernel > W4A4_KERNEL_SMALLM_TC) return W4A4_ERR_INVALID_ARG;
    if (M < 0) return W4A4_ERR_INVALID_ARG;
    w4a4_status st = check_kn(N, K, r);
    if (st != W4A4_OK) return st;
    if (M == 0) return W4A4_OK;
    if (!act_ws || !packed || !P) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(act_ws) || !aligned16(packed)) return W4A4_ERR_MISALIGNED;
    const ActLayout AL = act_layout(M, K, r);
    if (act_ws_bytes < AL.total || packed_bytes < packed_layout(N, K, r).total) return W4A4_ERR_WORKSPACE;
    if ((st = check_device()) != W4A4_OK) return st;
    const uint8_t* ws = static_cast<const uint8_t*>(act_ws);
    const uint8_t* pk = static_cast<const uint8_t*>(packed);
    // the kernel and schedule w4a4_linear_select would run, with the dump on and no output
    const int k = pick_kernel(M, kernel);
    if (k == W4A4_KERNEL_TC) {
        const bool sk_room = AL.full > AL.total && act_ws_bytes >= AL.full;
        st = launch_gemm_tc(ws, pk, nullptr, nullptr, M, N, K, r, nullptr, P, sk_room, 0, stream);
    } else if (k == W4A4_KERNEL_SMALLM_TC) {
        st = launch_gemm_smallm_tc(ws, pk, nullptr, nullptr, M, N, K, r, nullptr, P, 0, stream);
    } else {
        st = launch_gemm_smallm(ws, pk, nullptr, nullptr, M, N, K, r, nullptr, P, stream);
    }
    if (st != W4A4_OK) return st;
    if ((st = sync_status(stream)) != W4A4_OK) return st;
    return device_status_words();
}

w4a4_status w4a4_debug_forward_partials(const uint16_t* X, const void* packed, size_t packed_bytes, int M, int N,
                                        int K, int r, void* act_ws, size_t act_ws_bytes, int32_t* P,
                                        cudaStream_t stream) {
    if (M < 0) return W4A4_ERR_INVALID_ARG;
    w4a4_status st = check_kn(N, K, r);
    if (st != W4A4_OK) return st;
    if (M == 0) return W4A4_OK;
    if (!X || !packed || !P) return W4A4_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(packed) || (act_ws && !aligned16(act_ws))) return W4A4_ERR_MISALIGNED;
    if (packed_bytes < packed_layout(N, K, r).total) return W4A4_ERR_WORKSPACE;
    if (act_ws && act_ws_bytes < act_layout(M, K, r).total) return W4A4_ERR_WORKSPACE;
    if (!fused_eligible(M, N, K, r)) return W4A4_ERR_UNSUPPORTED_SHAPE;
    if ((st = check_device()) != W4A4_OK) return st;
    st = launch_linear_fused(X, static_cast<const uint8_t*>(packed), nullptr, nullptr, M, N, K, r, nullptr,
                             static_cast<uint8_t*>(act_ws), P, stream);
    if (st != W4A4_OK) return st;
    if ((st = sync_status(stream)) != W4A4_OK) return st;
    return device_status_words();
}

w4a4_status w4a4_device_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return W4A4_ERR_CUDA;
    }
    return device_status_words();
}

}  // extern "C"
