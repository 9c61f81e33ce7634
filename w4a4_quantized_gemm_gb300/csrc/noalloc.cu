// Allocation-free variant of the whole layer: quantise X and run the GEMM with
// the activation workspace held in a fixed-size array that lives in the
// library's own device memory, for callers that cannot allocate device memory
// themselves (for example code running inside an allocator callback, a
// host-side runtime whose memory is owned by someone else, or a plugin ABI
// that only hands over input and output pointers).
//
// The array is reserved when the library is loaded onto a device and stays
// there until the process exits.  Every call uses the same array and leaves
// its contents behind; nothing in it needs to start at zero because each call
// rewrites every workspace row that can influence its output.  Two calls whose
// work overlaps on the GPU (different streams, or different host threads on
// one device) race on the array and give undefined results.
#include <mutex>

#include "kernels.h"

namespace w4a4 {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_ws[W4A4_NOALLOC_WORKSPACE_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

// Device address of the array on the current device.  The host-side name of
// the array is only a stand-in, so the address must come from the runtime; it
// is looked up once per device, on the first call made with that device current.
w4a4_status noalloc_workspace(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return W4A4_ERR_NO_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return W4A4_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return W4A4_OK;
}

}  // namespace
}  // namespace w4a4

extern "C" w4a4_status w4a4_linear_noalloc(const uint16_t* X, const void* packed, size_t packed_bytes,
                                           const uint16_t* colscale, const uint16_t* bias, int M, int N, int K,
                                           int r, uint16_t* Y, cudaStream_t stream) {
    // Every argument is checked before anything is launched or looked up: the
    // shapes, the pointers of both steps, packed_bytes, and the array's size.
    // The device is checked last, so that a bad call is refused the same way
    // with or without a usable GPU.
    if (M < 0 || N < 0 || K < 0 || r < 0) return W4A4_ERR_INVALID_ARG;
    if (K < w4a4::kGroup || K % w4a4::kGroup != 0 || N < 16 || N % 16 != 0 || r % 16 != 0 || r > W4A4_MAX_RANK)
        return W4A4_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return W4A4_OK;
    if (!X) return W4A4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(X) & 15u) != 0) return W4A4_ERR_MISALIGNED;
    // the workspace every call needs must fit the array; the GEMM's optional
    // stream-K hand-over area never does, so that schedule is not used here
    if (w4a4::act_layout(M, K, r).total > size_t(W4A4_NOALLOC_WORKSPACE_BYTES)) return W4A4_ERR_WORKSPACE;
    w4a4_status st = w4a4::linear_checks_no_ws(packed, packed_bytes, colscale, bias, M, N, K, r, Y);
    if (st != W4A4_OK) return st;
    void* ws = nullptr;
    st = w4a4::noalloc_workspace(&ws);
    if (st != W4A4_OK) return st;
    st = w4a4_quantize_act(X, packed, packed_bytes, M, K, r, ws, W4A4_NOALLOC_WORKSPACE_BYTES, stream);
    if (st != W4A4_OK) return st;
    return w4a4_linear(ws, W4A4_NOALLOC_WORKSPACE_BYTES, packed, packed_bytes, colscale, bias, M, N, K, r, Y, stream);
}
