"""GB300 (sm_103a) W4A4 + LoRA quantized linear layer.

Thin Python binding of the C ABI in ``include/w4a4.h`` (library
``libw4a4.so`` built in-tree by ``build.py``).  Functions keep the C names and
only marshal arguments: every step of the layer runs in the CUDA kernels.
PyTorch is used by callers for device memory and streams.

There is no CPU fallback: if the library is missing or no sm_103 device is
current, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a4.so")

W4A4_OK = 0
W4A4_ERR_TIMEOUT = 6
KERNEL_AUTO, KERNEL_TC, KERNEL_SMALLM, KERNEL_SMALLM_TC, KERNEL_FUSED = 0, 1, 2, 3, 4
GROUP = 64

_STATUS = {
    0: "W4A4_OK", 1: "W4A4_ERR_INVALID_ARG", 2: "W4A4_ERR_UNSUPPORTED_SHAPE", 3: "W4A4_ERR_MISALIGNED",
    4: "W4A4_ERR_WORKSPACE", 5: "W4A4_ERR_CUDA", 6: "W4A4_ERR_TIMEOUT", 7: "W4A4_ERR_NO_DEVICE",
}


class W4A4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)} ({lib().w4a4_status_string(status).decode()})")


_lib = None

# (name, restype, argtypes) for every entry point of include/w4a4.h
P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "w4a4_packed_weights_bytes": (Z, [I, I, I]),
    "w4a4_act_workspace_bytes": (Z, [I, I, I]),
    "w4a4_act_workspace_min_bytes": (Z, [I, I, I]),
    "w4a4_pack_weights": (I, [P, P, P, I, I, I, P, Z, P]),
    "w4a4_pack_weight_codes": (I, [P, P, P, P, I, I, I, P, Z, P]),
    "w4a4_quantize_act": (I, [P, P, Z, I, I, I, P, Z, P]),
    "w4a4_linear": (I, [P, Z, P, Z, P, P, I, I, I, I, P, P]),
    "w4a4_linear_select": (I, [P, Z, P, Z, P, P, I, I, I, I, P, I, P]),
    "w4a4_linear_noalloc": (I, [P, P, Z, P, P, I, I, I, I, P, P]),
    "w4a4_forward": (I, [P, P, Z, P, P, I, I, I, I, P, P, Z, I, P]),
    "w4a4_forward_is_fused": (I, [I, I, I, I]),
    "w4a4_debug_forward_partials": (I, [P, P, Z, I, I, I, I, P, Z, P, P]),
    "w4a4_rmsnorm_f16": (I, [P, I, I, I, P, P]),
    "w4a4_quantize_act_rmsnorm": (I, [P, I, P, Z, I, I, I, P, Z, P]),
    "w4a16_linear": (I, [P, P, Z, P, P, I, I, I, I, P, P]),
    "w4a16_pack_weights_asym": (I, [P, P, P, I, I, I, P, Z, P]),
    "w4a4_pack_weights_gate_up": (I, [P, P, P, I, I, I, P, Z, P]),
    "w4a4_svd_lora_scratch_bytes": (Z, [I, I, I]),
    "w4a4_pack_weights_svd": (I, [P, I, I, I, I, I, ctypes.c_ulonglong, P, Z, P, P, P, P, Z, P]),
    "w4a4_truncated_svd": (I, [P, I, I, I, I, ctypes.c_ulonglong, P, P, P, P, Z, P]),
    "w4a4_linear_silu_mul": (I, [P, Z, P, Z, P, P, I, I, I, I, P, P]),
    "w4a16_linear_asym": (I, [P, P, Z, P, P, I, I, I, I, P, P]),
    "w4a4_debug_unpack_weights": (I, [P, I, I, I, P, P, P, P, P]),
    "w4a4_debug_unpack_act": (I, [P, I, I, I, P, P, P, P, P]),
    "w4a4_debug_group_partials": (I, [P, Z, P, Z, I, I, I, I, I, P, P]),
    "w4a4_device_status": (I, []),
    "w4a4_status_string": (ctypes.c_char_p, [I]),
    "w4a4_last_dispatch": (ctypes.c_char_p, []),
    "w4a4_small_m_threshold": (I, []),
    "w4a4_stream_k": (I, []),
    "w4a4_set_stream_k": (None, [I]),
    "w4a4_set_small_m_threshold": (None, [I]),
    "w4a4_layout_version": (I, []),
}


def lib():
    """Load libw4a4.so (raises if it was not built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                              "or python w4a4_quantized_gemm_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != W4A4_OK:
        raise W4A4Error(status, where)


def _ptr(t):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "device tensors must be contiguous CUDA tensors"
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _nbytes(t):
    return t.numel() * t.element_size()


# ---------------------------------------------------------------- size queries
def packed_weights_bytes(N: int, K: int, r: int) -> int:
    n = lib().w4a4_packed_weights_bytes(N, K, r)
    if n == 0:
        raise W4A4Error(2, "w4a4_packed_weights_bytes")
    return n


def act_workspace_bytes(M: int, K: int, r: int) -> int:
    n = lib().w4a4_act_workspace_bytes(M, K, r)
    if n == 0 and M > 0:
        raise W4A4Error(2, "w4a4_act_workspace_bytes")
    return n


def act_workspace_min_bytes(M: int, K: int, r: int) -> int:
    """Bytes every call needs (without the GEMM's optional stream-K hand-over area)."""
    n = lib().w4a4_act_workspace_min_bytes(M, K, r)
    if n == 0 and M > 0:
        raise W4A4Error(2, "w4a4_act_workspace_min_bytes")
    return n


# ------------------------------------------------------------------ entry points
def w4a4_pack_weights(W, L_down, L_up, packed, r: int, stream=None):
    N, K = W.shape
    _check(lib().w4a4_pack_weights(_ptr(W), _ptr(L_down), _ptr(L_up), N, K, r, _ptr(packed), _nbytes(packed),
                                   _stream(stream)), "w4a4_pack_weights")


def w4a4_pack_weight_codes(codes, scales, L_down, L_up, packed, r: int, stream=None):
    N, K = codes.shape
    _check(lib().w4a4_pack_weight_codes(_ptr(codes), _ptr(scales), _ptr(L_down), _ptr(L_up), N, K, r,
                                        _ptr(packed), _nbytes(packed), _stream(stream)), "w4a4_pack_weight_codes")


def w4a4_quantize_act(X, packed, act_ws, r: int, stream=None):
    M, K = X.shape
    _check(lib().w4a4_quantize_act(_ptr(X), _ptr(packed), _nbytes(packed) if packed is not None else 0, M, K, r,
                                   _ptr(act_ws), _nbytes(act_ws),
                                   _stream(stream)), "w4a4_quantize_act")


def w4a16_linear(X, packed, colscale, bias, Y, r: int, stream=None):
    """W4A16 linear: fp16 X [M, K] against the packed INT4 weights -> Y [M, N]."""
    M, K = X.shape
    N = Y.shape[1]
    _check(lib().w4a16_linear(_ptr(X), _ptr(packed), _nbytes(packed), _ptr(colscale), _ptr(bias), M, N, K, r, _ptr(Y),
                              _stream(stream)), "w4a16_linear")


def w4a4_pack_weights_gate_up(W, L_down, L_up, packed, r: int, stream=None):
    """Fused gate|up weights W [N, K] (gate rows first) packed for w4a4_linear_silu_mul."""
    N, K = W.shape
    _check(lib().w4a4_pack_weights_gate_up(_ptr(W), _ptr(L_down), _ptr(L_up), N, K, r, _ptr(packed),
                                           _nbytes(packed), _stream(stream)), "w4a4_pack_weights_gate_up")


def w4a4_linear_silu_mul(act_ws, packed, colscale, bias, H, K: int, r: int, stream=None):
    """H [M, N/2] = silu(gate) * up of the fused gate|up W4A4 linear (colscale, bias [N])."""
    M, I = H.shape
    _check(lib().w4a4_linear_silu_mul(_ptr(act_ws), _nbytes(act_ws), _ptr(packed), _nbytes(packed), _ptr(colscale),
                                      _ptr(bias), M, 2 * I, K, r, _ptr(H), _stream(stream)), "w4a4_linear_silu_mul")


def svd_lora_scratch_bytes(N: int, K: int, r: int) -> int:
    n = lib().w4a4_svd_lora_scratch_bytes(N, K, r)
    if n == 0:
        raise W4A4Error(2, "w4a4_svd_lora_scratch_bytes")
    return n


def w4a4_pack_weights_svd(W, r: int, packed, rounds: int = 3, power_iters: int = 16, seed: int = 0,
                          scratch=None, stream=None):
    """Quantise W [N, K] and derive its rank-r LoRA from the quantisation error
    (SVD refit rounds).  Returns (L_down fp16 [K, r], L_up fp16 [r, N], per-round
    residuals) and fills `packed`."""
    N, K = W.shape
    dev = W.device
    Ld = torch.empty((K, r), dtype=torch.float16, device=dev)
    Lu = torch.empty((r, N), dtype=torch.float16, device=dev)
    if scratch is None:
        scratch = torch.empty(svd_lora_scratch_bytes(N, K, r), dtype=torch.uint8, device=dev)
    errs = (ctypes.c_float * rounds)()
    _check(lib().w4a4_pack_weights_svd(_ptr(W), N, K, r, rounds, power_iters, seed, _ptr(packed), _nbytes(packed),
                                       _ptr(Ld), _ptr(Lu), ctypes.cast(errs, ctypes.c_void_p), _ptr(scratch),
                                       _nbytes(scratch), _stream(stream)), "w4a4_pack_weights_svd")
    return Ld, Lu, [float(e) for e in errs]


def w4a4_truncated_svd(A, r: int, power_iters: int = 16, seed: int = 0, scratch=None, stream=None):
    """Rank-r SVD of A fp32 [N, K] on the GPU: (U [N, r], S [r], V [K, r])."""
    N, K = A.shape
    dev = A.device
    U = torch.empty((N, r), dtype=torch.float32, device=dev)
    S = torch.empty((r,), dtype=torch.float32, device=dev)
    V = torch.empty((K, r), dtype=torch.float32, device=dev)
    if scratch is None:
        scratch = torch.empty(svd_lora_scratch_bytes(N, K, r), dtype=torch.uint8, device=dev)
    _check(lib().w4a4_truncated_svd(_ptr(A), N, K, r, power_iters, seed, _ptr(U), _ptr(S), _ptr(V), _ptr(scratch),
                                    _nbytes(scratch), _stream(stream)), "w4a4_truncated_svd")
    return U, S, V


def w4a16_pack_weights_asym(W, L_down, L_up, packed, r: int, stream=None):
    """Asymmetric group-128 INT4 weights (fp16 scale + zero point per group) into `packed`."""
    N, K = W.shape
    _check(lib().w4a16_pack_weights_asym(_ptr(W), _ptr(L_down), _ptr(L_up), N, K, r, _ptr(packed), _nbytes(packed),
                                         _stream(stream)), "w4a16_pack_weights_asym")


def w4a16_linear_asym(X, packed, colscale, bias, Y, r: int, stream=None):
    """W4A16 linear on weights packed by w4a16_pack_weights_asym."""
    M, K = X.shape
    N = Y.shape[1]
    _check(lib().w4a16_linear_asym(_ptr(X), _ptr(packed), _nbytes(packed), _ptr(colscale), _ptr(bias), M, N, K, r,
                                   _ptr(Y), _stream(stream)), "w4a16_linear_asym")


def w4a4_quantize_act_rmsnorm(Y, K: int, packed, act_ws, r: int, stream=None):
    """RMSNorm of the first K columns of each row of Y [M, ld], then the
    activation step of the next linear on the normalised values."""
    M, ld = Y.shape
    _check(lib().w4a4_quantize_act_rmsnorm(_ptr(Y), ld, _ptr(packed), _nbytes(packed) if packed is not None else 0,
                                           M, K, r, _ptr(act_ws), _nbytes(act_ws),
                                           _stream(stream)), "w4a4_quantize_act_rmsnorm")


def w4a4_linear(act_ws, packed, colscale, bias, Y, K: int, r: int, kernel: int = KERNEL_AUTO, stream=None):
    M, N = Y.shape
    _check(lib().w4a4_linear_select(_ptr(act_ws), _nbytes(act_ws), _ptr(packed), _nbytes(packed), _ptr(colscale),
                                    _ptr(bias), M, N, K, r, _ptr(Y), kernel, _stream(stream)), "w4a4_linear")


def w4a4_forward(X, packed, colscale, bias, Y, r: int, act_ws=None, kernel: int = KERNEL_AUTO, stream=None):
    """The whole layer from fp16 X [M, K] into Y [M, N] in one call (one fused
    kernel at small M, else quantise + GEMM on act_ws; see include/w4a4.h)."""
    M, K = X.shape
    N = Y.shape[1]
    _check(lib().w4a4_forward(_ptr(X), _ptr(packed), _nbytes(packed), _ptr(colscale), _ptr(bias), M, N, K, r,
                              _ptr(Y), _ptr(act_ws), 0 if act_ws is None else _nbytes(act_ws), kernel,
                              _stream(stream)), "w4a4_forward")


def w4a4_forward_is_fused(M: int, N: int, K: int, r: int) -> bool:
    return bool(lib().w4a4_forward_is_fused(M, N, K, r))


def w4a4_linear_noalloc(X, packed, colscale, bias, Y, r: int, stream=None):
    """Quantise X and run the layer with the library's built-in workspace (no
    allocation anywhere; see include/w4a4.h for its size limit and sharing rules)."""
    M, K = X.shape
    N = Y.shape[1]
    _check(lib().w4a4_linear_noalloc(_ptr(X), _ptr(packed), _nbytes(packed), _ptr(colscale), _ptr(bias), M, N, K,
                                     r, _ptr(Y), _stream(stream)), "w4a4_linear_noalloc")


NOALLOC_WORKSPACE_BYTES = 8 << 20


def w4a4_rmsnorm_f16(Y, K: int, X, stream=None):
    """RMSNorm (unit gain) of the first K columns of each row of Y into X [M, K]."""
    M, ld = Y.shape
    if X.shape[0] != M or X.shape[1] != K:
        raise W4A4Error(1, "w4a4_rmsnorm_f16")
    _check(lib().w4a4_rmsnorm_f16(_ptr(Y), M, ld, K, _ptr(X), _stream(stream)), "w4a4_rmsnorm_f16")


def w4a4_debug_unpack_weights(packed, N: int, K: int, r: int, stream=None):
    dev = packed.device
    codes = torch.empty((N, K), dtype=torch.int8, device=dev)
    scales = torch.empty((N, K // GROUP), dtype=torch.float16, device=dev)
    Ld = torch.empty((K, r), dtype=torch.float16, device=dev) if r else None
    Lu = torch.empty((r, N), dtype=torch.float16, device=dev) if r else None
    _check(lib().w4a4_debug_unpack_weights(_ptr(packed), N, K, r, _ptr(codes), _ptr(scales), _ptr(Ld), _ptr(Lu),
                                           _stream(stream)), "w4a4_debug_unpack_weights")
    return codes, scales, Ld, Lu


def w4a4_debug_unpack_act(act_ws, M: int, K: int, r: int, stream=None):
    dev = act_ws.device
    codes = torch.empty((M, K), dtype=torch.int8, device=dev)
    sA = torch.empty((M, K // GROUP), dtype=torch.float32, device=dev)
    SA = torch.empty((M, K // GROUP), dtype=torch.float32, device=dev)
    lora = torch.empty((M, r), dtype=torch.float32, device=dev) if r else None
    _check(lib().w4a4_debug_unpack_act(_ptr(act_ws), M, K, r, _ptr(codes), _ptr(sA), _ptr(SA), _ptr(lora),
                                       _stream(stream)), "w4a4_debug_unpack_act")
    return codes, sA, SA, lora


def w4a4_debug_group_partials(act_ws, packed, M: int, N: int, K: int, r: int, kernel: int, stream=None):
    P_ = torch.empty((M, N, K // GROUP), dtype=torch.int32, device=act_ws.device)
    _check(lib().w4a4_debug_group_partials(_ptr(act_ws), _nbytes(act_ws), _ptr(packed), _nbytes(packed), M, N, K,
                                           r, kernel, _ptr(P_), _stream(stream)), "w4a4_debug_group_partials")
    return P_


def w4a4_debug_forward_partials(X, packed, N: int, r: int, act_ws=None, stream=None):
    M, K = X.shape
    P_ = torch.empty((M, N, K // GROUP), dtype=torch.int32, device=X.device)
    _check(lib().w4a4_debug_forward_partials(_ptr(X), _ptr(packed), _nbytes(packed), M, N, K, r, _ptr(act_ws),
                                             0 if act_ws is None else _nbytes(act_ws), _ptr(P_), _stream(stream)),
           "w4a4_debug_forward_partials")
    return P_


def w4a4_device_status() -> int:
    return lib().w4a4_device_status()


def w4a4_last_dispatch() -> str:
    return lib().w4a4_last_dispatch().decode()


def w4a4_small_m_threshold() -> int:
    return lib().w4a4_small_m_threshold()


def w4a4_set_small_m_threshold(m: int):
    lib().w4a4_set_small_m_threshold(int(m))


def w4a4_stream_k() -> bool:
    return bool(lib().w4a4_stream_k())


def w4a4_set_stream_k(on: bool):
    lib().w4a4_set_stream_k(1 if on else 0)


# ------------------------------------------------------------- layer helper
class W4A4Linear:
    """One packed layer: buffers allocated with torch, compute in the library.

    ``forward(X)`` = w4a4_quantize_act + w4a4_linear (two kernel launches).
    """

    def __init__(self, W, L_down, L_up, colscale, bias=None, stream=None):
        self.N, self.K = W.shape
        self.r = 0 if L_down is None else L_down.shape[1]
        dev = W.device
        self.packed = torch.empty(packed_weights_bytes(self.N, self.K, self.r), dtype=torch.uint8, device=dev)
        w4a4_pack_weights(W.contiguous(), L_down, L_up, self.packed, self.r, stream)
        self.colscale = colscale.contiguous()
        self.bias = None if bias is None else bias.contiguous()
        self._ws = None

    def workspace(self, M: int):
        need = act_workspace_bytes(M, self.K, self.r)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.packed.device)
        return self._ws

    def forward(self, X, out=None, kernel: int = KERNEL_AUTO, stream=None):
        M = X.shape[0]
        ws = self.workspace(M)
        Y = out if out is not None else torch.empty((M, self.N), dtype=torch.float16, device=X.device)
        w4a4_quantize_act(X, self.packed, ws, self.r, stream)
        w4a4_linear(ws, self.packed, self.colscale, self.bias, Y, self.K, self.r, kernel, stream)
        return Y

    __call__ = forward
