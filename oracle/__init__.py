"""CPU oracle for the W4A4 + LoRA quantized linear layer (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``.  The product path
(``w4a4_quantized_gemm_gb300``) never imports it, and this package imports
nothing from the product.

The arithmetic lives in ``w4a4_oracle.c`` (plain single-threaded C, fp64 /
int64 accumulation); this file only compiles it with gcc and marshals numpy
arrays.  See the C file's header for the passages each function follows.

Status of the pins (tests/test_oracle_pins.py):
  * fp16 conversions          -- pinned (exhaustive + numpy's float16 cast)
  * quantize_act/_weights     -- pinned (invariants, crafted ties, closed forms)
  * group_partials            -- pinned (brute force, all -8 = 4096, cancellation)
  * lora_down / linear        -- pinned (numpy fp64 matmul special cases:
                                 rank 0, zero weights, dequantised reference)
  * w4a16                     -- pinned (one-hot rows, exact homogeneity, the W4A4
                                 layer on exactly quantisable inputs, numpy matmul)
  * quantize_weights_asym /   -- pinned (exactly representable groups: codes, scale,
    w4a16_asym                   zero and values recovered; code range and the
                                 half-step bound; the layer on such weights equals
                                 a numpy fp64 matmul; one-hot rows)
  * svd_lora                  -- pinned (a planted low-rank quantisation error is
                                 recovered exactly; full rank leaves no error;
                                 exactly representable W gives no LoRA; one round
                                 reduces to the plain quantiser; errors fall)
  * silu_mul                  -- pinned (closed forms: silu(0) = 0, silu(ln 3) =
                                 (3/4) ln 3, silu(v) -> v and -> 0 in the tails;
                                 the gate/up column split on crafted rows)
  * rmsnorm_f16 / f64_to_f16  -- pinned (constant rows -> +-1 exactly, a zero row
                                 -> 0, columns past K ignored, odd symmetry, unit
                                 mean square; the encoder against numpy's rounding)
  * linear_sampled /          -- pinned (equal to the full evaluators on the same
    silu_mul_linear_sampled /    rows and columns)
    linear_rows
  * pack_weights_v1 /         -- pinned (every code, scale and LoRA value lands in
    pack_act_v1                  exactly one place, the defined bytes tile each
                                 section; hand-derived byte positions of the layout
                                 statement in tests/golden/layout_v1_positions.txt;
                                 E4M3 bytes against torch's float8_e4m3fn cast;
                                 decoding the bytes back gives the inputs)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GROUP = 64
CFLAGS = ["-O3", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fno-unsafe-math-optimizations", "-frounding-math"]


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/liboracle.so (gcc, portable flags)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int64
        lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_f16.restype = ctypes.c_uint16
        lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_f16.restype = ctypes.c_uint16
        lib.oracle_rmsnorm_f16.argtypes = [P, I, I, I, ctypes.c_double, P]
        lib.oracle_f64_to_f16_array.argtypes = [P, I, P]
        lib.oracle_quantize_act.argtypes = [P, I, I, P, P]
        lib.oracle_quantize_weights.argtypes = [P, I, I, P, P]
        lib.oracle_group_partials.argtypes = [P, P, I, I, I, P]
        lib.oracle_group_partials.restype = I
        lib.oracle_lora_down.argtypes = [P, P, I, I, I, P]
        lib.oracle_linear_from_codes.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, P]
        lib.oracle_linear_sampled.argtypes = [P, P, P, P, P, P, I, I, I, I, P, P, I, P, P, P, P, P, P]
        lib.oracle_w4a16_from_codes.argtypes = [P, P, P, P, P, P, P, I, I, I, I, P]
        lib.oracle_quantize_weights_asym.argtypes = [P, I, I, P, P, P]
        lib.oracle_silu_mul.argtypes = [P, I, I, P]
        lib.oracle_w4a16_asym_from_codes.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, P]
        lib.oracle_linear_rows.argtypes = [P, P, P, P, P, P, I, I, I, P, I, P, P, P, P, P, P]
        lib.oracle_packed_offsets.argtypes = [I, I, I, P]
        lib.oracle_act_offsets.argtypes = [I, I, I, P]
        lib.oracle_e4m3_of_int.argtypes = [ctypes.c_int]
        lib.oracle_e4m3_of_int.restype = ctypes.c_uint8
        lib.oracle_pack_weights_v1.argtypes = [P, P, P, P, I, I, I, P, P]
        lib.oracle_pack_act_v1.argtypes = [P, P, P, I, I, I, P, P]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def f16_to_f32(h: int) -> float:
    return float(_load().oracle_f16_to_f32(int(h)))


def f32_to_f16(x: float) -> int:
    return int(_load().oracle_f32_to_f16(float(np.float32(x))))


def f16_to_f32_array(h: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(h, dtype=np.uint16).ravel()
    out = np.fromiter((lib.oracle_f16_to_f32(int(v)) for v in flat), dtype=np.float32, count=flat.size)
    return out.reshape(np.shape(h))


def quantize_act(X: np.ndarray):
    """X: fp16 bits [M, K] -> (codes int8 [M, K], scales fp32 [M, K/64])."""
    X = _c(X, np.uint16)
    M, K = X.shape
    assert K % GROUP == 0
    q = np.empty((M, K), np.int8)
    s = np.empty((M, K // GROUP), np.float32)
    _load().oracle_quantize_act(_ptr(X), M, K, _ptr(q), _ptr(s))
    return q, s


def quantize_weights(W: np.ndarray):
    """W: fp32 [N, K] -> (codes int8 [N, K], scales fp16 bits [N, K/64])."""
    W = _c(W, np.float32)
    N, K = W.shape
    assert K % GROUP == 0
    q = np.empty((N, K), np.int8)
    s = np.empty((N, K // GROUP), np.uint16)
    _load().oracle_quantize_weights(_ptr(W), N, K, _ptr(q), _ptr(s))
    return q, s


def group_partials(qA: np.ndarray, qW: np.ndarray) -> np.ndarray:
    """int32 [M, N, K/64] exact per-group integer dot products."""
    qA = _c(qA, np.int8)
    qW = _c(qW, np.int8)
    M, K = qA.shape
    N, K2 = qW.shape
    assert K == K2 and K % GROUP == 0
    P = np.empty((M, N, K // GROUP), np.int32)
    bad = _load().oracle_group_partials(_ptr(qA), _ptr(qW), M, N, K, _ptr(P))
    assert bad == 0, f"{bad} partial sums overflow int32"
    return P


def lora_down(X: np.ndarray, L_down: np.ndarray) -> np.ndarray:
    """fp64 [M, r] = X (fp16) @ L_down (fp16 [K, r])."""
    X = _c(X, np.uint16)
    M, K = X.shape
    Ld = np.zeros((K, 0), np.uint16) if L_down is None else _c(L_down, np.uint16).reshape(K, -1)
    K2, r = Ld.shape
    assert K2 == K
    D = np.zeros((M, r), np.float64)
    if r:
        _load().oracle_lora_down(_ptr(X), _ptr(Ld), M, K, r, _ptr(D))
    return D


def linear_from_codes(qA, sA, qW, sW, D, L_up, colscale, bias) -> np.ndarray:
    qA = _c(qA, np.int8); sA = _c(sA, np.float32)
    qW = _c(qW, np.int8); sW = _c(sW, np.uint16)
    M, K = qA.shape
    N = qW.shape[0]
    D = _c(D, np.float64).reshape(M, -1)
    r = D.shape[1]
    Lup = _c(L_up, np.uint16).reshape(r, N) if r else np.zeros((0, N), np.uint16)
    cs = _c(colscale, np.uint16)
    b = np.zeros(N, np.uint16) if bias is None else _c(bias, np.uint16)
    Y = np.empty((M, N), np.float64)
    _load().oracle_linear_from_codes(_ptr(qA), _ptr(sA), _ptr(qW), _ptr(sW), _ptr(D), _ptr(Lup),
                                     _ptr(cs), _ptr(b), M, N, K, r, _ptr(Y))
    return Y


class Reference:
    """Every intermediate of the oracle for one layer (small and medium sizes)."""

    def __init__(self, X, W, L_down, L_up, colscale, bias):
        self.qA, self.sA = quantize_act(X)
        self.qW, self.sW = quantize_weights(W)
        self.D = lora_down(X, L_down)
        self.Y = linear_from_codes(self.qA, self.sA, self.qW, self.sW, self.D, L_up, colscale, bias)

    def partials(self):
        return group_partials(self.qA, self.qW)


def linear(X, W, L_down, L_up, colscale, bias) -> np.ndarray:
    """fp64 Y [M, N] of the whole layer from raw inputs."""
    return Reference(X, W, L_down, L_up, colscale, bias).Y


def linear_sampled(X, W, L_down, L_up, colscale, bias, rows, cols) -> np.ndarray:
    """fp64 Y[rows[i], cols[i]] from raw inputs (sorted by row for reuse)."""
    X = _c(X, np.uint16); W = _c(W, np.float32)
    M, K = X.shape
    N = W.shape[0]
    r = 0 if L_down is None else np.asarray(L_down).reshape(K, -1).shape[1]
    Ld = _c(L_down, np.uint16).reshape(K, r) if r else np.zeros((K, 0), np.uint16)
    Lup = _c(L_up, np.uint16).reshape(r, N) if r else np.zeros((0, N), np.uint16)
    rows = _c(rows, np.int64); cols = _c(cols, np.int64)
    order = np.lexsort((cols, rows))
    rs, cs_ = np.ascontiguousarray(rows[order]), np.ascontiguousarray(cols[order])
    out = np.empty(rows.size, np.float64)
    qa = np.empty(K, np.int8); sa = np.empty(K // GROUP, np.float32)
    qw = np.empty(K, np.int8); sw = np.empty(K // GROUP, np.uint16)
    d = np.zeros(max(r, 1), np.float64)
    _load().oracle_linear_sampled(_ptr(X), _ptr(W), _ptr(Ld), _ptr(Lup), _ptr(_c(colscale, np.uint16)),
                                  _ptr(_c(bias, np.uint16)), M, N, K, r, _ptr(rs), _ptr(cs_), rows.size,
                                  _ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw), _ptr(d), _ptr(out))
    res = np.empty_like(out)
    res[order] = out
    return res


def w4a16_from_codes(X, qW, sW, D, L_up, colscale, bias) -> np.ndarray:
    """fp64 Y [M, N] of the W4A16 layer: fp16 X against the dequantised INT4 weights."""
    X = _c(X, np.uint16)
    qW = _c(qW, np.int8); sW = _c(sW, np.uint16)
    M, K = X.shape
    N = qW.shape[0]
    D = _c(D, np.float64).reshape(M, -1)
    r = D.shape[1]
    Lup = _c(L_up, np.uint16).reshape(r, N) if r else np.zeros((0, N), np.uint16)
    cs = _c(colscale, np.uint16)
    b = np.zeros(N, np.uint16) if bias is None else _c(bias, np.uint16)
    Y = np.empty((M, N), np.float64)
    _load().oracle_w4a16_from_codes(_ptr(X), _ptr(qW), _ptr(sW), _ptr(D), _ptr(Lup), _ptr(cs), _ptr(b),
                                    M, N, K, r, _ptr(Y))
    return Y


def w4a16_linear(X, W, L_down, L_up, colscale, bias) -> np.ndarray:
    """fp64 Y [M, N] of the W4A16 layer from raw inputs (the same weight quantiser and LoRA)."""
    qW, sW = quantize_weights(W)
    return w4a16_from_codes(X, qW, sW, lora_down(X, L_down), L_up, colscale, bias)


GROUP_ASYM = 128


def quantize_weights_asym(W: np.ndarray):
    """W fp32 [N, K] -> (codes uint8 [N, K] in 0..15, scale fp16 bits [N, K/128],
    zero fp16 bits [N, K/128]): asymmetric 4-bit with a zero point per group of 128."""
    W = _c(W, np.float32)
    N, K = W.shape
    q = np.empty((N, K), np.uint8)
    s = np.empty((N, K // GROUP_ASYM), np.uint16)
    z = np.empty((N, K // GROUP_ASYM), np.uint16)
    _load().oracle_quantize_weights_asym(_ptr(W), N, K, _ptr(q), _ptr(s), _ptr(z))
    return q, s, z


def w4a16_asym_from_codes(X, q, scale, zero, D, L_up, colscale, bias) -> np.ndarray:
    """fp64 Y [M, N]: fp16 X against (q - zero) * scale, plus the LoRA and the column affine."""
    X = _c(X, np.uint16)
    q = _c(q, np.uint8); scale = _c(scale, np.uint16); zero = _c(zero, np.uint16)
    M, K = X.shape
    N = q.shape[0]
    D = _c(D, np.float64).reshape(M, -1)
    r = D.shape[1]
    Lup = _c(L_up, np.uint16).reshape(r, N) if r else np.zeros((0, N), np.uint16)
    cs = _c(colscale, np.uint16)
    b = np.zeros(N, np.uint16) if bias is None else _c(bias, np.uint16)
    Y = np.empty((M, N), np.float64)
    _load().oracle_w4a16_asym_from_codes(_ptr(X), _ptr(q), _ptr(scale), _ptr(zero), _ptr(D), _ptr(Lup), _ptr(cs),
                                         _ptr(b), M, N, K, r, _ptr(Y))
    return Y


def w4a16_asym_linear(X, W, L_down, L_up, colscale, bias) -> np.ndarray:
    """fp64 Y [M, N] of the W4A16 layer with asymmetric group-128 weights, from raw inputs."""
    q, s, z = quantize_weights_asym(W)
    return w4a16_asym_from_codes(X, q, s, z, lora_down(X, L_down), L_up, colscale, bias)


def dequantize_weights(qW: np.ndarray, sW: np.ndarray) -> np.ndarray:
    """fp64 [N, K]: codes times their fp16 group-64 scale."""
    q = np.asarray(qW, np.float64)
    s = f16_to_f32_array(np.asarray(sW, np.uint16)).astype(np.float64)
    return q * np.repeat(s, GROUP, axis=1)


def truncated_svd(A: np.ndarray, r: int):
    """Rank-r truncated SVD of A in fp64 (LAPACK): U [N, r], S [r], V [K, r]."""
    U, S, Vt = np.linalg.svd(np.asarray(A, np.float64), full_matrices=False)
    return U[:, :r], S[:r], Vt[:r].T


def svd_lora(W: np.ndarray, r: int, rounds: int = 3):
    """LoRA correction of the INT4 weights from W alone ("W4A4 CUDA Kernel for
    Voice Clone", 2.1: the quantisation error E = W - Q(W) and its rank-r SVD,
    L_up = (U_r S_r)^T, L_down = V_r; 2.2: rounds that quantise W - LoRA_previous
    and refit the SVD to the new error, stopping when the error stops falling),
    with the plain round-to-nearest quantiser in place of GPTQ (no calibration
    data).  The residual handed to the quantiser is rounded to fp32, its input
    type.  Returns the round with the smallest ||W - Q - L_down L_up^T||_F as a
    dict (codes, scales, L_down fp64 [K, r], L_up fp64 [r, N], err) and the list
    of every round's error."""
    W64 = np.asarray(W, np.float32).astype(np.float64)
    LW = np.zeros_like(W64)
    best, errs = None, []
    for _ in range(rounds):
        q, sc = quantize_weights((W64 - LW).astype(np.float32))
        E = W64 - dequantize_weights(q, sc)
        U, S, V = truncated_svd(E, r)
        L_new = (U * S) @ V.T
        err = float(np.linalg.norm(E - L_new))
        errs.append(err)
        if best is not None and err >= best["err"]:
            break
        best = dict(codes=q, scales=sc, L_down=V, L_up=(U * S).T, err=err)
        LW = L_new
    return best, errs


def silu_mul(Y: np.ndarray) -> np.ndarray:
    """fp64 H [M, I] = silu(Y[:, :I]) * Y[:, I:] for a fused gate|up output Y fp64 [M, 2I]."""
    Y = _c(Y, np.float64)
    M, N2 = Y.shape
    H = np.empty((M, N2 // 2), np.float64)
    _load().oracle_silu_mul(_ptr(Y), M, N2 // 2, _ptr(H))
    return H


def silu_mul_linear(X, W, L_down, L_up, colscale, bias) -> np.ndarray:
    """fp64 H [M, N/2]: the W4A4 layer on a fused gate|up weight W [N, K] (gate rows
    first), then silu(gate) * up."""
    return silu_mul(linear(X, W, L_down, L_up, colscale, bias))


def silu_mul_linear_sampled(X, W, L_down, L_up, colscale, bias, rows, cols) -> np.ndarray:
    """fp64 H[rows[i], cols[i]] from raw inputs (the gate and up outputs of each pair sampled)."""
    rows = np.asarray(rows, np.int64); cols = np.asarray(cols, np.int64)
    I = np.asarray(W).shape[0] // 2
    y = linear_sampled(X, W, L_down, L_up, colscale, bias, np.r_[rows, rows], np.r_[cols, cols + I])
    return silu_mul(np.stack([y[: rows.size], y[rows.size:]], axis=1)).ravel()


RMSNORM_EPS = 1e-6


def f64_to_f16(x: float) -> int:
    """Nearest binary16 (ties to even) of a double, in one rounding; returns the bits."""
    return int(_load().oracle_f64_to_f16(float(x)))


def f64_to_f16_array(a: np.ndarray) -> np.ndarray:
    """Elementwise nearest binary16 (ties to even) of doubles -> uint16 bits, same shape."""
    a = _c(a, np.float64)
    out = np.empty(a.shape, np.uint16)
    _load().oracle_f64_to_f16_array(_ptr(a), a.size, _ptr(out))
    return out


def rmsnorm_f16(Y: np.ndarray, K: int, eps: float = RMSNORM_EPS) -> np.ndarray:
    """RMSNorm with unit gain of the first K columns of each row of Y (fp16 bits,
    uint16 [M, ld]) -> fp16 bits uint16 [M, K] ("W4A4 CUDA Kernel for Voice
    Clone", 3.9): x = fp16(y / sqrt(mean(y^2) + eps)), sum in double."""
    Y = _c(Y, np.uint16)
    M, ld = Y.shape
    X = np.empty((M, K), dtype=np.uint16)
    _load().oracle_rmsnorm_f16(_ptr(Y), M, ld, K, float(eps), _ptr(X))
    return X


def linear_rows(X, W, L_down, L_up, colscale, bias, rows) -> np.ndarray:
    """fp64 Y[rows[i], :] (every output column of the listed rows) from raw inputs;
    the weights are quantised once."""
    X = _c(X, np.uint16); W = _c(W, np.float32)
    M, K = X.shape
    N = W.shape[0]
    r = 0 if L_down is None else np.asarray(L_down).reshape(K, -1).shape[1]
    Ld = _c(L_down, np.uint16).reshape(K, r) if r else np.zeros((K, 0), np.uint16)
    Lup = _c(L_up, np.uint16).reshape(r, N) if r else np.zeros((0, N), np.uint16)
    rows = _c(rows, np.int64)
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < M)
    qW = np.empty((N, K), np.int8); sW = np.empty((N, K // GROUP), np.uint16)
    qa = np.empty(K, np.int8); sa = np.empty(K // GROUP, np.float32)
    d = np.zeros(max(r, 1), np.float64)
    Y = np.empty((rows.size, N), np.float64)
    _load().oracle_linear_rows(_ptr(X), _ptr(W), _ptr(Ld), _ptr(Lup), _ptr(_c(colscale, np.uint16)),
                               _ptr(_c(bias, np.uint16)), N, K, r, _ptr(rows), rows.size, _ptr(qW), _ptr(sW),
                               _ptr(qa), _ptr(sa), _ptr(d), _ptr(Y))
    return Y


def packed_offsets(N: int, K: int, r: int) -> dict:
    """Section offsets of the packed weight buffer (layout version 1)."""
    off = np.zeros(5, np.int64)
    _load().oracle_packed_offsets(N, K, r, _ptr(off))
    return dict(zip(("Ld", "qW", "sW", "Lu", "total"), (int(v) for v in off)))


def act_offsets(M: int, K: int, r: int) -> dict:
    """Section offsets of the activation workspace (layout version 1, minimum size)."""
    off = np.zeros(5, np.int64)
    _load().oracle_act_offsets(M, K, r, _ptr(off))
    return dict(zip(("qA", "sS", "La", "flags", "total"), (int(v) for v in off)))


def e4m3_of_int(c: int) -> int:
    """FP8 E4M3 byte of an integer in [-8, 8]."""
    return int(_load().oracle_e4m3_of_int(int(c)))


def pack_weights_v1(qW, sW, L_down, L_up):
    """Packed-weight bytes (layout version 1) of codes int8 [N, K], fp16 scales
    (uint16 bits) [N, K/64] and the LoRA factors (uint16 bits [K, r], [r, N] or
    None).  Returns (bytes uint8 [total], defined uint8 [total]): defined marks the
    bytes the layout specifies (section padding is not)."""
    qW = _c(qW, np.int8); sW = _c(sW, np.uint16)
    N, K = qW.shape
    r = 0 if L_down is None else np.asarray(L_down).reshape(K, -1).shape[1]
    Ld = _c(L_down, np.uint16).reshape(K, r) if r else np.zeros((K, 0), np.uint16)
    Lup = _c(L_up, np.uint16).reshape(r, N) if r else np.zeros((0, N), np.uint16)
    total = packed_offsets(N, K, r)["total"]
    out = np.zeros(total, np.uint8); defined = np.zeros(total, np.uint8)
    _load().oracle_pack_weights_v1(_ptr(qW), _ptr(sW), _ptr(Ld), _ptr(Lup), N, K, r, _ptr(out), _ptr(defined))
    return out, defined


def pack_act_v1(qA, sA, La_f16, r: int):
    """Activation-workspace bytes (layout version 1) of rows m < M: codes int8
    [M, K], fp32 scales [M, K/64], lora_act as fp16 bits uint16 [M, r] (None when
    r == 0).  Returns (bytes, defined) of the minimum workspace size."""
    qA = _c(qA, np.int8); sA = _c(sA, np.float32)
    M, K = qA.shape
    La = _c(La_f16, np.uint16).reshape(M, r) if r else np.zeros((M, 0), np.uint16)
    total = act_offsets(M, K, r)["total"]
    out = np.zeros(total, np.uint8); defined = np.zeros(total, np.uint8)
    _load().oracle_pack_act_v1(_ptr(qA), _ptr(sA), _ptr(La), M, K, r, _ptr(out), _ptr(defined))
    return out, defined
