"""Fused gate|up linear with the SiLU(gate) * up epilogue against the CPU
oracle ("W4A4 CUDA Kernel for Voice Clone", 1: the decoder MLP's
SiLU(gate_proj x) * up_proj x): packed codes, scales and L_up bit-exact in the
documented gate|up row order; H within |H - h| <= 2e-3 (1 + |h|) of the
oracle's fp64 h."""
import numpy as np
import pytest
import torch

import oracle
import w4a4_quantized_gemm_gb300 as w4
from synthetic import make_linear_case
from tests.helpers import check_tol, quantize, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from w4a4_quantized_gemm_gb300 import build
    build.build()
    w4.lib()
    torch.cuda.init()


def _order(N):
    """Original row of each packed row, from the formula in include/w4a4.h."""
    I = N // 2
    p = np.arange(N)
    t, s, w = p // 128, (p % 128) // 32, p % 32
    j = 64 * t + 16 * s + w % 16
    return np.where(w < 16, j, I + j)


def _pack(c, t):
    packed = torch.empty(w4.packed_weights_bytes(c.N, c.K, c.r), dtype=torch.uint8, device="cuda")
    w4.w4a4_pack_weights_gate_up(t["W"], t["L_down"], t["L_up"], packed, c.r)
    return packed


@pytest.mark.parametrize("N,K,r", [(32, 64, 0), (96, 192, 16), (6144, 1024, 32)])
def test_pack_gate_up_order_bitexact(N, K, r):
    c = make_linear_case(1, K, N, r, seed=N + 3 * K)
    t = to_dev(c)
    codes, scales, Ld, Lu = w4.w4a4_debug_unpack_weights(_pack(c, t), N, K, r)
    qW, sW = oracle.quantize_weights(c.W)
    o = _order(N)
    assert sorted(o) == list(range(N))
    assert np.array_equal(codes.cpu().numpy(), qW[o])
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), sW[o])
    if r:
        assert np.array_equal(Ld.cpu().numpy().view(np.uint16), c.L_down)
        assert np.array_equal(Lu.cpu().numpy().view(np.uint16), c.L_up[:, o])


# M <= 32: the tcgen05 weight-streaming kernel (16 and 32 token blocks, a cluster
# split of K); above: every schedule of the tcgen05 tile kernel -- stream-K (with the
# hand-over area), split-K over clusters (a narrow N without it); a partial last
# tile (N/2 = 48), ranks 0..128
@pytest.mark.parametrize("M,N,K,r,minimal_ws", [(1, 64, 128, 16, False), (5, 96, 192, 16, False),
                                                (32, 4096, 1024, 32, False), (64, 256, 256, 32, False),
                                                (37, 96, 192, 0, False), (200, 544, 512, 128, False),
                                                (300, 1024, 2048, 32, True), (700, 6144, 1024, 32, False)])
def test_linear_silu_mul_matches_oracle(M, N, K, r, minimal_ws):
    c = make_linear_case(M, K, N, r, seed=M + N + 11 * K)
    t = to_dev(c)
    packed = _pack(c, t)
    ws = quantize(c, t, packed)
    if minimal_ws:
        ws = ws[: w4.act_workspace_min_bytes(M, K, r)]
    H = torch.full((M, N // 2), float("nan"), dtype=torch.float16, device="cuda")
    w4.w4a4_linear_silu_mul(ws, packed, t["colscale"], t["bias"], H, K, r)
    torch.cuda.synchronize()
    d = w4.w4a4_last_dispatch()
    assert "silu(gate)*up" in d, d
    if minimal_ws:
        assert "split-K" in d and "stream-K" not in d, d
    assert w4.w4a4_device_status() == 0
    if M * N * K <= 200 * 2 ** 20:
        check_tol(H, oracle.silu_mul_linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias), f"silu {M}x{N}x{K}")
    else:
        rows = np.unique(np.r_[0, 127, 128, M - 1, np.arange(3, M, 101)])
        rr, cc = np.repeat(rows, N // 2), np.tile(np.arange(N // 2), rows.size)
        h = oracle.silu_mul_linear_sampled(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias, rr, cc)
        check_tol(H.cpu()[rows], h.reshape(rows.size, N // 2), f"silu {M}x{N}x{K} (sampled rows)")
