"""The W4A16 linear (fp16 activations against the packed INT4 weights) against
the CPU oracle: Y within |Y - y| <= 2e-3 (1 + |y|) of the oracle's fp64 y
("INT4 Kernel Architecture, in depth", "W4A16 versus W4A4")."""
import numpy as np
import pytest
import torch

import oracle
import w4a4_quantized_gemm_gb300 as w4
from synthetic import make_linear_case
from tests.helpers import check_tol, pack, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from w4a4_quantized_gemm_gb300 import build
    build.build()
    w4.lib()
    torch.cuda.init()


def _run(c, t, packed, bias=True):
    Y = torch.empty((c.M, c.N), dtype=torch.float16, device="cuda")
    w4.w4a16_linear(t["X"], packed, t["colscale"], t["bias"] if bias else None, Y, c.r)
    torch.cuda.synchronize()
    assert "gemm_w4a16" in w4.w4a4_last_dispatch()
    assert w4.w4a4_device_status() == 0
    return Y


# decode shapes, ragged column tiles, every token-block size, K shares that do not
# divide evenly over the cluster, ranks 0..128, more rows than one token block
@pytest.mark.parametrize("M,N,K,r", [(1, 256, 1024, 32), (5, 48, 192, 16), (16, 400, 832, 32), (33, 144, 448, 0),
                                     (64, 1024, 1024, 128), (70, 96, 256, 32), (1, 4096, 4096, 32),
                                     (32, 4096, 4096, 32), (3, 12800, 1280, 64)])
def test_w4a16_matches_oracle(M, N, K, r):
    c = make_linear_case(M, K, N, r, seed=31 + M + N + K)
    t = to_dev(c)
    packed = pack(c, t)
    Y = _run(c, t, packed)
    y = oracle.w4a16_linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    check_tol(Y, y, f"w4a16 {M}x{N}x{K} r={r}")


def test_w4a16_zero_input_gives_bias_exactly():
    c = make_linear_case(9, 256, 64, 32, seed=5)
    c.X = np.zeros_like(c.X)
    t = to_dev(c)
    Y = _run(c, t, pack(c, t)).cpu().numpy().view(np.uint16)
    assert np.array_equal(Y, np.broadcast_to(c.bias, Y.shape))


def test_w4a16_no_bias_and_determinism():
    c = make_linear_case(12, 512, 96, 32, seed=8)
    t = to_dev(c)
    packed = pack(c, t)
    Y1 = _run(c, t, packed, bias=False)
    Y2 = _run(c, t, packed, bias=False)
    assert torch.equal(Y1, Y2)
    c.bias = np.zeros_like(c.bias)
    check_tol(Y1, oracle.w4a16_linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias), "w4a16 no bias")


def test_w4a16_output_guard_regions_untouched():
    """Y written only inside [M, N] (canaries around the buffer)."""
    M, N, K, r = 11, 80, 192, 16
    c = make_linear_case(M, K, N, r, seed=4)
    t = to_dev(c)
    packed = pack(c, t)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), 0x5A5A, dtype=torch.int16, device="cuda")
    Y = buf[guard:guard + M * N].view(torch.float16).view(M, N)
    w4.w4a16_linear(t["X"], packed, t["colscale"], t["bias"], Y, r)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:guard] == 0x5A5A) and np.all(b[guard + M * N:] == 0x5A5A)
    check_tol(Y, oracle.w4a16_linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias), "w4a16 guarded")


# ---- asymmetric group-128 weights with a zero point ("INT4 Kernel Architecture,
# in depth", "How the weights are stored")
def _pack_asym(c, t):
    packed = torch.empty(w4.packed_weights_bytes(c.N, c.K, c.r), dtype=torch.uint8, device="cuda")
    w4.w4a16_pack_weights_asym(t["W"], t["L_down"], t["L_up"], packed, c.r)
    return packed


@pytest.mark.parametrize("N,K,r", [(16, 128, 0), (48, 384, 16), (4096, 1024, 32)])
def test_pack_asym_bitexact(N, K, r):
    """Codes, fp16 scales and fp16 zero points equal the oracle's bit for bit."""
    c = make_linear_case(1, K, N, r, seed=N + 7 * K)
    c.W[3 % N] = np.abs(c.W[3 % N]) + 0.05   # an all-positive row: negative zero points
    t = to_dev(c)
    packed = _pack_asym(c, t)
    codes, planes, Ld, Lu = w4.w4a4_debug_unpack_weights(packed, N, K, r)
    q, s, z = oracle.quantize_weights_asym(c.W)
    assert np.array_equal(codes.cpu().numpy().astype(np.int16) + 8, q.astype(np.int16))
    pl = planes.cpu().numpy().view(np.uint16)
    assert np.array_equal(pl[:, 0::2], s)
    assert np.array_equal(pl[:, 1::2], z)
    if r:
        assert np.array_equal(Ld.cpu().numpy().view(np.uint16), c.L_down)
        assert np.array_equal(Lu.cpu().numpy().view(np.uint16), c.L_up)


@pytest.mark.parametrize("M,N,K,r", [(1, 256, 1024, 32), (5, 48, 256, 16), (16, 400, 896, 32), (33, 144, 384, 0),
                                     (64, 1024, 1024, 128), (1, 4096, 4096, 32), (32, 4096, 4096, 32)])
def test_w4a16_asym_matches_oracle(M, N, K, r):
    c = make_linear_case(M, K, N, r, seed=41 + M + N + K)
    c.W[1] = np.abs(c.W[1]) + 0.05
    t = to_dev(c)
    packed = _pack_asym(c, t)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    w4.w4a16_linear_asym(t["X"], packed, t["colscale"], t["bias"], Y, r)
    torch.cuda.synchronize()
    assert "asymmetric" in w4.w4a4_last_dispatch(), w4.w4a4_last_dispatch()
    assert w4.w4a4_device_status() == 0
    y = oracle.w4a16_asym_linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    check_tol(Y, y, f"w4a16 asym {M}x{N}x{K} r={r}")


def test_asym_rejects_k_not_multiple_of_128_and_far_zero_points():
    c = make_linear_case(2, 192, 32, 16, seed=3)
    t = to_dev(c)
    packed = torch.empty(w4.packed_weights_bytes(32, 192, 16), dtype=torch.uint8, device="cuda")
    with pytest.raises(w4.W4A4Error):
        w4.w4a16_pack_weights_asym(t["W"], t["L_down"], t["L_up"], packed, 16)
    c = make_linear_case(2, 256, 32, 16, seed=4)
    c.W[0] = 10.0 + np.linspace(0, 1e-3, 256, dtype=np.float32)  # zero point about -1.5e5
    t = to_dev(c)
    packed = torch.empty(w4.packed_weights_bytes(32, 256, 16), dtype=torch.uint8, device="cuda")
    with pytest.raises(w4.W4A4Error):
        w4.w4a16_pack_weights_asym(t["W"], t["L_down"], t["L_up"], packed, 16)
