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
