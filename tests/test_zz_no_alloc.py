"""The allocation-free entry point, w4a4_linear_noalloc.

Some callers cannot allocate device memory at all: code running inside an
allocator or a memory-pool callback, a runtime that owns every byte of device
memory, or a plugin interface that only hands over its input and output
buffers.  For them the library quantises X into a fixed workspace array of its
own and runs the GEMM from there.

Checked here, through the C ABI: on calls in a row whose shapes and data differ
(the shared array keeps the previous call's contents), Y has exactly the bits of
the regular two-call path (w4a4_quantize_act into a caller-allocated workspace
of the minimum size, then w4a4_linear: the same kernels on the same workspace
contents), and lies within the oracle's tolerance.  The calls cover the tiled
tcgen05 GEMM, the small-M kernel (M <= 32) and the largest M whose workspace
fits the array; the next M is refused.

Kept in a file of its own, named so that pytest collects it last."""
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


def _largest_m_that_fits(K, r):
    M = 1
    while w4.act_workspace_min_bytes(M + 1, K, r) <= w4.NOALLOC_WORKSPACE_BYTES:
        M += 1
    return M


def _regular_and_noalloc(c, t, packed):
    ws = torch.empty(w4.act_workspace_min_bytes(c.M, c.K, c.r), dtype=torch.uint8, device="cuda")
    w4.w4a4_quantize_act(t["X"], packed, ws, c.r)
    Y_ref = torch.full((c.M, c.N), float("nan"), dtype=torch.float16, device="cuda")
    w4.w4a4_linear(ws, packed, t["colscale"], t["bias"], Y_ref, c.K, c.r)
    Y = torch.full((c.M, c.N), float("nan"), dtype=torch.float16, device="cuda")
    w4.w4a4_linear_noalloc(t["X"], packed, t["colscale"], t["bias"], Y, c.r)
    torch.cuda.synchronize()
    assert w4.w4a4_device_status() == 0
    return Y_ref.cpu(), Y.cpu()


def test_noalloc_matches_regular_path_calls_in_a_row():
    K_big, r_big = 4096, 32
    M_max = _largest_m_that_fits(K_big, r_big)
    # tiled GEMM, then the small-M kernel on a smaller layer (stale rows of the
    # first call stay in the array), then the largest workspace the array holds
    cases = [(300, 1024, 256, 32, 1), (16, 512, 96, 16, 2), (M_max, K_big, 128, r_big, 3)]
    for (M, K, N, r, seed) in cases:
        c = make_linear_case(M, K, N, r, seed=seed)
        t = to_dev(c)
        packed = pack(c, t)
        Y_ref, Y = _regular_and_noalloc(c, t, packed)
        assert not torch.isnan(Y.float()).any()
        assert torch.equal(Y.view(torch.int16), Y_ref.view(torch.int16)), f"M={M}: bits differ from the two-call path"
        if M <= 300:
            y = oracle.linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
            check_tol(Y, y, f"noalloc M={M}")
        else:
            rows = np.array([0, 1, 127, 128, M // 2, M - 2, M - 1])
            cols = np.arange(N)
            rr, cc = np.repeat(rows, N), np.tile(cols, rows.size)
            y = oracle.linear_sampled(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias, rr, cc)
            check_tol(Y.numpy()[rr, cc], y, f"noalloc M={M} sampled rows")


def test_noalloc_refuses_the_first_size_over_the_array():
    K, N, r = 4096, 128, 32
    M = _largest_m_that_fits(K, r) + 1
    assert w4.act_workspace_min_bytes(M, K, r) > w4.NOALLOC_WORKSPACE_BYTES
    X = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    packed = torch.zeros(w4.packed_weights_bytes(N, K, r), dtype=torch.uint8, device="cuda")
    cs = torch.ones(N, dtype=torch.float16, device="cuda")
    Y = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    with pytest.raises(w4.W4A4Error) as e:
        w4.w4a4_linear_noalloc(X, packed, cs, None, Y, r)
    assert e.value.status == 4  # W4A4_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(Y).item() == 0  # nothing was launched
