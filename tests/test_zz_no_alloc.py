"""The allocation-free entry point, for callers that cannot allocate device
memory: it must give the same output as the regular two-call path
(w4a4_quantize_act into a caller-allocated workspace, then w4a4_linear), on two
calls in a row whose shapes and data differ (the shared built-in workspace keeps
the previous call's contents), and refuse shapes whose workspace would not fit.

Kept in a file of its own, named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import w4a4_quantized_gemm_gb300 as w4
from synthetic import make_linear_case
from tests.helpers import TOL_REL, pack, quantize, run_linear, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from w4a4_quantized_gemm_gb300 import build
    build.build()
    w4.lib()


def _regular_and_noalloc(M, K, N, r, seed):
    c = make_linear_case(M, K, N, r, seed=seed)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    Y_ref = run_linear(c, t, packed, ws)
    Y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    w4.w4a4_linear_noalloc(t["X"], packed, t["colscale"], t["bias"], Y, r)
    torch.cuda.synchronize()
    return Y_ref.float().cpu().numpy(), Y.float().cpu().numpy()


def test_noalloc_matches_regular_path_two_calls_in_a_row():
    # first call: tensor-core path (M > 64); second: a smaller, different layer on
    # the small-M path, so stale workspace rows from the first call are present
    for (M, K, N, r, seed) in [(300, 1024, 256, 32, 1), (37, 512, 96, 16, 2)]:
        y_ref, y = _regular_and_noalloc(M, K, N, r, seed)
        assert not np.isnan(y).any()
        np.testing.assert_array_less(np.abs(y - y_ref), TOL_REL * (1.0 + np.abs(y_ref)) + 1e-30)


def test_noalloc_rejects_oversized_workspace():
    M, K, N, r = 8192, 4096, 128, 32  # needs ~38 MB of workspace
    assert w4.act_workspace_bytes(M, K, r) > w4.NOALLOC_WORKSPACE_BYTES
    X = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    packed = torch.zeros(w4.packed_weights_bytes(N, K, r), dtype=torch.uint8, device="cuda")
    cs = torch.ones(N, dtype=torch.float16, device="cuda")
    Y = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    with pytest.raises(w4.W4A4Error) as e:
        w4.w4a4_linear_noalloc(X, packed, cs, None, Y, r)
    assert e.value.status == 4  # W4A4_ERR_WORKSPACE
