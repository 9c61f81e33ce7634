"""The decoder-layer stack (four W4A4 + LoRA linears per layer, RMSNorm glue
between them) against the CPU oracle.

The oracle runs its own chain from the seeded input: its fp64 Y rounded to
fp16 ("W4A4 CUDA Kernel for Voice Clone", 3.7: the kernel writes fp16), then
its RMSNorm of the columns the next linear reads (same post, 3.9).  Every GPU
step is checked on the oracle's input for that step -- GPU linear on the
oracle's X_i: codes and scales bit-exact, Y within |Y - y| <= 2e-3 (1 + |y|);
GPU RMSNorm on the oracle's fp16 Y_i: the same fp16 bits as the oracle's
X_{i+1} (both sides use the same fp64 arithmetic; only the order of the fp64
additions differs, which may move a value lying on an fp16 rounding boundary
by one ulp).  The GPU's own chain is not compared element by element with the
oracle's: a one-ulp difference in an fp16 input legitimately moves a
quantisation code, and the two chains drift apart.
"""
import numpy as np
import pytest
import torch

import oracle
import w4a4_quantized_gemm_gb300 as w4
from synthetic import STACK_LAYERS, STACK_LINEARS, make_activations, make_stack_input, make_stack_linear
from tests.helpers import check_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from w4a4_quantized_gemm_gb300 import build
    build.build()
    w4.lib()
    torch.cuda.init()


def _f16(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.float16).copy()).to(dev)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def _assert_f16_equal(got: np.ndarray, want: np.ndarray, what: str):
    ulps = np.abs(got.astype(np.int32) - want.astype(np.int32))
    assert ulps.max() <= 1 and (ulps > 0).sum() <= 1, f"{what}: {(ulps > 0).sum()} elements differ, max {ulps.max()}"


@pytest.mark.parametrize("M,ld,K", [(37, 6144, 3072), (19, 14336, 14336), (5, 1040, 1032)])
def test_rmsnorm_matches_oracle(M, ld, K):
    """Ragged row counts, a row stride wider than K, rows held in registers and
    rows read twice (K > 4096), K not a multiple of 256, an all-zero row, outliers."""
    rng = np.random.default_rng(11 + K)
    Y, _ = make_activations(rng, M, ld)
    Y[min(5, M - 1)] = 0
    X = torch.empty((M, K), dtype=torch.float16, device="cuda")
    w4.w4a4_rmsnorm_f16(_f16(Y), K, X)
    torch.cuda.synchronize()
    _assert_f16_equal(_bits(X), oracle.rmsnorm_f16(Y, K), "rmsnorm")


def _step_checks(stack, i, c, X, rows=None):
    """Run GPU linear i on the oracle's input X (placed in `rows` of the GPU
    buffer, all rows if None) and GPU glue i on the oracle's fp16 output;
    return the oracle's next input."""
    rows_t = slice(None) if rows is None else torch.tensor(rows, device="cuda")
    L = stack.layers[i]
    L["X"][rows_t] = _f16(X)
    stack.run_linear(i)
    torch.cuda.synchronize()
    codes, sA, _, _ = w4.w4a4_debug_unpack_act(L["ws"], stack.M, c.K, c.r)
    qa, sa = oracle.quantize_act(X)
    sel = slice(None) if rows is None else list(rows)
    assert np.array_equal(codes.cpu().numpy()[sel], qa), f"linear {i}: codes"
    assert np.array_equal(sA.cpu().numpy()[sel], sa), f"linear {i}: scales"
    y = oracle.linear(X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    check_tol(L["Y"][rows_t], y, f"linear {i} ({c.name})")
    Yh = oracle.f64_to_f16_array(y)
    Xn = oracle.rmsnorm_f16(Yh, L["k_next"])
    L["Y"][rows_t] = _f16(Yh)
    stack.run_glue(i)
    torch.cuda.synchronize()
    _assert_f16_equal(_bits(stack.next_input(i)[rows_t]), Xn, f"glue {i}")
    return Xn


def test_stack_two_layers_teacher_forced():
    """Eight linears at M = 192 (tensor-core path, a ragged 128-row tile)."""
    from w4a4_quantized_gemm_gb300.stack import W4A4Stack
    M = 192
    linears = [make_stack_linear(l, j) for l in range(2) for j in range(len(STACK_LINEARS))]
    stack = W4A4Stack(linears, M)
    X = make_stack_input(M)
    for i, c in enumerate(linears):
        X = _step_checks(stack, i, c, X)


def test_stack_full_size_graph_and_sampled_rows():
    """The 28-layer, M = 700 stack as the benchmark runs it: the CUDA-graph
    forward equals the eager one bit for bit, every RMSNorm output row has mean
    square 1, and two sampled rows (the first and the ragged last) are checked
    step by step against the oracle's chain through all 112 linears."""
    from w4a4_quantized_gemm_gb300.stack import W4A4Stack
    M = 700
    nl = len(STACK_LINEARS)
    stack = W4A4Stack((make_stack_linear(l, j) for l in range(STACK_LAYERS) for j in range(nl)), M)
    X0 = make_stack_input(M)
    g = stack.capture()
    stack.X0.copy_(_f16(X0))
    g.replay()
    torch.cuda.synchronize()
    out_graph = stack.out.clone()
    norms = [stack.next_input(i).clone() for i in range(0, len(stack.layers), 9)]
    stack.X0.copy_(_f16(X0))
    stack.forward()
    torch.cuda.synchronize()
    assert torch.equal(stack.out, out_graph), "graph and eager forward differ"
    for x in norms:
        ms = x.float().pow(2).mean(dim=1)
        assert torch.isfinite(x).all() and float((ms - 1).abs().max()) < 2e-3
    rows = [0, M - 1]
    X = X0[rows]
    for i in range(len(stack.layers)):
        c = make_stack_linear(i // nl, i % nl)
        X = _step_checks(stack, i, c, X, rows)
