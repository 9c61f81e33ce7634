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
by one ulp).  In the fused stack the GPU step takes the oracle's fp16 Y_{i-1}
and normalises it itself; its codes and scales must equal those the oracle
computes from its own X_i.  The GPU's own chain is not compared element by element with the
oracle's: a one-ulp difference in an fp16 input legitimately moves a
quantisation code, and the two chains drift apart.
"""
import numpy as np
import pytest
import torch

import oracle
import w4a4_quantized_gemm_gb300 as w4
from synthetic import (STACK_LAYERS, STACK_LINEARS, make_activations, make_linear_case, make_stack_input,
                       make_stack_linear)
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


def _step_checks(stack, i, c, X, Yprev=None, rows=None):
    """Run GPU linear i on the oracle's input for that step (placed in `rows`
    of the GPU buffers, all rows if None): X itself, or in the fused stack the
    oracle's fp16 output Yprev of linear i-1, which the GPU normalises into X.
    Where the stack has a glue kernel after linear i, run it on the oracle's
    fp16 output.  Returns the oracle's next input and its fp16 output."""
    rows_t = slice(None) if rows is None else torch.tensor(rows, device="cuda")
    L = stack.layers[i]
    if stack.reads_previous_output(i):
        stack.layers[i - 1]["Y"][rows_t] = _f16(Yprev)
    else:
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
    if stack.has_glue(i):
        L["Y"][rows_t] = _f16(Yh)
        stack.run_glue(i)
        torch.cuda.synchronize()
        _assert_f16_equal(_bits(stack.next_input(i)[rows_t]), Xn, f"glue {i}")
    return Xn, Yh


@pytest.mark.parametrize("fused", [False, True], ids=["glue_kernel", "fused"])
def test_stack_two_layers_teacher_forced(fused):
    """Eight linears at M = 192 (tensor-core path, a ragged 128-row tile)."""
    from w4a4_quantized_gemm_gb300.stack import W4A4Stack
    M = 192
    linears = [make_stack_linear(l, j) for l in range(2) for j in range(len(STACK_LINEARS))]
    stack = W4A4Stack(linears, M, fused=fused)
    X, Yh = make_stack_input(M), None
    for i, c in enumerate(linears):
        X, Yh = _step_checks(stack, i, c, X, Yh)


@pytest.mark.parametrize("M,ld,K,r", [(37, 6144, 3072, 32), (130, 4096, 2048, 0), (5, 1032, 1024, 128),
                                      (200, 1024, 1024, 16), (11, 10304, 10240, 32), (2053, 6144, 5120, 32)])
def test_fused_rmsnorm_quantize_matches_oracle(M, ld, K, r):
    """The fused kernel on a wider-than-K row stride, ragged row counts, an
    all-zero row and outlier columns: codes and scales bit-exact against the
    oracle's quantiser on the oracle's normalised input, lora_act within the
    fp16 rounding of fp64 X_norm . L_down."""
    rng = np.random.default_rng(5 + K + r)
    Y, _ = make_activations(rng, M, ld)
    Y[min(3, M - 1)] = 0
    c = make_linear_case(M, K, 64, r, seed=K + r)
    Xn = oracle.rmsnorm_f16(Y, K)
    W = torch.from_numpy(c.W).cuda()
    Ld, Lu = _f16(c.L_down), _f16(c.L_up)
    packed = torch.empty(w4.packed_weights_bytes(64, K, r), dtype=torch.uint8, device="cuda")
    w4.w4a4_pack_weights(W, Ld, Lu, packed, r)
    ws = torch.empty(w4.act_workspace_bytes(M, K, r), dtype=torch.uint8, device="cuda")
    w4.w4a4_quantize_act_rmsnorm(_f16(Y), K, packed, ws, r)
    assert "RMSNorm fused" in w4.w4a4_last_dispatch()
    codes, sA, _, lora = w4.w4a4_debug_unpack_act(ws, M, K, r)
    qa, sa = oracle.quantize_act(Xn)
    assert np.array_equal(codes.cpu().numpy(), qa), "codes"
    assert np.array_equal(sA.cpu().numpy(), sa), "scales"
    if r:
        xf = Xn.view(np.float16).astype(np.float64)
        want = xf @ c.L_down.view(np.float16).astype(np.float64)
        got = lora.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - want) <= 1e-3 * (1 + np.abs(want))), "lora_act"


def test_stack_full_size_graph_and_sampled_rows():
    """The 28-layer, M = 700 stack as the benchmark runs it (the RMSNorm fused
    into the activation kernels): the CUDA-graph forward equals the eager one
    bit for bit, the normalised output rows have mean square 1, and two sampled
    rows (the first and the ragged last) are checked step by step against the
    oracle's chain through all 112 linears."""
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
    norms = [stack.out.clone()]
    stack.X0.copy_(_f16(X0))
    stack.forward()
    torch.cuda.synchronize()
    assert torch.equal(stack.out, out_graph), "graph and eager forward differ"
    for x in norms:
        ms = x.float().pow(2).mean(dim=1)
        assert torch.isfinite(x).all() and float((ms - 1).abs().max()) < 2e-3
    rows = [0, M - 1]
    X, Yh = X0[rows], None
    for i in range(len(stack.layers)):
        c = make_stack_linear(i // nl, i % nl)
        X, Yh = _step_checks(stack, i, c, X, Yh, rows)
