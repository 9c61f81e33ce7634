"""The whole linear from fp16 activations in one call (w4a4_forward), and its
fused small-M kernel: quantisation and LoRA down of X, the exact per-group
products, LoRA up and the affine in one launch ("W4A4 CUDA Kernel for Voice
Clone", 3.6-3.7; "INT4 Kernel Architecture, in depth", "One token versus a
thousand").

Against the oracle, on the fused kernel's own outputs:
  * the codes, sA and SA it writes into the optional workspace: bit-exact;
  * lora_act: within half an fp16 step plus fp32 accumulation noise;
  * the per-group integer partials of its partials variant: bit-exact;
  * Y within 2e-3 (1 + |y|).
The sizes cover the decode sweep at K = N = 4096 (M = 1, 4, 16, 32, the
benchmark's shapes), both token blocks (16 and 32), split factors 1 to 8 with
equal and unequal K slices, a ragged last weight tile, r = 0 and M not a
multiple of 4.  Shapes the fused kernel does not take run the two-call path and
give exactly its bits."""
import numpy as np
import pytest
import torch

import oracle
import w4a4_quantized_gemm_gb300 as w4
from synthetic import SMALL_M_SWEEP, make_linear_case
from tests.helpers import check_tol, pack, quantize, run_linear, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from w4a4_quantized_gemm_gb300 import build
    build.build()
    w4.lib()


DECODE = [(s["M"], s["K"], s["N"], s["r"]) for s in SMALL_M_SWEEP if s["M"] <= 32]
EDGE = [(3, 1024, 2048, 16), (17, 512, 256, 0), (31, 4096, 1024, 32), (8, 192, 48, 16), (32, 64, 16, 16),
        (5, 2048, 400, 32), (1, 128, 4096, 32), (16, 4096, 4096, 0), (29, 320, 1040, 32)]


def _forward(c, t, packed, ws=None, kernel=w4.KERNEL_AUTO):
    Y = torch.full((c.M, c.N), float("nan"), dtype=torch.float16, device="cuda")
    w4.w4a4_forward(t["X"], packed, t["colscale"], t["bias"], Y, c.r, act_ws=ws, kernel=kernel)
    torch.cuda.synchronize()
    assert w4.w4a4_device_status() == 0
    return Y


@pytest.mark.parametrize("M,K,N,r", DECODE + EDGE, ids=lambda v: str(v))
def test_fused_forward_matches_oracle(M, K, N, r):
    c = make_linear_case(M, K, N, r, seed=M * 31 + K + N + r)
    t = to_dev(c)
    packed = pack(c, t)
    assert w4.w4a4_forward_is_fused(M, N, K, r) == (M <= 8)
    ws = torch.zeros(w4.act_workspace_min_bytes(M, K, r), dtype=torch.uint8, device="cuda")
    Y = _forward(c, t, packed, ws, kernel=w4.KERNEL_FUSED)
    assert "linear_fused" in w4.w4a4_last_dispatch()
    assert not torch.isnan(Y.float()).any()
    y = oracle.linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    check_tol(Y, y, f"fused M={M} K={K} N={N} r={r}")
    # codes, scales and SA as written by the fused kernel
    codes, sA, SA, lora = w4.w4a4_debug_unpack_act(ws, M, K, r)
    qA, sA_ref = oracle.quantize_act(c.X)
    assert np.array_equal(codes.cpu().numpy(), qA)
    assert np.array_equal(sA.cpu().numpy(), sA_ref)
    assert np.array_equal(SA.cpu().numpy(), qA.reshape(M, -1, 64).sum(axis=2).astype(np.float32))
    if r:
        D = oracle.lora_down(c.X, c.L_down)
        err = np.abs(lora.cpu().numpy().astype(np.float64) - D)
        assert np.all(err <= 2.0 ** -11 * np.abs(D) + 1e-5 * (1 + np.abs(D)))
    # without the workspace: the same Y bits
    Y2 = _forward(c, t, packed, None, kernel=w4.KERNEL_FUSED)
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))


@pytest.mark.parametrize("M,K,N,r", DECODE + EDGE[:6], ids=lambda v: str(v))
def test_fused_partials_bitexact(M, K, N, r):
    c = make_linear_case(M, K, N, r, seed=M + 3 * K + N)
    t = to_dev(c)
    packed = pack(c, t)
    P = w4.w4a4_debug_forward_partials(t["X"], packed, N, r)
    assert "linear_fused" in w4.w4a4_last_dispatch() and "partials" in w4.w4a4_last_dispatch()
    qA, _ = oracle.quantize_act(c.X)
    qW, _ = oracle.quantize_weights(c.W)
    assert np.array_equal(P.cpu().numpy(), oracle.group_partials(qA, qW))


def test_fused_zero_and_outlier_rows():
    M, K, N, r = 12, 1024, 512, 32
    c = make_linear_case(M, K, N, r, seed=5)
    X = c.X.copy()
    X[0, :] = 0
    X[1, :64] = np.float16(60000).view(np.uint16)
    X[2, 64:128] = np.float16(-3.5).view(np.uint16)
    c.X = X
    t = to_dev(c)
    packed = pack(c, t)
    ws = torch.zeros(w4.act_workspace_min_bytes(M, K, r), dtype=torch.uint8, device="cuda")
    Y = _forward(c, t, packed, ws)
    codes, sA, _, _ = w4.w4a4_debug_unpack_act(ws, M, K, r)
    qA, sA_ref = oracle.quantize_act(X)
    assert np.array_equal(codes.cpu().numpy(), qA)
    assert np.array_equal(sA.cpu().numpy(), sA_ref)
    # row 1's products reach ~1e5 and cancel: fp32 accumulation (the pages' arithmetic)
    # is not within the relative bound there, so that row is only required to be finite
    y = oracle.linear(X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    rows = [m for m in range(M) if m != 1]
    check_tol(Y[rows], y[rows], "zero and outlier rows")
    assert torch.isfinite(Y[1].float()).all()


@pytest.mark.parametrize("M,K,N,r", [(8, 1024, 512, 64), (4, 8192, 1024, 32), (40, 512, 256, 16), (16, 4096, 4096, 32)],
                         ids=lambda v: str(v))
def test_forward_two_call_path_where_auto_does_not_fuse(M, K, N, r):
    c = make_linear_case(M, K, N, r, seed=M + K)
    t = to_dev(c)
    packed = pack(c, t)
    assert not w4.w4a4_forward_is_fused(M, N, K, r)
    ws = torch.empty(w4.act_workspace_min_bytes(M, K, r), dtype=torch.uint8, device="cuda")
    Y = _forward(c, t, packed, ws)
    ws2 = quantize(c, t, packed)
    Y_ref = run_linear(c, t, packed, ws2)
    assert torch.equal(Y.view(torch.int16), Y_ref.view(torch.int16))
    with pytest.raises(w4.W4A4Error) as e:
        _forward(c, t, packed, None)
    assert e.value.status == 1  # W4A4_ERR_INVALID_ARG: the two-call path needs the workspace
    if M > 32 or r > 32 or K > 4096:
        with pytest.raises(w4.W4A4Error) as e:
            _forward(c, t, packed, ws, kernel=w4.KERNEL_FUSED)
        assert e.value.status == 2  # W4A4_ERR_UNSUPPORTED_SHAPE


def test_forward_back_to_back_calls_in_a_graph():
    """Calls in a row on different inputs (the decode benchmark's pattern): each Y
    matches its own call outside the graph bit for bit."""
    M, K, N, r = 4, 4096, 4096, 32
    cases = [make_linear_case(M, K, N, r, seed=s) for s in range(3)]
    ts = [to_dev(c) for c in cases]
    packs = [pack(c, t) for c, t in zip(cases, ts)]
    Ys = [torch.zeros((M, N), dtype=torch.float16, device="cuda") for _ in cases]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for c, t, p, Y in zip(cases, ts, packs, Ys):  # the first call outside any capture
            w4.w4a4_forward(t["X"], p, t["colscale"], t["bias"], Y, r)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    refs = [Y.clone() for Y in Ys]
    for Y in Ys:
        Y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c, t, p, Y in zip(cases, ts, packs, Ys):
            w4.w4a4_forward(t["X"], p, t["colscale"], t["bias"], Y, r)
    g.replay()
    torch.cuda.synchronize()
    assert w4.w4a4_device_status() == 0
    for Y, Yr in zip(Ys, refs):
        assert torch.equal(Y.view(torch.int16), Yr.view(torch.int16))


def test_crafted_ties_codes_both_kernels():
    """Exact rounding ties (tests/golden/act_quant_ties.txt, hand-computed from the
    rule of "W4A4 CUDA Kernel for Voice Clone", 3.6: round to nearest even): the
    activation kernel and the fused kernel give the oracle's codes bit for bit."""
    import os
    gold = os.path.join(os.path.dirname(__file__), "golden", "act_quant_ties.txt")
    groups = []
    for line in open(gold):
        if line.startswith("#") or not line.strip():
            continue
        gid, _, xs, _ = [p.strip() for p in line.split("|")]
        groups.append([float(v) for v in xs.split()])
    K = 64 * 8
    M, N, r = 3, 256, 16
    c = make_linear_case(M, K, N, r, seed=11)
    X = c.X.view(np.float16).astype(np.float32)
    for m in range(M):  # the crafted groups, rotated per row, in the first groups of each row
        for g in range(min(len(groups), K // 64)):
            vals = groups[(g + m) % len(groups)]
            X[m, 64 * g:64 * g + 64] = 0
            X[m, 64 * g:64 * g + len(vals)] = vals
    c.X = X.astype(np.float16).view(np.uint16)
    t = to_dev(c)
    packed = pack(c, t)
    qA, sA_ref = oracle.quantize_act(c.X)
    ws = quantize(c, t, packed)
    codes, sA, _, _ = w4.w4a4_debug_unpack_act(ws, M, K, r)
    assert np.array_equal(codes.cpu().numpy(), qA) and np.array_equal(sA.cpu().numpy(), sA_ref)
    ws2 = torch.zeros(w4.act_workspace_min_bytes(M, K, r), dtype=torch.uint8, device="cuda")
    _forward(c, t, packed, ws2, kernel=w4.KERNEL_FUSED)
    codes2, sA2, _, _ = w4.w4a4_debug_unpack_act(ws2, M, K, r)
    assert np.array_equal(codes2.cpu().numpy(), qA) and np.array_equal(sA2.cpu().numpy(), sA_ref)
