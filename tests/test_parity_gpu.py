"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Bit-exact: weight codes and fp16 scales, activation codes and fp32 scales,
per-group integer partial sums of each GEMM kernel.  Within tolerance
|Y - y| <= 2e-3 (1 + |y|) (y the oracle's fp64 output): the fp16 output.
"""
import numpy as np
import pytest
import torch

import oracle
import w4a4_quantized_gemm_gb300 as w4
from synthetic import make_linear_case, random_codes, random_f16
from tests.helpers import check_tol, pack, quantize, run_linear, to_dev

pytestmark = pytest.mark.gpu

KERNELS = [w4.KERNEL_SMALLM, w4.KERNEL_TC, w4.KERNEL_SMALLM_TC, w4.KERNEL_AUTO]  # every one has a partials dump
YKERNELS = [w4.KERNEL_SMALLM, w4.KERNEL_TC, w4.KERNEL_SMALLM_TC]
KNAMES = {w4.KERNEL_SMALLM: "smallm", w4.KERNEL_TC: "tc", w4.KERNEL_SMALLM_TC: "smallm_tc", w4.KERNEL_AUTO: "auto"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from w4a4_quantized_gemm_gb300 import build
    build.build()
    w4.lib()
    torch.cuda.init()


def _kernel_available(k):
    return True


# ------------------------------------------------------------------ packing
@pytest.mark.parametrize("N,K,r", [(16, 64, 0), (48, 192, 16), (256, 1024, 32), (4096, 1024, 32)])
def test_pack_weights_bitexact(N, K, r):
    c = make_linear_case(1, K, N, r, seed=N + K)
    t = to_dev(c)
    packed = pack(c, t)
    codes, scales, Ld, Lu = w4.w4a4_debug_unpack_weights(packed, N, K, r)
    qW, sW = oracle.quantize_weights(c.W)
    assert np.array_equal(codes.cpu().numpy(), qW)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), sW)
    if r:
        assert np.array_equal(Ld.cpu().numpy().view(np.uint16), c.L_down)
        assert np.array_equal(Lu.cpu().numpy().view(np.uint16), c.L_up)


def test_pack_weight_codes_full_range_roundtrip():
    rng = np.random.default_rng(3)
    N, K, r = 64, 256, 16
    codes = random_codes(rng, (N, K))
    codes[0, :] = -8
    codes[1, :] = 7
    scales = random_f16(rng, (N, K // 64), 1e-3, 1e-2)
    dev = lambda a: torch.from_numpy(a).cuda()
    Ld = dev(random_f16(rng, (K, r), -0.1, 0.1).view(np.float16))
    Lu = dev(random_f16(rng, (r, N), -0.1, 0.1).view(np.float16))
    packed = torch.empty(w4.packed_weights_bytes(N, K, r), dtype=torch.uint8, device="cuda")
    w4.w4a4_pack_weight_codes(dev(codes), dev(scales.view(np.float16)), Ld, Lu, packed, r)
    c2, s2, _, _ = w4.w4a4_debug_unpack_weights(packed, N, K, r)
    assert np.array_equal(c2.cpu().numpy(), codes)
    assert np.array_equal(s2.cpu().numpy().view(np.uint16), scales)


# -------------------------------------------------------- activation kernel
@pytest.mark.parametrize("M,K,r", [(1, 64, 0), (17, 128, 16), (64, 1024, 32), (200, 3072, 32), (33, 512, 128),
                                   (2061, 5120, 32), (2048, 640, 16)])
def test_quantize_act_bitexact(M, K, r):
    """Includes the prefill cluster split (M >= 2048): K in two cluster ranks with
    a ragged last row block, and a single CTA per row block with unequal groups
    per warp."""
    c = make_linear_case(M, K, 32, r, seed=M * 7 + K)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    codes, sA, SA, lora = w4.w4a4_debug_unpack_act(ws, M, K, r)
    qA, sA_ref = oracle.quantize_act(c.X)
    assert np.array_equal(codes.cpu().numpy(), qA)
    assert np.array_equal(sA.cpu().numpy(), sA_ref)
    assert np.array_equal(SA.cpu().numpy(), qA.reshape(M, -1, 64).sum(axis=2).astype(np.float32))
    if r:
        D = oracle.lora_down(c.X, c.L_down)
        # fp32 accumulation + fp16 storage: half an fp16 ulp plus accumulation noise
        err = np.abs(lora.cpu().numpy().astype(np.float64) - D)
        assert np.all(err <= 2.0 ** -11 * np.abs(D) + 1e-5 * (1 + np.abs(D)))


def test_quantize_act_zero_and_outlier_rows():
    M, K = 24, 256
    c = make_linear_case(M, K, 16, 16, seed=1)
    X = c.X.copy()
    X[0, :] = 0                      # all-zero row: scale 1e-10, codes 0
    X[1, :64] = np.float16(60000).view(np.uint16)   # large values
    X[2, 64:128] = np.float16(-3.5).view(np.uint16)
    c.X = X
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    codes, sA, SA, _ = w4.w4a4_debug_unpack_act(ws, M, K, 16)
    qA, sA_ref = oracle.quantize_act(X)
    assert np.array_equal(codes.cpu().numpy(), qA)
    assert np.array_equal(sA.cpu().numpy(), sA_ref)
    assert sA_ref[0, 0] == np.float32(1e-10)


# ------------------------------------------------------------ exact partials
@pytest.mark.parametrize("kernel", KERNELS, ids=lambda k: KNAMES[k])
@pytest.mark.parametrize("M,N,K,r", [(1, 16, 64, 0), (7, 48, 128, 16), (33, 144, 192, 32), (130, 256, 256, 0),
                                     (300, 400, 128, 32), (64, 1024, 1024, 128), (20, 272, 4096, 32)])
def test_group_partials_bitexact(kernel, M, N, K, r):
    """Each kernel's dump comes from the schedule its output would use (split-K
    clusters, ragged tiles, the 3-stage variant at rank 128, the LoRA planes)."""
    c = make_linear_case(M, K, N, r, seed=M + N)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    P = w4.w4a4_debug_group_partials(ws, packed, M, N, K, r, kernel).cpu().numpy()
    assert "partials dump" in w4.w4a4_last_dispatch(), w4.w4a4_last_dispatch()
    ref = oracle.Reference(c.X, c.W, None, None, c.colscale, c.bias)
    assert np.array_equal(P, oracle.group_partials(ref.qA, ref.qW))


@pytest.mark.parametrize("kernel", KERNELS, ids=lambda k: KNAMES[k])
def test_group_partials_extreme_codes(kernel):
    """All -8 x -8 (P = 4096), alternating signs (P = 0) and random full-range codes."""
    rng = np.random.default_rng(9)
    M, N, K = 40, 64, 256
    qW = random_codes(rng, (N, K))
    qW[0, :] = -8
    qW[1, :] = np.tile([7, -8], K // 2)
    sW = random_f16(rng, (N, K // 64), 0.01, 0.02)
    c = make_linear_case(M, K, N, 0, seed=2)
    X = c.X.view(np.float16).copy()
    X[0, :] = -7.0  # codes -7 after quantisation (absmax/7 scale)
    X[1, :] = np.tile(np.float16([3.5, -3.5]), K // 2)
    c.X = X.view(np.uint16)
    t = to_dev(c)
    packed = torch.empty(w4.packed_weights_bytes(N, K, 0), dtype=torch.uint8, device="cuda")
    w4.w4a4_pack_weight_codes(torch.from_numpy(qW).cuda(), torch.from_numpy(sW.view(np.float16)).cuda(),
                              None, None, packed, 0)
    ws = quantize(c, t, packed)
    P = w4.w4a4_debug_group_partials(ws, packed, M, N, K, 0, kernel).cpu().numpy()
    qA, _ = oracle.quantize_act(c.X)
    ref = oracle.group_partials(qA, qW)
    assert ref[0, 0, 0] == 7 * 8 * 64
    assert np.array_equal(P, ref)


# ------------------------------------------------------------------ output Y
SHAPES = [(1, 16, 64, 0), (5, 32, 128, 16), (16, 256, 256, 32), (37, 144, 192, 32), (64, 1024, 1024, 32),
          (129, 272, 320, 32), (200, 512, 512, 64), (300, 128, 1024, 128)]


@pytest.mark.parametrize("kernel", YKERNELS, ids=lambda k: KNAMES[k])
@pytest.mark.parametrize("M,N,K,r", SHAPES)
def test_linear_within_tolerance(kernel, M, N, K, r):
    c = make_linear_case(M, K, N, r, seed=M + 3 * N + K)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    Y = run_linear(c, t, packed, ws, kernel)
    y = oracle.linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    check_tol(Y, y, f"{KNAMES[kernel]} {M}x{N}x{K} r={r}")


@pytest.mark.parametrize("kernel", YKERNELS, ids=lambda k: KNAMES[k])
def test_zero_input_gives_bias_exactly(kernel):
    c = make_linear_case(20, 256, 64, 32, seed=5)
    c.X = np.zeros_like(c.X)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    Y = run_linear(c, t, packed, ws, kernel).cpu().numpy().view(np.uint16)
    assert np.array_equal(Y, np.broadcast_to(c.bias, Y.shape))


@pytest.mark.parametrize("kernel", YKERNELS, ids=lambda k: KNAMES[k])
def test_no_bias_and_determinism(kernel):
    c = make_linear_case(70, 256, 96, 32, seed=8)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    Y1 = run_linear(c, t, packed, ws, kernel, bias=False)
    Y2 = run_linear(c, t, packed, ws, kernel, bias=False)
    assert torch.equal(Y1, Y2)
    c0 = make_linear_case(70, 256, 96, 32, seed=8)
    c0.bias = np.zeros_like(c0.bias)
    y = oracle.linear(c0.X, c0.W, c0.L_down, c0.L_up, c0.colscale, c0.bias)
    check_tol(Y1, y, "no bias")


def test_m_zero_is_noop():
    c = make_linear_case(1, 128, 32, 16, seed=1)
    t = to_dev(c)
    packed = pack(c, t)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    Y = torch.empty((0, 32), dtype=torch.float16, device="cuda")
    w4.w4a4_quantize_act(t["X"][:0], packed, ws, 16)
    w4.w4a4_linear(ws, packed, t["colscale"], t["bias"], Y, 128, 16)


@pytest.mark.parametrize("kernel", YKERNELS, ids=lambda k: KNAMES[k])
def test_output_guard_regions_untouched(kernel):
    """Y written only inside [M, N]: canaries before/after the buffer and the
    columns of a wider row stride stay intact (stand-in for a memory checker)."""
    M, N, K, r = 45, 80, 192, 16
    c = make_linear_case(M, K, N, r, seed=4)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), 0x5A5A, dtype=torch.int16, device="cuda")
    Y = buf[guard:guard + M * N].view(torch.float16).view(M, N)
    w4.w4a4_linear(ws, packed, t["colscale"], t["bias"], Y, K, r, kernel)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:guard] == 0x5A5A) and np.all(b[guard + M * N:] == 0x5A5A)
    y = oracle.linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    check_tol(Y, y, "guarded")


@pytest.mark.parametrize("silu,N", [(False, 512), (False, 528), (True, 512)], ids=["plain", "plain-N528", "silu"])
def test_tiled_store_alignment_same_bits(silu, N):
    """The tiled kernel stores 32 bytes of an output row at a time when the output
    is 32-byte aligned (rows are N x 2 bytes with N a multiple of 16, and N/2 x 2
    bytes with N a multiple of 32 for the SiLU epilogue), else 16 bytes at a
    time: both give the same bits, within tolerance of the oracle, and nothing
    outside the output is written."""
    M, K, r = 200, 256, 32
    c = make_linear_case(M, K, N, r, seed=21 + N)
    t = to_dev(c)
    if silu:
        packed = torch.empty(w4.packed_weights_bytes(N, K, r), dtype=torch.uint8, device="cuda")
        w4.w4a4_pack_weights_gate_up(t["W"], t["L_down"], t["L_up"], packed, r)
    else:
        packed = pack(c, t)
    ws = quantize(c, t, packed)
    cols = N // 2 if silu else N
    outs = []
    for off in (0, 8):  # fp16 elements past a 256-byte aligned base: 0 and 16 bytes
        buf = torch.full((off + M * cols + 64,), 0x5A5A, dtype=torch.int16, device="cuda")
        Y = buf[off:off + M * cols].view(torch.float16).view(M, cols)
        assert (Y.data_ptr() % 32 == 0) == (off == 0)
        if silu:
            w4.w4a4_linear_silu_mul(ws, packed, t["colscale"], t["bias"], Y, K, r)
        else:
            w4.w4a4_linear(ws, packed, t["colscale"], t["bias"], Y, K, r, w4.KERNEL_TC)
        torch.cuda.synchronize()
        assert "gemm_tc" in w4.w4a4_last_dispatch()
        assert w4.w4a4_device_status() == 0
        b = buf.cpu().numpy()
        assert np.all(b[:off] == 0x5A5A) and np.all(b[off + M * cols:] == 0x5A5A)
        outs.append(Y.cpu())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    if silu:
        y = oracle.silu_mul_linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    else:
        y = oracle.linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    check_tol(outs[0], y, "store alignment")


def test_dispatch_is_logged():
    c = make_linear_case(3, 128, 32, 16, seed=1)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    run_linear(c, t, packed, ws, w4.KERNEL_SMALLM)
    assert "gemm_smallm" in w4.w4a4_last_dispatch()


# Small-M kernel with K split over a cluster: uneven group shares (G not a
# multiple of the split), a ragged last column tile (warps without rows), and
# more than one chunk of 8 groups per CTA.
def _expected_split(M, N, K):
    tok = 8 if M <= 8 else 16 if M <= 16 else 32 if M <= 32 else 64
    tiles = -(-N // 128) * -(-M // tok)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ks = 1
    while ks < 8 and tiles * ks * 2 <= 2 * sms and ks * 2 <= K // 64:
        ks *= 2
    return ks


@pytest.mark.parametrize("M,N,K,r", [(3, 400, 832, 32), (40, 144, 448, 16), (2, 48, 4480, 32), (1, 12800, 1280, 32),
                                     (12, 1024, 4096, 64)])
def test_smallm_split_k_cluster(M, N, K, r):
    ks = _expected_split(M, N, K)
    c = make_linear_case(M, K, N, r, seed=M + N + K)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    Y = run_linear(c, t, packed, ws, w4.KERNEL_SMALLM)
    assert f"split-K={ks} " in w4.w4a4_last_dispatch(), w4.w4a4_last_dispatch()
    y = oracle.linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    check_tol(Y, y, f"smallm split {M}x{N}x{K} r={r}")
    assert w4.w4a4_device_status() == 0


# The tcgen05 small-M kernel on the split shapes above, every token-block size
# (16, 32, 64), ragged column tiles, ranks 0..128, more rows than one block.
@pytest.mark.parametrize("M,N,K,r", [(3, 400, 832, 32), (40, 144, 448, 16), (2, 48, 4480, 32), (1, 12800, 1280, 32),
                                     (12, 1024, 4096, 64), (32, 4096, 4096, 32), (64, 1024, 1024, 128),
                                     (70, 96, 256, 32), (17, 272, 320, 0)])
def test_smallm_tc_matches_oracle(M, N, K, r):
    c = make_linear_case(M, K, N, r, seed=M + 2 * N + K)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    Y = run_linear(c, t, packed, ws, w4.KERNEL_SMALLM_TC)
    assert "gemm_smallm_tc" in w4.w4a4_last_dispatch(), w4.w4a4_last_dispatch()
    y = oracle.linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    check_tol(Y, y, f"smallm_tc {M}x{N}x{K} r={r}")
    assert w4.w4a4_device_status() == 0


# The tcgen05 GEMM's stream-K schedule: every CTA takes an equal run of jobs,
# tiles cut between CTAs are finished by the CTA holding their first job.
# Shapes: the layer's qkv and o linears (tiles cut in two and three), a tile cut
# between 32 CTAs (one job each), rank 128 (3-stage variant), a ragged M tail.
@pytest.mark.parametrize("M,N,K,r", [(700, 4096, 1024, 32), (700, 1024, 2048, 32), (129, 256, 4096, 32),
                                     (300, 512, 640, 128), (200, 144, 1024, 16)])
def test_stream_k_matches_oracle(M, N, K, r):
    was = w4.w4a4_stream_k()
    w4.w4a4_set_stream_k(True)
    try:
        _stream_k_case(M, N, K, r)
    finally:
        w4.w4a4_set_stream_k(was)


def _stream_k_case(M, N, K, r):
    c = make_linear_case(M, K, N, r, seed=M + 5 * N + K)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    Y = run_linear(c, t, packed, ws, w4.KERNEL_TC)
    assert "stream-K" in w4.w4a4_last_dispatch(), w4.w4a4_last_dispatch()
    assert w4.w4a4_device_status() == 0
    # oracle on sampled rows (every column) for the large shapes
    rows = np.arange(M) if M * N * K <= 200 * 2 ** 20 else np.unique(np.r_[0, 1, 127, 128, M - 1, np.arange(5, M, 97)])
    rr, cc = np.repeat(rows, N), np.tile(np.arange(N), rows.size)
    y = oracle.linear_sampled(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias, rr, cc).reshape(rows.size, N)
    check_tol(Y.cpu()[rows], y, f"stream-K {M}x{N}x{K} r={r}")
    # a second call on the same workspace finds the flags cleared: the same bits
    Y2 = run_linear(c, t, packed, ws, w4.KERNEL_TC)
    assert torch.equal(Y, Y2)
    # the stream-K schedule's own integer partials, on the sampled rows
    if M * N * K <= 1 << 31:
        P = w4.w4a4_debug_group_partials(ws, packed, M, N, K, r, w4.KERNEL_TC)
        assert "stream-K" in w4.w4a4_last_dispatch() and "partials dump" in w4.w4a4_last_dispatch()
        qA, _ = oracle.quantize_act(c.X[rows])
        qW, _ = oracle.quantize_weights(c.W)
        assert np.array_equal(P.cpu().numpy()[rows], oracle.group_partials(qA, qW))
        assert w4.w4a4_device_status() == 0
    # without the hand-over area the GEMM takes another schedule, within tolerance too
    ws_min = ws[: w4.act_workspace_min_bytes(M, K, r)]
    Y3 = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    w4.w4a4_linear(ws_min, packed, t["colscale"], t["bias"], Y3, K, r, w4.KERNEL_TC)
    torch.cuda.synchronize()
    assert "stream-K" not in w4.w4a4_last_dispatch(), w4.w4a4_last_dispatch()
    check_tol(Y3.cpu()[rows], y, f"round-robin {M}x{N}x{K} r={r}")
    assert w4.w4a4_device_status() == 0


def test_stream_k_wait_runs_out_and_reports_timeout():
    """A bounded wait that can never be satisfied: the stream-K finisher waits for
    its hand-over counters to reach 32, and the test sets them to a value that the
    producers' increments cannot bring there.  The launch must end by itself with
    W4A4_ERR_TIMEOUT in the status word, and the context must stay usable: the
    same linear, re-quantised, then matches the oracle."""
    M, N, K, r = 129, 256, 4096, 32
    was = w4.w4a4_stream_k()
    w4.w4a4_set_stream_k(True)
    try:
        c = make_linear_case(M, K, N, r, seed=77)
        t = to_dev(c)
        packed = pack(c, t)
        ws = quantize(c, t, packed)
        flags_end = w4.act_workspace_min_bytes(M, K, r)
        ws[flags_end - 160 * 16 * 4: flags_end] = 0xFF  # counters at 2^32 - 1: +32 never gives 32
        run_linear(c, t, packed, ws, w4.KERNEL_TC)
        assert "stream-K" in w4.w4a4_last_dispatch(), w4.w4a4_last_dispatch()
        assert w4.w4a4_device_status() == w4.W4A4_ERR_TIMEOUT
        assert w4.w4a4_device_status() == 0  # read and cleared
        ws = quantize(c, t, packed)  # the activation kernel clears the counters
        Y = run_linear(c, t, packed, ws, w4.KERNEL_TC)
        assert w4.w4a4_device_status() == 0
        y = oracle.linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
        check_tol(Y, y, "after a timed-out launch")
    finally:
        w4.w4a4_set_stream_k(was)
