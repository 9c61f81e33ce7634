"""Parity at the full sizes of the workloads, in the dispatch the benchmark uses.

Whole-output comparison where the oracle finishes in seconds (single linear,
decoder-layer linears at M = 700, the small-M sweep at K = N = 4096); for the
M = 8192 prefill shapes, whole output rows (every column) at the first and the
last row of every 128-row tile, so that every output tile is compared.
Bit-exact per-group partial sums from the kernel and schedule AUTO runs: the
four decoder-layer linears (whole tiles with the last round split over K in
the same launch, split-K clusters, round-robin tiles), the
small-M sweep at M <= 32 (the tcgen05 small-M kernel), and the stream-K
schedule on the qkv linear.
"""
import numpy as np
import pytest
import torch

import oracle
import w4a4_quantized_gemm_gb300 as w4
from synthetic import DECODER_LAYER_M700, PREFILL, SINGLE_LINEAR, SMALL_M_SWEEP, make_linear_case
from tests.helpers import check_tol, pack, quantize, run_linear, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from w4a4_quantized_gemm_gb300 import build
    build.build()
    w4.lib()


def _full_check(shape, seed, kernel=w4.KERNEL_AUTO):
    c = make_linear_case(seed=seed, **shape)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    Y = run_linear(c, t, packed, ws, kernel)
    y = oracle.linear(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias)
    return check_tol(Y, y, str(shape))


@pytest.mark.parametrize("kernel", [w4.KERNEL_AUTO, w4.KERNEL_TC, w4.KERNEL_SMALLM])
def test_single_linear_m64(kernel):
    _full_check(SINGLE_LINEAR, 0, kernel)


@pytest.mark.parametrize("name", list(DECODER_LAYER_M700))
def test_decoder_layer_linears_m700(name):
    _full_check(DECODER_LAYER_M700[name], list(DECODER_LAYER_M700).index(name))


def _partials_check(shape, seed, stream_k=False):
    c = make_linear_case(seed=seed, **shape)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    was = w4.w4a4_stream_k()
    w4.w4a4_set_stream_k(stream_k)
    try:
        P = w4.w4a4_debug_group_partials(ws, packed, c.M, c.N, c.K, c.r, w4.KERNEL_AUTO)
        dispatch = w4.w4a4_last_dispatch()
    finally:
        w4.w4a4_set_stream_k(was)
    assert w4.w4a4_device_status() == 0
    qA, _ = oracle.quantize_act(c.X)
    qW, _ = oracle.quantize_weights(c.W)
    assert np.array_equal(P.cpu().numpy(), oracle.group_partials(qA, qW)), dispatch
    return dispatch


@pytest.mark.parametrize("name", list(DECODER_LAYER_M700))
def test_decoder_layer_partials_bitexact(name):
    d = _partials_check(DECODER_LAYER_M700[name], list(DECODER_LAYER_M700).index(name))
    assert "gemm_tc" in d
    if name in ("o", "down"):
        assert "split-K=" in d, d  # N = 1024: the cluster split-K schedule
    if name == "qkv":
        assert "split-K=2 in the same launch" in d, d  # 192 tiles: 152 whole, the last 40 split over K


def test_qkv_m700_stream_k_partials_bitexact():
    d = _partials_check(DECODER_LAYER_M700["qkv"], 0, stream_k=True)
    assert "stream-K" in d, d


@pytest.mark.parametrize("shape", [s for s in SMALL_M_SWEEP if s["M"] <= 32], ids=lambda s: f"M{s['M']}")
def test_small_m_partials_bitexact(shape):
    d = _partials_check(shape, shape["M"])
    assert "gemm_smallm_tc" in d, d


@pytest.mark.parametrize("shape", SMALL_M_SWEEP, ids=lambda s: f"M{s['M']}")
def test_small_m_sweep(shape):
    _full_check(shape, shape["M"])


@pytest.mark.parametrize("name", list(PREFILL))
def test_prefill_m8192_every_tile(name):
    s = PREFILL[name]
    c = make_linear_case(seed=5, **s)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    Y = run_linear(c, t, packed, ws, w4.KERNEL_AUTO)
    assert w4.w4a4_device_status() == 0
    # first and last row of every 128-row tile, every column: every (M tile, N tile) pair
    rows = np.unique(np.r_[np.arange(0, c.M, 128), np.minimum(np.arange(127, c.M + 127, 128), c.M - 1)])
    y = oracle.linear_rows(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias, rows)
    Ys = Y[torch.from_numpy(rows).cuda()]
    check_tol(Ys, y, name)
    mt_hit = np.unique(rows // 128)
    assert mt_hit.size == -(-c.M // 128)
    # codes and scales of those rows are bit-exact at full size
    codes, sA, _, _ = w4.w4a4_debug_unpack_act(ws, c.M, c.K, c.r)
    qA, sA_ref = oracle.quantize_act(c.X[rows])
    assert np.array_equal(codes.cpu().numpy()[rows], qA)
    assert np.array_equal(sA.cpu().numpy()[rows], sA_ref)


@pytest.mark.parametrize("M,K,N,r,mode", [(256, 1024, 10240, 32, "inline"), (1280, 1536, 2048, 16, "inline"),
                                            (256, 4096, 10240, 32, "second")], ids=lambda v: str(v))
def test_thin_last_round_runs_split_over_k(M, K, N, r, mode):
    """A last round of tiles that fills at most half the SMs runs split over K after
    the full rounds of whole tiles: in the same launch on clusters of two when the
    tiles are short ("inline"), or as a launch of its own on larger clusters when
    they are long ("second").  Every output tile, on the first and last row of
    every 128-row tile; the group partials of the same schedule bit-exact on those
    rows."""
    expect = "split-K=2 in the same launch" if mode == "inline" else "round-robin, last"
    c = make_linear_case(M, K, N, r, seed=M + N)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    Y = run_linear(c, t, packed, ws, w4.KERNEL_AUTO)
    d = w4.w4a4_last_dispatch()
    assert w4.w4a4_device_status() == 0
    assert expect in d, d
    rows = np.unique(np.r_[np.arange(0, c.M, 128), np.minimum(np.arange(127, c.M + 127, 128), c.M - 1)])
    y = oracle.linear_rows(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias, rows)
    check_tol(Y[torch.from_numpy(rows).cuda()], y, f"thin last round {M}x{K}x{N}")
    P = w4.w4a4_debug_group_partials(ws, packed, M, N, K, r, w4.KERNEL_AUTO)
    assert expect in w4.w4a4_last_dispatch()
    assert w4.w4a4_device_status() == 0
    qA, _ = oracle.quantize_act(c.X[rows])
    qW, _ = oracle.quantize_weights(c.W)
    assert np.array_equal(P[torch.from_numpy(rows).cuda()].cpu().numpy(), oracle.group_partials(qA, qW))
