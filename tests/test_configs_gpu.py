"""Parity at the full sizes of the workloads, in the dispatch the benchmark uses.

Whole-output comparison where the oracle finishes in seconds (single linear,
decoder-layer linears at M = 700, the small-M sweep at K = N = 4096); sampled
outputs for the M = 8192 prefill shapes.  Bit-exact partial sums for the qkv
linear at M = 700.
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


def test_qkv_m700_partials_bitexact():
    s = DECODER_LAYER_M700["qkv"]
    c = make_linear_case(seed=0, **s)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    P = w4.w4a4_debug_group_partials(ws, packed, c.M, c.N, c.K, c.r, w4.KERNEL_TC).cpu().numpy()
    ref = oracle.Reference(c.X, c.W, None, None, c.colscale, c.bias)
    assert np.array_equal(P, oracle.group_partials(ref.qA, ref.qW))


@pytest.mark.parametrize("shape", SMALL_M_SWEEP, ids=lambda s: f"M{s['M']}")
def test_small_m_sweep(shape):
    _full_check(shape, shape["M"])


@pytest.mark.parametrize("name", list(PREFILL))
def test_prefill_m8192_sampled(name):
    s = PREFILL[name]
    c = make_linear_case(seed=5, **s)
    t = to_dev(c)
    packed = pack(c, t)
    ws = quantize(c, t, packed)
    Y = run_linear(c, t, packed, ws, w4.KERNEL_AUTO)
    rng = np.random.default_rng(1)
    rows = np.concatenate([rng.integers(0, c.M, 1500), [0, c.M - 1, 127, 128, 8191]])
    cols = np.concatenate([rng.integers(0, c.N, 1500), [0, c.N - 1, 127, 128, c.N - 128]])
    y = oracle.linear_sampled(c.X, c.W, c.L_down, c.L_up, c.colscale, c.bias, rows, cols)
    Ys = Y[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    check_tol(Ys, y, name)
    # codes of sampled rows are bit-exact at full size
    codes, sA, _, _ = w4.w4a4_debug_unpack_act(ws, c.M, c.K, c.r)
    sel = np.unique(rows[:64])
    qA, sA_ref = oracle.quantize_act(c.X[sel])
    assert np.array_equal(codes.cpu().numpy()[sel], qA)
    assert np.array_equal(sA.cpu().numpy()[sel], sA_ref)
