"""The C-ABI library builds, loads and exports every declared entry point; host
argument checks reject bad calls before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest
import torch

import w4a4_quantized_gemm_gb300 as w4
from w4a4_quantized_gemm_gb300 import build as wbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a4.h")


@pytest.fixture(scope="module")
def L():
    wbuild.build()
    return w4.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a(?:4|16)_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ("w4a4_pack_weights", "w4a4_quantize_act", "w4a4_linear"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in w4.SIGNATURES, f"binding has no signature for {name}"


def declared_arity():
    """Parameter count of every declared entry point, read off its prototype."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    out = {}
    for m in re.finditer(r"\b(w4a(?:4|16)_[a-z0-9_]+)\s*\(", src):
        depth, i = 1, m.end()
        while depth:
            depth += {"(": 1, ")": -1}.get(src[i], 0)
            i += 1
        params = src[m.end():i - 1].strip()
        if src[i:].lstrip().startswith(";") or src[i:].lstrip().startswith("{"):
            out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header_arity():
    arity = declared_arity()
    assert set(arity) == set(declared_functions())
    for name, n in arity.items():
        assert len(w4.SIGNATURES[name][1]) == n, f"{name}: header {n} parameters, binding {len(w4.SIGNATURES[name][1])}"


def test_size_queries(L):
    G = 1024 // 64
    # packed: L_down first, then codes, scales, L_up; 256-byte aligned sections
    al = lambda x: (x + 255) // 256 * 256
    exp = al(al(al(1024 * 32 * 2) + G * 4096 * 32) + G * 4096 * 2)
    exp = al(exp + 32 * 4096 * 2)
    assert w4.packed_weights_bytes(4096, 1024, 32) == exp
    MT = (700 + 127) // 128
    ws = al(al(al(al(MT * G * 2 * 128 * 32) + MT * G * 128 * 8) + MT * 2 * 128 * 32) + 160 * 16 * 4)
    assert w4.act_workspace_min_bytes(700, 1024, 32) == ws
    # the tcgen05 GEMM's stream-K hand-over area: 160 CTAs x 16 warps x 4 KB, from M = 33 on
    assert w4.act_workspace_bytes(700, 1024, 32) == ws + 160 * 16 * 4096
    assert w4.act_workspace_bytes(32, 1024, 32) == w4.act_workspace_min_bytes(32, 1024, 32)
    assert L.w4a4_packed_weights_bytes(4096, 1000, 32) == 0   # K % 64
    assert L.w4a4_packed_weights_bytes(4100, 1024, 32) == 0   # N % 16
    assert L.w4a4_packed_weights_bytes(4096, 1024, 24) == 0   # r % 16
    assert L.w4a4_packed_weights_bytes(4096, 1024, 144) == 0  # r > 128
    assert L.w4a4_layout_version() == 1


def _vp(x):
    return ctypes.c_void_p(x)


def test_argument_checks_precede_any_launch(L):
    A = _vp(0x10000)  # never dereferenced: every call below fails on the host
    big = 1 << 40
    lin = lambda M, N, K, r, ws=A, pk=A, cs=A, y=A, wsb=big, pkb=big: L.w4a4_linear(
        ws, wsb, pk, pkb, cs, None, M, N, K, r, y, None)
    assert lin(64, 1024, 1000, 32) == 2
    assert lin(64, 1000, 1024, 32) == 2
    assert lin(64, 1024, 1024, 40) == 2
    assert lin(64, 1024, 1024, 256) == 2
    assert lin(-1, 1024, 1024, 32) == 1
    assert lin(0, 1024, 1024, 32) == 0            # M == 0: no-op
    assert lin(64, 1024, 1024, 32, ws=None) == 1
    assert lin(64, 1024, 1024, 32, y=_vp(0x10008)) == 3
    assert lin(64, 1024, 1024, 32, wsb=100) == 4
    assert lin(64, 1024, 1024, 32, pkb=100) == 4
    assert L.w4a4_quantize_act(A, A, big, 64, 100, 32, A, big, None) == 2
    assert L.w4a4_quantize_act(_vp(0x10002), A, big, 64, 128, 32, A, big, None) == 3
    assert L.w4a4_quantize_act(A, A, big, 64, 128, 32, A, 10, None) == 4
    # the activation kernel reads L_down (K r 2 bytes) from the packed buffer
    assert L.w4a4_quantize_act(A, A, 128 * 32 * 2 - 1, 64, 128, 32, A, big, None) == 4
    assert L.w4a4_quantize_act(A, None, 0, 64, 128, 32, A, big, None) == 1   # r > 0 needs L_down
    assert L.w4a4_pack_weights(None, A, A, 64, 128, 32, A, big, None) == 1
    assert L.w4a4_pack_weights(A, None, A, 64, 128, 32, A, big, None) == 1  # r > 0 needs LoRA factors
    assert L.w4a4_linear_select(A, big, A, big, A, None, 64, 1024, 1024, 32, A, 7, None) == 1
    assert L.w4a4_rmsnorm_f16(A, 64, 1024, 1004, A, None) == 2    # K % 8 != 0
    assert L.w4a4_rmsnorm_f16(A, 64, 1000, 1024, A, None) == 1    # ld_y < K
    assert L.w4a4_rmsnorm_f16(A, 64, 1028, 1024, A, None) == 2    # ld_y % 8 != 0
    assert L.w4a4_rmsnorm_f16(_vp(0x10002), 64, 1024, 1024, A, None) == 3
    assert L.w4a4_rmsnorm_f16(A, 0, 1024, 1024, A, None) == 0     # M == 0: no-op
    assert L.w4a4_rmsnorm_f16(A, 4, 16392, 16392, A, None) == 2   # K > 16384
    big = 1 << 40
    assert L.w4a4_quantize_act_rmsnorm(A, 1000, A, big, 64, 1024, 32, A, big, None) == 1  # ld_y < K
    assert L.w4a4_quantize_act_rmsnorm(A, 1028, A, big, 64, 1024, 32, A, big, None) == 2  # ld_y % 8 != 0
    assert L.w4a4_quantize_act_rmsnorm(A, 1024, A, big, 64, 1000, 32, A, big, None) == 2  # K % 64 != 0
    assert L.w4a4_quantize_act_rmsnorm(A, 1024, A, big, 64, 1024, 24, A, big, None) == 2  # r % 16 != 0
    assert L.w4a4_quantize_act_rmsnorm(A, 1024, None, big, 64, 1024, 32, A, big, None) == 1  # r > 0 needs L_down
    assert L.w4a4_quantize_act_rmsnorm(_vp(0x10008), 1024, A, big, 64, 1024, 32, A, big, None) == 3
    assert L.w4a4_quantize_act_rmsnorm(A, 1024, A, big, 64, 1024, 32, A, 16, None) == 4  # workspace too small
    assert L.w4a4_quantize_act_rmsnorm(A, 1024, A, big, 0, 1024, 32, A, big, None) == 0  # M == 0: no-op
    assert L.w4a4_quantize_act_rmsnorm(A, 1024, A, 100, 64, 1024, 32, A, big, None) == 4  # packed below L_down


def test_argument_checks_of_the_variant_entry_points(L):
    """W4A16 (plain and asymmetric), the gate|up packer and SiLU linear, the SVD
    LoRA calls and the allocation-free layer refuse bad calls on the host."""
    A = _vp(0x10000)
    big = 1 << 40
    w16 = lambda M, N, K, r, X=A, y=A, pkb=big: L.w4a16_linear(X, A, pkb, A, None, M, N, K, r, y, None)
    assert w16(4, 1024, 1000, 32) == 2
    assert w16(-1, 1024, 1024, 32) == 1
    assert w16(0, 1024, 1024, 32) == 0
    assert w16(4, 1024, 1024, 32, X=None) == 1
    assert w16(4, 1024, 1024, 32, y=_vp(0x10008)) == 3
    assert w16(4, 1024, 1024, 32, pkb=100) == 4
    wa = lambda M, N, K, r, pkb=big: L.w4a16_linear_asym(A, A, pkb, A, None, M, N, K, r, A, None)
    assert wa(4, 1024, 192, 32) == 2           # K % 128 != 0 (group-128 weights)
    assert wa(-1, 1024, 1024, 32) == 1
    assert wa(0, 1024, 1024, 32) == 0
    assert wa(4, 1024, 1024, 32, pkb=100) == 4
    pa = lambda N, K, r, W=A, pkb=big: L.w4a16_pack_weights_asym(W, A, A, N, K, r, A, pkb, None)
    assert pa(1024, 192, 32) == 2
    assert pa(1024, 1024, 32, W=None) == 1
    assert pa(1024, 1024, 32, W=_vp(0x10004)) == 3
    assert pa(1024, 1024, 32, pkb=100) == 4
    gu = lambda N, K, r, W=A, pkb=big: L.w4a4_pack_weights_gate_up(W, A, A, N, K, r, A, pkb, None)
    assert gu(48, 1024, 32) == 2                # gate|up halves of 16 columns each: N % 32 != 0
    assert gu(1024, 1024, 32, W=None) == 1
    assert gu(1024, 1024, 32, pkb=100) == 4
    sm = lambda M, N, K, r, wsb=big: L.w4a4_linear_silu_mul(A, wsb, A, big, A, None, M, N, K, r, A, None)
    assert sm(64, 48, 1024, 32) == 2
    assert sm(-1, 1024, 1024, 32) == 1
    assert sm(0, 1024, 1024, 32) == 0
    assert sm(64, 1024, 1024, 32, wsb=100) == 4
    sv = lambda r=32, rounds=3, power=8, scratch=A, sb=big, W=A: L.w4a4_pack_weights_svd(
        W, 1024, 1024, r, rounds, power, 7, A, big, A, A, None, scratch, sb, None)
    assert sv(r=0) == 2 and sv(r=8) == 2        # rank below 16, or not a multiple of 16
    assert sv(rounds=0) == 1 and sv(rounds=17) == 1 and sv(power=-1) == 1 and sv(power=65) == 1
    assert sv(scratch=None) == 1
    assert sv(W=_vp(0x10004)) == 3
    assert sv(sb=16) == 4
    ts = lambda r=32, power=8, U=A, sb=big, Amat=A: L.w4a4_truncated_svd(
        Amat, 1024, 1024, r, power, 7, U, A, A, A, sb, None)
    assert ts(r=0) == 2 and ts(power=-1) == 1 and ts(power=65) == 1 and ts(U=None) == 1
    assert ts(Amat=_vp(0x10004)) == 3
    assert ts(sb=16) == 4
    assert L.w4a4_svd_lora_scratch_bytes(1024, 1024, 0) == 0
    assert L.w4a4_svd_lora_scratch_bytes(1024, 1000, 32) == 0
    assert L.w4a4_svd_lora_scratch_bytes(1024, 1024, 32) > 0
    # every check of both steps comes before any launch and before the device check: on a
    # machine without a GPU a bad call gets its own error, never W4A4_ERR_NO_DEVICE
    na = lambda M, N, K, r, X=A, pkb=big, cs=A, y=A, b=None: L.w4a4_linear_noalloc(
        X, A, pkb, cs, b, M, N, K, r, y, None)
    assert na(-1, 1024, 1024, 32) == 1
    assert na(0, 1024, 1024, 32) == 0
    assert na(64, 1024, 1000, 32) == 2 and na(64, 1024, 1024, 24) == 2
    assert na(64, 1000, 1024, 32) == 2 and na(64, 8, 1024, 32) == 2     # N % 16, N < 16
    assert na(64, 1024, 1024, 32, X=None) == 1
    assert na(64, 1024, 1024, 32, X=_vp(0x10004)) == 3
    assert na(64, 1024, 1024, 32, cs=None) == 1                          # null colscale
    assert na(64, 1024, 1024, 32, y=None) == 1
    assert na(64, 1024, 1024, 32, cs=_vp(0x10008)) == 3
    assert na(64, 1024, 1024, 32, b=_vp(0x10008)) == 3
    assert na(64, 1024, 1024, 32, y=_vp(0x10002)) == 3
    assert na(64, 1024, 1024, 32, pkb=w4.packed_weights_bytes(1024, 1024, 32) - 16) == 4  # packed too small
    assert na(8192, 1024, 4096, 32) == 4        # the workspace would not fit the library's array


def test_noalloc_size_limit_is_the_minimum_workspace(L):
    """The array bounds w4a4_act_workspace_min_bytes, not the size with the stream-K area:
    the largest M that fits is accepted up to the device check, the next one refused."""
    A = _vp(0x10000)
    lim = w4.NOALLOC_WORKSPACE_BYTES
    K, N, r = 4096, 1024, 32
    M = 1
    while w4.act_workspace_min_bytes(M + 1, K, r) <= lim:
        M += 1
    assert w4.act_workspace_min_bytes(M, K, r) <= lim < w4.act_workspace_min_bytes(M + 1, K, r)
    assert w4.act_workspace_bytes(M, K, r) > lim  # (the stream-K area alone is 10 MiB)
    call = lambda m: L.w4a4_linear_noalloc(A, A, 1 << 40, A, None, m, N, K, r, A, None)
    assert call(M + 1) == 4
    if not torch.cuda.is_available():
        assert call(M) == 7   # every argument check passed; only the device is missing


def test_stream_k_switch(L):
    before = L.w4a4_stream_k()
    try:
        L.w4a4_set_stream_k(1)
        assert L.w4a4_stream_k() == 1
        L.w4a4_set_stream_k(0)
        assert L.w4a4_stream_k() == 0
    finally:
        L.w4a4_set_stream_k(before)


def test_small_m_threshold_setting(L):
    before = L.w4a4_small_m_threshold()
    assert before >= 0
    try:
        L.w4a4_set_small_m_threshold(16)
        assert L.w4a4_small_m_threshold() == 16
        L.w4a4_set_small_m_threshold(-5)          # negative means never: the tiled kernel for every M
        assert L.w4a4_small_m_threshold() == 0
    finally:
        L.w4a4_set_small_m_threshold(before)
    assert L.w4a4_small_m_threshold() == before


@pytest.mark.skipif(torch.cuda.is_available(), reason="valid shapes would launch on a machine with a GPU")
def test_valid_call_without_device_reports_no_device(L):
    A = _vp(0x10000)
    st = L.w4a4_linear(A, 1 << 40, A, 1 << 40, A, None, 64, 1024, 1024, 32, A, None)
    assert st == 7


def test_status_strings(L):
    for s in range(8):
        assert L.w4a4_status_string(s)
    assert b"unknown" in L.w4a4_status_string(99)
