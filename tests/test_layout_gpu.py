"""The CUDA packer and the CUDA activation kernel write exactly the bytes of the
buffer layout (version 1) that the oracle's own packer produces from the
oracle's codes and scales ("INT4 Kernel Architecture, in depth", "Failure
modes": a wrong packing order is one of the ways these kernels go wrong).

Bit-exact: every byte of the packed weights that the layout defines, and the
code planes, (sA, SA) pairs and stream-K flags of the workspace.  lora_act is
fp16 of an fp32 sum on the GPU and of the fp64 sum in the oracle, so its bytes
are compared as fp16 values within half an fp16 step plus accumulation noise."""
import numpy as np
import pytest
import torch

import oracle
import w4a4_quantized_gemm_gb300 as w4
from synthetic import DECODER_LAYER_M700, make_linear_case
from tests.helpers import pack, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from w4a4_quantized_gemm_gb300 import build
    build.build()
    w4.lib()


SHAPES = [(1, 64, 16, 0), (37, 192, 48, 16), (300, 1024, 256, 32), (130, 512, 96, 128)] + \
    [(s["M"], s["K"], s["N"], s["r"]) for s in DECODER_LAYER_M700.values()]


@pytest.mark.parametrize("M,K,N,r", SHAPES, ids=lambda v: str(v))
def test_packed_weight_bytes_equal_oracle_packer(M, K, N, r):
    c = make_linear_case(M, K, N, r, seed=K + N + r)
    t = to_dev(c)
    packed = pack(c, t).cpu().numpy()
    qW, sW = oracle.quantize_weights(c.W)
    want, defined = oracle.pack_weights_v1(qW, sW, c.L_down if r else None, c.L_up if r else None)
    assert packed.size == want.size
    d = defined == 1
    bad = np.flatnonzero(packed[d] != want[d])
    assert bad.size == 0, f"{bad.size} bytes differ, first at defined byte {bad[:5]}"


@pytest.mark.parametrize("M,K,N,r", SHAPES, ids=lambda v: str(v))
def test_workspace_bytes_equal_oracle_packer(M, K, N, r):
    c = make_linear_case(M, K, N, r, seed=M + K)
    t = to_dev(c)
    packed = pack(c, t)
    ws = torch.empty(w4.act_workspace_min_bytes(M, K, r), dtype=torch.uint8, device="cuda")
    w4.w4a4_quantize_act(t["X"], packed, ws, r)
    got = ws.cpu().numpy()
    off = oracle.act_offsets(M, K, r)
    # code 0 may be stored as E4M3 -0 (0x80: x / sA rounded to -0): the value is
    # what is unique, so the code planes are compared with -0 read as +0
    codes = got[off["qA"]:off["sS"]]
    codes[codes == 0x80] = 0x00
    qA, sA = oracle.quantize_act(c.X)
    D = oracle.lora_down(c.X, c.L_down) if r else None
    La = oracle.f64_to_f16_array(D) if r else None
    want, defined = oracle.pack_act_v1(qA, sA, La, r)
    assert got.size == want.size
    exact = np.zeros(want.size, bool)
    exact[off["qA"]:off["La"]] = True
    exact[off["flags"]:off["total"]] = True
    d = (defined == 1) & exact
    bad = np.flatnonzero(got[d] != want[d])
    assert bad.size == 0, f"{bad.size} code/scale/flag bytes differ"
    if r:
        sl = slice(off["La"], off["flags"])
        dl = defined[sl] == 1
        g16 = got[sl][dl].view(np.float16).astype(np.float64)
        w16 = want[sl][dl].view(np.float16).astype(np.float64)
        assert g16.size == M * r
        assert np.all(np.abs(g16 - w16) <= 2.0 ** -10 * np.abs(w16) + 1e-5)
