"""Shared helpers for the GPU parity tests: upload a synthetic case, run the
CUDA path through the C ABI, and compare with the oracle."""
import numpy as np
import torch

import w4a4_quantized_gemm_gb300 as w4

TOL_REL = 2e-3  # |Y - y| <= 2e-3 * (1 + |y|), y the oracle's fp64 output


def to_dev(c, device="cuda"):
    t = {}
    t["X"] = torch.from_numpy(c.X.view(np.float16).copy()).to(device)
    t["W"] = torch.from_numpy(c.W.copy()).to(device)
    if c.r:
        t["L_down"] = torch.from_numpy(c.L_down.view(np.float16).copy()).to(device)
        t["L_up"] = torch.from_numpy(c.L_up.view(np.float16).copy()).to(device)
    else:
        t["L_down"] = t["L_up"] = None
    t["colscale"] = torch.from_numpy(c.colscale.view(np.float16).copy()).to(device)
    t["bias"] = torch.from_numpy(c.bias.view(np.float16).copy()).to(device)
    return t


def pack(c, t):
    packed = torch.empty(w4.packed_weights_bytes(c.N, c.K, c.r), dtype=torch.uint8, device="cuda")
    w4.w4a4_pack_weights(t["W"], t["L_down"], t["L_up"], packed, c.r)
    return packed


def quantize(c, t, packed, M=None):
    M = c.M if M is None else M
    ws = torch.empty(max(w4.act_workspace_bytes(M, c.K, c.r), 16), dtype=torch.uint8, device="cuda")
    w4.w4a4_quantize_act(t["X"][:M], packed, ws, c.r)
    return ws


def run_linear(c, t, packed, ws, kernel=w4.KERNEL_AUTO, bias=True):
    Y = torch.full((c.M, c.N), float("nan"), dtype=torch.float16, device="cuda")
    w4.w4a4_linear(ws, packed, t["colscale"], t["bias"] if bias else None, Y, c.K, c.r, kernel)
    torch.cuda.synchronize()
    return Y


def check_tol(Y, y_ref, what=""):
    Yf = Y.float().cpu().numpy().astype(np.float64) if isinstance(Y, torch.Tensor) else np.asarray(Y, np.float64)
    err = np.abs(Yf - y_ref)
    bound = TOL_REL * (1.0 + np.abs(y_ref))
    bad = ~(err <= bound)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst "
                           f"{(err / bound).max():.3f}x bound at {np.unravel_index(np.argmax(err / bound), err.shape)}")
    return float((err / bound).max())
