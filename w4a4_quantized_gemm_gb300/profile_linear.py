"""Profiling driver: one W4A4 linear of the M=700 decoder layer, called in a loop.

    python -m w4a4_quantized_gemm_gb300.profile_linear <qkv|o|gate_up|down|prefill_up|prefill_down|m1|m4|m16|m32> [iters]
    python -m w4a4_quantized_gemm_gb300.profile_linear norm_gate_up [iters]
    python -m w4a4_quantized_gemm_gb300.profile_linear fwd_<m1|m4|m16|m32> [iters]
    python -m w4a4_quantized_gemm_gb300.profile_linear single [iters]
    python -m w4a4_quantized_gemm_gb300.profile_linear stack [forwards]

`single` is the single linear M=64, K=N=1024.  `stack` builds the 28-layer
stack (112 linears, RMSNorm folded into each next activation kernel) and runs
that many eager forward passes (336 launches each).  The fwd_ forms call
w4a4_forward instead (the whole layer from fp16 X in one
call: the fused small-M kernel up to M = 8).  The norm_gate_up form runs the
stack's RMSNorm glue alone: the gate_up output
[700, 6144] normalised over its first 3072 columns into the down linear's
input, on replicas of the buffers.

Each iteration runs the layer's two kernels (quantize + LoRA down, then GEMM +
LoRA up + affine) on one of R replicas of the inputs, so that consecutive
launches read distinct buffers (the replicas total more than the 129 MB L2
for the M=700 shapes).  Meant to be run under a profiler that captures one
launch after a few warm-up ones (e.g. `-k regex:gemm -s 25 -c 1`).  Prints
one line with the kernel the dispatcher chose.
"""
from __future__ import annotations

import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from synthetic import DECODER_LAYER_M700, SINGLE_LINEAR, make_linear_case  # noqa: E402

SHAPES = dict(DECODER_LAYER_M700)
SHAPES.update({
    "single": dict(SINGLE_LINEAR),
    "prefill_up": dict(M=8192, K=4096, N=14336, r=32),
    "prefill_down": dict(M=8192, K=14336, N=4096, r=32),
    "m1": dict(M=1, K=4096, N=4096, r=32),
    "m4": dict(M=4, K=4096, N=4096, r=32),
    "m16": dict(M=16, K=4096, N=4096, r=32),
    "m32": dict(M=32, K=4096, N=4096, r=32),
})


def main() -> int:
    import torch

    from w4a4_quantized_gemm_gb300 import build as wbuild
    wbuild.build()
    import w4a4_quantized_gemm_gb300 as w4

    name = sys.argv[1] if len(sys.argv) > 1 else "qkv"
    iters = int(sys.argv[2]) if len(sys.argv) > 2 else 30
    if name == "stack":
        from synthetic import STACK_LAYERS, STACK_LINEARS, make_stack_input, make_stack_linear
        from w4a4_quantized_gemm_gb300.stack import W4A4Stack
        dev = torch.device("cuda", 0)
        nl = len(STACK_LINEARS)
        stack = W4A4Stack((make_stack_linear(l, j) for l in range(STACK_LAYERS) for j in range(nl)), 700, dev)
        stack.X0.copy_(torch.from_numpy(make_stack_input(700).view(np.float16).copy()).to(dev))
        for _ in range(iters):
            stack.forward()
        torch.cuda.synchronize()
        print(f"stack: {len(stack.layers)} linears, {stack.launches_per_forward()} launches per forward, "
              f"forwards={iters} status={w4.w4a4_device_status()}")
        return 0
    if name == "norm_gate_up":
        dev = torch.device("cuda", 0)
        g = torch.Generator(device="cpu").manual_seed(0)
        Y0 = (torch.randn(700, 6144, generator=g) * 3).half().to(dev)
        R = 24
        Ys = [Y0.clone() for _ in range(R)]
        Xs = [torch.empty((700, 3072), dtype=torch.float16, device=dev) for _ in range(R)]
        for i in range(iters):
            w4.w4a4_rmsnorm_f16(Ys[i % R], 3072, Xs[i % R])
        torch.cuda.synchronize()
        print(f"{name}: M=700 ld=6144 K=3072 replicas={R} iters={iters} dispatch={w4.w4a4_last_dispatch()}")
        return 0
    fwd = name.startswith("fwd_")
    s = SHAPES[name[4:] if fwd else name]
    M, K, N, r = s["M"], s["K"], s["N"], s["r"]
    c = make_linear_case(M=M, K=K, N=N, r=r, seed=0)
    dev = torch.device("cuda", 0)
    per_rep = N * K // 2 + 2 * M * (K + N)
    R = 1 if per_rep > 256 * 2 ** 20 else max(2, min(24, (300 * 2 ** 20) // per_rep))
    X = torch.from_numpy(c.X.view(np.float16).copy()).to(dev)
    W = torch.from_numpy(c.W).to(dev)
    Ld = torch.from_numpy(c.L_down.view(np.float16).copy()).to(dev)
    Lu = torch.from_numpy(c.L_up.view(np.float16).copy()).to(dev)
    cs = torch.from_numpy(c.colscale.view(np.float16).copy()).to(dev)
    b = torch.from_numpy(c.bias.view(np.float16).copy()).to(dev)
    packed = torch.empty(w4.packed_weights_bytes(N, K, r), dtype=torch.uint8, device=dev)
    w4.w4a4_pack_weights(W, Ld, Lu, packed, r)
    del W
    Xs = [X.clone() for _ in range(R)]
    Ps = [packed.clone() for _ in range(R)]
    WS = [torch.empty(w4.act_workspace_bytes(M, K, r), dtype=torch.uint8, device=dev) for _ in range(R)]
    Ys = [torch.empty((M, N), dtype=torch.float16, device=dev) for _ in range(R)]
    for i in range(iters):
        j = i % R
        if fwd:
            w4.w4a4_forward(Xs[j], Ps[j], cs, b, Ys[j], r, act_ws=WS[j])
        else:
            w4.w4a4_quantize_act(Xs[j], Ps[j], WS[j], r)
            w4.w4a4_linear(WS[j], Ps[j], cs, b, Ys[j], K, r)
    torch.cuda.synchronize()
    print(f"{name}: M={M} K={K} N={N} r={r} replicas={R} iters={iters} dispatch={w4.w4a4_last_dispatch()}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
