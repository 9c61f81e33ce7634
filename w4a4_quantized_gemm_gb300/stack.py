"""A stack of W4A4 + LoRA linears with RMSNorm glue (the 28-layer decoder
stack of four linears per layer).

Per linear i: quantise X_i (w4a4_quantize_act), GEMM + LoRA + affine
(w4a4_linear) into Y_i, then RMSNorm of the first K_{i+1} columns of Y_i into
X_{i+1} (w4a4_rmsnorm_f16) -- "W4A4 CUDA Kernel for Voice Clone", 3.4 (the
kernels of one linear) and 3.9 (RMSNorm between the linears).  With
`fused=True` (the default) the norm and the next quantisation are one kernel
(w4a4_quantize_act_rmsnorm reads Y_i directly; X_{i+1} is never written) and
only the last output is normalised by the glue kernel, into `out`.  The module
only allocates device buffers and issues the C-ABI calls, on one stream, and
can capture one forward pass as a CUDA graph ("W4A4 CUDA Kernel for Voice
Clone", 4: CUDA graphs remove the per-kernel launch overhead).
"""
from __future__ import annotations

from typing import Iterable, List

import numpy as np
import torch

import w4a4_quantized_gemm_gb300 as w4


class W4A4Stack:
    def __init__(self, linears: Iterable, M: int, device="cuda", fused: bool = True):
        """`linears`: objects with K, N, r, W (float32 [N, K]), L_down, L_up,
        colscale, bias (fp16 bit arrays), in forward order.  Weights are packed
        on the device one at a time and the fp32 copies dropped."""
        self.M = M
        self.fused = fused
        self.dev = torch.device(device)
        self.layers: List[dict] = []
        lin = list(linears)
        for i, c in enumerate(lin):
            k_next = lin[(i + 1) % len(lin)].K
            W = torch.from_numpy(c.W).to(self.dev)
            Ld = torch.from_numpy(c.L_down.view(np.float16).copy()).to(self.dev)
            Lu = torch.from_numpy(c.L_up.view(np.float16).copy()).to(self.dev)
            packed = torch.empty(w4.packed_weights_bytes(c.N, c.K, c.r), dtype=torch.uint8, device=self.dev)
            w4.w4a4_pack_weights(W, Ld, Lu, packed, c.r)
            del W, Ld, Lu
            self.layers.append(dict(
                K=c.K, N=c.N, r=c.r, k_next=k_next, packed=packed,
                cs=torch.from_numpy(c.colscale.view(np.float16).copy()).to(self.dev),
                b=torch.from_numpy(c.bias.view(np.float16).copy()).to(self.dev),
                X=torch.empty((M, c.K), dtype=torch.float16, device=self.dev),
                ws=torch.empty(w4.act_workspace_bytes(M, c.K, c.r), dtype=torch.uint8, device=self.dev),
                Y=torch.empty((M, c.N), dtype=torch.float16, device=self.dev)))
        self.out = torch.empty((M, lin[0].K), dtype=torch.float16, device=self.dev)
        torch.cuda.synchronize(self.dev)

    @property
    def X0(self) -> torch.Tensor:
        return self.layers[0]["X"]

    def next_input(self, i: int) -> torch.Tensor:
        return self.layers[i + 1]["X"] if i + 1 < len(self.layers) else self.out

    def reads_previous_output(self, i: int) -> bool:
        """Whether linear i takes its input straight from linear i-1's output."""
        return self.fused and i > 0

    def run_linear(self, i: int, stream=None):
        """Quantise layer i's input (fused: normalise linear i-1's output on the
        way in) and run its GEMM."""
        L = self.layers[i]
        if self.reads_previous_output(i):
            w4.w4a4_quantize_act_rmsnorm(self.layers[i - 1]["Y"], L["K"], L["packed"], L["ws"], L["r"], stream)
        else:
            w4.w4a4_quantize_act(L["X"], L["packed"], L["ws"], L["r"], stream)
        w4.w4a4_linear(L["ws"], L["packed"], L["cs"], L["b"], L["Y"], L["K"], L["r"], w4.KERNEL_AUTO, stream)

    def run_glue(self, i: int, stream=None):
        """RMSNorm of layer i's output into the next linear's input (or `out`)."""
        L = self.layers[i]
        w4.w4a4_rmsnorm_f16(L["Y"], L["k_next"], self.next_input(i), stream)

    def has_glue(self, i: int) -> bool:
        return not self.fused or i == len(self.layers) - 1

    def forward(self, stream=None):
        for i in range(len(self.layers)):
            self.run_linear(i, stream)
            if self.has_glue(i):
                self.run_glue(i, stream)

    def capture(self) -> torch.cuda.CUDAGraph:
        """One forward pass as a CUDA graph (warm the kernels up first)."""
        self.forward()
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.forward(torch.cuda.current_stream())
        torch.cuda.synchronize(self.dev)
        return g

    def launches_per_forward(self) -> int:
        return 2 * len(self.layers) + sum(self.has_glue(i) for i in range(len(self.layers)))
