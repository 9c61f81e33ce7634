"""Operation and byte counts of the W4A4 + LoRA linear (host-side arithmetic
for the benchmark's throughput and roofline numbers).

Units of work, per linear layer of shape (M, N, K) and LoRA rank r:
  effective ops  = 2 M N K + 2 M r (K + N)     (main GEMM + LoRA down + up)
  weight bytes   = N K / 2 + 2 N K / 64         (4-bit codes + fp16 group scales)
"""
from __future__ import annotations

GROUP = 64


def linear_ops(M: int, N: int, K: int, r: int) -> int:
    return 2 * M * N * K + 2 * M * r * (K + N)


def weight_bytes(N: int, K: int, group: int = GROUP, scale_bytes: int = 2) -> float:
    """Packed 4-bit weights plus one scale per group of `group` input channels."""
    return N * K / 2 + scale_bytes * N * K / group


def bits_per_weight(group: int, scale_bytes: int = 2) -> float:
    return 4 + 8 * scale_bytes / group


def gemm_bytes(M: int, N: int, K: int, r: int) -> int:
    """Algorithmic HBM bytes of one GEMM launch (w4a4_linear): reads packed
    weights, scales, L_up, colscale/bias, the activation workspace (E4M3 codes,
    (sA, SA) per group, fp16 lora_act), writes fp16 Y."""
    G = K // GROUP
    return (N * K // 2 + 2 * N * G + 2 * r * N + 4 * N      # weight side
            + M * K + 8 * M * G + 2 * M * r                  # activation workspace
            + 2 * M * N)                                     # Y


def act_bytes(M: int, K: int, r: int) -> int:
    """Algorithmic HBM bytes of one activation-kernel launch (w4a4_quantize_act)."""
    G = K // GROUP
    return 2 * M * K + 2 * K * r + M * K + 8 * M * G + 2 * M * r


def w4a16_intensity(M: int, group: int = 128, scale_bytes: int = 2) -> float:
    """Decode arithmetic intensity, flops per byte of weight traffic, of a
    4-bit GEMM with M tokens ("INT4 Kernel Architecture, in depth", roofline
    section: about 3.9 M for 4.125-bit weights)."""
    return 2.0 * M / (0.5 + scale_bytes / group)


def crossover_m(ridge_flops_per_byte: float, group: int = 128, scale_bytes: int = 2) -> float:
    """M where the 4-bit GEMM stops being bound by weight bandwidth."""
    return ridge_flops_per_byte / w4a16_intensity(1, group, scale_bytes)


def dense_gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K
