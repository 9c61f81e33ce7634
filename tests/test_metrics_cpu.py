"""The benchmark's byte and intensity arithmetic against the decode roofline
worked example printed in "INT4 Kernel Architecture, in depth", section "Why
INT4 kernels exist: the roofline" (values in tests/golden)."""
import math
import os

import pytest

from w4a4_quantized_gemm_gb300 import metrics

GOLD = os.path.join(os.path.dirname(__file__), "golden", "int4_roofline_worked_example.txt")


def _load():
    vals = {}
    with open(GOLD) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, value, sig, mode = [p.strip() for p in line.split("|")]
            vals[name] = (float(value), int(sig), mode)
    return vals


def _agrees(x, printed, sig, mode="nearest"):
    """x rounds (or truncates) to the page's figure at the significant figures it prints."""
    e = math.floor(math.log10(abs(printed)))
    unit = 10.0 ** (e - sig + 1)
    if mode == "truncated":
        return printed <= x < printed + unit * (1 + 1e-12)
    return abs(x - printed) <= 0.5 * unit * (1 + 1e-12)


V = _load()


def test_rounding_helper_rejects_a_neighbour():
    assert _agrees(4.806, 4.8, 2) and not _agrees(4.86, 4.8, 2)
    assert _agrees(4.15, 4.1, 2, "truncated") and not _agrees(4.21, 4.1, 2, "truncated") and not _agrees(4.09, 4.1, 2, "truncated")


def test_bits_per_weight_of_group_128_fp16_scales():
    assert metrics.bits_per_weight(128) == V["int4_g128_bits"][0]
    assert metrics.bits_per_weight(64) == 4.25  # the packed format of this library


def test_decode_floors_of_the_8b_model():
    params = V["fp16_weight_bytes"][0] / 2          # the page's fp16 bytes fix the parameter count
    bw = V["hbm_bytes_per_s"][0]
    assert _agrees(params * 2 / bw, *V["fp16_floor_s"])
    # weight_bytes(N, K) of one N x K matrix scales with N K: a single row of `params` weights
    int4 = metrics.weight_bytes(1, params, group=128)
    assert _agrees(int4, *V["int4_g128_weight_bytes"])
    assert _agrees(int4 / bw, *V["int4_g128_floor_s"])
    assert _agrees(int4 / params, *V["bytes_per_weight"])


@pytest.mark.parametrize("M", [1, 4, 16, 32, 76])
def test_intensity_is_about_3_9_m(M):
    assert _agrees(metrics.w4a16_intensity(M, group=128) / M, *V["intensity_per_token"])
    # the same rule for this library's group-64 format: 2 flops per 0.53125 bytes
    assert metrics.w4a16_intensity(M, group=64) == pytest.approx(2 * M / 0.53125, rel=1e-15)


def test_ridge_and_crossover():
    ridge = V["dense_fp16_flops"][0] / V["hbm_bytes_per_s"][0]
    assert _agrees(ridge, *V["ridge_flops_per_byte"])
    assert _agrees(metrics.crossover_m(ridge, group=128), *V["crossover_m"])


# Per-config totals as tabulated from the definition ops = 2MNK + 2Mr(K+N) and
# bytes = codes + fp16 group scales (hand-computed, one line per config).
OPS = {
    (64, 1024, 1024): 142_606_336,
    (700, 4096, 1024): 6_101_401_600,      # qkv (M, N, K)
    (700, 1024, 2048): 3_073_638_400,      # o
    (700, 6144, 1024): 9_129_164_800,      # gate_up
    (700, 1024, 3072): 4_587_520_000,      # down
    (8192, 14336, 4096): 971_736_350_720,  # prefill, gate/up-style
    (8192, 4096, 14336): 971_736_350_720,  # prefill, down-style
}


@pytest.mark.parametrize("MNK,ops", list(OPS.items()))
def test_linear_ops_per_config(MNK, ops):
    assert metrics.linear_ops(*MNK, 32) == ops


def test_workload_totals():
    import bench
    assert bench.layer_ops() == 6_101_401_600 + 3_073_638_400 + 9_129_164_800 + 4_587_520_000
    assert bench.stack_ops() == 640_968_294_400
    assert metrics.weight_bytes(4096, 4096) == 8_912_896     # the small-M sweep's packed weights + scales
    assert metrics.weight_bytes(1024, 1024) == 524_288 + 32_768


def test_bench_traffic_is_tied_to_the_kernel_source_it_was_measured_on():
    """roofline.traffic comes from an ncu capture of a given gemm_tc.cu: reported only while the
    source still hashes to the key it was recorded under, null once the kernel changes."""
    import bench
    key = bench.kernel_source_hash("gemm_tc.cu")
    rec = bench.NCU_TRAFFIC.get((bench.WORKLOAD, key))
    got = bench.ncu_traffic(bench.WORKLOAD)
    if rec is None:
        assert got is None
    else:
        assert got["bytes_per_pass"] == sum(rec["per_linear"].values())
    assert bench.ncu_traffic("no such workload") is None


def test_gemm_launch_count_per_schedule():
    """gpu_launches counts two GEMM launches for a call whose last round of tiles runs in a
    launch of its own, one for every other schedule (the inline split of that round included)."""
    import bench
    second = ("gemm_tc tcgen05.f8f6f4 tile=128x128 groups/job=2 stages=4 tiles=2048: 1976 round-robin, last 72 "
              "split-K=2 (cluster) N-tiles-fastest")
    inline = ("gemm_tc tcgen05.f8f6f4 tile=128x128 groups/job=2 stages=3 tiles=192: 152 whole, last 40 split-K=2 "
              "in the same launch (cluster)")
    plain = "gemm_tc tcgen05.f8f6f4 tile=128x128 groups/job=2 stages=3 split-K=2 (cluster) tiles=48 grid=96"
    assert bench.gemm_launches(second) == 2
    assert bench.gemm_launches(inline) == 1
    assert bench.gemm_launches(plain) == 1
