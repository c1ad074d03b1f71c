"""The bench's choice of roofline per prefill workload: the tensor peak above
the ridge point (burst tensor peak over copy bandwidth), HBM below it, with
the byte floor as the algorithmic bytes."""
import types

import bench

PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _case(flops, nbytes):
    return types.SimpleNamespace(flops=flops, bytes=nbytes, flop_note="test")


def test_byte_floor_counts_q_o_k_v_and_lse():
    # 1 query row of 2 heads (d = 4) against 3 keys of 1 KV head:
    # Q + O = 2 * 1*2*4*2 B, K + V = 2 * 3*1*4*2 B, lse = 1*2*4 B
    assert bench.byte_floor(1, 2, 3, 1, 4) == 32 + 48 + 8


def test_above_ridge_is_tensor_bound():
    ridge = 1900e12 / 6800e9  # about 279 flop per byte
    r = bench.workload_roofline(_case(2 * ridge * 1e9, 1e9), 1.0, PEAKS, "measured", None)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 2 * ridge * 1e9 / 1e-3 / 1e12) < 0.01
    assert abs(r["frac"] - r["achieved"] / 1900.0) < 1e-4


def test_below_ridge_is_hbm_bound():
    # 100 flop per byte: 1 GB in 0.2 ms is 5000 GB/s
    r = bench.workload_roofline(_case(100e9, 1e9), 0.2, PEAKS, "measured", 123)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 5000.0) < 0.1
    assert abs(r["frac"] - 5000.0 / 6800.0) < 1e-4
    assert r["traffic"] == 123


def test_workloads_have_their_expected_bounds():
    ridge = PEAKS["bf16_tflops"] * 1e12 / (PEAKS["hbm_gbs"] * 1e9)
    short = bench.make_case("gqa_short_query_32x32q4kv_16x4096")
    gqa = bench.make_case("gqa_causal_4x32q8kv_4096")
    assert short.flops / short.bytes < ridge < gqa.flops / gqa.bytes
