"""Host-side helpers of bench.py (no GPU): the comment-free source
fingerprint that ties the committed ncu traffic figures to the kernel code,
and the algorithmic byte/FLOP accounting."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from serving_moe_route_gb300 import workloads as W  # noqa: E402


def test_strip_c_comments_keeps_code_and_strings():
    src = 'int a = 1; // note\n/* block\n comment */ asm("x // not a comment");\nchar c = \'/\';'
    assert bench.strip_c_comments(src) == 'int a = 1; asm("x // not a comment"); char c = \'/\';'


def test_fingerprint_ignores_comments_only():
    a = "__global__ void k(int* p) { p[0] = 1; }"
    b = "// header\n__global__ void k(int* p) {  /* store */ p[0] = 1; }\n"
    c = "__global__ void k(int* p) { p[0] = 2; }"
    assert bench.strip_c_comments(a) == bench.strip_c_comments(b)
    assert bench.strip_c_comments(a) != bench.strip_c_comments(c)


def test_committed_traffic_matches_current_kernels():
    # the profiles/ncu_traffic.json figures come from the kernels as they
    # stand; after a kernel change without a new capture the bench reports
    # traffic null, and this test says so
    import pytest
    if bench.ncu_traffic("decode_bf16") is None:
        pytest.skip("kernel code changed since the committed ncu traffic capture")
    assert bench.ncu_traffic("decode_bf16") > 1_200_000_000  # the touched weights, read once


def test_algorithmic_accounting_decode():
    wl = W.workloads()["decode_bf16"]
    counts = [8] * wl.E  # every expert touched
    acc = bench.algorithmic(wl, counts)
    assert acc["flops"] == 6.0 * 128 * 8 * 2048 * 768
    assert acc["w13_bytes_per_expert"] == 2 * 768 * 2048 * 2
    assert acc["w2_bytes_per_expert"] == 2048 * 768 * 2
    assert acc["touched"] == 128
    # layer bytes: touched weights + logits + x + out
    assert acc["layer_bytes"] == 128 * (6291456 + 3145728) + 128 * 128 * 2 + 2 * 128 * 2048 * 2


def test_tensor_peak_per_operand_type():
    pk = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "measured"}
    wls = W.workloads()
    assert bench.tensor_peak(wls["decode_bf16"], pk)[0] == 1900.0
    assert bench.tensor_peak(wls["tiny_f32"], pk)[0] == 950.0
    # FP8 without a probe: the nominal 2x ratio, and it says so
    v, src = bench.tensor_peak(wls["fp8_T16"], pk)
    assert v == 3800.0 and "nominal" in src
    pk["fp8_tflops"] = 3500.0
    v, src = bench.tensor_peak(wls["fp8_T16"], pk)
    assert v == 3500.0 and "measured" in src


def test_estimate_ablation_pairs_old_and_new():
    rows = [{"workload": "a", "us_median": 50.0}, {"workload": "a_old_est", "us_median": 100.0},
            {"workload": "b", "us_median": 10.0}]
    ab = bench.estimate_ablation(rows)
    assert list(ab) == ["a"] and ab["a"]["old_over_new"] == 2.0


def test_every_benchmarked_workload_is_a_named_workload():
    # the GPU parity suite runs every named workload on all of its tokens,
    # so nothing the sweep times goes without a parity test
    assert set(bench.SWEEP) <= set(W.workloads())
    assert "decode_bf16" in bench.SWEEP


class _Plan:
    def __init__(self, gemm_pair=0, gemm_tm=0, gemm_dyn=0):
        self.gemm_pair, self.gemm_tm, self.gemm_dyn = gemm_pair, gemm_tm, gemm_dyn


def test_gemm_roofline_attributes_the_launch_that_ran():
    # stage times in ms; acc: GEMM1 and GEMM2 algorithmic bytes and FLOPs
    pk = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "measured"}
    acc = {"g1_bytes": 600e6, "g2_bytes": 300e6, "flops": 3e9}
    wl = W.workloads()["sparse_concentrated_bf16"]
    # a per-call plan that picked CTA pairs: the single-CTA launch (stage
    # 'gemm1') returned at once, both GEMMs ran in stage 'gemm2'
    st = {"gemm1": [0.006], "gemm2": [0.043]}
    name, r = bench.gemm_roofline(wl, st, acc, pk, family=2, plan=_Plan(gemm_dyn=1))
    assert "CTA pairs" in name and r["kernel"].startswith("moe_gemm_pair_kernel")
    assert r["mean_ms"] == 0.043 and r["algorithmic_bytes"] == int(900e6)
    # the same plan when the one-CTA-per-tile family ran (fused, stage 'gemm1')
    st = {"gemm1": [0.55], "gemm2": [0.008]}
    name, r = bench.gemm_roofline(wl, st, acc, pk, family=1, plan=_Plan(gemm_dyn=1))
    assert "fused" in name and r["kernel"].startswith("moe_gemm_kernel")
    assert r["mean_ms"] == 0.55
    # plans that fix the family: the fused launch is recognised by an empty GEMM2 stage
    name, r = bench.gemm_roofline(wl, st, acc, pk, family=None, plan=_Plan())
    assert name == "gemm1+gemm2 fused"
    # FP8 token-major plans name their kernel
    wl8 = W.workloads()["fp8_T4096"]
    st = {"gemm1": [0.176], "gemm2": [0.117]}
    name, r = bench.gemm_roofline(wl8, st, acc, pk, family=None, plan=_Plan(gemm_tm=1))
    assert name == "gemm1" and r["kernel"].startswith("moe_gemm_tm_kernel")
