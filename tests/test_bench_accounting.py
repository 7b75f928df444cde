"""CPU checks of the benchmark's FLOP accounting against the convention it
reports in: pairs = T(T+1)/2, forward = 4 B NH hd pairs, backward = 2.5 x
forward; the per-kernel roofline FLOPs add up to the step's (the dK/dV kernel
4 GEMM units, the dQ kernel 1, the forward 2), and the table's figures for the
two GQA workloads."""
import pytest

import bench
from causal_attention_gqa_gb300.workloads import WORKLOADS


@pytest.mark.parametrize("name,fwd_gflop,bwd_gflop", [
    ("gqa_block", 68.75, 171.88),
    ("long_context_gqa", 549.8, 1374.6),
    ("gpt2_124m_mha", 12.90, 32.24),
])
def test_step_flops_match_the_convention(name, fwd_gflop, bwd_gflop):
    w = WORKLOADS[name]
    pairs = w.T * (w.T + 1) // 2
    assert w.flops_fwd() == 4 * w.B * w.NH * w.hd * pairs
    assert w.flops_bwd() == 2.5 * w.flops_fwd()
    assert bench.flops_per_step(w) == w.flops_fwd() + w.flops_bwd()
    assert abs(w.flops_fwd() / 1e9 - fwd_gflop) < 0.01 * fwd_gflop
    assert abs(w.flops_bwd() / 1e9 - bwd_gflop) < 0.01 * bwd_gflop


def test_kernel_flops_add_up_to_the_step():
    w = WORKLOADS["gqa_block"]
    k = {n: bench.kernel_algorithmic_flops(n, w) for n in ("fwd_tc05", "bwd_dkdv_tc05", "bwd_dq_tc05")}
    assert k["fwd_tc05"] == w.flops_fwd()
    assert k["bwd_dkdv_tc05"] + k["bwd_dq_tc05"] == w.flops_bwd()
    assert sum(k.values()) == bench.flops_per_step(w)
    assert bench.kernel_algorithmic_flops("rope_qk", w) is None     # memory pass: no FLOP roofline


def test_peak_choice_follows_the_length_of_the_timed_region():
    peaks = {"bf16_tflops": 1842.5, "bf16_tflops_sustained": 1679.4}
    tf, desc = bench.choose_peak(peaks, "measured", 0.0064)
    assert tf == 1842.5 and "burst" in desc
    tf, desc = bench.choose_peak(peaks, "measured", 3.0)
    assert tf == 1679.4 and "sustained" in desc


def test_combined_backward_fraction_counts_five_units_over_both_kernels():
    w = WORKLOADS["gqa_block"]
    # per-kernel events: (launches, total ms)
    prof = {"fwd_tc05": (10, 0.665), "bwd_dkdv_tc05": (10, 1.173), "bwd_dq_tc05": (10, 1.128),
            "rope_qk": (10, 0.192)}
    roof, comb = bench.roofline_of(prof, w, 1842.5, "burst")
    assert roof["kernel"] == "bwd_dkdv_tc05"
    assert abs(roof["achieved"] - 4 * 2.0 * w.B * w.NH * w.hd * w.causal_pairs / 0.1173e-3 / 1e12) < 1e-6
    assert comb["algorithmic_flop_per_step"] == w.flops_bwd()
    assert abs(comb["ms"] - 0.2301) < 1e-9
    assert abs(comb["achieved"] - w.flops_bwd() / 0.2301e-3 / 1e12) < 1e-6
    assert abs(comb["frac"] - comb["achieved"] / 1842.5) < 1e-12
