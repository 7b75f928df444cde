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
