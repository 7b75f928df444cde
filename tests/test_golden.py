"""The stored oracle fixture under tests/golden/ (written by
tests/golden/make_golden.py from the oracle alone).

CPU: the fixture's inputs are the seeded generator's, the oracle still
reproduces the stored values, and the stored values meet facts the
definition fixes on their own (position 0 attends only to itself; the
rotation is the identity at t = 0; the two query heads of the kv group add
their dV).  GPU: the float32 path against the stored values.
"""
import math
import os
import sys

import numpy as np
import pytest

import oracle
from causal_attention_gqa_gb300.workloads import make_inputs, shape_workload
from helpers import TOL, rel_err, run_gpu

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))
import make_golden  # noqa: E402


@pytest.fixture(scope="module")
def golden():
    return make_golden.load()


def test_fixture_inputs_are_the_generators(golden):
    w = shape_workload(**make_golden.CASE)
    qkv, dout = make_inputs(w, "f32")
    assert np.array_equal(golden["qkv"], qkv.astype(np.float64))
    assert np.array_equal(golden["dout"], dout.astype(np.float64))


def test_oracle_reproduces_the_fixture(golden):
    _, arr = make_golden.arrays()
    for name in ("out", "lse", "dqkv"):
        np.testing.assert_allclose(arr[name], golden[name], rtol=1e-12, atol=1e-14)


def test_fixture_meets_the_definition(golden):
    c = make_golden.CASE
    B, T, C, NH, NKV = c["B"], c["T"], c["C"], c["NH"], c["NKV"]
    hd, grp = C // NH, NH // NKV
    Q, K, V = oracle.split_qkv(golden["qkv"], C, NH, NKV)
    out = golden["out"].reshape(B, T, NH, hd)
    _, _, dV = oracle.split_qkv(golden["dqkv"], C, NH, NKV)
    dout = golden["dout"].reshape(B, T, NH, hd)
    for b in range(B):
        for h in range(NH):
            kh = h // grp
            # position 0 sees only itself: its output is V_0 and its lse the
            # scaled score of q_0 with k_0 (no rotation at t = 0)
            np.testing.assert_allclose(out[b, 0, h], V[b, 0, kh], rtol=0, atol=1e-15)
            s00 = float(np.dot(Q[b, 0, h], K[b, 0, kh])) / math.sqrt(hd)
            assert abs(golden["lse"][b, h, 0] - s00) <= 1e-13 * max(1.0, abs(s00))
    # every row's output is a convex combination of the visible value rows
    for b in range(B):
        for t in range(T):
            for h in range(NH):
                vis = V[b, : t + 1, h // grp]
                assert np.all(out[b, t, h] <= vis.max(axis=0) + 1e-12)
                assert np.all(out[b, t, h] >= vis.min(axis=0) - 1e-12)
    # sum over value rows of dV equals the sum of dO over the group's heads
    # and positions (each row's probabilities sum to one)
    for b in range(B):
        for kh in range(NKV):
            got = dV[b, :, kh].sum(axis=0)
            want = dout[b, :, kh * grp:(kh + 1) * grp].sum(axis=(0, 1))
            np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.gpu
def test_gpu_against_the_fixture(lib, golden):
    """The float32 path (head size 4, GQA, RoPE) on the fixture's inputs
    against the stored oracle values, at the float32 bar."""
    w = shape_workload(**make_golden.CASE)
    qkv, dout = make_inputs(w, "f32")
    got = run_gpu(lib, w, qkv, dout, "f32")
    for name in ("out", "lse", "dqkv"):
        err = rel_err(got[name], golden[name])
        assert err <= TOL["f32"], (name, err)
