"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle,
element by element on the same seeded inputs.

Bars (normalised max error, max|gpu - oracle| / max|oracle|): 1e-4 for the
float32 path, 2e-2 for the bf16 path, on out, lse and dqkv (and separately
on its dQ, dK, dV blocks).
"""
import numpy as np
import pytest

import oracle
from causal_attention_gqa_gb300.workloads import WORKLOADS, make_inputs, sample_rows, shape_workload
from helpers import TOL, rel_err, run_gpu

pytestmark = pytest.mark.gpu


def check_full(lib, w, dtype, backward=True, fwd_ws=False):
    qkv, dout = make_inputs(w, dtype)
    got = run_gpu(lib, w, qkv, dout, dtype, backward=backward, fwd_ws=fwd_ws)
    tol = TOL[dtype]
    if backward:
        ref_dqkv, aux = oracle.attention_backward(qkv, dout, w.C, w.NH, w.NKV, w.rope_theta, return_aux=True)
        ref_out, ref_lse = aux["out"], aux["lse"]
    else:
        ref_out, ref_lse = oracle.attention_forward(qkv, w.C, w.NH, w.NKV, w.rope_theta)
    errs = {"out": rel_err(got["out"], ref_out), "lse": rel_err(got["lse"], ref_lse)}
    lse_abs = float(np.abs(got["lse"] - ref_lse).max())
    if backward:
        errs["dqkv"] = rel_err(got["dqkv"], ref_dqkv)
        gq, gk, gv = oracle.split_qkv(got["dqkv"], w.C, w.NH, w.NKV)
        rq, rk, rv = oracle.split_qkv(ref_dqkv, w.C, w.NH, w.NKV)
        errs.update(dq=rel_err(gq, rq), dk=rel_err(gk, rk), dv=rel_err(gv, rv))
    assert np.isfinite(got["out"]).all() and np.isfinite(got["lse"]).all()
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{w.name} {dtype}: errors {errs} exceed {tol}"
    assert lse_abs <= tol * max(1.0, float(np.abs(ref_lse).max())), lse_abs
    return errs


# ------------------------------------------------------------------ float32 path
@pytest.mark.parametrize("name", ["microgpt_tiny", "qwen2_single_head"])
def test_f32_tiny_workloads(lib, name):
    check_full(lib, WORKLOADS[name], "f32")


def test_f32_gpt2_mha_full(lib):
    check_full(lib, WORKLOADS["gpt2_124m_mha"], "f32")


@pytest.mark.parametrize("B,T,C,NH,NKV,theta", [
    (1, 1, 16, 4, 4, 0.0), (2, 17, 16, 4, 2, 1e6), (1, 33, 32, 2, 1, 1e4), (3, 95, 64, 4, 1, 0.0),
    (1, 129, 256, 2, 2, 1e6), (2, 70, 96, 3, 1, 0.0), (1, 200, 512, 8, 2, 1e6), (1, 40, 48, 8, 8, 1e6),
])
def test_f32_shapes(lib, B, T, C, NH, NKV, theta):
    check_full(lib, shape_workload(B, T, C, NH, NKV, theta, seed=B * 1000 + T), "f32")


@pytest.mark.parametrize("B,T,C,NH,NKV,theta", [
    # head size 64: the register-tiled float32 kernels (64 x 64 tiles):
    # T = 1, one exact tile, ragged tails, GQA groups of 2 and 3
    (1, 1, 64, 1, 1, 1e6), (1, 64, 64, 1, 1, 0.0), (2, 130, 256, 4, 2, 1e6), (3, 200, 384, 6, 2, 1e4),
])
def test_f32_head64_tiled(lib, B, T, C, NH, NKV, theta):
    check_full(lib, shape_workload(B, T, C, NH, NKV, theta, seed=B * 1000 + T + 17), "f32")


def test_f32_head64_unaligned_tensors(lib):
    """Float32 tensors only 4-byte aligned go to the row-per-warp kernels
    (the tiled ones move 16-byte pieces); both meet the bar."""
    import torch
    from helpers import to_numpy
    w = shape_workload(1, 100, 128, 2, 1, 1e6, seed=41)
    qkv_np, dout_np = make_inputs(w, "f32")

    def shifted(a):
        flat = torch.zeros(a.size + 1, dtype=torch.float32, device="cuda")
        v = flat[1:].view(a.shape)
        v.copy_(torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)))
        return v

    qkv, dout = shifted(qkv_np), shifted(dout_np)
    out = shifted(np.zeros((w.B, w.T, w.C)))
    lse = torch.empty((w.B, w.NH, w.T), dtype=torch.float32, device="cuda")
    dqkv = shifted(np.zeros(qkv_np.shape))
    lib.attn_fwd(out, lse, qkv, w.B, w.T, w.C, w.NH, w.NKV, w.rope_theta, lib.DTYPE_F32)
    nb = lib.attn_bwd_workspace_bytes(w.B, w.T, w.C, w.NH, w.NKV, lib.DTYPE_F32)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    lib.attn_bwd(dqkv, qkv, out, dout, lse, w.B, w.T, w.C, w.NH, w.NKV, w.rope_theta, lib.DTYPE_F32, ws, nb)
    torch.cuda.synchronize()
    ref_dqkv, aux = oracle.attention_backward(qkv_np, dout_np, w.C, w.NH, w.NKV, w.rope_theta, return_aux=True)
    errs = {"out": rel_err(to_numpy(out), aux["out"]), "lse": rel_err(to_numpy(lse), aux["lse"]),
            "dqkv": rel_err(to_numpy(dqkv), ref_dqkv)}
    assert all(v <= TOL["f32"] for v in errs.values()), errs


def test_tf32_forward_without_workspace_runs_the_float32_kernels(lib):
    """attn_fwd takes no workspace, so with ATTN_DTYPE_TF32 it runs the exact
    float32 kernels (the tensor-core path needs scratch for its bf16 parts):
    bit-identical to ATTN_DTYPE_F32, and within the float32 bar."""
    import torch
    from helpers import to_device, to_numpy
    w = shape_workload(2, 70, 128, 2, 1, 1e6, seed=31)
    qkv_np, _ = make_inputs(w, "f32")
    qkv = to_device(qkv_np, "f32")
    res = {}
    for code in (lib.DTYPE_F32, lib.DTYPE_TF32):
        res[code] = lib.forward(qkv, w.NH, w.NKV, w.rope_theta, dtype=code)
    torch.cuda.synchronize()
    for a, b in zip(res[lib.DTYPE_F32], res[lib.DTYPE_TF32]):
        assert torch.equal(a, b)
    out, lse = res[lib.DTYPE_TF32]
    ref_out, ref_lse = oracle.attention_forward(qkv_np, w.C, w.NH, w.NKV, w.rope_theta)
    assert rel_err(to_numpy(out), ref_out) <= TOL["f32"] and rel_err(to_numpy(lse), ref_lse) <= TOL["f32"]


# ------------------------------------------------------------------ bf16 forward
@pytest.mark.parametrize("B,T,C,NH,NKV,theta", [
    (1, 1, 128, 1, 1, 0.0), (1, 128, 128, 1, 1, 0.0), (1, 129, 256, 2, 1, 1e6), (2, 300, 512, 8, 2, 1e6),
    (1, 77, 512, 4, 4, 0.0), (1, 256, 256, 4, 1, 1e4), (2, 513, 1024, 8, 8, 0.0), (1, 1000, 512, 4, 1, 1e6),
])
def test_bf16_forward_shapes(lib, B, T, C, NH, NKV, theta):
    check_full(lib, shape_workload(B, T, C, NH, NKV, theta, seed=B * 1000 + T + 7), "bf16", backward=False)


@pytest.mark.parametrize("B,T,C,NH,NKV,theta", [
    # head size 128 with an even number of query heads per kv head: the
    # paired-head forward kernel (ragged T, T = 1, one tile, several items)
    (2, 385, 1024, 8, 2, 0.0), (1, 1, 256, 2, 1, 0.0), (1, 128, 256, 2, 1, 0.0), (3, 200, 1024, 8, 4, 0.0),
    (1, 700, 2048, 16, 2, 0.0),
    # head size 64, an even number of query heads: heads sharing a kv head,
    # one kv head per query head, and groups of three (a pair can straddle
    # two kv heads)
    (2, 300, 512, 8, 4, 0.0), (1, 200, 256, 4, 4, 0.0), (1, 1, 128, 2, 2, 0.0), (2, 385, 384, 6, 2, 0.0),
    (1, 640, 768, 12, 12, 0.0),
])
def test_bf16_forward_paired_heads(lib, B, T, C, NH, NKV, theta):
    check_full(lib, shape_workload(B, T, C, NH, NKV, theta, seed=B * 1000 + T + 13), "bf16", backward=False)


@pytest.mark.parametrize("B,T,C,NH,NKV,theta", [
    (1, 1, 128, 1, 1, 1e6), (1, 129, 256, 2, 1, 1e6), (2, 300, 512, 8, 2, 1e6), (1, 256, 256, 4, 1, 1e4),
    (1, 1000, 512, 4, 1, 1e6), (1, 77, 512, 4, 4, 0.0), (3, 200, 1024, 8, 4, 1e6),
    # rows a block wide (the prologue's per-group row dot) in four-row groups
    # that run from one batch row into the next
    (3, 101, 2048, 16, 4, 1e6),
])
def test_bf16_forward_workspace_shapes(lib, B, T, C, NH, NKV, theta):
    """attn_fwd_ws (Q/K rotated once into the workspace, then attention) and
    attn_bwd_rot reading that rotated copy."""
    check_full(lib, shape_workload(B, T, C, NH, NKV, theta, seed=B * 1000 + T + 9), "bf16", fwd_ws=True)


@pytest.mark.parametrize("B,T,C,NH,NKV,theta", [
    (1, 1, 128, 1, 1, 0.0), (1, 129, 256, 2, 1, 1e6), (2, 300, 512, 8, 2, 1e6), (1, 77, 512, 4, 4, 0.0),
    (1, 256, 256, 4, 1, 1e4), (1, 640, 1024, 8, 2, 1e6),
    # rows of at least 256 16-byte chunks whose count is not a multiple of 32
    # (the prologue's per-group row dot with a partial last warp)
    (1, 100, 2112, 33, 11, 1e6), (1, 70, 2176, 17, 17, 0.0),
    # the same with four-row groups running into the next batch row
    (2, 70, 2112, 33, 11, 1e6),
])
def test_bf16_backward_shapes(lib, B, T, C, NH, NKV, theta):
    check_full(lib, shape_workload(B, T, C, NH, NKV, theta, seed=B * 1000 + T + 11), "bf16")


def test_bf16_gpt2_mha_reduced_batch(lib):
    w = WORKLOADS["gpt2_124m_mha"].replace(B=2)
    check_full(lib, w, "bf16")


# ------------------------------------------------------------------ full-size, sampled
def check_sampled(lib, w, dtype, n_rows=64, kv_groups=None, fwd_ws=False):
    """Full-size run in the benchmark's launch configuration (fwd_ws: the
    forward through attn_fwd_ws, as bench.py calls it); the oracle is
    evaluated on seeded query rows of every head (out, lse, dQ) and on seeded
    key rows of a few kv groups (dK, dV)."""
    qkv, dout = make_inputs(w, dtype)
    got = run_gpu(lib, w, qkv, dout, dtype, fwd_ws=fwd_ws)
    qr = sample_rows(w.T, n_rows, w.seed + 1)
    kr = sample_rows(w.T, n_rows, w.seed + 2)
    if kv_groups is None:
        kv_groups = [(0, 0), (w.B - 1, w.NKV - 1)]
    ref = oracle.attention_sampled(qkv, dout, w.C, w.NH, w.NKV, w.rope_theta, qr, kv_groups, kr)
    tol = TOL[dtype]
    hd = w.hd
    gq, gk, gv = oracle.split_qkv(got["dqkv"], w.C, w.NH, w.NKV)
    errs = {
        "out": rel_err(got["out"][:, qr], ref["out_rows"]),
        "lse": rel_err(got["lse"][:, :, qr], ref["lse_rows"]),
        "dq": rel_err(gq[:, qr], ref["dq_rows"]),
        "dk": rel_err(np.stack([gk[b, kr, kh] for (b, kh) in kv_groups]),
                      np.stack([ref["dk_rows"][g] for g in kv_groups])),
        "dv": rel_err(np.stack([gv[b, kr, kh] for (b, kh) in kv_groups]),
                      np.stack([ref["dv_rows"][g] for g in kv_groups])),
    }
    for k in ("out", "lse", "dqkv"):
        assert np.isfinite(got[k]).all(), k
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{w.name} {dtype}: errors {errs} exceed {tol}"
    return errs


def test_bf16_gpt2_mha_full_sampled(lib):
    check_sampled(lib, WORKLOADS["gpt2_124m_mha"], "bf16")


def test_bf16_gqa_block_full_sampled(lib):
    check_sampled(lib, WORKLOADS["gqa_block"], "bf16", fwd_ws=True)


def test_bf16_gqa_block_full_sampled_in_kernel_rope(lib):
    check_sampled(lib, WORKLOADS["gqa_block"], "bf16", fwd_ws=False)


def test_bf16_long_context_full_sampled(lib):
    # dK/dV on every kv group (each needs every query row of its four heads
    # in the oracle, a few seconds per group).
    w = WORKLOADS["long_context_gqa"]
    check_sampled(lib, w, "bf16", kv_groups=[(0, kh) for kh in range(w.NKV)], fwd_ws=True)
