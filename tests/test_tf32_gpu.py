"""GPU parity of the float32 tensor-core path (ATTN_DTYPE_TF32, head size 64)
against the float64 oracle, at the float32 bar (1e-4, normalised max error).

The path splits every float32 operand into bf16 parts hi + lo and takes each
product as hi*hi + hi*lo + lo*hi on the tensor cores, with P and dS split the
same way; it runs through attn_fwd_ws and attn_bwd / attn_bwd_rot (the parts
live in the caller's workspace).  The library's per-kernel events show which
kernels ran, so the tests also check that the tensor-core kernels did.
"""
import numpy as np
import pytest

import oracle
from causal_attention_gqa_gb300.workloads import WORKLOADS, make_inputs, shape_workload
from helpers import TOL, rel_err, to_device, to_numpy

pytestmark = pytest.mark.gpu
SPLIT_KERNELS = {"split_prep", "fwd_split", "bwd_dkdv_split", "bwd_dq_split"}


def run_tf32(lib, w, qkv_np, dout_np, interleaved=False, via_rot=False):
    import torch
    qkv, dout = to_device(qkv_np, "f32"), to_device(dout_np, "f32")
    lib.attn_profile_start()
    out, lse, fws = lib.forward_ws(qkv, w.NH, w.NKV, w.rope_theta, dtype=lib.DTYPE_TF32,
                                   rope_interleaved=interleaved)
    dqkv = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, w.rope_theta, dtype=lib.DTYPE_TF32,
                        rope_interleaved=interleaved, qk_rot=fws if via_rot else None)
    torch.cuda.synchronize()
    ran = set(lib.attn_profile_stop())
    assert SPLIT_KERNELS <= ran, ran
    assert lib.attn_device_status() == 0
    return to_numpy(out), to_numpy(lse), to_numpy(dqkv)


def check_tf32(lib, w, interleaved=False, via_rot=False):
    qkv_np, dout_np = make_inputs(w, "f32")
    out, lse, dqkv = run_tf32(lib, w, qkv_np, dout_np, interleaved, via_rot)
    ref_dqkv, aux = oracle.attention_backward(qkv_np, dout_np, w.C, w.NH, w.NKV, w.rope_theta,
                                              rope_interleaved=interleaved, return_aux=True)
    errs = {"out": rel_err(out, aux["out"]), "lse": rel_err(lse, aux["lse"]), "dqkv": rel_err(dqkv, ref_dqkv)}
    gq, gk, gv = oracle.split_qkv(dqkv, w.C, w.NH, w.NKV)
    rq, rk, rv = oracle.split_qkv(ref_dqkv, w.C, w.NH, w.NKV)
    errs.update(dq=rel_err(gq, rq), dk=rel_err(gk, rk), dv=rel_err(gv, rv))
    assert np.isfinite(out).all() and np.isfinite(dqkv).all()
    bad = {k: v for k, v in errs.items() if not v <= TOL["f32"]}
    assert not bad, f"{w.name}: errors {errs} exceed {TOL['f32']}"
    return errs


@pytest.mark.parametrize("B,T,C,NH,NKV,theta", [
    (1, 1, 64, 1, 1, 0.0),            # one token
    (2, 70, 128, 2, 1, 1e6),          # ragged tile, two query heads per kv head, RoPE
    (1, 300, 256, 4, 4, 0.0),         # three query tiles, MHA
    (1, 257, 512, 8, 2, 1e4),         # one row past two tiles, grp 4
    (2, 129, 384, 6, 3, 1e6),
])
def test_tf32_tensor_path_shapes(lib, B, T, C, NH, NKV, theta):
    check_tf32(lib, shape_workload(B, T, C, NH, NKV, theta, seed=B * 1000 + T + 5))


def test_tf32_tensor_path_interleaved_rope_and_rot_entry(lib):
    check_tf32(lib, shape_workload(1, 200, 256, 4, 2, 1e4, seed=77), interleaved=True, via_rot=True)


def test_tf32_gpt2_mha_full(lib):
    """The GPT-2-shaped workload (B=8, T=1024, C=768, NH=NKV=12, head size 64)
    in float32, whole tensors against the oracle."""
    errs = check_tf32(lib, WORKLOADS["gpt2_124m_mha"])
    assert max(errs.values()) <= TOL["f32"]


def test_tf32_backward_is_deterministic(lib):
    import torch
    w = shape_workload(2, 300, 256, 4, 2, 1e6, seed=9)
    qkv_np, dout_np = make_inputs(w, "f32")
    qkv, dout = to_device(qkv_np, "f32"), to_device(dout_np, "f32")
    out, lse, _ = lib.forward_ws(qkv, w.NH, w.NKV, w.rope_theta, dtype=lib.DTYPE_TF32)
    a = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, w.rope_theta, dtype=lib.DTYPE_TF32)
    b = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, w.rope_theta, dtype=lib.DTYPE_TF32)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
