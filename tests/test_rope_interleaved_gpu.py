"""GPU parity with the interleaved (GPT-J) RoPE pairing (ATTN_FLAG_ROPE_INTERLEAVED)
against the float64 oracle: the bf16 path through attn_fwd_ws + attn_bwd_rot
(paired-head and single-head forward kernels), through attn_bwd's own
rotation, and through attn_fwd's rotation inside the attention kernel; the
float32 path (row-per-warp and tiled kernels)."""
import numpy as np
import pytest

import oracle
from causal_attention_gqa_gb300.workloads import make_inputs, shape_workload
from helpers import TOL, rel_err, to_device, to_numpy

pytestmark = pytest.mark.gpu


def check(lib, w, dtype, use_rot=True, in_kernel=False):
    import torch
    qkv_np, dout_np = make_inputs(w, dtype)
    qkv, dout = to_device(qkv_np, dtype), to_device(dout_np, dtype)
    if dtype == "bf16" and in_kernel:
        out, lse = lib.forward(qkv, w.NH, w.NKV, w.rope_theta, rope_interleaved=True)   # attn_fwd
        dqkv = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, w.rope_theta, rope_interleaved=True)
    elif dtype == "bf16":
        out, lse, fws = lib.forward_ws(qkv, w.NH, w.NKV, w.rope_theta, rope_interleaved=True)
        dqkv = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, w.rope_theta, qk_rot=fws if use_rot else None,
                            rope_interleaved=True)
    else:
        out, lse = lib.forward(qkv, w.NH, w.NKV, w.rope_theta, rope_interleaved=True)
        dqkv = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, w.rope_theta, rope_interleaved=True)
    torch.cuda.synchronize()
    ref_dqkv, aux = oracle.attention_backward(qkv_np, dout_np, w.C, w.NH, w.NKV, w.rope_theta, return_aux=True,
                                              rope_interleaved=True)
    errs = {"out": rel_err(to_numpy(out), aux["out"]), "lse": rel_err(to_numpy(lse), aux["lse"]),
            "dqkv": rel_err(to_numpy(dqkv), ref_dqkv)}
    assert all(v <= TOL[dtype] for v in errs.values()), errs
    assert lib.attn_device_status() == 0
    return errs


@pytest.mark.parametrize("B,T,C,NH,NKV,theta", [
    (2, 300, 512, 8, 2, 1e4),      # head size 64
    (1, 257, 1024, 8, 4, 1e6),     # head size 128, paired-head forward
    (2, 130, 768, 6, 2, 1e4),      # head size 128, three query heads per kv head
])
def test_bf16_interleaved_through_the_rotated_copy(lib, B, T, C, NH, NKV, theta):
    check(lib, shape_workload(B, T, C, NH, NKV, theta, seed=B * 100 + T + 61), "bf16")


def test_bf16_interleaved_through_attn_bwd_rotation(lib):
    check(lib, shape_workload(2, 200, 1024, 8, 2, 1e4, seed=62), "bf16", use_rot=False)


@pytest.mark.parametrize("B,T,C,NH,NKV,theta", [
    (2, 70, 64, 4, 2, 1e4),        # head size 16, row-per-warp kernels
    (2, 130, 256, 4, 2, 1e4),      # head size 64, tiled kernels
])
def test_f32_interleaved(lib, B, T, C, NH, NKV, theta):
    check(lib, shape_workload(B, T, C, NH, NKV, theta, seed=B * 100 + T + 63), "f32")


@pytest.mark.parametrize("B,T,C,NH,NKV,theta", [
    (2, 300, 512, 8, 2, 1e4),      # head size 64
    (1, 257, 1024, 8, 4, 1e6),     # head size 128
    (1, 1, 256, 2, 1, 1e4),        # one token
])
def test_bf16_interleaved_rotated_inside_the_forward_kernel(lib, B, T, C, NH, NKV, theta):
    """attn_fwd (bf16) rotates each Q tile and every landed K tile in shared
    memory: with the flag it turns each bf16 pair (2i, 2i+1) in place."""
    check(lib, shape_workload(B, T, C, NH, NKV, theta, seed=B * 100 + T + 64), "bf16", in_kernel=True)
