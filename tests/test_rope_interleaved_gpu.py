"""GPU parity with the interleaved (GPT-J) RoPE pairing (ATTN_FLAG_ROPE_INTERLEAVED)
against the float64 oracle: the bf16 path through attn_fwd_ws + attn_bwd_rot
(paired-head and single-head forward kernels) and through attn_bwd's own
rotation, and the float32 path (row-per-warp and tiled kernels)."""
import numpy as np
import pytest

import oracle
from causal_attention_gqa_gb300.workloads import make_inputs, shape_workload
from helpers import TOL, rel_err, to_device, to_numpy

pytestmark = pytest.mark.gpu


def check(lib, w, dtype, use_rot=True):
    import torch
    qkv_np, dout_np = make_inputs(w, dtype)
    qkv, dout = to_device(qkv_np, dtype), to_device(dout_np, dtype)
    if dtype == "bf16":
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


def test_bf16_attn_fwd_rejects_interleaved(lib):
    """attn_fwd (bf16) rotates inside its attention kernel, NEOX pairs only."""
    import torch
    from causal_attention_gqa_gb300.binding import AttnError
    qkv = torch.zeros((1, 128, 3 * 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((1, 128, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(AttnError) as ei:
        lib.attn_fwd(out, lse, qkv, 1, 128, 128, 1, 1, 1e4, lib.DTYPE_BF16 | lib.FLAG_ROPE_INTERLEAVED)
    assert ei.value.status == -3
    lib.attn_fwd(out, lse, qkv, 1, 128, 128, 1, 1, 0.0, lib.DTYPE_BF16 | lib.FLAG_ROPE_INTERLEAVED)  # no RoPE: ignored
    torch.cuda.synchronize()
