"""GPU parity of attn_qkv_proj (QKV projection with the RoPE rotation in its
epilogue) against the float64 oracle, and the attention run from its rotated
copy (attn_fwd_rot + attn_bwd_rot)."""
import numpy as np
import pytest

import oracle
from causal_attention_gqa_gb300.workloads import make_inputs, make_proj_inputs
from helpers import TOL, rel_err, to_numpy

pytestmark = pytest.mark.gpu


def pair_perm(hd):
    return np.concatenate([np.arange(0, hd, 2), np.arange(1, hd, 2)])


def run_proj(lib, B, T, Cm, NH, NKV, hd, theta, interleaved):
    import torch
    N = (NH + 2 * NKV) * hd
    x_np, w_np = make_proj_inputs(B * T, Cm, N, seed=B * 1000 + T + Cm + NH)
    x = torch.from_numpy(x_np).to("cuda", torch.bfloat16)
    w = torch.from_numpy(w_np).to("cuda", torch.bfloat16)
    qkv, rot = lib.qkv_proj(x, w, T, NH, NKV, theta, rope_interleaved=interleaved)
    torch.cuda.synchronize()
    return x_np, w_np, qkv, rot


@pytest.mark.parametrize("B,T,Cm,NH,NKV,hd,theta,interleaved", [
    (2, 200, 256, 4, 2, 64, 1e4, False),       # M tail (400 rows)
    (1, 300, 1024, 8, 2, 128, 1e6, False),
    (2, 77, 200, 3, 1, 64, 1e4, True),         # K tail (Cm = 200), N tail (N = 320)
    (1, 129, 512, 4, 4, 128, 1e4, True),
    (1, 64, 128, 2, 1, 128, 0.0, False),       # no RoPE: no copy
    (4, 2048, 2048, 16, 4, 128, 1e6, False),   # the GQA block's projection: several tiles per CTA pair
])
def test_qkv_projection_matches_oracle(lib, B, T, Cm, NH, NKV, hd, theta, interleaved):
    x_np, w_np, qkv, rot = run_proj(lib, B, T, Cm, NH, NKV, hd, theta, interleaved)
    ref_qkv, ref_rot = oracle.qkv_projection(x_np, w_np, T, NH, NKV, theta, rope_interleaved=interleaved)
    M, N, NQK = B * T, (NH + 2 * NKV) * hd, (NH + NKV) * hd
    got = to_numpy(qkv).reshape(M, N)
    assert rel_err(got, ref_qkv) <= TOL["bf16"], rel_err(got, ref_qkv)
    if theta > 0:
        import torch
        got_rot = rot[:M * NQK * 2].view(torch.bfloat16).float().cpu().numpy().astype(np.float64).reshape(M, NQK)
        if interleaved:        # the copy keeps each head in NEOX slot order
            p = pair_perm(hd)
            ref_rot = ref_rot.reshape(M, NH + NKV, hd)[..., p].reshape(M, NQK)
        assert rel_err(got_rot, ref_rot) <= TOL["bf16"], rel_err(got_rot, ref_rot)
    else:
        assert rot is None
    assert lib.attn_device_status() == 0


@pytest.mark.parametrize("interleaved", [False, True])
def test_attention_from_the_projection_copy(lib, interleaved):
    """projection -> attn_fwd_rot -> attn_bwd_rot (no rotation pass) against
    the oracle attention of the projected qkv."""
    import torch
    B, T, Cm, NH, NKV, hd, theta = 2, 200, 512, 8, 2, 128, 1e4
    C = NH * hd
    x_np, w_np, qkv, rot = run_proj(lib, B, T, Cm, NH, NKV, hd, theta, interleaved)
    code = lib.DTYPE_BF16 | (lib.FLAG_ROPE_INTERLEAVED if interleaved else 0)
    out = torch.empty((B, T, C), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, NH, T), dtype=torch.float32, device="cuda")
    lib.attn_fwd_rot(out, lse, qkv, rot, B, T, C, NH, NKV, theta, code)
    rng = np.random.default_rng(3)
    dout_np = (rng.standard_normal((B, T, C)) * 1e-2).astype(np.float32)
    dout = torch.from_numpy(dout_np).to("cuda", torch.bfloat16)
    dqkv = lib.backward(qkv, out, dout, lse, NH, NKV, theta, qk_rot=rot, rope_interleaved=interleaved)
    torch.cuda.synchronize()
    qkv_np = to_numpy(qkv)
    dout_ref = to_numpy(dout)
    ref_dqkv, aux = oracle.attention_backward(qkv_np, dout_ref, C, NH, NKV, theta, return_aux=True,
                                              rope_interleaved=interleaved)
    errs = {"out": rel_err(to_numpy(out), aux["out"]), "lse": rel_err(to_numpy(lse), aux["lse"]),
            "dqkv": rel_err(to_numpy(dqkv), ref_dqkv)}
    assert all(v <= TOL["bf16"] for v in errs.values()), errs
    assert lib.attn_device_status() == 0
