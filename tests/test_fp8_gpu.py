"""GPU check of the e4m3 (FP8) forward (attn_fwd_fp8) against the float64
oracle on the original inputs.

Bars, from the e4m3 rounding model (3 mantissa bits: a value scaled into the
e4m3 range is rounded with a relative error of at most 2^-4):
  * out: out = sum_j P_j V_j / l with every P_j and every V element rounded,
    so |out - ref| <= (2^-4 + 2^-4 + 2^-8) max|V| = 0.129 max|V| from those
    two roundings (rows that see a single key reach it: out = the rounded
    V_0), plus the absolute error of weights in the e4m3 subnormal range.
    The kernel stores 112 p (p = 2^(s - m) <= 4 with a lazily renewed row
    maximum m), so a weight with 112 p < 2^-6 is off by at most 2^-10 / 112,
    and l >= 1: at most T 2^-10 / 112 max|V| over a row.
  * lse: the scores s = q . k / sqrt(hd) inherit the rounding of Q and K;
    its worst case (all 128 products rounded the same way) is far larger
    than what random inputs show, so the bar, 0.1 max(1, max|lse|), is an
    empirical margin over the measured ~0.01 relative error.
"""
import numpy as np
import pytest

import oracle
from causal_attention_gqa_gb300.workloads import WORKLOADS, make_inputs, sample_rows, shape_workload
from helpers import rel_err, to_device, to_numpy

pytestmark = pytest.mark.gpu
P_SUBNORMAL = 2.0 ** -10 / 112.0     # absolute error of one stored weight below the normal range


def out_bar(T):   # times max|V|
    return 2.0 ** -4 + 2.0 ** -4 + 2.0 ** -8 + T * P_SUBNORMAL
LSE_BAR = 0.1      # times max(1, max|lse|)


@pytest.mark.parametrize("B,T,C,NH,NKV,theta,interleaved", [
    (2, 300, 1024, 8, 2, 1e6, False),
    (1, 257, 2048, 16, 4, 1e4, True),
    (1, 128, 256, 2, 1, 0.0, False),
    (1, 1, 256, 2, 1, 1e6, False),
])
def test_fp8_forward_within_bar(lib, B, T, C, NH, NKV, theta, interleaved):
    import torch
    w = shape_workload(B, T, C, NH, NKV, theta, seed=B * 100 + T + 71)
    qkv_np, _ = make_inputs(w, "bf16")
    qkv = to_device(qkv_np, "bf16")
    out, lse = lib.forward_fp8(qkv, NH, NKV, theta, rope_interleaved=interleaved)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.attention_forward(qkv_np, C, NH, NKV, theta, rope_interleaved=interleaved)
    _, _, V = oracle.split_qkv(qkv_np, C, NH, NKV)
    e_out = float(np.abs(to_numpy(out) - ref_out).max()) / float(np.abs(V).max())
    e_lse = float(np.abs(to_numpy(lse) - ref_lse).max()) / max(1.0, float(np.abs(ref_lse).max()))
    assert np.isfinite(to_numpy(out)).all()
    assert e_out <= out_bar(T) and e_lse <= LSE_BAR, (e_out, e_lse)
    # and in the normalised metric of the other paths (reported on failure)
    assert rel_err(to_numpy(out), ref_out) <= 2 * out_bar(T)
    assert lib.attn_device_status() == 0


@pytest.mark.parametrize("B,T,C,NH,NKV", [
    (2, 300, 1024, 8, 2),
    (1, 257, 2048, 16, 4),
    (1, 1000, 512, 4, 1),
    (1, 128, 256, 2, 1),
    (1, 1, 256, 2, 1),
])
def test_fp8_forward_matches_quantized_oracle(lib, B, T, C, NH, NKV):
    """Without RoPE both sides quantize the same float32 values with the same
    float32 scale arithmetic, so every Q/K/V code agrees; what remains is the
    kernel's e4m3 rounding of the softmax weights (stored as 112 p, p <= 4)
    before PV.  With out = sum_j P8_j Vd_j / l, l >= 1 (the row maximum
    contributes at least 1), a weight rounds with relative error <= 2^-4 in
    the normal range and absolute error <= 2^-10 / 112 below it
    (112 p < 2^-6), and out is rounded to bf16 (2^-8 relative), so
    |out - ref| <= max|Vd| (2^-4 + T 2^-10 / 112 + 2^-8).  lse uses the
    unrounded float32 weights: float32 score sums and exp2/log2
    approximations give ~1e-6; the bar is 1e-3 max(1, |lse|)."""
    import torch
    from oracle.e4m3 import attention_forward_e4m3
    w = shape_workload(B, T, C, NH, NKV, 0.0, seed=B * 100 + T + 79)
    qkv_np, _ = make_inputs(w, "bf16")
    qkv = to_device(qkv_np, "bf16")
    out, lse = lib.forward_fp8(qkv, NH, NKV, 0.0)
    torch.cuda.synchronize()
    ref_out, ref_lse, Vd = attention_forward_e4m3(qkv_np, C, NH, NKV, 0.0)
    vmax = float(np.abs(Vd).max())
    bar_out = vmax * (2.0 ** -4 + T * P_SUBNORMAL + 2.0 ** -8)
    lse_bar = 1e-3 * max(1.0, float(np.abs(ref_lse).max()))
    e_out = float(np.abs(to_numpy(out) - ref_out).max())
    e_lse = float(np.abs(to_numpy(lse) - ref_lse).max())
    assert np.isfinite(to_numpy(out)).all()
    assert e_out <= bar_out and e_lse <= lse_bar, (e_out, bar_out, e_lse, lse_bar)
    assert lib.attn_device_status() == 0


def test_fp8_forward_rejects_unsupported_shapes(lib):
    import torch
    from causal_attention_gqa_gb300.binding import AttnError
    qkv = torch.zeros((1, 64, (3 + 2) * 128), dtype=torch.bfloat16, device="cuda")   # NH 3: odd group
    with pytest.raises(AttnError) as ei:
        lib.forward_fp8(qkv, 3, 1, 0.0)
    assert ei.value.status == -3


@pytest.mark.parametrize("name", ["gqa_block", "long_context_gqa"])
def test_fp8_forward_full_size_sampled(lib, name):
    """Full-size call as bench.py --fp8 makes it (caller workspace); the
    oracle is evaluated on seeded query rows of every head."""
    import torch
    from causal_attention_gqa_gb300 import binding
    w = WORKLOADS[name]
    qkv_np, dout_np = make_inputs(w, "bf16")
    qkv = to_device(qkv_np, "bf16")
    out = torch.empty((w.B, w.T, w.C), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.NH, w.T), dtype=torch.float32, device="cuda")
    nb = binding.attn_fwd_fp8_workspace_bytes(w.B, w.T, w.C, w.NH, w.NKV, binding.DTYPE_BF16)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    binding.attn_fwd_fp8(out, lse, qkv, w.B, w.T, w.C, w.NH, w.NKV, w.rope_theta, binding.DTYPE_BF16, ws, nb)
    torch.cuda.synchronize()
    qr = sample_rows(w.T, 48, w.seed + 11)
    ref = oracle.attention_sampled(qkv_np, dout_np, w.C, w.NH, w.NKV, w.rope_theta, qr, [], qr)
    _, _, V = oracle.split_qkv(qkv_np, w.C, w.NH, w.NKV)
    got_out = to_numpy(out)[:, qr]
    got_lse = to_numpy(lse)[:, :, qr]
    assert np.isfinite(got_out).all() and np.isfinite(got_lse).all()
    e_out = float(np.abs(got_out - ref["out_rows"]).max()) / float(np.abs(V).max())
    e_lse = float(np.abs(got_lse - ref["lse_rows"]).max()) / max(1.0, float(np.abs(ref["lse_rows"]).max()))
    assert e_out <= out_bar(w.T) and e_lse <= LSE_BAR, (e_out, e_lse)
    assert lib.attn_device_status() == 0
