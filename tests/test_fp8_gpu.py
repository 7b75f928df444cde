"""GPU check of the e4m3 (FP8) forward (attn_fwd_fp8) against the float64
oracle on the original inputs.

Bars, from the e4m3 rounding model (3 mantissa bits: a value scaled into the
e4m3 range is rounded with a relative error of at most 2^-4):
  * out: out = sum_j P_j V_j / l with every P_j and every V element rounded,
    so |out - ref| <= (2^-4 + 2^-4 + 2^-8) max|V| = 0.129 max|V| from those
    two roundings; rows that see a single key reach it (out = the rounded
    V_0).  The bar is 0.13 max|V|.
  * lse: the scores s = q . k / sqrt(hd) inherit the rounding of Q and K;
    its worst case (all 128 products rounded the same way) is far larger
    than what random inputs show, so the bar, 0.1 max(1, max|lse|), is an
    empirical margin over the measured ~0.01 relative error.
"""
import numpy as np
import pytest

import oracle
from causal_attention_gqa_gb300.workloads import make_inputs, shape_workload
from helpers import rel_err, to_device, to_numpy

pytestmark = pytest.mark.gpu
OUT_BAR = 0.13     # times max|V|
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
    assert e_out <= OUT_BAR and e_lse <= LSE_BAR, (e_out, e_lse)
    # and in the normalised metric of the other paths (reported on failure)
    assert rel_err(to_numpy(out), ref_out) <= 2 * OUT_BAR
    assert lib.attn_device_status() == 0


def test_fp8_forward_rejects_unsupported_shapes(lib):
    import torch
    from causal_attention_gqa_gb300.binding import AttnError
    qkv = torch.zeros((1, 64, (3 + 2) * 128), dtype=torch.bfloat16, device="cuda")   # NH 3: odd group
    with pytest.raises(AttnError) as ei:
        lib.forward_fp8(qkv, 3, 1, 0.0)
    assert ei.value.status == -3
