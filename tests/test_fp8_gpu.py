"""GPU check of the e4m3 (FP8) forward (attn_fwd_fp8) against the e4m3
oracle (oracle/e4m3.py), which restates every step the kernel takes: Q/K
quantized per 128-row tile after RoPE, V per head, and the softmax weights
rounded to e4m3 as P8 = e4m3(112 * 2^(s - m)) with the lazily renewed row
maximum, walking the keys in 128-key blocks.

The bar is element-wise and does not grow with T.  It is the sum of:
  * the bf16 rounding of out (8 significant bits): 2^-8 |out|;
  * float32 evaluation order (the sum l of up to T weights, the O
    accumulator's rescales, the final scaling): |out| * (l_rel + 2^-16), with
    l_rel the oracle's bound on how far l moves when every weight is
    evaluated in float32 (see weighted_row_e4m3);
  * the weights that lie within float32 reach of an e4m3 midpoint (they may
    round either way): the oracle's o_bound, one code step times |V| for
    each such weight, over l; zero for most rows;
  * the tensor core's accumulation of the PV products: MMA_REL per added
    K slice times the sum of |P8 V8|, over l.
With RoPE the rotated Q/K values differ from the oracle's by the rotation's
float32 arithmetic and angle error (at most ANGLE_ERROR times the pair's
norm); the oracle carries that into the score reach, so Q/K codes next to a
midpoint are covered the same way.  A row whose renewal decision is open
(its block maximum within reach of m + 2) may follow either branch; the
oracle evaluates both.

lse: the kernel's l sums unrounded weights, so lse is the log-sum-exp of the
quantized scores whatever the rounding: |lse - ref| <= ln 2 * (score reach)
+ float32 terms.
"""
import numpy as np
import pytest

from causal_attention_gqa_gb300.workloads import WORKLOADS, make_inputs, sample_rows, shape_workload
from helpers import to_device, to_numpy

pytestmark = pytest.mark.gpu
ANGLE_ERROR = 2e-6          # rotation error per unit pair norm (angle ~6e-7 rad plus float32 products)
MMA_REL = 2.0 ** -22        # rounding of one tensor-core accumulation step, relative to what it adds


def fp8_reference(qkv_np, w, theta, interleaved=False, rows=None):
    from oracle.e4m3 import attention_forward_e4m3
    return attention_forward_e4m3(qkv_np, w.C, w.NH, w.NKV, theta, rope_interleaved=interleaved, rows=rows,
                                  angle_error=ANGLE_ERROR if theta > 0 else 0.0, mma_rel=MMA_REL)


def check_against_e4m3_oracle(got_out, got_lse, ref, rows, hd):
    """Element-wise comparison with the bar described above; returns the
    largest error / bar, the bars of every checked element over max|V|, and
    the number of rows with an open renewal decision."""
    ref_out, ref_lse, Vd, reach = ref
    vmax = float(np.abs(Vd).max())
    B, T, C = ref_out.shape
    NH = ref_lse.shape[1]
    worst = 0.0
    bars = []
    open_rows = 0
    for b in range(B):
        for t in rows:
            for h in range(NH):
                cols = slice(h * hd, (h + 1) * hd)
                g = got_out[b, t, cols]
                assert np.isfinite(g).all()
                cand = [(ref_out[b, t, cols], reach["o_bound"][b, t, cols], reach["l_rel"][b, h, t])]
                cand += reach["open"].get((b, h, int(t)), [])
                open_rows += len(cand) > 1
                best = None
                for o_ref, o_bnd, l_rel in cand:
                    bar = (2.0 ** -8 * np.abs(o_ref)
                           + (1 + 2.0 ** -8) * (o_bnd + np.abs(o_ref) * (l_rel + 2.0 ** -16)
                                                + reach["o_acc"][b, t, cols])
                           + 2.0 ** -30 * vmax)
                    r = float((np.abs(g - o_ref) / bar).max())
                    if best is None or r < best[0]:
                        best = (r, bar)
                worst = max(worst, best[0])
                bars.append(best[1] / vmax)
                lse_bar = (np.log(2.0) * reach["s_reach"][b, h, t] + 2.0 ** -18
                           + 2.0 ** -20 * abs(ref_lse[b, h, t]))
                e_lse = abs(got_lse[b, h, t] - ref_lse[b, h, t])
                assert e_lse <= lse_bar, (b, h, t, e_lse, lse_bar)
    assert worst <= 1.0, f"out error reaches {worst:.3f} of the bar"
    return worst, np.concatenate(bars), open_rows


def assert_bar_is_tight(bars):
    """The bar does not hide a loose comparison: on a typical element it is
    within two bf16 steps of max|V| (measured medians: 1e-4 without RoPE,
    2e-3 to 4e-3 with it, where most rows have a Q/K code within the
    rotation's reach of a midpoint), and nowhere more than the error one
    rounded weight can make (2^-4 relative)."""
    assert np.median(bars) <= 2.0 ** -7, np.median(bars)
    assert bars.max() <= 2.0 ** -4, bars.max()


@pytest.mark.parametrize("B,T,C,NH,NKV,theta,interleaved", [
    (2, 300, 1024, 8, 2, 0.0, False),
    (1, 257, 2048, 16, 4, 0.0, False),
    (1, 1000, 512, 4, 1, 0.0, False),
    (1, 128, 256, 2, 1, 0.0, False),
    (1, 1, 256, 2, 1, 0.0, False),
    (2, 300, 1024, 8, 2, 1e6, False),
    (1, 257, 2048, 16, 4, 1e4, True),
    (1, 1, 256, 2, 1, 1e6, False),
])
def test_fp8_forward_matches_e4m3_oracle(lib, B, T, C, NH, NKV, theta, interleaved):
    import torch
    w = shape_workload(B, T, C, NH, NKV, theta, seed=B * 100 + T + 71)
    qkv_np, _ = make_inputs(w, "bf16")
    qkv = to_device(qkv_np, "bf16")
    out, lse = lib.forward_fp8(qkv, NH, NKV, theta, rope_interleaved=interleaved)
    torch.cuda.synchronize()
    ref = fp8_reference(qkv_np, w, theta, interleaved)
    worst, bars, _ = check_against_e4m3_oracle(to_numpy(out), to_numpy(lse), ref, range(T), w.hd)
    assert_bar_is_tight(bars)
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
    """Full-size call as bench.py --fp8 makes it (caller workspace, RoPE
    1e6); the e4m3 oracle is evaluated on seeded query rows of every head."""
    import torch
    from causal_attention_gqa_gb300 import binding
    w = WORKLOADS[name]
    qkv_np, _ = make_inputs(w, "bf16")
    qkv = to_device(qkv_np, "bf16")
    out = torch.empty((w.B, w.T, w.C), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.NH, w.T), dtype=torch.float32, device="cuda")
    nb = binding.attn_fwd_fp8_workspace_bytes(w.B, w.T, w.C, w.NH, w.NKV, binding.DTYPE_BF16)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    binding.attn_fwd_fp8(out, lse, qkv, w.B, w.T, w.C, w.NH, w.NKV, w.rope_theta, binding.DTYPE_BF16, ws, nb)
    torch.cuda.synchronize()
    qr = sample_rows(w.T, 48, w.seed + 11)
    ref = fp8_reference(qkv_np, w, w.rope_theta, rows=qr)
    worst, bars, _ = check_against_e4m3_oracle(to_numpy(out), to_numpy(lse), ref, qr, w.hd)
    assert_bar_is_tight(bars)
    assert lib.attn_device_status() == 0
