"""GPU parity of attn_decode (single-query attention over a KV cache)
against the float64 oracle: ragged lengths, chunk boundaries (128 cache rows
per chunk), grouped heads, both element types; determinism and the
length-range rule."""
import numpy as np
import pytest

import oracle
from causal_attention_gqa_gb300.workloads import make_decode_inputs
from helpers import TOL, rel_err

pytestmark = pytest.mark.gpu


def run_decode(lib, q_np, k_np, v_np, lens, dtype):
    import torch
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.from_numpy(q_np).to("cuda", tdt)
    k = torch.from_numpy(k_np).to("cuda", tdt)
    v = torch.from_numpy(v_np).to("cuda", tdt)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out, lse = lib.decode(q, k, v, lens_t)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,NH,NKV,hd,max_len,lens", [
    (1, 1, 1, 64, 1, [1]),
    (3, 8, 2, 128, 300, [1, 129, 300]),
    (2, 4, 4, 64, 1000, [1000, 513]),
    (2, 32, 8, 128, 2048, [2048, 1537]),
    (1, 6, 1, 128, 257, [256]),       # grp 6: two head groups of one kv head
    (2, 12, 12, 64, 128, [128, 127]),
])
def test_decode_matches_oracle(lib, dtype, B, NH, NKV, hd, max_len, lens):
    q, k, v = make_decode_inputs(B, NH, NKV, hd, max_len, dtype, seed=B * 100 + NH + max_len)
    out, lse = run_decode(lib, q, k, v, lens, dtype)
    ref_out, ref_lse = oracle.attention_decode(q, k, v, lens)
    tol = TOL[dtype]
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert rel_err(out, ref_out) <= tol, rel_err(out, ref_out)
    assert float(np.abs(lse - ref_lse).max()) <= tol * max(1.0, float(np.abs(ref_lse).max()))
    assert lib.attn_device_status() == 0


def test_decode_is_deterministic(lib):
    q, k, v = make_decode_inputs(2, 16, 4, 128, 4096, "bf16", seed=5)
    a = run_decode(lib, q, k, v, [4096, 3000], "bf16")
    b = run_decode(lib, q, k, v, [4096, 3000], "bf16")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_decode_length_out_of_range_is_clamped_and_recorded(lib):
    """seq_lens outside [1, max_len] are clamped into it (the launch still
    computes something defined) and ATTN_ERR_BAD_ARGUMENT is recorded."""
    q, k, v = make_decode_inputs(2, 4, 2, 64, 50, "f32", seed=9)
    assert lib.attn_device_status(reset=True) == 0
    out, lse = run_decode(lib, q, k, v, [0, 99], "f32")
    assert lib.attn_device_status(reset=True) == -8
    ref_out, ref_lse = oracle.attention_decode(q, k, v, [1, 50])
    assert rel_err(out, ref_out) <= TOL["f32"]
    assert lib.attn_device_status() == 0
