"""The allocation-free backward entry point, attn_bwd_noalloc.

It exists for callers that cannot allocate device memory at the point where
they run the backward (allocator or memory-pool callbacks, runtimes with a
fixed memory budget, plugins handed only input/output pointers).  These tests
call it through the C ABI and compare its dqkv with the regular attn_bwd
(caller-provided workspace) on the same inputs, twice in a row, because the
built-in scratch buffer is shared by every call and keeps the previous call's
contents.  Both entry points run the same deterministic kernels on the same
workspace layout, so the results must agree bit for bit: a tolerance would hide
a scratch-layout mistake.  This file is collected last so that a run stopping
at the first failure has already run every other test.
"""
import numpy as np
import pytest

from causal_attention_gqa_gb300.workloads import make_inputs, shape_workload
from helpers import TOL, rel_err, to_device, to_numpy

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,shape,theta", [
    ("bf16", (2, 300, 512, 8, 2), 1e6),     # uses the rotated Q/K scratch
    ("bf16", (1, 257, 512, 4, 4), 0.0),
    ("f32", (2, 70, 64, 4, 2), 1e4),
])
def test_noalloc_backward_matches_workspace_backward_twice(lib, dtype, shape, theta):
    import torch
    B, T, C, NH, NKV = shape
    w = shape_workload(B, T, C, NH, NKV, theta, seed=31 + T)
    qkv_np, dout_np = make_inputs(w, dtype)
    qkv, dout = to_device(qkv_np, dtype), to_device(dout_np, dtype)
    out, lse = lib.forward(qkv, NH, NKV, theta)
    ref = lib.backward(qkv, out, dout, lse, NH, NKV, theta)
    code = lib.dtype_code(qkv)
    for _ in range(2):
        dqkv = torch.full_like(qkv, float("nan"))
        lib.attn_bwd_noalloc(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, theta, code)
        torch.cuda.synchronize()
        got = to_numpy(dqkv)
        assert np.isfinite(got).all()
        assert rel_err(got, to_numpy(ref)) <= TOL[dtype]
        assert torch.equal(dqkv, ref), "attn_bwd_noalloc differs from attn_bwd on the same inputs"
    assert lib.attn_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_buffer(lib):
    """The long-context bf16 shape needs ~90 MB of scratch, more than the
    64 MiB built-in buffer: rejected with ATTN_ERR_WORKSPACE, nothing run."""
    import torch
    from causal_attention_gqa_gb300.binding import AttnError, DTYPE_BF16
    B, T, C, NH, NKV = 1, 8192, 4096, 32, 8
    need = lib.attn_bwd_workspace_bytes(B, T, C, NH, NKV, DTYPE_BF16)
    assert need > 64 * 1024 * 1024
    W = (NH + 2 * NKV) * (C // NH)
    qkv = torch.zeros((B, T, W), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, T, C), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, NH, T), dtype=torch.float32, device="cuda")
    dqkv = torch.zeros_like(qkv)
    with pytest.raises(AttnError) as ei:
        lib.attn_bwd_noalloc(dqkv, qkv, out, out, lse, B, T, C, NH, NKV, 1e6, DTYPE_BF16)
    assert ei.value.status == -5
    torch.cuda.synchronize()
    assert lib.attn_device_status() == 0
