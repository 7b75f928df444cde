"""GPU robustness: determinism, guard bands, argument errors that must launch
nothing, and the bounded-wait failure path (a wait that nothing completes
must expire, report ATTN_ERR_DEVICE_TIMEOUT and leave the device usable)."""
import numpy as np
import pytest

from causal_attention_gqa_gb300.workloads import make_inputs, shape_workload
from helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,theta", [("f32", 1e6), ("bf16", 1e6), ("bf16", 0.0)])
def test_backward_is_deterministic(lib, dtype, theta):
    import torch
    w = shape_workload(2, 333, 512, 8, 2, theta, seed=21)
    qkv_np, dout_np = make_inputs(w, dtype)
    qkv, dout = to_device(qkv_np, dtype), to_device(dout_np, dtype)
    out, lse = lib.forward(qkv, w.NH, w.NKV, theta)
    out2, lse2 = lib.forward(qkv, w.NH, w.NKV, theta)
    d1 = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, theta)
    d2 = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, theta)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    assert torch.equal(d1, d2)


@pytest.mark.parametrize("theta", [1e6, 0.0])
def test_benchmark_path_is_deterministic(lib, theta):
    """Head size 128, four query heads per kv head: the paired-head forward
    (attn_fwd_ws), and attn_bwd_rot whose dQ kernel hands out work items
    dynamically; every output element still has one writer and one summation
    order, so repeated calls are bit-identical."""
    import torch
    w = shape_workload(2, 333, 1024, 8, 2, theta, seed=23)
    qkv_np, dout_np = make_inputs(w, "bf16")
    qkv, dout = to_device(qkv_np, "bf16"), to_device(dout_np, "bf16")
    out, lse, fws = lib.forward_ws(qkv, w.NH, w.NKV, theta)
    out2, lse2, fws2 = lib.forward_ws(qkv, w.NH, w.NKV, theta)
    d1 = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, theta, qk_rot=fws)
    d2 = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, theta, qk_rot=fws2)
    d3 = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, theta)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    assert torch.equal(d1, d2) and torch.equal(d1, d3)


def test_guard_bands_untouched_benchmark_path(lib):
    """The tile stores of the paired-head forward and of the gradient
    epilogues clip rows past T: nothing outside the outputs changes."""
    import torch
    w = shape_workload(1, 200, 1024, 8, 2, 1e6, seed=24)
    qkv_np, dout_np = make_inputs(w, "bf16")
    qkv, dout = to_device(qkv_np, "bf16"), to_device(dout_np, "bf16")
    pad = 4096
    canary = -12288.0

    def guarded(n, dt):
        buf = torch.full((pad + n + pad,), canary, dtype=dt, device="cuda")
        return buf, buf[pad:pad + n]

    B, T, C, NH, NKV = w.B, w.T, w.C, w.NH, w.NKV
    out_buf, out = guarded(B * T * C, torch.bfloat16)
    lse_buf, lse = guarded(B * NH * T, torch.float32)
    dq_buf, dqkv = guarded(B * T * w.qkv_width, torch.bfloat16)
    code = lib.DTYPE_BF16
    fb = lib.attn_fwd_workspace_bytes(B, T, C, NH, NKV, code)
    fws = torch.empty(fb, dtype=torch.uint8, device="cuda")
    lib.attn_fwd_ws(out, lse, qkv, B, T, C, NH, NKV, w.rope_theta, code, fws, fb)
    nbytes = lib.attn_bwd_workspace_bytes(B, T, C, NH, NKV, code)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    lib.attn_bwd_rot(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, w.rope_theta, code, fws, ws, nbytes)
    torch.cuda.synchronize()
    for buf in (out_buf, lse_buf, dq_buf):
        host = buf.float().cpu().numpy()
        assert np.all(host[:pad] == canary) and np.all(host[-pad:] == canary)
    assert torch.isfinite(out).all() and torch.isfinite(dqkv).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_guard_bands_untouched(lib, dtype):
    """Outputs live inside larger buffers filled with a canary; nothing outside
    the output extents may change (stands in for a memory checker)."""
    import torch
    w = shape_workload(1, 200, 256, 4, 2, 1e6, seed=22)
    qkv_np, dout_np = make_inputs(w, dtype)
    qkv, dout = to_device(qkv_np, dtype), to_device(dout_np, dtype)
    tdt = qkv.dtype
    pad = 4096
    canary = -12288.0  # exactly representable in bf16 and float32

    def guarded(n, dt):
        buf = torch.full((pad + n + pad,), canary, dtype=dt, device="cuda")
        return buf, buf[pad:pad + n]

    B, T, C, NH, NKV = w.B, w.T, w.C, w.NH, w.NKV
    out_buf, out = guarded(B * T * C, tdt)
    lse_buf, lse = guarded(B * NH * T, torch.float32)
    dq_buf, dqkv = guarded(B * T * w.qkv_width, tdt)
    code = lib.dtype_code(qkv)
    lib.attn_fwd(out, lse, qkv, B, T, C, NH, NKV, w.rope_theta, code)
    nbytes = lib.attn_bwd_workspace_bytes(B, T, C, NH, NKV, code)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    lib.attn_bwd(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, w.rope_theta, code, ws, nbytes)
    torch.cuda.synchronize()
    for buf in (out_buf, lse_buf, dq_buf):
        host = buf.float().cpu().numpy()
        assert np.all(host[:pad] == canary) and np.all(host[-pad:] == canary)
    assert torch.isfinite(out).all() and torch.isfinite(dqkv).all()


def test_invalid_arguments_launch_nothing(lib):
    import torch
    from causal_attention_gqa_gb300.binding import AttnError
    qkv = torch.zeros((1, 128, 3 * 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((1, 128, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device="cuda")
    cases = [
        (dict(C=128, NH=3, NKV=1), -2),           # C % NH
        (dict(C=128, NH=2, NKV=3), -2),           # NH % NKV (and C/NH)
        (dict(C=96 * 3, NH=3, NKV=3), -3),         # hd 96 unsupported on bf16
    ]
    for kw, code in cases:
        with pytest.raises(AttnError) as ei:
            lib.attn_fwd(out, lse, qkv, 1, 128, kw["C"], kw["NH"], kw["NKV"], 0.0, lib.DTYPE_BF16)
        assert ei.value.status == code
    with pytest.raises(AttnError) as ei:   # misaligned bf16 pointer
        lib.attn_fwd(out.data_ptr() + 2, lse, qkv, 1, 128, 128, 1, 1, 0.0, lib.DTYPE_BF16)
    assert ei.value.status == -4
    with pytest.raises(AttnError) as ei:   # TF32 runs the float32 kernels: hd 256 unsupported
        lib.attn_fwd(out, lse, qkv, 1, 128, 256, 1, 1, 0.0, lib.DTYPE_TF32)
    assert ei.value.status == -3
    with pytest.raises(AttnError) as ei:   # workspace too small
        lib.attn_bwd(qkv, qkv, out, out, lse, 1, 128, 128, 1, 1, 0.0, lib.DTYPE_BF16, qkv, 16)
    assert ei.value.status == -5
    torch.cuda.synchronize()
    assert lib.attn_device_status() == 0


def test_bounded_wait_expires_and_device_stays_usable(lib):
    import torch
    assert lib.attn_selftest_wait_timeout(2_000_000) == -7   # 2 ms limit
    x = torch.arange(10, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 45.0
    assert lib.attn_device_status() == 0  # the self test reports separately


def test_no_device_errors_recorded(lib):
    assert lib.attn_device_status(reset=True) == 0


@pytest.mark.parametrize("dtype,theta,fwd_ws", [("bf16", 1e6, True), ("bf16", 0.0, False), ("f32", 1e6, False)])
def test_cuda_graph_capture_replays_identically(lib, dtype, theta, fwd_ws):
    """A forward + backward captured into a CUDA graph (the launch-overhead
    remedy for small problems) replays bit-identically to eager calls: none of
    these four entry points synchronises, allocates or reads host state on the
    stream."""
    import torch
    w = shape_workload(2, 200, 1024 if dtype == "bf16" else 128, 8, 2, theta, seed=51)
    qkv_np, dout_np = make_inputs(w, dtype)
    qkv, dout = to_device(qkv_np, dtype), to_device(dout_np, dtype)
    code = lib.DTYPE_BF16 if dtype == "bf16" else lib.DTYPE_F32
    B, T, C, NH, NKV = w.B, w.T, w.C, w.NH, w.NKV
    out = torch.empty((B, T, C), dtype=qkv.dtype, device="cuda")
    lse = torch.empty((B, NH, T), dtype=torch.float32, device="cuda")
    dqkv = torch.empty_like(qkv)
    wsb = lib.attn_bwd_workspace_bytes(B, T, C, NH, NKV, code)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    fwsb = lib.attn_fwd_workspace_bytes(B, T, C, NH, NKV, code)
    fws = torch.empty(max(fwsb, 1), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        s = stream.cuda_stream
        if fwd_ws:
            lib.attn_fwd_ws(out, lse, qkv, B, T, C, NH, NKV, theta, code, fws, fwsb, s)
            lib.attn_bwd_rot(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, theta, code, fws, ws, wsb, s)
        else:
            lib.attn_fwd(out, lse, qkv, B, T, C, NH, NKV, theta, code, s)
            lib.attn_bwd(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, theta, code, ws, wsb, s)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    ref = [out.clone(), lse.clone(), dqkv.clone()]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for t in (out, lse, dqkv):
        t.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1]) and torch.equal(dqkv, ref[2])
    assert lib.attn_device_status() == 0
