"""World-size-2 CPU (gloo) checks of the multi-rank host logic: the slowest
rank's times reach every rank, and sharding the batch rows over ranks is
exact -- the oracle on each rank's shard equals the matching rows of the
oracle on the global batch (batch rows are independent problems, which is why
the path needs no collective)."""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2
SHAPE = dict(B=2, T=70, C=64, NH=4, NKV=2, rope_theta=1e4, seed=321)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    import oracle
    from causal_attention_gqa_gb300.workloads import make_inputs, rank_shard, shape_workload
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        # slowest rank's numbers, element by element
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 5.0], "cpu")
        w = rank_shard(shape_workload(**SHAPE), rank, WORLD)
        qkv, dout = make_inputs(w, "f32")
        out, lse = oracle.attention_forward(qkv, w.C, w.NH, w.NKV, w.rope_theta)
        dist.barrier()
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), reduced=np.array(got), qkv=qkv, dout=dout, out=out, lse=lse)
    finally:
        dist.destroy_process_group()


def test_two_rank_reduction_and_exact_batch_sharding(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    mp.spawn(_rank_main, args=(_free_port(), str(tmp_path)), nprocs=WORLD, join=True)
    import oracle
    from causal_attention_gqa_gb300.workloads import shape_workload
    parts = [np.load(tmp_path / f"rank{r}.npz") for r in range(WORLD)]
    for p in parts:
        np.testing.assert_array_equal(p["reduced"], [2.0, 10.0, 5.0])
    # the ranks drew different batch rows
    assert not np.array_equal(parts[0]["qkv"], parts[1]["qkv"])
    w = shape_workload(**SHAPE)
    qkv_global = np.concatenate([p["qkv"] for p in parts], axis=0)
    out_g, lse_g = oracle.attention_forward(qkv_global, w.C, w.NH, w.NKV, w.rope_theta)
    for r, p in enumerate(parts):
        rows = slice(r * w.B, (r + 1) * w.B)
        np.testing.assert_array_equal(p["out"], out_g[rows])
        np.testing.assert_array_equal(p["lse"], lse_g[rows])
    # and the backward's gradients of a shard are the global gradients' rows
    dout_global = np.concatenate([p["dout"] for p in parts], axis=0)
    g_global = oracle.attention_backward(qkv_global, dout_global, w.C, w.NH, w.NKV, w.rope_theta)
    g_shard = oracle.attention_backward(parts[1]["qkv"], parts[1]["dout"], w.C, w.NH, w.NKV, w.rope_theta)
    np.testing.assert_array_equal(g_shard, g_global[w.B:2 * w.B])


def test_rank_shard_rules():
    from causal_attention_gqa_gb300.workloads import WORKLOADS, rank_shard
    w = WORKLOADS["gqa_block"]
    assert rank_shard(w, 0, 4) is w
    seeds = {rank_shard(w, r, 4).seed for r in range(4)}
    assert len(seeds) == 4
    assert all(rank_shard(w, r, 4).B == w.B for r in range(4))
    with pytest.raises(ValueError):
        rank_shard(w, 4, 4)
