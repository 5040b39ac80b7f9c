"""The multi-rank path on CPU (gloo, world size 2): batch shards cover the
batch exactly once, sharded results equal the unsharded ones, and the
max-over-ranks timing reduction used by bench.py picks the slowest rank."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from exact_attention_71_gb300.shard import batch_shard


def test_batch_shard_partitions_the_batch():
    for B in range(0, 13):
        for world in range(1, 6):
            owned = []
            for r in range(world):
                s, e = batch_shard(B, world, r)
                assert 0 <= s <= e <= B
                owned.extend(range(s, e))
            assert owned == list(range(B))
    with pytest.raises(ValueError):
        batch_shard(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from exact_attention_71_gb300 import synth
    B, N, H, d = 5, 40, 2, 16
    q, k, v = synth.qkv_bf16(B, N, H, d, seed=3)
    s, e = batch_shard(B, world, rank)
    o, lse = oracle.attention(q[s:e], k[s:e], v[s:e], causal=True)
    parts = [None] * world
    dist.all_gather_object(parts, (s, e, o, lse))
    t = torch.tensor([float(rank + 1)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        o_all = np.concatenate([p[2] for p in parts], axis=0)
        l_all = np.concatenate([p[3] for p in parts], axis=0)
        o_ref, l_ref = oracle.attention(q, k, v, causal=True)
        ok = np.array_equal(o_all, o_ref) and np.array_equal(l_all, l_ref) and t.item() == world
        with open(out_path, "w") as f:
            f.write("ok" if ok else "mismatch")
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_reduce(tmp_path):
    out = str(tmp_path / "result.txt")
    mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
    assert open(out).read() == "ok"


def test_job_end_to_end_figure_from_the_slowest_rank():
    """bench.py's end-to-end line at N ranks: all ranks' work over the
    slowest rank's step time, bytes summed over the ranks."""
    import bench
    rank_e2e = {"value": 100.0, "unit": "TFLOPS", "h2d_bytes_per_step": 1000, "d2h_bytes_per_step": 10,
                "ms_per_step": 1.0}
    out = bench.job_e2e(rank_e2e, 2.0, 4, 1e12)
    assert out["value"] == 2000.0          # 4 x 1e12 FLOP / 2 ms
    assert out["h2d_bytes_per_step"] == 4000 and out["d2h_bytes_per_step"] == 40
    assert out["ms_per_step"] == 2.0 and out["ranks"] == 4
    assert rank_e2e["h2d_bytes_per_step"] == 1000   # the rank's own figure is left as it was
