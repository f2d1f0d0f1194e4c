"""The N > 1 host logic of bench.py with 2 gloo ranks on CPU: sharding of
independent sequences, the max-over-ranks of the elapsed time and the
whole-job rate.  Each rank also builds its own share of a workload's block
tables with the C++ block manager (no GPU, no collective on the data path)."""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import paged_kv_cache_13_gb300 as pkv
        import synthetic as syn
        w = syn.workload("llama3_8b_b64")
        lens = syn.context_lengths(w)
        lo, hi = bench.shard(len(lens), world, rank)
        pool = pkv.pkv_pool_create(w["num_blocks"], 16, syn.free_order(w))
        seqs = []
        for L in lens[lo:hi]:
            s = pkv.pkv_seq_create(pool)
            pkv.pkv_seq_append(pool, s, L)
            seqs.append(s)
        _, ctx = pkv.pkv_build_block_tables(pool, seqs, 256)
        my_bytes = int(ctx.sum()) * bench.KV_BYTES_PER_TOKEN
        fake_seconds = 1.0 + rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(fake_seconds, dist, torch.device("cpu"))
        t = torch.tensor([my_bytes], dtype=torch.float64)
        dist.all_reduce(t)
        q.put((rank, lo, hi, my_bytes, slowest, float(t.item())))
        pkv.pkv_pool_destroy(pool)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import bench
    import synthetic as syn
    lens = syn.context_lengths(syn.workload("llama3_8b_b64"))
    # shards are disjoint and cover the batch
    assert res[0][1] == 0 and res[0][2] == res[1][1] and res[1][2] == len(lens)
    total = sum(r[3] for r in res)
    assert total == sum(lens) * bench.KV_BYTES_PER_TOKEN
    assert all(r[4] == 2.0 for r in res)  # the slowest rank's time on every rank
    assert all(r[5] == total for r in res)
    # weak-scaling rate: units of all ranks over the slowest time
    assert bench.whole_job_rate(100.0, 2, 2.0) == 100.0


def test_shard_covers_any_size():
    import bench
    for n in (0, 1, 7, 64, 65):
        for world in (1, 2, 3, 8):
            parts = [bench.shard(n, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            assert all(parts[i][1] == parts[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1
