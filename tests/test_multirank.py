"""The N > 1 host logic of bench.py with 2 gloo ranks on CPU: every rank
builds its own replica of the workload's block tables with the C++ block
manager (replicas only: no GPU, no collective on the data path), the
max-over-ranks of the elapsed time, and the whole-job rate over all
replicas."""

import hashlib
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


def tables_digest(pkv, pool, seqs):
    tables, ctx = pkv.pkv_build_block_tables(pool, seqs, 256)
    return hashlib.sha256(tables.tobytes() + ctx.tobytes()).hexdigest()


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
        pool = pkv.pkv_pool_create(w["num_blocks"], 16, syn.free_order(w))
        seqs = []
        for L in lens:
            s = pkv.pkv_seq_create(pool)
            pkv.pkv_seq_append(pool, s, L)
            seqs.append(s)
        _, ctx = pkv.pkv_build_block_tables(pool, seqs, 256)
        my_bytes = int(ctx.sum()) * bench.KV_BYTES_PER_TOKEN
        fake_seconds = 1.0 + rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(fake_seconds, dist, torch.device("cpu"))
        t = torch.tensor([my_bytes], dtype=torch.float64)
        dist.all_reduce(t)
        q.put((rank, tables_digest(pkv, pool, seqs), my_bytes, slowest, float(t.item())))
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
    # every rank holds the same replica: identical tables, the whole batch
    assert res[0][1] == res[1][1]
    replica = sum(lens) * bench.KV_BYTES_PER_TOKEN
    assert all(r[2] == replica for r in res)
    total = sum(r[2] for r in res)
    assert total == world * replica
    assert all(r[3] == 2.0 for r in res)  # the slowest rank's time on every rank
    assert all(r[4] == total for r in res)
    # weak-scaling rate: units of all ranks over the slowest time
    assert bench.whole_job_rate(replica, world, 2.0) == total / 2.0
