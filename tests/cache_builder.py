"""Builds a workload's paged KV cache on the GPU through the library's own
entry points (host block manager + KV-append + copy-on-write copy), and the
oracle's expected decode outputs from the same seeded logical rows."""

import numpy as np
import torch

import synthetic as syn
from oracle import attention as oatt
from oracle import kvcache as okv


class GpuCache:
    pass


def _rows_source(w):
    """handle, start, n -> (k, v) CPU 16-bit rows of that handle's tokens."""
    cache = {}
    prefix = "prompt" in w

    def rows(handle, start, n):
        if prefix and handle == 0:
            if "prompt" not in cache:
                cache["prompt"] = syn.prompt_kv(w)
            k, v = cache["prompt"]
        else:
            i = handle - 1 if prefix else handle
            if i not in cache:
                cache[i] = syn.sequence_kv(w, i)
            k, v = cache[i]
        return k[start:start + n], v[start:start + n]

    return rows


def build(pkv, w, device, quant=None, empty_fill=None, step_append=True):
    """Prefill the workload and run its decode-step append.

    quant: None for a 16-bit cache, "int4" / "fp8" for a quantised cache.
    Returns a GpuCache with pools, tables, lens, q and bookkeeping.
    """
    NB, BS, Hkv, D = w["num_blocks"], w["block_size"], w["hkv"], w["d"]
    dt = w["torch_dtype"]
    order = syn.free_order(w)
    pool = pkv.pkv_pool_create(NB, BS, order)
    c = GpuCache()
    c.w, c.pool, c.quant = w, pool, quant
    if quant is None:
        c.k_pool = torch.empty((NB, Hkv, BS, D), dtype=dt, device=device)
        c.v_pool = torch.empty((NB, Hkv, BS, D), dtype=dt, device=device)
        if empty_fill is not None:
            c.k_pool.fill_(empty_fill)
            c.v_pool.fill_(empty_fill)
        c.pools = [c.k_pool, c.v_pool]
    else:
        g = w.get("group_size", D) if quant == "int4" else D
        cb = D // 2 if quant == "int4" else D
        ng = D // g if quant == "int4" else 1
        u8 = torch.uint8
        c.cache = {
            "k_codes": torch.empty((NB, Hkv, BS, cb), dtype=u8, device=device),
            "v_codes": torch.empty((NB, Hkv, BS, cb), dtype=u8, device=device),
            "k_scale": torch.empty((NB, Hkv, BS, ng), dtype=torch.float16, device=device),
            "v_scale": torch.empty((NB, Hkv, BS, ng), dtype=torch.float16, device=device),
        }
        if quant == "int4":
            c.cache["k_zero"] = torch.empty((NB, Hkv, BS, ng), dtype=torch.float16, device=device)
            c.cache["v_zero"] = torch.empty((NB, Hkv, BS, ng), dtype=torch.float16, device=device)
        c.group_size = g
        c.pools = [c.cache[k] for k in ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero")
                   if k in c.cache]
    ops, decoded = syn.prefill_schedule(w)
    B = len(decoded)
    c.decoded = decoded
    n_sink = w.get("n_sink", 0)
    c.n_sink = n_sink
    if quant is not None:
        ns = max(n_sink, 1)
        c.cache["sink_k"] = torch.zeros((B, ns, Hkv, D), dtype=dt, device=device)
        c.cache["sink_v"] = torch.zeros((B, ns, Hkv, D), dtype=dt, device=device)
        c.window = w.get("window", 0)
        if c.window:
            R = c.window // BS + 1
            c.cache["win_k"] = torch.zeros((B, R, Hkv, BS, D), dtype=dt, device=device)
            c.cache["win_v"] = torch.zeros((B, R, Hkv, BS, D), dtype=dt, device=device)
    row_of_handle = {h: i for i, h in enumerate(decoded)}
    rows = _rows_source(w)
    lens = {}
    pending = []  # (slots, k, v, positions, rows)

    def flush():
        if not pending:
            return
        slots = torch.from_numpy(np.concatenate([p[0] for p in pending])).to(device)
        k = torch.cat([p[1] for p in pending]).to(device)
        v = torch.cat([p[2] for p in pending]).to(device)
        if quant is None:
            pkv.pkv_kv_append(k, v, slots, c.k_pool, c.v_pool)
        else:
            pos = torch.from_numpy(np.concatenate([p[3] for p in pending]).astype(np.int32)).to(device)
            sidx = torch.from_numpy(np.concatenate([p[4] for p in pending]).astype(np.int32)).to(device)
            pkv.pkv_kv_append_quant(k, v, slots, pos, sidx, c.cache, n_sink, quant, c.group_size,
                                    window=getattr(c, "window", 0))
        pending.clear()

    c.all_pairs = []

    def do_append(h, n, slots, pairs):
        start = lens.get(h, 0)
        c.all_pairs += list(pairs)
        if pairs:
            flush()
            pr = torch.tensor(np.array(pairs, dtype=np.int32).reshape(-1, 2), device=device)
            pkv.pkv_copy_blocks(c.pools, pr)
        k, v = rows(h, start, n)
        pos = np.arange(start, start + n)
        # sink rows go to the decoded handle's batch row; a prompt holder
        # (not decoded) writes row 0, and every child's row gets the prompt's
        # sink tokens after the prefill
        sidx = np.full(n, row_of_handle.get(h, 0))
        pending.append((np.asarray(slots, dtype=np.int64), k, v, pos, sidx))
        lens[h] = start + n

    for op in ops:
        if op[0] == "create":
            pkv.pkv_seq_create(pool)
        elif op[0] == "fork":
            child = pkv.pkv_seq_fork(pool, op[1])
            lens[child] = lens.get(op[1], 0)
        else:
            _, h, n = op
            slots, pairs = pkv.pkv_seq_append(pool, h, n)
            do_append(h, n, slots, pairs)
    flush()
    if quant is not None and "prompt" in w:
        # children inherit the prompt's sink tokens: copy them into each row
        kp, vp = rows(0, 0, n_sink)
        for r in range(B):
            c.cache["sink_k"][r, :n_sink] = kp.to(device)
            c.cache["sink_v"][r, :n_sink] = vp.to(device)
    # the decode step: one token per decoded sequence
    slots, pairs = pkv.pkv_seq_append_batch(pool, decoded, 1)
    if len(pairs):
        pkv.pkv_copy_blocks(c.pools, torch.from_numpy(np.ascontiguousarray(pairs)).to(device))
    c.step_pairs = [tuple(int(x) for x in p) for p in pairs]
    c.all_pairs += c.step_pairs
    c.step_slots = slots.copy()
    if step_append:
        for i, h in enumerate(decoded):
            do_append(h, 1, slots[i:i + 1], [])
        flush()
    else:
        # leave the step's rows unwritten: a fused append+decode writes them
        nk, nv = [], []
        for h in decoded:
            k, v = rows(h, lens.get(h, 0), 1)
            nk.append(k[0])
            nv.append(v[0])
            lens[h] = lens.get(h, 0) + 1
        c.new_k = torch.stack(nk).to(device)
        c.new_v = torch.stack(nv).to(device)
    c.max_blocks = max(pkv.pkv_seq_num_blocks(pool, h) for h in decoded)
    tables, ctx = pkv.pkv_build_block_tables(pool, decoded, c.max_blocks)
    c.tables_host, c.lens_host = tables, ctx
    c.tables = torch.from_numpy(tables).to(device)
    c.lens = torch.from_numpy(ctx).to(device)
    c.q = syn.query(w).to(device)
    c.rows = rows
    c.handle_len = lens
    torch.cuda.synchronize()
    return c


def logical_rows(c, i):
    """Logical (k, v) rows of decoded sequence i as float32 NumPy arrays."""
    h = c.decoded[i]
    L = int(c.lens_host[i])
    w = c.w
    if "prompt" in w:
        k, v = syn.sequence_kv(w, h - 1)
    else:
        k, v = syn.sequence_kv(w, h)
    assert k.shape[0] == L
    return syn.kv_rows_to_numpy(k), syn.kv_rows_to_numpy(v)


def expected(c, seq_ids=None):
    """Oracle decode output [len(seq_ids), Hq, D] (float64)."""
    q = syn.kv_rows_to_numpy(syn.query(c.w))
    ids = range(len(c.decoded)) if seq_ids is None else seq_ids
    out = []
    for i in ids:
        k, v = logical_rows(c, i)
        if c.quant is None:
            out.append(oatt.sequence_attention(q[i], k, v, c.w["scale"]))
        else:
            out.append(okv.sequence_attention_quant(q[i], k, v, c.w["scale"], c.n_sink, c.quant,
                                                    getattr(c, "group_size", c.w["d"]),
                                                    window=getattr(c, "window", 0)))
    return np.stack(out)


def _expected_one(args):
    """Oracle output of one sequence, regenerated from the seeded workload
    (runs in a worker process)."""
    w, idx, q_row, quant, n_sink, group_size, window = args
    k, v = syn.sequence_kv(w, idx)
    k, v = syn.kv_rows_to_numpy(k), syn.kv_rows_to_numpy(v)
    if quant is None:
        return oatt.sequence_attention(q_row, k, v, w["scale"])
    return okv.sequence_attention_quant(q_row, k, v, w["scale"], n_sink, quant, group_size,
                                        window=window)


def expected_parallel(c, seq_ids=None, workers=None):
    """``expected`` computed in worker processes, one sequence each.

    The pool is started with ``spawn``: the calling process already holds a
    CUDA context, and a forked child of it would hang."""
    import multiprocessing
    import os
    from concurrent.futures import ProcessPoolExecutor
    q = syn.kv_rows_to_numpy(syn.query(c.w))
    ids = list(range(len(c.decoded)) if seq_ids is None else seq_ids)
    prefix = "prompt" in c.w
    jobs = [(c.w, (c.decoded[i] - 1) if prefix else c.decoded[i], q[i], c.quant, c.n_sink,
             getattr(c, "group_size", c.w["d"]), getattr(c, "window", 0)) for i in ids]
    n = workers or max(1, min(len(jobs), (os.cpu_count() or 1), 16))
    with ProcessPoolExecutor(max_workers=n, mp_context=multiprocessing.get_context("spawn")) as ex:
        return np.stack(list(ex.map(_expected_one, jobs)))


def assert_close(got, want, atol=2e-3, rtol=1e-2, what=""):
    """|got - want| <= atol + rtol * |want| element-wise (the acceptance bound)."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d / %d elements out of tolerance; max abs err %.3g; first %s"
                             % (what, bad.sum(), bad.size, err.max(), idx.tolist()))
    return float(err.max())
