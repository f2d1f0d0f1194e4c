"""GPU decode through block tables that the host prefix cache produced.

"Capítulo 8 — Gerenciamento de KV Cache de Próxima Geração", §8.3: a new
request's prompt is cut into block-sized chunks; every chunk already in the
cache is mapped into the request's table and its prefill skipped, and only
the rest is computed.  "The 8GB VRAM Breakthrough", §3 "Copy-on-Write (CoW)
Prefix Sharing": samples forked from one request share its blocks until a
write into the shared, partially filled tail block clones that block.

Each test drives the whole path through the library -- prefix match, the
KV-append of the unmatched rows, the batch append with its copy-on-write
pairs, the block copy and the fused append + decode -- and checks every
decoded output against the oracle's attention over that sequence's logical
rows, the tables against the oracle's allocator and prefix cache run on the
same operations, and the block accounting against the pages' best-of-8
figures.
"""

import math

import numpy as np
import pytest
import torch

import synthetic as syn
from cache_builder import assert_close
from oracle import allocator
from oracle import attention as oatt

pytestmark = pytest.mark.gpu


def _tokens(seed, n):
    return [int(x) for x in np.random.default_rng(seed).integers(0, 128256, size=n)]


class _Path:
    """The library's pool and device pools, with the oracle's allocator and
    prefix cache run on the same operations alongside."""

    def __init__(self, pkv, w, dev):
        self.pkv, self.w, self.dev = pkv, w, dev
        NB, BS = w["num_blocks"], w["block_size"]
        order = syn.free_order(w)
        self.pool = pkv.pkv_pool_create(NB, BS, order)
        self.m = allocator.KVCacheManager(NB, BS, order)
        self.cache = allocator.PrefixCache(self.m)
        shape = (NB, w["hkv"], BS, w["d"])
        # unwritten slots hold NaN: a row read from a slot nobody wrote shows
        self.kp = torch.full(shape, float("nan"), dtype=w["torch_dtype"], device=dev)
        self.vp = torch.full(shape, float("nan"), dtype=w["torch_dtype"], device=dev)
        self.copies = []

    def write(self, k, v, slots):
        if len(slots) == 0:
            return
        s = torch.from_numpy(np.ascontiguousarray(slots, dtype=np.int64)).to(self.dev)
        self.pkv.pkv_kv_append(k.contiguous().to(self.dev), v.contiguous().to(self.dev), s,
                               self.kp, self.vp)

    def append(self, sid, rsid, n):
        slots, pairs = self.pkv.pkv_seq_append(self.pool, sid, n)
        rslots, rpairs = self.m.append(rsid, n)
        np.testing.assert_array_equal(slots, np.array(rslots, dtype=np.int64))
        assert pairs == rpairs
        self.copy(np.array(pairs, dtype=np.int32).reshape(-1, 2))
        return slots

    def append_batch(self, sids, rsids):
        slots, pairs = self.pkv.pkv_seq_append_batch(self.pool, sids, 1)
        rslots, rpairs = [], []
        for r in rsids:
            s, p = self.m.append(r, 1)
            rslots += s
            rpairs += p
        np.testing.assert_array_equal(slots, np.array(rslots, dtype=np.int64))
        assert [tuple(int(x) for x in p) for p in pairs] == rpairs
        self.copy(pairs)
        return slots

    def copy(self, pairs):
        if len(pairs) == 0:
            return
        self.copies += [tuple(int(x) for x in p) for p in pairs]
        pr = torch.from_numpy(np.ascontiguousarray(pairs, dtype=np.int32)).to(self.dev)
        self.pkv.pkv_copy_blocks([self.kp, self.vp], pr)

    def decode_step(self, sids, rsids, q, new_k, new_v):
        """One decode step: reserve one slot per sequence, clone what must be
        cloned, then write the new rows and attend (fused)."""
        pkv, w = self.pkv, self.w
        slots = self.append_batch(sids, rsids)
        mb = max(pkv.pkv_seq_num_blocks(self.pool, s) for s in sids)
        tables, lens = pkv.pkv_build_block_tables(self.pool, sids, mb)
        rtables, rlens = self.m.block_tables(rsids, mb)
        np.testing.assert_array_equal(tables, np.array(rtables, dtype=np.int32))
        np.testing.assert_array_equal(lens, np.array(rlens, dtype=np.int32))
        B = len(sids)
        out = torch.empty((B, w["hq"], w["d"]), dtype=w["torch_dtype"], device=self.dev)
        ws = torch.empty(max(pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], mb), 16),
                         dtype=torch.uint8, device=self.dev)
        pkv.pkv_paged_attention_decode_append(
            q.to(self.dev), new_k.to(self.dev), new_v.to(self.dev),
            torch.from_numpy(slots.copy()).to(self.dev), self.kp, self.vp,
            torch.from_numpy(tables).to(self.dev), torch.from_numpy(lens).to(self.dev),
            w["scale"], out, workspace=ws)
        torch.cuda.synchronize()
        assert pkv.pkv_device_status() == 0
        return out.float().cpu().numpy(), tables, lens


def _expected(w, q, rows):
    qn = syn.kv_rows_to_numpy(q)
    return np.stack([oatt.sequence_attention(qn[i], syn.kv_rows_to_numpy(k), syn.kv_rows_to_numpy(v),
                                             w["scale"]) for i, (k, v) in enumerate(rows)])


def test_best_of_8_through_prefix_match_cow_and_decode(pkv, cuda_dev):
    """An earlier request computed a 2,008-token prompt and registered its
    125 full blocks.  A new request with that prompt maps them, prefills only
    the 8 unmatched tokens, and forks 8 samples (best-of-8) that share its
    partial tail block.  Each sample's first write clones that block (8
    clones, the request keeps the original); each then decodes over its own
    tail of 1..300 tokens."""
    w = syn.workload("prefix_cow_2008")
    P, bs = w["prompt"], w["block_size"]
    tails = syn.tails(w)
    path = _Path(pkv, w, cuda_dev)
    pk, pv = syn.prompt_kv(w)
    ids = _tokens(2008, P)

    a = pkv.pkv_seq_create(path.pool)
    ra = path.m.create()
    path.write(pk, pv, path.append(a, ra, P))
    n_reg = pkv.pkv_prefix_register(path.pool, a, ids)
    assert n_reg == path.cache.register(ra, ids) == P // bs
    pkv.pkv_seq_free(path.pool, a)
    path.m.free(ra)

    r, matched = pkv.pkv_prefix_match(path.pool, ids)
    rr, rmatched = path.cache.match(ids)
    assert (r, matched) == (rr, rmatched) and matched == P // bs * bs == 2000
    path.write(pk[matched:], pv[matched:], path.append(r, rr, P - matched))
    assert path.copies == []
    shared_tail = int(pkv.pkv_seq_block_table(path.pool, r)[-1])

    kids = [pkv.pkv_seq_fork(path.pool, r) for _ in tails]
    rkids = [path.m.fork(rr) for _ in tails]
    assert kids == rkids
    rows = [syn.sequence_kv(w, i) for i in range(len(tails))]
    # the first tail token of every sample that has one before the decode
    # token goes in through one batch append: the copy-on-write step
    first = [i for i, t in enumerate(tails) if t >= 2]
    slots = path.append_batch([kids[i] for i in first], [rkids[i] for i in first])
    path.write(torch.stack([rows[i][0][P] for i in first]),
               torch.stack([rows[i][1][P] for i in first]), slots)
    for i in first:
        n = tails[i] - 2
        if n > 0:
            path.write(rows[i][0][P + 1:P + 1 + n], rows[i][1][P + 1:P + 1 + n],
                       path.append(kids[i], rkids[i], n))
    q = syn.query(w)
    new_k = torch.stack([k[-1] for k, _ in rows])
    new_v = torch.stack([v[-1] for _, v in rows])
    got, tables, lens = path.decode_step(kids, rkids, q, new_k, new_v)
    np.testing.assert_array_equal(lens, [P + t for t in tails])

    # every sample cloned the shared partial block exactly once
    assert len(path.copies) == len(tails)
    assert all(src == shared_tail for src, _ in path.copies)
    assert len({dst for _, dst in path.copies}) == len(tails)
    # shared blocks counted once: 125 cached, the request's tail, and each
    # sample's own blocks from the clone on
    held = set(tables[tables >= 0].tolist()) | set(pkv.pkv_seq_block_table(path.pool, r).tolist())
    assert len(held) == P // bs + 1 + sum(math.ceil((P % bs + t) / bs) for t in tails)
    for b in pkv.pkv_seq_block_table(path.pool, r)[:-1]:
        assert pkv.pkv_block_refcount(path.pool, int(b)) == 1 + 1 + len(tails)  # cache, request, samples
    assert pkv.pkv_block_refcount(path.pool, shared_tail) == 1
    entries, lookups, hit_blocks = pkv.pkv_prefix_stats(path.pool)
    assert (entries, lookups, hit_blocks) == (len(path.cache.entries), path.cache.lookups,
                                              path.cache.hit_blocks)
    assert hit_blocks == P // bs

    assert_close(got, _expected(w, q, rows), what="best-of-8 through the prefix cache")
    pkv.pkv_pool_destroy(path.pool)


def test_shared_system_prompt_requests_decode_exactly(pkv, cuda_dev):
    """Eight requests share a 2,000-token system prompt and differ after it.
    They arrive one after another: the first computes and registers every
    full block it holds, each later one maps the 125 prompt blocks, prefills
    only its own suffix and registers its own full blocks.  All eight then
    decode one step together."""
    w = syn.workload("prefix_cow")
    P, bs = w["prompt"], w["block_size"]
    lens_all = syn.context_lengths(w)
    path = _Path(pkv, w, cuda_dev)
    prompt_ids = _tokens(2000, P)
    rows = [syn.sequence_kv(w, i) for i in range(len(lens_all))]
    sids, rsids = [], []
    for i, L in enumerate(lens_all):
        ids = prompt_ids + _tokens(3000 + i, L - 1 - P)
        sid, matched = pkv.pkv_prefix_match(path.pool, ids)
        rsid, rmatched = path.cache.match(ids)
        assert (sid, matched) == (rsid, rmatched)
        assert matched == (0 if i == 0 else P)
        k, v = rows[i]
        path.write(k[matched:L - 1], v[matched:L - 1], path.append(sid, rsid, L - 1 - matched))
        assert (pkv.pkv_prefix_register(path.pool, sid, ids)
                == path.cache.register(rsid, ids))
        sids.append(sid)
        rsids.append(rsid)
    assert path.copies == []
    q = syn.query(w)
    new_k = torch.stack([k[-1] for k, _ in rows])
    new_v = torch.stack([v[-1] for _, v in rows])
    got, tables, lens = path.decode_step(sids, rsids, q, new_k, new_v)
    np.testing.assert_array_equal(lens, lens_all)
    # the prompt's blocks are the same physical blocks in every table
    assert (tables[:, :P // bs] == tables[0, :P // bs]).all()
    held = set(tables[tables >= 0].tolist())
    assert len(held) == P // bs + sum(math.ceil((L - P) / bs) for L in lens_all)
    entries, lookups, hit_blocks = pkv.pkv_prefix_stats(path.pool)
    assert hit_blocks == (len(lens_all) - 1) * (P // bs)
    assert (entries, lookups, hit_blocks) == (len(path.cache.entries), path.cache.lookups,
                                              path.cache.hit_blocks)
    assert_close(got, _expected(w, q, rows), what="system prompt through the prefix cache")
    pkv.pkv_pool_destroy(path.pool)
