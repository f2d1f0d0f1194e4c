"""Prefix cache ("Capítulo 8 — Gerenciamento de KV Cache de Próxima
Geração", §8.3): the oracle's cache against the pages' accounting, and the
C++ cache (through the C ABI, no GPU) against the oracle, op by op."""

import random

import numpy as np
import pytest

from conftest import read_golden
from oracle import allocator


def _tokens(rng, n):
    return [int(x) for x in rng.integers(0, 128256, size=n)]


def test_oracle_best_of_8_through_the_prefix_cache():
    """Eight samples of one 2,000-token prompt: the first computes and
    registers the prompt's 125 blocks, the other seven map them; each sample
    then decodes 100 tokens of its own.  Token slots: 2,000 + 8 x 100 =
    2,800 instead of 16,800 (the pages' best-of-8 figures), 181 blocks."""
    g = {k: v for k, v in read_golden("best_of_8.txt")}
    P, S = int(g["prompt"]), int(g["samples"])
    per_sample = (int(g["unshared_token_slots"]) // S) - P
    m = allocator.KVCacheManager(4096)
    cache = allocator.PrefixCache(m)
    prompt = _tokens(np.random.default_rng(0), P)
    first = m.create()
    m.append(first, P)
    assert cache.register(first, prompt) == P // 16
    sids = [first]
    for _ in range(S - 1):
        sid, matched = cache.match(prompt)
        assert matched == P
        sids.append(sid)
    for sid in sids:
        m.append(sid, per_sample)
    tokens_held = P + sum(m.length(s) - P for s in sids)
    assert tokens_held == int(g["shared_token_slots"])
    assert S * (P + per_sample) == int(g["unshared_token_slots"])
    assert m.unique_blocks(sids) == P // 16 + S * -(-per_sample // 16) == 181


def test_oracle_chunks_are_position_dependent():
    m = allocator.KVCacheManager(64)
    cache = allocator.PrefixCache(m)
    rng = np.random.default_rng(1)
    a, b = _tokens(rng, 16), _tokens(rng, 16)
    s = m.create()
    m.append(s, 32)
    assert cache.register(s, a + b) == 2
    assert cache.match(b + a)[1] == 0        # b is cached only after a
    assert cache.match(a + _tokens(rng, 16))[1] == 16
    assert cache.match(a + b + a)[1] == 32
    assert cache.match(a[:15])[1] == 0       # only full blocks


def test_oracle_system_prompt_hit_rate():
    """A shared 1,024-token system prompt with a 200-token user suffix per
    request: after the first request every later one maps the whole prompt
    (the pages cite >99% hit rates for a chat service's system prompt)."""
    m = allocator.KVCacheManager(20000)
    cache = allocator.PrefixCache(m)
    rng = np.random.default_rng(2)
    system = _tokens(rng, 1024)
    hits = 0
    for r in range(100):
        prompt = system + _tokens(rng, 200)
        sid, matched = cache.match(prompt)
        m.append(sid, len(prompt) - matched)
        cache.register(sid, prompt)
        hits += matched // 16
        m.free(sid)
    later = 99 * (1024 // 16)
    assert hits >= later  # every system-prompt block after the first request
    assert hits / (99 * (len(system) + 200) // 16) > 0.8


def test_oracle_eviction_frees_lru_leaves_only():
    m = allocator.KVCacheManager(16)
    cache = allocator.PrefixCache(m)
    rng = np.random.default_rng(3)
    t = _tokens(rng, 48)
    s = m.create()
    m.append(s, 48)
    cache.register(s, t)
    assert cache.evict(1) == 0          # the sequence still holds every block
    m.free(s)
    assert m.pool.num_free() == 16 - 3  # the cache holds them
    assert cache.evict(1) == 1          # the leaf (third block) goes first
    assert cache.match(t)[1] == 32
    assert cache.evict(10) == 0         # the match's sequence holds the rest
    cache.clear()


def _state(pkv, pool, m, cache, live):
    for sid in live:
        np.testing.assert_array_equal(pkv.pkv_seq_block_table(pool, sid), np.array(m.table(sid), dtype=np.int32))
        assert pkv.pkv_seq_len(pool, sid) == m.length(sid)
    assert pkv.pkv_pool_num_free(pool) == m.pool.num_free()
    for b in range(m.pool.num_blocks):
        assert pkv.pkv_block_refcount(pool, b) == m.pool.ref[b]
    assert pkv.pkv_prefix_stats(pool) == (len(cache.entries), cache.lookups, cache.hit_blocks)


@pytest.mark.parametrize("seed", range(6))
def test_cpp_prefix_cache_matches_oracle(pkv, seed):
    rnd = random.Random(seed)
    rng = np.random.default_rng(seed)
    NB, bs = 96, 16
    order = rng.permutation(NB).astype(np.int32)
    m = allocator.KVCacheManager(NB, bs, order)
    cache = allocator.PrefixCache(m)
    pool = pkv.pkv_pool_create(NB, bs, order)
    prompts = [_tokens(rng, rnd.randrange(0, 120)) for _ in range(4)]
    live = {}  # sid -> tokens it holds
    for step in range(120):
        op = rnd.random()
        if op < 0.35:   # a request: match, prefill the rest, register
            base = rnd.choice(prompts)
            toks = base[:rnd.randrange(0, len(base) + 1)] + _tokens(rng, rnd.randrange(0, 40))
            sid, matched = pkv.pkv_prefix_match(pool, toks)
            rsid, rmatched = cache.match(toks)
            assert (sid, matched) == (rsid, rmatched)
            need = len(toks) - matched
            try:
                rs, _ = m.append(rsid, need)
            except allocator.OutOfBlocks:
                with pytest.raises(pkv.PkvError):
                    pkv.pkv_seq_append(pool, sid, need)
                live[sid] = toks[:matched]
            else:
                slots, _ = pkv.pkv_seq_append(pool, sid, need)
                np.testing.assert_array_equal(slots, np.array(rs, dtype=np.int64))
                live[sid] = toks
            assert pkv.pkv_prefix_register(pool, sid, live[sid]) == cache.register(rsid, live[sid])
        elif op < 0.6 and live:   # finish a request
            sid = rnd.choice(sorted(live))
            pkv.pkv_seq_free(pool, sid)
            m.free(sid)
            del live[sid]
        elif op < 0.85:           # evict
            n = rnd.randrange(0, 6)
            assert pkv.pkv_prefix_evict(pool, n) == cache.evict(n)
        elif op < 0.9:
            pkv.pkv_prefix_clear(pool)
            cache.clear()
        _state(pkv, pool, m, cache, live)
    for sid in list(live):
        pkv.pkv_seq_free(pool, sid)
        m.free(sid)
    pkv.pkv_prefix_clear(pool)
    cache.clear()
    assert pkv.pkv_pool_num_free(pool) == NB
    pkv.pkv_pool_destroy(pool)


def test_cpp_prefix_errors(pkv):
    pool = pkv.pkv_pool_create(8, 16, None)
    s = pkv.pkv_seq_create(pool)
    pkv.pkv_seq_append(pool, s, 20)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_prefix_register(pool, s, list(range(21)))  # more tokens than held
    with pytest.raises(pkv.PkvError):
        pkv.pkv_prefix_register(pool, 12345, list(range(16)))  # no such sequence
    assert pkv.pkv_prefix_register(pool, s, list(range(20))) == 1  # one full block
    seq, matched = pkv.pkv_prefix_match(pool, list(range(40)))
    assert matched == 16 and pkv.pkv_block_refcount(pool, pkv.pkv_seq_block_table(pool, s)[0]) == 3
    pkv.pkv_pool_destroy(pool)
