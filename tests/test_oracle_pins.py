"""Pins of the oracle's byte accounting and allocator to what the pages print."""

import math
import random

import pytest

from conftest import read_golden
from oracle import allocator, kv_bytes

GiB = 1 << 30
KiB = 1 << 10


def _golden_dict(name):
    return {r[0]: r[1:] for r in read_golden(name)}


# ---------------------------------------------------------------- bytes
def test_kv_bytes_match_printed_figures():
    g = {k: float(v[0]) for k, v in _golden_dict("kv_bytes.txt").items()}
    L, H, D = 32, 8, 128
    bpt = kv_bytes.kv_bytes_per_token(L, H, D, 2)
    assert bpt == g["fp16_bytes_per_token"]
    assert bpt / KiB == g["fp16_kib_per_token"]
    for s, key in ((8192, "fp16_gib_at_8192"), (32768, "fp16_gib_at_32768"), (65536, "fp16_gib_at_65536")):
        assert kv_bytes.kv_cache_bytes(L, H, D, s, 1, 2) / GiB == g[key]
    assert kv_bytes.fp8_code_bytes_per_token(L, H, D) / KiB == g["fp8_kib_per_token"]
    assert kv_bytes.fp8_code_bytes_per_token(L, H, D) * 65536 / GiB == g["fp8_gib_at_65536"]
    assert kv_bytes.int4_group_bytes(64) == g["int4_g64_bytes_per_group"]
    assert kv_bytes.int4_group_bytes(64) * 8 / 64 == g["int4_g64_bits_per_element"]
    assert 2 * L * H * D == g["int4_elements_per_token"]
    ipt = kv_bytes.int4_bytes_per_token(L, H, D, 64)
    assert ipt == g["int4_g64_bytes_per_token"]
    assert ipt / KiB == g["int4_g64_kib_per_token"]
    assert ipt * 65536 / GiB == g["int4_g64_gib_at_65536"]


def test_kv_equation_is_linear_in_every_factor():
    base = kv_bytes.kv_cache_bytes(2, 3, 5, 7, 11, 2)
    assert kv_bytes.kv_cache_bytes(4, 3, 5, 7, 11, 2) == 2 * base
    assert kv_bytes.kv_cache_bytes(2, 3, 5, 14, 11, 2) == 2 * base
    assert kv_bytes.kv_cache_bytes(2, 3, 5, 7, 22, 2) == 2 * base
    assert kv_bytes.kv_cache_bytes(2, 3, 5, 7, 11, 1) * 2 == base


def test_per_layer_bytes_used_by_the_measurements():
    # one layer, 8 KV heads, head dim 128: bf16 K+V, INT4 (group = dim), FP8
    assert kv_bytes.kv_bytes_per_token(1, 8, 128, 2) == 4096
    assert kv_bytes.int4_bytes_per_token_per_layer(8, 128, 128) == 1088
    assert kv_bytes.fp8_bytes_per_token_per_layer_with_scales(8, 128) == 2080


# ------------------------------------------------------------ allocator
def test_worked_allocation_25_47_12():
    g = _golden_dict("worked_allocation.txt")
    bs = int(g["block_size"][0])
    lens = [int(x) for x in g["lens"]]
    m = allocator.KVCacheManager(num_blocks=64, block_size=bs)
    sids = []
    for L in lens:
        s = m.create()
        m.append(s, L)
        sids.append(s)
    used_blocks = sum(len(m.table(s)) for s in sids)
    assert used_blocks * bs == int(g["paged_slots"][0])
    per_request_max = int(g["contiguous_slots"][0]) // len(lens)
    assert per_request_max * len(lens) == int(g["contiguous_slots"][0])
    assert int(g["contiguous_slots"][0]) // (used_blocks * bs) == int(g["ratio"][0])
    assert m.pool.num_free() == 64 - used_blocks


def test_block_table_example():
    rows = [[int(x) for x in r] for r in read_golden("block_table_example.txt")]
    first = [r[3] for r in rows]
    order = first + [b for b in range(1024) if b not in first]
    m = allocator.KVCacheManager(num_blocks=1024, block_size=16, free_order=order)
    s = m.create()
    slots, copies = m.append(s, 48)
    assert copies == []
    assert m.table(s) == first
    for logical, t0, t1, phys in rows:
        for t in (t0, t1):
            assert t // 16 == logical
            assert slots[t] == phys * 16 + t % 16


def test_best_of_8_accounting():
    g = _golden_dict("best_of_8.txt")
    prompt, n = int(g["prompt"][0]), int(g["samples"][0])
    unshared, shared = int(g["unshared_token_slots"][0]), int(g["shared_token_slots"][0])
    c = (unshared - n * prompt) // n
    assert n * (prompt + c) == unshared and prompt + n * c == shared
    m = allocator.KVCacheManager(num_blocks=4096)
    p = m.create()
    m.append(p, prompt)
    kids = [m.fork(p) for _ in range(n)]
    copies = []
    for k in kids:
        copies += m.append(k, c)[1]
    assert copies == []  # 2000 = 125 * 16: the shared tail block is full
    unique = m.unique_blocks([p] + kids)
    assert unique == prompt // 16 + n * math.ceil(c / 16) == 181
    # token slots actually holding tokens: shared prompt once + each continuation
    assert prompt + n * c == shared
    assert unique * 16 >= shared


def test_tail_waste_at_most_block_minus_one():
    rnd = random.Random(7)
    m = allocator.KVCacheManager(num_blocks=100000)
    for _ in range(200):
        L = rnd.randint(1, 5000)
        s = m.create()
        m.append(s, L)
        waste = len(m.table(s)) * 16 - L
        assert 0 <= waste <= 15


def test_on_demand_growth_one_block_per_16_tokens():
    m = allocator.KVCacheManager(num_blocks=64)
    s = m.create()
    for L in range(1, 100):
        m.append(s, 1)
        assert len(m.table(s)) == -(-L // 16)


def test_cow_clones_only_partial_shared_block():
    m = allocator.KVCacheManager(num_blocks=4096)
    p = m.create()
    m.append(p, 2008)
    shared_tail = m.table(p)[-1]
    kids = [m.fork(p) for _ in range(8)]
    assert m.pool.ref[shared_tail] == 9
    clones = []
    for i, k in enumerate(kids):
        slots, copies = m.append(k, 1)
        assert len(copies) == 1 and copies[0][0] == shared_tail
        clones.append(copies[0][1])
        assert m.table(k)[:-1] == m.table(p)[:-1]  # full blocks stay shared
        assert m.table(k)[-1] == copies[0][1]
        assert slots[0] == copies[0][1] * 16 + 2008 % 16
        assert m.pool.ref[shared_tail] == 9 - (i + 1)
    assert len(set(clones)) == 8
    # the holder keeps the original block; full prompt blocks counted once
    assert m.unique_blocks([p] + kids) == 126 + 8
    # a second write to a child's own (now private) block clones nothing
    assert m.append(kids[0], 1)[1] == []


def test_cow_full_tail_block_needs_no_clone():
    m = allocator.KVCacheManager(num_blocks=4096)
    p = m.create()
    m.append(p, 2000)
    kids = [m.fork(p) for _ in range(8)]
    for k in kids:
        slots, copies = m.append(k, 1)
        assert copies == []
        assert len(m.table(k)) == 126
    assert m.unique_blocks([p] + kids) == 125 + 8


def test_last_owner_writes_in_place():
    m = allocator.KVCacheManager(num_blocks=64)
    p = m.create()
    m.append(p, 20)
    k = m.fork(p)
    m.free(p)
    assert m.append(k, 1)[1] == []  # ref back to 1: no clone


def test_refcounts_return_to_zero_and_stack_refills():
    rnd = random.Random(3)
    order = list(range(256))
    rnd.shuffle(order)
    m = allocator.KVCacheManager(num_blocks=256, free_order=order)
    live = []
    for _ in range(300):
        op = rnd.random()
        if op < 0.3 or not live:
            s = m.create()
            live.append(s)
        elif op < 0.45:
            live.append(m.fork(rnd.choice(live)))
        elif op < 0.85:
            try:
                m.append(rnd.choice(live), rnd.randint(1, 40))
            except allocator.OutOfBlocks:
                pass
        else:
            s = live.pop(rnd.randrange(len(live)))
            m.free(s)
    for s in live:
        m.free(s)
    assert all(r == 0 for r in m.pool.ref)
    assert sorted(m.pool.free) == list(range(256))


def test_out_of_blocks_is_atomic():
    m = allocator.KVCacheManager(num_blocks=4)
    s = m.create()
    m.append(s, 40)  # 3 blocks
    before = (m.table(s), m.length(s), list(m.pool.free), list(m.pool.ref))
    with pytest.raises(allocator.OutOfBlocks):
        m.append(s, 30)  # needs 2 more, only 1 free
    assert (m.table(s), m.length(s), list(m.pool.free), list(m.pool.ref)) == before


def test_double_free_detected():
    pool = allocator.BlockPool(4)
    b = pool.alloc()
    pool.decref(b)
    with pytest.raises(allocator.DoubleFree):
        pool.decref(b)


def test_lifo_reuse_of_freed_block():
    pool = allocator.BlockPool(8, free_order=[5, 3, 1, 0, 2, 4, 6, 7])
    assert [pool.alloc() for _ in range(3)] == [5, 3, 1]
    pool.decref(3)
    assert pool.alloc() == 3
    assert pool.alloc() == 0
