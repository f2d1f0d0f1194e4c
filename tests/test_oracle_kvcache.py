"""Pins of the oracle's KV-append scatter and copy-on-write block copy.

These two functions are the expected values of the GPU append and CoW tests,
so they are pinned here to what the pages fix rather than to themselves:

* the slot rule of "The 8GB VRAM Breakthrough", §3 "How Logical-to-Physical
  Block Tables Work": the token at logical position t of a sequence whose
  table maps logical block t // 16 to physical block b lives at offset
  t % 16 of b (the page's 412 / 089 / 903 table is the worked case);
* "PagedAttention aplica memória virtual ao cache KV de LLMs", section
  "Compartilhamento e compromissos": paging changes the layout, not the
  result, and a write to shared memory copies only the block it touches;
* "A Ideia de 60 Anos Que Domou a Memória da GPU", section "o bônus que paga
  o ingresso: compartilhar": only the affected block is copied, then written.

Each check is built so that a transposed (block, offset) pair, a head/offset
swap, a dropped negative-slot test, or a copy of more than the named blocks
fails at least one of them.
"""

import numpy as np
import pytest

from conftest import read_golden
from oracle import allocator, attention, kvcache


def _distinct_rows(rng, T, Hkv, D):
    """Rows whose every element is different, so any misplacement shows."""
    base = np.arange(T * Hkv * D, dtype=np.float64).reshape(T, Hkv, D)
    return base + rng.random((T, Hkv, D)) * 0.5


# ------------------------------------------------------------------ kv_append
def test_append_lands_at_the_pages_table_positions():
    # The page's table: logical block 0 -> #412, 1 -> #089, 2 -> #903.  The
    # slots below are worked by hand from it: token 5 -> 412*16+5 = 6597,
    # token 20 -> 89*16+4 = 1428, token 47 -> 903*16+15 = 14463, token 0 ->
    # 6592, token 16 -> 1424, token 32 -> 14448.
    rows = [[int(x) for x in r] for r in read_golden("block_table_example.txt")]
    assert [r[3] for r in rows] == [412, 89, 903]
    cases = [  # (slot, physical block, offset) -- literal, not recomputed
        (6597, 412, 5), (1428, 89, 4), (14463, 903, 15),
        (6592, 412, 0), (1424, 89, 0), (14448, 903, 0),
    ]
    Hkv, D, NB = 3, 5, 1024
    rng = np.random.default_rng(11)
    k = _distinct_rows(rng, len(cases), Hkv, D)
    v = -_distinct_rows(rng, len(cases), Hkv, D)
    k_pool = np.full((NB, Hkv, 16, D), np.nan)
    v_pool = np.full((NB, Hkv, 16, D), np.nan)
    kvcache.kv_append(k, v, [c[0] for c in cases], k_pool, v_pool)
    written = np.zeros((NB, 16), dtype=bool)
    for t, (_, blk, off) in enumerate(cases):
        for h in range(Hkv):
            np.testing.assert_array_equal(k_pool[blk, h, off], k[t, h])
            np.testing.assert_array_equal(v_pool[blk, h, off], v[t, h])
        written[blk, off] = True
    # nothing else was touched
    by_slot_k = k_pool.transpose(0, 2, 1, 3)  # [NB, 16, Hkv, D]
    by_slot_v = v_pool.transpose(0, 2, 1, 3)
    assert np.isnan(by_slot_k[~written]).all() and np.isnan(by_slot_v[~written]).all()


def test_append_skips_negative_slots():
    Hkv, D = 2, 4
    rng = np.random.default_rng(12)
    k = _distinct_rows(rng, 4, Hkv, D)
    v = _distinct_rows(rng, 4, Hkv, D) + 1000
    k_pool = np.zeros((4, Hkv, 16, D))
    v_pool = np.zeros((4, Hkv, 16, D))
    # slot 17 is block 1, offset 1; slot 63 is block 3, offset 15
    kvcache.kv_append(k, v, [-1, 17, -5, 63], k_pool, v_pool)
    np.testing.assert_array_equal(k_pool[1, :, 1], k[1])
    np.testing.assert_array_equal(v_pool[3, :, 15], v[3])
    k_pool[1, :, 1] = 0
    k_pool[3, :, 15] = 0
    v_pool[1, :, 1] = 0
    v_pool[3, :, 15] = 0
    assert not k_pool.any() and not v_pool.any()


def test_append_honours_block_size():
    # block size 8: slot 13 is block 1, offset 5; slot 8 is block 1, offset 0
    k = np.arange(2 * 1 * 3, dtype=np.float64).reshape(2, 1, 3) + 1
    k_pool = np.zeros((4, 1, 8, 3))
    v_pool = np.zeros((4, 1, 8, 3))
    kvcache.kv_append(k, -k, [13, 8], k_pool, v_pool, block_size=8)
    np.testing.assert_array_equal(k_pool[1, 0, 5], k[0, 0])
    np.testing.assert_array_equal(v_pool[1, 0, 0], -k[1, 0])
    assert np.count_nonzero(k_pool) == 6


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_scatter_through_manager_slots_equals_slab_attention(seed):
    # Interleaved appends of several sequences through a shuffled pool, every
    # row written by kv_append at the manager's slot.  Paged attention through
    # the tables must then equal attention over each sequence's contiguous
    # slab, bit for bit (paging changes layout, not results).
    rng = np.random.default_rng(100 + seed)
    Hkv, G, D, NB, bs = 2, 3, 8, 96, 16
    order = rng.permutation(NB)
    m = allocator.KVCacheManager(NB, bs, free_order=order)
    lens_target = [int(x) for x in rng.integers(1, 120, size=5)]
    sids = [m.create() for _ in lens_target]
    slab_k = np.zeros((len(sids), Hkv, max(lens_target), D))
    slab_v = np.zeros_like(slab_k)
    k_pool = np.full((NB, Hkv, bs, D), np.nan)
    v_pool = np.full((NB, Hkv, bs, D), np.nan)
    done = [0] * len(sids)
    while done != lens_target:
        i = int(rng.integers(len(sids)))
        n = min(int(rng.integers(1, 20)), lens_target[i] - done[i])
        if n == 0:
            continue
        slots, copies = m.append(sids[i], n)
        assert copies == []
        k = rng.standard_normal((n, Hkv, D))
        v = rng.standard_normal((n, Hkv, D))
        kvcache.kv_append(k, v, slots, k_pool, v_pool, block_size=bs)
        slab_k[i, :, done[i]:done[i] + n] = k.transpose(1, 0, 2)
        slab_v[i, :, done[i]:done[i] + n] = v.transpose(1, 0, 2)
        done[i] += n
    tables, lens = m.block_tables(sids, max(len(m.table(s)) for s in sids))
    q = rng.standard_normal((len(sids), Hkv * G, D))
    paged = attention.paged_attention_decode(q, k_pool, v_pool, tables, lens, 0.35, block_size=bs)
    slab = attention.slab_attention_decode(q, slab_k, slab_v, lens, 0.35)
    np.testing.assert_array_equal(paged, slab)


def test_planted_transpose_in_append_is_caught():
    # The same scatter with (block, offset) swapped, planted here on the CPU,
    # breaks the slab equality: the check above can see this mistake.
    rng = np.random.default_rng(5)
    Hkv, D, NB = 1, 4, 32
    m = allocator.KVCacheManager(NB, 16, free_order=rng.permutation(NB))
    s = m.create()
    slots, _ = m.append(s, 40)
    k = rng.standard_normal((40, Hkv, D))
    v = rng.standard_normal((40, Hkv, D))
    k_pool = np.zeros((NB, Hkv, 16, D))
    v_pool = np.zeros((NB, Hkv, 16, D))
    for t, slot in enumerate(slots):
        blk, off = divmod(slot, 16)
        if off < NB and blk < 16:
            k_pool[off, :, blk] = k[t]
            v_pool[off, :, blk] = v[t]
    tables, lens = m.block_tables([s], 3)
    q = rng.standard_normal((1, 1, D))
    paged = attention.paged_attention_decode(q, k_pool, v_pool, tables, lens, 0.5)
    slab = attention.slab_attention_decode(q, k.transpose(1, 0, 2)[None], v.transpose(1, 0, 2)[None],
                                           lens, 0.5)
    assert not np.array_equal(paged, slab)


# ---------------------------------------------------------------- copy_blocks
def _cow_setup(prompt_len, n_fork, seed):
    rng = np.random.default_rng(seed)
    Hkv, D, NB, bs = 2, 8, 64, 16
    m = allocator.KVCacheManager(NB, bs, free_order=rng.permutation(NB))
    p = m.create()
    slots, _ = m.append(p, prompt_len)
    pk = rng.standard_normal((prompt_len, Hkv, D))
    pv = rng.standard_normal((prompt_len, Hkv, D))
    # four pools of different shapes, as a quantised cache has (codes,
    # scales, zeros) besides K and V; every entry distinct
    pools = [np.full((NB, Hkv, bs, D), np.nan), np.full((NB, Hkv, bs, D), np.nan),
             np.arange(NB * Hkv * bs * 3, dtype=np.float64).reshape(NB, Hkv, bs, 3),
             np.arange(NB * 7, dtype=np.float64).reshape(NB, 7) * -1]
    kvcache.kv_append(pk, pv, slots, pools[0], pools[1])
    kids = [m.fork(p) for _ in range(n_fork)]
    return rng, m, p, kids, pools, pk, pv


def test_copy_blocks_clones_only_the_written_block():
    # 24-token prompt: its second block holds 8 tokens and is shared after the
    # fork, so a child's first write clones exactly that block.
    rng, m, p, kids, pools, pk, pv = _cow_setup(24, 3, 21)
    shared_tail = m.table(p)[1]
    for child in kids:
        slots, copies = m.append(child, 1)
        assert len(copies) == 1 and copies[0][0] == shared_tail
        before = [x.copy() for x in pools]
        kvcache.copy_blocks(pools, copies)
        src, dst = copies[0]
        for x, old in zip(pools, before):
            np.testing.assert_array_equal(x[dst], old[src])
            keep = np.ones(x.shape[0], dtype=bool)
            keep[dst] = False
            np.testing.assert_array_equal(x[keep], old[keep])  # nothing else changed
        # then the child's new row goes into the clone, not the shared block
        nk = rng.standard_normal((1, 2, 8))
        kvcache.kv_append(nk, -nk, slots, pools[0], pools[1])
        np.testing.assert_array_equal(pools[0][dst, :, 8], nk[0])
        np.testing.assert_array_equal(pools[0][shared_tail, :, :8],
                                      pk[16:24].transpose(1, 0, 2))
        assert np.isnan(pools[0][shared_tail, :, 8]).all()


def test_copy_on_write_keeps_every_sequence_exact():
    # After the clones and one private token per child, paged attention of
    # the holder and of every child equals attention over its logical rows.
    rng, m, p, kids, pools, pk, pv = _cow_setup(40, 4, 22)
    logical = {p: (pk, pv)}
    for child in kids:
        slots, copies = m.append(child, 3)
        kvcache.copy_blocks(pools, copies)
        nk = rng.standard_normal((3, 2, 8))
        nv = rng.standard_normal((3, 2, 8))
        kvcache.kv_append(nk, nv, slots, pools[0], pools[1])
        logical[child] = (np.concatenate([pk, nk]), np.concatenate([pv, nv]))
    sids = [p] + kids
    tables, lens = m.block_tables(sids, 3)
    q = rng.standard_normal((len(sids), 4, 8))
    paged = attention.paged_attention_decode(q, pools[0], pools[1], tables, lens, 0.4)
    for i, s in enumerate(sids):
        k, v = logical[s]
        want = attention.sequence_attention(q[i], k, v, 0.4)
        np.testing.assert_array_equal(paged[i], want)
    # shared full block counted once, tail cloned per child
    assert m.unique_blocks(sids) == 2 + 1 + len(kids)


def test_copy_blocks_applies_every_pair_to_every_pool():
    # several pairs that do not chain (no dst is another pair's src)
    pools = [np.arange(6 * 2, dtype=np.float64).reshape(6, 2),
             np.arange(6, dtype=np.float64) * 10]
    kvcache.copy_blocks(pools, [(0, 5), (2, 3), (4, 1)])
    np.testing.assert_array_equal(pools[0], [[0, 1], [8, 9], [4, 5], [4, 5], [8, 9], [0, 1]])
    np.testing.assert_array_equal(pools[1], [0, 40, 20, 20, 40, 0])


def test_planted_whole_pool_copy_is_caught():
    # A copy that writes more than the named block, planted here, changes
    # blocks outside the pair: the "nothing else changed" check sees it.
    pools = [np.arange(8 * 3, dtype=np.float64).reshape(8, 3)]
    before = pools[0].copy()
    pools[0][:] = pools[0][2]
    keep = np.ones(8, dtype=bool)
    keep[6] = False
    assert not np.array_equal(pools[0][keep], before[keep])
