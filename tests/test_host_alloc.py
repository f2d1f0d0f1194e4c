"""The C++ block manager (through the C ABI, no GPU) against the oracle's:
block tables, slot mappings and copy-on-write pairs must be bit-exact."""

import random

import numpy as np
import pytest

import synthetic as syn
from oracle import allocator


def _run_schedule_both(pkv, w):
    """Build the workload's cache layout with both managers, op by op."""
    order = syn.free_order(w)
    ref = allocator.KVCacheManager(w["num_blocks"], w["block_size"], order)
    pool = pkv.pkv_pool_create(w["num_blocks"], w["block_size"], order)
    ops, decoded = syn.prefill_schedule(w)
    for op in ops:
        if op[0] == "create":
            assert pkv.pkv_seq_create(pool) == ref.create()
        elif op[0] == "fork":
            assert pkv.pkv_seq_fork(pool, op[1]) == ref.fork(op[1])
        else:
            _, s, n = op
            slots, pairs = pkv.pkv_seq_append(pool, s, n)
            rs, rp = ref.append(s, n)
            np.testing.assert_array_equal(slots, np.array(rs, dtype=np.int64))
            assert pairs == rp
    # the decode step: one token for every decoded sequence
    slots, pairs = pkv.pkv_seq_append_batch(pool, decoded, 1)
    want_slots, want_pairs = [], []
    for s in decoded:
        rs, rp = ref.append(s, 1)
        want_slots += rs
        want_pairs += rp
    np.testing.assert_array_equal(slots, np.array(want_slots, dtype=np.int64))
    np.testing.assert_array_equal(pairs.reshape(-1, 2), np.array(want_pairs, dtype=np.int32).reshape(-1, 2))
    max_blocks = max(len(ref.table(s)) for s in decoded)
    tables, lens = pkv.pkv_build_block_tables(pool, decoded, max_blocks)
    rt, rl = ref.block_tables(decoded, max_blocks)
    np.testing.assert_array_equal(tables, np.array(rt, dtype=np.int32))
    np.testing.assert_array_equal(lens, np.array(rl, dtype=np.int32))
    assert list(lens) == syn.context_lengths(w)
    assert pkv.pkv_pool_num_free(pool) == ref.pool.num_free()
    for b in set(int(x) for x in tables.ravel() if x >= 0):
        assert pkv.pkv_block_refcount(pool, b) == ref.pool.ref[b]
    return pool, ref, decoded, want_pairs


@pytest.mark.parametrize("name", ["tiny", "llama3_8b_b64", "long_splitk", "quant", "prefix_cow",
                                  "prefix_cow_2008"])
def test_workload_tables_bit_exact(pkv, name):
    w = syn.workload(name)
    pool, ref, decoded, pairs = _run_schedule_both(pkv, w)
    if name == "prefix_cow":
        assert pairs == []  # 2000 = 125 * 16: the shared tail block is full
        assert ref.unique_blocks(decoded) == 125 + sum(
            len(ref.table(s)) - 125 for s in decoded)
    if name == "prefix_cow_2008":
        # every child clones the shared partial block exactly once, in the
        # append that first writes to it (prefill or the decode step)
        assert ref.pool.ref[ref.table(0)[-1]] == 1
    if name == "long_splitk":
        # round-robin allocation interleaves the sequences' blocks
        tables, _ = pkv.pkv_build_block_tables(pool, decoded, 4096)
        assert not np.array_equal(np.sort(tables[1, :2048]), np.sort(tables[2, :2048]))
    for s in list(ref.tables):
        pkv.pkv_seq_free(pool, s)
        ref.free(s)
    assert pkv.pkv_pool_num_free(pool) == w["num_blocks"]
    pkv.pkv_pool_destroy(pool)


def test_prefix_2008_clone_count(pkv):
    w = syn.workload("prefix_cow_2008")
    order = syn.free_order(w)
    pool = pkv.pkv_pool_create(w["num_blocks"], 16, order)
    p = pkv.pkv_seq_create(pool)
    pkv.pkv_seq_append(pool, p, 2008)
    kids = [pkv.pkv_seq_fork(pool, p) for _ in range(8)]
    shared = pkv.pkv_seq_block_table(pool, p)[-1]
    assert pkv.pkv_block_refcount(pool, shared) == 9
    slots, pairs = pkv.pkv_seq_append_batch(pool, kids, 1)
    assert pairs.shape == (8, 2) and (pairs[:, 0] == shared).all()
    assert len(set(pairs[:, 1])) == 8
    assert pkv.pkv_block_refcount(pool, shared) == 1
    pkv.pkv_pool_destroy(pool)


def test_random_operations_match_oracle(pkv):
    rnd = random.Random(1234)
    for trial in range(5):
        nb = rnd.choice([8, 32, 200])
        order = list(range(nb))
        rnd.shuffle(order)
        ref = allocator.KVCacheManager(nb, 16, order)
        pool = pkv.pkv_pool_create(nb, 16, order)
        live = []
        for _ in range(400):
            r = rnd.random()
            if r < 0.2 or not live:
                assert pkv.pkv_seq_create(pool) == ref.create()
                live.append(ref._next_id - 1)
            elif r < 0.35:
                parent = rnd.choice(live)
                assert pkv.pkv_seq_fork(pool, parent) == ref.fork(parent)
                live.append(ref._next_id - 1)
            elif r < 0.85:
                s, n = rnd.choice(live), rnd.randint(0, 40)
                try:
                    want = ref.append(s, n)
                except allocator.OutOfBlocks:
                    with pytest.raises(pkv.PkvError) as e:
                        pkv.pkv_seq_append(pool, s, n)
                    assert e.value.name == "PKV_ERR_OUT_OF_BLOCKS"
                else:
                    slots, pairs = pkv.pkv_seq_append(pool, s, n)
                    assert list(slots) == want[0] and pairs == want[1]
            else:
                s = live.pop(rnd.randrange(len(live)))
                pkv.pkv_seq_free(pool, s)
                ref.free(s)
            assert pkv.pkv_pool_num_free(pool) == ref.pool.num_free()
        for s in live:
            assert list(pkv.pkv_seq_block_table(pool, s)) == ref.table(s)
            assert pkv.pkv_seq_len(pool, s) == ref.length(s)
            pkv.pkv_seq_free(pool, s)
        assert pkv.pkv_pool_num_free(pool) == nb
        pkv.pkv_pool_destroy(pool)


def test_error_paths(pkv):
    E = pkv.PkvError
    with pytest.raises(E) as e:
        pkv.pkv_pool_create(4, 16, [0, 1, 1, 2])
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    pool = pkv.pkv_pool_create(4, 16)
    with pytest.raises(E) as e:
        pkv.pkv_seq_free(pool, 99)
    assert e.value.name == "PKV_ERR_BAD_SEQ"
    b = pkv.pkv_block_alloc(pool)
    pkv.pkv_block_decref(pool, b)
    with pytest.raises(E) as e:
        pkv.pkv_block_decref(pool, b)
    assert e.value.name == "PKV_ERR_DOUBLE_FREE"
    with pytest.raises(E) as e:
        pkv.pkv_block_incref(pool, b)
    assert e.value.name == "PKV_ERR_DOUBLE_FREE"
    s = pkv.pkv_seq_create(pool)
    pkv.pkv_seq_append(pool, s, 40)  # 3 blocks
    before = (list(pkv.pkv_seq_block_table(pool, s)), pkv.pkv_seq_len(pool, s), pkv.pkv_pool_num_free(pool))
    with pytest.raises(E) as e:
        pkv.pkv_seq_append(pool, s, 30)
    assert e.value.name == "PKV_ERR_OUT_OF_BLOCKS"
    assert (list(pkv.pkv_seq_block_table(pool, s)), pkv.pkv_seq_len(pool, s), pkv.pkv_pool_num_free(pool)) == before
    with pytest.raises(E) as e:
        pkv.pkv_build_block_tables(pool, [s], 2)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(E) as e:
        pkv.pkv_seq_append_batch(pool, [s, s], 1)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    pkv.pkv_pool_destroy(pool)


def test_fault_injection_keeps_appends_atomic(pkv):
    pool = pkv.pkv_pool_create(64, 16)
    s = pkv.pkv_seq_create(pool)
    pkv.pkv_seq_append(pool, s, 16)
    pkv.pkv_debug_fail_after(pool, 1)
    snap = (list(pkv.pkv_seq_block_table(pool, s)), pkv.pkv_seq_len(pool, s), pkv.pkv_pool_num_free(pool))
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_seq_append(pool, s, 17)  # needs 2 blocks, 1 allowed
    assert e.value.name == "PKV_ERR_OUT_OF_BLOCKS"
    assert (list(pkv.pkv_seq_block_table(pool, s)), pkv.pkv_seq_len(pool, s), pkv.pkv_pool_num_free(pool)) == snap
    pkv.pkv_seq_append(pool, s, 16)  # 1 block: allowed
    with pytest.raises(pkv.PkvError):
        pkv.pkv_block_alloc(pool)
    pkv.pkv_debug_fail_after(pool, -1)
    pkv.pkv_block_alloc(pool)
    # a batch step fails as a whole
    t = pkv.pkv_seq_create(pool)
    pkv.pkv_debug_fail_after(pool, 1)
    n_free = pkv.pkv_pool_num_free(pool)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_seq_append_batch(pool, [s, t], 1)  # both need a new block
    assert pkv.pkv_pool_num_free(pool) == n_free and pkv.pkv_seq_len(pool, t) == 0
    pkv.pkv_pool_destroy(pool)


def test_worked_allocation_through_c_abi(pkv):
    pool = pkv.pkv_pool_create(64, 16)
    seqs = []
    for L in (25, 47, 12):
        s = pkv.pkv_seq_create(pool)
        pkv.pkv_seq_append(pool, s, L)
        seqs.append(s)
    tables, lens = pkv.pkv_build_block_tables(pool, seqs, 3)
    assert (tables >= 0).sum() * 16 == 96
    assert list(lens) == [25, 47, 12]
    pkv.pkv_pool_destroy(pool)
