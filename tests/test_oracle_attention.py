"""Pins of the oracle's attention to library routines, closed forms and the
pages' invariance statement (paging changes layout, not results)."""

import numpy as np
import pytest
import torch

from oracle import allocator, attention


def _sdpa64(q, K, V, scale):
    """torch scaled_dot_product_attention in float64, one query row."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64))[None, None, None, :]
    kt = torch.from_numpy(np.asarray(K, dtype=np.float64))[None, None]
    vt = torch.from_numpy(np.asarray(V, dtype=np.float64))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[0, 0, 0].numpy()


@pytest.mark.parametrize("T,D", [(1, 4), (3, 8), (17, 16), (40, 64)])
def test_reference_matches_torch_sdpa(T, D):
    rng = np.random.default_rng(T * 100 + D)
    for _ in range(5):
        q = rng.standard_normal(D)
        K = rng.standard_normal((T, D)) * 2
        V = rng.standard_normal((T, D))
        scale = 1 / np.sqrt(D)
        np.testing.assert_allclose(attention.attention_reference(q, K, V, scale),
                                   _sdpa64(q, K, V, scale), rtol=1e-12, atol=1e-13)


def test_brute_force_softmax_tiny():
    # explicit exponentials without max subtraction, 3 tokens
    q = np.array([0.5, -1.0])
    K = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    V = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]])
    s = [0.5 * 0.7, -1.0 * 0.7, -0.5 * 0.7]
    e = [np.exp(x) for x in s]
    want = sum(ei * vi for ei, vi in zip(e, V)) / sum(e)
    np.testing.assert_allclose(attention.attention_reference(q, K, V, 0.7), want, rtol=1e-14)


def test_closed_forms():
    rng = np.random.default_rng(0)
    D = 8
    V = rng.standard_normal((5, D))
    K = rng.standard_normal((5, D))
    # one token: the output is that token's value row
    np.testing.assert_array_equal(attention.attention_reference(rng.standard_normal(D), K[:1], V[:1], 0.3), V[0])
    # all logits equal (q = 0): the mean of V
    np.testing.assert_allclose(attention.attention_reference(np.zeros(D), K, V, 0.3), V.mean(0), rtol=1e-14)
    # one dominant logit: that row
    Kd = np.zeros((5, D))
    Kd[3, 0] = 1.0
    q = np.zeros(D)
    q[0] = 1e4
    np.testing.assert_allclose(attention.attention_reference(q, Kd, V, 1.0), V[3], rtol=0, atol=1e-300)
    # zero context gives zeros
    np.testing.assert_array_equal(attention.attention_reference(np.ones(D), K[:0], V[:0], 1.0), np.zeros(D))


def test_gqa_mapping_matches_torch_enable_gqa():
    rng = np.random.default_rng(1)
    Hq, Hkv, D, T = 8, 2, 16, 9
    q = rng.standard_normal((Hq, D))
    k = rng.standard_normal((T, Hkv, D))
    v = rng.standard_normal((T, Hkv, D))
    got = attention.sequence_attention(q, k, v, 0.25)
    qt = torch.from_numpy(q)[None, :, None, :]
    kt = torch.from_numpy(k.transpose(1, 0, 2).copy())[None]
    vt = torch.from_numpy(v.transpose(1, 0, 2).copy())[None]
    want = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.25, enable_gqa=True)
    np.testing.assert_allclose(got, want[0, :, 0].numpy(), rtol=1e-12, atol=1e-13)


def _build_paged(lens, Hkv, D, num_blocks, order, k_rows, v_rows, bs=16):
    m = allocator.KVCacheManager(num_blocks, bs, order)
    kp = np.zeros((num_blocks, Hkv, bs, D))
    vp = np.zeros((num_blocks, Hkv, bs, D))
    sids = []
    for i, L in enumerate(lens):
        s = m.create()
        slots, _ = m.append(s, L)
        for t, slot in enumerate(slots):
            kp[slot // bs, :, slot % bs] = k_rows[i][t]
            vp[slot // bs, :, slot % bs] = v_rows[i][t]
        sids.append(s)
    max_blocks = max(len(m.table(s)) for s in sids)
    tables, ctx = m.block_tables(sids, max_blocks)
    return kp, vp, tables, ctx


def test_paged_equals_slab_for_every_permutation():
    """100 seeded block-table permutations, bit-identical float64 results."""
    rng = np.random.default_rng(11)
    lens = [25, 47, 12]
    Hq, Hkv, D, NB = 8, 2, 64, 64
    q = rng.standard_normal((3, Hq, D))
    k_rows = [rng.standard_normal((L, Hkv, D)) for L in lens]
    v_rows = [rng.standard_normal((L, Hkv, D)) for L in lens]
    maxL = max(lens)
    k_slab = np.zeros((3, Hkv, maxL, D))
    v_slab = np.zeros((3, Hkv, maxL, D))
    for i, L in enumerate(lens):
        k_slab[i, :, :L] = k_rows[i].transpose(1, 0, 2)
        v_slab[i, :, :L] = v_rows[i].transpose(1, 0, 2)
    want = attention.slab_attention_decode(q, k_slab, v_slab, lens, 0.125)
    seen = set()
    for p in range(100):
        order = rng.permutation(NB)
        kp, vp, tables, ctx = _build_paged(lens, Hkv, D, NB, order, k_rows, v_rows)
        seen.add(tuple(tuple(t) for t in tables))
        got = attention.paged_attention_decode(q, kp, vp, tables, ctx, 0.125)
        np.testing.assert_array_equal(got, want)
    assert len(seen) == 100


def test_paged_with_shared_blocks_equals_slab():
    rng = np.random.default_rng(12)
    Hq, Hkv, D, NB, bs = 4, 1, 8, 32, 16
    m = allocator.KVCacheManager(NB, bs, rng.permutation(NB))
    kp = np.zeros((NB, Hkv, bs, D))
    vp = np.zeros((NB, Hkv, bs, D))
    p = m.create()
    prompt_k = rng.standard_normal((20, Hkv, D))
    prompt_v = rng.standard_normal((20, Hkv, D))
    for t, slot in enumerate(m.append(p, 20)[0]):
        kp[slot // bs, :, slot % bs] = prompt_k[t]
        vp[slot // bs, :, slot % bs] = prompt_v[t]
    kids = [m.fork(p) for _ in range(3)]
    rows_k, rows_v = [], []
    for c in kids:
        tk = rng.standard_normal((5, Hkv, D))
        tv = rng.standard_normal((5, Hkv, D))
        slots, copies = m.append(c, 5)
        for src, dst in copies:
            kp[dst] = kp[src]
            vp[dst] = vp[src]
        for t, slot in enumerate(slots):
            kp[slot // bs, :, slot % bs] = tk[t]
            vp[slot // bs, :, slot % bs] = tv[t]
        rows_k.append(np.concatenate([prompt_k, tk]))
        rows_v.append(np.concatenate([prompt_v, tv]))
    tables, ctx = m.block_tables(kids, 2)
    q = rng.standard_normal((3, Hq, D))
    got = attention.paged_attention_decode(q, kp, vp, tables, ctx, 0.3)
    for i in range(3):
        want = attention.sequence_attention(q[i], rows_k[i], rows_v[i], 0.3)
        np.testing.assert_array_equal(got[i], want)


def test_planted_mistakes_are_caught():
    """A transposed gather or a wrong head mapping breaks the pins above."""
    rng = np.random.default_rng(5)
    Hq, Hkv, D = 4, 2, 8
    q = rng.standard_normal((Hq, D))
    k = rng.standard_normal((6, Hkv, D))
    v = rng.standard_normal((6, Hkv, D))
    good = attention.sequence_attention(q, k, v, 0.5)
    # head h -> h % Hkv instead of h // G
    bad = np.stack([attention.attention_reference(q[h], k[:, h % Hkv], v[:, h % Hkv], 0.5) for h in range(Hq)])
    assert not np.allclose(good, bad)
    # softmax over the wrong axis / missing scale
    bad2 = np.stack([attention.attention_reference(q[h], k[:, h // 2], v[:, h // 2], 1.0) for h in range(Hq)])
    assert not np.allclose(good, bad2)
