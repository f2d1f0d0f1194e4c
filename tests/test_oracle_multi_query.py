"""Pins of the oracle's multi-query (causal) attention: torch's causal SDPA
for a whole prefill, the decode oracle for one query, invariance to tokens
past each query's position, and paging invariance."""

import numpy as np
import pytest
import torch

from oracle import allocator, attention


def _causal_sdpa64(q, k, v, scale):
    """torch scaled_dot_product_attention, float64, queries = the last L of
    T keys (bottom-right aligned causal mask), GQA by enable_gqa."""
    L, Hq, D = q.shape
    T = k.shape[0]
    mask = torch.ones(L, T, dtype=torch.bool).tril(diagonal=T - L)
    qt = torch.from_numpy(q.transpose(1, 0, 2).copy())[None]
    kt = torch.from_numpy(k.transpose(1, 0, 2).copy())[None]
    vt = torch.from_numpy(v.transpose(1, 0, 2).copy())[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale,
                                                         enable_gqa=True)
    return o[0].numpy().transpose(1, 0, 2)


@pytest.mark.parametrize("L,T,Hq,Hkv", [(5, 5, 4, 1), (1, 9, 8, 2), (6, 40, 8, 2), (17, 17, 4, 4), (3, 70, 6, 3)])
def test_matches_torch_causal_sdpa(L, T, Hq, Hkv):
    rng = np.random.default_rng(L * 1000 + T)
    D = 16
    q = rng.standard_normal((L, Hq, D))
    k = rng.standard_normal((T, Hkv, D)) * 2
    v = rng.standard_normal((T, Hkv, D))
    got = attention.multi_query_attention(q, k, v, 0.3)
    np.testing.assert_allclose(got, _causal_sdpa64(q, k, v, 0.3), rtol=1e-12, atol=1e-13)


def test_one_query_is_decode():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 8, 32))
    k = rng.standard_normal((50, 2, 32))
    v = rng.standard_normal((50, 2, 32))
    np.testing.assert_array_equal(attention.multi_query_attention(q, k, v, 0.2)[0],
                                  attention.sequence_attention(q[0], k, v, 0.2))


def test_future_tokens_do_not_matter():
    """Changing K/V after a query's position leaves that query's output
    unchanged (the causal mask); the first query of a full prefill sees only
    token 0, so its output is V_0."""
    rng = np.random.default_rng(8)
    L, T, D = 6, 20, 8
    q = rng.standard_normal((L, 4, D))
    k = rng.standard_normal((T, 2, D))
    v = rng.standard_normal((T, 2, D))
    base = attention.multi_query_attention(q, k, v, 0.5)
    for i in range(L):
        p = T - L + i
        k2, v2 = k.copy(), v.copy()
        k2[p + 1:] = rng.standard_normal(k2[p + 1:].shape) * 5
        v2[p + 1:] = rng.standard_normal(v2[p + 1:].shape) * 5
        np.testing.assert_array_equal(attention.multi_query_attention(q, k2, v2, 0.5)[i], base[i])
    full = attention.multi_query_attention(q[:1], k[:1], v[:1], 0.5)
    np.testing.assert_array_equal(full[0, 0], v[0, 0])
    # more queries than tokens: the queries at negative positions get zeros
    short = attention.multi_query_attention(q, k[:3], v[:3], 0.5)
    np.testing.assert_array_equal(short[:3], np.zeros((3, 4, D)))
    np.testing.assert_array_equal(short[3], attention.multi_query_attention(q[3:4], k[:1], v[:1], 0.5)[0])


def test_paged_equals_contiguous():
    rng = np.random.default_rng(9)
    Hq, Hkv, D, bs = 8, 2, 16, 16
    lens, qlens = [40, 17, 5, 64], [6, 1, 5, 16]
    ks = [rng.standard_normal((L, Hkv, D)) for L in lens]
    vs = [rng.standard_normal((L, Hkv, D)) for L in lens]
    m = allocator.KVCacheManager(32, bs, rng.permutation(32))
    kp, vp = np.zeros((32, Hkv, bs, D)), np.zeros((32, Hkv, bs, D))
    sids = []
    for i, L in enumerate(lens):
        s = m.create()
        for t, slot in enumerate(m.append(s, L)[0]):
            kp[slot // bs, :, slot % bs] = ks[i][t]
            vp[slot // bs, :, slot % bs] = vs[i][t]
        sids.append(s)
    tables, ctx = m.block_tables(sids, 4)
    q_start = np.concatenate([[0], np.cumsum(qlens)])
    q = rng.standard_normal((q_start[-1], Hq, D))
    got = attention.paged_multi_query_attention(q, q_start, kp, vp, tables, ctx, 0.25)
    for b in range(len(lens)):
        want = attention.multi_query_attention(q[q_start[b]:q_start[b + 1]], ks[b], vs[b], 0.25)
        np.testing.assert_array_equal(got[q_start[b]:q_start[b + 1]], want)


def test_planted_mask_mistake_is_caught():
    """A mask shifted by one (each query also seeing the next token) fails
    the torch comparison."""
    rng = np.random.default_rng(10)
    L, T, D = 4, 12, 8
    q = rng.standard_normal((L, 2, D))
    k = rng.standard_normal((T, 1, D))
    v = rng.standard_normal((T, 1, D))
    wrong = np.stack([np.stack([attention.attention_reference(q[i, h], k[:T - L + i + 2, 0], v[:T - L + i + 2, 0], 0.4)
                                if T - L + i + 2 <= T else attention.attention_reference(q[i, h], k[:, 0], v[:, 0], 0.4)
                                for h in range(2)]) for i in range(L)])
    assert not np.allclose(wrong, _causal_sdpa64(q, k, v, 0.4), rtol=1e-6, atol=1e-8)
