"""Single-query (decode) attention, contiguous and paged (test infrastructure).

What is computed is ordinary scaled-dot-product attention for one new query
per sequence.  Paging "changes only the layout and retrieval of the KV cache,
not the computation or its results" ("PagedAttention aplica memória virtual
ao cache KV de LLMs", section "Compartilhamento e compromissos"), so the
oracle is the plain definition applied to the tokens the block table gathers
("The 8GB VRAM Breakthrough", §3 "How Logical-to-Physical Block Tables
Work": the kernel walks the table and gathers the scattered physical blocks
for the QK^T product and the softmax-weighted sum of V).

Grouped-query attention: query head h reads KV head floor(h / G) with
G = Hq / Hkv (the pages give the 32-query / 8-KV-head layout of an 8B model,
§2, but not the mapping; contiguous groups are the common convention).

All arithmetic is float64.  Nothing is blocked, fused or reordered beyond
the definition.
"""

import numpy as np


def attention_reference(q, K, V, scale):
    """out = sum_t softmax_t(scale * <q, K_t>) V_t, in float64.

    q: [D]; K, V: [T, D].  T == 0 gives zeros (no token to attend to).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(q.shape[0], dtype=np.float64)
    s = float(scale) * (K @ q)
    s = s - s.max()
    p = np.exp(s)
    p = p / p.sum()
    return p @ V


def gather_tokens(pool, table, ctx, kv_head, block_size):
    """Rows of one KV head for logical tokens 0..ctx-1, through the table.

    pool: [num_blocks, Hkv, block_size, D]; token t lives in physical block
    table[t // block_size] at offset t % block_size.
    """
    rows = []
    for t in range(ctx):
        rows.append(pool[table[t // block_size], kv_head, t % block_size])
    if not rows:
        return np.zeros((0, pool.shape[-1]), dtype=np.float64)
    return np.stack(rows).astype(np.float64)


def paged_attention_decode(q, k_pool, v_pool, block_tables, context_lens, scale, block_size=16):
    """Decode attention through block tables.

    q: [B, Hq, D]; k_pool, v_pool: [num_blocks, Hkv, block_size, D];
    block_tables: [B, max_blocks] (entries past the context unused);
    context_lens: [B] tokens per sequence (including the one just appended).
    Returns float64 [B, Hq, D].
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        ctx = int(context_lens[b])
        for g in range(Hkv):
            K = gather_tokens(k_pool, block_tables[b], ctx, g, block_size)
            V = gather_tokens(v_pool, block_tables[b], ctx, g, block_size)
            for h in range(g * G, (g + 1) * G):
                out[b, h] = attention_reference(q[b, h], K, V, scale)
    return out


def slab_attention_decode(q, k_slab, v_slab, context_lens, scale):
    """The same attention over a contiguous per-sequence slab.

    k_slab, v_slab: [B, Hkv, max_len, D] -- the naive contiguous layout of
    "The 8GB VRAM Breakthrough", §3 (one tensor sized to max_seq_len).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_slab.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        ctx = int(context_lens[b])
        for h in range(Hq):
            g = h // G
            out[b, h] = attention_reference(q[b, h], k_slab[b, g, :ctx], v_slab[b, g, :ctx], scale)
    return out


def sequence_attention(q_seq, k_seq, v_seq, scale):
    """Decode attention for one sequence from its logical K/V rows.

    q_seq: [Hq, D]; k_seq, v_seq: [ctx, Hkv, D] in logical token order.
    Returns float64 [Hq, D].  Used for sampled checks at full size, where the
    per-sequence tokens are regenerated from their seed instead of being read
    back from any pool.
    """
    q_seq = np.asarray(q_seq, dtype=np.float64)
    Hq, D = q_seq.shape
    Hkv = k_seq.shape[1]
    G = Hq // Hkv
    out = np.zeros((Hq, D), dtype=np.float64)
    for h in range(Hq):
        g = h // G
        out[h] = attention_reference(q_seq[h], k_seq[:, g, :], v_seq[:, g, :], scale)
    return out


def multi_query_attention(q_rows, k_seq, v_seq, scale):
    """Causal attention of L new query tokens of one sequence.

    The L queries are the last L of the sequence's ctx tokens ("The 8GB VRAM
    Breakthrough", §6: the target model's one parallel pass over the
    gamma + 1 draft tokens; §5: a slice of a chunked prefill), so query i
    sits at position p = ctx - L + i and attends to tokens 0..p.
    q_rows: [L, Hq, D]; k_seq, v_seq: [ctx, Hkv, D] in logical order.
    Returns float64 [L, Hq, D]; a query at a negative position (ctx < L)
    gets zeros.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    L, Hq, D = q_rows.shape
    ctx, Hkv = k_seq.shape[0], k_seq.shape[1]
    G = Hq // Hkv
    out = np.zeros((L, Hq, D), dtype=np.float64)
    for i in range(L):
        p = ctx - L + i
        if p < 0:
            continue
        for h in range(Hq):
            g = h // G
            out[i, h] = attention_reference(q_rows[i, h], k_seq[:p + 1, g, :], v_seq[:p + 1, g, :], scale)
    return out


def paged_multi_query_attention(q, q_start, k_pool, v_pool, block_tables, context_lens, scale,
                                block_size=16):
    """Multi-query attention through block tables.

    q: [T, Hq, D] with sequence b's queries at rows q_start[b] .. q_start[b+1]-1;
    pools [num_blocks, Hkv, block_size, D]; context_lens include the new
    tokens.  Returns float64 [T, Hq, D].
    """
    q = np.asarray(q, dtype=np.float64)
    T, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    out = np.zeros((T, Hq, D), dtype=np.float64)
    for b in range(len(context_lens)):
        lo, hi = int(q_start[b]), int(q_start[b + 1])
        if hi == lo:
            continue
        ctx = int(context_lens[b])
        k = np.stack([gather_tokens(k_pool, block_tables[b], ctx, g, block_size) for g in range(Hkv)], axis=1) \
            if ctx else np.zeros((0, Hkv, D))
        v = np.stack([gather_tokens(v_pool, block_tables[b], ctx, g, block_size) for g in range(Hkv)], axis=1) \
            if ctx else np.zeros((0, Hkv, D))
        out[lo:hi] = multi_query_attention(q[lo:hi], k, v, scale)
    return out
