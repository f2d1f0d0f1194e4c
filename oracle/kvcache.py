"""KV-append scatter, quantised append with sinks, copy-on-write block copy,
and attention over a quantised cache (test infrastructure).

* Append: each decode step writes one new K/V vector per sequence into the
  cache ("The 8GB VRAM Breakthrough", §1: the GPU must "write one new KV
  vector back" per generated token); with paging the write goes to the slot
  ``block * block_size + offset`` the block table reserved (§3).
* Quantised append: the body of the context is stored as INT4 or FP8 codes,
  the first ``n_sink`` tokens (attention sinks) stay in 16-bit (§4 "The Hybrid
  Solution: Sink-FP16 + Group-Wise Asymmetric INT4 / FP8"; §5 flowchart
  "Token Position Router").  Reading used: codes are written for every token
  (sink slots included) and the sink tokens are *also* copied into a
  per-sequence 16-bit buffer ``sink[seq, pos, head, :]``; attention reads the
  sink buffer for positions < n_sink and the codes elsewhere.
* Local window: the most recent tokens also stay in 16-bit ("The 8GB VRAM
  Breakthrough", §5 flowchart: the "Token Position Router" sends "Sink
  (0..7) or Local Window (Last 128)" to the high-precision FP16 pool, the
  middle context body to the quantiser).  Reading used: every token is
  quantised as above *and* copied to a per-sequence 16-bit ring of
  ``window / block_size + 1`` blocks (token p in ring block
  ``(p // bs) % R``, offset ``p % bs``); attention reads 16-bit values for
  the whole blocks from ``window_start`` on -- the last ``window`` tokens
  rounded down to a block boundary, so between window and window + bs - 1
  tokens -- and codes before that.
* Copy-on-write: cloning a shared block copies the whole physical block
  ("A Ideia de 60 Anos...", section "o bônus que paga o ingresso:
  compartilhar": copy only the affected block, then write).

Pool layouts (per layer): values ``[num_blocks, Hkv, block_size, D]``;
INT4 codes ``[num_blocks, Hkv, block_size, D/2]`` with fp16 scale and zero
``[num_blocks, Hkv, block_size, D/group]``; FP8 codes
``[num_blocks, Hkv, block_size, D]`` with fp16 scale
``[num_blocks, Hkv, block_size, 1]`` -- the packed layout of §7's Triton
pattern.
"""

import numpy as np

from . import quant
from .attention import attention_reference


def kv_append(k, v, slot_mapping, k_pool, v_pool, block_size=16):
    """pool[slot // bs, :, slot % bs, :] = new row; negative slots skipped."""
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = divmod(slot, block_size)
        k_pool[blk, :, off, :] = k[t]
        v_pool[blk, :, off, :] = v[t]


def quantize_token(x_heads, qmode, group_size):
    """Quantise one token's rows [Hkv, D] -> (codes, scale, zero or None)."""
    Hkv, D = x_heads.shape
    if qmode == "int4":
        codes, s, z = [], [], []
        for h in range(Hkv):
            cs, ss, zs = [], [], []
            for g0 in range(0, D, group_size):
                c, s16, z16 = quant.int4_quantize_group(x_heads[h, g0:g0 + group_size])
                cs.append(c)
                ss.append(s16)
                zs.append(z16)
            codes.append(quant.pack_nibbles(np.concatenate(cs)))
            s.append(ss)
            z.append(zs)
        return (np.array(codes, dtype=np.uint8), np.array(s, dtype=np.float16),
                np.array(z, dtype=np.float16))
    if qmode == "fp8":
        codes, s = [], []
        for h in range(Hkv):
            c, s16 = quant.fp8_quantize_row(x_heads[h])
            codes.append(c)
            s.append([s16])
        return np.array(codes, dtype=np.uint8), np.array(s, dtype=np.float16), None
    raise ValueError(qmode)


def window_start(ctx, window, block_size=16):
    """First position read from the 16-bit window: the last ``window``
    tokens rounded down to a block boundary (ctx when there is no window)."""
    if window <= 0:
        return ctx
    return max(0, ctx - window) // block_size * block_size


def ring_blocks(window, block_size=16):
    """Blocks in a sequence's 16-bit window ring."""
    return window // block_size + 1


def kv_append_quant(k, v, slot_mapping, positions, seq_idx, cache, n_sink, qmode,
                    group_size, block_size=16, window=0):
    """Quantised scatter of new tokens plus the 16-bit sink copies.

    k, v: [T, Hkv, D] values exact in binary32; cache: dict with
    ``k_codes, k_scale, k_zero, v_codes, v_scale, v_zero, sink_k, sink_v``
    (zero arrays absent for FP8); sink_*: [B, n_sink, Hkv, D].
    """
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = divmod(slot, block_size)
        for name, x in (("k", k[t]), ("v", v[t])):
            codes, s, z = quantize_token(np.asarray(x, dtype=np.float32), qmode, group_size)
            cache[name + "_codes"][blk, :, off, :] = codes
            cache[name + "_scale"][blk, :, off, :] = s
            if z is not None:
                cache[name + "_zero"][blk, :, off, :] = z
        pos = int(positions[t])
        if pos < n_sink:
            cache["sink_k"][int(seq_idx[t]), pos] = k[t]
            cache["sink_v"][int(seq_idx[t]), pos] = v[t]
        if window > 0:
            rb = (pos // block_size) % ring_blocks(window, block_size)
            cache["win_k"][int(seq_idx[t]), rb, :, pos % block_size] = k[t]
            cache["win_v"][int(seq_idx[t]), rb, :, pos % block_size] = v[t]


def dequantize_cache_row(cache, name, blk, head, off, qmode, group_size):
    codes = cache[name + "_codes"][blk, head, off]
    s = cache[name + "_scale"][blk, head, off]
    if qmode == "int4":
        full = quant.unpack_nibbles(codes)
        z = cache[name + "_zero"][blk, head, off]
        out = np.empty(full.shape[0], dtype=np.float64)
        for gi in range(full.shape[0] // group_size):
            sl = slice(gi * group_size, (gi + 1) * group_size)
            out[sl] = quant.int4_dequantize(full[sl], s[gi], z[gi])
        return out
    return quant.E4M3_VALUES[codes.astype(np.int64)] * float(s[0])


def paged_attention_decode_quant(q, cache, block_tables, context_lens, scale, n_sink, qmode,
                                 group_size, block_size=16, window=0):
    """Attention over the dequantised cache, sink and window positions read
    in 16-bit (window ring ``win_k/win_v [B, R, Hkv, block_size, D]``)."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = cache["k_codes"].shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        ctx = int(context_lens[b])
        ws = window_start(ctx, window, block_size)
        for g in range(Hkv):
            K = np.zeros((ctx, D))
            V = np.zeros((ctx, D))
            for t in range(ctx):
                if t >= ws:
                    rb = (t // block_size) % ring_blocks(window, block_size)
                    K[t] = cache["win_k"][b, rb, g, t % block_size]
                    V[t] = cache["win_v"][b, rb, g, t % block_size]
                    continue
                if t < n_sink:
                    K[t] = cache["sink_k"][b, t, g]
                    V[t] = cache["sink_v"][b, t, g]
                    continue
                blk = block_tables[b][t // block_size]
                off = t % block_size
                K[t] = dequantize_cache_row(cache, "k", blk, g, off, qmode, group_size)
                V[t] = dequantize_cache_row(cache, "v", blk, g, off, qmode, group_size)
            for h in range(g * G, (g + 1) * G):
                out[b, h] = attention_reference(q[b, h], K, V, scale)
    return out


def quantize_sequence(x_seq, qmode, group_size):
    """Vectorised quantisation of one sequence's rows [ctx, Hkv, D].

    Returns the dequantised float64 values and the raw codes/scales/zeros
    ([ctx, Hkv, ...]) for bit-exact comparison with a device cache.
    """
    ctx, Hkv, D = x_seq.shape
    X = np.asarray(x_seq, dtype=np.float32).reshape(ctx * Hkv, D)
    if qmode == "int4":
        codes, s, z = quant.int4_quantize_rows(X, group_size)
        deq = quant.int4_dequantize_rows(codes, s, z, group_size)
        return (deq.reshape(ctx, Hkv, D), quant.pack_nibbles(codes).reshape(ctx, Hkv, D // 2),
                s.reshape(ctx, Hkv, -1), z.reshape(ctx, Hkv, -1))
    if qmode == "fp8":
        codes, s = quant.fp8_quantize_rows(X)
        deq = quant.fp8_dequantize_rows(codes, s)
        return deq.reshape(ctx, Hkv, D), codes.reshape(ctx, Hkv, D), s.reshape(ctx, Hkv, 1), None
    raise ValueError(qmode)


def sequence_attention_quant(q_seq, k_seq, v_seq, scale, n_sink, qmode, group_size, window=0):
    """Decode attention of one sequence over its quantised cache.

    The cache holds the oracle's own quantisation of the logical rows; the
    first n_sink positions and the positions from window_start on use the
    16-bit originals.  q_seq: [Hq, D]; k_seq, v_seq: [ctx, Hkv, D].
    """
    k_deq = quantize_sequence(k_seq, qmode, group_size)[0]
    v_deq = quantize_sequence(v_seq, qmode, group_size)[0]
    ns = min(n_sink, k_seq.shape[0])
    k_deq[:ns] = np.asarray(k_seq[:ns], dtype=np.float64)
    v_deq[:ns] = np.asarray(v_seq[:ns], dtype=np.float64)
    ws = window_start(k_seq.shape[0], window)
    k_deq[ws:] = np.asarray(k_seq[ws:], dtype=np.float64)
    v_deq[ws:] = np.asarray(v_seq[ws:], dtype=np.float64)
    q_seq = np.asarray(q_seq, dtype=np.float64)
    Hq, D = q_seq.shape
    Hkv = k_seq.shape[1]
    G = Hq // Hkv
    out = np.zeros((Hq, D))
    for h in range(Hq):
        out[h] = attention_reference(q_seq[h], k_deq[:, h // G], v_deq[:, h // G], scale)
    return out


def copy_blocks(pools, pairs):
    """For each (src, dst): every pool's block dst becomes a copy of block src."""
    for src, dst in pairs:
        for p in pools:
            p[int(dst)] = p[int(src)]
