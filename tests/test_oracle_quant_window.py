"""Pins of the oracle's 16-bit local window over the quantised cache."""

import numpy as np
import pytest

from oracle import attention, kvcache


@pytest.mark.parametrize("ctx,start", [(1, 0), (100, 0), (128, 0), (129, 0), (143, 0), (144, 16),
                                       (145, 16), (160, 32), (1000, 864)])
def test_window_start_rounds_down_to_blocks(ctx, start):
    assert kvcache.window_start(ctx, 128) == start
    assert kvcache.window_start(ctx, 0) == ctx
    # between window and window + 15 tokens stay in 16-bit
    assert min(ctx, 128) <= ctx - start <= 128 + 15


def test_ring_holds_every_window_block():
    """The blocks from window_start on never share a ring block."""
    for ctx in range(1, 600):
        ws = kvcache.window_start(ctx, 128)
        blocks = range(ws // 16, (ctx + 15) // 16)
        assert len({b % kvcache.ring_blocks(128) for b in blocks}) == len(blocks)


@pytest.mark.parametrize("qmode", ["int4", "fp8"])
def test_full_window_is_exact_attention(qmode):
    """A window covering the whole context leaves nothing quantised: the
    result is the plain attention of the 16-bit rows."""
    rng = np.random.default_rng(1)
    ctx, Hq, Hkv, D = 90, 8, 2, 64
    q = rng.standard_normal((Hq, D))
    k = rng.standard_normal((ctx, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((ctx, Hkv, D)).astype(np.float32)
    got = kvcache.sequence_attention_quant(q, k, v, 0.2, 0, qmode, D, window=128)
    np.testing.assert_array_equal(got, attention.sequence_attention(q, k, v, 0.2))
    # without the window the quantised result differs
    assert not np.array_equal(kvcache.sequence_attention_quant(q, k, v, 0.2, 0, qmode, D), got)


def test_paged_window_reads_the_ring():
    """The paged form (codes + ring) equals the sequence form, and what it
    reads at window positions is the ring, not the codes."""
    rng = np.random.default_rng(2)
    ctx, Hkv, D, bs, W = 200, 2, 64, 16, 128
    k = rng.standard_normal((ctx, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((ctx, Hkv, D)).astype(np.float32)
    q = rng.standard_normal((1, 4, D))
    nb = ctx // bs + 1
    R = kvcache.ring_blocks(W)
    cache = {"k_codes": np.zeros((nb, Hkv, bs, D // 2), np.uint8), "v_codes": np.zeros((nb, Hkv, bs, D // 2), np.uint8),
             "k_scale": np.zeros((nb, Hkv, bs, 1), np.float16), "v_scale": np.zeros((nb, Hkv, bs, 1), np.float16),
             "k_zero": np.zeros((nb, Hkv, bs, 1), np.float16), "v_zero": np.zeros((nb, Hkv, bs, 1), np.float16),
             "sink_k": np.zeros((1, 4, Hkv, D)), "sink_v": np.zeros((1, 4, Hkv, D)),
             "win_k": np.zeros((1, R, Hkv, bs, D)), "win_v": np.zeros((1, R, Hkv, bs, D))}
    table = rng.permutation(nb)
    slots = [int(table[t // bs]) * bs + t % bs for t in range(ctx)]
    kvcache.kv_append_quant(k, v, slots, list(range(ctx)), [0] * ctx, cache, 4, "int4", D, window=W)
    got = kvcache.paged_attention_decode_quant(q, cache, [table], [ctx], 0.3, 4, "int4", D, window=W)
    want = kvcache.sequence_attention_quant(q[0], k, v, 0.3, 4, "int4", D, window=W)
    np.testing.assert_allclose(got[0], want, rtol=1e-12, atol=1e-13)
    # poisoning the codes of window positions changes nothing
    ws = kvcache.window_start(ctx, W)
    for t in range(ws, ctx):
        cache["k_codes"][table[t // bs], :, t % bs] = 0xFF
    np.testing.assert_array_equal(
        kvcache.paged_attention_decode_quant(q, cache, [table], [ctx], 0.3, 4, "int4", D, window=W), got)
