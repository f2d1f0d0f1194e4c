"""GPU quantised KV path: INT4 / FP8 codes bit-exact with the oracle's
binary32 quantiser, and decode attention over the quantised cache (sinks in
16-bit) within the acceptance bound of the oracle's attention over the
dequantised cache."""

import numpy as np
import pytest
import torch

import synthetic as syn
from cache_builder import assert_close, build, expected, expected_parallel, logical_rows
from oracle import kvcache as okv

pytestmark = pytest.mark.gpu


def _rand16(rng, shape, dtype, outliers=0.0):
    x = rng.standard_normal(shape).astype(np.float32)
    if outliers:
        hit = rng.random(shape) < outliers
        x = np.where(hit, np.where(rng.random(shape) < 0.5, -8.0, 8.0), x).astype(np.float32)
    return torch.from_numpy(x).to(dtype)


def _empty_cache(qmode, NB, Hkv, D, g, dev, B=1, n_sink=4, dtype=torch.bfloat16):
    cb = D // 2 if qmode == "int4" else D
    ng = D // g if qmode == "int4" else 1
    c = {
        "k_codes": torch.zeros((NB, Hkv, 16, cb), dtype=torch.uint8, device=dev),
        "v_codes": torch.zeros((NB, Hkv, 16, cb), dtype=torch.uint8, device=dev),
        "k_scale": torch.zeros((NB, Hkv, 16, ng), dtype=torch.float16, device=dev),
        "v_scale": torch.zeros((NB, Hkv, 16, ng), dtype=torch.float16, device=dev),
        "sink_k": torch.zeros((B, max(n_sink, 1), Hkv, D), dtype=dtype, device=dev),
        "sink_v": torch.zeros((B, max(n_sink, 1), Hkv, D), dtype=dtype, device=dev),
    }
    if qmode == "int4":
        c["k_zero"] = torch.zeros((NB, Hkv, 16, ng), dtype=torch.float16, device=dev)
        c["v_zero"] = torch.zeros((NB, Hkv, 16, ng), dtype=torch.float16, device=dev)
    return c


@pytest.mark.parametrize("qmode,D,g,dtype", [
    ("int4", 128, 128, torch.bfloat16), ("int4", 128, 64, torch.bfloat16), ("int4", 128, 32, torch.float16),
    ("int4", 64, 64, torch.float16), ("fp8", 128, 128, torch.bfloat16), ("fp8", 64, 64, torch.float16),
    ("int4", 256, 256, torch.bfloat16), ("fp8", 256, 256, torch.bfloat16)])
def test_append_quant_codes_bit_exact(pkv, cuda_dev, qmode, D, g, dtype):
    rng = np.random.default_rng(D + g)
    NB, Hkv, T, n_sink = 24, 4, 200, 4
    k = _rand16(rng, (T, Hkv, D), dtype, 0.01)
    v = _rand16(rng, (T, Hkv, D), dtype, 0.01) * 3
    # a few degenerate rows: constant, zero, huge spread
    k[0] = 1.5
    k[1] = 0.0
    k[2, :, 0] = 3e4 if dtype == torch.float16 else 3e30
    slots = rng.choice(NB * 16, size=T, replace=False).astype(np.int64)
    slots[-3:] = -1
    positions = np.arange(T, dtype=np.int32)
    seq_idx = np.zeros(T, dtype=np.int32)
    cache = _empty_cache(qmode, NB, Hkv, D, g, cuda_dev, 1, n_sink, dtype)
    pkv.pkv_kv_append_quant(k.to(cuda_dev), v.to(cuda_dev), torch.from_numpy(slots).to(cuda_dev),
                            torch.from_numpy(positions).to(cuda_dev), torch.from_numpy(seq_idx).to(cuda_dev),
                            cache, n_sink, qmode, g)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    got = {n: t.cpu().numpy() for n, t in cache.items() if not n.startswith("sink")}
    for name, x in (("k", k), ("v", v)):
        _, codes, s, z = okv.quantize_sequence(x.float().numpy(), qmode, g)
        for t in range(T):
            if slots[t] < 0:
                continue
            blk, off = divmod(int(slots[t]), 16)
            assert np.array_equal(got[name + "_codes"][blk, :, off], codes[t]), (name, t)
            assert got[name + "_scale"][blk, :, off].tobytes() == s[t].tobytes(), (name, t)
            if qmode == "int4":
                assert got[name + "_zero"][blk, :, off].tobytes() == z[t].tobytes(), (name, t)
    assert torch.equal(cache["sink_k"][0, :n_sink].cpu(), k[:n_sink])
    assert torch.equal(cache["sink_v"][0, :n_sink].cpu(), v[:n_sink])


def _decode_quant(pkv, c, partition_size=0):
    w = c.w
    B = len(c.decoded)
    out = torch.empty((B, w["hq"], w["d"]), dtype=w["torch_dtype"], device=c.q.device)
    n = pkv.pkv_decode_workspace_bytes(B, w["hq"], w["d"], c.max_blocks, 16, partition_size)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=c.q.device)
    pkv.pkv_paged_attention_decode_quant(c.q, c.cache, c.n_sink, c.tables, c.lens, w["scale"], out,
                                         c.quant, c.group_size, ws, partition_size,
                                         window=getattr(c, "window", 0))
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    return out.float().cpu().numpy()


@pytest.mark.parametrize("qmode", ["int4", "fp8"])
@pytest.mark.parametrize("ps", [0, 64, 4096])
def test_quant_decode_small(pkv, cuda_dev, qmode, ps):
    w = syn.workload("quant", batch=5, ctx=1000, num_blocks=1024)
    c = build(pkv, w, cuda_dev, quant=qmode)
    want = expected(c)
    got = _decode_quant(pkv, c, ps)
    assert_close(got, want, what="%s ps %d" % (qmode, ps))


@pytest.mark.parametrize("qmode", ["int4", "fp8"])
@pytest.mark.parametrize("ctx", [1, 3, 4, 5, 15, 16, 17, 33])
def test_quant_decode_short_contexts_and_sinks(pkv, cuda_dev, qmode, ctx):
    w = syn.workload("quant", batch=3, ctx=ctx, num_blocks=64)
    c = build(pkv, w, cuda_dev, quant=qmode)
    want = expected(c)
    for ps in (0, 16):
        got = _decode_quant(pkv, c, ps)
        assert_close(got, want, what="%s ctx %d" % (qmode, ctx))


@pytest.mark.parametrize("qmode", ["int4", "fp8"])
def test_quant_decode_fp16_head64(pkv, cuda_dev, qmode):
    w = syn.workload("quant", batch=4, ctx=300, num_blocks=256, hq=8, hkv=2, d=64, dtype="fp16",
                     group_size=64)
    c = build(pkv, w, cuda_dev, quant=qmode)
    assert_close(_decode_quant(pkv, c, 64), expected(c), what=qmode)


def _codes_match(c, i, qmode):
    """Every token's codes, scales (and zeros) of sequence i, K and V, equal
    the oracle quantiser's, read through the sequence's table."""
    k, v = logical_rows(c, i)
    table = c.tables_host[i]
    t = np.arange(k.shape[0])
    blk, off = table[t // 16], t % 16
    for name, x in (("k", k), ("v", v)):
        _, codes, s, z = okv.quantize_sequence(x, qmode, c.group_size)
        np.testing.assert_array_equal(c.cache[name + "_codes"].cpu().numpy()[blk, :, off], codes)
        assert c.cache[name + "_scale"].cpu().numpy()[blk, :, off].tobytes() == s.tobytes()
        if qmode == "int4":
            assert c.cache[name + "_zero"].cpu().numpy()[blk, :, off].tobytes() == z.tobytes()


@pytest.mark.parametrize("qmode", ["int4", "fp8"])
def test_quant_workload_full_size(pkv, cuda_dev, qmode):
    """32 sequences x 16,384 tokens, 4 sinks, 1% outliers at +-8: every
    sequence's output within the bound (balanced split), and every code,
    scale and zero of three sequences bit-exact."""
    w = syn.workload("quant")
    c = build(pkv, w, cuda_dev, quant=qmode)
    got = _decode_quant(pkv, c, 0)
    assert np.isfinite(got).all()
    assert_close(got, expected_parallel(c), what="quant %s" % qmode)
    for i in (0, 13, 31):
        _codes_match(c, i, qmode)


def test_quant_prefix_cow_int4(pkv, cuda_dev):
    """Copy-on-write of a quantised block copies codes, scales and zeros."""
    w = syn.workload("prefix_cow_2008", n_sink=4, group_size=128)
    c = build(pkv, w, cuda_dev, quant="int4")
    assert len(c.all_pairs) == 8
    assert_close(_decode_quant(pkv, c, 0), expected(c), what="prefix int4")


# The pages' own INT4 layout: groups of 64 along the head dim (two (scale,
# zero) pairs per token and head at D = 128) and 8 sink tokens.

@pytest.mark.parametrize("ps", [0, 64, 4096])
def test_int4_group64_decode(pkv, cuda_dev, ps):
    w = syn.workload("quant", batch=5, ctx=1000, num_blocks=1024, group_size=64, n_sink=8)
    c = build(pkv, w, cuda_dev, quant="int4")
    assert c.group_size == 64
    assert_close(_decode_quant(pkv, c, ps), expected(c), what="g64 ps %d" % ps)


@pytest.mark.parametrize("ctx", [1, 7, 8, 9, 16, 17, 33])
def test_int4_group64_short_contexts_and_8_sinks(pkv, cuda_dev, ctx):
    w = syn.workload("quant", batch=3, ctx=ctx, num_blocks=64, group_size=64, n_sink=8)
    c = build(pkv, w, cuda_dev, quant="int4")
    want = expected(c)
    for ps in (0, 16):
        assert_close(_decode_quant(pkv, c, ps), want, what="g64 ctx %d" % ctx)


def test_int4_group64_full_size(pkv, cuda_dev):
    """32 sequences x 16,384 tokens in the pages' layout (g = 64, 8 sinks):
    every output within the bound (balanced split), every code of one
    sequence bit-exact."""
    w = syn.workload("quant", group_size=64, n_sink=8)
    c = build(pkv, w, cuda_dev, quant="int4")
    got = _decode_quant(pkv, c, 0)
    assert_close(got, expected_parallel(c), what="g64 full size")
    _codes_match(c, 21, "int4")


def test_int4_group_size_checks(pkv, cuda_dev):
    """Decode supports g = head dim, and g = 64 at head dim 128."""
    w = syn.workload("quant", batch=2, ctx=40, num_blocks=64, group_size=32)
    c = build(pkv, w, cuda_dev, quant="int4")
    with pytest.raises(pkv.PkvError):
        _decode_quant(pkv, c, 0)


# The pages' full layout: INT4 groups of 64, 8 sinks, and the last 128
# tokens kept in 16-bit (a per-sequence window ring).

@pytest.mark.parametrize("ctx", [1, 100, 128, 129, 143, 144, 145, 161, 500])
@pytest.mark.parametrize("qmode", ["int4", "fp8"])
def test_window_boundaries(pkv, cuda_dev, qmode, ctx):
    w = syn.workload("quant", batch=3, ctx=ctx, num_blocks=256, group_size=64 if qmode == "int4" else 128,
                     n_sink=8, window=128)
    c = build(pkv, w, cuda_dev, quant=qmode)
    want = expected(c)
    for ps in (0, 16, 64):
        assert_close(_decode_quant(pkv, c, ps), want, what="%s window ctx %d ps %d" % (qmode, ctx, ps))


def test_window_ring_holds_the_last_tokens(pkv, cuda_dev):
    """Every token of every sequence passed through its ring: the ring's
    blocks from the window start on equal the 16-bit rows."""
    w = syn.workload("quant", batch=2, ctx=300, num_blocks=128, group_size=64, n_sink=8, window=128)
    c = build(pkv, w, cuda_dev, quant="int4")
    R = 128 // 16 + 1
    for i in range(2):
        k, v = logical_rows(c, i)
        L = k.shape[0]
        ws = max(L - 128, 0) // 16 * 16
        wk = c.cache["win_k"][i].float().cpu().numpy()
        for t in range(ws, L):
            np.testing.assert_array_equal(wk[(t // 16) % R, :, t % 16], k[t])


def test_pages_layout_full_size(pkv, cuda_dev):
    """32 x 16,384 tokens in the pages' BIE layout (INT4 g = 64, 8 sinks,
    128-token 16-bit window): every output within the bound."""
    w = syn.workload("quant", group_size=64, n_sink=8, window=128)
    c = build(pkv, w, cuda_dev, quant="int4")
    got = _decode_quant(pkv, c, 0)
    assert_close(got, expected_parallel(c), what="BIE layout full size")


@pytest.mark.parametrize("qmode,mag", [("int4", 4000.0), ("fp8", 60000.0)])
def test_large_value_scales_take_the_exact_max(pkv, cuda_dev, qmode, mag):
    """Outliers large enough that a token's V scale exceeds 128 (INT4: a
    range of +-4,000; FP8: an amax of 60,000): the blocks holding them take
    the exact softmax max (weights <= 1), so W = P s stays inside fp16."""
    w = syn.workload("quant", batch=4, ctx=700, num_blocks=256, outlier_frac=0.02, outlier_mag=mag)
    c = build(pkv, w, cuda_dev, quant=qmode)
    want = expected(c)
    got = _decode_quant(pkv, c)
    assert np.isfinite(got).all()
    assert_close(got, want, what="%s outliers +-%g" % (qmode, mag))
