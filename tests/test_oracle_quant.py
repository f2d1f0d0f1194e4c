"""Pins of the oracle's INT4 / FP8 quantisers."""

import numpy as np
import pytest
import torch

from oracle import kvcache, quant


# ------------------------------------------------------------------ FP8
def test_e4m3_table_matches_torch_for_all_256_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = quant.E4M3_VALUES
    nan = np.isnan(vals)
    assert (nan == np.isnan(ours)).all()
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    np.testing.assert_array_equal(ours[~nan], vals[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_encoder_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    finite = quant.E4M3_VALUES[~np.isnan(quant.E4M3_VALUES)]
    pos = np.unique(finite[finite >= 0])
    mids = (pos[:-1] + pos[1:]) / 2  # exact ties: must go to the even mantissa
    vals = np.concatenate([
        rng.standard_normal(3000) * 30,
        rng.uniform(-448, 448, 2000),
        rng.standard_normal(500) * 1e-3,
        mids, -mids, pos, -pos,
    ]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448]
    want = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got_vec = quant.e4m3_encode_array(vals)
    np.testing.assert_array_equal(got_vec, want)
    for v in vals[::23]:
        assert quant.e4m3_encode(v) == want[list(vals).index(v)]


def test_e4m3_saturation_and_signed_zero():
    assert quant.e4m3_encode(np.float32(448)) == 0x7E
    assert quant.e4m3_encode(np.float32(470)) == 0x7E
    assert quant.e4m3_encode(np.float32(1e9)) == 0x7E
    assert quant.e4m3_encode(np.float32(-1e9)) == 0xFE
    assert quant.e4m3_encode(np.float32(-0.0)) == 0x80
    assert quant.e4m3_encode(np.float32(-1e-6)) == 0x80
    v = np.array([470, -500, 1e30, -0.0, 2.0 ** -10, 3 * 2.0 ** -10, 3 * 2.0 ** -11], dtype=np.float32)
    np.testing.assert_array_equal(quant.e4m3_encode_array(v), [0x7E, 0xFE, 0x7E, 0x80, 0x00, 0x02, 0x01])


def test_fp8_row_scale_and_roundtrip():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(128) * 3).astype(np.float32)
    codes, s16 = quant.fp8_quantize_row(x)
    assert s16 == np.float16(np.float32(np.abs(x).max()) / np.float32(448))
    deq = quant.E4M3_VALUES[codes] * float(s16)
    # relative error of E4M3 (3 mantissa bits) is at most 2^-4 for normals
    big = np.abs(x) > 2 ** -6 * float(s16)
    assert np.all(np.abs(deq[big] - x[big]) <= 2.0 ** -4 * np.abs(x[big]) + 1e-12)
    # the largest magnitude lands on (or next to) 448 * s
    assert np.abs(quant.E4M3_VALUES[codes]).max() >= 416
    codes2, s2 = quant.fp8_quantize_rows(x[None, :])
    np.testing.assert_array_equal(codes2[0], codes)
    assert s2[0] == s16


def test_fp8_zero_row_uses_unit_scale():
    codes, s16 = quant.fp8_quantize_row(np.zeros(16, np.float32))
    assert s16 == 1 and (codes == 0).all()


# ------------------------------------------------------------------ INT4
def test_int4_hand_worked_group():
    x = np.array([-1.0, 0.0, 0.5, 2.0], dtype=np.float32)
    codes, s16, z16 = quant.int4_quantize_group(x)
    assert s16 == np.float16(0.2)  # (2 - (-1)) / 15
    assert z16 == np.float16(5.0)  # 1 / 0.19995 = 5.0012 -> fp16 5.0
    assert list(codes) == [0, 5, 8, 15]
    np.testing.assert_allclose(quant.int4_dequantize(codes, s16, z16),
                               [-5 * 0.199951171875, 0.0, 3 * 0.199951171875, 10 * 0.199951171875])


def test_int4_exact_grid_roundtrip():
    """Values already on a representable grid come back exactly, codes too."""
    rng = np.random.default_rng(3)
    for _ in range(200):
        s = float(2.0 ** rng.integers(-6, 3))
        z = float(rng.integers(0, 16))
        q = rng.integers(0, 16, size=32).astype(np.uint8)
        q[0], q[1] = 0, 15  # the range is exactly 15 steps
        x = ((q.astype(np.float64) - z) * s).astype(np.float32)
        codes, s16, z16 = quant.int4_quantize_group(x)
        assert float(s16) == s and float(z16) == z
        np.testing.assert_array_equal(codes, q)
        np.testing.assert_array_equal(quant.int4_dequantize(codes, s16, z16), x)


def test_int4_error_bound():
    rng = np.random.default_rng(4)
    for _ in range(300):
        x = (rng.standard_normal(64) * rng.uniform(0.01, 10)).astype(np.float32)
        codes, s16, z16 = quant.int4_quantize_group(x)
        deq = quant.int4_dequantize(codes, s16, z16)
        s = float(s16)
        # half a step, plus the fp16 rounding of s (15 steps) and of z
        slack = 0.5 * s + 15 * abs(s - (float(x.max()) - float(x.min())) / 15) + abs(float(z16)) * s * 2 ** -10 + 1e-6
        assert np.max(np.abs(deq - x)) <= slack
        assert codes.min() >= 0 and codes.max() <= 15


def test_int4_degenerate_and_saturating_groups():
    codes, s16, z16 = quant.int4_quantize_group(np.full(8, 3.0, np.float32))
    assert s16 == 1 and z16 == np.float16(-3.0) and (codes == 0).all()
    codes, s16, z16 = quant.int4_quantize_group(np.zeros(8, np.float32))
    assert s16 == 1 and (codes == 0).all()
    big = np.array([-3e38, 3e38], dtype=np.float32)
    codes, s16, z16 = quant.int4_quantize_group(big)
    assert s16 == np.float16(65504)
    assert np.isfinite(float(z16)) and abs(float(z16)) == 65504


def test_int4_rows_matches_scalar_definition():
    rng = np.random.default_rng(5)
    X = (rng.standard_normal((300, 128)) * 2).astype(np.float32)
    X[rng.random(X.shape) < 0.01] = 8.0
    X = torch.from_numpy(X).to(torch.bfloat16).float().numpy()
    for g in (128, 64, 32):
        codes, s, z = quant.int4_quantize_rows(X, g)
        for r in range(0, 300, 37):
            for gi in range(128 // g):
                c1, s1, z1 = quant.int4_quantize_group(X[r, gi * g:(gi + 1) * g])
                np.testing.assert_array_equal(codes[r, gi * g:(gi + 1) * g], c1)
                assert s[r, gi].tobytes() == s1.tobytes() and z[r, gi].tobytes() == z1.tobytes()


def test_nibble_packing_layout():
    # [.., head_dim // 2] bytes, element 2i low nibble, 2i+1 high nibble
    assert list(quant.pack_nibbles(np.array([1, 2, 15, 0], np.uint8))) == [0x21, 0x0F]
    rng = np.random.default_rng(6)
    c = rng.integers(0, 16, size=(5, 128)).astype(np.uint8)
    p = quant.pack_nibbles(c)
    assert p.shape == (5, 64)
    np.testing.assert_array_equal(quant.unpack_nibbles(p), c)


def test_fp16_rounding_agrees_with_torch():
    rng = np.random.default_rng(8)
    v = (rng.standard_normal(20000) * 10.0 ** rng.uniform(-8, 4, 20000)).astype(np.float32)
    ours = np.array([quant.fp16_sat(x) for x in v[:2000]], dtype=np.float16)
    want = torch.from_numpy(v[:2000]).to(torch.float16).numpy()
    np.testing.assert_array_equal(ours.view(np.uint16), want.view(np.uint16))


# --------------------------------------------------- quantised attention
def test_quant_append_and_attention_small():
    """Cache-level oracle (paged, slot writes) == sequence-level oracle."""
    rng = np.random.default_rng(9)
    Hq, Hkv, D, bs, NB, n_sink = 4, 2, 16, 16, 8, 4
    ctx = 37
    k = torch.from_numpy(rng.standard_normal((ctx, Hkv, D)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    v = torch.from_numpy(rng.standard_normal((ctx, Hkv, D)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    q = rng.standard_normal((1, Hq, D))
    table = [5, 2, 7]
    slots = [table[t // bs] * bs + t % bs for t in range(ctx)]
    for qmode in ("int4", "fp8"):
        cb = D // 2 if qmode == "int4" else D
        cache = {
            "k_codes": np.zeros((NB, Hkv, bs, cb), np.uint8), "v_codes": np.zeros((NB, Hkv, bs, cb), np.uint8),
            "k_scale": np.zeros((NB, Hkv, bs, 1), np.float16), "v_scale": np.zeros((NB, Hkv, bs, 1), np.float16),
            "k_zero": np.zeros((NB, Hkv, bs, 1), np.float16), "v_zero": np.zeros((NB, Hkv, bs, 1), np.float16),
            "sink_k": np.zeros((1, n_sink, Hkv, D)), "sink_v": np.zeros((1, n_sink, Hkv, D)),
        }
        kvcache.kv_append_quant(k, v, slots, list(range(ctx)), [0] * ctx, cache, n_sink, qmode, D)
        got = kvcache.paged_attention_decode_quant(q, cache, [table], [ctx], 0.25, n_sink, qmode, D)
        want = kvcache.sequence_attention_quant(q[0], k, v, 0.25, n_sink, qmode, D)
        np.testing.assert_allclose(got[0], want, rtol=1e-12, atol=1e-12)
        # sinks are the originals; the body differs from the unquantised attention only slightly
        np.testing.assert_array_equal(cache["sink_k"][0], k[:n_sink])
        from oracle.attention import sequence_attention
        exact = sequence_attention(q[0], k, v, 0.25)
        assert np.max(np.abs(got[0] - exact)) < 0.25
        # codes at slot positions equal the vectorised sequence quantiser's
        _, kc, ks, kz = kvcache.quantize_sequence(k, qmode, D)
        for t in (0, 5, 36):
            np.testing.assert_array_equal(cache["k_codes"][slots[t] // bs, :, slots[t] % bs], kc[t])
            assert cache["k_scale"][slots[t] // bs, :, slots[t] % bs].tobytes() == ks[t].tobytes()
