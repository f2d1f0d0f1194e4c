"""KV-cache quantisers (test infrastructure; see ``oracle/__init__``).

Asymmetric INT4 -- "The 8GB VRAM Breakthrough", §4 "Sink-Preserving
Group-Wise INT4 Mode": codes q in [0, 15], an fp16 scale s and an fp16 zero
point z per group, dequantised as x = (q - z) * s.  The page fixes the code
range, the storage precision of s and z and the dequantisation; it does not
say how s, z and q are chosen.  Reading used here (the plainest one that fits
the stored types), every step an IEEE binary32 operation, in this order:

1. mn, mx = min and max of the group (exact in binary32 for 16-bit inputs);
2. s = fp16(binary32(mx - mn) / 15); if mx == mn or s == 0 then s = 1;
3. z = fp16(binary32(-mn) / s)            (a floating zero point, stored fp16;
   a zero point of -0 is stored as +0, since min(-0, +0) may be either);
4. q = clamp(rint_half_even(binary32(binary32(x / s) + z)), 0, 15);
   fp16() rounds to nearest even and saturates to +-65504.

Two codes share a byte: element 2i in the low nibble, 2i+1 in the high one.
The Triton pattern of §7 ("Register-Level INT4 Dequantization") unpacks a low
and a high nibble per byte but does not say which element is which; this
pairing is our reading.

FP8 E4M3 -- §4 "FP8 (E4M3) Mode": values are cast to OCP float8_e4m3fn
(sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, 0x7F and
0xFF are NaN, largest finite 448) after division by a dynamic scale.  The
page attaches one scale per head; here it is per (token, head):
a = max |x| (binary32); s = fp16(a / 448), s = 1 if it is 0;
code = nearest E4M3 value of binary32(x / s), ties to even mantissa,
magnitudes above 448 saturate to 448; dequantised as e4m3(code) * s.

The scalar encoders below are the definitions; the ``*_rows`` versions apply
the same binary32 operations element-wise with NumPy (float32 NumPy array
arithmetic is IEEE round-to-nearest per element) for full-size sampled
checks, and tests assert the two agree.
"""

from fractions import Fraction

import numpy as np

F16_MAX = 65504.0
E4M3_MAX = 448.0


# ---------------------------------------------------------------- helpers
def fp16_sat(x32):
    """Round a binary32 value to fp16 (nearest even), saturating to +-65504."""
    with np.errstate(over="ignore"):
        h = np.float16(np.float32(x32))
    if np.isinf(h):
        h = np.float16(np.copysign(F16_MAX, float(x32)))
    return h


def _fp16_sat_array(x32):
    with np.errstate(over="ignore"):
        h = np.asarray(x32, dtype=np.float32).astype(np.float16)
    inf = np.isinf(h)
    if inf.any():
        h[inf] = np.copysign(np.float16(F16_MAX), h[inf])
    return h


# ------------------------------------------------------------------- INT4
def int4_quantize_group(x):
    """Quantise one group (1-D values exact in binary32). Returns (codes, s16, z16)."""
    x = np.asarray(x, dtype=np.float32)
    mn = np.float32(x.min())
    mx = np.float32(x.max())
    with np.errstate(over="ignore"):
        s16 = fp16_sat(np.float32(mx - mn) / np.float32(15.0))
    if mx == mn or s16 == 0:
        s16 = np.float16(1.0)
    z16 = fp16_sat(np.float32(-mn) / np.float32(s16))
    if z16 == 0:
        z16 = np.float16(0.0)
    codes = np.empty(x.shape[0], dtype=np.uint8)
    s32 = np.float32(s16)
    z32 = np.float32(z16)
    for i, xi in enumerate(x):
        v = np.float32(np.float32(xi) / s32)
        v = np.float32(v + z32)
        r = np.rint(v)
        codes[i] = int(min(max(r, 0.0), 15.0))
    return codes, s16, z16


def int4_dequantize(codes, s16, z16):
    """x = (q - z) * s, exact in float64."""
    return (np.asarray(codes, dtype=np.float64) - float(z16)) * float(s16)


def int4_quantize_rows(X, group_size):
    """Element-wise binary32 version of ``int4_quantize_group`` over rows.

    X: [N, D] values exact in binary32.  Returns (codes uint8 [N, D],
    s16 [N, D/g], z16 [N, D/g]).
    """
    X = np.asarray(X, dtype=np.float32)
    N, D = X.shape
    assert D % group_size == 0
    Xg = X.reshape(N, D // group_size, group_size)
    mn = Xg.min(axis=-1)
    mx = Xg.max(axis=-1)
    with np.errstate(over="ignore"):
        s16 = _fp16_sat_array((mx - mn) / np.float32(15.0))
    degenerate = (mx == mn) | (s16 == 0)
    s16[degenerate] = np.float16(1.0)
    s32 = s16.astype(np.float32)
    z16 = _fp16_sat_array((-mn) / s32)
    z16[z16 == 0] = np.float16(0.0)
    z32 = z16.astype(np.float32)
    v = (Xg / s32[..., None]) + z32[..., None]
    q = np.clip(np.rint(v), 0.0, 15.0).astype(np.uint8)
    return q.reshape(N, D), s16, z16


def int4_dequantize_rows(codes, s16, z16, group_size):
    N, D = codes.shape
    c = codes.reshape(N, D // group_size, group_size).astype(np.float64)
    out = (c - z16.astype(np.float64)[..., None]) * s16.astype(np.float64)[..., None]
    return out.reshape(N, D)


def pack_nibbles(codes):
    """[..., D] codes in 0..15 -> [..., D/2] bytes, element 2i low, 2i+1 high."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed):
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0x0F
    out[..., 1::2] = packed >> 4
    return out


# -------------------------------------------------------------- FP8 E4M3
def e4m3_decode_exact(code):
    """Exact value of an OCP E4M3 (fn) code as a Fraction; None for NaN."""
    code = int(code)
    sign = -1 if code & 0x80 else 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return None
    if e == 0:
        mag = Fraction(m, 8) * Fraction(1, 64)  # subnormal: 0.m * 2^-6
    else:
        mag = (1 + Fraction(m, 8)) * (Fraction(2) ** (e - 7))
    return sign * mag


E4M3_VALUES = np.array(
    [np.nan if e4m3_decode_exact(c) is None else float(e4m3_decode_exact(c)) for c in range(256)],
    dtype=np.float64,
)
# Finite non-negative codes 0x00..0x7E in increasing magnitude.
_E4M3_POS = E4M3_VALUES[:0x7F]


def e4m3_encode(v):
    """Nearest E4M3 code of a finite binary32 value, ties to even mantissa,
    saturating at +-448 (sign of zero kept).  Exact rational comparison."""
    v = np.float32(v)
    if np.isnan(v):
        raise ValueError("NaN has no E4M3 encoding here")
    sign = 0x80 if np.signbit(v) else 0x00
    mag = Fraction(abs(float(v)))
    if mag >= Fraction(448):
        return sign | 0x7E
    best, best_d = None, None
    for c in range(0x7F):
        d = abs(e4m3_decode_exact(c) - mag)
        if best is None or d < best_d or (d == best_d and (c & 1) == 0):
            best, best_d = c, d
    return sign | best


def e4m3_encode_array(values):
    """Vectorised nearest-with-ties-to-even over the sorted magnitude table."""
    v = np.asarray(values, dtype=np.float32)
    if np.isnan(v).any():
        raise ValueError("NaN has no E4M3 encoding here")
    sign = np.where(np.signbit(v), 0x80, 0x00).astype(np.uint8)
    mag = np.abs(v).astype(np.float64)
    mag = np.minimum(mag, E4M3_MAX)
    hi = np.searchsorted(_E4M3_POS, mag, side="left")  # first table value >= mag
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E4M3_POS[hi] - mag
    d_lo = mag - _E4M3_POS[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    # exact hits: hi value == mag -> d_hi == 0, never loses to lo unless lo == hi
    code = np.where(pick_lo & (d_hi != 0), lo, hi).astype(np.uint8)
    return code | sign


def fp8_quantize_row(x):
    """Quantise one (token, head) row. Returns (codes uint8 [D], s16)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.float32(np.abs(x).max())
    s16 = fp16_sat(a / np.float32(E4M3_MAX))
    if s16 == 0:
        s16 = np.float16(1.0)
    s32 = np.float32(s16)
    codes = np.array([e4m3_encode(np.float32(xi / s32)) for xi in x], dtype=np.uint8)
    return codes, s16


def fp8_quantize_rows(X):
    """Element-wise version of ``fp8_quantize_row``. X: [N, D]."""
    X = np.asarray(X, dtype=np.float32)
    a = np.abs(X).max(axis=-1)
    s16 = _fp16_sat_array(a / np.float32(E4M3_MAX))
    s16[s16 == 0] = np.float16(1.0)
    s32 = s16.astype(np.float32)
    codes = e4m3_encode_array(X / s32[:, None])
    return codes, s16


def fp8_dequantize_rows(codes, s16):
    return E4M3_VALUES[np.asarray(codes, dtype=np.int64)] * s16.astype(np.float64)[:, None]
