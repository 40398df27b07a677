"""Number formats used by the layer, written out from their definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

All routines take / return NumPy arrays and work elementwise.  Values are
carried as float64, which holds every bf16, fp16, e4m3, E2M1 and E8M0 value
(and every product of a codebook value with a bf16 scale) exactly.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# bf16 / fp16 / fp32
# ---------------------------------------------------------------------------


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values (bf16 is the upper
    half of an fp32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round-to-nearest-even of fp32 values to bf16 (IEEE 754 rounding
    applied to the 8-bit significand); NaN stays NaN (quiet), inf stays inf."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint32)
    nan = np.isnan(a)
    r = np.where(nan, ((u >> 16) | 0x40).astype(np.uint32), r)
    return r.astype(np.uint16)


def rne_bf16(a) -> np.ndarray:
    """Value of bf16 RNE(a) for float64 input a: a is first rounded to the
    nearest fp32 (RNE), then to bf16.  For the layer this double rounding is
    the definition: the values rounded to bf16 are fp32 results."""
    return bf16_bits_to_f64(f32_to_bf16_bits(np.asarray(a, dtype=np.float64).astype(np.float32)))


def fp16_to_f64(h: np.ndarray) -> np.ndarray:
    return np.asarray(h, dtype=np.float16).astype(np.float64)


def to_f32(a) -> np.ndarray:
    """Round float64 to the nearest fp32 (as float64)."""
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# 2-bit codebook {-4, -1, 1, 4} with fp16 group-32 scales
# ---------------------------------------------------------------------------

# Code c (0..3) names the c-th entry of the sign-symmetric codebook in
# ascending order.  The pages give the codebook {-4,-1,1,4} (blog
# "这个项目我们能学到什么?" on vLLM-Moet) but not the code -> entry order; the
# ascending order is this library's convention.
W2_CODEBOOK = np.array([-4.0, -1.0, 1.0, 4.0])


def unpack_w2_codes(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., K/4] -> code indices uint8 [..., K]; element i sits at bits
    2*(i%4) .. 2*(i%4)+1 of byte i//4."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 4,), dtype=np.uint8)
    for j in range(4):
        out[..., j::4] = (p >> (2 * j)) & 3
    return out


def w2_effective_scale(scales_fp16: np.ndarray) -> np.ndarray:
    """The group scale a bf16 dequantised tile carries: RNE_bf16(fp16 scale).

    The codebook entries are +-1 and +-4 (powers of two), so
    entry * RNE_bf16(s) == RNE_bf16(entry * s) exactly: the dequantised weight
    is the bf16 value nearest to entry * s."""
    return rne_bf16(fp16_to_f64(scales_fp16))


def decode_w2(packed: np.ndarray, scales_fp16: np.ndarray) -> np.ndarray:
    """Dequantise 2-bit codebook weights: [..., K/4] codes + [..., K/32] fp16
    scales -> float64 [..., K] with w = codebook[c] * RNE_bf16(scale)."""
    codes = unpack_w2_codes(packed)
    vals = W2_CODEBOOK[codes]
    s = w2_effective_scale(scales_fp16)
    return vals * np.repeat(s, 32, axis=-1)


# ---------------------------------------------------------------------------
# OCP MX formats: E2M1 (FP4), E8M0 (shared scale), E4M3 (FP8)
# ---------------------------------------------------------------------------

def e2m1_value(nib) -> np.ndarray:
    """E2M1 (1 sign, 2 exponent, 1 mantissa bit, bias 1, no inf/NaN):
    exponent field 0 is subnormal (0 or 0.5); otherwise 2^(e-1) * (1 + m/2).
    Nibble 0b1000 is -0."""
    nib = np.asarray(nib, dtype=np.int64)
    s = (nib >> 3) & 1
    e = (nib >> 1) & 3
    m = nib & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return np.where(s == 1, -mag, mag)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] -> nibbles uint8 [..., K]; element 2i is the LOW nibble."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def e8m0_value(b) -> np.ndarray:
    """E8M0 byte b -> 2^(b-127); b = 255 is NaN."""
    b = np.asarray(b, dtype=np.int64)
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


def decode_mxfp4(packed: np.ndarray, e8m0: np.ndarray) -> np.ndarray:
    """MXFP4 dequantisation: value = E2M1 * 2^(E8M0-127) per block of 32
    along the last axis (exact in float64; NaN where the scale byte is 255)."""
    v = e2m1_value(unpack_e2m1(packed))
    return v * np.repeat(e8m0_value(e8m0), 32, axis=-1)


def _e4m3_table() -> np.ndarray:
    """Values of the 127 finite non-negative E4M3 codes 0x00..0x7E (bias 7;
    exponent field 0 is subnormal m/8 * 2^-6; 0x7F is NaN; no infinities)."""
    c = np.arange(127)
    e = c >> 3
    m = c & 7
    return np.where(e == 0, m / 8.0 * 2.0 ** -6, np.ldexp(1.0 + m / 8.0, e - 7))


E4M3_TABLE = _e4m3_table()
E4M3_MAX = 448.0


def e4m3_value(b) -> np.ndarray:
    """E4M3 byte -> value (NaN for 0x7F / 0xFF)."""
    b = np.asarray(b, dtype=np.int64)
    mag_code = b & 0x7F
    mag = np.where(mag_code == 0x7F, np.nan, E4M3_TABLE[np.minimum(mag_code, 126)])
    return np.where((b & 0x80) != 0, -mag, mag)


def e4m3_encode(a) -> np.ndarray:
    """Round-to-nearest-even into E4M3 with saturation to +-448 (OCP "satfinite"
    conversion).  NaN -> 0x7F; the sign of zero is kept (-0 -> 0x80).

    Ties go to the code with an even mantissa, which for adjacent codes of the
    monotone table is the even code."""
    a = np.asarray(a, dtype=np.float64)
    mag = np.abs(a)
    sat = mag >= E4M3_MAX
    magc = np.where(sat | np.isnan(mag), 0.0, mag)
    hi = np.searchsorted(E4M3_TABLE, magc, side="left")         # first table value >= mag
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    dlo = magc - E4M3_TABLE[lo]
    dhi = E4M3_TABLE[hi] - magc
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(sat, 126, code)
    neg = np.signbit(a)
    out = (code | np.where(neg, 0x80, 0)).astype(np.uint8)
    return np.where(np.isnan(a), np.uint8(0x7F), out).astype(np.uint8)


def mxfp4_to_e4m3(packed: np.ndarray, e8m0: np.ndarray) -> np.ndarray:
    """The online MXFP4 -> FP8 conversion ("国产GPU完成MoE大模型Day-0适配", §四):
    each weight's value E2M1 * 2^(E8M0-127) is written as one E4M3 byte of a
    plain FP8 tensor (scale folded in), RNE + saturation; a NaN scale gives
    0x7F.  Exact whenever the value is an E4M3 value, i.e. for every code when
    E8M0-127 lies in [-8, 6]."""
    return e4m3_encode(decode_mxfp4(packed, e8m0))


# ---------------------------------------------------------------------------
# MXFP8 activation quantisation (E4M3 elements, one E8M0 scale per 32)
# ---------------------------------------------------------------------------

def mxfp8_quantize(a: np.ndarray):
    """OCP MX conversion of fp32 values along the last axis in blocks of 32.

    Per block: amax = max |a|; X = floor(log2(amax)) - 8 (8 = exponent of
    E4M3's largest normal), taken from the binary exponent of amax; amax == 0
    gives X = -127; X is clamped to [-127, 127].  Elements are
    q = E4M3_RNE_satfinite(a * 2^-X).  Returns (q uint8 [...], X+127 uint8
    [..., K/32])."""
    a = np.asarray(a, dtype=np.float64)
    blk = a.reshape(a.shape[:-1] + (a.shape[-1] // 32, 32))
    amax = np.max(np.abs(blk), axis=-1)
    _, ex = np.frexp(amax)                       # amax = f * 2^ex, f in [0.5, 1)
    X = np.where(amax == 0, -127, ex - 1 - 8)
    X = np.clip(X, -127, 127)
    q = e4m3_encode(blk * np.ldexp(1.0, -X)[..., None])
    return q.reshape(a.shape), (X + 127).astype(np.uint8)


def mxfp8_dequantize(q: np.ndarray, sbytes: np.ndarray) -> np.ndarray:
    v = e4m3_value(q)
    return v * np.repeat(e8m0_value(sbytes), 32, axis=-1)
