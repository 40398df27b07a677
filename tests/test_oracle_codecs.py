"""Pins for the oracle's number formats (no GPU).

Every check compares the oracle against something other than itself: the
pages' codebook, the OCP specification tables under tests/golden/, exact
rational arithmetic (fractions), Python's own float formatting, and torch's
independent dtype casts.
"""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import codecs as C

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    for line in open(os.path.join(GOLD, name), encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append(line.split())
    return rows


# --------------------------------------------------------------------------- 2-bit

def test_w2_codebook_matches_pages():
    tab = {int(a): float(b) for a, b in _read_table("w2_codebook.txt")}
    assert [tab[c] for c in range(4)] == list(C.W2_CODEBOOK)


def test_w2_unpack_all_bytes():
    """All 256 bytes: element i of a byte is bits 2i..2i+1, read here from the
    binary string of the byte."""
    b = np.arange(256, dtype=np.uint8)[:, None]
    got = C.unpack_w2_codes(b)
    for v in range(256):
        s = format(v, "08b")[::-1]            # s[i] = bit i
        want = [int(s[2 * i]) + 2 * int(s[2 * i + 1]) for i in range(4)]
        assert list(got[v]) == want


def test_w2_decode_exhaustive_codes_with_scales():
    """Every byte with several fp16 scales (normal, subnormal, ties for the bf16
    rounding): value == codebook * bf16(scale), bf16 taken from torch."""
    tab = {int(a): float(b) for a, b in _read_table("w2_codebook.txt")}
    scales = np.array([0.02, 1.0, 6.1e-5, 3.0e-7, 0.0131, 65504.0, 0.00999, 1.0 + 2 ** -8],
                      dtype=np.float16)
    for s in scales:
        packed = np.tile(np.arange(256, dtype=np.uint8), 8)[None, :]      # 2048 elements
        sc = np.full((1, packed.shape[1] * 4 // 32), s, dtype=np.float16)
        got = C.decode_w2(packed, sc)[0]
        sb = float(torch.tensor(float(s), dtype=torch.float32).to(torch.bfloat16).float())
        codes = [(int(byte) >> (2 * i)) & 3 for byte in packed[0] for i in range(4)]
        want = np.array([tab[c] * sb for c in codes])
        assert np.array_equal(got, want)
        # "entry * bf16(s) == bf16(entry * s)": the codebook is powers of two
        for c in range(4):
            direct = float(torch.tensor(tab[c] * float(s), dtype=torch.float32).to(torch.bfloat16).float())
            assert direct == tab[c] * sb


# --------------------------------------------------------------------------- bf16

def test_bf16_rne_matches_torch_including_ties():
    g = np.random.default_rng(7)
    a = g.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    # exact ties: low 16 bits == 0x8000 with both parities of the kept lsb
    u = g.integers(0, 2 ** 31, 4000, dtype=np.uint64).astype(np.uint32)
    ties = ((u & 0x7FFF0000) | 0x8000).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 1e-40, -1e-44], dtype=np.float32)
    a = np.concatenate([a, ties, special])
    a = a[np.isfinite(a) | np.isinf(a)]
    got = C.f32_to_bf16_bits(a)
    want = torch.from_numpy(a.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    assert np.isnan(C.bf16_bits_to_f64(C.f32_to_bf16_bits(np.array([np.nan], np.float32)))[0])


def test_fp16_decode_matches_struct():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    got = C.fp16_to_f64(h)
    for bits in range(0, 65536, 97):
        (v,) = struct.unpack("<e", struct.pack("<H", bits))
        if math.isnan(v):
            assert math.isnan(got[bits])
        else:
            assert got[bits] == v


# --------------------------------------------------------------------------- E2M1 / E8M0

def test_e2m1_table_matches_ocp():
    tab = _read_table("e2m1_ocp.txt")
    got = C.e2m1_value(np.arange(16))
    for nib, v in tab:
        assert got[int(nib)] == float(v)
        assert math.copysign(1.0, got[int(nib)]) == math.copysign(1.0, float(v))


def test_e2m1_matches_torch_fp4():
    packed = np.arange(256, dtype=np.uint8)
    nibs = C.unpack_e2m1(packed[None, :])[0]
    ours = C.e2m1_value(nibs)
    tv = torch.from_numpy(packed.copy()).view(torch.float4_e2m1fn_x2)
    # torch's fp4 container has no float cast; decode by its documented nibble order:
    # element 0 of the pair is the low nibble.
    lo = np.array([float(C.e2m1_value(b & 15)) for b in range(256)])
    assert np.array_equal(ours[0::2], lo)
    assert tv.numel() == 256


def test_e8m0_all_bytes():
    b = np.arange(256)
    got = C.e8m0_value(b)
    for v in range(255):
        assert got[v] == math.ldexp(1.0, v - 127)
    assert np.isnan(got[255])
    t = torch.tensor([2.0 ** (v - 127) for v in range(1, 255)], dtype=torch.float32)
    assert list(t.to(torch.float8_e8m0fnu).view(torch.uint8).numpy()) == list(range(1, 255))


def test_mxfp4_decode_layout():
    """Low nibble first; the block scale applies to 32 consecutive elements."""
    packed = np.array([[0x21] * 16 + [0xF7] * 16], dtype=np.uint8)        # 64 elements
    sc = np.array([[127, 130]], dtype=np.uint8)
    v = C.decode_mxfp4(packed, sc)[0]
    assert list(v[:4]) == [0.5, 1.0, 0.5, 1.0]
    assert list(v[32:34]) == [6.0 * 8, -6.0 * 8]


# --------------------------------------------------------------------------- E4M3

def test_e4m3_landmarks():
    for row in _read_table("e4m3_landmarks.txt"):
        if row[0] == "sat":
            assert int(C.e4m3_encode(np.array([float(row[1])]))[0]) == int(row[2], 16)
            continue
        byte, val = int(row[0], 16), float(row[1])
        got = C.e4m3_value(np.array([byte]))[0]
        assert got == val and math.copysign(1, got) == math.copysign(1, val)
        assert int(C.e4m3_encode(np.array([val]))[0]) == byte
    assert int(C.e4m3_encode(np.array([np.nan]))[0]) == 0x7F
    assert np.isnan(C.e4m3_value(np.array([0x7F, 0xFF]))).all()


def test_e4m3_encode_matches_torch_in_range():
    g = np.random.default_rng(3)
    a = np.concatenate([g.standard_normal(50000) * 40, g.standard_normal(20000) * 1e-2,
                        g.uniform(-463.99, 463.99, 20000)])
    # all midpoints between adjacent codes (ties) and the codes themselves
    t = C.E4M3_TABLE
    mids = (t[1:] + t[:-1]) / 2
    a = np.concatenate([a, mids, -mids, t, -t]).astype(np.float32).astype(np.float64)
    got = C.e4m3_encode(a)
    want = torch.from_numpy(a.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def _e4m3_values_exact():
    vals = {}
    for c in range(127):
        e, m = c >> 3, c & 7
        vals[c] = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return vals


def test_mxfp4_to_e4m3_exhaustive_against_fractions():
    """All 16 codes x 256 scale bytes, brute force over the 127 E4M3 values in
    exact rational arithmetic (nearest, ties to even mantissa, saturation)."""
    ev = _e4m3_values_exact()
    e2m1 = {0: Fraction(0), 1: Fraction(1, 2), 2: Fraction(1), 3: Fraction(3, 2), 4: Fraction(2),
            5: Fraction(3), 6: Fraction(4), 7: Fraction(6)}
    nib = np.arange(16, dtype=np.uint8)
    for b in range(256):
        packed = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
        packed = np.tile(packed, 2)[None, :]                       # 32 elements = one block
        got = C.mxfp4_to_e4m3(packed, np.array([[b]], dtype=np.uint8))[0][:16]
        for n in range(16):
            if b == 255:
                assert got[n] == 0x7F
                continue
            mag = e2m1[n & 7] * Fraction(2) ** (b - 127)
            if mag >= 448:
                code = 126
            else:
                best = None
                for c, v in ev.items():
                    d = abs(v - mag)
                    if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
                        best = (d, c)
                code = best[1]
            want = code | (0x80 if n & 8 else 0)
            assert got[n] == want, (b, n)


def test_mxfp4_to_e4m3_is_exact_in_the_stated_range():
    nib = np.arange(16, dtype=np.uint8)
    packed = np.tile((nib[0::2] | (nib[1::2] << 4)).astype(np.uint8), 2)[None, :]
    for b in range(127 - 8, 127 + 7):
        s = np.array([[b]], dtype=np.uint8)
        assert np.array_equal(C.e4m3_value(C.mxfp4_to_e4m3(packed, s)), C.decode_mxfp4(packed, s))


# --------------------------------------------------------------------------- MXFP8

def _mxfp8_bruteforce(block):
    """Scale exponent by search: the X with 2^8 <= amax*2^-X < 2^9; elements by
    torch's RNE cast after clamping to +-448 (saturation)."""
    amax = max(abs(float(v)) for v in block)
    if amax == 0:
        X = -127
    else:
        X = 0
        while amax * 2.0 ** -X >= 512:
            X += 1
        while amax * 2.0 ** -X < 256:
            X -= 1
        X = max(-127, min(127, X))
    scaled = np.clip(np.asarray(block, dtype=np.float64) * 2.0 ** -X, -448, 448)
    q = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return q, X + 127


def test_mxfp8_quantize_bruteforce():
    g = np.random.default_rng(11)
    a = np.concatenate([g.standard_normal(32 * 64) * 3.0,
                        np.zeros(32),
                        g.standard_normal(32) * 1e-30,
                        np.full(32, 511.0), np.full(32, 512.0)]).astype(np.float32).astype(np.float64)
    a[5] = 1000.0
    q, s = C.mxfp8_quantize(a[None, :])
    for blk in range(a.size // 32):
        qb, sb = _mxfp8_bruteforce(a[blk * 32:(blk + 1) * 32])
        assert s[0, blk] == sb, blk
        assert np.array_equal(q[0, blk * 32:(blk + 1) * 32], qb), blk
