"""Pins for oracle.formats: closed forms, library routines, brute force.

None of these tests reuses the oracle's own formula: decode tables are
checked against PyTorch's float8_e4m3fn bit casts and a literal E2M1 table,
encoding against brute-force nearest search over the representable values
and against PyTorch's RNE cast, rule Q against an exhaustive scan over the
scale exponent, and bf16 rounding against exact rational arithmetic.
"""
from fractions import Fraction
import math
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ decode
def test_e4m3_table_matches_torch_bitcast():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = F.e4m3_decode_table()
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok]))


def test_format_endpoints_fixture():
    for fmt, code, val in _golden("format_endpoints.txt"):
        code = int(code, 16)
        want = float("nan") if val == "nan" else float(Fraction(val))
        if fmt == "e4m3":
            got = F.e4m3_decode_table()[code]
        elif fmt == "e2m1":
            got = F.e2m1_decode_table()[code]
        else:
            got = float(F.ue8m0_decode(code))
        if math.isnan(want):
            assert math.isnan(got), (fmt, code)
        else:
            assert got == want, (fmt, hex(code), got, want)


def test_e2m1_literal_table():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    want = np.array(mags + [-m for m in mags])
    got = F.e2m1_decode_table()
    assert np.array_equal(got, want)
    assert np.signbit(got[8])  # 0x8 is negative zero


def test_ue8m0_every_code():
    b = np.arange(256)
    got = F.ue8m0_decode(b)
    for v in range(255):
        assert got[v] == math.ldexp(1.0, v - 127)
    assert math.isnan(got[255])


def test_e2m1_nibble_order():
    # element 2c in the low nibble of byte c
    codes = np.array([[1, 2, 3, 15]], dtype=np.uint8)
    packed = F.pack_e2m1(codes)
    assert packed.tolist() == [[0x21, 0xF3]]
    assert np.array_equal(F.unpack_e2m1(packed), codes)


# ------------------------------------------------------------------ encode
def _brute_encode(v, fmt):
    """Nearest representable by exhaustive search, ties to the even code,
    saturating; sign bit from the sign of v."""
    tab = F.e4m3_decode_table() if fmt == F.E4M3 else F.e2m1_decode_table()
    n = 128 if fmt == F.E4M3 else 8
    sign_bit = 0x80 if fmt == F.E4M3 else 0x8
    mags = [(c, tab[c]) for c in range(n) if not math.isnan(tab[c])]
    vmax = max(m for _, m in mags)
    out = []
    for x in np.asarray(v, dtype=np.float64).reshape(-1):
        a = min(abs(Fraction(float(x))), Fraction(vmax))
        best = None
        for c, m in mags:
            d = abs(Fraction(m) - a)
            if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
                best = (d, c)
        c = best[1]
        if math.copysign(1.0, x) < 0:
            c |= sign_bit
        out.append(c)
    return np.array(out, dtype=np.uint8)


@pytest.mark.parametrize("fmt", [F.E4M3, F.E2M1])
def test_encode_roundtrip_every_representable(fmt):
    tab = F.e4m3_decode_table() if fmt == F.E4M3 else F.e2m1_decode_table()
    codes = np.array([c for c in range(len(tab)) if not math.isnan(tab[c])], dtype=np.uint8)
    assert np.array_equal(F.encode(tab[codes], fmt), codes)


@pytest.mark.parametrize("fmt", [F.E4M3, F.E2M1])
def test_encode_midpoints_and_random_vs_brute_force(fmt):
    tab = F.e4m3_decode_table() if fmt == F.E4M3 else F.e2m1_decode_table()
    n = 127 if fmt == F.E4M3 else 8
    pos = np.sort(tab[:n])
    mids = (pos[1:] + pos[:-1]) / 2          # exact ties
    rng = np.random.default_rng(1)
    vmax = pos[-1]
    rnd = rng.uniform(-1.2 * vmax, 1.2 * vmax, 400)
    small = rng.uniform(-pos[2], pos[2], 100)
    v = np.concatenate([mids, -mids, rnd, small, [0.0, -0.0, -1e-300, 1e30, -1e30]])
    assert np.array_equal(F.encode(v, fmt), _brute_encode(v, fmt))


def test_e4m3_encode_matches_torch_rne_cast():
    rng = np.random.default_rng(2)
    v = np.concatenate([
        rng.standard_normal(20000) * 30.0,
        rng.standard_normal(5000) * 2.0 ** -8,   # subnormal range
        (F.e4m3_decode_table()[1:126] + F.e4m3_decode_table()[2:127]) / 2,  # ties
    ]).astype(np.float32)
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.encode(v.astype(np.float64), F.E4M3)
    assert np.array_equal(got, ref)


def test_negative_zero_and_saturation():
    assert F.encode(np.array([-1e-30]), F.E4M3)[0] == 0x80
    assert F.encode(np.array([-1e-30]), F.E2M1)[0] == 0x8
    assert F.encode(np.array([1000.0]), F.E4M3)[0] == 0x7E
    assert F.encode(np.array([-7.0]), F.E2M1)[0] == 0xF


# ------------------------------------------------------------------ rule Q
def _brute_scale(a, fmt):
    Fmax = Fraction(448) if fmt == F.E4M3 else Fraction(6)
    if a == 0:
        return 0
    fa = Fraction(float(a))
    for s in range(-127, 128):
        if fa <= Fmax * Fraction(2) ** s:
            return s
    return 127


@pytest.mark.parametrize("fmt", [F.E4M3, F.E2M1])
def test_scale_exponent_vs_exhaustive_scan(fmt):
    rng = np.random.default_rng(3)
    Fmax = 448.0 if fmt == F.E4M3 else 6.0
    a = np.exp2(rng.uniform(-140, 120, 3000)) * rng.uniform(1, 2, 3000)
    edges = []
    for s in (-130, -127, -126, -20, -1, 0, 1, 7, 50, 120):
        x = math.ldexp(Fmax, s)
        edges += [x, np.nextafter(x, 0), np.nextafter(x, np.inf)]
    a = np.concatenate([a, edges, [0.0]])
    got = F.scale_exponent(a, fmt)
    want = np.array([_brute_scale(x, fmt) for x in a])
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", [F.E4M3, F.E2M1])
def test_quantize_block_properties(fmt):
    rng = np.random.default_rng(4)
    Fmax = 448.0 if fmt == F.E4M3 else 6.0
    v = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-30, 30, (64, 1)))
    v[3, :32] = 0.0
    codes, sf = F.quantize_mx(v, fmt)
    s = sf.astype(np.int64) - 127
    blocks = np.abs(v).reshape(64, 8, 32).max(-1)
    scale = np.ldexp(1.0, s)
    nz = blocks > 0
    assert np.all(blocks[nz] <= Fmax * scale[nz])            # fits
    assert np.all(blocks[nz] > Fmax * scale[nz] / 2)         # smallest such s
    assert sf[3, 0] == 127
    dec = F.decode(codes, fmt).reshape(64, 8, 32)
    assert np.all(np.abs(dec) <= Fmax)
    # every element is the nearest representable of v / 2^s
    q = v.reshape(64, 8, 32) / scale[..., None]
    sub = q.reshape(-1)[:1500]
    assert np.array_equal(codes.reshape(-1)[:1500], _brute_encode(sub, fmt))


def test_quantize_roundtrip_on_representable_blocks():
    """A block whose values are representable at its own scale comes back exactly."""
    rng = np.random.default_rng(5)
    tab = F.e4m3_decode_table()[:127]
    for _ in range(50):
        s = int(rng.integers(-20, 20))
        vals = rng.choice(tab, 32) * rng.choice([-1.0, 1.0], 32)
        vals[0] = 448.0 if rng.random() < 0.5 else 320.0   # pins the block max
        v = vals * 2.0 ** s
        codes, sf = F.quantize_mx(v[None, :], F.E4M3)
        assert np.array_equal(F.dequantize(codes, sf, F.E4M3)[0], v)


# ------------------------------------------------------------------ bf16
def _bf16_exact(x: float) -> float:
    if x == 0:
        return x
    fx = abs(Fraction(x))
    e = math.floor(math.log2(fx))
    while Fraction(2) ** e > fx:
        e -= 1
    while Fraction(2) ** (e + 1) <= fx:
        e += 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 7)
    q = fx / ulp
    n = math.floor(q)
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * ulp
    if r > (2 - Fraction(1, 128)) * Fraction(2) ** 127:
        return math.copysign(math.inf, x)
    return math.copysign(float(r), x)


def test_bf16_round_vs_exact_rationals():
    rng = np.random.default_rng(6)
    v = np.concatenate([
        rng.standard_normal(3000) * np.exp2(rng.uniform(-140, 130, 3000)),
        # exact ties in fp64 (not representable in fp32): 1 + 2^-8 + tiny
        [1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -40, -(1 + 2 ** -8),
         3.3895313892515355e38, 3.4e38, 1e-45, 2 ** -133, 2 ** -134, 3 * 2 ** -135],
    ])
    got = F.bf16_round(v)
    want = np.array([_bf16_exact(float(x)) for x in v])
    assert np.array_equal(got, want)


def test_bf16_round_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(20000) * 100).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).float().double().numpy()
    assert np.array_equal(F.bf16_round(v.astype(np.float64)), ref)
    bits = F.bf16_bits(v.astype(np.float64))
    assert np.array_equal(bits, torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
