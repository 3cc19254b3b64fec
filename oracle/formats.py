"""Number formats of the layer, written from their definitions (fp64 throughout).

The pages name the formats only: FP8 activations with UE8M0 scale factors,
FP4 weights, recipe ``(1, 1, 32)`` (one scale per 32 elements along K) --
DeepGEMM ``fp8_fp4_mega_moe`` call on the digest page of sglang PR #36657,
section 关键源码片段; the ``x_sf`` / ``l1_acts_sf`` views of the DeepGEMM SM90
MegaMoE dev log, Phase 1 entry.  The element formats are those of the OCP
Microscaling (MX) specification v1.0:

* E4M3 ("fn"): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; no
  infinities; S.1111.111 is NaN; largest finite 448; subnormal step 2^-9.
* E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes
  {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* UE8M0: unsigned 8-bit exponent, value 2^(b - 127); b = 255 is NaN.

Block quantiser ("rule Q"): for each run of 32 elements with largest
magnitude a, the scale exponent s is the smallest integer with a <= F * 2^s
(F = 448 for E4M3, 6 for E2M1), clamped to [-127, 127]; an all-zero block
takes s = 0 (byte 127).  Each element becomes RNE(v / 2^s) in the element
format.  The pages do not spell the rule out; rounding the scale *up* is the
one choice that never saturates an element (it is also the ceil-to-power-of-
two scale used for UE8M0 casts in the DeepSeek/DeepGEMM tooling).
"""
from __future__ import annotations

import numpy as np

E4M3 = "e4m3"
E2M1 = "e2m1"

# (mantissa bits, exponent bias, min normal exponent, largest finite)
_SPEC = {
    E4M3: (3, 7, -6, 448.0),
    E2M1: (1, 1, 0, 6.0),
}
BLOCK = 32


# ---------------------------------------------------------------- decoding
def e4m3_decode_table() -> np.ndarray:
    """Value of every E4M3 code 0..255 (NaN for 0x7F / 0xFF)."""
    out = np.empty(256, dtype=np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            out[c] = np.nan
        elif e == 0:
            out[c] = sign * m * 2.0 ** -9          # m/8 * 2^(1-7)
        else:
            out[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


def e2m1_decode_table() -> np.ndarray:
    """Value of every E2M1 code 0..15."""
    out = np.empty(16, dtype=np.float64)
    for c in range(16):
        sign = -1.0 if c & 0x8 else 1.0
        e = (c >> 1) & 0x3
        m = c & 0x1
        if e == 0:
            out[c] = sign * m * 0.5                # m/2 * 2^(1-1)
        else:
            out[c] = sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return out


_E4M3_TAB = e4m3_decode_table()
_E2M1_TAB = e2m1_decode_table()


def ue8m0_decode(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.int64)
    out = np.ldexp(1.0, b - 127).astype(np.float64)
    return np.where(b == 255, np.nan, out)


def decode(codes, fmt: str) -> np.ndarray:
    """Unpacked element codes (one per byte) -> fp64 values."""
    codes = np.asarray(codes, dtype=np.uint8)
    tab = _E4M3_TAB if fmt == E4M3 else _E2M1_TAB
    return tab[codes]


def unpack_e2m1(packed) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] codes; element 2c is the low nibble of byte c."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def pack_e2m1(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] & 0xF) | ((codes[..., 1::2] & 0xF) << 4)


def dequantize(codes, sf, fmt: str) -> np.ndarray:
    """codes [..., K] (unpacked), sf [..., K/32] -> fp64 [..., K]."""
    v = decode(codes, fmt)
    scale = ue8m0_decode(sf)
    shp = v.shape
    return (v.reshape(shp[:-1] + (shp[-1] // BLOCK, BLOCK)) * scale[..., None]).reshape(shp)


# ---------------------------------------------------------------- encoding
def encode(v, fmt: str) -> np.ndarray:
    """Round-to-nearest-even into the element format, saturating at the
    largest finite value; the sign bit follows the sign of v (so a negative
    value that rounds to zero gives negative zero).  v must be finite."""
    mbits, bias, emin, vmax = _SPEC[fmt]
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("encode: non-finite input")
    mag = np.abs(v)
    _, p = np.frexp(mag)                     # mag = f * 2^p, f in [0.5, 1)
    E = np.maximum(p - 1, emin)              # exponent of the binade (subnormals share emin)
    ulp = np.ldexp(1.0, E - mbits)
    r = np.rint(mag / ulp) * ulp             # exact: mag/ulp is exact, rint is RNE
    r = np.minimum(r, vmax)
    # code of r
    _, pr = np.frexp(r)
    Er = pr - 1
    normal = r >= np.ldexp(1.0, emin)
    sub_code = np.rint(r / np.ldexp(1.0, emin - mbits)).astype(np.int64)
    mant = np.rint((r / np.ldexp(1.0, np.where(normal, Er, 0)) - 1.0) * (1 << mbits)).astype(np.int64)
    norm_code = ((Er + bias).astype(np.int64) << mbits) | mant
    code = np.where(normal, norm_code, sub_code)
    sign_bit = 0x80 if fmt == E4M3 else 0x8
    code = np.where(np.signbit(v), code | sign_bit, code)
    return code.astype(np.uint8)


def scale_exponent(amax, fmt: str) -> np.ndarray:
    """Rule Q: smallest integer s with amax <= F * 2^s, clamped to [-127, 127];
    0 for amax == 0.  Exact (integer arithmetic on the binary exponent)."""
    a = np.asarray(amax, dtype=np.float64)
    f, p = np.frexp(a)                       # a = (2f) * 2^(p-1), 2f in [1, 2)
    P = p - 1
    m = 2.0 * f
    if fmt == E4M3:                          # F = 1.75 * 2^8
        s = np.where(m <= 1.75, P - 8, P - 7)
    else:                                    # F = 1.5 * 2^2
        s = np.where(m <= 1.5, P - 2, P - 1)
    s = np.clip(s, -127, 127)
    return np.where(a == 0, 0, s).astype(np.int64)


def quantize_mx(v, fmt: str):
    """Rule Q over blocks of 32 along the last axis.

    Returns (codes uint8 [..., K] unpacked, sf uint8 [..., K/32])."""
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    if K % BLOCK:
        raise ValueError("last dimension must be a multiple of 32")
    blocks = v.reshape(v.shape[:-1] + (K // BLOCK, BLOCK))
    amax = np.max(np.abs(blocks), axis=-1) if K else np.zeros(v.shape[:-1] + (0,))
    s = scale_exponent(amax, fmt)
    q = blocks / np.ldexp(1.0, s)[..., None]
    codes = encode(q, fmt).reshape(v.shape)
    sf = (s + 127).astype(np.uint8)
    return codes, sf


# ---------------------------------------------------------------- bfloat16
def bf16_round(v) -> np.ndarray:
    """One round-to-nearest-even of an fp64 value to bfloat16 (8 significant
    bits, fp32 exponent range, subnormal step 2^-133), returned as fp64."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.abs(v)
    _, p = np.frexp(mag)
    E = np.maximum(p - 1, -126)
    ulp = np.ldexp(1.0, E - 7)
    r = np.rint(mag / ulp) * ulp
    bf_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(r > bf_max, np.inf, r)
    return np.copysign(r, v)


def bf16_bits(v) -> np.ndarray:
    """bf16 bit patterns (uint16) of bf16_round(v)."""
    r = np.asarray(bf16_round(v), dtype=np.float32)     # exact: r is a bf16 value
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
