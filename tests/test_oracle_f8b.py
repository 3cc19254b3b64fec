"""Pins for oracle.moe_f8b, the (1, 128, 128) recipe.

* the block scale against the exact rational a / 448 rounded to the nearest
  fp32, found without numpy;
* every element code against an exhaustive search of the E4M3 grid for the
  value nearest to the exactly rounded fp32 quotient (ties to the even code,
  saturation at 448);
* an exact round trip of values that the format holds;
* zero blocks, the 128 x 128 block geometry of weights;
* the 1-token / 1-expert layer against an independent scalar computation in
  exact rational arithmetic (except exp);
* the closed form when every expert holds the same weights; token order;
* a planted change of the quantisation rule (multiplying by 448 / a instead
  of dividing by the fp32 scale) is caught.
"""
from fractions import Fraction
import math

import numpy as np
import pytest

from oracle import formats as F
from oracle import moe_f8b as M8
from oracle.routing import route


def _nearest_f32(x: Fraction) -> Fraction:
    """Round-to-nearest-even of a rational to fp32 (normal and subnormal)."""
    if x == 0:
        return Fraction(0)
    ax = abs(x)
    e = 0
    while Fraction(2) ** e > ax:
        e -= 1
    while Fraction(2) ** (e + 1) <= ax:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    q = ax / ulp
    n = math.floor(q)
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2):
        n += 1
    return (1 if x > 0 else -1) * n * ulp


def _e4m3_value(code):
    s = -1 if code & 0x80 else 1
    e, m = (code >> 3) & 15, code & 7
    if e == 0:
        return s * Fraction(m, 512)
    return s * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


_GRID = {c: _e4m3_value(c) for c in range(127)}           # non-negative finite codes 0 .. 448
_SORTED = sorted((v, c) for c, v in _GRID.items())          # increasing value (codes increase with value)
_VALUES = [v for v, _ in _SORTED]


def _nearest_e4m3(q: Fraction) -> Fraction:
    """The E4M3 value nearest to q (ties to the even code), saturating at 448."""
    import bisect

    a = min(abs(q), Fraction(448))
    i = bisect.bisect_left(_VALUES, a)
    cands = [_SORTED[j] for j in (i - 1, i) if 0 <= j < len(_SORTED)]
    d = min(abs(v - a) for v, _ in cands)
    near = [(v, c) for v, c in cands if abs(v - a) == d]
    v, c = min(near, key=lambda vc: vc[1] % 2) if len(near) > 1 else near[0]
    return v if q >= 0 else -v


def _exact_block(vals):
    """(scale, decoded values) of one block by the rule, in exact arithmetic."""
    a = max(abs(Fraction(float(v))) for v in vals)
    s = Fraction(1) if a == 0 else _nearest_f32(a / 448)
    return s, [_nearest_e4m3(_nearest_f32(Fraction(float(v)) / s)) * s for v in vals]


def test_block_scale_and_codes_by_brute_force():
    rng = np.random.default_rng(41)
    for trial in range(6):
        v = (rng.standard_normal((2, 256)) * np.exp(rng.uniform(-8, 8))).astype(np.float32)
        if trial == 1:
            v[0, :128] *= 1e-30                               # tiny values: subnormal codes
        codes, s = M8.quantize_f8b(v, 1)
        assert s.dtype == np.float32 and s.shape == (2, 2)
        dec = M8.dequantize_f8b(codes, s, 1)
        for r in range(2):
            for b in range(2):
                blk = v[r, 128 * b:128 * b + 128]
                es, ev = _exact_block(blk)
                assert Fraction(float(s[r, b])) == es, (trial, r, b)
                assert all(Fraction(float(dec[r, 128 * b + i])) == ev[i] for i in range(128)), (trial, r, b)


def test_round_trip_of_representable_blocks():
    rng = np.random.default_rng(42)
    for j in (-20, -3, 0, 5, 30):
        codes = rng.integers(0, 126, 128).astype(np.uint8) | (rng.integers(0, 2, 128).astype(np.uint8) << 7)
        codes[17] = 0x7E                                       # 448: the block's largest magnitude
        v = F.decode(codes, F.E4M3) * 2.0 ** j
        c2, s = M8.quantize_f8b(v[None, :].astype(np.float32), 1)
        assert float(s[0, 0]) == 2.0 ** j
        assert np.array_equal(F.decode(c2[0], F.E4M3), F.decode(codes, F.E4M3))


def test_zero_block_and_weight_block_geometry():
    v = np.zeros((256, 384), np.float32)
    v[5, 200] = 3.0                       # block (0, 1)
    v[130, 10] = -896.0                   # block (1, 0)
    codes, s = M8.quantize_f8b(v, 128)
    assert s.shape == (2, 3)
    assert np.array_equal(s, np.array([[1.0, 3.0 / 448, 1.0], [2.0, 1.0, 1.0]], np.float32))
    assert codes[5, 200] == 0x7E and codes[130, 10] == 0xFE
    assert np.count_nonzero(codes) == 2
    with pytest.raises(ValueError):
        M8.quantize_f8b(np.zeros((100, 128), np.float32), 128)


def _exact_layer_one_token(x32, W1, W2, clamp, I):
    """Scalar computation of y for k = 1, E = 1, w = 1, independent of the
    oracle: exact rationals for the quantisers and sums, float only for exp."""
    H = x32.shape[0]

    def quant_rows(m, block_rows):
        out = [[None] * m.shape[1] for _ in range(m.shape[0])]
        for r0 in range(0, m.shape[0], block_rows):
            for c0 in range(0, m.shape[1], 128):
                blk = [m[r, c] for r in range(r0, r0 + block_rows) for c in range(c0, c0 + 128)]
                _, ev = _exact_block(blk)
                n = 0
                for r in range(r0, r0 + block_rows):
                    for c in range(c0, c0 + 128):
                        out[r][c] = ev[n]
                        n += 1
        return out

    xs = quant_rows(x32[None, :], 1)[0]
    w1 = quant_rows(W1, 128)
    w2 = quant_rows(W2, 128)
    a1 = [sum(xs[h] * w1[n][h] for h in range(H)) for n in range(2 * I)]
    hv = []
    for i in range(I):
        g, u = a1[i], a1[I + i]
        if clamp:
            L = Fraction(clamp)
            g = min(g, L)
            u = max(min(u, L), -L)
        gf = float(g)
        sig = Fraction(1) / (1 + Fraction(math.exp(-gf)))
        hv.append(Fraction(gf) * sig * Fraction(float(u)))
    h32 = [_nearest_f32(v) for v in hv]                        # the decision is taken in fp32
    hq = []
    for b in range(0, I, 128):
        hq += _exact_block([float(v) for v in h32[b:b + 128]])[1]
    o = [sum(hq[i] * w2[n][i] for i in range(I)) for n in range(H)]
    return np.array([float(F.bf16_round(np.array([float(v)]))[0]) if abs(float(v)) > 0 else 0.0 for v in o])


@pytest.mark.parametrize("clamp", [7.0, 0.0, 0.05])
def test_one_token_one_expert_exact(clamp):
    rng = np.random.default_rng(43)
    H, I = 128, 128
    x = rng.standard_normal(H).astype(np.float32)
    W1 = (rng.standard_normal((2 * I, H)) / math.sqrt(H)).astype(np.float32)
    W2 = (rng.standard_normal((H, I)) / math.sqrt(I)).astype(np.float32)
    xc, xs = M8.quantize_tokens_f8b(x[None, :])
    ex = M8.quantize_expert_f8b(W1, W2)
    y = M8.moe_forward_f8b(xc, xs, np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), lambda e: ex, clamp, 1)
    want = _exact_layer_one_token(x, W1, W2, clamp, I)
    assert np.array_equal(y[0], want)


def test_identical_experts_closed_form():
    rng = np.random.default_rng(44)
    T, H, I, E, k = 20, 256, 128, 5, 3
    x = rng.standard_normal((T, H)).astype(np.float32)
    xc, xs = M8.quantize_tokens_f8b(x)
    ex = M8.quantize_expert_f8b((rng.standard_normal((2 * I, H)) / 16).astype(np.float32),
                                (rng.standard_normal((H, I)) / 11).astype(np.float32))
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32) + 0.1
    y = M8.moe_forward_f8b(xc, xs, idx, w, lambda e: ex, 7.0, E)
    w1d, w2d = ex.decoded()
    o, _, _ = M8.expert_mlp_f8b(M8.dequantize_f8b(xc, xs, 1), w1d, w2d, 7.0)
    want = F.bf16_round(o * w.astype(np.float64).sum(axis=1, keepdims=True))
    ulp = np.ldexp(1.0, np.frexp(np.abs(want))[1] - 8)
    assert np.all(np.abs(y - want) <= ulp + 1e-300)
    assert np.mean(y == want) > 0.99


def test_token_order_invariance_and_empty_slots():
    rng = np.random.default_rng(45)
    T, H, I, E, k = 16, 128, 128, 4, 2
    x = rng.standard_normal((T, H)).astype(np.float32)
    xc, xs = M8.quantize_tokens_f8b(x)
    exs = [M8.quantize_expert_f8b((rng.standard_normal((2 * I, H)) / 11).astype(np.float32),
                                  (rng.standard_normal((H, I)) / 11).astype(np.float32)) for _ in range(E)]
    idx = rng.integers(0, E, (T, k)).astype(np.int32)
    idx[3, :] = -1
    w = rng.random((T, k)).astype(np.float32)
    y = M8.moe_forward_f8b(xc, xs, idx, w, lambda e: exs[e], 7.0, E)
    assert np.all(y[3] == 0)
    p = rng.permutation(T)
    y2 = M8.moe_forward_f8b(xc[p], xs[p], idx[p], w[p], lambda e: exs[e], 7.0, E)
    assert np.array_equal(y2, y[p])
    c, o, _, _ = route(idx, E)
    assert c.sum() == (idx >= 0).sum()


def test_planted_reciprocal_rule_is_caught():
    """Multiplying by 448 / a instead of dividing by the fp32 scale a / 448
    moves about one code in five million; on this block (one value and the
    block's largest magnitude, fp32 bit patterns) the two rules give
    neighbouring codes, and the brute-force rule sides with the oracle."""
    v = np.zeros((1, 128), np.float32)
    v[0, 0] = np.uint32(0xBE8E2114).view(np.float32)
    v[0, 1] = np.uint32(0x3F093A6B).view(np.float32)          # the block's largest magnitude
    codes, s = M8.quantize_f8b(v, 1)
    amax = np.float32(v[0, 1])
    alt = F.encode((v * (np.float32(448.0) / amax)).astype(np.float32).astype(np.float64), F.E4M3)
    assert alt[0, 0] != codes[0, 0]
    _, ev = _exact_block(v[0])
    assert Fraction(float(F.decode(codes[:, :1], F.E4M3)[0, 0]) * Fraction(float(s[0, 0]))) == ev[0]
    assert Fraction(float(F.decode(alt[:, :1], F.E4M3)[0, 0]) * Fraction(float(s[0, 0]))) != ev[0]
