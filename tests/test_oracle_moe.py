"""Pins for oracle.routing and oracle.moe.

* routing against a brute-force Python loop;
* the 1-token / 1-expert layer against an independent scalar computation in
  exact rational arithmetic (Fraction), except for exp();
* fp64 accumulation against exact sums;
* the closed form when every expert holds the same weights;
* invariance to token order and to relabelling the experts;
* special cases: no tokens, empty experts, all-empty rows, clamp that never
  binds, k = 1 with w = 1 (a dense MLP);
* planted mistakes in the oracle are caught by these pins.
"""
from fractions import Fraction
import math

import numpy as np
import pytest

from oracle import formats as F
from oracle import moe as M
from oracle.routing import route


# ------------------------------------------------------------------ helpers
def _rand_layer(rng, T, H, I, E, k, empty_frac=0.0, scale_x=1.0):
    x = rng.standard_normal((T, H)) * scale_x
    xc, xsf = F.quantize_mx(x, F.E4M3)
    experts = []
    for _ in range(E):
        w1 = rng.standard_normal((2 * I, H)) / math.sqrt(H)
        w2 = rng.standard_normal((H, I)) / math.sqrt(I)
        experts.append(M.quantize_expert(w1, w2))
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else \
        np.zeros((0, k), np.int32)
    if empty_frac:
        idx[rng.random(idx.shape) < empty_frac] = -1
    w = rng.random((T, k)).astype(np.float32) + 0.05
    w /= w.sum(axis=1, keepdims=True)
    return xc, xsf, idx, w.astype(np.float32), experts


# ------------------------------------------------------------------ routing
def _route_brute(idx, E):
    flat = [int(v) for v in np.asarray(idx).reshape(-1)]
    counts = [0] * E
    for v in flat:
        if v >= 0:
            counts[v] += 1
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    fill = list(offsets[:-1])
    perm = [0] * offsets[-1]
    inv = [-1] * len(flat)
    for f, v in enumerate(flat):          # ascending flat order -> stable
        if v >= 0:
            perm[fill[v]] = f
            inv[f] = fill[v]
            fill[v] += 1
    return counts, offsets, perm, inv


@pytest.mark.parametrize("T,E,k,empty", [(0, 4, 2, 0.0), (1, 1, 1, 0.0), (37, 5, 3, 0.2),
                                         (200, 16, 4, 0.05), (64, 8, 8, 0.0)])
def test_route_vs_brute_force(T, E, k, empty):
    rng = np.random.default_rng(T * 7 + E)
    idx = rng.integers(0, E, (T, k)).astype(np.int32)     # duplicates allowed
    idx[rng.random((T, k)) < empty] = -1
    counts, offsets, perm, inv = route(idx, E)
    bc, bo, bp, bi = _route_brute(idx, E)
    assert counts.tolist() == bc
    assert offsets.tolist() == bo
    assert perm.tolist() == bp
    assert inv.tolist() == bi


def test_route_bad_index_raises():
    with pytest.raises(ValueError):
        route(np.array([[0, 4]]), 4)
    with pytest.raises(ValueError):
        route(np.array([[-2, 0]]), 4)


# ------------------------------------------------- 1 token, 1 expert, exact
def _exact_e4m3(code):
    s = -1 if code & 0x80 else 1
    e, m = (code >> 3) & 15, code & 7
    if e == 0:
        return s * Fraction(m, 512)
    return s * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


_E2M1_LIT = [Fraction(v) for v in ("0", "1/2", "1", "3/2", "2", "3", "4", "6")]


def _exact_e2m1(code):
    return (-1 if code & 8 else 1) * _E2M1_LIT[code & 7]


def _exact_quant_e4m3(vals):
    """Rule Q on 32 values by exhaustive search (exact)."""
    a = max(abs(v) for v in vals)
    if a == 0:
        s = 0
    else:
        s = next(s for s in range(-127, 128) if a <= 448 * Fraction(2) ** s)
    grid = sorted({abs(_exact_e4m3(c)) for c in range(127)})
    out = []
    for v in vals:
        q = abs(v) / Fraction(2) ** s
        best = min(grid, key=lambda g: (abs(g - q), 0))
        ties = [g for g in grid if abs(g - q) == abs(best - q)]
        if len(ties) == 2:   # tie: even mantissa = even code
            codes = {abs(_exact_e4m3(c)): c for c in range(127)}
            best = ties[0] if codes[ties[0]] % 2 == 0 else ties[1]
        out.append((best if v >= 0 else -best) * Fraction(2) ** s)
    return out


def _bf16_exact(x: Fraction) -> float:
    if x == 0:
        return 0.0
    ax = abs(x)
    e = 0
    while Fraction(2) ** e > ax:
        e -= 1
    while Fraction(2) ** (e + 1) <= ax:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 7)
    q = ax / ulp
    n = math.floor(q)
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2):
        n += 1
    return math.copysign(float(n * ulp), x)


def _exact_layer_one_token(xc, xsf, w, ex: M.ExpertWeights, clamp, H, I):
    """Scalar, independent computation of y for k = 1, E = 1."""
    xs = [_exact_e4m3(int(xc[0, h])) * Fraction(2) ** (int(xsf[0, h // 32]) - 127) for h in range(H)]
    w1c = F.unpack_e2m1(ex.w1)
    w2c = F.unpack_e2m1(ex.w2)
    W1 = [[_exact_e2m1(int(w1c[n, h])) * Fraction(2) ** (int(ex.w1_sf[n, h // 32]) - 127)
           for h in range(H)] for n in range(2 * I)]
    W2 = [[_exact_e2m1(int(w2c[n, i])) * Fraction(2) ** (int(ex.w2_sf[n, i // 32]) - 127)
           for i in range(I)] for n in range(H)]
    a1 = [sum(xs[h] * W1[n][h] for h in range(H)) for n in range(2 * I)]
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
    hq = []
    for b in range(I // 32):
        hq += _exact_quant_e4m3(hv[32 * b:32 * b + 32])
    o = [sum(hq[i] * W2[n][i] for i in range(I)) for n in range(H)]
    wf = Fraction(float(w[0, 0]))
    return np.array([_bf16_exact(wf * o[n]) for n in range(H)])


@pytest.mark.parametrize("clamp", [7.0, 0.0, 0.05])
def test_one_token_one_expert_exact(clamp):
    rng = np.random.default_rng(11)
    H, I = 64, 32
    xc, xsf, _, _, experts = _rand_layer(rng, 1, H, I, 1, 1)
    idx = np.zeros((1, 1), np.int32)
    w = np.ones((1, 1), np.float32)
    y = M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], clamp, 1)
    want = _exact_layer_one_token(xc, xsf, w, experts[0], clamp, H, I)
    assert np.array_equal(y[0], want)


def test_fp64_accumulation_is_exact_enough():
    """Each product of two decoded values is exact in fp64; the fp64 sum of
    H of them is within a few ulp of the exact rational sum."""
    rng = np.random.default_rng(12)
    H, I = 256, 32
    xc, xsf, _, _, experts = _rand_layer(rng, 2, H, I, 1, 1)
    xd = F.dequantize(xc, xsf, F.E4M3)
    w1d, _ = experts[0].decoded()
    a1 = xd @ w1d.T
    for t in range(2):
        for n in range(0, 2 * I, 7):
            exact = sum(Fraction(float(xd[t, h])) * Fraction(float(w1d[n, h])) for h in range(H))
            assert abs(Fraction(float(a1[t, n])) - exact) <= abs(exact) * Fraction(1, 10 ** 13) + Fraction(1, 10 ** 30)


# ------------------------------------------------------------------ closed form
def test_identical_experts_closed_form():
    rng = np.random.default_rng(13)
    T, H, I, E, k = 24, 128, 64, 6, 3
    xc, xsf, idx, w, experts = _rand_layer(rng, T, H, I, E, k)
    ex = experts[0]
    y = M.moe_forward(xc, xsf, idx, w, lambda e: ex, 7.0, E)
    # dense MLP per token, then times the sum of its weights
    xd = F.dequantize(xc, xsf, F.E4M3)
    w1d, w2d = ex.decoded()
    o, _, _ = M.expert_mlp(xd, w1d, w2d, 7.0)
    want = F.bf16_round(o * w.astype(np.float64).sum(axis=1, keepdims=True))
    ulp = np.ldexp(1.0, np.frexp(np.abs(want))[1] - 8)
    diff = np.abs(y - want)
    assert np.all(diff <= ulp + 1e-300)              # at most one bf16 step (sum order)
    assert np.mean(diff == 0) > 0.99


def test_dense_mlp_when_k1_w1():
    rng = np.random.default_rng(14)
    T, H, I, E = 10, 96, 64, 3
    xc, xsf, _, _, experts = _rand_layer(rng, T, H, I, E, 1)
    idx = rng.integers(0, E, (T, 1)).astype(np.int32)
    w = np.ones((T, 1), np.float32)
    y = M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], 7.0, E)
    xd = F.dequantize(xc, xsf, F.E4M3)
    for t in range(T):
        w1d, w2d = experts[idx[t, 0]].decoded()
        o, _, _ = M.expert_mlp(xd[t:t + 1], w1d, w2d, 7.0)
        assert np.array_equal(y[t], F.bf16_round(o[0]))


# ------------------------------------------------------------------ invariances
def test_token_permutation_invariance():
    rng = np.random.default_rng(15)
    T, H, I, E, k = 30, 64, 32, 5, 2
    xc, xsf, idx, w, experts = _rand_layer(rng, T, H, I, E, k, empty_frac=0.1)
    y = M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], 7.0, E)
    p = rng.permutation(T)
    y2 = M.moe_forward(xc[p], xsf[p], idx[p], w[p], lambda e: experts[e], 7.0, E)
    assert np.array_equal(y2, y[p])
    c1, *_ = route(idx, E)
    c2, *_ = route(idx[p], E)
    assert np.array_equal(c1, c2)


def test_expert_relabel_invariance():
    rng = np.random.default_rng(16)
    T, H, I, E, k = 20, 64, 32, 6, 3
    xc, xsf, idx, w, experts = _rand_layer(rng, T, H, I, E, k, empty_frac=0.1)
    y = M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], 7.0, E)
    sigma = rng.permutation(E)                       # new label of expert e
    relab = np.where(idx >= 0, sigma[np.maximum(idx, 0)], -1).astype(np.int32)
    inv_sigma = np.argsort(sigma)
    y2 = M.moe_forward(xc, xsf, relab, w, lambda e: experts[inv_sigma[e]], 7.0, E)
    assert np.array_equal(y, y2)


# ------------------------------------------------------------------ special cases
def test_zero_tokens():
    rng = np.random.default_rng(17)
    _, _, _, _, experts = _rand_layer(rng, 1, 64, 32, 2, 1)
    y = M.moe_forward(np.zeros((0, 64), np.uint8), np.zeros((0, 2), np.uint8),
                      np.zeros((0, 2), np.int32), np.zeros((0, 2), np.float32),
                      lambda e: experts[e], 7.0, 2)
    assert y.shape == (0, 64)


def test_empty_rows_and_empty_experts():
    rng = np.random.default_rng(18)
    T, H, I, E, k = 12, 64, 32, 8, 2
    xc, xsf, idx, w, experts = _rand_layer(rng, T, H, I, E, k)
    idx[:, :] = np.where(idx % 2 == 0, idx, 0)       # odd experts get nothing
    idx[3, :] = -1                                   # token 3 routed nowhere
    calls = []

    def ex(e):
        calls.append(e)
        return experts[e]
    y = M.moe_forward(xc, xsf, idx, w, ex, 7.0, E)
    assert np.all(y[3] == 0)
    assert all(e % 2 == 0 for e in calls)
    counts, *_ = route(idx, E)
    assert np.all(counts[1::2] == 0)


def test_clamp_that_never_binds_equals_no_clamp():
    rng = np.random.default_rng(19)
    xc, xsf, idx, w, experts = _rand_layer(rng, 16, 64, 32, 4, 2)
    a = M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], 1e30, 4)
    b = M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], 0.0, 4)
    c = M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], float("inf"), 4)
    assert np.array_equal(a, b) and np.array_equal(b, c)


def test_clamp_binds_changes_output():
    rng = np.random.default_rng(20)
    xc, xsf, idx, w, experts = _rand_layer(rng, 16, 64, 32, 4, 2, scale_x=4.0)
    a = M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], 0.1, 4)
    b = M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], 0.0, 4)
    assert not np.array_equal(a, b)


def test_token_subset_matches_full():
    rng = np.random.default_rng(21)
    xc, xsf, idx, w, experts = _rand_layer(rng, 40, 64, 32, 6, 3)
    full = M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], 7.0, 6)
    sub = M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], 7.0, 6, tokens=[0, 5, 39])
    assert np.array_equal(sub, full[[0, 5, 39]])


# ------------------------------------------------------------------ planted mistakes
def test_pins_catch_planted_mistakes(monkeypatch):
    """Each planted mistake in the oracle makes one of the pins above fail."""
    rng = np.random.default_rng(11)
    H, I = 64, 32
    xc, xsf, _, _, experts = _rand_layer(rng, 1, H, I, 1, 1)
    idx = np.zeros((1, 1), np.int32)
    w = np.ones((1, 1), np.float32)
    want = _exact_layer_one_token(xc, xsf, w, experts[0], 0.05, H, I)

    def run():
        return M.moe_forward(xc, xsf, idx, w, lambda e: experts[e], 0.05, 1)[0]

    assert np.array_equal(run(), want)
    orig = M.swiglu
    # gate and up swapped
    monkeypatch.setattr(M, "swiglu", lambda a1, I_, c: orig(np.concatenate([a1[..., I_:], a1[..., :I_]], -1), I_, c))
    assert not np.array_equal(run(), want)
    monkeypatch.setattr(M, "swiglu", orig)
    # clamp dropped
    monkeypatch.setattr(M, "swiglu", lambda a1, I_, c: orig(a1, I_, 0.0))
    assert not np.array_equal(run(), want)
    monkeypatch.setattr(M, "swiglu", orig)
    # scale exponent rounded down instead of up: a one-step scale change only
    # shows when the block maximum saturates, so the rule-Q scan pin catches it
    from test_oracle_formats import _brute_scale
    orig_s = F.scale_exponent
    monkeypatch.setattr(F, "scale_exponent", lambda a, fmt: orig_s(a, fmt) - 1)
    a = np.array([0.3, 5.0, 448.0, 1e-3])
    assert [int(v) for v in F.scale_exponent(a, F.E4M3)] != [_brute_scale(v, F.E4M3) for v in a]
