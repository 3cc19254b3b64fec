"""Pins for oracle.moe_bf16 (the bf16 x bf16 layer):

* brute force: a pure-Python loop over tokens, slots, features and sums
  (math.exp, no numpy) on tiny random layers;
* closed forms of SwiGLU: a gate at 0 gives 0; a large gate passes u through
  (silu(g) = g to fp64 precision); a clamped gate and up give the known value
  7 * 7 / (1 + e^-7), rounded to bf16;
* exact invariances: doubling topk_w doubles y; relabelling the experts, or
  permuting the tokens, permutes nothing else;
* special cases: empty slots and tokens routed nowhere give zero rows.
A planted mistake (no bf16 rounding of the L1 activations, or the gate and up
halves swapped) is caught.
"""
import math

import numpy as np
import pytest

from oracle import formats as F
from oracle import moe_bf16 as MB


def _bf(a):
    return F.bf16_round(np.asarray(a, dtype=np.float64))


def _rand(rng, T, H, I, E, k, empty_frac=0.0):
    x = _bf(rng.standard_normal((T, H)))
    experts = [(_bf(rng.standard_normal((2 * I, H)) / math.sqrt(H)), _bf(rng.standard_normal((H, I)) / math.sqrt(I)))
               for _ in range(E)]
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    if empty_frac:
        idx[rng.random(idx.shape) < empty_frac] = -1
    w = (rng.random((T, k)) + 0.05).astype(np.float32)
    return x, idx, w, experts


def _bf_scalar(v: float) -> float:
    return float(F.bf16_round(np.float64(v)))


def _brute(x, idx, w, experts, clamp):
    """Pure-Python restatement: loops and math.exp only."""
    T, k = idx.shape
    H = len(x[0])
    y = []
    for t in range(T):
        acc = [0.0] * H
        for j in range(k):
            e = int(idx[t][j])
            if e < 0:
                continue
            w1, w2 = experts[e]
            I = len(w1) // 2
            h = []
            for i in range(I):
                g = sum(float(x[t][c]) * float(w1[i][c]) for c in range(H))
                u = sum(float(x[t][c]) * float(w1[I + i][c]) for c in range(H))
                if clamp is not None and clamp > 0:
                    g = min(g, clamp)
                    u = min(max(u, -clamp), clamp)
                h.append(_bf_scalar(g / (1.0 + math.exp(-g)) * u))
            for o in range(H):
                acc[o] += float(w[t][j]) * sum(h[i] * float(w2[o][i]) for i in range(I))
        y.append([_bf_scalar(a) for a in acc])
    return np.array(y)


@pytest.mark.parametrize("seed,clamp,empty", [(0, 7.0, 0.0), (1, 0.0, 0.3), (2, 1.5, 0.1)])
def test_brute_force(seed, clamp, empty):
    rng = np.random.default_rng(seed)
    x, idx, w, experts = _rand(rng, T=5, H=12, I=6, E=4, k=2, empty_frac=empty)
    y = MB.moe_forward_bf16(x, idx, w, lambda e: experts[e], clamp, 4)
    ref = _brute(x, idx, w, experts, clamp)
    # different fp64 summation orders can move a bf16 rounding by one step at a tie
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(ref), 1e-30))[1] - 8)
    assert np.all(np.abs(y - ref) <= ulp)
    assert np.mean(y == ref) >= 0.95


def _one_feature_layer(g_in, u_in, w, clamp):
    """E = 1, k = 1, I = 1, H = 2: the gate row picks x[0], the up row x[1],
    and W2 sends h to output 0 only."""
    x = np.array([[g_in, u_in]], dtype=np.float64)
    w1 = np.array([[1.0, 0.0], [0.0, 1.0]])
    w2 = np.array([[1.0], [0.0]])
    return MB.moe_forward_bf16(x, np.array([[0]]), np.array([[w]], np.float32), lambda e: (w1, w2), clamp, 1)


def test_closed_forms_of_swiglu():
    # silu(0) = 0
    assert np.all(_one_feature_layer(0.0, 3.0, 1.0, None) == 0.0)
    # silu(g) = g for g = 48 (e^-48 is far below fp64 resolution): h = 48 * 0.5 = 24, y = 0.25 * 24
    y = _one_feature_layer(48.0, 0.5, 0.25, None)
    assert y[0, 0] == 6.0 and y[0, 1] == 0.0
    # clamp 7 on gate and up: h = bf16(7 * 7 / (1 + e^-7)) = bf16(48.955...) = 49 (bf16 step 0.25 in [32, 64))
    y = _one_feature_layer(48.0, 10.0, 1.0, 7.0)
    assert y[0, 0] == 49.0
    # a clamp that is off (0) leaves the product: h = bf16(48 * 10) = 480
    assert _one_feature_layer(48.0, 10.0, 1.0, 0.0)[0, 0] == 480.0


def test_doubling_weights_doubles_output():
    rng = np.random.default_rng(3)
    x, idx, w, experts = _rand(rng, T=6, H=16, I=8, E=5, k=3)
    y1 = MB.moe_forward_bf16(x, idx, w, lambda e: experts[e], 7.0, 5)
    y2 = MB.moe_forward_bf16(x, idx, (2 * w).astype(np.float32), lambda e: experts[e], 7.0, 5)
    assert np.array_equal(y2, 2 * y1)


def test_relabelling_experts_and_permuting_tokens():
    rng = np.random.default_rng(4)
    x, idx, w, experts = _rand(rng, T=7, H=16, I=8, E=5, k=2)
    y = MB.moe_forward_bf16(x, idx, w, lambda e: experts[e], 7.0, 5)
    relabel = rng.permutation(5)
    inv = np.argsort(relabel)
    y_r = MB.moe_forward_bf16(x, relabel[idx], w, lambda e: experts[inv[e]], 7.0, 5)
    assert np.array_equal(y, y_r)
    order = rng.permutation(7)
    y_p = MB.moe_forward_bf16(x[order], idx[order], w[order], lambda e: experts[e], 7.0, 5)
    assert np.array_equal(y_p, y[order])


def test_empty_rows_are_zero():
    rng = np.random.default_rng(5)
    x, idx, w, experts = _rand(rng, T=4, H=8, I=4, E=3, k=2)
    idx[2, :] = -1
    y = MB.moe_forward_bf16(x, idx, w, lambda e: experts[e], 7.0, 3)
    assert np.all(y[2] == 0)


def test_planted_mistakes_are_caught(monkeypatch):
    rng = np.random.default_rng(0)
    x, idx, w, experts = _rand(rng, T=5, H=12, I=6, E=4, k=2)
    ref = _brute(x, idx, w, experts, 7.0)

    def no_rounding(xd, w1d, w2d, clamp):
        I = w1d.shape[0] // 2
        h = MB.swiglu(xd @ w1d.T, I, clamp)
        return h @ w2d.T, h

    def swapped(xd, w1d, w2d, clamp):
        I = w1d.shape[0] // 2
        a1 = xd @ w1d.T
        h = F.bf16_round(MB.swiglu(np.concatenate([a1[:, I:], a1[:, :I]], axis=1), I, clamp))
        return h @ w2d.T, h

    for bad in (no_rounding, swapped):
        monkeypatch.setattr(MB, "expert_mlp_bf16", bad)
        y = MB.moe_forward_bf16(x, idx, w, lambda e: experts[e], 7.0, 4)
        assert not np.array_equal(y, ref)
        monkeypatch.undo()
