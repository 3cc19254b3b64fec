"""The bf16 x bf16 variant of the fused MoE expert layer, plain and in fp64.

Test infrastructure: only the tests, the package's smoke check and the
benchmark's CPU-baseline leg use this module; the library never does.

The pages name a second MegaMoE kernel beside the FP8 x FP4 one, the BF16
MegaMoE (DeepGEMM PR #451, "Reset MegaMoE combine readiness for CUDA graph
replay": the fix and its review cover both the FP8/FP4 and the BF16 kernel,
with the same dispatch, readiness and combine protocol), but not its
arithmetic.  The reading taken here is the FP8 x FP4 layer (``moe.py``) with
every quantisation step replaced by bfloat16:

1. x [T, H], W1 [E, 2I, H] and W2 [E, H, I] hold bfloat16 values;
2. route the assignments (``routing``);
3. for each assignment (t, j) with expert e = topk_idx[t, j]:
   a1 = x[t] . W1[e]^T                      (fp64 sums)
   g = a1[:I], u = a1[I:];  the clamp and SwiGLU of ``moe.swiglu``
   h -> bfloat16, round to nearest even     (the L1 activations are bf16)
   o = h . W2[e]^T                          (fp64 sums)
4. y[t] = bf16_RNE( sum over j ascending of topk_w[t, j] * o_(t,j) ).
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from .moe import swiglu
from .routing import route


def expert_mlp_bf16(xd: np.ndarray, w1d: np.ndarray, w2d: np.ndarray, clamp):
    """One expert on rows xd [n, H] (bf16 values): returns (o [n, H] fp64,
    the bf16 L1 activations [n, I] as fp64)."""
    I = w1d.shape[0] // 2
    a1 = xd @ w1d.T
    h = F.bf16_round(swiglu(a1, I, clamp))
    return h @ w2d.T, h


def moe_forward_bf16(x, topk_idx, topk_w, expert, clamp, E: int, tokens=None, want_intermediates: bool = False):
    """The bf16 layer.

    x        fp64 [T, H]  bfloat16 values
    topk_idx int  [T, k]  expert ids, -1 = empty slot
    topk_w   f32  [T, k]
    expert   callable e -> (W1 [2I, H], W2 [H, I]) as fp64 arrays of bfloat16 values
    tokens   optional sorted token ids: compute only these rows of y
    Returns y as fp64 values that are exactly bf16, plus intermediates if asked.
    """
    x = np.asarray(x, dtype=np.float64)
    topk_idx = np.asarray(topk_idx)
    T, k = topk_idx.shape
    H = x.shape[1] if x.ndim == 2 else 0
    counts, offsets, perm, inv = route(topk_idx, E)
    if tokens is None:
        tokens = np.arange(T, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    want = np.zeros(T, dtype=bool)
    want[tokens] = True

    contrib = {}
    l1 = {}
    w_flat = np.asarray(topk_w, dtype=np.float64).reshape(-1)
    for e in range(E):
        flats = perm[offsets[e]:offsets[e + 1]]
        flats = flats[want[flats // k]]
        if len(flats) == 0:
            continue
        w1d, w2d = expert(e)
        o, h = expert_mlp_bf16(x[flats // k], w1d, w2d, clamp)
        for n, f in enumerate(flats):
            contrib[int(f)] = w_flat[f] * o[n]
            if want_intermediates:
                l1[int(f)] = h[n]

    y = np.zeros((len(tokens), H), dtype=np.float64)
    for r, t in enumerate(tokens):
        acc = np.zeros(H, dtype=np.float64)
        for j in range(k):
            f = int(t) * k + j
            if f in contrib:
                acc = acc + contrib[f]
        y[r] = F.bf16_round(acc)
    if want_intermediates:
        return y, {"counts": counts, "offsets": offsets, "perm": perm, "inv": inv, "contrib": contrib, "l1": l1}
    return y
