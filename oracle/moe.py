"""The fused MoE expert layer, plain and in fp64.

What the layer computes (single GPU; the cross-rank dispatch/combine of the
DeepGEMM kernel is not part of it):

1. decode every input byte exactly (``formats``);
2. route the assignments (``routing``);
3. for each assignment (t, j) with expert e = topk_idx[t, j]:
   a1 = x[t] . W1[e]^T                      (L1 gate/up GEMM, fp64 sums)
   g = a1[:I], u = a1[I:]                   (gate rows first, then up rows)
   if a clamp L applies:  g = min(g, L);  u = min(max(u, -L), L)
   h = g / (1 + exp(-g)) * u                (SwiGLU)
   h -> E4M3 + UE8M0 per 32 (rule Q), decoded again
   o = h . W2[e]^T                          (L2 down GEMM, fp64 sums)
4. y[t] = bf16_RNE( sum over j ascending of topk_w[t, j] * o_(t,j) ).

Sources: the fused FP8 x FP4 MegaMoE call on the digest page of sglang PR
#36657 (section 关键源码片段): it takes the output, both layers' weights and
a shared buffer, the per-32 (1, 1, 32) recipe, SwiGLU with an optional
activation clamp, and keeps the first num_tokens output rows; the buffer views x,
x_sf, topk_idx, topk_weights, l1_acts, l1_acts_sf, l2_acts, l2_acts_sf
(DeepGEMM SM90 MegaMoE dev log, Phase 1 entry); the dispatch/combine
ordering (same log, Phase 2 entry; DeepGEMM PR #451 "Reset MegaMoE combine
readiness for CUDA graph replay").  The pages do not define the clamp form,
the gate/up order, or where topk_weights is applied; the readings taken here
are: one-sided clamp on the gate, two-sided on the up projection; gate rows
[0, I) then up rows [I, 2I); the weight is applied to the L2 output in the
combine.  A clamp applies iff it is finite and > 0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import formats as F
from .routing import route


def clamp_applies(clamp) -> bool:
    return clamp is not None and math.isfinite(clamp) and clamp > 0


@dataclass
class ExpertWeights:
    """Quantised weights of one expert in the layer's canonical layouts."""
    w1: np.ndarray      # uint8 [2I, H/2]  E2M1 packed, element 2c in the low nibble
    w1_sf: np.ndarray   # uint8 [2I, H/32] UE8M0
    w2: np.ndarray      # uint8 [H, I/2]
    w2_sf: np.ndarray   # uint8 [H, I/32]

    def decoded(self):
        w1 = F.dequantize(F.unpack_e2m1(self.w1), self.w1_sf, F.E2M1)
        w2 = F.dequantize(F.unpack_e2m1(self.w2), self.w2_sf, F.E2M1)
        return w1, w2


def swiglu(a1: np.ndarray, I: int, clamp) -> np.ndarray:
    g = a1[..., :I]
    u = a1[..., I:]
    if clamp_applies(clamp):
        L = float(clamp)
        g = np.minimum(g, L)
        u = np.minimum(np.maximum(u, -L), L)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def expert_mlp(xd: np.ndarray, w1d: np.ndarray, w2d: np.ndarray, clamp):
    """One expert on decoded rows xd [n, H]: returns (o [n, H] fp64,
    l1 codes uint8 [n, I], l1 sf uint8 [n, I/32])."""
    I = w1d.shape[0] // 2
    a1 = xd @ w1d.T
    h = swiglu(a1, I, clamp)
    codes, sf = F.quantize_mx(h, F.E4M3)
    hd = F.dequantize(codes, sf, F.E4M3)
    return hd @ w2d.T, codes, sf


def moe_forward(x, x_sf, topk_idx, topk_w, expert, clamp, E: int, tokens=None,
                want_intermediates: bool = False):
    """The layer.

    x        uint8 [T, H]     E4M3 codes;   x_sf uint8 [T, H/32]
    topk_idx int   [T, k]     expert ids, -1 = empty slot
    topk_w   f32   [T, k]
    expert   callable e -> ExpertWeights
    tokens   optional sorted token ids: compute only these rows of y
    Returns y as fp64 values that are exactly bf16 (rows of ``tokens`` if
    given), plus a dict of intermediates if asked.
    """
    x = np.asarray(x, dtype=np.uint8)
    topk_idx = np.asarray(topk_idx)
    T, k = topk_idx.shape
    H = x.shape[1] if x.ndim == 2 else 0
    counts, offsets, perm, inv = route(topk_idx, E)
    if tokens is None:
        tokens = np.arange(T, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    want = np.zeros(T, dtype=bool)
    want[tokens] = True

    contrib = {}                  # flat index -> fp64 [H] weighted expert output
    l1 = {}
    w_flat = np.asarray(topk_w, dtype=np.float64).reshape(-1)
    for e in range(E):
        flats = perm[offsets[e]:offsets[e + 1]]
        flats = flats[want[flats // k]]
        if len(flats) == 0:
            continue
        rows = flats // k
        xd = F.dequantize(x[rows], x_sf[rows], F.E4M3)
        w1d, w2d = expert(e).decoded()
        o, codes, sf = expert_mlp(xd, w1d, w2d, clamp)
        for n, f in enumerate(flats):
            contrib[int(f)] = w_flat[f] * o[n]
            if want_intermediates:
                l1[int(f)] = (codes[n], sf[n])

    y = np.zeros((len(tokens), H), dtype=np.float64)
    for r, t in enumerate(tokens):
        acc = np.zeros(H, dtype=np.float64)
        for j in range(k):
            f = int(t) * k + j
            if f in contrib:
                acc = acc + contrib[f]
        y[r] = F.bf16_round(acc)
    if want_intermediates:
        return y, {"counts": counts, "offsets": offsets, "perm": perm, "inv": inv,
                   "contrib": contrib, "l1": l1}
    return y


def quantize_expert(w1_f32: np.ndarray, w2_f32: np.ndarray) -> ExpertWeights:
    """fp32 weights of one expert -> E2M1 + UE8M0/32 (rule Q), packed."""
    c1, s1 = F.quantize_mx(w1_f32, F.E2M1)
    c2, s2 = F.quantize_mx(w2_f32, F.E2M1)
    return ExpertWeights(F.pack_e2m1(c1), s1, F.pack_e2m1(c2), s2)


def quantize_tokens(x_f32: np.ndarray):
    """fp32 activations -> E4M3 codes + UE8M0/32 (rule Q)."""
    return F.quantize_mx(x_f32, F.E4M3)
