"""The fused expert layer in the (1, 128, 128) recipe, plain and in fp64.

Test infrastructure: only tests/, the smoke check and the benchmark's CPU
baseline use this module; the product never does.

Source: DeepGEMM fork, "SM90 MegaMoE 开发日志", Phase 1 entry -- on SM90 the
Python wrapper of the MegaMoE call takes the (1, 128, 128) recipe with float
scale factors (the SM100 call of the same pages uses recipe (1, 1, 32) with
UE8M0 scales, oracle.moe).  The recipe's three numbers are the block shapes of
its scales: activations carry one fp32 scale per token and 128 consecutive
elements along K, weights one fp32 scale per block of 128 rows x 128 columns,
and the L1 activations between the two GEMMs are requantised like the
activations (one scale per token and 128 features).  Elements are FP8 E4M3.

The pages give none of the arithmetic.  Readings taken here:
* scale of a block with largest magnitude a: s = a / 448 rounded to fp32
  (round to nearest); an all-zero block takes s = 1;
* element code: RNE into E4M3 of the fp32 quotient v / s (an IEEE fp32
  division), saturating at 448;
* the quantisation decision is taken in fp32: the values are rounded to fp32
  first (the inputs are fp32 already; the fp64 L1 activations of this oracle
  are rounded to fp32 before they are requantised, the precision in which the
  GPU holds them);
* everything else as in oracle.moe: exact decoding, fp64 sums, the clamp and
  SwiGLU, the top-k weight applied to the L2 output, one bf16 rounding of the
  fp64 sum over the token's slots in ascending order.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import formats as F
from .moe import swiglu
from .routing import route

BLOCK = 128
E4M3_MAX = 448.0


def block_scales(v32: np.ndarray, block_rows: int) -> np.ndarray:
    """fp32 scales of the blocks of block_rows x 128 of an fp32 matrix."""
    R, C = v32.shape
    if C % BLOCK or R % block_rows:
        raise ValueError("the matrix must split into blocks of block_rows x 128")
    blocks = np.abs(v32).reshape(R // block_rows, block_rows, C // BLOCK, BLOCK)
    amax = blocks.max(axis=(1, 3)) if R and C else np.zeros((R // block_rows, C // BLOCK), np.float32)
    amax = amax.astype(np.float32)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(amax == 0, np.float32(1.0), s).astype(np.float32)


def quantize_f8b(v, block_rows: int):
    """Matrix v [R, C] -> (E4M3 codes uint8 [R, C], fp32 scales
    [R / block_rows, C / 128]).  block_rows = 1 for activations, 128 for
    weights."""
    v32 = np.asarray(v, dtype=np.float32)
    if not np.all(np.isfinite(v32)):
        raise ValueError("quantize_f8b: non-finite input")
    s = block_scales(v32, block_rows)
    R, C = v32.shape
    s_full = np.repeat(np.repeat(s, block_rows, axis=0), BLOCK, axis=1)
    q = (v32 / s_full).astype(np.float32)          # IEEE fp32 division
    return F.encode(q.astype(np.float64), F.E4M3), s


def dequantize_f8b(codes, scales, block_rows: int) -> np.ndarray:
    """E4M3 codes [R, C] and fp32 block scales -> fp64 values (exact)."""
    v = F.decode(np.asarray(codes, np.uint8), F.E4M3)
    s = np.asarray(scales, np.float64)
    return v * np.repeat(np.repeat(s, block_rows, axis=0), BLOCK, axis=1)


@dataclass
class ExpertWeightsF8B:
    """One expert's weights: E4M3 codes and fp32 scales per 128 x 128 block."""
    w1: np.ndarray      # uint8 [2I, H]
    w1_s: np.ndarray    # f32 [2I/128, H/128]
    w2: np.ndarray      # uint8 [H, I]
    w2_s: np.ndarray    # f32 [H/128, I/128]

    def decoded(self):
        return dequantize_f8b(self.w1, self.w1_s, BLOCK), dequantize_f8b(self.w2, self.w2_s, BLOCK)


def quantize_expert_f8b(w1_f32, w2_f32) -> ExpertWeightsF8B:
    c1, s1 = quantize_f8b(w1_f32, BLOCK)
    c2, s2 = quantize_f8b(w2_f32, BLOCK)
    return ExpertWeightsF8B(c1, s1, c2, s2)


def quantize_tokens_f8b(x_f32):
    """fp32 activations [T, H] -> E4M3 codes + fp32 scales [T, H/128]."""
    return quantize_f8b(x_f32, 1)


def expert_mlp_f8b(xd: np.ndarray, w1d: np.ndarray, w2d: np.ndarray, clamp):
    """One expert on decoded rows xd [n, H]: returns (o [n, H] fp64, L1 codes
    uint8 [n, I], L1 scales f32 [n, I/128])."""
    I = w1d.shape[0] // 2
    a1 = xd @ w1d.T
    h = swiglu(a1, I, clamp)
    codes, s = quantize_f8b(h.astype(np.float32), 1)
    hd = dequantize_f8b(codes, s, 1)
    return hd @ w2d.T, codes, s


def moe_forward_f8b(x, x_s, topk_idx, topk_w, expert, clamp, E: int, tokens=None,
                    want_intermediates: bool = False):
    """The layer.

    x        uint8 [T, H]     E4M3 codes;   x_s f32 [T, H/128]
    topk_idx int   [T, k]     expert ids, -1 = empty slot
    topk_w   f32   [T, k]
    expert   callable e -> ExpertWeightsF8B
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

    contrib = {}
    l1 = {}
    w_flat = np.asarray(topk_w, dtype=np.float64).reshape(-1)
    for e in range(E):
        flats = perm[offsets[e]:offsets[e + 1]]
        flats = flats[want[flats // k]]
        if len(flats) == 0:
            continue
        rows = flats // k
        xd = dequantize_f8b(x[rows], np.asarray(x_s)[rows], 1)
        w1d, w2d = expert(e).decoded()
        o, codes, s = expert_mlp_f8b(xd, w1d, w2d, clamp)
        for n, f in enumerate(flats):
            contrib[int(f)] = w_flat[f] * o[n]
            if want_intermediates:
                l1[int(f)] = (codes[n], s[n])

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
