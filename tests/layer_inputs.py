"""Test-side construction of the layer's inputs, on both sides.

GPU side: fp32 values from the device build of the shared generator,
quantised by the library's own kernel (mm_quantize_mx).  Oracle side: the
same fp32 values from the host build of the generator, quantised by the
oracle.  The quantiser parity test checks that both give identical bytes.
"""
from __future__ import annotations

import numpy as np
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from oracle import formats as OF
from oracle import moe as OM

# tolerance of the layer output against the oracle
TOL_NL2 = 5e-3
TOL_MAXREL = 3e-2
REL_FLOOR = 1e-2


def gpu_quantize(src: torch.Tensor, rows: int, cols: int, fmt: int, out=None, out_sf=None):
    dev = src.device
    if out is None:
        out = torch.empty(rows, cols if fmt == mm.MM_FMT_E4M3 else cols // 2, dtype=torch.uint8, device=dev)
    if out_sf is None:
        out_sf = torch.empty(rows, cols // 32, dtype=torch.uint8, device=dev)
    rc = mm.mm_quantize_mx(src, rows, cols, fmt, out, out_sf)
    assert rc == mm.MM_OK, mm.STATUS_NAMES.get(rc, rc)
    return out, out_sf


class GpuWeights:
    """Quantised expert weights; l1_sf / l2_sf hold the prepared scales that
    mm_forward takes, l1_sf_rows / l2_sf_rows the quantiser's row layout."""

    def __init__(self, cfg, device="cuda", chunk=8):
        E, H, I = cfg.E, cfg.H, cfg.I
        self.l1_w = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=device)
        self.l1_sf_rows = torch.empty(E, 2 * I, H // 32, dtype=torch.uint8, device=device)
        self.l2_w = torch.empty(E, H, I // 2, dtype=torch.uint8, device=device)
        self.l2_sf_rows = torch.empty(E, H, I // 32, dtype=torch.uint8, device=device)
        n1, n2 = 2 * I * H, H * I
        buf = torch.empty(min(chunk, E) * n1, dtype=torch.float32, device=device)
        for e0 in range(0, E, chunk):
            e1 = min(E, e0 + chunk)
            b = buf[: (e1 - e0) * n1]
            synth.normal_f32_cuda(cfg.seed, synth.TENSOR_W1, e0 * n1, b, synth.weight_scale(H))
            gpu_quantize(b, (e1 - e0) * 2 * I, H, mm.MM_FMT_E2M1, self.l1_w[e0:e1], self.l1_sf_rows[e0:e1])
            b = buf[: (e1 - e0) * n2]
            synth.normal_f32_cuda(cfg.seed, synth.TENSOR_W2, e0 * n2, b, synth.weight_scale(I))
            gpu_quantize(b, (e1 - e0) * H, I, mm.MM_FMT_E2M1, self.l2_w[e0:e1], self.l2_sf_rows[e0:e1])
        del buf
        self.l1_sf = mm.prepare_weight_scales(self.l1_sf_rows, H)
        self.l2_sf = mm.prepare_weight_scales(self.l2_sf_rows, I)
        torch.cuda.synchronize(device)


class GpuTokens:
    def __init__(self, cfg, seed=None, device="cuda", routing=None):
        T, H = cfg.T, cfg.H
        s = cfg.seed if seed is None else seed
        xf = torch.empty(max(T * H, 1), dtype=torch.float32, device=device)
        if T:
            synth.normal_f32_cuda(s, synth.TENSOR_X, 0, xf[: T * H])
        self.x = torch.empty(T, H, dtype=torch.uint8, device=device)
        self.x_sf = torch.empty(T, H // 32, dtype=torch.uint8, device=device)
        if T:
            gpu_quantize(xf[: T * H], T, H, mm.MM_FMT_E4M3, self.x, self.x_sf)
        idx, w, _ = synth.routing(cfg, s) if routing is None else routing
        self.idx_np, self.w_np = idx, w
        self.topk_idx = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to(device)
        self.topk_w = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).to(device)


def oracle_expert(cfg, e):
    return OM.quantize_expert(synth.w1_f32(cfg, e), synth.w2_f32(cfg, e))


def oracle_tokens(cfg, seed=None, rows=None):
    return OF.quantize_mx(synth.x_f32(cfg, seed, rows), OF.E4M3)


class ExpertCache:
    def __init__(self, cfg):
        self.cfg, self.cache = cfg, {}

    def __call__(self, e):
        if e not in self.cache:
            self.cache[e] = oracle_expert(self.cfg, e)
        return self.cache[e]


def run_layer(cfg, w: GpuWeights, tok: GpuTokens, num_sms=0, clamp=None, workspace=None, stream=None):
    T = cfg.T
    nbytes = mm.mm_workspace_size(max(T, 1), cfg.E, cfg.k, cfg.H, cfg.I)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=w.l1_w.device)
    y = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=w.l1_w.device)
    rc = mm.mm_forward(T, cfg.E, cfg.k, cfg.H, cfg.I, tok.x, tok.x_sf, tok.topk_idx, tok.topk_w, w.l1_w, w.l1_sf,
                       w.l2_w, w.l2_sf, y, cfg.clamp if clamp is None else clamp, num_sms, workspace,
                       stream=stream)
    assert rc == mm.MM_OK, mm.STATUS_NAMES.get(rc, rc)
    st, sm, info = mm.mm_get_status(workspace, stream)
    assert st == mm.MM_OK, (mm.STATUS_NAMES.get(st, st), sm, hex(info))
    return y, workspace


# token rows per block of each layer variant (mm_layer_variant's numbering)
BLOCK_ROWS = {0: 128, 1: 32, 2: 128, 3: 32, 4: 256}


def atom_pos(r):
    """Byte of row r (< 128) within a 512-byte scale atom (lane r % 32, word r / 32)."""
    r = np.asarray(r)
    return (r % 32) * 16 + (r // 32) * 4


def token_scale_rows(ws: torch.Tensor, cfg, which: str, variant: int, idx=None) -> np.ndarray:
    """The UE8M0 token scales a forward left in the workspace ("xs_sf": the
    dispatched x scales, K = H; "l1_acts_sf": the L1 activation scales, K = I),
    read back from their atoms into rows [n_valid, K/32] in slot order."""
    from oracle.routing import route

    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    K = H if which == "xs_sf" else I
    S = K // 128
    idx = np.asarray(cfg_routing_idx(cfg) if idx is None else idx)
    counts, offsets, _, _ = route(idx, E)
    rows_max = BLOCK_ROWS[variant]
    halves = 2 if variant == 4 else 1
    nb = -(-counts // rows_max)
    first = np.concatenate([[0], np.cumsum(nb)])
    n = int(offsets[-1])
    off, nbytes = mm.mm_workspace_region(which, max(T, 1), E, k, H, I)
    raw = ws[off:off + nbytes].cpu().numpy()
    out = np.zeros((n, K // 32), np.uint8)
    for e in range(E):
        c = int(counts[e])
        if c == 0:
            continue
        mbk = int(nb[e])
        rpb = -(-c // mbk)
        i = np.arange(c)
        mb, row = i // rpb, i % rpb
        b = first[e] + mb
        base = ((b * halves + row // 128) * S) * 512 + atom_pos(row % 128)
        for s in range(S):
            for j in range(4):
                out[offsets[e] + i, 4 * s + j] = raw[base + s * 512 + j]
    return out


def cfg_routing_idx(cfg):
    idx, _, _ = synth.routing(cfg)
    return idx


def bf16_to_np(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


def close_enough(y: np.ndarray, ref: np.ndarray):
    """(ok, normalised L2 error, max relative error over |ref| > 1e-2)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return True, 0.0, 0.0
    if not np.all(np.isfinite(y)):
        return False, float("inf"), float("inf")
    den = np.linalg.norm(ref)
    nl2 = float(np.linalg.norm(y - ref) / den) if den > 0 else float(np.linalg.norm(y))
    m = np.abs(ref) > REL_FLOOR
    mr = float(np.max(np.abs(y[m] - ref[m]) / np.abs(ref[m]))) if m.any() else 0.0
    return (nl2 <= TOL_NL2 and mr <= TOL_MAXREL), nl2, mr
