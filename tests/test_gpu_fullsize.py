"""Full-size configurations, in the launch configuration bench.py times
(num_sms = 0, default reserve of two SMs).

The oracle cannot compute whole batches of this size in seconds, so:
* routing (counts, offsets, permutation, inverse) is compared in full, bit
  for bit;
* every output element is finite;
* dense per-expert parity: for four experts of each configuration (the
  hottest, the coldest non-empty one, one whose last token block is short,
  and the highest non-empty id) EVERY slot is compared with the oracle: the
  requantised L1 activations against the oracle's codes (one E4M3 step at
  most, 99% exact), and the weighted L2 row the layer kernel leaves in the
  workspace (fp32, indexed by the flat assignment) against the oracle's L2
  on those activations and against the oracle end to end;
* sampled output rows are compared with the oracle, which computes them one
  token at a time (each row depends only on its own token and its experts);
* a captured graph replayed 12 times with changed inputs equals the eager
  launch bit for bit (decode, prefill, skew; Kimi-style also with a side
  stream holding one SM), and the first replay's sampled rows match the
  oracle."""
import numpy as np
import pytest
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from oracle import formats as OF
from oracle import moe as OM
from oracle.routing import route
from helpers import blocker
from layer_inputs import (TOL_NL2, ExpertCache, GpuTokens, GpuWeights, bf16_to_np, close_enough, oracle_tokens,
                          run_layer, token_scale_rows)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample_tokens(cfg, idx):
    """Two tokens: the first one, and one routed to the most loaded expert
    (the largest N blocks and, for skewed routing, the split experts)."""
    counts = np.bincount(idx.reshape(-1)[idx.reshape(-1) >= 0], minlength=cfg.E)
    hot = int(np.argmax(counts))
    t_hot = int(np.nonzero((idx == hot).any(axis=1))[0][-1])
    return sorted({0, t_hot})


def _oracle_rows(cfg, idx, w, toks, seed=None, cache=None):
    xc, xsf = oracle_tokens(cfg, seed=seed, rows=toks)
    cache = cache or ExpertCache(cfg)
    return OM.moe_forward(xc, xsf, idx[toks], w[toks], cache, cfg.clamp, cfg.E), cache


def _check_routing(cfg, ws, idx):
    rc, c, o, p, i = mm.mm_read_routing(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, ws)
    assert rc == mm.MM_OK
    rc_, ro, rp, ri = route(idx, cfg.E)
    assert np.array_equal(c, rc_) and np.array_equal(o, ro)
    assert np.array_equal(p[: int(ro[-1])], rp) and np.array_equal(i, ri)
    return rc_, ro, rp


def _block_rows(cfg):
    """Largest token block of the kernel variant the host picks for this batch."""
    return 32 if cfg.T * cfg.k <= 16 * cfg.E else 128


def pick_experts(cfg, counts):
    """The hottest expert, the coldest non-empty one, the one whose last
    (balanced) token block is shortest among those split into several blocks,
    and the highest non-empty id."""
    nz = np.nonzero(counts)[0]
    hot = int(nz[np.argmax(counts[nz])])
    cold = int(nz[np.argmin(counts[nz])])
    m = _block_rows(cfg)
    short, best = None, None
    for e in nz:
        c = int(counts[e])
        nb = (c + m - 1) // m
        if nb < 2:
            continue
        rpb = (c + nb - 1) // nb
        last = c - (nb - 1) * rpb
        if best is None or last < best:
            short, best = int(e), last
    picked = {hot, cold, int(nz[-1])}
    if short is not None:
        picked.add(short)
    return sorted(picked)


# The weighted L2 row of one slot, recomputed in fp64 from the GPU's own L1
# activations, may differ from the GPU's fp32 row only by the rounding of the
# fp32 accumulation: at most 2^-12 of the sum of the absolute terms.
L2_FROM_GPU_CODES_REL = 2.0 ** -12


def _dense_expert_parity(cfg, ws, tok, routing):
    """Every slot of the picked experts, checked in three parts:
    1. the requantised L1 activations against the oracle's codes (one E4M3
       step at most, 99% exact: near a rounding tie the fp32 and fp64
       accumulators may round to neighbouring codes, or a block scale near a
       power of two to the neighbouring exponent);
    2. the weighted fp32 L2 rows against the oracle's L2 GEMM applied to the
       GPU's own L1 activations, which leaves only the fp32 summation
       rounding;
    3. the weighted L2 rows against the oracle end to end, by normalised L2
       error (an element-wise bound on intermediate rows would count the
       one-step code moves of part 1 many times over)."""
    counts, offsets, perm = routing
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    st_off, _ = mm.mm_workspace_region("stage", T, E, k, H, I)
    l1_off, _ = mm.mm_workspace_region("l1_acts", T, E, k, H, I)
    stage = ws[st_off:st_off + T * k * H * 4].view(torch.float32).view(T * k, H)
    l1a = ws[l1_off:l1_off + T * k * I].view(T * k, I)
    l1s = token_scale_rows(ws, cfg, "l1_acts_sf", mm.mm_layer_variant(T, E, k, H), idx=tok.idx_np)
    cache = ExpertCache(cfg)
    w_flat = tok.w_np.reshape(-1).astype(np.float64)
    report = {}
    for e in pick_experts(cfg, counts):
        slots = np.arange(offsets[e], offsets[e + 1])
        flats = perm[slots]
        rows = flats // k
        xc, xsf = oracle_tokens(cfg, rows=rows)
        w1d, w2d = cache(e).decoded()
        o, codes, sf = OM.expert_mlp(OF.dequantize(xc, xsf, OF.E4M3), w1d, w2d, cfg.clamp)
        wt = w_flat[flats][:, None]
        sl = torch.from_numpy(slots.astype(np.int64)).cuda()
        fl = torch.from_numpy(flats.astype(np.int64)).cuda()
        got = stage.index_select(0, fl).cpu().numpy().astype(np.float64)
        # 1. L1 activations
        g = OF.dequantize(l1a.index_select(0, sl).cpu().numpy(), l1s[slots], OF.E4M3)
        r = OF.dequantize(codes, sf, OF.E4M3)
        step = np.ldexp(1.0, np.frexp(np.maximum(np.abs(r), np.abs(g)))[1] - 4)   # one E4M3 step
        assert np.all(np.abs(g - r) <= step + 1e-300), (cfg.name, e)
        exact = float(np.mean(g == r))
        assert exact >= 0.99, (cfg.name, e, exact)
        # 2. L2 on the GPU's own activations
        want_g = wt * (g @ w2d.T)
        bound = L2_FROM_GPU_CODES_REL * (np.abs(wt) * (np.abs(g) @ np.abs(w2d).T)) + 1e-30
        worst = float(np.max(np.abs(got - want_g) / bound))
        assert worst <= 1.0, (cfg.name, e, worst)
        # 3. end to end
        want = wt * o
        den = np.linalg.norm(want)
        nl2 = float(np.linalg.norm(got - want) / den) if den > 0 else float(np.linalg.norm(got))
        assert nl2 <= TOL_NL2, (cfg.name, e, len(slots), nl2)
        report[e] = (len(slots), exact, worst, nl2)
    return report


@pytest.mark.parametrize("name", ["decode", "prefill", "skew", "kimi"])
def test_full_size_dense_expert_parity(name):
    cfg = synth.CONFIGS[name]
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg)
    y, ws = run_layer(cfg, w, tok)
    routing = _check_routing(cfg, ws, tok.idx_np)
    yn = bf16_to_np(y)
    assert np.all(np.isfinite(yn))
    report = _dense_expert_parity(cfg, ws, tok, routing)
    print(f"dense parity {name}: " + ", ".join(f"e{e}: {n} slots, L1 exact {ex:.6f}, L2 worst/bound {wb:.2e}, "
                                                f"nl2 {nl:.2e}" for e, (n, ex, wb, nl) in report.items()))
    assert len(report) >= 3, report
    toks = _sample_tokens(cfg, tok.idx_np)
    ref, _ = _oracle_rows(cfg, tok.idx_np, tok.w_np, toks)
    ok, nl2, mr = close_enough(yn[toks], ref)
    assert ok, (name, toks, nl2, mr)


@pytest.mark.parametrize("name", ["decode", "prefill", "skew"])
def test_full_size_graph_replays(name):
    cfg = synth.CONFIGS[name]
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg, seed=0)
    ws_g = torch.empty(mm.mm_workspace_size(T, E, k, H, I), dtype=torch.uint8, device="cuda")
    ws_e = torch.empty_like(ws_g)
    y_g = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    y_e = torch.empty_like(y_g)

    def fwd(y, ws, stream=None):
        return mm.mm_forward(T, E, k, H, I, tok.x, tok.x_sf, tok.topk_idx, tok.topk_w, w.l1_w, w.l1_sf, w.l2_w,
                             w.l2_sf, y, cfg.clamp, 0, ws, stream=stream)

    assert fwd(y_g, ws_g) == mm.MM_OK
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        assert fwd(y_g, ws_g, torch.cuda.current_stream()) == mm.MM_OK
    torch.cuda.synchronize()
    held = None
    for r in range(1, 13):
        new = GpuTokens(cfg, seed=r)
        tok.x.copy_(new.x); tok.x_sf.copy_(new.x_sf)
        tok.topk_idx.copy_(new.topk_idx); tok.topk_w.copy_(new.topk_w)
        graph.replay()
        assert fwd(y_e, ws_e) == mm.MM_OK
        torch.cuda.current_stream().synchronize()
        assert mm.mm_get_status(ws_g)[0] == mm.MM_OK
        assert mm.mm_get_status(ws_e)[0] == mm.MM_OK
        assert torch.equal(y_g.view(torch.int16), y_e.view(torch.int16)), f"replay {r}"
        if r == 1:
            toks = _sample_tokens(cfg, new.idx_np)
            held = (y_g[toks].clone(), new.idx_np, new.w_np, toks)
    y1, idx1, w1, toks = held
    ref, _ = _oracle_rows(cfg, idx1, w1, toks, seed=1)
    ok, nl2, mr = close_enough(bf16_to_np(y1), ref)
    assert ok, (toks, nl2, mr)


def test_kimi_reserve_side_stream_and_graph_replays():
    cfg = synth.CONFIGS["kimi"]
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg, seed=0)
    ws_g = torch.empty(mm.mm_workspace_size(T, E, k, H, I), dtype=torch.uint8, device="cuda")
    ws_e = torch.empty_like(ws_g)
    y_g = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    y_e = torch.empty_like(y_g)

    def fwd(y, ws, stream=None):
        return mm.mm_forward(T, E, k, H, I, tok.x, tok.x_sf, tok.topk_idx, tok.topk_w, w.l1_w, w.l1_sf, w.l2_w,
                             w.l2_sf, y, cfg.clamp, 0, ws, stream=stream)

    prev = mm.mm_set_reserved_sms(2)
    try:
        assert fwd(y_g, ws_g) == mm.MM_OK
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            assert fwd(y_g, ws_g, torch.cuda.current_stream()) == mm.MM_OK
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        started = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert blocker().occupy_one_sm(3_000_000_000, 200 * 1024, started.data_ptr(), side.cuda_stream) == 0
        overlapped = True
        cache = ExpertCache(cfg)
        for r in range(1, 13):
            new = GpuTokens(cfg, seed=r)
            tok.x.copy_(new.x); tok.x_sf.copy_(new.x_sf)
            tok.topk_idx.copy_(new.topk_idx); tok.topk_w.copy_(new.topk_w)
            graph.replay()
            assert fwd(y_e, ws_e) == mm.MM_OK
            torch.cuda.current_stream().synchronize()
            assert mm.mm_get_status(ws_g)[0] == mm.MM_OK
            assert mm.mm_get_status(ws_e)[0] == mm.MM_OK
            assert torch.equal(y_g.view(torch.int16), y_e.view(torch.int16)), f"replay {r}"
            if r == 1:
                overlapped = not side.query()
                yn = bf16_to_np(y_g)
                assert np.all(np.isfinite(yn))
                toks = _sample_tokens(cfg, new.idx_np)
                held = (y_g[toks].clone(), new.idx_np, new.w_np, toks)
        side.synchronize()
    finally:
        mm.mm_set_reserved_sms(prev)
    assert overlapped, "the side stream finished before the first replay"
    y1, idx1, w1, toks = held
    ref, _ = _oracle_rows(cfg, idx1, w1, toks, seed=1, cache=cache)
    ok, nl2, mr = close_enough(bf16_to_np(y1), ref)
    assert ok, (toks, nl2, mr)
