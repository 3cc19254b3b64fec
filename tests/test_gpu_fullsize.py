"""Full-size configurations, in the launch configuration bench.py times
(num_sms = 0, default reserve of two SMs).

The oracle cannot compute whole batches of this size in seconds, so:
* routing (counts, offsets, permutation, inverse) is compared in full, bit
  for bit;
* every output element is finite, and a token with no routed slot is zero;
* sampled output rows are compared with the oracle, which computes them one
  token at a time (each row depends only on its own token and its experts).
The Kimi-style case also runs with a side stream holding one SM and replays a
captured graph 12 times with changed inputs (bit-equal to eager)."""
import numpy as np
import pytest
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from oracle import formats as OF
from oracle import moe as OM
from oracle.routing import route
from helpers import blocker
from layer_inputs import (ExpertCache, GpuTokens, GpuWeights, bf16_to_np, close_enough, oracle_tokens,
                          run_layer)

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("name", ["decode", "prefill", "skew"])
def test_full_size_sampled_parity(name):
    cfg = synth.CONFIGS[name]
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg)
    y, ws = run_layer(cfg, w, tok)
    _check_routing(cfg, ws, tok.idx_np)
    yn = bf16_to_np(y)
    assert np.all(np.isfinite(yn))
    toks = _sample_tokens(cfg, tok.idx_np)
    ref, _ = _oracle_rows(cfg, tok.idx_np, tok.w_np, toks)
    ok, nl2, mr = close_enough(yn[toks], ref)
    assert ok, (name, toks, nl2, mr)


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
