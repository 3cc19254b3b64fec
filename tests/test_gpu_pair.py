"""The two-CTA tiles (tcgen05 cta_group::2, M = 256: a cluster of two CTAs
shares each MMA tile, each CTA holding 128 of its token rows and 128 of its
256 weight rows) against the fp64 oracle, and against one-CTA tiles of the
same batch.  Shapes: token blocks of 256 rows split 128 + 128 (two 128-row
boxes), blocks whose odd half is short or empty, hot experts split into
several blocks, empty experts, no clamp.  Also: graph replays with changed
inputs equal to eager, results independent of the grid size, a bad index
reported and cleared by the next launch."""
import numpy as np
import pytest
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from oracle import moe as OM
from oracle.routing import route
from layer_inputs import ExpertCache, GpuTokens, GpuWeights, bf16_to_np, close_enough, oracle_tokens, run_layer

pytestmark = pytest.mark.gpu

PAIR = 4


@pytest.fixture(scope="module", autouse=True)
def pair_on():
    """The two-CTA tiles are off by default; this module runs with them on."""
    prev = mm.mm_set_pair_mma(1)
    yield
    mm.mm_set_pair_mma(prev)


CASES = {
    # 300 assignments per expert: two blocks of 150 rows (128 on the even CTA, 22 on the odd one)
    "pair-two-blocks": synth.Config("pair-two-blocks", T=600, H=512, I=256, E=4, k=2, clamp=7.0, seed=30),
    # 50 per expert: one block, the odd CTA's half empty
    "pair-half-empty": synth.Config("pair-half-empty", T=200, H=256, I=128, E=8, k=2, clamp=7.0, seed=31),
    # 256 per expert: one block, both halves full (single 128-row token boxes)
    "pair-full": synth.Config("pair-full", T=512, H=1024, I=384, E=2, k=1, clamp=7.0, seed=32),
    # skewed routing: hot experts in several blocks, cold and empty experts, no clamp
    "pair-skew": synth.Config("pair-skew", T=320, H=512, I=256, E=64, k=4, clamp=0.0, skew=True, seed=33),
}


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    cfg = CASES[request.param]
    assert mm.mm_get_pair_mma() == 1
    assert mm.mm_layer_variant(cfg.T, cfg.E, cfg.k, cfg.H) == PAIR
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg)
    y, ws = run_layer(cfg, w, tok)
    return cfg, w, tok, y, ws


def test_pair_matches_oracle(case):
    cfg, w, tok, y, ws = case
    rc, c, o, p, i = mm.mm_read_routing(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, ws)
    rc_, ro, rp, ri = route(tok.idx_np, cfg.E)
    assert rc == mm.MM_OK and np.array_equal(c, rc_) and np.array_equal(o, ro)
    assert np.array_equal(p[: int(ro[-1])], rp) and np.array_equal(i, ri)
    xc, xsf = oracle_tokens(cfg)
    ref = OM.moe_forward(xc, xsf, tok.idx_np, tok.w_np, ExpertCache(cfg), cfg.clamp, cfg.E)
    ok, nl2, mr = close_enough(bf16_to_np(y), ref)
    assert ok, (cfg.name, nl2, mr)


def test_pair_equals_one_cta_tiles(case):
    """The same products summed in the same order: the two tilings agree bit for bit."""
    cfg, w, tok, y, ws = case
    prev = mm.mm_set_pair_mma(0)
    try:
        assert mm.mm_layer_variant(cfg.T, cfg.E, cfg.k, cfg.H) == 0
        y1, _ = run_layer(cfg, w, tok)
    finally:
        mm.mm_set_pair_mma(prev)
    ok, nl2, mr = close_enough(bf16_to_np(y1), bf16_to_np(y))
    assert ok, (cfg.name, nl2, mr)
    assert torch.equal(y1.view(torch.int16), y.view(torch.int16)), cfg.name


def test_pair_independent_of_grid_size(case):
    cfg, w, tok, y, ws = case
    for num_sms in (2, 6, 77):
        y2, _ = run_layer(cfg, w, tok, num_sms=num_sms, workspace=ws)
        assert torch.equal(y2.view(torch.int16), y.view(torch.int16)), num_sms


def test_pair_graph_replays_equal_eager():
    cfg = CASES["pair-skew"]
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
    for r in range(1, 13):
        new = GpuTokens(cfg, seed=r)
        tok.x.copy_(new.x); tok.x_sf.copy_(new.x_sf)
        tok.topk_idx.copy_(new.topk_idx); tok.topk_w.copy_(new.topk_w)
        y_g.fill_(float("nan"))
        graph.replay()
        assert fwd(y_e, ws_e) == mm.MM_OK
        torch.cuda.synchronize()
        assert mm.mm_get_status(ws_g)[0] == mm.MM_OK and mm.mm_get_status(ws_e)[0] == mm.MM_OK
        assert torch.equal(y_g.view(torch.int16), y_e.view(torch.int16)), f"replay {r}"


def test_pair_bad_index_then_recovers():
    cfg = CASES["pair-two-blocks"]
    routing = synth.routing(cfg)
    w = GpuWeights(cfg)
    bad = routing[0].copy()
    bad[7, 1] = cfg.E
    tok_bad = GpuTokens(cfg, routing=(bad, routing[1], 0.0))
    ws = torch.empty(mm.mm_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I), dtype=torch.uint8, device="cuda")
    y = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    rc = mm.mm_forward(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, tok_bad.x, tok_bad.x_sf, tok_bad.topk_idx, tok_bad.topk_w,
                       w.l1_w, w.l1_sf, w.l2_w, w.l2_sf, y, cfg.clamp, 0, ws)
    assert rc == mm.MM_OK
    st, sm, info = mm.mm_get_status(ws)
    assert st == mm.MM_ERR_BAD_INDEX and info == 7 * cfg.k + 1
    tok = GpuTokens(cfg, routing=routing)
    y2, _ = run_layer(cfg, w, tok, workspace=ws)
    xc, xsf = oracle_tokens(cfg)
    ref = OM.moe_forward(xc, xsf, routing[0], routing[1], ExpertCache(cfg), cfg.clamp, cfg.E)
    assert close_enough(bf16_to_np(y2), ref)[0]


def test_pair_bf16_activations_equal_quantize_then_forward():
    """mm_forward_bf16 with two-CTA tiles: the dispatch quantises each token
    and writes its scales into both 128-row halves of the token blocks' scale
    atoms; the result equals mm_forward on mm_quantize_mx of the same values,
    bit for bit (blocks of 150 rows: 128 on the even CTA, 22 on the odd one)."""
    from layer_inputs import gpu_quantize
    cfg = CASES["pair-two-blocks"]
    T, H = cfg.T, cfg.H
    assert mm.mm_layer_variant(T, cfg.E, cfg.k, H) == PAIR
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg)
    xf = torch.empty(T * H, dtype=torch.float32, device="cuda")
    synth.normal_f32_cuda(cfg.seed, synth.TENSOR_X, 0, xf)
    xb = xf.view(T, H).to(torch.bfloat16)
    ws = torch.empty(mm.mm_workspace_size(T, cfg.E, cfg.k, H, cfg.I), dtype=torch.uint8, device="cuda")
    y_fold = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    assert mm.mm_forward_bf16(T, cfg.E, cfg.k, H, cfg.I, xb, tok.topk_idx, tok.topk_w, w.l1_w, w.l1_sf, w.l2_w,
                              w.l2_sf, y_fold, cfg.clamp, 0, ws) == mm.MM_OK
    assert mm.mm_get_status(ws)[0] == mm.MM_OK
    x8, sf8 = gpu_quantize(xb.float().reshape(-1), T, H, mm.MM_FMT_E4M3)
    y_sep = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    assert mm.mm_forward(T, cfg.E, cfg.k, H, cfg.I, x8, sf8, tok.topk_idx, tok.topk_w, w.l1_w, w.l1_sf, w.l2_w,
                         w.l2_sf, y_sep, cfg.clamp, 0, ws) == mm.MM_OK
    assert mm.mm_get_status(ws)[0] == mm.MM_OK
    assert torch.equal(y_fold.view(torch.int16), y_sep.view(torch.int16))
