"""The fused layer on the GPU against the fp64 oracle, on shapes the oracle
finishes in seconds that still span several L1/L2 tiles, split experts into
several token blocks, leave ragged tails and exercise both kernel variants."""
import numpy as np
import pytest
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from oracle import formats as OF
from oracle import moe as OM
from layer_inputs import (ExpertCache, GpuTokens, GpuWeights, bf16_to_np, close_enough, oracle_tokens, token_scale_rows,
                          run_layer)

pytestmark = pytest.mark.gpu

SMALL = {
    # thin variant (<= 16 assignments per expert on average: 32-row token stages)
    "tiny": synth.CONFIGS["tiny"],
    # wide variant: ~267 assignments per expert -> 3 token blocks (one of them a full
    # 128-row block, loaded as one 128-row box), L2 tail of 128 hidden rows (H = 384)
    "ragged": synth.Config("ragged", T=400, H=384, I=256, E=3, k=2, clamp=7.0, seed=1),
    # many experts with 0-3 tokens, some slots empty, no clamp
    "sparse": synth.Config("sparse", T=37, H=256, I=128, E=16, k=4, clamp=0.0, seed=2),
    # skewed routing (hot experts split into several 32-row blocks), 4 L2 / 3 L1 weight blocks
    "wide": synth.Config("wide", T=129, H=1024, I=384, E=96, k=8, clamp=10.0, skew=True, seed=3),
    # ~6 tokens per expert, a hot expert split into several blocks
    "thin": synth.Config("thin", T=100, H=512, I=256, E=64, k=4, clamp=7.0, skew=True, seed=5),
    # thin variant with the 128-row L2 tail (H = 384)
    "thin_tail": synth.Config("thin_tail", T=48, H=384, I=128, E=8, k=2, clamp=7.0, seed=6),
    # wide variant, one ~75-token block per expert: five 16-row token boxes split 3/2
    # between the two producers
    "odd_boxes": synth.Config("odd_boxes", T=150, H=256, I=128, E=2, k=1, clamp=7.0, seed=7),
}


def _routing(cfg):
    idx, w, f = synth.routing(cfg)
    if cfg.name == "sparse":
        rng = np.random.default_rng(5)
        idx = idx.copy()
        idx[rng.random(idx.shape) < 0.15] = -1
        idx[4, :] = -1            # a token routed nowhere
    return idx, w, f


def _oracle(cfg, idx, w, tokens=None):
    xc, xsf = oracle_tokens(cfg)
    return OM.moe_forward(xc, xsf, idx, w, ExpertCache(cfg), cfg.clamp, cfg.E, tokens=tokens,
                          want_intermediates=True)


@pytest.fixture(scope="module", params=list(SMALL))
def case(request):
    cfg = SMALL[request.param]
    routing = _routing(cfg)
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg, routing=routing)
    y, ws = run_layer(cfg, w, tok)
    ref, inter = _oracle(cfg, routing[0], routing[1])
    return cfg, w, tok, y, ws, ref, inter


def test_output_matches_oracle(case):
    cfg, w, tok, y, ws, ref, _ = case
    ok, nl2, mr = close_enough(bf16_to_np(y), ref)
    assert ok, (cfg.name, nl2, mr)


def test_empty_rows_are_zero(case):
    cfg, w, tok, y, ws, ref, _ = case
    empty = np.all(tok.idx_np < 0, axis=1)
    if empty.any():
        assert torch.all(y[torch.from_numpy(empty).cuda()] == 0)


def test_routing_in_workspace(case):
    cfg, w, tok, y, ws, ref, inter = case
    rc, c, o, p, i = mm.mm_read_routing(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, ws)
    assert rc == mm.MM_OK
    n = int(inter["offsets"][-1])
    assert np.array_equal(c, inter["counts"]) and np.array_equal(o, inter["offsets"])
    assert np.array_equal(p[:n], inter["perm"]) and np.array_equal(i, inter["inv"])


def test_dispatched_scales_are_the_tokens_scales(case):
    """The dispatch writes each slot's UE8M0 scale bytes into its token
    block's scale atoms; read back into rows, slot s holds exactly the
    x_sf row of the token perm[s] // k."""
    cfg, w, tok, y, ws, ref, inter = case
    variant = mm.mm_layer_variant(cfg.T, cfg.E, cfg.k, cfg.H)
    got = token_scale_rows(ws, cfg, "xs_sf", variant, idx=tok.idx_np)
    xsf = tok.x_sf.cpu().numpy()
    want = xsf[inter["perm"] // cfg.k]
    assert np.array_equal(got, want), cfg.name


def test_l1_activations_close_to_oracle(case):
    """Diagnostic of the requantised L1 activations: the GPU accumulates in
    fp32 and the oracle in fp64, so a code may move by one step near a
    rounding tie (or a block scale near a power of two); nothing more."""
    cfg, w, tok, y, ws, ref, inter = case
    off, nb = mm.mm_workspace_region("l1_acts", cfg.T, cfg.E, cfg.k, cfg.H, cfg.I)
    codes = ws[off:off + nb].view(cfg.T * cfg.k, cfg.I).cpu().numpy()
    variant = mm.mm_layer_variant(cfg.T, cfg.E, cfg.k, cfg.H)
    sfs = token_scale_rows(ws, cfg, "l1_acts_sf", variant, idx=tok.idx_np)
    inv = inter["inv"]
    same = total = 0
    for f, (oc, osf) in inter["l1"].items():
        s = inv[f]
        g = OF.dequantize(codes[s][None], sfs[s][None], OF.E4M3)[0]
        r = OF.dequantize(oc[None], osf[None], OF.E4M3)[0]
        step = np.ldexp(1.0, np.frexp(np.maximum(np.abs(r), np.abs(g)))[1] - 4)   # one E4M3 step
        assert np.all(np.abs(g - r) <= step + 1e-300), (cfg.name, f)
        same += int(np.sum(g == r))
        total += g.size
    assert same >= 0.99 * total, (same, total)


def test_result_independent_of_grid_size(case):
    cfg, w, tok, y, ws, ref, _ = case
    for num_sms in (2, 16, 77):
        y2, _ = run_layer(cfg, w, tok, num_sms=num_sms, workspace=ws)
        assert torch.equal(y2.view(torch.int16), y.view(torch.int16)), num_sms


def test_repeat_launch_is_bit_identical(case):
    cfg, w, tok, y, ws, ref, _ = case
    y2, _ = run_layer(cfg, w, tok, workspace=ws)
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))


def test_binding_clamp():
    cfg = synth.Config("clamp", T=48, H=256, I=128, E=4, k=2, clamp=0.25, seed=7)
    routing = synth.routing(cfg)
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg, routing=routing)
    y, _ = run_layer(cfg, w, tok)
    ref, _ = _oracle(cfg, routing[0], routing[1])
    ok, nl2, mr = close_enough(bf16_to_np(y), ref)
    assert ok, (nl2, mr)
    y0, _ = run_layer(cfg, w, tok, clamp=0.0)
    assert not torch.equal(y0, y)


def test_single_token_single_expert():
    cfg = synth.Config("one", T=1, H=128, I=128, E=1, k=1, clamp=7.0, seed=8)
    routing = (np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), 0.0)
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg, routing=routing)
    y, _ = run_layer(cfg, w, tok)
    ref, _ = _oracle(cfg, routing[0], routing[1])
    ok, nl2, mr = close_enough(bf16_to_np(y), ref)
    assert ok, (nl2, mr)


def test_bad_index_leaves_status_and_next_launch_recovers():
    cfg = SMALL["tiny"]
    routing = synth.routing(cfg)
    w = GpuWeights(cfg)
    bad = routing[0].copy()
    bad[3, 1] = cfg.E + 5
    tok_bad = GpuTokens(cfg, routing=(bad, routing[1], 0.0))
    ws = torch.empty(mm.mm_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I), dtype=torch.uint8, device="cuda")
    y = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    rc = mm.mm_forward(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, tok_bad.x, tok_bad.x_sf, tok_bad.topk_idx, tok_bad.topk_w,
                       w.l1_w, w.l1_sf, w.l2_w, w.l2_sf, y, cfg.clamp, 0, ws)
    assert rc == mm.MM_OK
    st, sm, info = mm.mm_get_status(ws)
    assert st == mm.MM_ERR_BAD_INDEX and info == 3 * cfg.k + 1
    tok = GpuTokens(cfg, routing=routing)
    y2, _ = run_layer(cfg, w, tok, workspace=ws)       # asserts status OK after the relaunch
    ref, _ = _oracle(cfg, routing[0], routing[1])
    assert close_enough(bf16_to_np(y2), ref)[0]
