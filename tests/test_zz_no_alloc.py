"""mm_forward_noalloc: the layer for callers that cannot allocate device
memory where they run it (a runtime whose pool allocator owns all device
memory, a plugin handed only its inputs and outputs, a loop that forbids
allocation after start-up).  Its workspace is the library's fixed 64 MiB
device array, and mm_noalloc_get_status reads that array's status word.

Checked through the C ABI against mm_forward with a caller-owned workspace,
within the layer's output tolerance, on two calls in a row with different
inputs; against the oracle on one shape; a shape whose workspace exceeds the
array is refused before anything is enqueued; and a bad expert index put into
the input on the host is reported through mm_noalloc_get_status, after which
a clean call succeeds.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from oracle import moe as OM
from layer_inputs import ExpertCache, GpuTokens, GpuWeights, bf16_to_np, close_enough, oracle_tokens

pytestmark = pytest.mark.gpu

MID = synth.Config("noalloc-mid", T=96, H=1024, I=512, E=24, k=4, clamp=7.0, seed=4)
CASES = [synth.CONFIGS["tiny"], MID]


def _noalloc(cfg, w, tok):
    y = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = mm.mm_forward_noalloc(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, tok.x, tok.x_sf, tok.topk_idx, tok.topk_w,
                               w.l1_w, w.l1_sf, w.l2_w, w.l2_sf, y, cfg.clamp, 0)
    assert rc == mm.MM_OK, mm.STATUS_NAMES.get(rc, rc)
    return y


def _with_workspace(cfg, w, tok):
    ws = torch.empty(mm.mm_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I), dtype=torch.uint8, device="cuda")
    y = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    rc = mm.mm_forward(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, tok.x, tok.x_sf, tok.topk_idx, tok.topk_w, w.l1_w,
                       w.l1_sf, w.l2_w, w.l2_sf, y, cfg.clamp, 0, ws)
    assert rc == mm.MM_OK
    st, sm, info = mm.mm_get_status(ws)
    assert st == mm.MM_OK, (mm.STATUS_NAMES.get(st, st), sm, info)
    return y


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_noalloc_matches_workspace_path_two_calls(cfg):
    w = GpuWeights(cfg)
    for seed in (cfg.seed, cfg.seed + 100):           # two calls in a row, different tokens
        tok = GpuTokens(cfg, seed=seed)
        got = _noalloc(cfg, w, tok)
        st, sm, info = mm.mm_noalloc_get_status()
        assert st == mm.MM_OK, (mm.STATUS_NAMES.get(st, st), sm, info)
        want = _with_workspace(cfg, w, tok)
        ok, nl2, mr = close_enough(bf16_to_np(got), bf16_to_np(want))
        assert ok, (cfg.name, seed, nl2, mr)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_noalloc_matches_oracle():
    cfg = MID
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg)
    got = _noalloc(cfg, w, tok)
    assert mm.mm_noalloc_get_status()[0] == mm.MM_OK
    xc, xsf = oracle_tokens(cfg)
    ref = OM.moe_forward(xc, xsf, tok.idx_np, tok.w_np, ExpertCache(cfg), cfg.clamp, cfg.E)
    ok, nl2, mr = close_enough(bf16_to_np(got), ref)
    assert ok, (nl2, mr)


def test_noalloc_reports_a_bad_index_then_recovers():
    cfg = synth.CONFIGS["tiny"]
    routing = synth.routing(cfg)
    w = GpuWeights(cfg)
    bad = routing[0].copy()
    bad[5, 0] = cfg.E + 3                             # outside [-1, E): the routing kernel rejects it
    _noalloc(cfg, w, GpuTokens(cfg, routing=(bad, routing[1], 0.0)))
    st, sm, info = mm.mm_noalloc_get_status()
    assert st == mm.MM_ERR_BAD_INDEX and info == 5 * cfg.k + 0, (mm.STATUS_NAMES.get(st, st), info)
    tok = GpuTokens(cfg, routing=routing)
    got = _noalloc(cfg, w, tok)
    assert mm.mm_noalloc_get_status()[0] == mm.MM_OK   # the next call reset the status
    want = _with_workspace(cfg, w, tok)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    assert np.all(np.isfinite(bf16_to_np(got)))


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # 1024 tokens x top-8 at hidden 7168 needs ~300 MB of workspace
    big = synth.Config("too-big", T=1024, H=7168, I=2048, E=256, k=8, clamp=7.0)
    assert mm.mm_workspace_size(big.T, big.E, big.k, big.H, big.I) > 64 << 20
    x = torch.empty(16, dtype=torch.uint8, device="cuda")
    rc = mm.mm_forward_noalloc(big.T, big.E, big.k, big.H, big.I, x, x, x, x, x, x, x, x, x, 7.0, 0)
    assert rc == mm.MM_ERR_WORKSPACE_TOO_SMALL
