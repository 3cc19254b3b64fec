"""Liveness of the persistent grid while another stream holds an SM.

The scenario of sglang PR #36657 (Root cause; Validation: "GB300 side-stream
repro"): a kernel on a side stream occupies one SM.  With the default reserve
of two SMs the persistent grid still fits and the layer completes while the
side stream is busy; with the reserve disabled one CTA cannot become
resident until the side stream ends.  The dispatch is a static grid-stride
loop, so the tokens that CTA copies arrive only once it runs.  The layer
kernel has no whole-grid barrier and its tile schedule is dynamic: when other
CTAs run out of tiles and exit, the late CTA takes their SM, and the layer may
complete.  In a single-expert layer every tile needs every CTA's tokens, so
no CTA can finish first: the bounded wait on the expert's arrival count
reports MM_ERR_TIMEOUT instead of hanging -- after which the next launch
succeeds (every launch resets its counters).  The blocker is a bounded spin (it always
ends by itself), and no GPU is faulted or hung."""
import time

import pytest
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from helpers import blocker
from layer_inputs import GpuTokens, GpuWeights

pytestmark = pytest.mark.gpu

CFG = synth.Config("liveness", T=512, H=1024, I=512, E=32, k=8, clamp=7.0, seed=11)
# One expert; 2048 slots, so every CTA of a 152-CTA grid (12 warps each) dispatches some; 640 tiles
# (16 token blocks x (32 L1 + 8 L2)), more than the two each CTA claims before its first wait, so
# every resident CTA holds a tile that needs the late CTA's tokens and none can exit first.
CFG_ONE = synth.Config("liveness-one-expert", T=2048, H=2048, I=4096, E=1, k=1, clamp=7.0, seed=12)
BLOCKER_SMEM = 200 * 1024     # leaves no room for a layer CTA on that SM


def _make(cfg):
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg)
    ws = torch.empty(mm.mm_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I), dtype=torch.uint8, device="cuda")
    return cfg, w, tok, ws


@pytest.fixture(scope="module")
def layer():
    return _make(CFG)


@pytest.fixture(scope="module")
def layer_one():
    return _make(CFG_ONE)


def _forward(layer, y, stream=None):
    cfg, w, tok, ws = layer
    return mm.mm_forward(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, tok.x, tok.x_sf, tok.topk_idx, tok.topk_w, w.l1_w,
                         w.l1_sf, w.l2_w, w.l2_sf, y, cfg.clamp, 0, ws, stream=stream)


def _reference(layer):
    cfg, w, tok, ws = layer
    y = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    assert _forward(layer, y) == mm.MM_OK
    assert mm.mm_get_status(ws)[0] == mm.MM_OK
    return y


def _occupy(ns):
    side = torch.cuda.Stream()
    started = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    rc = blocker().occupy_one_sm(ns, BLOCKER_SMEM, started.data_ptr(), side.cuda_stream)
    assert rc == 0
    time.sleep(0.05)            # let it take its SM
    return side


def _full_grid_under_side_stream(layer, ns):
    """One launch with no reserve and a 50 ms wait limit while a side stream holds an SM."""
    ws = layer[3]
    prev = mm.mm_set_reserved_sms(0)
    prev_to = mm.mm_get_wait_timeout_ns()
    mm.mm_set_wait_timeout_ns(50_000_000)
    try:
        side = _occupy(ns)
        y = torch.empty(layer[0].T, layer[0].H, dtype=torch.bfloat16, device="cuda")
        assert _forward(layer, y) == mm.MM_OK
        st = mm.mm_get_status(ws)
        side.synchronize()
    finally:
        mm.mm_set_reserved_sms(prev)
        mm.mm_set_wait_timeout_ns(prev_to)
    return y, st


def test_reserve_two_completes_while_side_stream_holds_an_sm(layer):
    ws = layer[3]
    want = _reference(layer)
    prev = mm.mm_set_reserved_sms(2)
    try:
        side = _occupy(1_500_000_000)
        y = torch.empty_like(want)
        assert _forward(layer, y) == mm.MM_OK
        st = mm.mm_get_status(ws)
        still_busy = not side.query()
        side.synchronize()
    finally:
        mm.mm_set_reserved_sms(prev)
    assert st[0] == mm.MM_OK, st
    assert still_busy, "the side stream finished before the layer: the scenario did not overlap"
    assert torch.equal(y.view(torch.int16), want.view(torch.int16))


def test_full_grid_completes_or_reports_timeout(layer):
    """Many experts: the late CTA may run on an SM another CTA left.  Either
    the result is exact or the launch reports a timeout -- never a hang, never
    a silent wrong result."""
    want = _reference(layer)
    y, (st, sm, info) = _full_grid_under_side_stream(layer, 800_000_000)
    assert st in (mm.MM_OK, mm.MM_ERR_TIMEOUT), (st, sm, hex(info))
    if st == mm.MM_OK:
        assert torch.equal(y.view(torch.int16), want.view(torch.int16))


def test_single_expert_full_grid_times_out_then_recovers(layer_one):
    want = _reference(layer_one)
    y, (st, sm, info) = _full_grid_under_side_stream(layer_one, 800_000_000)
    assert st == mm.MM_ERR_TIMEOUT, (st, sm, hex(info))
    # the next launch resets every counter and succeeds
    y2 = torch.empty_like(want)
    assert _forward(layer_one, y2) == mm.MM_OK
    assert mm.mm_get_status(layer_one[3])[0] == mm.MM_OK
    assert torch.equal(y2.view(torch.int16), want.view(torch.int16))
