"""Liveness of the whole-grid barrier while another stream holds an SM.

The scenario of sglang PR #36657 (Root cause; Validation: "GB300 side-stream
repro"): a kernel on a side stream occupies one SM.  With the default reserve
of two SMs the persistent grid still fits and the layer completes while the
side stream is busy; with the reserve disabled one CTA cannot become
resident, the grid barrier cannot complete, and the bounded wait reports
MM_ERR_TIMEOUT instead of hanging -- after which the next launch succeeds
(every launch resets its counters).  The blocker is a bounded spin (it always
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
BLOCKER_SMEM = 200 * 1024     # leaves no room for a layer CTA on that SM


@pytest.fixture(scope="module")
def layer():
    w = GpuWeights(CFG)
    tok = GpuTokens(CFG)
    ws = torch.empty(mm.mm_workspace_size(CFG.T, CFG.E, CFG.k, CFG.H, CFG.I), dtype=torch.uint8, device="cuda")
    return w, tok, ws


def _forward(w, tok, ws, y, stream=None):
    return mm.mm_forward(CFG.T, CFG.E, CFG.k, CFG.H, CFG.I, tok.x, tok.x_sf, tok.topk_idx, tok.topk_w, w.l1_w,
                         w.l1_sf, w.l2_w, w.l2_sf, y, CFG.clamp, 0, ws, stream=stream)


def _reference(layer):
    w, tok, ws = layer
    y = torch.empty(CFG.T, CFG.H, dtype=torch.bfloat16, device="cuda")
    assert _forward(w, tok, ws, y) == mm.MM_OK
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


def test_reserve_two_completes_while_side_stream_holds_an_sm(layer):
    w, tok, ws = layer
    want = _reference(layer)
    prev = mm.mm_set_reserved_sms(2)
    try:
        side = _occupy(1_500_000_000)
        y = torch.empty_like(want)
        assert _forward(w, tok, ws, y) == mm.MM_OK
        st = mm.mm_get_status(ws)
        still_busy = not side.query()
        side.synchronize()
    finally:
        mm.mm_set_reserved_sms(prev)
    assert st[0] == mm.MM_OK, st
    assert still_busy, "the side stream finished before the layer: the scenario did not overlap"
    assert torch.equal(y.view(torch.int16), want.view(torch.int16))


def test_full_grid_times_out_then_recovers(layer):
    w, tok, ws = layer
    want = _reference(layer)
    prev = mm.mm_set_reserved_sms(0)
    prev_to = mm.mm_get_wait_timeout_ns()
    mm.mm_set_wait_timeout_ns(50_000_000)
    try:
        side = _occupy(800_000_000)
        y = torch.empty_like(want)
        assert _forward(w, tok, ws, y) == mm.MM_OK
        st, sm, info = mm.mm_get_status(ws)
        side.synchronize()
    finally:
        mm.mm_set_reserved_sms(prev)
        mm.mm_set_wait_timeout_ns(prev_to)
    assert st == mm.MM_ERR_TIMEOUT, (st, sm, hex(info))
    # the next launch resets every counter and succeeds
    y2 = torch.empty_like(want)
    assert _forward(w, tok, ws, y2) == mm.MM_OK
    assert mm.mm_get_status(ws)[0] == mm.MM_OK
    assert torch.equal(y2.view(torch.int16), want.view(torch.int16))
