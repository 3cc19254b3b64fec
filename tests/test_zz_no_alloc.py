"""mm_forward_noalloc: the layer for callers that cannot allocate device
memory (a stream under CUDA-graph capture, a runtime whose pool allocator owns
all device memory, a loop that forbids allocation after start-up).  Its
workspace is the library's fixed 48 MiB device array.

Checked through the C ABI against mm_forward with a caller-owned workspace,
within the layer's output tolerance, on two calls in a row with different
inputs; and a shape whose workspace exceeds the array is refused before
anything is enqueued.  This file is collected last on purpose."""
import pytest
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from layer_inputs import GpuTokens, GpuWeights, bf16_to_np, close_enough

pytestmark = pytest.mark.gpu

CASES = [
    synth.CONFIGS["tiny"],
    synth.Config("noalloc-mid", T=96, H=1024, I=512, E=24, k=4, clamp=7.0, seed=4),
]


def _noalloc(cfg, w, tok):
    y = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = mm.mm_forward_noalloc(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, tok.x, tok.x_sf, tok.topk_idx, tok.topk_w,
                               w.l1_w, w.l1_sf, w.l2_w, w.l2_sf, y, cfg.clamp, 0)
    assert rc == mm.MM_OK, mm.STATUS_NAMES.get(rc, rc)
    torch.cuda.synchronize()
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
        want = _with_workspace(cfg, w, tok)
        ok, nl2, mr = close_enough(bf16_to_np(got), bf16_to_np(want))
        assert ok, (cfg.name, seed, nl2, mr)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # 1024 tokens x top-8 at hidden 7168 needs ~300 MB of workspace
    big = synth.Config("too-big", T=1024, H=7168, I=2048, E=256, k=8, clamp=7.0)
    assert mm.mm_workspace_size(big.T, big.E, big.k, big.H, big.I) > 48 << 20
    x = torch.empty(16, dtype=torch.uint8, device="cuda")
    rc = mm.mm_forward_noalloc(big.T, big.E, big.k, big.H, big.I, x, x, x, x, x, x, x, x, x, 7.0, 0)
    assert rc == mm.MM_ERR_WORKSPACE_TOO_SMALL
