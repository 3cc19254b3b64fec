"""mm_forward_bf16: bf16 activations, quantised to E4M3 + UE8M0/32 inside the
layer's dispatch, checked two ways on the same seeded inputs:

* bit for bit against mm_forward on the library's own quantisation
  (mm_quantize_mx) of the same values -- the fold must not change a byte;
* against the fp64 oracle fed with the oracle's quantisation (the scale rule
  and round-to-nearest-even) of the same bf16 values.

Cases cover both kernel variants (thin: few tokens per expert; wide: 128-row
token blocks) and empty slots."""
import numpy as np
import pytest
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from oracle import formats as OF
from oracle import moe as OM
from layer_inputs import ExpertCache, GpuTokens, GpuWeights, bf16_to_np, close_enough, gpu_quantize

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": synth.CONFIGS["tiny"],                                                        # thin variant
    "ragged": synth.Config("ragged", T=400, H=384, I=256, E=3, k=2, clamp=7.0, seed=1),  # wide variant
    "sparse": synth.Config("sparse", T=37, H=256, I=128, E=16, k=4, clamp=0.0, seed=2),  # empty slots
}


def _routing(cfg):
    idx, w, f = synth.routing(cfg)
    if cfg.name == "sparse":
        rng = np.random.default_rng(5)
        idx = idx.copy()
        idx[rng.random(idx.shape) < 0.15] = -1
        idx[4, :] = -1            # a token routed nowhere
    return idx, w, f


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    cfg = CASES[request.param]
    T, H = cfg.T, cfg.H
    routing = _routing(cfg)
    w = GpuWeights(cfg)
    tok = GpuTokens(cfg, routing=routing)
    xf = torch.empty(T * H, dtype=torch.float32, device="cuda")
    synth.normal_f32_cuda(cfg.seed, synth.TENSOR_X, 0, xf)
    xb = xf.view(T, H).to(torch.bfloat16)                      # round to nearest even
    ws = torch.empty(mm.mm_workspace_size(T, cfg.E, cfg.k, H, cfg.I), dtype=torch.uint8, device="cuda")

    y_fold = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    rc = mm.mm_forward_bf16(T, cfg.E, cfg.k, H, cfg.I, xb, tok.topk_idx, tok.topk_w, w.l1_w, w.l1_sf, w.l2_w,
                            w.l2_sf, y_fold, cfg.clamp, 0, ws)
    assert rc == mm.MM_OK, mm.STATUS_NAMES.get(rc, rc)
    st = mm.mm_get_status(ws)
    assert st[0] == mm.MM_OK, st

    x8, sf8 = gpu_quantize(xb.float().reshape(-1), T, H, mm.MM_FMT_E4M3)
    y_sep = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    rc = mm.mm_forward(T, cfg.E, cfg.k, H, cfg.I, x8, sf8, tok.topk_idx, tok.topk_w, w.l1_w, w.l1_sf, w.l2_w,
                       w.l2_sf, y_sep, cfg.clamp, 0, ws)
    assert rc == mm.MM_OK, mm.STATUS_NAMES.get(rc, rc)
    st = mm.mm_get_status(ws)
    assert st[0] == mm.MM_OK, st
    return cfg, routing, xb.cpu(), y_fold, y_sep


def test_fold_is_bit_identical_to_quantize_then_forward(case):
    cfg, routing, xb, y_fold, y_sep = case
    assert torch.equal(y_fold.view(torch.int16), y_sep.view(torch.int16)), cfg.name


def test_fold_matches_oracle(case):
    cfg, routing, xb, y_fold, y_sep = case
    codes, sf = OF.quantize_mx(xb.float().numpy().astype(np.float64), OF.E4M3)
    ref = OM.moe_forward(codes, sf, routing[0], routing[1], ExpertCache(cfg), cfg.clamp, cfg.E)
    ok, nl2, mr = close_enough(bf16_to_np(y_fold), ref)
    assert ok, (cfg.name, nl2, mr)


def test_fold_leaves_empty_tokens_zero(case):
    cfg, routing, xb, y_fold, y_sep = case
    empty = np.all(routing[0] < 0, axis=1)
    if empty.any():
        assert torch.all(y_fold[torch.from_numpy(empty).cuda()] == 0)
