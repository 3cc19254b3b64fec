"""mm_quantize_mx against the oracle's block quantiser: bit-exact codes and
scales (both sides decide each code on the same exact fp32 value)."""
import numpy as np
import pytest
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from oracle import formats as OF
from layer_inputs import gpu_quantize

pytestmark = pytest.mark.gpu


def _both(vals: np.ndarray, fmt_gpu, fmt_or):
    rows, cols = vals.shape
    src = torch.from_numpy(np.ascontiguousarray(vals, np.float32)).cuda()
    c, s = gpu_quantize(src, rows, cols, fmt_gpu)
    torch.cuda.synchronize()
    oc, osf = OF.quantize_mx(vals.astype(np.float64), fmt_or)
    if fmt_or == OF.E2M1:
        oc = OF.pack_e2m1(oc)
    return c.cpu().numpy(), s.cpu().numpy(), oc, osf


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_x_quantisation_bit_exact(name):
    cfg = synth.CONFIGS[name]
    x = synth.x_f32(cfg)
    c, s, oc, osf = _both(x, mm.MM_FMT_E4M3, OF.E4M3)
    assert np.array_equal(s, osf)
    assert np.array_equal(c, oc)


@pytest.mark.parametrize("name,experts", [("tiny", [0, 5]), ("decode", [3])])
def test_weight_quantisation_bit_exact(name, experts):
    cfg = synth.CONFIGS[name]
    for e in experts:
        for w in (synth.w1_f32(cfg, e), synth.w2_f32(cfg, e)):
            c, s, oc, osf = _both(w, mm.MM_FMT_E2M1, OF.E2M1)
            assert np.array_equal(s, osf)
            assert np.array_equal(c, oc)


@pytest.mark.parametrize("fmt_gpu,fmt_or", [(mm.MM_FMT_E4M3, OF.E4M3), (mm.MM_FMT_E2M1, OF.E2M1)])
def test_edge_values_bit_exact(fmt_gpu, fmt_or):
    rng = np.random.default_rng(9)
    tab = OF.e4m3_decode_table()[:127] if fmt_or == OF.E4M3 else OF.e2m1_decode_table()[:8]
    pos = np.sort(tab)
    mids = (pos[1:] + pos[:-1]) / 2
    rows = []
    # exact ties at scale 2^0 (block max pinned to the top of the range)
    for i in range(0, len(mids), 31):
        r = np.zeros(32)
        r[0] = pos[-1]
        seg = mids[i:i + 31]
        r[1:1 + len(seg)] = seg * rng.choice([-1, 1], len(seg))
        rows.append(r)
    rows.append(np.zeros(32))                                   # all-zero block
    rows.append(np.full(32, -1e-30))                            # tiny negatives
    rows.append(rng.standard_normal(32) * 1e-38)                # near fp32 subnormal range
    rows.append(rng.standard_normal(32) * 3e37)                 # huge
    r = rng.standard_normal(32); r[5] = 448.0 * 2 ** 3; rows.append(r)   # max exactly F * 2^s
    vals = np.stack(rows).astype(np.float32).astype(np.float64)
    c, s, oc, osf = _both(vals, fmt_gpu, fmt_or)
    assert np.array_equal(s, osf)
    assert np.array_equal(c, oc)
