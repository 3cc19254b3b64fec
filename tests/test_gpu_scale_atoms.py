"""mm_prepare_weight_scales: the block scales of a weight matrix rearranged
into 512-byte atoms, byte for byte as include/megamoe.h defines them (atom
(b, s), byte 16 l + 4 c + j = scale of row 128 b + 32 c + l, block 4 s + j)."""
import numpy as np
import pytest
import torch

import moe_expert_layer_idx_gb300 as mm

pytestmark = pytest.mark.gpu


def _atoms_by_definition(sf: np.ndarray) -> np.ndarray:
    rows, kb = sf.shape
    out = np.empty(rows * kb, np.uint8)
    for b in range(rows // 128):
        for s in range(kb // 4):
            base = (b * (kb // 4) + s) * 512
            for l in range(32):
                for c in range(4):
                    for j in range(4):
                        out[base + 16 * l + 4 * c + j] = sf[128 * b + 32 * c + l, 4 * s + j]
    return out


@pytest.mark.parametrize("rows,k", [(128, 128), (256, 512), (384, 1024), (128, 7168)])
def test_atoms_match_the_definition(rows, k):
    rng = np.random.default_rng(rows + k)
    sf = rng.integers(0, 256, (rows, k // 32), dtype=np.uint8)
    d_sf = torch.from_numpy(sf).cuda()
    out = torch.empty(rows * k // 32, dtype=torch.uint8, device="cuda")
    assert mm.mm_prepare_weight_scales(d_sf, rows, k, out) == mm.MM_OK
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.array_equal(got, _atoms_by_definition(sf))
    assert np.array_equal(np.sort(got), np.sort(sf.reshape(-1)))     # a permutation of the bytes


def test_torch_helper_keeps_shape_and_bytes():
    rng = np.random.default_rng(7)
    sf = torch.from_numpy(rng.integers(0, 256, (2, 256, 16), dtype=np.uint8)).cuda()   # E = 2, rows 256, K = 512
    out = mm.prepare_weight_scales(sf, 512)
    torch.cuda.synchronize()
    assert out.shape == sf.shape
    assert np.array_equal(out.cpu().numpy().reshape(-1), _atoms_by_definition(sf.cpu().numpy().reshape(512, 16)))
