"""Routing kernel against the oracle: counts, offsets, permutation and its
inverse bit-exact (the stable order makes them unique)."""
import numpy as np
import pytest
import torch

import moe_expert_layer_idx_gb300 as mm
import synth
from oracle.routing import route

pytestmark = pytest.mark.gpu


def _gpu_route(idx: np.ndarray, E: int, H=256, I=128):
    T, k = idx.shape
    ws = torch.empty(mm.mm_workspace_size(max(T, 1), E, k, H, I), dtype=torch.uint8, device="cuda")
    d_idx = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda()
    assert mm.mm_route(T, E, k, H, I, d_idx, ws) == mm.MM_OK
    st = mm.mm_get_status(ws)
    rc, counts, offsets, perm, inv = mm.mm_read_routing(T, E, k, H, I, ws)
    assert rc == mm.MM_OK
    return st, counts, offsets, perm, inv


def _check(idx, E):
    st, c, o, p, i = _gpu_route(idx, E)
    assert st[0] == mm.MM_OK
    rc, ro, rp, ri = route(idx, E)
    n = int(ro[-1])
    assert np.array_equal(c, rc)
    assert np.array_equal(o, ro)
    assert np.array_equal(p[:n], rp)
    assert np.array_equal(i, ri)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skew", "kimi"])
def test_routing_of_the_configs(name):
    cfg = synth.CONFIGS[name]
    idx, _, _ = synth.routing(cfg)
    _check(idx, cfg.E)


@pytest.mark.parametrize("T,E,k,empty", [(1, 1, 1, 0.0), (8, 4, 3, 0.0), (48, 16, 2, 0.3), (192, 1024, 16, 0.1),
                                         (33, 7, 5, 0.0), (1000, 3, 1, 0.5), (5, 1024, 1, 0.0),
                                         (3001, 37, 7, 0.05), (20000, 256, 8, 0.02)])
def test_routing_edge_shapes(T, E, k, empty):
    rng = np.random.default_rng(T + E + k)
    idx = rng.integers(0, E, (T, k)).astype(np.int32)          # duplicate experts per token allowed
    idx[rng.random((T, k)) < empty] = -1
    _check(idx, E)


def test_all_slots_empty():
    _check(np.full((40, 4), -1, np.int32), 8)


def test_bad_index_is_reported():
    idx = np.zeros((20, 2), np.int32)
    idx[7, 1] = 8          # E = 8 -> out of range
    idx[12, 0] = -3
    st, *_ = _gpu_route(idx, 8)
    assert st[0] == mm.MM_ERR_BAD_INDEX
    assert st[2] == 7 * 2 + 1   # first bad flat index


def test_bad_index_is_reported_across_chunks():
    """Above 2048 assignments the flat array is split into chunks of ~1024;
    the smallest bad flat index over all chunks is reported."""
    idx = np.zeros((1000, 8), np.int32)          # 8000 assignments: 8 chunks
    idx[900, 3] = 16                             # chunk 7
    idx[400, 5] = -7                             # chunk 3: the first bad one
    idx[700, 0] = 99
    st, *_ = _gpu_route(idx, 16)
    assert st[0] == mm.MM_ERR_BAD_INDEX
    assert st[2] == 400 * 8 + 5


# token rows per block of each layer variant (mm_layer_variant's numbering)
BLOCK_ROWS = {0: 128, 1: 32, 2: 128, 3: 32, 4: 256}


def _region(ws, name, T, E, k, H, I, count):
    off, nb = mm.mm_workspace_region(name, T, E, k, H, I)
    assert count * 4 <= nb
    return ws[off:off + 4 * count].view(torch.int32).cpu().numpy()


@pytest.mark.parametrize("T,E,k,pair", [(128, 256, 8, False), (8192, 256, 8, False), (4096, 256, 8, False),
                                        (3001, 37, 7, False), (40, 8, 4, False), (2048, 64, 8, True),
                                        (700, 5, 3, True)])
def test_token_block_tables(T, E, k, pair):
    """items[e] = the first token block of expert e (prefix sum of
    ceil(count / block rows)), and token block b of expert e carries the
    record {e, items[e], offsets[e], counts[e]}: both exact, for thin, wide
    and two-CTA blocks."""
    H, I = 512, 256
    rng = np.random.default_rng(T * 7 + E)
    idx = rng.integers(0, E, (T, k)).astype(np.int32)
    idx[rng.random((T, k)) < 0.05] = -1
    prev = mm.mm_get_pair_mma()
    mm.mm_set_pair_mma(1 if pair else 0)
    try:
        variant = mm.mm_layer_variant(T, E, k, H)
        assert variant == (4 if pair else (1 if T * k <= 16 * E else 0))
        ws = torch.empty(mm.mm_workspace_size(T, E, k, H, I), dtype=torch.uint8, device="cuda")
        d_idx = torch.from_numpy(idx).cuda()
        assert mm.mm_route(T, E, k, H, I, d_idx, ws) == mm.MM_OK
        torch.cuda.synchronize()
    finally:
        mm.mm_set_pair_mma(prev)
    counts, offsets, _, _ = route(idx, E)
    nb = (counts + BLOCK_ROWS[variant] - 1) // BLOCK_ROWS[variant]
    want_items = np.concatenate([[0], np.cumsum(nb)]).astype(np.int32)
    items = _region(ws, "items", T, E, k, H, I, E + 1)
    assert np.array_equal(items, want_items)
    n = int(want_items[-1])
    rec = _region(ws, "token_blocks", T, E, k, H, I, 4 * n).reshape(n, 4)
    e = np.repeat(np.arange(E), nb)
    want = np.stack([e, want_items[e], offsets[e], counts[e]], axis=1).astype(np.int32)
    assert np.array_equal(rec, want)
