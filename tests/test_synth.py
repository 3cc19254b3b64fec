"""The shared input generator: host build against its pure-Python definition,
and the routing recipe's stated properties."""
import numpy as np
import pytest

import synth


def test_host_build_matches_python_definition():
    tab = synth.normal_table()
    rng = np.random.default_rng(0)
    for seed, tid in [(0, 1), (3, 2), (12, 4), (2 ** 40 + 5, 3)]:
        idx = rng.integers(0, 2 ** 40, 40).tolist() + [0, 1, 2, 3, 4, 5, 6, 7]
        for i in idx:
            got = synth.normal_f32(seed, tid, i, 1, 0.125)[0]
            want = np.float32(tab[synth.index16_py(seed, tid, i)]) * np.float32(0.125)
            assert got == want


def test_contiguous_ranges_agree():
    a = synth.normal_f32(5, 2, 1000, 777)
    b = synth.normal_f32(5, 2, 1003, 100)
    assert np.array_equal(a[3:103], b)


def test_u64_is_splitmix_stream():
    out = synth.u64(7, 5, 0, 4)
    key = synth.key_of(7, 5)
    assert [int(v) for v in out] == [synth.mix64(key + (n + 1) * synth.GOLDEN) for n in range(4)]


def test_table_is_standard_normal():
    t = synth.normal_table().astype(np.float64)
    assert abs(t.mean()) < 1e-6
    assert abs(t.std() - 1.0) < 2e-3
    assert np.all(np.diff(t) > 0)
    v = synth.normal_f32(1, 1, 0, 1 << 18)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_routing_recipe(name):
    cfg = synth.CONFIGS[name]
    idx, w, _ = synth.routing(cfg)
    assert idx.shape == (cfg.T, cfg.k) and w.shape == (cfg.T, cfg.k)
    assert np.all((idx >= 0) & (idx < cfg.E))
    assert all(len(set(r)) == cfg.k for r in idx.tolist())        # k distinct experts
    assert np.allclose(w.sum(1), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)                         # descending weight


def test_skew_recipe_properties():
    cfg = synth.CONFIGS["skew"]
    idx, w, factor = synth.routing(cfg)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
    mean = cfg.T * cfg.k / cfg.E
    assert counts.min() == 0 and counts.max() > 10 * mean
    assert factor >= 1.0
