"""Host-side checks of the C ABI, no GPU needed: the library builds and loads,
exports every entry point declared in include/*.h, rejects bad arguments
before touching the device, and sizes the persistent grid as the pages do."""
import glob
import math
import os
import re

import pytest

import moe_expert_layer_idx_gb300 as mm
from moe_expert_layer_idx_gb300 import build as mmbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mmbuild.build()
    return mm.lib()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(mm_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_abi():
    names = _declared()
    for want in ("mm_workspace_size", "mm_forward", "mm_set_reserved_sms"):
        assert want in names


def test_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


# ---------------------------------------------------------------- launch size
def _pages_rule(device_sms, reserve, current):
    """The SM-reserve arithmetic of sglang PR #36657 (digest page, 关键源码片段):
    max_num_sms = max(2, physical - max(reserve, 0)); target = min(max, current);
    target -= target % 2."""
    max_num = max(2, device_sms - max(reserve, 0))
    target = min(max_num, current)
    target -= target % 2
    return target


@pytest.mark.parametrize("sms", [148, 152, 160, 7])
@pytest.mark.parametrize("reserve", [-3, 0, 1, 2, 3, 10, 500])
@pytest.mark.parametrize("current", [0, 1, 2, 3, 75, 150, 151, 152, 1000])
def test_grid_size_follows_the_pages(lib, sms, reserve, current):
    got = mm.mm_grid_size(sms, reserve, current, 0)
    cur = min(current, sms) if current > 0 else sms
    want = _pages_rule(sms, reserve, cur)
    assert got == max(want, 2)          # our floor: never fewer than one 2-CTA pair
    assert got % 2 == 0


def test_grid_size_examples(lib):
    assert mm.mm_grid_size(152, 2, 0, 0) == 150      # default reserve of two
    assert mm.mm_grid_size(152, 0, 0, 0) == 152      # reserve disabled
    assert mm.mm_grid_size(152, 1, 0, 0) == 150      # odd -> even
    assert mm.mm_grid_size(152, 400, 0, 0) == 2      # excessive reserve floors at 2
    assert mm.mm_grid_size(152, 2, 0, 140) == 140    # never more CTAs than can be resident
    assert mm.mm_grid_size(152, 2, 0, 141) == 140
    assert mm.mm_grid_size(1, 0, 0, 0) == mm.MM_ERR_INVALID_ARG


def test_reserved_sms_setting(lib):
    prev = mm.mm_get_reserved_sms()
    if "MM_RESERVED_SMS" not in os.environ:
        assert prev == 2
    try:
        assert mm.mm_set_reserved_sms(-4) == prev
        assert mm.mm_get_reserved_sms() == 0
        assert mm.mm_set_reserved_sms(6) == 0
        assert mm.mm_get_reserved_sms() == 6
    finally:
        mm.mm_set_reserved_sms(prev)


def test_wait_timeout_setting(lib):
    prev = mm.mm_get_wait_timeout_ns()
    try:
        mm.mm_set_wait_timeout_ns(12345)
        assert mm.mm_get_wait_timeout_ns() == 12345
        mm.mm_set_wait_timeout_ns(0)
        assert mm.mm_get_wait_timeout_ns() == 2_000_000_000
    finally:
        mm.mm_set_wait_timeout_ns(prev)


# ---------------------------------------------------------------- workspace
def test_workspace_size_depends_on_shape_only(lib):
    a = mm.mm_workspace_size(128, 256, 8, 7168, 2048)
    assert a > 0
    assert mm.mm_workspace_size(129, 256, 8, 7168, 2048) > a
    # the dispatched tokens, L1 activations, weighted L2 rows and the token-scale
    # atoms (room for 2E + A/32 block halves per 128-wide K stage) dominate
    A, E = 128 * 8, 256
    big = A * (7168 + 2048 + 4 * 7168) + (2 * E + A // 32) * (7168 // 128 + 2048 // 128) * 512
    assert big <= a < big + 64 * 1024


@pytest.mark.parametrize("args", [(16, 8, 2, 100, 128), (16, 8, 2, 256, 64), (16, 0, 2, 256, 128),
                                  (16, 8, 17, 256, 128), (16, 1025, 2, 256, 128), (-1, 8, 2, 256, 128)])
def test_workspace_size_rejects_unsupported(lib, args):
    assert mm.mm_workspace_size(*args) == 0


def test_workspace_regions_are_disjoint_and_aligned(lib):
    shape = (100, 16, 4, 512, 256)
    total = mm.mm_workspace_size(*shape)
    end = 0
    for name in mm.REGIONS:
        off, nb = mm.mm_workspace_region(name, *shape)
        assert off % 256 == 0 and off >= end
        end = off + nb
    assert end <= total
    # routing chunk table: [E][C] counts and C bad-index words; one chunk up to 2048 assignments
    assert mm.mm_workspace_region("route_chunks", *shape)[1] == 4 * 16 * 1 + 4
    assert mm.mm_workspace_region("route_chunks", 20000, 256, 8, 512, 256)[1] == 4 * 256 * 128 + 4 * 128
    assert mm.mm_workspace_region("route_chunks", 300, 256, 8, 512, 256)[1] == 4 * 256 * 3 + 4 * 3


@pytest.mark.parametrize("A,chunks", [(1, 1), (2048, 1), (2049, 3), (4096, 4), (4097, 5), (131072, 128),
                                      (131073, 128), (1 << 24, 128)])
def test_routing_chunk_count(lib, A, chunks):
    """One routing CTA up to 2048 assignments, else ceil(A / 1024) chunks, at most 128."""
    E = 16
    assert mm.mm_workspace_region("route_chunks", A, E, 1, 128, 128)[1] == 4 * E * chunks + 4 * chunks


# ---------------------------------------------------------------- argument errors
FAKE = 1 << 20        # an aligned address that is never dereferenced


def _fwd(**kw):
    a = dict(num_tokens=64, experts=8, topk=2, hidden=256, inter=128, x=FAKE, x_sf=FAKE, topk_idx=FAKE,
             topk_w=FAKE, l1_w=FAKE, l1_sf=FAKE, l2_w=FAKE, l2_sf=FAKE, y=FAKE, clamp=7.0, num_sms=0,
             workspace=FAKE, workspace_bytes=1 << 40, stream=0)
    a.update(kw)
    return mm.mm_forward(**a)


def test_forward_argument_errors(lib):
    assert _fwd(num_tokens=0) == mm.MM_OK                      # nothing to do, nothing launched
    assert _fwd(hidden=200) == mm.MM_ERR_UNSUPPORTED_SHAPE
    assert _fwd(inter=192) == mm.MM_ERR_UNSUPPORTED_SHAPE
    assert _fwd(topk=17) == mm.MM_ERR_UNSUPPORTED_SHAPE
    assert _fwd(experts=0) == mm.MM_ERR_INVALID_ARG
    assert _fwd(x=0) == mm.MM_ERR_INVALID_ARG
    assert _fwd(y=0) == mm.MM_ERR_INVALID_ARG
    assert _fwd(x=FAKE + 8) == mm.MM_ERR_INVALID_ARG            # x needs 16-byte alignment
    assert _fwd(l1_w=FAKE + 16) == mm.MM_ERR_INVALID_ARG        # packed FP4 weights need 32
    assert _fwd(l2_sf=FAKE + 4) == mm.MM_ERR_INVALID_ARG        # prepared scales need 16 (bulk copies)
    assert _fwd(workspace=FAKE + 128) == mm.MM_ERR_INVALID_ARG  # workspace needs 256
    assert _fwd(clamp=math.nan) == mm.MM_ERR_INVALID_ARG
    need = mm.mm_workspace_size(64, 8, 2, 256, 128)
    assert _fwd(workspace_bytes=need - 1) == mm.MM_ERR_WORKSPACE_TOO_SMALL


def _fwd_bf16(**kw):
    a = dict(num_tokens=64, experts=8, topk=2, hidden=256, inter=128, x_bf16=FAKE, topk_idx=FAKE,
             topk_w=FAKE, l1_w=FAKE, l1_sf=FAKE, l2_w=FAKE, l2_sf=FAKE, y=FAKE, clamp=7.0, num_sms=0,
             workspace=FAKE, workspace_bytes=1 << 40, stream=0)
    a.update(kw)
    return mm.mm_forward_bf16(**a)


def test_forward_bf16_argument_errors(lib):
    assert _fwd_bf16(num_tokens=0) == mm.MM_OK
    assert _fwd_bf16(hidden=200) == mm.MM_ERR_UNSUPPORTED_SHAPE
    assert _fwd_bf16(x_bf16=0) == mm.MM_ERR_INVALID_ARG            # no activations of either kind
    assert _fwd_bf16(x_bf16=FAKE + 8) == mm.MM_ERR_INVALID_ARG     # bf16 rows need 16-byte alignment
    assert _fwd_bf16(topk_w=0) == mm.MM_ERR_INVALID_ARG
    need = mm.mm_workspace_size(64, 8, 2, 256, 128)
    assert _fwd_bf16(workspace_bytes=need - 1) == mm.MM_ERR_WORKSPACE_TOO_SMALL


def _bf16_layer(**kw):
    a = dict(num_tokens=64, experts=8, topk=2, hidden=256, inter=128, x=FAKE, topk_idx=FAKE, topk_w=FAKE,
             l1_w=FAKE, l2_w=FAKE, y=FAKE, clamp=7.0, num_sms=0, workspace=FAKE, workspace_bytes=1 << 40, stream=0)
    a.update(kw)
    return mm.mm_bf16_forward(**a)


def test_bf16_layer_workspace_and_argument_errors(lib):
    fp8 = mm.mm_workspace_size(64, 8, 2, 256, 128)
    bf = mm.mm_bf16_workspace_size(64, 8, 2, 256, 128)
    assert bf > fp8                                            # 2-byte activations
    assert mm.mm_bf16_workspace_size(64, 8, 2, 200, 128) == 0
    assert _bf16_layer(num_tokens=0) == mm.MM_OK
    assert _bf16_layer(hidden=200) == mm.MM_ERR_UNSUPPORTED_SHAPE
    assert _bf16_layer(x=0) == mm.MM_ERR_INVALID_ARG
    assert _bf16_layer(l2_w=0) == mm.MM_ERR_INVALID_ARG
    assert _bf16_layer(x=FAKE + 8) == mm.MM_ERR_INVALID_ARG
    assert _bf16_layer(workspace_bytes=fp8) == mm.MM_ERR_WORKSPACE_TOO_SMALL   # the FP8 layer's size is short


def test_route_and_quantize_argument_errors(lib):
    assert mm.mm_route(64, 8, 2, 256, 128, FAKE, FAKE, 10, 0) == mm.MM_ERR_WORKSPACE_TOO_SMALL
    assert mm.mm_route(64, 8, 2, 256, 128, 0, FAKE, 1 << 40, 0) == mm.MM_ERR_INVALID_ARG
    assert mm.mm_quantize_mx(FAKE, 4, 48, mm.MM_FMT_E4M3, FAKE, FAKE, 0) == mm.MM_ERR_INVALID_ARG
    assert mm.mm_quantize_mx(FAKE, 4, 64, 7, FAKE, FAKE, 0) == mm.MM_ERR_INVALID_ARG
    assert mm.mm_quantize_mx(FAKE, 0, 64, mm.MM_FMT_E4M3, FAKE, FAKE, 0) == mm.MM_OK


def test_forward_without_device(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd() == mm.MM_ERR_NO_DEVICE
    assert _fwd_bf16() == mm.MM_ERR_NO_DEVICE
    assert _bf16_layer() == mm.MM_ERR_NO_DEVICE


def test_layer_variant_choice(lib):
    """Host-side choice of the layer kernel (no GPU needed): decode-sized
    batches (at most 16 assignments per expert on average) take the thin
    stages; larger ones take two-CTA tiles when hidden is a multiple of 256
    and the pair switch is on, else one-CTA tiles; the bf16 layer never pairs."""
    import moe_expert_layer_idx_gb300 as mm

    prev = mm.mm_set_pair_mma(1)
    try:
        assert mm.mm_layer_variant(128, 256, 8, 7168) == 1          # decode: 4 per expert
        assert mm.mm_layer_variant(512, 256, 8, 7168) == 1          # exactly 16 per expert
        assert mm.mm_layer_variant(8192, 256, 8, 7168) == 4         # prefill: pair
        assert mm.mm_layer_variant(400, 3, 2, 384) == 0             # hidden 384: one-CTA tiles
        assert mm.mm_layer_variant(8192, 256, 8, 7168, True) == 3 - 1   # bf16 wide
        assert mm.mm_layer_variant(128, 256, 8, 7168, True) == 3    # bf16 thin
        assert mm.mm_set_pair_mma(0) == 1
        assert mm.mm_get_pair_mma() == 0
        assert mm.mm_layer_variant(8192, 256, 8, 7168) == 0
        assert mm.mm_layer_variant(0, 8, 2, 256) == 1
        assert mm.mm_layer_variant(-1, 8, 2, 256) == mm.MM_ERR_INVALID_ARG
    finally:
        mm.mm_set_pair_mma(prev)


def test_prepare_weight_scales_argument_errors(lib):
    """Rows and K must be multiples of 128 and the buffers aligned; checked
    before any device work (nothing is dereferenced here)."""
    assert mm.mm_prepare_weight_scales(FAKE, 0, 256, FAKE, stream=0) == mm.MM_OK       # nothing to do
    assert mm.mm_prepare_weight_scales(FAKE, 100, 256, FAKE, stream=0) == mm.MM_ERR_INVALID_ARG
    assert mm.mm_prepare_weight_scales(FAKE, 128, 192, FAKE, stream=0) == mm.MM_ERR_INVALID_ARG
    assert mm.mm_prepare_weight_scales(FAKE + 2, 128, 256, FAKE, stream=0) == mm.MM_ERR_INVALID_ARG
    assert mm.mm_prepare_weight_scales(FAKE, 128, 256, FAKE + 8, stream=0) == mm.MM_ERR_INVALID_ARG
    assert mm.mm_prepare_weight_scales(0, 128, 256, FAKE, stream=0) == mm.MM_ERR_INVALID_ARG
