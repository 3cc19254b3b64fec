"""GB300 (sm_103a) fused MoE expert layer -- Python binding of libmegamoe.so.

Argument marshalling only: every step of the layer runs in the CUDA kernels
of ``csrc/`` behind the C ABI of ``include/megamoe.h``.  The functions keep
the C names; tensors may be passed as torch tensors (their ``data_ptr()`` is
used) or as raw integer addresses.  There is no CPU fallback: if the library
is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmegamoe.so")

MM_OK = 0
MM_ERR_INVALID_ARG = -1
MM_ERR_UNSUPPORTED_SHAPE = -2
MM_ERR_WORKSPACE_TOO_SMALL = -3
MM_ERR_CUDA = -4
MM_ERR_TIMEOUT = -5
MM_ERR_BAD_INDEX = -6
MM_ERR_BOUNDS = -7
MM_ERR_NO_DEVICE = -8
STATUS_NAMES = {0: "MM_OK", -1: "MM_ERR_INVALID_ARG", -2: "MM_ERR_UNSUPPORTED_SHAPE",
                -3: "MM_ERR_WORKSPACE_TOO_SMALL", -4: "MM_ERR_CUDA", -5: "MM_ERR_TIMEOUT",
                -6: "MM_ERR_BAD_INDEX", -7: "MM_ERR_BOUNDS", -8: "MM_ERR_NO_DEVICE"}

MM_FMT_E4M3 = 0
MM_FMT_E2M1 = 1

REGIONS = {"ctrl": 0, "counts": 1, "offsets": 2, "items": 3, "arrival": 4, "l1_done": 5, "perm": 6,
           "inv": 7, "xs": 8, "xs_sf": 9, "l1_acts": 10, "l1_acts_sf": 11, "stage": 12, "route_chunks": 13,
           "token_blocks": 14}

_lib = None
_c_int, _c_size, _c_vp, _c_ll = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_longlong

_SIGS = {
    "mm_workspace_size": (_c_size, [_c_int] * 5),
    "mm_forward": (_c_int, [_c_int] * 5 + [_c_vp] * 9 + [ctypes.c_float, _c_int, _c_vp, _c_size, _c_vp]),
    "mm_set_reserved_sms": (_c_int, [_c_int]),
    "mm_get_reserved_sms": (_c_int, []),
    "mm_set_pair_mma": (_c_int, [_c_int]),
    "mm_get_pair_mma": (_c_int, []),
    "mm_layer_variant": (_c_int, [_c_int] * 5),
    "mm_grid_size": (_c_int, [_c_int] * 4),
    "mm_set_wait_timeout_ns": (None, [ctypes.c_ulonglong]),
    "mm_get_wait_timeout_ns": (ctypes.c_ulonglong, []),
    "mm_get_status": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp]),
    "mm_route": (_c_int, [_c_int] * 5 + [_c_vp, _c_vp, _c_size, _c_vp]),
    "mm_read_routing": (_c_int, [_c_int] * 5 + [_c_vp] * 5),
    "mm_workspace_region": (_c_int, [_c_int] * 6 + [_c_vp, _c_vp]),
    "mm_quantize_mx": (_c_int, [_c_vp, _c_ll, _c_ll, _c_int, _c_vp, _c_vp, _c_vp]),
    "mm_prepare_weight_scales": (_c_int, [_c_vp, _c_ll, _c_ll, _c_vp, _c_vp]),
    "mm_forward_noalloc": (_c_int, [_c_int] * 5 + [_c_vp] * 9 + [ctypes.c_float, _c_int, _c_vp]),
    "mm_noalloc_get_status": (_c_int, [_c_vp, _c_vp, _c_vp]),
    "mm_forward_bf16": (_c_int, [_c_int] * 5 + [_c_vp] * 8 + [ctypes.c_float, _c_int, _c_vp, _c_size, _c_vp]),
    "mm_bf16_workspace_size": (_c_size, [_c_int] * 5),
    "mm_bf16_forward": (_c_int, [_c_int] * 5 + [_c_vp] * 6 + [ctypes.c_float, _c_int, _c_vp, _c_size, _c_vp]),
    "mm_f8b_forward": (_c_int, [_c_int] * 5 + [_c_vp] * 9 + [ctypes.c_float, _c_int, _c_vp, _c_size, _c_vp]),
    "mm_quantize_f8b": (_c_int, [_c_vp, _c_ll, _c_ll, _c_int, _c_vp, _c_vp, _c_vp]),
}


class MegaMoEError(RuntimeError):
    def __init__(self, what: str, code: int):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}")
        self.code = code


def lib():
    """The loaded libmegamoe.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ C ABI
def mm_workspace_size(max_tokens, experts, topk, hidden, inter) -> int:
    return lib().mm_workspace_size(max_tokens, experts, topk, hidden, inter)


def mm_forward(num_tokens, experts, topk, hidden, inter, x, x_sf, topk_idx, topk_w, l1_w, l1_sf,
               l2_w, l2_sf, y, clamp, num_sms, workspace, workspace_bytes=None, stream=None) -> int:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    return lib().mm_forward(num_tokens, experts, topk, hidden, inter, _ptr(x), _ptr(x_sf), _ptr(topk_idx),
                            _ptr(topk_w), _ptr(l1_w), _ptr(l1_sf), _ptr(l2_w), _ptr(l2_sf), _ptr(y),
                            float(clamp), num_sms, _ptr(workspace), workspace_bytes, _stream(stream))


def mm_forward_bf16(num_tokens, experts, topk, hidden, inter, x_bf16, topk_idx, topk_w, l1_w, l1_sf,
                    l2_w, l2_sf, y, clamp, num_sms, workspace, workspace_bytes=None, stream=None) -> int:
    """mm_forward on bf16 activations [T, H], quantised to E4M3 + UE8M0/32 in the layer's dispatch."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    return lib().mm_forward_bf16(num_tokens, experts, topk, hidden, inter, _ptr(x_bf16), _ptr(topk_idx),
                                 _ptr(topk_w), _ptr(l1_w), _ptr(l1_sf), _ptr(l2_w), _ptr(l2_sf), _ptr(y),
                                 float(clamp), num_sms, _ptr(workspace), workspace_bytes, _stream(stream))


def mm_bf16_workspace_size(max_tokens, experts, topk, hidden, inter) -> int:
    return lib().mm_bf16_workspace_size(max_tokens, experts, topk, hidden, inter)


def mm_bf16_forward(num_tokens, experts, topk, hidden, inter, x, topk_idx, topk_w, l1_w, l2_w, y, clamp,
                    num_sms, workspace, workspace_bytes=None, stream=None) -> int:
    """The bf16 x bf16 layer (bf16 activations and weights, no scale factors)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    return lib().mm_bf16_forward(num_tokens, experts, topk, hidden, inter, _ptr(x), _ptr(topk_idx), _ptr(topk_w),
                                 _ptr(l1_w), _ptr(l2_w), _ptr(y), float(clamp), num_sms, _ptr(workspace),
                                 workspace_bytes, _stream(stream))


def mm_f8b_forward(num_tokens, experts, topk, hidden, inter, x, x_sf, topk_idx, topk_w, l1_w, l1_sf, l2_w,
                   l2_sf, y, clamp, num_sms, workspace, workspace_bytes=None, stream=None) -> int:
    """The layer in the (1, 128, 128) recipe: E4M3 activations and weights with
    float32 scales per 1 x 128 (x_sf) and 128 x 128 (l1_sf, l2_sf) blocks."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    return lib().mm_f8b_forward(num_tokens, experts, topk, hidden, inter, _ptr(x), _ptr(x_sf), _ptr(topk_idx),
                                _ptr(topk_w), _ptr(l1_w), _ptr(l1_sf), _ptr(l2_w), _ptr(l2_sf), _ptr(y),
                                float(clamp), num_sms, _ptr(workspace), workspace_bytes, _stream(stream))


def mm_quantize_f8b(src, rows, cols, block_rows, dst, dst_sf, stream=None) -> int:
    """fp32 [rows, cols] -> E4M3 codes + float32 scales per block_rows x 128 block."""
    return lib().mm_quantize_f8b(_ptr(src), rows, cols, block_rows, _ptr(dst), _ptr(dst_sf), _stream(stream))


def mm_set_reserved_sms(n) -> int:
    return lib().mm_set_reserved_sms(n)


def mm_get_reserved_sms() -> int:
    return lib().mm_get_reserved_sms()


def mm_set_pair_mma(enable) -> int:
    """Two-CTA (M = 256) tiles for wide batches on (1) or off (0); returns the previous setting."""
    return lib().mm_set_pair_mma(int(enable))


def mm_get_pair_mma() -> int:
    return lib().mm_get_pair_mma()


VARIANT_NAMES = {0: "wide (one CTA, 128-token tiles)", 1: "thin (one CTA, 32-token stages)",
                 2: "bf16 wide", 3: "bf16 thin", 4: "pair (two CTAs, 256-token tiles)"}


def mm_layer_variant(num_tokens, experts, topk, hidden, bf16_layer=False) -> int:
    return lib().mm_layer_variant(num_tokens, experts, topk, hidden, int(bool(bf16_layer)))


def mm_grid_size(device_sms, reserved_sms, num_sms, max_resident=0) -> int:
    return lib().mm_grid_size(device_sms, reserved_sms, num_sms, max_resident)


def mm_set_wait_timeout_ns(ns) -> None:
    lib().mm_set_wait_timeout_ns(ns)


def mm_get_wait_timeout_ns() -> int:
    return lib().mm_get_wait_timeout_ns()


def mm_get_status(workspace, stream=None):
    """Returns (status, sm, info)."""
    sm, info = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().mm_get_status(_ptr(workspace), _stream(stream), ctypes.addressof(sm), ctypes.addressof(info))
    return rc, sm.value, info.value


def mm_route(num_tokens, experts, topk, hidden, inter, topk_idx, workspace, workspace_bytes=None,
             stream=None) -> int:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    return lib().mm_route(num_tokens, experts, topk, hidden, inter, _ptr(topk_idx), _ptr(workspace),
                          workspace_bytes, _stream(stream))


def mm_read_routing(num_tokens, experts, topk, hidden, inter, workspace):
    """Returns (rc, counts, offsets, perm, inv) as numpy int32 arrays."""
    import numpy as np

    A = num_tokens * topk
    counts = np.zeros(experts, np.int32)
    offsets = np.zeros(experts + 1, np.int32)
    perm = np.zeros(A, np.int32)
    inv = np.zeros(A, np.int32)
    rc = lib().mm_read_routing(num_tokens, experts, topk, hidden, inter, _ptr(workspace),
                               counts.ctypes.data, offsets.ctypes.data, perm.ctypes.data, inv.ctypes.data)
    return rc, counts, offsets, perm, inv


def mm_workspace_region(which, num_tokens, experts, topk, hidden, inter):
    """Returns (offset, bytes) of a workspace region (name from REGIONS, or its number)."""
    w = REGIONS[which] if isinstance(which, str) else which
    off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    rc = lib().mm_workspace_region(w, num_tokens, experts, topk, hidden, inter,
                                   ctypes.addressof(off), ctypes.addressof(nb))
    if rc != MM_OK:
        raise MegaMoEError("mm_workspace_region", rc)
    return off.value, nb.value


def mm_quantize_mx(src, rows, cols, fmt, dst, dst_sf, stream=None) -> int:
    return lib().mm_quantize_mx(_ptr(src), rows, cols, fmt, _ptr(dst), _ptr(dst_sf), _stream(stream))


def mm_prepare_weight_scales(sf, rows, k, out, stream=None) -> int:
    """UE8M0 scales [rows, k/32] of a weight matrix -> the prepared layout that
    mm_forward takes for l1_sf / l2_sf (same byte count; see include/megamoe.h)."""
    return lib().mm_prepare_weight_scales(_ptr(sf), rows, k, _ptr(out), _stream(stream))


def prepare_weight_scales(sf, k, stream=None):
    """Torch convenience: a new tensor holding the prepared scales of `sf`
    (uint8, rows x k/32 bytes in any shape whose last dimension is k/32)."""
    import torch

    rows = sf.numel() // (k // 32)
    out = torch.empty_like(sf, memory_format=torch.contiguous_format)
    rc = mm_prepare_weight_scales(sf, rows, k, out, stream)
    if rc != MM_OK:
        raise MegaMoEError("mm_prepare_weight_scales", rc)
    return out


def mm_forward_noalloc(num_tokens, experts, topk, hidden, inter, x, x_sf, topk_idx, topk_w, l1_w, l1_sf,
                       l2_w, l2_sf, y, clamp, num_sms, stream=None) -> int:
    """mm_forward with the library's fixed 64 MiB device scratch as workspace,
    for callers that cannot allocate device memory (see include/megamoe.h);
    device-side errors are read with mm_noalloc_get_status."""
    return lib().mm_forward_noalloc(num_tokens, experts, topk, hidden, inter, _ptr(x), _ptr(x_sf),
                                    _ptr(topk_idx), _ptr(topk_w), _ptr(l1_w), _ptr(l1_sf), _ptr(l2_w),
                                    _ptr(l2_sf), _ptr(y), float(clamp), num_sms, _stream(stream))


def mm_noalloc_get_status(stream=None):
    """Status of the calls of mm_forward_noalloc on the current device: (status, sm, info)."""
    sm, info = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().mm_noalloc_get_status(_stream(stream), ctypes.addressof(sm), ctypes.addressof(info))
    return rc, sm.value, info.value


# ------------------------------------------------------------------ convenience
class MegaMoELayer:
    """Resident expert weights plus a caller-owned workspace (torch tensors).

    ``l1_sf`` / ``l2_sf`` are the UE8M0 scales as ``mm_quantize_mx`` writes
    them; the layer keeps its own prepared copies (mm_prepare_weight_scales).
    ``forward`` enqueues ``mm_forward`` on the current (or given) stream.  All
    arithmetic happens in the library's kernels.
    """

    def __init__(self, experts, topk, hidden, inter, l1_w, l1_sf, l2_w, l2_sf, max_tokens,
                 clamp=0.0, num_sms=0, device=None):
        import torch

        self.E, self.k, self.H, self.I = experts, topk, hidden, inter
        self.l1_w, self.l2_w = l1_w, l2_w
        self.l1_sf = prepare_weight_scales(l1_sf, hidden)
        self.l2_sf = prepare_weight_scales(l2_sf, inter)
        self.clamp, self.num_sms = clamp, num_sms
        self.max_tokens = max_tokens
        nbytes = mm_workspace_size(max_tokens, experts, topk, hidden, inter)
        if nbytes == 0:
            raise MegaMoEError("mm_workspace_size", MM_ERR_UNSUPPORTED_SHAPE)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device or l1_w.device)

    def forward(self, x, x_sf, topk_idx, topk_w, y=None, stream=None):
        import torch

        T = x.shape[0]
        if y is None:
            y = torch.empty(T, self.H, dtype=torch.bfloat16, device=x.device)
        rc = mm_forward(T, self.E, self.k, self.H, self.I, x, x_sf, topk_idx, topk_w, self.l1_w,
                        self.l1_sf, self.l2_w, self.l2_sf, y, self.clamp, self.num_sms, self.workspace,
                        stream=stream)
        if rc != MM_OK:
            raise MegaMoEError("mm_forward", rc)
        return y

    def status(self, stream=None):
        return mm_get_status(self.workspace, stream)
