"""Seeded synthetic inputs for the fused MoE expert layer (shared by both sides).

This module only *draws* inputs.  It holds none of the layer's arithmetic:
no FP8/FP4 quantisation, no routing of tokens to experts, no matmul.  The
quantised bytes that the layer consumes are made by each side from the fp32
values drawn here (the CPU oracle with its own quantiser, the GPU path with
its own kernel), so the two sides never share a code path.

Generator (see synth.h for the exact definition): SplitMix64 streams keyed
by (seed, tensor id); each 16-bit field of a stream output indexes a table
of standard-normal quantiles.  The host build (synth_cpu.c) and the device
build (synth_gpu.cu) compile the same header, so both produce identical fp32
values.

Workload recipe (the configurations of the fused MegaMoE expert layer on the
pages "[Blackwell] Reserve SMs for DeepGEMM MegaMoE grid barriers", Summary /
Fix, and the DeepGEMM FP8 x FP4 MegaMoE call (per-32 recipe, SwiGLU with an
activation clamp) shown on the digest of the same PR, section 关键源码片段):

* x  ~ N(0, 1)           [T, H]        tensor id 1
* W1 ~ N(0, 1/sqrt(H))   [E, 2I, H]    tensor id 2   (rows [0, I) gate, [I, 2I) up)
* W2 ~ N(0, 1/sqrt(I))   [E, H, I]     tensor id 3
* gate logits z ~ N(0,1) [T, E]        tensor id 4; softmax, top-k (ties to the
  lower expert id), weights renormalised to sum 1.
* skewed routing adds b_e = -1.2 * log(r_e), r a seeded permutation of 1..E
  (tensor id 5), doubled until some expert gets no token and one gets more
  than 10x the mean.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")

TENSOR_X = 1
TENSOR_W1 = 2
TENSOR_W2 = 3
TENSOR_LOGITS = 4
TENSOR_PERM = 5

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
STREAM_MULT = 0xD1B54A32D192ED03


# --------------------------------------------------------------------------
# configurations
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Config:
    name: str
    T: int            # tokens
    H: int            # hidden
    I: int            # intermediate per expert
    E: int            # experts
    k: int            # top-k
    clamp: float      # swiglu clamp; 0.0 = no clamp
    skew: bool = False
    seed: int = 0
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def assignments(self) -> int:
        return self.T * self.k

    def flops(self) -> int:
        """Algorithmic FLOPs: 2*H*2I (gate/up) + 2*I*H (down) per assignment."""
        return self.assignments * (2 * self.H * 2 * self.I + 2 * self.I * self.H)

    def expert_bytes(self) -> int:
        """FP4 weights + UE8M0/32 scales of one expert (L1 and L2)."""
        H, I = self.H, self.I
        return 2 * I * H // 2 + 2 * I * H // 32 + H * I // 2 + H * I // 32


CONFIGS = {
    "tiny": Config("tiny", T=64, H=256, I=128, E=8, k=2, clamp=7.0),
    "decode": Config("decode", T=128, H=7168, I=2048, E=256, k=8, clamp=7.0),
    "prefill": Config("prefill", T=8192, H=7168, I=2048, E=256, k=8, clamp=7.0),
    "skew": Config("skew", T=4096, H=7168, I=2048, E=256, k=8, clamp=0.0, skew=True),
    "kimi": Config("kimi", T=16384, H=7168, I=2048, E=384, k=8, clamp=10.0),
}


# --------------------------------------------------------------------------
# reference definition in pure Python (used only to pin the C/CUDA builds)
# --------------------------------------------------------------------------
def mix64(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def key_of(seed: int, tensor_id: int) -> int:
    return mix64((seed * GOLDEN + tensor_id * STREAM_MULT + 1) & MASK64)


def index16_py(seed: int, tensor_id: int, i: int) -> int:
    w = mix64(key_of(seed, tensor_id) + ((i >> 2) + 1) * GOLDEN)
    return (w >> (16 * (i & 3))) & 0xFFFF


# --------------------------------------------------------------------------
# quantile table
# --------------------------------------------------------------------------
_TABLE = None


def normal_table() -> np.ndarray:
    """table[j] = fp32(Phi^-1((j + 0.5) / 65536)), j < 65536."""
    global _TABLE
    if _TABLE is None:
        from scipy.special import ndtri

        j = np.arange(65536, dtype=np.float64)
        _TABLE = np.ascontiguousarray(ndtri((j + 0.5) / 65536.0).astype(np.float32))
    return _TABLE


# --------------------------------------------------------------------------
# host build (C, OpenMP)
# --------------------------------------------------------------------------
_CPU_LIB = None


def build_cpu(force: bool = False) -> str:
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, "libsynth_cpu.so")
    src = os.path.join(_HERE, "synth_cpu.c")
    hdr = os.path.join(_HERE, "synth.h")
    if force or not os.path.exists(out) or os.path.getmtime(out) < max(
        os.path.getmtime(src), os.path.getmtime(hdr)
    ):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
             src, "-o", tmp]
        )
        os.replace(tmp, out)
    return out


def _cpu():
    global _CPU_LIB
    if _CPU_LIB is None:
        lib = ctypes.CDLL(build_cpu())
        lib.synth_normal_f32.argtypes = [ctypes.c_uint64] * 4 + [
            ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_normal_f32.restype = None
        lib.synth_u64.argtypes = [ctypes.c_uint64] * 4 + [ctypes.c_void_p]
        lib.synth_u64.restype = None
        _CPU_LIB = lib
    return _CPU_LIB


def normal_f32(seed: int, tensor_id: int, start: int, n: int, scale: float = 1.0) -> np.ndarray:
    """Elements [start, start+n) of the stream (seed, tensor_id), host build."""
    out = np.empty(n, dtype=np.float32)
    if n:
        t = normal_table()
        _cpu().synth_normal_f32(seed, tensor_id, start, n, np.float32(scale).item(),
                                t.ctypes.data, out.ctypes.data)
    return out


def u64(seed: int, tensor_id: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    if n:
        _cpu().synth_u64(seed, tensor_id, start, n, out.ctypes.data)
    return out


def weight_scale(fan_in: int) -> float:
    """fp32(1/sqrt(K)): the standard deviation of a weight with fan-in K."""
    return float(np.float32(1.0 / math.sqrt(fan_in)))


# --------------------------------------------------------------------------
# per-tensor helpers (host)
# --------------------------------------------------------------------------
def x_f32(cfg: Config, seed: int | None = None, rows=None) -> np.ndarray:
    s = cfg.seed if seed is None else seed
    if rows is None:
        return normal_f32(s, TENSOR_X, 0, cfg.T * cfg.H).reshape(cfg.T, cfg.H)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((len(rows), cfg.H), dtype=np.float32)
    for n, t in enumerate(rows):
        out[n] = normal_f32(s, TENSOR_X, int(t) * cfg.H, cfg.H)
    return out


def w1_f32(cfg: Config, e: int) -> np.ndarray:
    n = 2 * cfg.I * cfg.H
    return normal_f32(cfg.seed, TENSOR_W1, e * n, n, weight_scale(cfg.H)).reshape(2 * cfg.I, cfg.H)


def w2_f32(cfg: Config, e: int) -> np.ndarray:
    n = cfg.H * cfg.I
    return normal_f32(cfg.seed, TENSOR_W2, e * n, n, weight_scale(cfg.I)).reshape(cfg.H, cfg.I)


# --------------------------------------------------------------------------
# routing inputs (gate + top-k are *inputs* of the layer; drawn here)
# --------------------------------------------------------------------------
def _topk(logits: np.ndarray, k: int):
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]
    w = np.take_along_axis(p, order, axis=1)
    w = w / w.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def routing(cfg: Config, seed: int | None = None):
    """Return (topk_idx int32 [T,k], topk_w f32 [T,k], bias_factor)."""
    s = cfg.seed if seed is None else seed
    T, E, k = cfg.T, cfg.E, cfg.k
    if T == 0:
        return np.zeros((0, k), np.int32), np.zeros((0, k), np.float32), 0.0
    z = normal_f32(s, TENSOR_LOGITS, 0, T * E).reshape(T, E).astype(np.float64)
    if not cfg.skew:
        idx, w = _topk(z, k)
        return idx, w, 0.0
    keys = u64(s, TENSOR_PERM, 0, E)
    r = np.empty(E, dtype=np.float64)
    r[np.argsort(keys, kind="stable")] = np.arange(1, E + 1, dtype=np.float64)
    bias = -1.2 * np.log(r)
    factor = 1.0
    mean = T * k / E
    for _ in range(16):
        idx, w = _topk(z + factor * bias, k)
        counts = np.bincount(idx.reshape(-1), minlength=E)
        if counts.min() == 0 and counts.max() > 10 * mean:
            return idx, w, factor
        factor *= 2.0
    raise RuntimeError("skewed routing recipe did not converge")


# --------------------------------------------------------------------------
# device build (CUDA) -- used by the GPU side only
# --------------------------------------------------------------------------
_GPU_LIB = None
_GPU_TABLES = {}


def build_gpu(force: bool = False, arch: str = "103a") -> str:
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, "libsynth_gpu.so")
    src = os.path.join(_HERE, "synth_gpu.cu")
    hdr = os.path.join(_HERE, "synth.h")
    if force or not os.path.exists(out) or os.path.getmtime(out) < max(
        os.path.getmtime(src), os.path.getmtime(hdr)
    ):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["nvcc", f"-gencode=arch=compute_{arch},code=sm_{arch}", "-O3", "-fmad=false",
             "-Xcompiler", "-fPIC", "-shared", src, "-o", tmp]
        )
        os.replace(tmp, out)
    return out


def _gpu():
    global _GPU_LIB
    if _GPU_LIB is None:
        lib = ctypes.CDLL(build_gpu())
        lib.synth_normal_f32_cuda.argtypes = [ctypes.c_uint64] * 4 + [
            ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_normal_f32_cuda.restype = ctypes.c_int
        _GPU_LIB = lib
    return _GPU_LIB


def normal_f32_cuda(seed: int, tensor_id: int, start: int, out, scale: float = 1.0, stream=None):
    """Fill the contiguous float32 CUDA tensor `out` with elements [start, start+numel)."""
    import torch

    dev = out.device
    tab = _GPU_TABLES.get(dev)
    if tab is None:
        tab = torch.from_numpy(normal_table()).to(dev)
        _GPU_TABLES[dev] = tab
    assert out.dtype == torch.float32 and out.is_contiguous()
    s = torch.cuda.current_stream(dev) if stream is None else stream
    rc = _gpu().synth_normal_f32_cuda(seed, tensor_id, start, out.numel(),
                                      np.float32(scale).item(), tab.data_ptr(),
                                      out.data_ptr(), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_normal_f32_cuda failed: cudaError {rc}")
    return out
