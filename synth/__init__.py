"""Seeded synthetic inputs for the routed MoE feed-forward step.

This module is the one thing the test harness, the oracle side and the CUDA
side share: it turns (seed, stream, index) into input numbers and nothing
else. It holds none of the MoE arithmetic (no router, no quantiser, no FFN).

Workloads are the layer shapes the routed-MoE pages speak of (the Flyweight
README's Qwen/DeepSeek-shaped MoE families, §Features and §Quantization), with
synthetic seeded values in place of checkpoints:

  hidden states   bf16, N(0, 1)
  router weights  fp32, N(0, sigma_router)  [E, H] row-major
  expert weights  fp32, N(0, sigma_w): gate/up [I, H], down [H, I] row-major,
                  to be quantised to Q8_0 by whichever side consumes them
  router bias     optional fp32 [E]: b_e = -s * ln(r_e), r a seeded permutation
                  of 1..E (a Zipf(s) skew of the routing odds)

Normals are Irwin-Hall(12) deviates (see synth_rng.h), identical on host and
device.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfwsynth.so")
_lib = None

KIND_GATE, KIND_UP, KIND_DOWN, KIND_ROUTER, KIND_BIAS_PERM, KIND_X = 0, 1, 2, 3, 4, 5


def build(force: bool = False) -> str:
    """Compile libfwsynth.so in place (host + sm_103a device code)."""
    from ._build import build_synth
    return build_synth(force=force)


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            build()
        L = ctypes.CDLL(_LIB_PATH)
        u64, f32 = ctypes.c_uint64, ctypes.c_float
        vp = ctypes.c_void_p
        L.synth_normal_f32.argtypes = [u64, u64, u64, u64, f32, vp]
        L.synth_normal_f32.restype = None
        L.synth_normal_bf16.argtypes = [u64, u64, u64, u64, f32, vp]
        L.synth_normal_bf16.restype = None
        L.synth_u64_fill.argtypes = [u64, u64, u64, u64, vp]
        L.synth_u64_fill.restype = None
        L.synth_normal_f32_device.argtypes = [u64, u64, u64, u64, f32, vp, vp]
        L.synth_normal_f32_device.restype = ctypes.c_int
        L.synth_normal_bf16_device.argtypes = [u64, u64, u64, u64, f32, vp, vp]
        L.synth_normal_bf16_device.restype = ctypes.c_int
        _lib = L
    return _lib


def stream_id(layer: int, expert: int, kind: int, redraw: int = 0) -> int:
    """Independent stream per (layer, expert, tensor kind, redraw round)."""
    return (layer << 40) | (redraw << 24) | (expert << 8) | kind


# ---------------------------------------------------------------- host fills
def normal_f32(seed: int, stream: int, n: int, sigma: float, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().synth_normal_f32(seed, stream, offset, n, sigma, out.ctypes.data)
    return out


def normal_bf16_bits(seed: int, stream: int, n: int, sigma: float, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    lib().synth_normal_bf16(seed, stream, offset, n, sigma, out.ctypes.data)
    return out


def u64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    lib().synth_u64_fill(seed, stream, offset, n, out.ctypes.data)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


# -------------------------------------------------------------- device fills
def _dev_ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def fill_normal_f32_device(tensor, seed: int, stream: int, sigma: float, offset: int = 0, cuda_stream=None):
    """Fill a contiguous float32 CUDA tensor in place (torch used for memory only)."""
    import torch
    assert tensor.is_cuda and tensor.dtype == torch.float32 and tensor.is_contiguous()
    s = cuda_stream if cuda_stream is not None else torch.cuda.current_stream().cuda_stream
    rc = lib().synth_normal_f32_device(seed, stream, offset, tensor.numel(), sigma, _dev_ptr(tensor),
                                       ctypes.c_void_p(s))
    if rc != 0:
        raise RuntimeError(f"synth_normal_f32_device failed: cudaError {rc}")


def fill_normal_bf16_device(tensor, seed: int, stream: int, sigma: float, offset: int = 0, cuda_stream=None):
    import torch
    assert tensor.is_cuda and tensor.dtype in (torch.bfloat16, torch.int16, torch.uint16) and tensor.is_contiguous()
    s = cuda_stream if cuda_stream is not None else torch.cuda.current_stream().cuda_stream
    rc = lib().synth_normal_bf16_device(seed, stream, offset, tensor.numel(), sigma, _dev_ptr(tensor),
                                        ctypes.c_void_p(s))
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16_device failed: cudaError {rc}")


# ------------------------------------------------------------------ workloads
@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    I: int
    E: int
    k: int
    S: int            # shared (always-on) experts: 0 or 1
    T: int
    sigma_router: float
    sigma_w: float
    seed: int
    layers: int = 1
    zipf_s: float = 0.0   # 0: no router bias
    note: str = ""

    @property
    def n_experts_total(self) -> int:
        return self.E + self.S

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    "tiny": Workload("tiny", H=256, I=128, E=8, k=2, S=0, T=4, sigma_router=0.05, sigma_w=0.02,
                     seed=0xF00D0001, note="tiny MoE layer, top-2 of 8"),
    "dec1": Workload("dec1", H=2048, I=768, E=128, k=8, S=0, T=1, sigma_router=0.02, sigma_w=0.02,
                     seed=0xF00D0002, layers=48, note="decode batch-1, 48 layers cycled (working set > L2)"),
    "dec16": Workload("dec16", H=2048, I=768, E=128, k=8, S=0, T=16, sigma_router=0.02, sigma_w=0.02,
                      seed=0xF00D0003, layers=48, note="multi-slot decode, 16 sequence slots"),
    "pre4096": Workload("pre4096", H=2048, I=768, E=128, k=8, S=0, T=4096, sigma_router=0.02, sigma_w=0.02,
                        seed=0xF00D0004, layers=4, zipf_s=1.1, note="prefill chunk, Zipf(1.1)-skewed routing"),
    "large1": Workload("large1", H=7168, I=2048, E=256, k=8, S=1, T=1, sigma_router=0.01, sigma_w=0.01,
                       seed=0xF00D0005, layers=4, note="large MoE decode, 256 routed + 1 shared"),
    "large2048": Workload("large2048", H=7168, I=2048, E=256, k=8, S=1, T=2048, sigma_router=0.01,
                          sigma_w=0.01, seed=0xF00D0005, layers=2, note="large MoE prefill, 2048 tokens"),
}


# ----------------------------------------------------------- tensor recipes
def expert_weight_f32(w: Workload, layer: int, expert: int, kind: int) -> np.ndarray:
    """fp32 weights of one expert matrix: gate/up [I, H], down [H, I] (row-major)."""
    rows, cols = (w.I, w.H) if kind in (KIND_GATE, KIND_UP) else (w.H, w.I)
    return normal_f32(w.seed, stream_id(layer, expert, kind), rows * cols, w.sigma_w).reshape(rows, cols)


def router_weight_f32(w: Workload, layer: int) -> np.ndarray:
    return normal_f32(w.seed, stream_id(layer, 0, KIND_ROUTER), w.E * w.H, w.sigma_router).reshape(w.E, w.H)


def router_bias_f32(w: Workload, layer: int):
    """Zipf(s) routing skew: b_e = -s ln r_e with r a seeded permutation of 1..E; None if s == 0."""
    if w.zipf_s == 0.0:
        return None
    r = seeded_permutation(w.seed, stream_id(layer, 0, KIND_BIAS_PERM), w.E) + 1
    return (-w.zipf_s * np.log(r.astype(np.float64))).astype(np.float32)


def seeded_permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of 0..n-1 driven by the stream's 64-bit outputs."""
    draws = u64(seed, stream, n)
    p = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(draws[i] % np.uint64(i + 1))
        p[i], p[j] = p[j], p[i]
    return p


def hidden_bf16_bits(w: Workload, layer: int, T: int | None = None, redraw: int = 0) -> np.ndarray:
    """Hidden states [T, H] as bf16 bit patterns."""
    T = w.T if T is None else T
    return normal_bf16_bits(w.seed, stream_id(layer, 0, KIND_X, redraw), T * w.H, 1.0).reshape(T, w.H)


def hidden_row_bf16_bits(w: Workload, layer: int, t: int, redraw: int) -> np.ndarray:
    """Row t of the hidden-state stream of one redraw round."""
    return normal_bf16_bits(w.seed, stream_id(layer, 0, KIND_X, redraw), w.H, 1.0, offset=t * w.H)
