"""ctypes front end of the fp64 C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
bench's CPU-baseline leg, never by the library. Arrays are numpy; all results
are fp64 (ids and permutation indices int32).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

Q8_0_BLOCK = 32
Q8_0_BYTES = 34


def build(force: bool = False) -> str:
    from ._build import build_oracle
    return build_oracle(force=force)


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = load(_LIB_PATH)
    return _lib


def load(path: str):
    """Load an oracle shared library and declare its C signatures."""
    L = ctypes.CDLL(path)
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_half_to_double.restype = ctypes.c_double
    L.oracle_double_to_half.argtypes = [ctypes.c_double]
    L.oracle_double_to_half.restype = ctypes.c_uint16
    L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_double.restype = ctypes.c_double
    L.oracle_q8_0_quantize.argtypes = [vp, i64, i64, vp]
    L.oracle_q8_0_quantize.restype = ctypes.c_int
    L.oracle_q8_0_dequantize.argtypes = [vp, i64, i64, vp]
    L.oracle_q8_0_dequantize.restype = ctypes.c_int
    L.oracle_router_logits.argtypes = [vp, i64, i64, vp, vp, i64, vp]
    L.oracle_router_logits.restype = None
    L.oracle_topk_gates.argtypes = [vp, i64, i64, i64, vp, vp]
    L.oracle_topk_gates.restype = None
    L.oracle_gates_full_softmax.argtypes = [vp, i64, i64, i64, vp, vp]
    L.oracle_gates_full_softmax.restype = None
    L.oracle_permutation.argtypes = [vp, i64, i64, i64, vp, vp, vp]
    L.oracle_permutation.restype = None
    L.oracle_expert_ffn.argtypes = [vp, vp, vp, i64, i64, vp, vp]
    L.oracle_expert_ffn.restype = None
    L.oracle_moe_forward.argtypes = [i64] * 6 + [vp] * 9
    L.oracle_moe_forward.restype = ctypes.c_int
    L.oracle_moe_experts.argtypes = [i64] * 6 + [vp] * 7
    L.oracle_q8_activations.argtypes = [vp, i64, i64, vp, vp, vp]
    L.oracle_q8_activations.restype = ctypes.c_int
    L.oracle_moe_experts_q8act.argtypes = [i64] * 6 + [vp] * 7
    L.oracle_moe_experts_q8act.restype = ctypes.c_int
    L.oracle_moe_experts.restype = ctypes.c_int
    return L


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def half_to_double(bits: int) -> float:
    return lib().oracle_half_to_double(bits)


def double_to_half(x: float) -> int:
    return lib().oracle_double_to_half(x)


def q8_0_quantize(w: np.ndarray) -> np.ndarray:
    """[rows, K] fp32 -> uint8 [rows, K/32*34] GGUF-style Q8_0 blocks."""
    w = _c(w, np.float32)
    rows, K = w.shape
    out = np.empty((rows, K // Q8_0_BLOCK * Q8_0_BYTES), dtype=np.uint8)
    if lib().oracle_q8_0_quantize(_p(w), rows, K, _p(out)) != 0:
        raise ValueError("bad Q8_0 sizes")
    return out


def q8_0_dequantize(blocks: np.ndarray, rows: int, K: int) -> np.ndarray:
    blocks = _c(blocks, np.uint8)
    out = np.empty((rows, K), dtype=np.float64)
    if lib().oracle_q8_0_dequantize(_p(blocks), rows, K, _p(out)) != 0:
        raise ValueError("bad Q8_0 sizes")
    return out


def router_logits(x_bits: np.ndarray, Wr: np.ndarray, bias=None) -> np.ndarray:
    x_bits = _c(x_bits, np.uint16)
    Wr = _c(Wr, np.float32)
    T, H = x_bits.shape
    E = Wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    z = np.empty((T, E), dtype=np.float64)
    lib().oracle_router_logits(_p(x_bits), T, H, _p(Wr), _p(b), E, _p(z))
    return z


def topk_gates(z: np.ndarray, k: int):
    z = _c(z, np.float64)
    T, E = z.shape
    ids = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float64)
    lib().oracle_topk_gates(_p(z), T, E, k, _p(ids), _p(gates))
    return ids, gates


def gates_full_softmax(z: np.ndarray, ids: np.ndarray) -> np.ndarray:
    z = _c(z, np.float64)
    ids = _c(ids, np.int32)
    T, E = z.shape
    k = ids.shape[1]
    g = np.empty((T, k), dtype=np.float64)
    lib().oracle_gates_full_softmax(_p(z), T, E, k, _p(ids), _p(g))
    return g


def permutation(ids: np.ndarray, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    inv = np.empty(T * k, dtype=np.int32)
    lib().oracle_permutation(_p(ids), T, k, E, _p(offsets), _p(perm), _p(inv))
    return offsets, perm, inv


def expert_ffn(wg: np.ndarray, wu: np.ndarray, wd: np.ndarray, H: int, I: int, x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float64)
    y = np.empty(H, dtype=np.float64)
    lib().oracle_expert_ffn(_p(_c(wg, np.uint8)), _p(_c(wu, np.uint8)), _p(_c(wd, np.uint8)), H, I, _p(x), _p(y))
    return y


def _ptr_array(blocks_list):
    arr = (ctypes.c_void_p * len(blocks_list))()
    keep = []
    for i, b in enumerate(blocks_list):
        if b is None:
            arr[i] = None
        else:
            b = _c(b, np.uint8)
            keep.append(b)
            arr[i] = b.ctypes.data
    return arr, keep


def moe_forward(x_bits, Wr, bias, w_gate, w_up, w_down, k: int, S: int = 0):
    """Whole step. w_* are lists of E+S Q8_0 arrays (None allowed for experts no
    token selects). Returns (ids [T,k] int32, gates [T,k] fp64, out [T,H] fp64)."""
    x_bits = _c(x_bits, np.uint16)
    Wr = _c(Wr, np.float32)
    T, H = x_bits.shape
    E = Wr.shape[0]
    I = None
    for b in w_gate:
        if b is not None:
            I = b.size // (H // Q8_0_BLOCK * Q8_0_BYTES)
            break
    b = None if bias is None else _c(bias, np.float32)
    g_arr, k1 = _ptr_array(w_gate)
    u_arr, k2 = _ptr_array(w_up)
    d_arr, k3 = _ptr_array(w_down)
    ids = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float64)
    out = np.empty((T, H), dtype=np.float64)
    rc = lib().oracle_moe_forward(T, H, I, E, k, S, _p(x_bits), _p(Wr), _p(b), g_arr, u_arr, d_arr,
                                  _p(ids), _p(gates), _p(out))
    if rc != 0:
        raise ValueError(f"oracle_moe_forward failed: {rc}")
    return ids, gates, out


def q8_activations(v: np.ndarray, blk: int):
    """Q8 activations of fp32 v (1-D, len % blk == 0): (q*d fp64, q int8, d fp32 per block)."""
    v = _c(np.asarray(v, dtype=np.float32).ravel(), np.float32)
    n = v.size
    out = np.empty(n, dtype=np.float64)
    q = np.empty(n, dtype=np.int8)
    d = np.empty(max(n // blk, 1), dtype=np.float32)
    if lib().oracle_q8_activations(_p(v), n, blk, _p(out), _p(q), _p(d)) != 0:
        raise ValueError("oracle_q8_activations: bad sizes")
    return out, q, d[:n // blk]


def moe_experts(x_bits, ids, gates, w_gate, w_up, w_down, E: int, S: int = 0, act_q8: bool = False):
    """Expert part only, from given routing (act_q8: with Q8 activations). Returns out [T,H] fp64."""
    x_bits = _c(x_bits, np.uint16)
    ids = _c(ids, np.int32)
    gates = _c(gates, np.float64)
    T, H = x_bits.shape
    k = ids.shape[1]
    I = None
    for b in w_gate:
        if b is not None:
            I = b.size // (H // Q8_0_BLOCK * Q8_0_BYTES)
            break
    g_arr, k1 = _ptr_array(w_gate)
    u_arr, k2 = _ptr_array(w_up)
    d_arr, k3 = _ptr_array(w_down)
    out = np.empty((T, H), dtype=np.float64)
    fn = lib().oracle_moe_experts_q8act if act_q8 else lib().oracle_moe_experts
    rc = fn(T, H, I, E, k, S, _p(x_bits), _p(ids), _p(gates), g_arr, u_arr, d_arr, _p(out))
    if rc != 0:
        raise ValueError(f"oracle_moe_experts failed: {rc}")
    return out
