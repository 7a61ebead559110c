"""Independent brute-force references used to pin the oracle (numpy only).

Nothing here calls or imports the oracle or the CUDA library. Q8_0 blocks are
parsed with numpy's own binary16 type; the FFN is evaluated densely for all E
experts and mixed with a length-E mask of gates; selection is a full
lexicographic sort.
"""
import numpy as np


def parse_q8_0(blocks: np.ndarray, rows: int, K: int) -> np.ndarray:
    """GGUF Q8_0 bytes [rows, K/32*34] -> fp64 weights [rows, K] (numpy float16 scales)."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(rows, K // 32, 34)
    d = b[:, :, 0:2].copy().view(np.float16).astype(np.float64)  # [rows, K/32, 1], little-endian
    q = b[:, :, 2:].copy().view(np.int8).astype(np.float64)      # [rows, K/32, 32]
    return (d * q).reshape(rows, K)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def sort_select(z: np.ndarray, k: int) -> np.ndarray:
    """ids [T,k]: full sort by (-z, id)."""
    T, E = z.shape
    ids = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = np.lexsort((np.arange(E), -z[t]))
        ids[t] = order[:k]
    return ids


def dense_masked_moe(X, Wg, Wu, Wd, mask, shared=None):
    """All E experts evaluated densely for every token, mixed by mask [T, E].

    X [T,H] fp64; Wg, Wu [E, I, H]; Wd [E, H, I]; shared = (Wg_s, Wu_s, Wd_s) or None."""
    T = X.shape[0]
    E = Wg.shape[0]
    out = np.zeros((T, Wd.shape[1]))
    for e in range(E):
        G = X @ Wg[e].T
        U = X @ Wu[e].T
        A = G / (1.0 + np.exp(-G)) * U
        Y = A @ Wd[e].T
        out += mask[:, e:e + 1] * Y
    if shared is not None:
        g_s, u_s, d_s = shared
        G = X @ g_s.T
        U = X @ u_s.T
        out += (G / (1.0 + np.exp(-G)) * U) @ d_s.T
    return out
