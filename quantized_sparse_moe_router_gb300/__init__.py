"""Python binding of libfwmoe.so (include/fwmoe.h): argument marshalling only.

Every step of the routed MoE feed-forward runs in the library's CUDA kernels;
PyTorch only provides device memory and the current stream. The binding does
not fall back to anything: if the library is missing it raises.

Low level: the C entry points under their own names (fw_moe_init, fw_moe_route,
fw_moe_ffn, fw_moe_forward, fw_moe_forward_host, fw_moe_get_permutation,
fw_moe_export_q8_0, fw_moe_status, fw_moe_free, fw_moe_last_error,
fw_q8_0_quantize), taking raw pointers and ints.

High level: `MoELayer` (one handle = one layer) and `quantize_q8_0`, taking
torch tensors.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfwmoe.so")

FW_OK, FW_EINVAL, FW_ENOMEM, FW_ECUDA, FW_EUNSUPPORTED, FW_ESTATE, FW_ETIMEOUT, FW_EDEVICE = 0, -1, -2, -3, -4, -5, -6, -7
STATUS_NAMES = {0: "FW_OK", -1: "FW_EINVAL", -2: "FW_ENOMEM", -3: "FW_ECUDA", -4: "FW_EUNSUPPORTED",
                -5: "FW_ESTATE", -6: "FW_ETIMEOUT", -7: "FW_EDEVICE"}


class FwMoeConfig(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("T_max", ctypes.c_int32), ("decode_T_max", ctypes.c_int32),
                ("act_q8", ctypes.c_int32)]


class FwMoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("router_w", "router_bias", "w_gate", "w_up", "w_down",
                                               "shared_gate", "shared_up", "shared_down")]


class FwError(RuntimeError):
    def __init__(self, status: int, where: str, text: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {text}")
        self.status = status


def build(force: bool = False) -> str:
    from ._build import build as _b
    return _b(force=force)


_lib = None

EXPORTED = ("fw_moe_init", "fw_moe_route", "fw_moe_ffn", "fw_moe_forward", "fw_moe_forward_host",
            "fw_moe_get_permutation", "fw_moe_export_q8_0", "fw_moe_status", "fw_moe_free", "fw_moe_last_error",
            "fw_q8_0_quantize", "fw_moe_profile_begin", "fw_moe_profile_end", "fw_moe_route_noalloc",
            "fw_moe_graph_create", "fw_moe_graph_launch", "fw_moe_graph_destroy")

KERNEL_KINDS = ("route_decode", "route_tiles", "route_scan", "route_scatter", "decode_experts", "reserved",
                "prefill_gateup", "prefill_down", "prefill_combine", "prefill_gather", "prefill_gateup_small",
                "prefill_down_small", "prefill_gateup_mid", "prefill_down_mid")


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with quantized_sparse_moe_router_gb300.build() "
                              "(nvcc, sm_103a); there is no fallback implementation")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        sig = {
            "fw_moe_init": [ctypes.POINTER(FwMoeConfig), ctypes.POINTER(FwMoeWeights), vp, ctypes.POINTER(vp)],
            "fw_moe_route": [vp, vp, i32, vp, vp, vp],
            "fw_moe_ffn": [vp, vp, i32, vp, vp],
            "fw_moe_forward": [vp, vp, i32, vp, vp, vp, vp],
            "fw_moe_forward_host": [vp, vp, i32, vp, vp, vp],
            "fw_moe_get_permutation": [vp, vp, vp, vp, vp],
            "fw_moe_export_q8_0": [vp, i32, i32, vp, vp],
            "fw_moe_status": [vp, vp],
            "fw_moe_free": [vp],
            "fw_q8_0_quantize": [vp, i64, i64, vp, vp],
            "fw_moe_profile_begin": [vp, i32],
            "fw_moe_profile_end": [vp, i32, vp, vp],
            "fw_moe_route_noalloc": [vp, i32, i32, vp, vp, i32, i32, vp, vp, vp],
            "fw_moe_graph_create": [vp, i32, i32, vp, vp, vp, ctypes.POINTER(vp)],
            "fw_moe_graph_launch": [vp, vp],
            "fw_moe_graph_destroy": [vp],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.fw_moe_last_error.argtypes = []
        L.fw_moe_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def fw_moe_last_error() -> str:
    return lib().fw_moe_last_error().decode()


def _check(rc: int, where: str):
    if rc != FW_OK:
        raise FwError(rc, where, fw_moe_last_error())


# Thin, same-named wrappers over the C entry points (raw pointers and ints).
def fw_moe_init(cfg: FwMoeConfig, weights: FwMoeWeights, stream: int) -> int:
    h = ctypes.c_void_p()
    _check(lib().fw_moe_init(ctypes.byref(cfg), ctypes.byref(weights), stream, ctypes.byref(h)), "fw_moe_init")
    return h.value


def fw_moe_route(h, x, T, expert_ids, gates, stream):
    _check(lib().fw_moe_route(h, x, T, expert_ids, gates, stream), "fw_moe_route")


def fw_moe_ffn(h, x, T, out, stream):
    _check(lib().fw_moe_ffn(h, x, T, out, stream), "fw_moe_ffn")


def fw_moe_forward(h, x, T, expert_ids, gates, out, stream):
    _check(lib().fw_moe_forward(h, x, T, expert_ids, gates, out, stream), "fw_moe_forward")


def fw_moe_forward_host(h, x_host, T, ids_host, out_host, stream):
    _check(lib().fw_moe_forward_host(h, x_host, T, ids_host, out_host, stream), "fw_moe_forward_host")


def fw_moe_get_permutation(h, offsets, perm, inv, stream):
    _check(lib().fw_moe_get_permutation(h, offsets, perm, inv, stream), "fw_moe_get_permutation")


def fw_moe_export_q8_0(h, expert, which, blocks, stream):
    _check(lib().fw_moe_export_q8_0(h, expert, which, blocks, stream), "fw_moe_export_q8_0")


def fw_moe_status(h, stream):
    _check(lib().fw_moe_status(h, stream), "fw_moe_status")


def fw_moe_free(h):
    _check(lib().fw_moe_free(h), "fw_moe_free")


def fw_moe_graph_create(handles, T, xs, outs, ids) -> int:
    """handles, xs, outs, ids: sequences of raw pointers (one per call)."""
    n = len(handles)
    arr = lambda seq: (ctypes.c_void_p * n)(*seq)
    g = ctypes.c_void_p()
    _check(lib().fw_moe_graph_create(arr(handles), n, T, arr(xs), arr(outs), arr(ids), ctypes.byref(g)),
           "fw_moe_graph_create")
    return g.value


def fw_moe_graph_launch(g, stream):
    _check(lib().fw_moe_graph_launch(g, stream), "fw_moe_graph_launch")


def fw_moe_graph_destroy(g):
    _check(lib().fw_moe_graph_destroy(g), "fw_moe_graph_destroy")


def fw_q8_0_quantize(w, rows, K, blocks, stream):
    _check(lib().fw_q8_0_quantize(w, rows, K, blocks, stream), "fw_q8_0_quantize")


def fw_moe_route_noalloc(x, T, H, router_w, router_bias, E, k, expert_ids, gates, stream):
    """Routing without a handle or any device allocation (see include/fwmoe.h)."""
    _check(lib().fw_moe_route_noalloc(x, T, H, router_w, router_bias, E, k, expert_ids, gates, stream),
           "fw_moe_route_noalloc")


def fw_moe_profile_begin(h, max_launches):
    _check(lib().fw_moe_profile_begin(h, max_launches), "fw_moe_profile_begin")


def fw_moe_profile_end(h):
    """-> {kind name: (total ms, launches)} for the kinds that launched."""
    n = 16
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int32 * n)()
    _check(lib().fw_moe_profile_end(h, n, ms, cnt), "fw_moe_profile_end")
    return {KERNEL_KINDS[i]: (ms[i], cnt[i]) for i in range(len(KERNEL_KINDS)) if cnt[i]}


# ------------------------------------------------------------ torch level
def _stream(stream=None) -> int:
    import torch
    return stream if stream is not None else torch.cuda.current_stream().cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def q8_0_bytes(rows: int, K: int) -> int:
    return rows * (K // 32) * 34


def quantize_q8_0(w, out=None, stream=None):
    """fp32 CUDA tensor [rows, K] -> uint8 CUDA tensor [rows, K/32*34] (GGUF Q8_0 blocks)."""
    import torch
    assert w.is_cuda and w.dtype == torch.float32 and w.is_contiguous() and w.dim() == 2
    rows, K = w.shape
    if out is None:
        out = torch.empty((rows, K // 32 * 34), dtype=torch.uint8, device=w.device)
    fw_q8_0_quantize(_ptr(w), rows, K, _ptr(out), _stream(stream))
    return out


class MoEGraph:
    """A chain of layer calls captured once as one CUDA graph and replayed by one
    launch (fw_moe_graph_* in include/fwmoe.h): call i is layers[i].forward of
    xs[i] into outs[i] with expert ids into ids[i] (outs[i] may be xs[i + 1])."""

    def __init__(self, layers, xs, outs, ids):
        T = xs[0].shape[0]
        self.graph = fw_moe_graph_create([L.handle for L in layers], T, [_ptr(x) for x in xs],
                                         [_ptr(o) for o in outs], [_ptr(i) for i in ids])
        self._keep = (list(layers), list(xs), list(outs), list(ids))  # the graph reads them at each launch

    def launch(self, stream=None):
        fw_moe_graph_launch(self.graph, _stream(stream))

    def close(self):
        if self.graph:
            g, self.graph = self.graph, None
            fw_moe_graph_destroy(g)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoELayer:
    """One routed-MoE layer: a handle of the C library.

    weights: dict of CUDA tensors: router_w fp32 [E, H], router_bias fp32 [E]
    or None, w_gate / w_up uint8 [E, I*H/32*34], w_down uint8 [E, H*I/32*34]
    (GGUF Q8_0 blocks), and shared_gate / shared_up / shared_down for
    n_shared == 1. The library copies what it needs: the tensors may be freed
    after construction.
    """

    def __init__(self, H, I, E, k, n_shared=0, T_max=16, decode_T_max=0, weights=None, stream=None, act_q8=False):
        self.H, self.I, self.E, self.k, self.S, self.T_max = H, I, E, k, n_shared, T_max
        cfg = FwMoeConfig(H, I, E, k, n_shared, T_max, decode_T_max, 1 if act_q8 else 0)
        w = FwMoeWeights()
        for name, _ in FwMoeWeights._fields_:
            t = weights.get(name) if weights else None
            setattr(w, name, _ptr(t))
        self.handle = fw_moe_init(cfg, w, _stream(stream))

    def route(self, x, expert_ids=None, gates=None, stream=None):
        import torch
        T = x.shape[0]
        if expert_ids is None:
            expert_ids = torch.empty((T, self.k), dtype=torch.int32, device=x.device)
        fw_moe_route(self.handle, _ptr(x), T, _ptr(expert_ids), _ptr(gates), _stream(stream))
        return expert_ids, gates

    def ffn(self, x, out=None, stream=None):
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device)
        fw_moe_ffn(self.handle, _ptr(x), T, _ptr(out), _stream(stream))
        return out

    def forward(self, x, expert_ids=None, gates=None, out=None, stream=None):
        import torch
        T = x.shape[0]
        if expert_ids is None:
            expert_ids = torch.empty((T, self.k), dtype=torch.int32, device=x.device)
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device)
        fw_moe_forward(self.handle, _ptr(x), T, _ptr(expert_ids), _ptr(gates), _ptr(out), _stream(stream))
        return expert_ids, out

    def forward_host(self, x_host, ids_host, out_host, stream=None):
        """Host (ideally pinned) CPU tensors in and out; synchronises the stream."""
        T = x_host.shape[0]
        fw_moe_forward_host(self.handle, _ptr(x_host), T, _ptr(ids_host), _ptr(out_host), _stream(stream))

    def permutation(self, T, stream=None):
        import torch
        dev = torch.device("cuda", torch.cuda.current_device())
        offsets = torch.empty(self.E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(max(T * self.k, 1), dtype=torch.int32, device=dev)
        inv = torch.empty(max(T * self.k, 1), dtype=torch.int32, device=dev)
        fw_moe_get_permutation(self.handle, _ptr(offsets), _ptr(perm), _ptr(inv), _stream(stream))
        return offsets, perm[:T * self.k], inv[:T * self.k]

    def export_q8_0(self, expert, which, stream=None):
        import torch
        rows, K = (self.I, self.H) if which in (0, 1) else (self.H, self.I)
        out = torch.empty((rows, K // 32 * 34), dtype=torch.uint8, device="cuda")
        fw_moe_export_q8_0(self.handle, expert, which, _ptr(out), _stream(stream))
        return out

    def status(self, stream=None):
        fw_moe_status(self.handle, _stream(stream))

    def close(self):
        if self.handle:
            h, self.handle = self.handle, None
            fw_moe_free(h)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
