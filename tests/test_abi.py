"""The C-ABI library: it loads, exports every entry point include/fwmoe.h
declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

import quantized_sparse_moe_router_gb300 as fw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    fw.build()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fwmoe.h")).read()
    return sorted(set(re.findall(r"^\s*(?:fw_status|const char \*)\s*(fw_\w+)\s*\(", src, re.M)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("fw_moe_init", "fw_moe_route", "fw_moe_ffn", "fw_moe_free", "fw_moe_last_error"):
        assert n in names
    assert set(names) == set(fw.EXPORTED)


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(fw.LIB_PATH)
    for n in declared_functions():
        assert hasattr(L, n), n


def _cfg(**kw):
    d = dict(H=256, I=128, E=8, k=2, n_shared=0, T_max=4, decode_T_max=0, act_q8=0)
    d.update(kw)
    return fw.FwMoeConfig(**d)


@pytest.mark.parametrize("bad, status", [
    (dict(H=96), fw.FW_EUNSUPPORTED), (dict(I=0), fw.FW_EUNSUPPORTED), (dict(E=0), fw.FW_EUNSUPPORTED),
    (dict(E=300), fw.FW_EUNSUPPORTED), (dict(k=0), fw.FW_EINVAL), (dict(k=9), fw.FW_EINVAL),
    (dict(k=17, E=32), fw.FW_EINVAL), (dict(n_shared=2), fw.FW_EINVAL), (dict(T_max=0), fw.FW_EINVAL),
    (dict(decode_T_max=17), fw.FW_EINVAL), (dict(act_q8=2), fw.FW_EINVAL),
])
def test_init_rejects_bad_config(bad, status):
    h = ctypes.c_void_p()
    w = fw.FwMoeWeights()
    rc = fw.lib().fw_moe_init(ctypes.byref(_cfg(**bad)), ctypes.byref(w), None, ctypes.byref(h))
    assert rc == status
    assert h.value is None
    assert fw.fw_moe_last_error()


def test_init_requires_weights():
    h = ctypes.c_void_p()
    w = fw.FwMoeWeights()
    assert fw.lib().fw_moe_init(ctypes.byref(_cfg()), ctypes.byref(w), None, ctypes.byref(h)) == fw.FW_EINVAL
    w.router_w = w.w_gate = w.w_up = w.w_down = 4096
    rc = fw.lib().fw_moe_init(ctypes.byref(_cfg(n_shared=1)), ctypes.byref(w), None, ctypes.byref(h))
    assert rc == fw.FW_EINVAL and "shared" in fw.fw_moe_last_error()


def test_calls_on_a_non_handle_are_rejected():
    L = fw.lib()
    assert L.fw_moe_route(None, None, 1, None, None, None) == fw.FW_EINVAL
    assert L.fw_moe_ffn(12345, None, 1, None, None) == fw.FW_EINVAL
    assert L.fw_moe_get_permutation(None, None, None, None, None) == fw.FW_EINVAL
    assert L.fw_moe_status(None, None) == fw.FW_EINVAL
    assert L.fw_moe_free(None) == fw.FW_OK  # NULL is a no-op
    assert L.fw_moe_free(777) == fw.FW_EINVAL


def test_quantize_rejects_bad_sizes():
    L = fw.lib()
    assert L.fw_q8_0_quantize(4096, 2, 48, 4096, None) == fw.FW_EINVAL
    assert L.fw_q8_0_quantize(4096, -1, 64, 4096, None) == fw.FW_EINVAL
    assert L.fw_q8_0_quantize(4100, 2, 64, 4096, None) == fw.FW_EINVAL  # misaligned fp32 source
    assert L.fw_q8_0_quantize(None, 0, 64, None, None) == fw.FW_OK      # nothing to do


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(fw, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(fw, "_lib", None)
    with pytest.raises(ImportError):
        fw.lib()


def test_noalloc_router_rejects_bad_arguments_before_any_device_call():
    """fw_moe_route_noalloc checks sizes, pointers and alignment on the host
    (no CUDA call happens for these), and T = 0 is a no-op."""
    L = fw.lib()
    ok = dict(x=4096, T=1, H=2048, w=4096, b=None, E=128, k=8, ids=4096, g=4096)

    def call(**over):
        a = dict(ok, **over)
        return L.fw_moe_route_noalloc(a["x"], a["T"], a["H"], a["w"], a["b"], a["E"], a["k"], a["ids"], a["g"], None)

    assert call(T=17) == fw.FW_EINVAL and "T must be" in fw.fw_moe_last_error()
    assert call(T=-1) == fw.FW_EINVAL
    assert call(E=257) == fw.FW_EINVAL and call(E=0) == fw.FW_EINVAL
    assert call(k=0) == fw.FW_EINVAL and call(k=17, E=64) == fw.FW_EINVAL and call(k=9, E=8) == fw.FW_EINVAL
    assert call(H=6) == fw.FW_EINVAL and call(H=0) == fw.FW_EINVAL
    assert call(x=None) == fw.FW_EINVAL and call(w=None) == fw.FW_EINVAL and call(ids=None) == fw.FW_EINVAL
    assert call(x=4100) == fw.FW_EINVAL            # x needs 8-byte alignment
    assert call(w=4104) == fw.FW_EINVAL            # router_w needs 16-byte alignment
    assert call(ids=4098) == fw.FW_EINVAL and call(g=4098) == fw.FW_EINVAL and call(b=4098) == fw.FW_EINVAL
    assert "alignment" in fw.fw_moe_last_error()
    assert call(T=0, x=None, w=None, ids=None) == fw.FW_OK  # nothing to route


def test_graph_calls_reject_bad_arguments_on_the_host():
    L = fw.lib()
    g = ctypes.c_void_p()
    assert L.fw_moe_graph_create(None, 1, 1, None, None, None, None) == fw.FW_EINVAL
    assert L.fw_moe_graph_create(None, 0, 1, None, None, None, ctypes.byref(g)) == fw.FW_EINVAL
    assert g.value is None
    one = (ctypes.c_void_p * 1)(4096)
    rc = L.fw_moe_graph_create(one, 1, 1, one, one, one, ctypes.byref(g))
    assert rc == fw.FW_EINVAL and "not a live handle" in fw.fw_moe_last_error()
    assert L.fw_moe_graph_create(one, 1, 0, one, one, one, ctypes.byref(g)) == fw.FW_EINVAL
    assert L.fw_moe_graph_launch(None, None) == fw.FW_EINVAL
    assert L.fw_moe_graph_launch(777, None) == fw.FW_EINVAL  # checked against the live set, not read
    assert L.fw_moe_graph_destroy(None) == fw.FW_OK  # NULL is a no-op
    assert L.fw_moe_graph_destroy(777) == fw.FW_EINVAL
