"""fw_moe_route_noalloc: routing for callers that must not allocate device
memory (a framework's memory manager owns the whole device, or a latency path
cannot take cudaMalloc's synchronisation). Its scratch is a static device
array inside the library; this checks, through the C ABI, that two calls in a
row give the fp64 oracle's ids (bit-exact) and gates (within the suite's gate
bound), and the same as the handle-based fw_moe_route, and that sizes beyond
the array are refused. Collected last on purpose."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import quantized_sparse_moe_router_gb300 as fw
import synth
from layer_inputs import GATE_TOL, DeviceLayer, OracleLayer, hidden_with_margins, to_device_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.mark.parametrize("name, over", [("tiny", dict(T=4)), ("dec16", {}), ("tiny", dict(T=16, E=256, k=8))])
def test_noalloc_route_matches_handle_route_twice(name, over):
    fw.build()
    torch.cuda.set_device(0)
    wl = synth.WORKLOADS[name].with_(**over)
    dl = DeviceLayer(wl, 0, DEV)
    ol = OracleLayer(wl, 0)
    layer = dl.make(T_max=wl.T)
    sp = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # two calls in a row share (and reuse) the static scratch
        x = hidden_with_margins(wl, call, ol.Wr, ol.bias)
        xd = to_device_bf16(x, DEV)
        g_ref = torch.empty((wl.T, wl.k), dtype=torch.float32, device=DEV)
        ids_ref, _ = layer.route(xd, gates=g_ref)
        ids = torch.full((wl.T, wl.k), -1, dtype=torch.int32, device=DEV)
        gates = torch.full((wl.T, wl.k), -1.0, dtype=torch.float32, device=DEV)
        bias_ptr = None if dl.router_bias is None else dl.router_bias.data_ptr()
        fw.fw_moe_route_noalloc(xd.data_ptr(), wl.T, wl.H, dl.router_w.data_ptr(), bias_ptr, wl.E, wl.k,
                                ids.data_ptr(), gates.data_ptr(), sp)
        torch.cuda.synchronize()
        ids_o, gates_o = ol.route(x)  # the oracle's routing of the same rows
        assert np.array_equal(ids.cpu().numpy(), ids_o)
        assert np.abs(gates.cpu().numpy() - gates_o).max() <= GATE_TOL
        assert torch.equal(ids, ids_ref)
        assert (gates - g_ref).abs().max().item() <= GATE_TOL
    layer.close()


def test_noalloc_route_refuses_sizes_beyond_its_scratch():
    fw.build()
    L = fw.lib()
    assert L.fw_moe_route_noalloc(4096, 17, 256, 4096, None, 8, 2, 4096, None, None) == fw.FW_EINVAL
    assert "16" in fw.fw_moe_last_error()
    assert L.fw_moe_route_noalloc(4096, 4, 256, 4096, None, 257, 2, 4096, None, None) == fw.FW_EINVAL
    assert L.fw_moe_route_noalloc(4096, 0, 256, 4096, None, 8, 2, 4096, None, None) == fw.FW_OK

