"""Chains of layer calls captured as one CUDA graph through the C ABI
(fw_moe_graph_create / launch): the replay gives the same bits as the same
calls made directly, on the decode and the prefill path, follows new input
contents from one launch to the next, and the first layer of the chain
matches the fp64 oracle (ids bit-exact, outputs within the suite's bound)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import quantized_sparse_moe_router_gb300 as fw
import synth
from layer_inputs import DeviceLayer, OracleLayer, hidden_with_margins, to_device_bf16, tolerance

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def built():
    fw.build()
    torch.cuda.set_device(0)


def direct_chain(layers, x, T, H, k):
    """The same calls made one by one: each layer's output is the next one's input."""
    outs, ids = [], []
    cur = x
    for L in layers:
        i = torch.empty((T, k), dtype=torch.int32, device=DEV)
        o = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        L.forward(cur, expert_ids=i, out=o)
        outs.append(o)
        ids.append(i)
        cur = o
    return ids, outs


@pytest.mark.parametrize("name, over", [("tiny", dict(T=4)), ("tiny", dict(T=1, S=1)), ("tiny", dict(T=40)),
                                        ("tiny", dict(T=16, S=1))])
def test_graph_chain_matches_direct_calls_and_oracle(name, over):
    wl = synth.WORKLOADS[name].with_(**over)
    n = 3
    dls = [DeviceLayer(wl, l, DEV) for l in range(n)]
    layers = [d.make(T_max=max(wl.T, 16)) for d in dls]
    ol0 = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol0.Wr, ol0.bias)
    bufs = [to_device_bf16(x, DEV)] + [torch.zeros((wl.T, wl.H), dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    ids = [torch.full((wl.T, wl.k), -1, dtype=torch.int32, device=DEV) for _ in range(n)]
    g = fw.MoEGraph(layers, bufs[:n], bufs[1:], ids)
    g.launch()
    torch.cuda.synchronize()
    for L in layers:
        L.status()
    ids_d, outs_d = direct_chain(layers, bufs[0], wl.T, wl.H, wl.k)
    torch.cuda.synchronize()
    for i in range(n):
        assert torch.equal(ids[i], ids_d[i]), f"layer {i}: ids differ from the direct call"
        assert torch.equal(bufs[i + 1], outs_d[i]), f"layer {i}: output differs from the direct call"
    ids_ref, _, out_ref = ol0.forward(x)
    assert np.array_equal(ids[0].cpu().numpy(), ids_ref)
    got = bufs[1].float().cpu().numpy().astype(np.float64)
    assert np.abs(got - out_ref).max() <= tolerance(out_ref)
    # new contents in the chain's input: the next launch reads them
    x2 = hidden_with_margins(wl, 1, ol0.Wr, ol0.bias)
    bufs[0].copy_(to_device_bf16(x2, DEV))
    g.launch()
    g.launch()  # a replay after a replay: the handles' workspaces are reused in order
    torch.cuda.synchronize()
    ids_d, outs_d = direct_chain(layers, bufs[0], wl.T, wl.H, wl.k)
    torch.cuda.synchronize()
    for i in range(n):
        assert torch.equal(ids[i], ids_d[i]) and torch.equal(bufs[i + 1], outs_d[i])
    ids_ref2, _, out_ref2 = ol0.forward(x2)
    assert np.array_equal(ids[0].cpu().numpy(), ids_ref2)
    assert np.abs(bufs[1].float().cpu().numpy().astype(np.float64) - out_ref2).max() <= tolerance(out_ref2)
    g.close()
    for L in layers:
        L.close()


def test_graph_refuses_a_profiling_layer():
    wl = synth.WORKLOADS["tiny"].with_(T=4)
    layer = DeviceLayer(wl, 0, DEV).make(T_max=16)
    x = torch.zeros((4, wl.H), dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(x)
    ids = torch.empty((4, wl.k), dtype=torch.int32, device=DEV)
    fw.fw_moe_profile_begin(layer.handle, 64)
    with pytest.raises(fw.FwError) as ei:
        fw.MoEGraph([layer], [x], [out], [ids])
    assert ei.value.status == fw.FW_ESTATE
    fw.fw_moe_profile_end(layer.handle)
    layer.close()


def test_graph_of_q8_activation_layers_matches_direct_calls():
    """The graph captures whatever each layer does: Q8-activation decode layers replay bit for bit."""
    wl = synth.WORKLOADS["tiny"].with_(T=3, S=1)
    n = 2
    layers = [DeviceLayer(wl, l, DEV).make(T_max=16, act_q8=True) for l in range(n)]
    ol0 = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol0.Wr, ol0.bias)
    bufs = [to_device_bf16(x, DEV)] + [torch.zeros((wl.T, wl.H), dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    ids = [torch.empty((wl.T, wl.k), dtype=torch.int32, device=DEV) for _ in range(n)]
    g = fw.MoEGraph(layers, bufs[:n], bufs[1:], ids)
    g.launch()
    torch.cuda.synchronize()
    ids_d, outs_d = direct_chain(layers, bufs[0], wl.T, wl.H, wl.k)
    torch.cuda.synchronize()
    for i in range(n):
        assert torch.equal(ids[i], ids_d[i]) and torch.equal(bufs[i + 1], outs_d[i])
    g.close()
    for L in layers:
        L.close()
