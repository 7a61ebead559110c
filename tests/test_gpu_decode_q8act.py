"""Q8 activations on the decode path (act_q8; the Flyweight README's
Q8-activation decode kernels, read as the Q8_0 rule on x per 32-block and on
h per 16-block, in fp32): parity with the oracle's Q8-activation step through
the C ABI -- ids bit-exact, gates within GATE_TOL, outputs within
1e-2 * max|oracle| + 1e-3 -- and, past the decode path, the unchanged
bf16-activation step."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle
import quantized_sparse_moe_router_gb300 as fw
import synth
from layer_inputs import GATE_TOL, DeviceLayer, OracleLayer, hidden_with_margins, to_device_bf16, tolerance

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def built():
    fw.build()
    torch.cuda.set_device(0)


CASES = [
    ("tiny", dict(T=1)),
    ("tiny", dict(T=4)),
    ("tiny", dict(T=16, k=8)),
    ("tiny", dict(T=5, S=1)),
    ("tiny", dict(T=1, H=4160, I=192)),       # one token, three down stages
    ("tiny", dict(T=16, E=32, k=16, S=1)),
    ("dec1", {}),
    ("dec16", {}),
    ("large1", dict(E=32)),                   # the large layer's shapes, fewer routed experts
]


@pytest.mark.parametrize("name, over", CASES, ids=[f"{n}-{'-'.join(f'{k}{v}' for k, v in o.items())}" for n, o in CASES])
def test_decode_q8act_parity(name, over):
    wl = synth.WORKLOADS[name].with_(**over)
    dl = DeviceLayer(wl, 0, DEV)
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    layer = dl.make(T_max=16, act_q8=True)
    xd = to_device_bf16(x, DEV)
    gates = torch.empty((wl.T, wl.k), dtype=torch.float32, device=DEV)
    ids, out = layer.forward(xd, gates=gates)
    torch.cuda.synchronize()
    layer.status()
    ids_ref, gates_ref = ol.route(x)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.abs(gates.cpu().numpy() - gates_ref).max() <= GATE_TOL
    g, u, d = ol.lists_for(ids_ref)
    out_ref = oracle.moe_experts(x, ids_ref, gates_ref, g, u, d, E=wl.E, S=wl.S, act_q8=True)
    got = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - out_ref).max()
    assert err <= tolerance(out_ref), f"max|err| {err} > {tolerance(out_ref)}"
    # the bf16-activation step differs from it by more than this error (the option is in effect)
    out_bf16 = oracle.moe_experts(x, ids_ref, gates_ref, g, u, d, E=wl.E, S=wl.S)
    assert np.abs(out_bf16 - out_ref).max() > err
    ids2, out2 = layer.forward(xd)
    assert torch.equal(ids, ids2) and torch.equal(out, out2)
    layer.close()


def test_q8act_leaves_the_prefill_path_in_bf16():
    wl = synth.WORKLOADS["tiny"].with_(T=40)
    dl = DeviceLayer(wl, 0, DEV)
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    layer = dl.make(T_max=64, act_q8=True)
    ids, out = layer.forward(to_device_bf16(x, DEV))
    torch.cuda.synchronize()
    ids_ref, _, out_ref = ol.forward(x)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.abs(out.float().cpu().numpy().astype(np.float64) - out_ref).max() <= tolerance(out_ref)
    layer.close()
