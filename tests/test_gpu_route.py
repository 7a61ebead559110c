"""GPU parity of the tiled router and the grouping (the path taken for T > 16):
ids, gates and the permutation against the oracle, over ragged tails, many
tiles, Zipf-skewed loads and ties."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle
import quantized_sparse_moe_router_gb300 as fw
import synth
from layer_inputs import GATE_TOL, DeviceLayer, OracleLayer, hidden_with_margins, to_device_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
# Gates from fp32-accurate logits: the decode router sums fp32 FMAs; the
# prefill router adds exact bf16-plane products in a tensor-core fp32
# accumulator over H/16 x 3 steps. Either stays far below the 1e-3 logit
# margin of the inputs (ids bit-exact); GATE_TOL is the suite's gate bound.


def route_and_check(wl, x, dl, ol, layer):
    T = x.shape[0]
    gates = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
    ids, _ = layer.route(to_device_bf16(x, DEV), gates=gates)
    torch.cuda.synchronize()
    ids_ref, gates_ref = ol.route(x)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.abs(gates.cpu().numpy() - gates_ref).max() <= GATE_TOL
    off, perm, inv = layer.permutation(T)
    o_ref, p_ref, i_ref = oracle.permutation(ids_ref, wl.E)
    assert np.array_equal(off.cpu().numpy(), o_ref)
    assert np.array_equal(perm.cpu().numpy(), p_ref)
    assert np.array_equal(inv.cpu().numpy(), i_ref)
    layer.status()
    return ids_ref


@pytest.mark.parametrize("T", [17, 33, 129, 1000])
@pytest.mark.parametrize("E, k", [(8, 2), (64, 8), (256, 8), (40, 5), (48, 12), (128, 16), (192, 6)])
def test_tiled_router_small(T, E, k):
    wl = synth.WORKLOADS["tiny"].with_(E=E, k=k, T=T, sigma_router=0.1)
    dl = DeviceLayer(wl, 0, DEV)
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    layer = dl.make(T_max=T)
    route_and_check(wl, x, dl, ol, layer)
    layer.close()


def test_router_prefill_full_size_zipf():
    """The 4096-token prefill workload: routing over all tokens, Zipf(1.1) skew."""
    wl = synth.WORKLOADS["pre4096"]
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    dl = DeviceLayer(wl.with_(E=wl.E), 0, DEV)
    layer = dl.make(T_max=wl.T)
    ids = route_and_check(wl, x, dl, ol, layer)
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    assert counts.max() > 8 * counts.mean()  # the skew is there
    layer.close()


@pytest.mark.parametrize("E, k", [(64, 8), (48, 12)])
def test_router_ties_tiled(E, k):
    wl = synth.WORKLOADS["tiny"].with_(E=E, k=k, T=100)
    dl = DeviceLayer(wl, 0, DEV, Wr=np.zeros((E, wl.H), np.float32))
    layer = dl.make(T_max=100)
    x = synth.hidden_bf16_bits(wl, 0)
    ids, _ = layer.route(to_device_bf16(x, DEV))
    assert ids.cpu().numpy().tolist() == [list(range(k))] * 100
    off, perm, inv = layer.permutation(100)
    o_ref, p_ref, _ = oracle.permutation(np.tile(np.arange(k, dtype=np.int32), (100, 1)), E)
    assert np.array_equal(off.cpu().numpy(), o_ref) and np.array_equal(perm.cpu().numpy(), p_ref)
    layer.close()
