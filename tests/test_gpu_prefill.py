"""GPU parity of the prefill path (T > decode limit: tiled router, grouping,
gather, tcgen05 grouped GEMMs with in-shared-memory Q8_0 dequantisation,
combine) against the fp64 oracle, through the C ABI.

Same bar as the decode path: ids and permutation bit-exact, outputs within
1e-2 * max|oracle| + 1e-3. At the full workload sizes the oracle checks a
sample of tokens (all of the routing is still checked)."""
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


def run_layer(wl, x, decode_T_max=0, T_max=None):
    dl = DeviceLayer(wl, 0, DEV)
    layer = dl.make(T_max=T_max or x.shape[0], decode_T_max=decode_T_max)
    T = x.shape[0]
    gates = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
    ids, out = layer.forward(to_device_bf16(x, DEV), gates=gates)
    torch.cuda.synchronize()
    layer.status()
    perm = layer.permutation(T)
    res = (ids.cpu().numpy(), gates.cpu().numpy(), out.float().cpu().numpy().astype(np.float64),
           [p.cpu().numpy() for p in perm])
    layer.close()
    return dl, res


def check(wl, x, res, ol, sample=None):
    ids, gates, out, (off, perm, inv) = res
    ids_ref, gates_ref = ol.route(x)
    assert np.array_equal(ids, ids_ref)
    assert np.abs(gates - gates_ref).max() <= GATE_TOL
    o_ref, p_ref, i_ref = oracle.permutation(ids_ref, wl.E)
    assert np.array_equal(off, o_ref) and np.array_equal(perm, p_ref) and np.array_equal(inv, i_ref)
    rows = np.arange(x.shape[0]) if sample is None else np.asarray(sample)
    g, u, d = ol.lists_for(ids_ref[rows])
    out_ref = oracle.moe_experts(x[rows], ids_ref[rows], gates_ref[rows], g, u, d, E=wl.E, S=wl.S)
    err = np.abs(out[rows] - out_ref).max()
    assert err <= tolerance(out_ref), f"max|err| {err} > {tolerance(out_ref)}"
    return err


CASES = [
    ("tiny", dict(T=17)),                              # one partial tile per expert
    ("tiny", dict(T=129, k=2)),
    ("tiny", dict(T=300, E=64, k=8, sigma_router=0.1)),  # many experts, several tiles, empty experts
    ("tiny", dict(T=200, S=1)),                         # shared expert rows
    ("tiny", dict(T=64, I=192)),                        # I % 128 == 64: half-empty last gate/up tile
    ("tiny", dict(T=40, H=320, E=8, k=3)),              # H % 256 != 0: partial last down tile
    ("tiny", dict(T=1000, k=2)),                        # 192-row tiles and small last tiles (both GEMM shapes)
    ("tiny", dict(T=700, k=2, I=192, S=1)),             # large remainders (> 64 rows), shared expert, odd blocks
]


@pytest.mark.parametrize("name, over", CASES, ids=[f"{n}-{'-'.join(f'{k}{v}' for k, v in o.items())}"
                                                    for n, o in CASES])
def test_prefill_parity_small(name, over):
    wl = synth.WORKLOADS[name].with_(**over)
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    _, res = run_layer(wl, x)
    check(wl, x, res, ol)


def test_decode_and_prefill_agree_at_T16():
    """The same 16 tokens through the decode path and (with decode_T_max=1)
    through the prefill path: both within tolerance of the oracle."""
    wl = synth.WORKLOADS["dec16"]
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    _, res_dec = run_layer(wl, x, decode_T_max=16)
    _, res_pre = run_layer(wl, x, decode_T_max=1)
    check(wl, x, res_dec, ol)
    check(wl, x, res_pre, ol)
    assert np.array_equal(res_dec[0], res_pre[0])


def test_prefill_full_size_4096_zipf():
    wl = synth.WORKLOADS["pre4096"]
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    _, res = run_layer(wl, x)
    rng = np.random.default_rng(0)
    sample = np.sort(rng.choice(wl.T, 40, replace=False))
    sample = np.concatenate([[0, wl.T - 1], sample])
    check(wl, x, res, ol, sample=sample)


def test_prefill_full_size_large_2048():
    """H=7168, I=2048, 256 routed + 1 shared expert, T=2048: routing for all
    tokens, outputs of a sample of tokens (the oracle quantises only the
    experts those tokens touch)."""
    wl = synth.WORKLOADS["large2048"]
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    _, res = run_layer(wl, x)
    check(wl, x, res, ol, sample=[0, 1337])
