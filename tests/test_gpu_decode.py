"""GPU parity of the quantiser, the repack, the routers and the decode path
(T <= 16) against the fp64 oracle, through the C ABI.

Bar: expert ids, offsets, perm and inv bit-exact; gates within GATE_TOL; outputs
max |gpu - oracle| <= 1e-2 * max|oracle| + 1e-3 (the GPU's bf16 widened
exactly to fp64)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle
import quantized_sparse_moe_router_gb300 as fw
import synth
from layer_inputs import GATE_TOL, DeviceLayer, OracleLayer, hidden_with_margins, to_device_bf16, tolerance
from synth import KIND_DOWN, KIND_GATE, KIND_UP

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def built():
    fw.build()
    torch.cuda.set_device(0)


def check_against_oracle(dl, ol, layer, x, ids, gates, out):
    ids_ref, gates_ref, out_ref = ol.forward(x)
    assert np.array_equal(ids.cpu().numpy(), ids_ref), "expert ids differ"
    assert np.abs(gates.cpu().numpy() - gates_ref).max() <= GATE_TOL
    w = dl.w
    T = x.shape[0]
    off, perm, inv = layer.permutation(T)
    o_ref, p_ref, i_ref = oracle.permutation(ids_ref, w.E)
    assert np.array_equal(off.cpu().numpy(), o_ref)
    assert np.array_equal(perm.cpu().numpy(), p_ref)
    assert np.array_equal(inv.cpu().numpy(), i_ref)
    got = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - out_ref).max()
    assert err <= tolerance(out_ref), f"max|err| {err} > {tolerance(out_ref)}"
    # the bytes the GPU quantised for the experts used equal the oracle's
    for e in sorted(set(np.unique(ids_ref).tolist()) | set(range(w.E, w.E + w.S)))[:12]:
        for kind in (KIND_GATE, KIND_UP, KIND_DOWN):
            assert np.array_equal(dl.q[kind][e].cpu().numpy(), ol.q(e, kind).ravel())
    return err


# ----------------------------------------------------------------- quantiser
def test_quantiser_bit_exact_against_oracle():
    rows, K = 300, 2048
    w = synth.normal_f32(77, 1, rows * K, 0.02).reshape(rows, K)
    w[0] = 0.0                                                    # all-zero blocks
    w[1, :32] = np.array([127.0, 2.5, -2.5, 0.5, -0.5, 126.5] + [1.5] * 26, np.float32)  # exact ties, d = 1
    w[2] *= 1e-4                                                  # subnormal binary16 scales
    w[3, :32] = (np.arange(-16, 16) * 2.0 ** -7).astype(np.float32)
    w[4] *= 1e4
    got = fw.quantize_q8_0(torch.from_numpy(w).to(DEV)).cpu().numpy()
    ref = oracle.q8_0_quantize(w)
    assert np.array_equal(got, ref)


def test_repack_round_trip():
    wl = synth.WORKLOADS["tiny"].with_(S=1)
    dl = DeviceLayer(wl, 0, DEV)
    layer = dl.make(T_max=4)
    for e in range(wl.E + 1):
        for kind in (KIND_GATE, KIND_UP, KIND_DOWN):
            assert torch.equal(layer.export_q8_0(e, kind), dl.q[kind][e].view(layer.export_q8_0(e, kind).shape))
    layer.close()


# --------------------------------------------------------------- decode path
DECODE_CASES = [
    ("tiny", {}),
    ("tiny", dict(T=1)),
    ("tiny", dict(T=3, k=1)),
    ("tiny", dict(T=16, k=8)),                 # k = E
    ("tiny", dict(T=5, S=1)),
    ("tiny", dict(T=1, H=2304, S=1)),          # one token, H past the several-token limit: two down stages
    ("tiny", dict(T=1, H=4160, I=192)),        # one token, three down stages (4160 = 3 x 1387 -> 1392-row stages)
    ("tiny", dict(T=2, H=2304)),               # several tokens with H > 2048: the prefill path takes them
    ("tiny", dict(T=1, H=14336, I=128)),       # one token at the largest H the decode kernel takes (two ring stages)
    ("tiny", dict(T=1, H=16384, I=128)),       # one token past it: the prefill path takes it
    ("tiny", dict(T=4, E=32, k=16)),           # the largest k
    ("tiny", dict(T=16, E=32, k=16, S=1)),     # largest k and T together, with a shared expert
    ("dec1", {}),
    ("dec16", {}),
    ("large1", {}),
]


@pytest.mark.parametrize("name, over", DECODE_CASES, ids=[f"{n}-{'-'.join(f'{k}{v}' for k, v in o.items())}"
                                                          for n, o in DECODE_CASES])
def test_decode_parity(name, over):
    wl = synth.WORKLOADS[name].with_(**over)
    dl = DeviceLayer(wl, 0, DEV)
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    layer = dl.make(T_max=max(wl.T, 16))
    xd = to_device_bf16(x, DEV)
    gates = torch.empty((wl.T, wl.k), dtype=torch.float32, device=DEV)
    ids, out = layer.forward(xd, gates=gates)
    torch.cuda.synchronize()
    layer.status()
    check_against_oracle(dl, ol, layer, x, ids, gates, out)
    # a second call on the same handle (ticket and workspace reuse) gives the same bits
    ids2, out2 = layer.forward(xd)
    assert torch.equal(ids, ids2) and torch.equal(out, out2)
    layer.close()


def test_decode_ties_and_forced_expert():
    """Zero router: every logit is exactly 0, so ids are 0..k-1 (ties to the lower
    id) and gates 1/k. A +50 bias on expert 5 forces every token onto it (one
    expert with all 16 tokens)."""
    wl = synth.WORKLOADS["tiny"].with_(T=16, k=3)
    ol = OracleLayer(wl, 0)
    zero = np.zeros((wl.E, wl.H), np.float32)
    dl = DeviceLayer(wl, 0, DEV, Wr=zero)
    layer = dl.make(T_max=16)
    x = synth.hidden_bf16_bits(wl, 0)
    gates = torch.empty((16, 3), dtype=torch.float32, device=DEV)
    ids, out = layer.forward(to_device_bf16(x, DEV), gates=gates)
    assert ids.cpu().numpy().tolist() == [[0, 1, 2]] * 16
    assert torch.all(gates == 1.0 / 3.0)
    g, u, d = ol.lists_for(np.array([[0, 1, 2]]))
    out_ref = oracle.moe_experts(x, np.tile([0, 1, 2], (16, 1)), np.full((16, 3), 1 / 3), g, u, d, E=wl.E)
    assert np.abs(out.float().cpu().numpy() - out_ref).max() <= tolerance(out_ref)
    layer.close()

    bias = np.zeros(wl.E, np.float32)
    bias[5] = 50.0
    ol.bias = bias
    dl2 = DeviceLayer(wl, 0, DEV, bias=bias)
    layer = dl2.make(T_max=16)
    x = hidden_with_margins(wl, 0, ol.Wr, bias)
    gates = torch.empty((16, 3), dtype=torch.float32, device=DEV)
    ids, out = layer.forward(to_device_bf16(x, DEV), gates=gates)
    torch.cuda.synchronize()
    assert np.all(ids.cpu().numpy()[:, 0] == 5)
    check_against_oracle(dl2, ol, layer, x, ids, gates, out)
    layer.close()


def test_call_contract():
    wl = synth.WORKLOADS["tiny"]
    dl = DeviceLayer(wl, 0, DEV)
    layer = dl.make(T_max=8)
    x = to_device_bf16(synth.hidden_bf16_bits(wl, 0, T=8), DEV)
    out = torch.empty((8, wl.H), dtype=torch.bfloat16, device=DEV)
    # ffn before any route
    with pytest.raises(fw.FwError) as ei:
        layer.ffn(x[:4], out=out[:4])
    assert ei.value.status == fw.FW_ESTATE
    layer.route(x[:4])
    with pytest.raises(fw.FwError) as ei:
        layer.ffn(x[:3], out=out[:3])
    assert ei.value.status == fw.FW_ESTATE
    with pytest.raises(fw.FwError) as ei:
        layer.route(torch.empty((9, wl.H), dtype=torch.bfloat16, device=DEV))
    assert ei.value.status == fw.FW_EINVAL
    # T = 0 is a no-op for both
    layer.route(x[:0])
    layer.ffn(x[:0], out=out[:0])
    layer.status()
    h = layer.handle
    layer.close()
    assert fw.lib().fw_moe_free(h) == fw.FW_EINVAL  # freed twice


def test_forward_host_matches_device_path():
    wl = synth.WORKLOADS["tiny"]
    dl = DeviceLayer(wl, 0, DEV)
    ol = OracleLayer(wl, 0)
    layer = dl.make(T_max=4)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    xd = to_device_bf16(x, DEV)
    ids, out = layer.forward(xd)
    xh = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    ids_h = torch.empty((4, wl.k), dtype=torch.int32).pin_memory()
    out_h = torch.empty((4, wl.H), dtype=torch.bfloat16).pin_memory()
    layer.forward_host(xh, ids_h, out_h)
    assert torch.equal(ids_h, ids.cpu()) and torch.equal(out_h, out.cpu())
    layer.close()


def test_decode_grid_wait_bound_gives_timeout_and_handle_recovers(monkeypatch):
    """A test hook makes the next two decode calls' grid-wide wait unreachable
    (one arrival more than the grid): the kernel gives up after its bound
    (1 ms here), records site 8 and returns; fw_moe_status reports
    FW_ETIMEOUT; the calls after that are correct again on the same handle.
    One call of each decode instantiation (one token, several tokens)."""
    wl = synth.WORKLOADS["tiny"]
    dl = DeviceLayer(wl, 0, DEV)
    ol = OracleLayer(wl, 0)
    monkeypatch.setenv("FWMOE_TEST_GRID_TIMEOUTS", "2")
    layer = dl.make(T_max=4)
    monkeypatch.delenv("FWMOE_TEST_GRID_TIMEOUTS")
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    xd = to_device_bf16(x, DEV)
    for T in (1, 4):
        layer.forward(xd[:T])
        with pytest.raises(fw.FwError) as ei:
            layer.status()
        assert ei.value.status == fw.FW_ETIMEOUT and "site 8" in str(ei.value)
    for T in (1, 4):
        gates = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
        ids, out = layer.forward(xd[:T], gates=gates)
        torch.cuda.synchronize()
        layer.status()
        check_against_oracle(dl, ol, layer, x[:T], ids, gates, out)
    layer.close()
