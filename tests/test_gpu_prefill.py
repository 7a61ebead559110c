"""GPU parity of the prefill path (T > decode limit: tiled router, grouping,
gather, tcgen05 grouped GEMMs with in-shared-memory Q8_0 dequantisation,
combine) against the fp64 oracle, through the C ABI.

Same bar as the decode path: ids and permutation bit-exact, outputs within
1e-2 * max|oracle| + 1e-3. At the full workload sizes every token's output is
checked too: the oracle's expert part runs in worker processes (one expert at
a time, the shared expert's tokens in ranges; tests/oracle_pool.py), which
gives the single-process oracle's result bit for bit."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle
import quantized_sparse_moe_router_gb300 as fw
import synth
from layer_inputs import GATE_TOL, DeviceLayer, OracleLayer, hidden_with_margins, to_device_bf16, tolerance
from oracle_pool import expert_outputs

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


def check(wl, x, res, ol, parallel=False):
    """Routing bit-exact, then every token's output within tolerance; with
    parallel=True the oracle's expert part runs over worker processes."""
    ids, gates, out, (off, perm, inv) = res
    ids_ref, gates_ref = ol.route(x)
    assert np.array_equal(ids, ids_ref)
    assert np.abs(gates - gates_ref).max() <= GATE_TOL
    o_ref, p_ref, i_ref = oracle.permutation(ids_ref, wl.E)
    assert np.array_equal(off, o_ref) and np.array_equal(perm, p_ref) and np.array_equal(inv, i_ref)
    if parallel:
        out_ref = expert_outputs(wl, ol.layer, x, ids_ref, gates_ref)
    else:
        g, u, d = ol.lists_for(ids_ref)
        out_ref = oracle.moe_experts(x, ids_ref, gates_ref, g, u, d, E=wl.E, S=wl.S)
    err = np.abs(out - out_ref).max()
    assert err <= tolerance(out_ref), f"max|err| {err} > {tolerance(out_ref)}"
    return ids_ref, err


CASES = [
    ("tiny", dict(T=17)),                              # one partial tile per expert
    ("tiny", dict(T=129, k=2)),
    ("tiny", dict(T=300, E=64, k=8, sigma_router=0.1)),  # many experts, several tiles, empty experts
    ("tiny", dict(T=200, S=1)),                         # shared expert rows
    ("tiny", dict(T=64, I=192)),                        # I % 128 == 64: half-empty last gate/up tile
    ("tiny", dict(T=40, H=320, E=8, k=3)),              # H % 256 != 0: partial last down tile
    ("tiny", dict(T=1000, k=2)),                        # 192-row tiles and small last tiles (both GEMM shapes)
    ("tiny", dict(T=700, k=2, I=192, S=1)),             # large remainders (> 64 rows), shared expert, odd blocks
    ("tiny", dict(T=330, k=2)),                         # about 82 rows per expert: too few mid tiles for their own launch
    ("tiny", dict(T=470, k=2, S=1)),                    # about 117 rows: big remainders; shared: 2 big + mid
    ("tiny", dict(T=40, E=32, k=16)),                   # the largest k (tensor-core router, 16-long top-k lists)
    ("tiny", dict(T=300, E=256, k=8)),                  # the largest E: 256 experts, most with a handful of rows
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
    """The 4096-token workload (Zipf(1.1)-skewed routing: a few experts with
    thousands of rows in many 192-row tiles, many with a handful): every
    token's output."""
    wl = synth.WORKLOADS["pre4096"]
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    _, res = run_layer(wl, x)
    ids, _ = check(wl, x, res, ol, parallel=True)
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    assert counts.max() > 2 * 192 and (counts[counts > 0] <= 64).any()  # both GEMM shapes ran


def test_prefill_mid_tiles_launch():
    """About 81 rows on each of 64 experts: more tiles of 65..96 rows than
    the rule that gives them a launch of their own needs (one tile per SM
    across the two weight blocks a CTA takes), so the mid-tile GEMMs run
    them; every token's output."""
    wl = synth.WORKLOADS["tiny"].with_(T=2600, E=64, k=2, H=1024, I=1024)
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    _, res = run_layer(wl, x)
    ids, _ = check(wl, x, res, ol, parallel=True)
    r = np.bincount(ids.ravel(), minlength=wl.E) % 192
    n_mid = int(((r > 64) & (r <= 96)).sum())
    per_tile = min((2 * wl.I // 128 + 1) // 2, (wl.H // 128 + 1) // 2)  # weight-block pairs per tile
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert n_mid * per_tile >= sms, n_mid


def test_prefill_full_size_large_2048():
    """H=7168, I=2048, 256 routed + 1 shared expert, T=2048: routing and
    every token's output; the call touches all 257 experts (so every expert's
    tiles, K offsets and both GEMM shapes are checked)."""
    wl = synth.WORKLOADS["large2048"]
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    _, res = run_layer(wl, x)
    ids, _ = check(wl, x, res, ol, parallel=True)
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    assert (counts > 0).all()


# ---------------------------------------------------------------- edge cases
def test_prefill_k_equals_E():
    """k = E on the prefill path: every token on every expert, gates the
    renormalised softmax of all E logits."""
    wl = synth.WORKLOADS["tiny"].with_(T=40, k=8)
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    _, res = run_layer(wl, x)
    check(wl, x, res, ol)
    assert (res[0] >= 0).all() and all(sorted(r) == list(range(8)) for r in res[0].tolist())


def test_prefill_zero_router_through_ffn():
    """A zero router makes every logit exactly 0: ids 0..k-1 (ties to the lower
    id), gates 1/k, through the tiled grouping and the GEMMs (experts 0..k-1
    get all T rows each: several 192-row tiles and a small last tile)."""
    wl = synth.WORKLOADS["tiny"].with_(T=430, k=3)
    zero = np.zeros((wl.E, wl.H), np.float32)
    ol = OracleLayer(wl, 0)
    dl = DeviceLayer(wl, 0, DEV, Wr=zero)
    layer = dl.make(T_max=wl.T)
    x = synth.hidden_bf16_bits(wl, 0)
    gates = torch.empty((wl.T, 3), dtype=torch.float32, device=DEV)
    ids, out = layer.forward(to_device_bf16(x, DEV), gates=gates)
    torch.cuda.synchronize()
    layer.status()
    ids_ref = np.tile(np.arange(3, dtype=np.int32), (wl.T, 1))
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert torch.all(gates == 1.0 / 3.0)
    off, perm, inv = layer.permutation(wl.T)
    o_ref, p_ref, i_ref = oracle.permutation(ids_ref, wl.E)
    assert np.array_equal(off.cpu().numpy(), o_ref) and np.array_equal(perm.cpu().numpy(), p_ref)
    assert np.array_equal(inv.cpu().numpy(), i_ref)
    g, u, d = ol.lists_for(ids_ref)
    out_ref = oracle.moe_experts(x, ids_ref, np.full((wl.T, 3), 1 / 3), g, u, d, E=wl.E)
    assert np.abs(out.float().cpu().numpy() - out_ref).max() <= tolerance(out_ref)
    layer.close()


def test_prefill_all_tokens_forced_onto_one_expert():
    """A +50 bias on expert 5 puts it first for every one of 430 tokens: one
    expert with 430 rows (two 192-row tiles and a 46-row small tile), the
    other slots spread over the rest."""
    wl = synth.WORKLOADS["tiny"].with_(T=430, k=2)
    bias = np.zeros(wl.E, np.float32)
    bias[5] = 50.0
    ol = OracleLayer(wl, 0)
    ol.bias = bias
    x = hidden_with_margins(wl, 0, ol.Wr, bias)
    dl = DeviceLayer(wl, 0, DEV, bias=bias)
    layer = dl.make(T_max=wl.T)
    gates = torch.empty((wl.T, wl.k), dtype=torch.float32, device=DEV)
    ids, out = layer.forward(to_device_bf16(x, DEV), gates=gates)
    torch.cuda.synchronize()
    layer.status()
    perm = layer.permutation(wl.T)
    res = (ids.cpu().numpy(), gates.cpu().numpy(), out.float().cpu().numpy().astype(np.float64),
           [p.cpu().numpy() for p in perm])
    layer.close()
    assert (res[0][:, 0] == 5).all()
    check(wl, x, res, ol)
