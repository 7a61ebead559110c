"""Pins of the fp64 oracle against things other than itself (no GPU).

Each pin is chosen so that a plausible slip in the oracle fails it: the
binary16 conversion against numpy's, the quantiser against closed-form blocks,
routing against a full sort, the FFN and combine against a dense all-experts
evaluation written independently in numpy, and a two-expert example whose
output has a closed form.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth
from brute import bf16_to_f64, dense_masked_moe, parse_q8_0, sort_select

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------- binary16 / bf16
def test_half_to_double_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    ours = np.array([oracle.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[np.isinf(ref)], ref[np.isinf(ref)])


def test_double_to_half_matches_numpy_rne():
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        # exact ties between neighbouring halves (normal and subnormal), both parities
        np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 2 ** -24 * 0.5, 2 ** -24 * 1.5, 2 ** -24 * 2.5,
                  65504.0, 65519.99, 65520.0, 2 ** -14, 2 ** -14 * (1 - 2 ** -11), 0.0, -0.0,
                  1 + 2 ** -11 + 2 ** -40, 1 / 127.0, 1e-3 / 127.0, 7.874e-9]),
    ])
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    ours = np.array([oracle.double_to_half(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_widening_matches_float32_halves():
    bits = synth.normal_bf16_bits(3, 9, 1000, 1.0)
    ours = np.array([oracle.lib().oracle_bf16_to_double(int(b)) for b in bits])
    assert np.array_equal(ours, bf16_to_f64(bits))


# -------------------------------------------------------------------- Q8_0
def _q_of(blocks, r=0, b=0):
    blk = blocks[r, b * 34:(b + 1) * 34]
    return blk[2:].view(np.int8).astype(int), int(blk[0]) | (int(blk[1]) << 8)


def test_q8_0_exact_codes_recovered():
    # values q * 2^-7 with +-127 present: d = 2^-7 exactly, codes come back unchanged
    q = np.array([127, -127] + list(range(-60, 60, 4)), dtype=np.int64)
    assert q.size == 32
    w = (q * 2.0 ** -7).astype(np.float32)[None, :]
    blocks = oracle.q8_0_quantize(w)
    codes, dbits = _q_of(blocks)
    assert dbits == 0x2000  # binary16 2^-7
    assert np.array_equal(codes, q)


def test_q8_0_zero_block():
    blocks = oracle.q8_0_quantize(np.zeros((2, 64), dtype=np.float32))
    assert blocks.shape == (2, 68) and not blocks.any()


def test_q8_0_round_half_away_from_zero():
    # amax = 127 -> d = 1 exactly, so w/d = w and the .5 cases are exact ties
    vals = [127.0, 2.5, -2.5, 0.5, -0.5, 126.5, -126.5, 1.5, -1.5, 3.49, -3.51] + [0.0] * 21
    blocks = oracle.q8_0_quantize(np.array(vals, dtype=np.float32)[None, :])
    codes, dbits = _q_of(blocks)
    assert dbits == 0x3C00  # 1.0
    assert list(codes[:11]) == [127, 3, -3, 1, -1, 127, -127, 2, -2, 3, -4]


def test_q8_0_subnormal_scale_and_unrounded_quantisation():
    # amax = 1e-3: d = 1e-3/127 is a binary16 subnormal; codes use the unrounded d
    rng = np.random.default_rng(1)
    w = rng.uniform(-1e-3, 1e-3, 32).astype(np.float32)
    w[5] = np.float32(1e-3)
    blocks = oracle.q8_0_quantize(w[None, :])
    codes, dbits = _q_of(blocks)
    d = float(np.float32(1e-3)) / 127.0
    assert dbits == np.float64(d).astype(np.float16).view(np.uint16)
    assert dbits < 0x0400  # subnormal
    expect = [int(math.copysign(math.floor(abs(float(x) / d) + 0.5), float(x))) for x in w]
    assert list(codes) == expect


def test_q8_0_layout_and_error_bound():
    rows, K = 5, 96
    w = synth.normal_f32(11, 1, rows * K, 0.02).reshape(rows, K)
    blocks = oracle.q8_0_quantize(w)
    assert blocks.shape == (rows, K // 32 * 34)
    deq = oracle.q8_0_dequantize(blocks, rows, K)
    assert np.array_equal(deq, parse_q8_0(blocks, rows, K))  # numpy parses the same layout
    for r in range(rows):
        for b in range(K // 32):
            x = w[r, b * 32:(b + 1) * 32].astype(np.float64)
            d = np.abs(x).max() / 127.0
            d16 = float(np.float64(d).astype(np.float16))
            q = np.abs(deq[r, b * 32:(b + 1) * 32]) / d16
            bound = d / 2 + q * abs(d - d16) + 1e-18
            assert np.all(np.abs(deq[r, b * 32:(b + 1) * 32] - x) <= bound)


# ---------------------------------------------------------------- routing
def _route_inputs(T=9, H=64, E=12, seed=5, sigma=0.1):
    x = synth.normal_bf16_bits(seed, 1, T * H, 1.0).reshape(T, H)
    Wr = synth.normal_f32(seed, 2, E * H, sigma).reshape(E, H)
    b = synth.normal_f32(seed, 3, E, 0.05)
    return x, Wr, b


def test_router_logits_match_numpy_matmul():
    x, Wr, b = _route_inputs()
    z = oracle.router_logits(x, Wr, b)
    ref = bf16_to_f64(x) @ Wr.astype(np.float64).T + b.astype(np.float64)
    assert np.allclose(z, ref, rtol=1e-13, atol=1e-14)
    z0 = oracle.router_logits(x, Wr, None)
    assert np.allclose(z0 + b.astype(np.float64), z, rtol=0, atol=1e-14)


@pytest.mark.parametrize("k", [1, 2, 5, 12])
def test_topk_matches_full_sort(k):
    x, Wr, b = _route_inputs()
    z = oracle.router_logits(x, Wr, b)
    ids, gates = oracle.topk_gates(z, k)
    assert np.array_equal(ids, sort_select(z, k))
    assert np.allclose(gates.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    assert np.all(np.diff(gates, axis=1) <= 0)  # descending logits give descending gates


def test_topk_ties_go_to_lower_id():
    z = np.array([[0.0] * 6, [1.0, 2.0, 2.0, 0.5, 2.0, 1.0], [3.0, 3.0, 1.0, 3.0, 2.0, 2.0]])
    ids, gates = oracle.topk_gates(z, 4)
    assert ids.tolist() == [[0, 1, 2, 3], [1, 2, 4, 0], [0, 1, 3, 4]]
    assert np.allclose(gates[0], 0.25, rtol=0, atol=1e-16)
    assert np.array_equal(ids, sort_select(z, 4))


def test_zero_router_uniform_gates():
    T, H, E, k = 3, 64, 8, 3
    x = synth.normal_bf16_bits(1, 1, T * H, 1.0).reshape(T, H)
    z = oracle.router_logits(x, np.zeros((E, H), np.float32), None)
    ids, gates = oracle.topk_gates(z, k)
    assert np.all(z == 0.0)
    assert ids.tolist() == [[0, 1, 2]] * T
    assert np.array_equal(gates, np.full((T, k), 1.0 / k))


def test_constant_shift_invariance():
    x, Wr, b = _route_inputs()
    z = oracle.router_logits(x, Wr, b)
    z2 = oracle.router_logits(x, Wr, (b.astype(np.float64) + 0.75).astype(np.float32))
    ids, g = oracle.topk_gates(z, 4)
    ids2, g2 = oracle.topk_gates(z2, 4)
    assert np.array_equal(ids, ids2)
    assert np.allclose(g, g2, rtol=0, atol=1e-7)  # fp32 bias rounding only


def test_two_experts_gate_is_logistic():
    z = np.array([[0.3, -1.1], [2.0, 2.5], [-0.25, -0.75]])
    ids, g = oracle.topk_gates(z, 2)
    for t in range(3):
        e0, e1 = ids[t]
        assert g[t, 0] == pytest.approx(1.0 / (1.0 + math.exp(z[t, e1] - z[t, e0])), rel=1e-15)


def test_gates_equal_literal_full_softmax_route():
    x, Wr, b = _route_inputs(T=20, E=30)
    z = oracle.router_logits(x, Wr, b)
    for k in (1, 3, 8, 30):
        ids, g = oracle.topk_gates(z, k)
        g_lit = oracle.gates_full_softmax(z, ids)
        assert np.allclose(g, g_lit, rtol=0, atol=1e-15)


# ------------------------------------------------------------- permutation
def test_permutation_brute_force_and_invariants():
    T, E, k = 37, 9, 3
    rng = np.random.default_rng(3)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    offsets, perm, inv = oracle.permutation(ids, E)
    pairs = sorted((int(ids[t, j]), t, t * k + j) for t in range(T) for j in range(k))
    assert perm.tolist() == [s for _, _, s in pairs]
    counts = np.bincount(ids.ravel(), minlength=E)
    assert offsets.tolist() == [0] + np.cumsum(counts).tolist()
    assert np.array_equal(inv[perm], np.arange(T * k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(ids.ravel()[seg] == e)
        assert np.all(np.diff(seg // k) > 0)  # ascending token within an expert


# ----------------------------------------------------------- experts, FFN
def _tiny_layer(E=4, H=64, I=96, S=0, seed=17, sigma=0.05):
    qs = {}
    for kind, (r, c) in ((0, (I, H)), (1, (I, H)), (2, (H, I))):
        qs[kind] = [oracle.q8_0_quantize(synth.normal_f32(seed, 100 * e + kind, r * c, sigma).reshape(r, c))
                    for e in range(E + S)]
    return qs


def test_expert_ffn_and_combine_match_dense_masked_evaluation():
    E, H, I, k, T = 5, 64, 96, 2, 7
    for S in (0, 1):
        qs = _tiny_layer(E=E, H=H, I=I, S=S)
        x = synth.normal_bf16_bits(2, 1, T * H, 1.0).reshape(T, H)
        Wr = synth.normal_f32(2, 2, E * H, 0.2).reshape(E, H)
        ids, gates, out = oracle.moe_forward(x, Wr, None, qs[0], qs[1], qs[2], k=k, S=S)
        Wg = np.stack([parse_q8_0(b, I, H) for b in qs[0][:E]])
        Wu = np.stack([parse_q8_0(b, I, H) for b in qs[1][:E]])
        Wd = np.stack([parse_q8_0(b, H, I) for b in qs[2][:E]])
        shared = None
        if S:
            shared = (parse_q8_0(qs[0][E], I, H), parse_q8_0(qs[1][E], I, H), parse_q8_0(qs[2][E], H, I))
        # independent routing: numpy logits, full softmax, full sort, mask
        z = bf16_to_f64(x) @ Wr.astype(np.float64).T
        p = np.exp(z - z.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        sel = sort_select(z, k)
        mask = np.zeros((T, E))
        for t in range(T):
            mask[t, sel[t]] = p[t, sel[t]] / p[t, sel[t]].sum()
        ref = dense_masked_moe(bf16_to_f64(x), Wg, Wu, Wd, mask, shared)
        assert np.array_equal(ids, sel)
        scale = np.abs(ref).max()
        assert np.abs(out - ref).max() <= 1e-12 * scale


def test_k_equals_E_uniform_gates_is_mean_of_experts():
    E, H, I, T = 4, 64, 96, 3
    qs = _tiny_layer(E=E, H=H, I=I)
    x = synth.normal_bf16_bits(4, 1, T * H, 1.0).reshape(T, H)
    ids, gates, out = oracle.moe_forward(x, np.zeros((E, H), np.float32), None, qs[0], qs[1], qs[2], k=E)
    assert np.array_equal(gates, np.full((T, E), 1.0 / E))
    Wg = np.stack([parse_q8_0(b, I, H) for b in qs[0]])
    Wu = np.stack([parse_q8_0(b, I, H) for b in qs[1]])
    Wd = np.stack([parse_q8_0(b, H, I) for b in qs[2]])
    mean = dense_masked_moe(bf16_to_f64(x), Wg, Wu, Wd, np.full((T, E), 1.0 / E))
    assert np.abs(out - mean).max() <= 1e-12 * np.abs(mean).max()
    # no residual: the output is not x plus anything
    assert np.abs(out).max() < 0.5 * np.abs(bf16_to_f64(x)).max()


def test_zero_gate_projection_gives_zero_output():
    E, H, I, T = 3, 64, 32, 2
    qs = _tiny_layer(E=E, H=H, I=I)
    zero = oracle.q8_0_quantize(np.zeros((I, H), np.float32))
    x = synth.normal_bf16_bits(4, 1, T * H, 1.0).reshape(T, H)
    Wr = synth.normal_f32(4, 2, E * H, 0.3).reshape(E, H)
    _, _, out = oracle.moe_forward(x, Wr, None, [zero] * E, qs[1], qs[2], k=2)
    assert np.all(out == 0.0)


def _hand_example():
    with open(os.path.join(GOLDEN, "hand_two_expert.json")) as f:
        return json.load(f)


def test_hand_two_expert_example():
    g = _hand_example()
    H = I = 32
    c = 127.0 / 128.0
    eye = np.eye(32, dtype=np.float32) * np.float32(c)
    q_pos = oracle.q8_0_quantize(eye)
    q_neg = oracle.q8_0_quantize(-eye)
    Wr = np.zeros((2, H), np.float32)
    Wr[0, 0] = 1.0
    Wr[1, 1] = 1.0
    x = np.zeros((2, H), np.float32)
    x[0, :6] = g["token0_x"]
    x[1, :6] = g["token1_x"]
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)  # all entries are exact in bf16
    for k in (1, 2):
        ids, gates, out = oracle.moe_forward(xb, Wr, None, [q_pos, q_pos], [q_pos, q_neg], [q_pos, q_pos], k=k)
        exp = g[f"k{k}"]
        assert ids.tolist() == exp["ids"]
        assert np.allclose(out[:, :6], exp["out"], rtol=0, atol=5e-10)
        assert np.all(out[:, 6:] == 0.0)
        # the same numbers from the closed form y0_i = c * SiLU(c x_i) * c x_i
        for t in range(2):
            xv = x[t, :6].astype(np.float64)
            y0 = c * (c * xv / (1 + np.exp(-c * xv))) * (c * xv)
            zt = xv[:2]
            if k == 1:
                ref = y0 if zt[0] > zt[1] else -y0
            else:
                ref = math.tanh((zt[0] - zt[1]) / 2) * y0
            assert np.allclose(out[t, :6], ref, rtol=1e-15, atol=1e-15)
        if k == 2:
            offsets, perm, inv = oracle.permutation(ids, 2)
            assert offsets.tolist() == exp["offsets"]
            assert perm.tolist() == exp["perm"]
            assert inv.tolist() == exp["inv"]


# ----------------------------------------------------------------- generator
def test_generator_is_counter_based_and_standardised():
    a = synth.normal_f32(123, 7, 200000, 1.0)
    b = synth.normal_f32(123, 7, 1000, 1.0, offset=5000)
    assert np.array_equal(a[5000:6000], b)
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1.0) < 0.01
    assert a.min() >= -6.0 and a.max() <= 6.0
    assert np.all(a * 65536.0 == np.round(a * 65536.0))  # 2^-16 grid
    c = synth.normal_f32(123, 8, 1000, 1.0)
    assert not np.array_equal(a[:1000], c)


def test_generator_bf16_is_round_to_nearest_even_of_f32():
    import torch
    f = synth.normal_f32(9, 4, 10000, 0.37)
    bits = synth.normal_bf16_bits(9, 4, 10000, 0.37)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)


# ------------------------------------------------------- Q8 activations
def test_q8_activations_closed_forms():
    # amax 127 gives d = 1 and codes round(v), ties away from zero
    v = np.array([127, 2.5, -2.5, 0.5, -0.5, 126.5, 0.49, -0.51] + [1.5] * 24, np.float32)
    out, q, d = oracle.q8_activations(v, 32)
    assert d.tolist() == [1.0]
    assert q[:8].tolist() == [127, 3, -3, 1, -1, 127, 0, -1] and set(q[8:].tolist()) == {2}
    assert np.array_equal(out, q.astype(np.float64))
    # an all-zero block: d = 0, codes 0, values 0; blocks are independent
    v = np.concatenate([np.zeros(16, np.float32), np.full(16, 3.0, np.float32)])
    out, q, d = oracle.q8_activations(v, 16)
    assert d[0] == 0.0 and not q[:16].any() and not out[:16].any()
    assert d[1] == np.float32(3.0) / np.float32(127.0) and set(q[16:].tolist()) == {127}
    # values already on the grid q * 2^-7 with amax = 127 * 2^-7 come back exactly
    codes = np.arange(-127, 129, 8)[:32].clip(-127, 127).astype(np.float32)
    codes[0] = -127.0
    v = codes * np.float32(2.0 ** -7)
    out, q, d = oracle.q8_activations(v, 32)
    assert d[0] == np.float32(2.0 ** -7) and np.array_equal(q.astype(np.float32), codes)
    assert np.array_equal(out, v.astype(np.float64))


def test_q8_activations_error_bound():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(64 * 32) * rng.choice([1e-3, 1.0, 40.0], 64).repeat(32)).astype(np.float32)
    out, q, d = oracle.q8_activations(v, 32)
    vb = v.reshape(64, 32).astype(np.float64)
    amax = np.abs(vb).max(axis=1)
    assert np.all(np.abs(q) <= 127) and np.all(np.abs(q.reshape(64, 32)).max(axis=1) == 127)
    assert np.allclose(d, amax / 127, rtol=2 ** -23, atol=0)          # d = amax/127 to fp32 rounding
    err = np.abs(out.reshape(64, 32) - vb)
    assert np.all(err <= d[:, None].astype(np.float64) * (0.5 + 1e-6))  # half a step, fp32 division slack


def test_q8act_experts_with_identity_weights_elementwise():
    """One expert whose gate, up and down matrices are s * identity (s = 127 * 2^-8: Q8_0 stores it
    exactly, d = 2^-8, code 127) reduces the Q8-activation step to element-wise operations: x on the
    2^-7 grid passes the x quantiser unchanged, g = u = s x, h = SiLU(g) u rounded to fp32 and
    quantised in blocks of 16 (here two blocks of very different size), y[o] = s h8[o] for o < I."""
    H, I = 64, 32
    s = 127 * 2.0 ** -8
    wg = np.zeros((I, H), np.float32)
    wg[np.arange(I), np.arange(I)] = s
    wd = np.zeros((H, I), np.float32)
    wd[np.arange(I), np.arange(I)] = s
    qg, qd = oracle.q8_0_quantize(wg), oracle.q8_0_quantize(wd)
    codes = np.concatenate([np.arange(-120, 120, 15)[:16], np.arange(-8, 8)[:16], np.arange(-127, 127, 4)[:32]])
    codes[0], codes[32] = -127, -127                     # every 32-block of x has amax 127 * 2^-7
    x = (codes.astype(np.float32) * np.float32(2.0 ** -7))
    x_bits = (x.view(np.uint32) >> 16).astype(np.uint16)[None, :]   # exact in bf16 (7-bit codes)
    ids = np.zeros((1, 1), np.int32)
    gates = np.ones((1, 1))
    out = oracle.moe_experts(x_bits, ids, gates, [qg], [qg], [qd], E=1, S=0, act_q8=True)[0]
    g = s * x[:I].astype(np.float64)
    h32 = (g / (1.0 + np.exp(-g)) * g).astype(np.float32)
    want = np.zeros(H)
    for b in range(I // 16):
        blk = h32[16 * b:16 * b + 16]
        db = np.float32(np.abs(blk).max()) / np.float32(127.0)
        r = (blk / db).astype(np.float64)                  # fp32 quotients
        qb = np.sign(r) * np.floor(np.abs(r) + 0.5)        # ties away (r is exact in fp64)
        want[16 * b:16 * b + 16] = s * qb * np.float64(db)
    assert np.allclose(out, want, rtol=1e-12, atol=1e-15)
    # the two h blocks differ in scale by far more than a code step: one 32-wide block would not match
    assert np.abs(h32[:16]).max() > 20 * np.abs(h32[16:]).max()


def test_q8act_experts_quantise_x_in_blocks_of_32():
    """Off the grid, x goes through the (separately pinned) activation quantiser in blocks of 32
    before the projections: with identity weights the output follows element by element."""
    H, I = 64, 32
    s = 127 * 2.0 ** -8
    wg = np.zeros((I, H), np.float32)
    wg[np.arange(I), np.arange(I)] = s
    wd = np.zeros((H, I), np.float32)
    wd[np.arange(I), np.arange(I)] = s
    qg, qd = oracle.q8_0_quantize(wg), oracle.q8_0_quantize(wd)
    rng = np.random.default_rng(11)
    x32 = (rng.standard_normal(H) * np.repeat([0.7, 0.05], 32)).astype(np.float32)
    u = x32.view(np.uint32)
    x_bits = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)[None, :]  # to bf16, nearest even
    xb = (x_bits[0].astype(np.uint32) << 16).view(np.float32)          # the bf16 values, exactly
    x8 = oracle.q8_activations(xb, 32)[0]
    assert not np.array_equal(x8, xb.astype(np.float64))              # the quantiser does change x here
    out = oracle.moe_experts(x_bits, np.zeros((1, 1), np.int32), np.ones((1, 1)), [qg], [qg], [qd], E=1, S=0,
                             act_q8=True)[0]
    g = s * x8[:I]
    h8 = oracle.q8_activations((g / (1.0 + np.exp(-g)) * g).astype(np.float32), 16)[0]
    want = np.concatenate([s * h8, np.zeros(H - I)])
    assert np.allclose(out, want, rtol=1e-12, atol=1e-15)
