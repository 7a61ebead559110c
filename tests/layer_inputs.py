"""Seeded layers and hidden states for the parity tests, built twice from the
same generator streams: once for the CUDA library (device fills, its own
quantiser) and once for the oracle (host fills, the oracle's quantiser).
Expected values never come from the CUDA side."""
from __future__ import annotations

import numpy as np

import oracle
import synth
from synth import KIND_DOWN, KIND_GATE, KIND_UP, stream_id

MARGIN = 1e-3  # adjacent sorted logits among the top k+1 differ by at least this


# Bound on |gate - oracle gate|. The gates only scale expert outputs, so an
# error d in a gate moves an output by at most d * max|expert output|: d = 1e-4
# keeps that at least two orders below the output bound (1e-2 * max|out|).
# (What the GPU gates actually show: fp32 logits summed over H terms -- on the
# tensor cores over 3 x H/16 MMA steps -- differ from the fp64 oracle by
# 1e-6 .. 1e-5 in the gates at H <= 7168.)
GATE_TOL = 1e-4


def tolerance(out_ref: np.ndarray) -> float:
    """max |gpu - oracle| allowed: 1e-2 * max|oracle| + 1e-3."""
    return 1e-2 * float(np.abs(out_ref).max()) + 1e-3


def margin_ok(z: np.ndarray, k: int) -> np.ndarray:
    """Per token: all adjacent gaps among the k+1 largest logits (k if k == E) are >= MARGIN."""
    E = z.shape[1]
    top = -np.sort(-z, axis=1)[:, :min(k + 1, E)]
    if top.shape[1] < 2:
        return np.ones(z.shape[0], dtype=bool)
    return (np.diff(-top, axis=1) >= MARGIN).all(axis=1)


def hidden_with_margins(w, layer, Wr, bias, T=None, max_rounds=200):
    """x [T, H] bf16 bits; rows whose oracle logits violate the margin are redrawn
    from the next redraw stream, row by row, until all pass."""
    T = w.T if T is None else T
    x = synth.hidden_bf16_bits(w, layer, T)
    bad = ~margin_ok(oracle.router_logits(x, Wr, bias), w.k)
    r = 0
    while bad.any():
        r += 1
        assert r <= max_rounds, "could not meet the logit margin"
        for t in np.nonzero(bad)[0]:
            x[t] = synth.hidden_row_bf16_bits(w, layer, int(t), r)
        idx = np.nonzero(bad)[0]
        bad[idx] = ~margin_ok(oracle.router_logits(x[idx], Wr, bias), w.k)
    return x


class DeviceLayer:
    """The layer's weights on the GPU, in the GGUF Q8_0 layout fw_moe_init takes."""

    def __init__(self, w, layer, device, Wr=None, bias=None):
        import torch
        import quantized_sparse_moe_router_gb300 as fw
        self.w, self.layer = w, layer
        H, I, E, S = w.H, w.I, w.E, w.S
        EU = E + S
        self.Wr = synth.router_weight_f32(w, layer) if Wr is None else Wr
        self.bias = synth.router_bias_f32(w, layer) if bias is None else bias
        gu_bytes = fw.q8_0_bytes(I, H)
        d_bytes = fw.q8_0_bytes(H, I)
        self.q = {KIND_GATE: torch.empty((EU, gu_bytes), dtype=torch.uint8, device=device),
                  KIND_UP: torch.empty((EU, gu_bytes), dtype=torch.uint8, device=device),
                  KIND_DOWN: torch.empty((EU, d_bytes), dtype=torch.uint8, device=device)}
        tmp = torch.empty(I * H, dtype=torch.float32, device=device)
        for e in range(EU):
            for kind in (KIND_GATE, KIND_UP, KIND_DOWN):
                synth.fill_normal_f32_device(tmp, w.seed, stream_id(layer, e, kind), w.sigma_w)
                rows, K = (I, H) if kind != KIND_DOWN else (H, I)
                fw.quantize_q8_0(tmp.view(rows, K), out=self.q[kind][e].view(rows, K // 32 * 34))
        del tmp
        self.router_w = torch.from_numpy(self.Wr).to(device)
        self.router_bias = None if self.bias is None else torch.from_numpy(self.bias).to(device)

    def weights(self):
        E = self.w.E
        d = {"router_w": self.router_w, "router_bias": self.router_bias,
             "w_gate": self.q[KIND_GATE][:E], "w_up": self.q[KIND_UP][:E], "w_down": self.q[KIND_DOWN][:E]}
        if self.w.S:
            d.update(shared_gate=self.q[KIND_GATE][E], shared_up=self.q[KIND_UP][E],
                     shared_down=self.q[KIND_DOWN][E])
        return d

    def make(self, T_max, decode_T_max=0, act_q8=False):
        import quantized_sparse_moe_router_gb300 as fw
        w = self.w
        return fw.MoELayer(w.H, w.I, w.E, w.k, n_shared=w.S, T_max=T_max, decode_T_max=decode_T_max,
                           weights=self.weights(), act_q8=act_q8)


class OracleLayer:
    """The same layer on the host, quantised by the oracle, experts made on demand."""

    def __init__(self, w, layer):
        self.w, self.layer = w, layer
        self.Wr = synth.router_weight_f32(w, layer)
        self.bias = synth.router_bias_f32(w, layer)
        self._q = {}

    def q(self, e, kind):
        key = (e, kind)
        if key not in self._q:
            self._q[key] = oracle.q8_0_quantize(synth.expert_weight_f32(self.w, self.layer, e, kind))
        return self._q[key]

    def lists_for(self, ids):
        """Per-kind lists of E+S Q8_0 arrays with only the experts in `ids` (and the shared one)."""
        w = self.w
        need = set(np.unique(ids).tolist()) | set(range(w.E, w.E + w.S))
        return [[self.q(e, kind) if e in need else None for e in range(w.E + w.S)]
                for kind in (KIND_GATE, KIND_UP, KIND_DOWN)]

    def route(self, x):
        z = oracle.router_logits(x, self.Wr, self.bias)
        return oracle.topk_gates(z, self.w.k)

    def forward(self, x):
        ids, gates = self.route(x)
        g, u, d = self.lists_for(ids)
        return ids, gates, oracle.moe_experts(x, ids, gates, g, u, d, E=self.w.E, S=self.w.S)


def to_device_bf16(x_bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(device).view(torch.bfloat16)
