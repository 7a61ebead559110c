"""The expert part of the fp64 oracle over every token of a large call, spread
over worker processes.

The oracle stays as it is: single-threaded C, called unchanged. What is split
is the work. A call's (token, slot) pairs are grouped by expert; a worker takes
one expert at a time, makes its fp32 weights from the generator streams,
quantises them with the oracle's own quantiser and evaluates that expert on its
tokens with `oracle.moe_experts` (one slot per token, the slot's gate as the
gate, so each result row is gate * y_e(x_t) exactly as the oracle forms it).
The shared expert's tokens are cut into ranges so that its work spreads too.
The parent adds each token's rows in slot order and the shared row last -- the
oracle's own order of additions -- so the result is the single-process
oracle's, bit for bit (a CPU test checks this on a small case).

Workers are started with the "spawn" method: a process forked after the
parent touched a GPU can hang.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_W = {}  # per worker process: the workload, the layer and the hidden rows


def _init(wl, layer, x_bits):
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    _W.update(wl=wl, layer=layer, x=x_bits, cache=(None, None))


def _expert_weights(e):
    import oracle
    import synth
    key, q = _W["cache"]
    if key != e:
        wl, layer = _W["wl"], _W["layer"]
        q = [oracle.q8_0_quantize(synth.expert_weight_f32(wl, layer, e, kind)) for kind in (0, 1, 2)]
        _W["cache"] = (e, q)
    return q


def _task(args):
    """(expert, token indices, gates) -> rows gate * y_e(x_t), fp64 [n, H]."""
    import oracle
    e, tok, g = args
    q = _expert_weights(e)
    n = len(tok)
    # one-expert call of the oracle's expert routine: experts 0..e, only e present
    lists = [[None] * e + [q[kind]] for kind in range(3)]
    out = oracle.moe_experts(_W["x"][tok], np.full((n, 1), e, np.int32), np.asarray(g, np.float64)[:, None],
                             lists[0], lists[1], lists[2], E=e + 1, S=0)
    return out


def expert_outputs(wl, layer, x_bits, ids, gates, procs=None, shared_chunk=128):
    """out [T, H] fp64 of the oracle's expert part (and combine) for routing
    (ids [T, k], gates [T, k]) of hidden rows x_bits [T, H] (bf16 bits)."""
    T, k = ids.shape
    procs = procs or max(1, min(os.cpu_count() or 1, 32))
    tasks = []
    order = np.argsort(ids.ravel(), kind="stable")  # slots grouped by expert, token ascending
    flat = ids.ravel()[order]
    starts = np.flatnonzero(np.r_[True, flat[1:] != flat[:-1]])
    ends = np.r_[starts[1:], len(flat)]
    for s0, s1 in zip(starts, ends):
        slots = order[s0:s1]
        tasks.append((int(flat[s0]), slots // k, gates.ravel()[slots], slots % k))
    for t0 in range(0, T if wl.S else 0, shared_chunk):
        tok = np.arange(t0, min(T, t0 + shared_chunk))
        tasks.append((wl.E, tok, np.ones(len(tok)), np.full(len(tok), k)))  # slot k: the shared row
    # the heaviest tasks first, so that no long one starts last
    tasks.sort(key=lambda a: -len(a[1]))
    contrib = np.zeros((T, k + 1, wl.H), np.float64)
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs, initializer=_init, initargs=(wl, layer, np.ascontiguousarray(x_bits))) as pool:
        for (e, tok, g, j), rows in zip(tasks, pool.imap(_task, [(e, tok, g) for e, tok, g, _ in tasks])):
            contrib[tok, j] = rows
    out = np.zeros((T, wl.H), np.float64)
    for j in range(k):
        out += contrib[:, j]
    if wl.S:
        out += contrib[:, k]
    return out
