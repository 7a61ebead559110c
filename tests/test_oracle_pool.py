"""The oracle run over worker processes (tests/oracle_pool.py) gives the
single-process oracle's output bit for bit: same routine, same per-slot
products, same order of additions."""
import numpy as np

import oracle
import synth
from layer_inputs import OracleLayer, hidden_with_margins
from oracle_pool import expert_outputs


def test_pool_equals_single_process_oracle():
    wl = synth.WORKLOADS["tiny"].with_(T=40, S=1, k=3)
    ol = OracleLayer(wl, 0)
    x = hidden_with_margins(wl, 0, ol.Wr, ol.bias)
    ids, gates = ol.route(x)
    g, u, d = ol.lists_for(ids)
    ref = oracle.moe_experts(x, ids, gates, g, u, d, E=wl.E, S=wl.S)
    got = expert_outputs(wl, 0, x, ids, gates, procs=3, shared_chunk=7)
    assert np.array_equal(got, ref)
