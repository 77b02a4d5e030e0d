"""Full-size OLMoE-shaped workload (16 layers x 64 experts, top-8, H 2048,
I 1024, bf16, 16 slots per layer) in the launch configuration the benchmark
times (the AUTO copy mode, batch 1): every layer step's slot trace bit-exact
against the oracle, and sampled (step, layer) outputs against the float64
oracle.  Layers are fed independent seeded hidden states so each sampled
output has an oracle input that never came from the GPU."""

import numpy as np
import pytest

from expert_slot_cache_topk_gb300 import synth
from oracle import router_topk
from tests.gpu_util import (OracleWeights, assert_close, empty_y, make_cache, oracle_slot_caches,
                            oracle_y, torch_x, y_to_f64)

pytestmark = pytest.mark.gpu


def test_olmoe_full_size_trace_and_sampled_outputs():
    import torch
    w = synth.WORKLOADS["olmoe"]
    steps = 48
    c = make_cache(w, copy_mode="auto")
    oc = oracle_slot_caches(w)
    lgs = [synth.routing_logits(w, l, steps) for l in range(w.layers)]
    xs = [synth.hidden_states(w, l, steps) for l in range(w.layers)]
    g = np.random.default_rng(7)
    sample = {(int(s), int(l)) for s, l in zip(g.integers(0, steps, 24), g.integers(0, w.layers, 24))}
    kept = {}
    for s in range(steps):
        for l in range(w.layers):
            y = empty_y(w, 1)
            c.forward(l, torch_x(w, xs[l][s]), torch.from_numpy(lgs[l][s]).cuda(), 1, y)
            rec = c.last_prepare(l)
            ids, _ = router_topk(lgs[l][s], w.top_k)
            ref = oc[l].prepare(ids)
            assert rec["hits"] == ref.hits and rec["misses"] == ref.misses, (s, l)
            if (s, l) in sample:
                kept[(s, l)] = y_to_f64(w, y)
    tot = c.stats(-1)
    assert tot["hits"] == sum(o.stats["hits"] for o in oc)
    assert tot["misses"] == sum(o.stats["misses"] for o in oc)
    for l in range(w.layers):
        assert c.verify_slots(l) == 0
    wt = OracleWeights(w)
    for (s, l), y in sorted(kept.items()):
        assert_close(y, oracle_y(w, wt, l, xs[l][s], lgs[l][s]), f"olmoe step {s} layer {l}")
    c.close()
