"""Eviction policies (LRU, LFU, FIFO, SLRU) on the GPU against the oracle, bit
for bit: the hand-worked traces, and seeded traces of single- and multi-token
steps with a small pool so that most misses evict (per step: hits, misses with
their slots and victims, slot ids; final pool state and counters)."""

import numpy as np
import pytest

from expert_slot_cache_topk_gb300 import synth
from oracle import router_topk
from oracle.slot_cache import POLICIES, LayerSlotCache, MovePolicy
from tests.gpu_util import OracleWeights, assert_close, make_cache, oracle_y, torch_x, y_to_f64
from tests.test_oracle_policies import TRACES

pytestmark = pytest.mark.gpu


def _prepare(c, layer, ids_np):
    import torch
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    out = torch.full(ids.shape, -99, dtype=torch.int32, device="cuda")
    c.prepare(layer, ids, ids.shape[0], out)
    return out.cpu().numpy()


def _check_step(c, oc, layer, ids, where):
    out = _prepare(c, layer, ids)
    ref = oc.prepare(ids)
    rec = c.last_prepare(layer)
    assert rec["bypass"] == ref.bypass, where
    assert rec["hits"] == ref.hits, where
    assert rec["misses"] == ref.misses, where
    assert (out == ref.slot_ids).all(), where
    return ref


def _final_state(c, oc, layer):
    sm, se, _, nfree = c.get_state(layer)
    assert (sm == oc.slot_map()).all() and (se == oc.slot_expert()).all()
    assert nfree == len(oc.free)
    s = c.stats(layer)
    for key, v in oc.stats.items():
        assert s[key] == v, key


@pytest.mark.parametrize("policy,E,N,steps,misses,hits", TRACES, ids=[t[0] for t in TRACES])
def test_hand_traces_on_gpu(policy, E, N, steps, misses, hits):
    from expert_slot_cache_topk_gb300._abi import MoECache
    c = MoECache(1, E, 1, 64, 128, "f32", N, 1, policy=policy)
    oc = LayerSlotCache(E, N, c.info()["expert_bytes"], policy=policy)
    for i, e in enumerate(steps, start=1):
        ref = _check_step(c, oc, 0, np.array([[e]]), (policy, i))
        assert ref.misses == misses.get(i, []) and ref.hits == hits.get(i, [])
    _final_state(c, oc, 0)
    c.close()


def test_slru_overflow_demotes_within_one_step_on_gpu():
    from expert_slot_cache_topk_gb300._abi import MoECache
    c = MoECache(1, 4, 2, 64, 128, "f32", 2, 1, policy="slru")
    oc = LayerSlotCache(4, 2, c.info()["expert_bytes"], policy="slru")
    for ids in ([0, 1], [0, 1], [1, 2], [3, 2], [0, 3]):
        _check_step(c, oc, 0, np.array([ids]), ids)
    _final_state(c, oc, 0)
    c.close()


@pytest.mark.parametrize("policy", POLICIES)
@pytest.mark.parametrize("slots,tokens", [(16, 1), (24, 3), (9, 1), (8, 1)])
def test_seeded_trace_matches_oracle(policy, slots, tokens):
    w = synth.WORKLOADS["olmoe"].with_(layers=1, hidden=128, inter=128, wdtype="f32", tokens=tokens)
    c = make_cache(w, slots=slots, fill=False, policy=policy)
    oc = LayerSlotCache(w.experts, slots, c.info()["expert_bytes"], policy=policy)
    lg = synth.routing_logits(w, 0, 300)
    for s in range(300):
        ids, _ = router_topk(lg[s], w.top_k)
        _check_step(c, oc, 0, ids, (policy, s))
    _final_state(c, oc, 0)
    assert oc.stats["evictions"] > 0
    c.close()


@pytest.mark.parametrize("policy", ["lfu", "slru"])
def test_policies_with_cold_set_and_moves(policy):
    w = synth.WORKLOADS["prefill_cold"].with_(layers=1, hidden=128, inter=128, wdtype="f32")
    mp = dict(interval=4, decay=float(np.float32(2.0 ** (-1.0 / 64.0))), threshold=0.5)
    cold = synth.cold_mask(w, 0)[None, :]
    c = make_cache(w, slots=12, fill=False, cold=cold, moves=mp, policy=policy)
    oc = LayerSlotCache(w.experts, 12, c.info()["expert_bytes"], cold_mask=cold[0], moves=MovePolicy(**mp),
                        policy=policy)
    lg = synth.routing_logits(w, 0, 400)
    for s in range(400):
        ids, _ = router_topk(lg[s], w.top_k)
        _check_step(c, oc, 0, ids, (policy, s))
        assert (c.get_cold(0) == oc.cold).all(), s
    _final_state(c, oc, 0)
    assert oc.stats["moves"] > 0 and oc.stats["evictions"] > 0
    c.close()


@pytest.mark.parametrize("policy", ["lfu", "fifo", "slru"])
def test_forward_under_each_policy_matches_oracle(policy):
    """The policy changes which slot holds an expert, never the result."""
    import torch
    w = synth.WORKLOADS["olmoe"].with_(layers=1)
    c = make_cache(w, slots=10, policy=policy)
    wt = OracleWeights(w)
    lgs = synth.routing_logits(w, 0, 12)
    xs = synth.hidden_states(w, 0, 12)
    for s in range(12):
        y = torch.empty((1, w.hidden), dtype=torch.bfloat16, device="cuda")
        c.forward(0, torch_x(w, xs[s]), torch.from_numpy(lgs[s]).cuda(), 1, y)
        torch.cuda.synchronize()
        assert_close(y_to_f64(w, y), oracle_y(w, wt, 0, xs[s], lgs[s]), f"{policy} step {s}")
    assert c.stats(0)["evictions"] > 0
    assert c.verify_slots(0) == 0
    c.check()
    c.close()
