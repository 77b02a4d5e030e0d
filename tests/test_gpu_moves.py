"""Run-time moves between the cold set and the pool on the GPU against the
oracle, bit for bit: the hand-worked move traces, and long seeded decode
traces of the prefill + cold-set shapes (per step: misses, hits, cold and
non-cold lists, slot ids; the cold set after every step; final pool state and
counters)."""

import numpy as np
import pytest

from expert_slot_cache_topk_gb300 import synth
from oracle import router_topk
from oracle.slot_cache import LayerSlotCache, MovePolicy
from tests.gpu_util import OracleWeights, assert_close, make_cache, oracle_y, torch_x, y_to_f64

pytestmark = pytest.mark.gpu
PAGES_DECAY = float(np.float32(2.0 ** (-1.0 / 64.0)))


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
    assert rec["cold"] == ref.cold and rec["noncold"] == ref.noncold, where
    assert (out == ref.slot_ids).all(), where
    assert (c.get_cold(layer) == oc.cold).all(), where
    return ref


def _final_state(c, oc, layer):
    sm, se, _, nfree = c.get_state(layer)
    assert (sm == oc.slot_map()).all() and (se == oc.slot_expert()).all()
    assert nfree == len(oc.free)
    s = c.stats(layer)
    for key, v in oc.stats.items():
        assert s[key] == v, key


@pytest.mark.parametrize("E,N,cold,mp,seq", [
    (3, 2, [0, 0, 1], dict(interval=2, decay=1.0, threshold=0.5), [0, 2, 2, 1, 1, 1, 0, 1]),
    (4, 2, [0, 0, 0, 1], dict(interval=2, decay=0.5, threshold=0.5), [3, 3, 3, 0, 0, 2, 0, 1, 2, 1, 0, 2, 1, 3]),
])
def test_hand_traces_on_gpu(E, N, cold, mp, seq):
    from expert_slot_cache_topk_gb300._abi import MoECache
    c = MoECache(1, E, 1, 64, 128, "f32", N, 1, cold_mask=np.array([cold], np.uint8), moves=mp)
    oc = LayerSlotCache(E, N, c.info()["expert_bytes"], cold_mask=cold, moves=MovePolicy(**mp))
    for i, e in enumerate(seq):
        _check_step(c, oc, 0, np.array([[e]]), i)
    _final_state(c, oc, 0)
    assert c.stats(0)["moves"] >= 2
    c.close()


@pytest.mark.parametrize("interval,threshold,slots", [(8, 2.0, 64), (4, 0.5, 16), (8, 2.0, 0)])
def test_decode_trace_with_moves_matches_oracle(interval, threshold, slots):
    w = synth.WORKLOADS["prefill_cold"].with_(layers=2, hidden=128, inter=128, wdtype="f32")
    mp = dict(interval=interval, decay=PAGES_DECAY, threshold=threshold, count_tokens=1)
    cold = np.stack([synth.cold_mask(w, l) for l in range(w.layers)])
    c = make_cache(w, slots=slots, fill=False, cold=cold, moves=mp)
    moved = 0
    for l in range(w.layers):
        oc = LayerSlotCache(w.experts, slots, c.info()["expert_bytes"], cold_mask=cold[l], moves=MovePolicy(**mp))
        lg = synth.routing_logits(w, l, 512)
        for s in range(512):
            ids, _ = router_topk(lg[s], w.top_k)
            _check_step(c, oc, l, ids, (l, s))
        _final_state(c, oc, l)
        moved += oc.stats["moves"]
    assert moved > 0
    c.close()


def test_multi_token_steps_count_when_allowed():
    w = synth.WORKLOADS["prefill_cold"].with_(layers=1, hidden=128, inter=128, wdtype="f32", tokens=4)
    mp = dict(interval=3, decay=PAGES_DECAY, threshold=1.0, count_tokens=4)
    cold = synth.cold_mask(w, 0)[None, :]
    c = make_cache(w, slots=64, fill=False, cold=cold, moves=mp)
    oc = LayerSlotCache(w.experts, 64, c.info()["expert_bytes"], cold_mask=cold[0], moves=MovePolicy(**mp))
    lg = synth.routing_logits(w, 0, 96)
    for s in range(96):
        ids, _ = router_topk(lg[s], w.top_k)
        _check_step(c, oc, 0, ids, s)
    _final_state(c, oc, 0)
    c.close()


def test_reset_restores_the_cold_set():
    w = synth.WORKLOADS["prefill_cold"].with_(layers=1, hidden=128, inter=128, wdtype="f32")
    mp = dict(interval=2, decay=1.0, threshold=0.0)
    cold = synth.cold_mask(w, 0)[None, :]
    c = make_cache(w, slots=16, fill=False, cold=cold, moves=mp)
    lg = synth.routing_logits(w, 0, 40)
    for s in range(40):
        ids, _ = router_topk(lg[s], w.top_k)
        _prepare(c, 0, ids)
    assert c.stats(0)["moves"] > 0 and (c.get_cold(0) != cold[0].astype(bool)).any()
    c.reset()
    assert (c.get_cold(0) == cold[0].astype(bool)).all() and c.stats(0)["moves"] == 0
    c.close()


def test_forward_with_moves_matches_oracle():
    """Moves change where experts are read from, never the result."""
    import torch
    w = synth.WORKLOADS["prefill_cold"].with_(layers=1)
    mp = dict(interval=2, decay=PAGES_DECAY, threshold=0.5)
    for mode in ("fused", "uva"):
        c = make_cache(w, slots=16, copy_mode=mode, moves=mp)
        wt = OracleWeights(w)
        lgs = synth.routing_logits(w, 0, 24)
        xs = synth.hidden_states(w, 0, 24)
        for s in range(24):
            y = torch.empty((1, w.hidden), dtype=torch.bfloat16, device="cuda")
            c.forward(0, torch_x(w, xs[s]), torch.from_numpy(lgs[s]).cuda(), 1, y)
            torch.cuda.synchronize()
            assert_close(y_to_f64(w, y), oracle_y(w, wt, 0, xs[s], lgs[s]), f"{mode} step {s}")
        assert c.stats(0)["moves"] > 0
        assert c.verify_slots(0) == 0
        c.check()
        c.close()
