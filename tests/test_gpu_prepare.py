"""Slot bookkeeping on the GPU: the hand-worked traces and full routing traces
of every workload must match the oracle bit for bit (slot ids, hits, misses,
evictions, bypass, cold, counters, final state)."""

import numpy as np
import pytest

from expert_slot_cache_topk_gb300 import synth
from oracle import router_topk
from tests.golden_traces import load_traces
from tests.gpu_util import make_cache, oracle_slot_caches

pytestmark = pytest.mark.gpu
TRACES = load_traces()


def _prepare(c, layer, ids_np):
    import torch
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    out = torch.full(ids.shape, -99, dtype=torch.int32, device="cuda")
    c.prepare(layer, ids, ids.shape[0], out)
    return out


@pytest.mark.parametrize("copy_mode", ["uva", "memcpy", "fused"])
@pytest.mark.parametrize("tr", TRACES, ids=[t.name for t in TRACES])
def test_golden_trace_on_gpu(tr, copy_mode):
    from expert_slot_cache_topk_gb300._abi import MoECache
    cold = np.zeros((1, tr.experts), np.uint8)
    cold[0, tr.cold] = 1
    maxT = max(len(s.ids) // tr.topk for s in tr.steps)
    c = MoECache(1, tr.experts, tr.topk, 64, 128, "f32", tr.slots, maxT, cold_mask=cold,
                 copy_mode=copy_mode)
    for i, st in enumerate(tr.steps):
        out = _prepare(c, 0, np.array(st.ids).reshape(-1, tr.topk))
        rec = c.last_prepare(0)
        assert rec["hits"] == st.hits, (tr.name, i)
        assert rec["misses"] == [tuple(m) for m in st.misses], (tr.name, i)
        assert rec["bypass"] == st.bypass, (tr.name, i)
        assert out.cpu().numpy().reshape(-1).astype(np.int64).tolist() == st.slots, (tr.name, i)
    s = c.stats(0)
    for key, v in tr.totals.items():
        assert s[key] == v, (tr.name, key)
    assert c.verify_slots(0) == 0
    c.close()


def _trace_workload(w, steps, layers=None, slots=None, prefill=False):
    """Run the integer trace of `w` through moe_cache_prepare and the oracle."""
    L = w.layers if layers is None else layers
    w = w.with_(layers=L)
    small = w.with_(hidden=128, inter=128, wdtype="f32")   # the trace does not depend on H, I, format
    T = w.prefill_tokens if prefill else w.tokens
    c = make_cache(small, slots=slots, max_tokens=max(T, w.tokens), fill=False,
                   cold=np.stack([synth.cold_mask(w, l) for l in range(L)]) if w.cold_frac else None)
    oc = oracle_slot_caches(small, slots=slots,
                            cold=np.stack([synth.cold_mask(w, l) for l in range(L)]) if w.cold_frac else None)
    for l in range(L):
        seq = []
        if prefill:
            seq.append(synth.prefill_logits(w, l))
        lg = synth.routing_logits(w, l, steps)
        seq.extend(lg[s] for s in range(steps))
        for i, logits in enumerate(seq):
            ids, _ = router_topk(logits, w.top_k)
            out = _prepare(c, l, ids)
            ref = oc[l].prepare(ids)
            rec = c.last_prepare(l)
            where = (w.name, l, i)
            assert rec["bypass"] == ref.bypass, where
            assert rec["hits"] == ref.hits, where
            assert rec["misses"] == ref.misses, where
            assert rec["cold"] == ref.cold and rec["noncold"] == ref.noncold, where
            assert (out.cpu().numpy() == ref.slot_ids).all(), where
        sm, se, _, nfree = c.get_state(l)
        assert (sm == oc[l].slot_map()).all() and (se == oc[l].slot_expert()).all()
        assert nfree == len(oc[l].free)
        s = c.stats(l)
        for key, v in oc[l].stats.items():
            assert s[key] == v * (1 if not key.startswith("bytes") else 1), (w.name, l, key)
    c.close()


def test_trace_tiny_full():
    _trace_workload(synth.WORKLOADS["tiny"], 64)


def test_trace_olmoe_full():
    _trace_workload(synth.WORKLOADS["olmoe"], 512)


@pytest.mark.parametrize("N", [0, 16, 32, 64])
def test_trace_int4_slots(N):
    _trace_workload(synth.WORKLOADS["int4"], 512, layers=4, slots=N)


def test_trace_batched_bypass():
    _trace_workload(synth.WORKLOADS["batched"], 64, layers=2)


def test_trace_prefill_then_decode_with_cold_set():
    _trace_workload(synth.WORKLOADS["prefill_cold"], 128, layers=2, prefill=True)


def test_trace_prefill_cold_all_noncold_resident():
    w = synth.WORKLOADS["prefill_cold"]
    _trace_workload(w, 64, layers=1, slots=w.experts - w.n_cold, prefill=True)
