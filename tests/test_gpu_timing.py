"""Timing records of the library on the GPU: per-launch miss counts and the
copy span of the staged kernel's copier warps (first chunk issued, last chunk
landed, experts copied), which the measurement of miss bandwidth divides by.
Checked against the oracle's miss / bypass lists of the same steps."""

import numpy as np
import pytest

from expert_slot_cache_topk_gb300 import synth
from oracle import router_topk
from tests.gpu_util import make_cache, oracle_slot_caches
from tests.test_gpu_forward import _forward_steps

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,slots", [("olmoe", 10), ("olmoe", 0), ("int4", 16)])
def test_copy_spans_count_the_copied_experts(name, slots):
    w = synth.WORKLOADS[name].with_(layers=1, slots=slots)
    steps = 12
    lgs = synth.routing_logits(w, 0, steps)
    xs = synth.hidden_states(w, 0, steps)
    c = make_cache(w, copy_mode="fused")
    c.set_timing(True, capacity=64)
    _forward_steps(c, w, 0, xs, lgs)
    ms, miss = c.read_timing_launches()
    spans = c.read_copy_spans()
    c.set_timing(False)
    c.check()
    c.close()
    oc = oracle_slot_caches(w)[0]
    assert len(spans) == len(ms) == steps
    for s in range(steps):
        ids, _ = router_topk(lgs[s], w.top_k)
        rec = oc.prepare(ids)
        copied = len(rec.copies)          # misses, or every non-cold expert of a bypass step
        assert copied == (len(rec.noncold) if rec.bypass else len(rec.misses))
        assert miss[s] == len(rec.misses), s
        assert int(spans[s][2]) == copied, (s, spans[s], copied)
        if copied:
            first, last = int(spans[s][0]), int(spans[s][1])
            assert 0 < first < last, (s, spans[s])
            # the copy ends within its own launch: the span is shorter than the launch
            assert (last - first) * 1e-6 <= ms[s] + 0.05, (s, last - first, ms[s])
        else:
            assert int(spans[s][1]) == 0
