"""One VMM table per layer (device rows = pool slots, then host rows = the
backing store; "Running 125B MoE on Two 32 GB Cards", section 4.2): the table's
shape, weights written by the CPU through the table, and decode / multi-token /
bypass results identical to the split layout in every copy mode."""

import numpy as np
import pytest

from expert_slot_cache_topk_gb300 import synth
from tests.gpu_util import OracleWeights, assert_close, make_cache, oracle_y, y_to_f64
from tests.test_gpu_forward import _forward_steps

pytestmark = pytest.mark.gpu
W = synth.WORKLOADS


def test_table_rows_are_adjacent():
    w = W["olmoe"].with_(layers=3)
    c = make_cache(w, slots=10, table="vmm", fill=False)
    info = c.info()
    assert info["table_layout"] == 1
    stride = info["slot_stride"]
    g = 2 << 20
    pool_part = (10 * stride + g - 1) // g * g
    host_part = (w.experts * stride + g - 1) // g * g
    pools = [c.pool_ptrs(l)[0] for l in range(3)]
    for l in range(3):
        back = c.backing_view(l).ctypes.data
        assert back == pools[l] + pool_part          # host rows follow the layer's device rows
        if l:
            assert pools[l] == pools[l - 1] + pool_part + host_part
    c.close()


@pytest.mark.parametrize("mode", ["uva", "fused", "memcpy"])
def test_decode_identical_to_split_layout(mode):
    import torch
    w = W["olmoe"].with_(layers=2)
    steps = 8
    outs = {}
    for table in ("split", "vmm"):
        c = make_cache(w, slots=w.top_k + 3, copy_mode=mode, table=table)
        ys = []
        for l in range(2):
            ys += [y.clone() for y in _forward_steps(c, w, l, synth.hidden_states(w, l, steps),
                                                     synth.routing_logits(w, l, steps))]
            assert c.verify_slots(l) == 0
        assert c.stats(-1)["misses"] > 0 and c.stats(-1)["evictions"] > 0
        c.check()
        c.close()
        outs[table] = ys
    for a, b in zip(outs["split"], outs["vmm"]):
        assert torch.equal(a, b)
    wt = OracleWeights(w)
    xs, lgs = synth.hidden_states(w, 1, steps), synth.routing_logits(w, 1, steps)
    for s in range(steps):
        assert_close(y_to_f64(w, outs["vmm"][steps + s]), oracle_y(w, wt, 1, xs[s], lgs[s]), f"{mode} step {s}")


def test_cold_set_bypass_and_multi_token_steps():
    import torch
    w = W["prefill_cold"].with_(layers=1, hidden=256, inter=128, tokens=24)
    cold = synth.cold_mask(w, 0)[None, :]
    lgs = synth.routing_logits(w, 0, 3)
    xs = synth.hidden_states(w, 0, 3)
    outs = {}
    for table in ("split", "vmm"):
        for slots in (64, 0):
            c = make_cache(w, slots=slots, cold=cold, table=table)
            outs[(table, slots)] = [y.clone() for y in _forward_steps(c, w, 0, xs, lgs)]
            st = c.stats(0)
            assert st["cold_reads"] > 0
            if slots == 0:
                assert st["bypass_steps"] == 3
            c.check()
            c.close()
    for slots in (64, 0):
        for a, b in zip(outs[("split", slots)], outs[("vmm", slots)]):
            assert torch.equal(a, b)


def test_load_expert_refreshes_a_resident_slot():
    w = W["tiny"]
    c = make_cache(w, slots=w.experts, table="vmm")
    _forward_steps(c, w, 0, synth.hidden_states(w, 0, 4), synth.routing_logits(w, 0, 4))
    sm, _, _, _ = c.get_state(0)
    e = int(np.nonzero(sm >= 0)[0][0])
    blk = synth.expert_block(w.with_(cfg_id=99), 0, e)
    c.load_expert(0, e, blk)
    assert c.verify_slots(0) == 0
    assert np.array_equal(c.backing_view(0)[e, : blk.size], blk)
    c.close()


def test_create_and_destroy_repeatedly():
    w = W["olmoe"].with_(layers=4)
    for _ in range(3):
        c = make_cache(w, slots=16, table="vmm", fill=False)
        c.close()
