"""Pins for the oracle's run-time moves between the cold set and the pool
("Running 125B MoE on Two 32 GB Cards", sections 4.3-4.4: decayed use counts,
every few steps the most used host expert and the least used GPU-side expert
trade places when their counts differ by more than a threshold).

The two traces below were worked out by hand from those rules (see the
MovePolicy docstring for the readings); decay factors and counts were chosen
so that every float32 value involved is exact.
"""

import numpy as np
import pytest

from oracle.slot_cache import LayerSlotCache, MovePolicy


def _run(cache, seq):
    recs = []
    for e in seq:
        recs.append(cache.prepare(np.array([[e]])))
    return recs


def test_hand_trace_resident_expert_demoted_frees_its_slot():
    # E=3, N=2, k=1, cold={2}, decisions every 2 counted steps, no decay, threshold 0.5
    c = LayerSlotCache(3, 2, cold_mask=[0, 0, 1], moves=MovePolicy(interval=2, decay=1.0, threshold=0.5))
    r = _run(c, [0, 2, 2, 1, 1, 1, 0, 1])
    # step 1: 0 misses into the highest free slot 1
    assert r[0].misses == [(0, 1, -1)] and r[0].move is None
    # step 2: 2 read cold; decision: counts [1,0,1]; cold c=2 (1), non-cold min h=1 (0); 1 > 0.5 -> move
    assert r[1].cold == [2] and r[1].move == (2, 1, -1)
    # step 3: 2 is no longer cold: a miss into slot 0
    assert r[2].misses == [(2, 0, -1)]
    # step 4: 1 read cold; decision: counts [1,1,2]; c=1 (1), h=0 (1); 0 > 0.5 false
    assert r[3].cold == [1] and r[3].move is None
    # step 6: counts [1,3,2]; c=1 (3), h=0 (1, resident in slot 1); 2 > 0.5 -> move, slot 1 freed
    assert r[5].move == (1, 0, 1)
    # step 7: 0 is cold now: read in place, no miss
    assert r[6].cold == [0] and r[6].misses == []
    # step 8: 1 misses into the freed slot 1; decision: counts [2,4,2]; c=0 (2), h=2 (2); no move
    assert r[7].misses == [(1, 1, -1)] and r[7].move is None
    assert c.cold.tolist() == [True, False, False]
    assert c.slot_map().tolist() == [-1, 1, 0]
    assert c.counts.tolist() == [2.0, 4.0, 2.0]
    st = c.stats
    assert (st["misses"], st["hits"], st["evictions"], st["moves"], st["cold_reads"]) == (3, 0, 0, 2, 5)


def test_hand_trace_with_decay_and_strict_threshold():
    # E=4, N=2, k=1, cold={3}, decisions every 2 counted steps, decay 0.5, threshold 0.5
    c = LayerSlotCache(4, 2, cold_mask=[0, 0, 0, 1], moves=MovePolicy(interval=2, decay=0.5, threshold=0.5))
    r = _run(c, [3, 3, 3, 0, 0, 2, 0, 1, 2, 1, 0, 2, 1, 3])
    moves = {i + 1: rec.move for i, rec in enumerate(r) if rec.move is not None}
    # step 2: counts [0,0,0,2]*0.5 = [0,0,0,1]; c=3, h=0 (tie 0/1/2 -> lowest id); 1 > 0.5
    # step 4: [1,0,0,2]*0.5 = [0.5,0,0,1]; c=0 (0.5), h=1 (0); 0.5 > 0.5 false
    # step 6: [1.5,0,1,1]*0.5 = [0.75,0,0.5,0.5]; c=0, h=1; 0.75 > 0.5 -> move
    # step 8: [1.75,1,0.5,0.5]*0.5 = [0.875,0.5,0.25,0.25]; c=1 (0.5), h=2 (0.25); 0.25 > 0.5 false
    # step 10: [0.875,1.5,1.25,0.25]*0.5 = [0.4375,0.75,0.625,0.125]; c=1, h=3 (0.125); 0.625 > 0.5 -> move
    # step 12: [1.4375,0.75,1.625,0.125]*0.5 = [0.71875,0.375,0.8125,0.0625]; c=3, h=1; negative
    # step 14: [0.71875,1.375,0.8125,1.0625]*0.5 = [0.359375,0.6875,0.40625,0.53125]; c=3, h=0; 0.171875
    assert moves == {2: (3, 0, -1), 6: (0, 1, -1), 10: (1, 3, -1)}
    assert [rec.misses for rec in r if rec.misses] == [
        [(3, 1, -1)],          # step 3: 3 is warm now, highest free slot
        [(2, 0, -1)],          # step 6
        [(0, 1, 3)],           # step 7: 0 warm again, evicts LRU 3 (last used step 3)
        [(1, 1, 0)],           # step 13: 1 warm, evicts LRU 0 (2 was hit at step 12)
    ]
    assert [i + 1 for i, rec in enumerate(r) if rec.hits] == [9, 11, 12]
    assert c.counts.tolist() == [0.359375, 0.6875, 0.40625, 0.53125]
    assert c.cold.tolist() == [False, False, False, True]
    assert c.stats["moves"] == 3 and c.stats["evictions"] == 2


def test_cold_set_size_is_invariant_and_cold_experts_never_resident():
    g = np.random.default_rng(3)
    E, N = 32, 6
    cold = np.zeros(E, bool)
    cold[g.choice(E, 5, replace=False)] = True
    c = LayerSlotCache(E, N, cold_mask=cold, moves=MovePolicy(interval=4, threshold=0.25))
    probs = g.dirichlet(np.full(E, 0.3))
    for _ in range(600):
        ids = g.choice(E, 2, replace=False, p=probs)
        c.prepare(ids[None, :])
        assert c.cold.sum() == 5
        assert not any(c.cold[e] for e in c.expert_to_slot)
        assert len(c.expert_to_slot) + len(c.free) == N
        assert sorted(list(c.expert_to_slot.values()) + c.free) == list(range(N))
    assert c.stats["moves"] > 0


def test_steps_over_the_token_limit_are_not_counted():
    c = LayerSlotCache(4, 2, cold_mask=[0, 0, 0, 1], moves=MovePolicy(interval=1, decay=1.0, count_tokens=1))
    c.prepare(np.array([[3], [3]]))          # two tokens: not counted, no decision
    assert c.counts.tolist() == [0, 0, 0, 0] and c.stats["moves"] == 0
    c.prepare(np.array([[3]]))               # counted: [0,0,0,1]; 1 > 2 false
    assert c.counts.tolist() == [0, 0, 0, 1] and c.stats["moves"] == 0


def test_reset_restores_the_initial_cold_set():
    c = LayerSlotCache(3, 2, cold_mask=[0, 0, 1], moves=MovePolicy(interval=2, decay=1.0, threshold=0.5))
    _run(c, [0, 2])
    assert c.cold.tolist() == [False, True, False]
    c.reset()
    assert c.cold.tolist() == [False, False, True] and c.counts.tolist() == [0, 0, 0]


class _NoDecay(LayerSlotCache):
    def _count_and_move(self, ids, rec):
        mp = self.moves
        self.moves = MovePolicy(mp.interval, 1.0, mp.threshold, mp.count_tokens)
        try:
            super()._count_and_move(ids, rec)
        finally:
            self.moves = mp


class _NonStrict(LayerSlotCache):
    def _count_and_move(self, ids, rec):
        mp = self.moves
        self.moves = MovePolicy(mp.interval, mp.decay, np.nextafter(np.float32(mp.threshold), np.float32(-1)),
                                mp.count_tokens)
        try:
            super()._count_and_move(ids, rec)
        finally:
            self.moves = mp


class _KeepSlot(LayerSlotCache):
    """Demoted expert keeps its slot (the freed-slot rule dropped)."""

    def _count_and_move(self, ids, rec):
        saved = dict(self.expert_to_slot), OrderedDict_copy(self.lru), list(self.free)
        super()._count_and_move(ids, rec)
        if rec.move is not None and rec.move[2] >= 0:
            self.expert_to_slot, self.lru, self.free = saved


def OrderedDict_copy(od):
    from collections import OrderedDict
    return OrderedDict(od)


@pytest.mark.parametrize("mutant", [_NoDecay, _NonStrict, _KeepSlot])
def test_planted_mistakes_fail_a_hand_trace(mutant):
    def trace_a(cls):
        c = cls(3, 2, cold_mask=[0, 0, 1], moves=MovePolicy(interval=2, decay=1.0, threshold=0.5))
        r = _run(c, [0, 2, 2, 1, 1, 1, 0, 1])
        return [x.move for x in r], [x.misses for x in r], c.slot_map().tolist()

    def trace_b(cls):
        c = cls(4, 2, cold_mask=[0, 0, 0, 1], moves=MovePolicy(interval=2, decay=0.5, threshold=0.5))
        r = _run(c, [3, 3, 3, 0, 0, 2, 0, 1, 2, 1, 0, 2, 1, 3])
        return [x.move for x in r], [x.misses for x in r]

    assert trace_a(mutant) != trace_a(LayerSlotCache) or trace_b(mutant) != trace_b(LayerSlotCache)
