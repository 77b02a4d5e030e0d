"""Pins for the slot-pool oracle: hand-worked traces, brute force, invariants,
and planted mistakes that the pins must catch."""

import numpy as np
import pytest

from oracle.slot_cache import LayerSlotCache, PrepareRecord, SLOT_POOL
from tests.golden_traces import load_traces

TRACES = load_traces()


def run_trace(tr, cls=LayerSlotCache):
    cold = np.zeros(tr.experts, dtype=bool)
    cold[tr.cold] = True
    c = cls(tr.experts, tr.slots, expert_bytes=1000, cold_mask=cold)
    recs = []
    for st in tr.steps:
        ids = np.array(st.ids, dtype=np.int64).reshape(-1, tr.topk)
        recs.append(c.prepare(ids))
    return c, recs


def trace_matches(tr, cls=LayerSlotCache) -> bool:
    try:
        c, recs = run_trace(tr, cls)
    except (KeyError, ValueError, IndexError):
        return False
    for st, rec in zip(tr.steps, recs):
        if rec.hits != st.hits or rec.misses != [tuple(m) for m in st.misses]:
            return False
        if rec.bypass != st.bypass or rec.slot_ids.reshape(-1).tolist() != st.slots:
            return False
    for key, v in tr.totals.items():
        if c.stats[key] != v:
            return False
    return True


@pytest.mark.parametrize("tr", TRACES, ids=[t.name for t in TRACES])
def test_golden_trace(tr):
    c, recs = run_trace(tr)
    for i, (st, rec) in enumerate(zip(tr.steps, recs)):
        assert rec.hits == st.hits, (tr.name, i)
        assert rec.misses == [tuple(m) for m in st.misses], (tr.name, i)
        assert rec.bypass == st.bypass, (tr.name, i)
        assert rec.slot_ids.reshape(-1).tolist() == st.slots, (tr.name, i)
    for key, v in tr.totals.items():
        assert c.stats[key] == v, (tr.name, key)
    assert c.stats["bytes_h2d_miss"] == 1000 * c.stats["misses"]


def _random_steps(seed, E, k, steps, T=1, skew=1.2):
    g = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=float) ** -skew
    p /= p.sum()
    out = []
    for _ in range(steps):
        t = g.integers(1, T + 1)
        out.append(np.stack([g.choice(E, size=k, replace=False, p=p) for _ in range(t)]))
    return out


@pytest.mark.parametrize("E,N,k,T", [(16, 4, 2, 1), (32, 8, 4, 3), (64, 16, 8, 1), (64, 16, 4, 6), (12, 12, 3, 2)])
def test_resident_set_brute_force(E, N, k, T):
    """LRU with capacity N holds the N most recently touched distinct experts.

    Brute force from the whole touch history (no OrderedDict): R_s = last N
    distinct experts touched; hits_s = |D_s & R_{s-1}|, misses_s = |D_s - R_{s-1}|,
    evicted_s = R_{s-1} - R_s.  A step touches its hits (ascending) and then its
    misses (ascending); bypass steps touch nothing.
    """
    c = LayerSlotCache(E, N, expert_bytes=7)
    history = []

    def resident():
        seen = []
        for e in reversed(history):
            if e not in seen:
                seen.append(e)
            if len(seen) == N:
                break
        return set(seen)

    tot_hits = tot_miss = 0
    for ids in _random_steps(E * 100 + N, E, k, 200, T):
        before = resident()
        D = sorted(set(ids.reshape(-1).tolist()))
        rec = c.prepare(ids)
        if len(D) > N:
            assert rec.bypass and resident() == before
            continue
        history.extend(sorted(set(D) & before) + sorted(set(D) - before))
        after = resident()
        assert set(rec.hits) == set(D) & before
        assert set(m[0] for m in rec.misses) == set(D) - before
        assert set(m[2] for m in rec.misses if m[2] >= 0) == before - after
        assert set(c.expert_to_slot) == after
        tot_hits += len(rec.hits)
        tot_miss += len(rec.misses)
        # slot_map and slot_expert are mutual inverses, slots in range
        sm, se = c.slot_map(), c.slot_expert()
        for e in range(E):
            if sm[e] >= 0:
                assert 0 <= sm[e] < N and se[sm[e]] == e
        for s in range(N):
            if se[s] >= 0:
                assert sm[se[s]] == s
        # every routed id resolves to the slot now holding its expert
        for e, v in zip(ids.reshape(-1), rec.slot_ids.reshape(-1)):
            assert v == (SLOT_POOL | int(sm[e]))
    assert c.stats["hits"] == tot_hits and c.stats["misses"] == tot_miss
    assert c.stats["bytes_h2d_miss"] == 7 * tot_miss


def test_capacity_equals_experts_no_misses_after_warmup():
    E, k = 32, 4
    c = LayerSlotCache(E, E)
    seen = set()
    for ids in _random_steps(5, E, k, 300):
        rec = c.prepare(ids)
        new = set(ids.reshape(-1).tolist()) - seen
        assert set(m[0] for m in rec.misses) == new
        seen |= new
    assert c.stats["misses"] == len(seen) and c.stats["evictions"] == 0


def test_full_miss_worst_case_disjoint_steps():
    E, k = 40, 4
    c = LayerSlotCache(E, k)
    for s in range(10):
        ids = np.arange(k * (s % 10), k * (s % 10) + k).reshape(1, k)
        rec = c.prepare(ids)
        assert len(rec.misses) == k and not rec.hits
    assert c.stats["evictions"] == 9 * k


def test_zero_slots_always_bypass_and_state_unchanged():
    E, k = 16, 3
    c = LayerSlotCache(E, 0, expert_bytes=5)
    n = 0
    for ids in _random_steps(9, E, k, 50, T=2):
        D = len(set(ids.reshape(-1).tolist()))
        rec = c.prepare(ids)
        assert rec.bypass and rec.copies == [(e, r) for r, e in enumerate(sorted(set(ids.reshape(-1).tolist())))]
        n += D
    assert c.stats["hits"] == c.stats["misses"] == 0
    assert c.stats["bypass_steps"] == 50 and c.stats["bytes_h2d_bypass"] == 5 * n


def test_bypass_does_not_touch_lru_order():
    E, N = 16, 4
    c = LayerSlotCache(E, N)
    for ids in ([[1]], [[2]], [[3]], [[4]]):
        c.prepare(np.array(ids))
    order, sm = c.lru_order(), c.slot_map().copy()
    rec = c.prepare(np.array([[5], [6], [7], [8], [9]]))
    assert rec.bypass
    assert c.lru_order() == order and (c.slot_map() == sm).all()


def test_empty_step_is_not_counted():
    c = LayerSlotCache(8, 2)
    rec = c.prepare(np.zeros((0, 2), dtype=np.int32))
    assert rec.slot_ids.shape == (0, 2) and c.stats["steps"] == 0


def test_out_of_range_id_raises():
    c = LayerSlotCache(8, 2)
    with pytest.raises(ValueError):
        c.prepare(np.array([[8]]))


# ---------------------------------------------------------------------------
# Planted mistakes: each plausible slip in the oracle must fail a pin.
# ---------------------------------------------------------------------------

class _SinglePass(LayerSlotCache):
    """The page's interleaved single ascending pass (hits and misses mixed)."""

    def prepare(self, topk_ids):
        ids = np.asarray(topk_ids, dtype=np.int64)
        D = sorted(set(ids.reshape(-1).tolist()))
        if ids.size == 0 or len(D) > self.N or self.cold.any():
            return super().prepare(ids)
        self.stats["steps"] += 1
        rec = PrepareRecord(distinct=D, noncold=D)
        for e in D:
            if e in self.expert_to_slot:
                self.lru.move_to_end(e)
                rec.hits.append(e)
                self.stats["hits"] += 1
                continue
            ev = -1
            if self.free:
                s = self.free.pop()
            else:
                ev, _ = self.lru.popitem(last=False)
                s = self.expert_to_slot.pop(ev)
                self.stats["evictions"] += 1
            self.expert_to_slot[e] = s
            self.lru[e] = None
            rec.misses.append((e, s, ev))
            self.stats["misses"] += 1
        rec.slot_ids = np.array([[self.expert_to_slot[int(e)] for e in row] for row in ids],
                                dtype=np.int32)
        return rec


class _EvictMRU(LayerSlotCache):
    """Evicts the most recently used expert not used in this step."""

    def _victim(self, step):
        return [e for e in self.lru if e not in step][-1]


class _FreeLowestFirst(LayerSlotCache):
    def reset(self):
        super().reset()
        self.free = list(range(self.N))[::-1]


class _BypassAtCapacity(LayerSlotCache):
    """Off-by-one: bypass when D >= N instead of D > N."""

    def prepare(self, topk_ids):
        n = self.N
        ids = np.asarray(topk_ids)
        if 0 < n == len(set(ids.reshape(-1).tolist())):
            self.N = n - 1
            try:
                return super().prepare(ids)
            finally:
                self.N = n
        return super().prepare(ids)


@pytest.mark.parametrize("mutant", [_SinglePass, _EvictMRU, _FreeLowestFirst, _BypassAtCapacity])
def test_planted_mistakes_fail_a_golden_trace(mutant):
    assert not all(trace_matches(tr, mutant) for tr in TRACES), mutant.__name__
