"""Pins for the oracle's eviction policies (vLLM PR #37190, the review thread
that added --moe-expert-cache-policy: lru, lfu = least frequently used,
fifo = insertion order, slru = probationary -> protected with a 20 % / 80 %
split).  Each trace was worked out by hand from the rules in the oracle's
docstring and is chosen so that it tells the policy apart from LRU."""

import numpy as np
import pytest

from oracle.slot_cache import POLICIES, LayerSlotCache

# (policy, E, N, steps (one expert per step), expected misses per step, expected hits per step)
TRACES = [
    # FIFO: a hit does not refresh; step 4 evicts 0 (first in), where LRU evicts 1
    ("fifo", 4, 2, [0, 1, 0, 2, 0, 3],
     {1: [(0, 1, -1)], 2: [(1, 0, -1)], 4: [(2, 1, 0)], 5: [(0, 0, 1)], 6: [(3, 1, 2)]}, {3: [0]}),
    # LFU: after steps 3-4 both residents were used in 2 steps; the tie goes to
    # the earliest inserted (0; LRU would evict 1); step 6 evicts 2 (used once;
    # FIFO would evict 1)
    ("lfu", 4, 2, [0, 1, 1, 0, 2, 3],
     {1: [(0, 1, -1)], 2: [(1, 0, -1)], 5: [(2, 1, 0)], 6: [(3, 1, 2)]}, {3: [1], 4: [0]}),
    # SLRU, N = 3, protected holds floor(2.4) = 2: step 5 evicts probationary 1
    # although protected 0 is older (LRU evicts 0); step 7 promotes 3 and
    # demotes 0 to probationary, which step 8 then evicts
    ("slru", 4, 3, [0, 0, 1, 2, 3, 2, 3, 1, 2, 0],
     {1: [(0, 2, -1)], 3: [(1, 1, -1)], 4: [(2, 0, -1)], 5: [(3, 1, 1)], 8: [(1, 2, 0)], 10: [(0, 2, 1)]},
     {2: [0], 6: [2], 7: [3], 9: [2]}),
]


def run(policy, E, N, steps):
    c = LayerSlotCache(E, N, policy=policy)
    recs = [c.prepare(np.array([[e]])) for e in steps]
    return c, recs


@pytest.mark.parametrize("policy,E,N,steps,misses,hits", TRACES, ids=[t[0] for t in TRACES])
def test_hand_trace(policy, E, N, steps, misses, hits):
    c, recs = run(policy, E, N, steps)
    for i, r in enumerate(recs, start=1):
        assert r.misses == misses.get(i, []), (policy, i)
        assert r.hits == hits.get(i, []), (policy, i)
    assert c.stats["evictions"] == sum(1 for m in misses.values() for x in m if x[2] >= 0)


@pytest.mark.parametrize("policy,E,N,steps,misses,hits", TRACES, ids=[t[0] for t in TRACES])
def test_trace_differs_from_lru(policy, E, N, steps, misses, hits):
    _, mine = run(policy, E, N, steps)
    _, lru = run("lru", E, N, steps)
    assert [r.misses for r in mine] != [r.misses for r in lru]


def test_slru_demotes_a_step_entry_when_protected_overflows():
    # N = 2: protected holds 1.  Step {0, 1} with both probationary: 0 is
    # promoted, then 1, which overflows the protected segment and demotes 0.
    c = LayerSlotCache(4, 2, policy="slru")
    c.prepare(np.array([[0, 1]]))
    c.prepare(np.array([[0, 1]]))
    assert list(c.prot) == [1] and list(c.prob) == [0]
    r = c.prepare(np.array([[1, 2]]))          # victim: probationary 0 (not in this step)
    assert r.misses == [(2, c.slot_map()[2], 0)]


@pytest.mark.parametrize("policy", POLICIES)
def test_invariants_and_never_evict_a_step_expert(policy):
    g = np.random.default_rng(11)
    E, N, k = 24, 7, 3
    c = LayerSlotCache(E, N, policy=policy)
    p = g.dirichlet(np.full(E, 0.4))
    for _ in range(500):
        ids = g.choice(E, k, replace=False, p=p)
        before = dict(c.expert_to_slot)
        r = c.prepare(ids[None, :])
        for e, s, ev in r.misses:
            assert ev not in set(ids.tolist())
            if ev >= 0:
                assert before[ev] == s
        assert sorted(list(c.expert_to_slot.values()) + c.free) == list(range(N))
        if policy == "slru":
            assert len(c.prot) <= (4 * N) // 5 and len(c.prot) + len(c.prob) == len(c.expert_to_slot)
    assert c.stats["hits"] + c.stats["misses"] == 500 * k - 0  # no bypass (k <= N), no cold


def test_unknown_policy_rejected():
    with pytest.raises(ValueError):
        LayerSlotCache(4, 2, policy="arc")
