"""Per-layer expert slot pool with LRU bookkeeping (oracle).

Test infrastructure: see the package docstring.

What it follows
---------------
* LRU kept as an ``OrderedDict`` with the front as least recently used: a hit
  moves the expert to the end; a miss takes a free slot with ``list.pop()``
  from ``list(range(capacity))`` (so the highest free index first), or else
  evicts the front with ``popitem(last=False)``; the id->slot mapping is
  updated in place and ``topk_ids`` are remapped through it
  (vLLM PR #37190 "Run MoE models exceeding VRAM via expert CPU offloading with
  GPU cache", sections "Architecture" and "How it works", and the review thread
  that replaced the list with an OrderedDict).
* The distinct experts of a step come from ``topk_ids.unique()``, i.e. in
  ascending id order (same page, "How it works").
* Bypass: a ubatch that touches more distinct experts than the pool has slots
  does not go through the pool and takes the selective-copy path; nothing is
  evicted (llama.cpp discussion #28248 "RFC: Persistent expert slot pool for
  MoE CPU offload", section "Why not the other approaches on the table" and
  "Design" item 2).  Rule used here: bypass iff (distinct non-cold experts) > N.
* Cold set: chosen experts stay in pinned host memory, are read through UVA
  and never enter the pool ("Running 125B MoE on Two 32 GB Cards", sections
  2 and 3 "Only the least used experts in host RAM (offload-02)").

Readings where the pages are open
---------------------------------
* Within a step, hits are touched first (ascending id), then misses are
  filled (ascending id).  Because the non-cold distinct count D is at most N on
  the pool path, the LRU front during the miss pass is never an expert used in
  this step.
* A bypass copies all D non-cold experts (resident ones too) into scratch at
  index = rank of the expert among them; LRU state and hit/miss counters are
  untouched.
* An empty step (no ids) is not a step: nothing changes and nothing is counted.

Slot-id encoding (the library's documented output encoding)
-----------------------------------------------------------
``kind << 29 | index`` with kind 0 = pool slot, 1 = bypass scratch position,
2 = cold expert id (read from host memory).
"""

from __future__ import annotations

from collections import OrderedDict
from dataclasses import dataclass, field

import numpy as np

SLOT_KIND_SHIFT = 29
SLOT_POOL = 0 << SLOT_KIND_SHIFT
SLOT_SCRATCH = 1 << SLOT_KIND_SHIFT
SLOT_COLD = 2 << SLOT_KIND_SHIFT


def decode_slot_id(v: int) -> tuple[str, int]:
    kind = v >> SLOT_KIND_SHIFT
    idx = v & ((1 << SLOT_KIND_SHIFT) - 1)
    return ({0: "pool", 1: "scratch", 2: "cold"}[kind], idx)


@dataclass
class PrepareRecord:
    distinct: list = field(default_factory=list)   # ascending distinct ids
    cold: list = field(default_factory=list)       # ascending cold ids
    noncold: list = field(default_factory=list)    # ascending non-cold ids (D)
    bypass: bool = False
    hits: list = field(default_factory=list)       # ascending
    misses: list = field(default_factory=list)     # (expert, slot, evicted|-1), ascending expert
    copies: list = field(default_factory=list)     # (expert, dest index) in copy order
    slot_ids: np.ndarray = None                    # int32, same shape as topk_ids
    move: tuple = None                             # (expert leaving the cold set, expert joining it,
                                                   #  slot freed by the latter or -1), if a move happened


POLICIES = ("lru", "lfu", "fifo", "slru")

STAT_KEYS = ("steps", "hits", "misses", "evictions", "bypass_steps", "cold_reads",
             "bytes_h2d_miss", "bytes_h2d_bypass", "bytes_uva_cold", "moves")


@dataclass
class MovePolicy:
    """Run-time moves between the cold set and the pool ("Running 125B MoE on
    Two 32 GB Cards", sections 4.3 "Moving experts at run time: simulation"
    and 4.4 "... implementation": per-layer use counts from the decode router,
    decayed, every few steps the most used host expert and the least used
    GPU-side expert trade places when their counts differ by more than a
    threshold, one pair per layer).

    Readings taken here:
    * a step is counted when it has at most ``count_tokens`` tokens (the pages
      count decode steps and not prefill; decode there is batch 1);
    * a counted step adds, to each expert, the number of its assignments in
      that step, in one float32 addition;
    * every ``interval`` counted steps, after the step's bookkeeping: the counts
      are multiplied by ``decay`` (float32; 0.5 ** (8 / 512) = 2 ** (-1/64) for
      the pages' interval 8 and half-life 512), then c = the cold expert with
      the largest count and h = the non-cold expert with the smallest count
      (ties to the lower id); if float32(count[c] - count[h]) > threshold, c
      leaves the cold set and h joins it;
    * nothing is copied at the decision: c is copied into a slot at its next
      use (an ordinary miss); if h holds a slot, the slot is freed (pushed on
      the free-slot stack, so the next miss takes it first) and h is read in
      place from then on;
    * all count arithmetic is float32, as on the GPU, so the integer outcomes
      (which experts move) are decided in the same precision.
    """

    interval: int = 8
    decay: float = float(np.float32(2.0 ** (-1.0 / 64.0)))
    threshold: float = 2.0
    count_tokens: int = 1


class LayerSlotCache:
    """One MoE layer's pool of ``slots`` expert slots."""

    def __init__(self, num_experts: int, slots: int, expert_bytes: int = 0, cold_mask=None,
                 moves: "MovePolicy | None" = None, policy: str = "lru"):
        if not 0 <= slots <= num_experts:
            raise ValueError("need 0 <= slots <= num_experts")
        if policy not in POLICIES:
            raise ValueError(f"policy must be one of {POLICIES}")
        self.policy = policy
        self.E = num_experts
        self.N = slots
        self.B = expert_bytes
        self.cold0 = (np.zeros(num_experts, dtype=bool) if cold_mask is None
                      else np.asarray(cold_mask, dtype=bool).copy())
        self.moves = moves
        self.reset()

    def reset(self):
        # lru: recency order (front = least recently used); fifo / lfu: insertion
        # order; slru: unused (prob / prot hold the two segments)
        self.lru: "OrderedDict[int, None]" = OrderedDict()
        self.freq: dict[int, int] = {}                        # lfu: steps used since insertion
        self.prob: "OrderedDict[int, None]" = OrderedDict()   # slru probationary, front = LRU
        self.prot: "OrderedDict[int, None]" = OrderedDict()   # slru protected, front = LRU
        self.expert_to_slot: dict[int, int] = {}
        self.free: list[int] = list(range(self.N))            # a stack: pop() from the end
        self.stats = {k: 0 for k in STAT_KEYS}
        self.cold = self.cold0.copy()
        self.counts = np.zeros(self.E, dtype=np.float32)
        self.counted_steps = 0

    # -- views used by tests -------------------------------------------------
    def slot_map(self) -> np.ndarray:
        m = np.full(self.E, -1, dtype=np.int32)
        for e, s in self.expert_to_slot.items():
            m[e] = s
        return m

    def slot_expert(self) -> np.ndarray:
        m = np.full(self.N, -1, dtype=np.int32)
        for e, s in self.expert_to_slot.items():
            m[s] = e
        return m

    def lru_order(self) -> list:
        return list(self.lru.keys())

    # -- one step --------------------------------------------------------------
    def prepare(self, topk_ids) -> PrepareRecord:
        ids = np.asarray(topk_ids, dtype=np.int64)
        rec = PrepareRecord()
        if ids.size == 0:
            rec.slot_ids = np.zeros(ids.shape, dtype=np.int32)
            return rec
        if ids.min() < 0 or ids.max() >= self.E:
            raise ValueError("expert id out of range")
        self.stats["steps"] += 1

        rec.distinct = sorted(set(int(e) for e in ids.reshape(-1)))
        rec.cold = [e for e in rec.distinct if self.cold[e]]
        rec.noncold = [e for e in rec.distinct if not self.cold[e]]
        self.stats["cold_reads"] += len(rec.cold)
        self.stats["bytes_uva_cold"] += len(rec.cold) * self.B

        scratch_pos = {}
        if len(rec.noncold) > self.N:
            rec.bypass = True
            self.stats["bypass_steps"] += 1
            self.stats["bytes_h2d_bypass"] += len(rec.noncold) * self.B
            for r, e in enumerate(rec.noncold):
                scratch_pos[e] = r
                rec.copies.append((e, r))
        else:
            step = set(rec.noncold)
            for e in rec.noncold:                      # hits first, ascending
                if e in self.expert_to_slot:
                    self._touch(e)
                    rec.hits.append(e)
                    self.stats["hits"] += 1
            for e in rec.noncold:                      # then misses, ascending
                if e in self.expert_to_slot:
                    continue
                evicted = -1
                if self.free:
                    s = self.free.pop()
                else:
                    evicted = self._victim(step)
                    self._remove(evicted)
                    s = self.expert_to_slot.pop(evicted)
                    self.stats["evictions"] += 1
                self.expert_to_slot[e] = s
                self._insert(e)
                rec.misses.append((e, s, evicted))
                rec.copies.append((e, s))
                self.stats["misses"] += 1
                self.stats["bytes_h2d_miss"] += self.B

        out = np.empty(ids.shape, dtype=np.int32)
        flat_in, flat_out = ids.reshape(-1), out.reshape(-1)
        for i, e in enumerate(flat_in):
            e = int(e)
            if self.cold[e]:
                flat_out[i] = SLOT_COLD | e
            elif rec.bypass:
                flat_out[i] = SLOT_SCRATCH | scratch_pos[e]
            else:
                flat_out[i] = SLOT_POOL | self.expert_to_slot[e]
        rec.slot_ids = out
        if self.moves is not None:
            self._count_and_move(ids, rec)
        return rec

    # -- eviction policies ---------------------------------------------------------
    # vLLM PR #37190 (the review thread that added --moe-expert-cache-policy):
    # lru = least recently used, lfu = least frequently used, fifo = insertion
    # order, slru = two segments, probationary -> protected, a 20 % / 80 %
    # split.  Readings: every policy keeps the hits-before-misses order, and
    # an expert used in the current step is never the victim; lfu counts the
    # steps an expert was used in since it was inserted, ties to the earliest
    # inserted; slru's protected segment holds floor(0.8 N) experts, a hit on
    # a probationary expert promotes it to the protected MRU end, overflow
    # demotes the protected LRU expert to the probationary MRU end, and the
    # victim is the probationary LRU expert (the protected LRU one when the
    # probationary segment has no candidate).
    def _touch(self, e: int):
        if self.policy == "lru":
            self.lru.move_to_end(e)
        elif self.policy == "lfu":
            self.freq[e] += 1
        elif self.policy == "slru":
            if e in self.prob:
                del self.prob[e]
                self.prot[e] = None
                if len(self.prot) > (4 * self.N) // 5:
                    k, _ = self.prot.popitem(last=False)
                    self.prob[k] = None
            else:
                self.prot.move_to_end(e)

    def _insert(self, e: int):
        if self.policy == "slru":
            self.prob[e] = None
        else:
            self.lru[e] = None
            if self.policy == "lfu":
                self.freq[e] = 1

    def _remove(self, e: int):
        if self.policy == "slru":
            self.prob.pop(e, None)
            self.prot.pop(e, None)
        else:
            del self.lru[e]
            self.freq.pop(e, None)

    def _victim(self, step: set) -> int:
        if self.policy == "slru":
            for seg in (self.prob, self.prot):
                for e in seg:
                    if e not in step:
                        return e
            raise AssertionError("no victim")
        cands = [e for e in self.lru if e not in step]     # in recency / insertion order
        if self.policy == "lfu":
            return min(cands, key=lambda e: self.freq[e])    # first of the minimum = earliest inserted
        return cands[0]

    # -- run-time moves between the cold set and the pool ------------------------
    def _count_and_move(self, ids: np.ndarray, rec: PrepareRecord):
        mp = self.moves
        tokens = ids.shape[0] if ids.ndim >= 2 else 1
        if tokens > mp.count_tokens:
            return
        n_sel = np.bincount(ids.reshape(-1), minlength=self.E)
        for e in np.nonzero(n_sel)[0]:
            self.counts[e] = np.float32(self.counts[e] + np.float32(n_sel[e]))
        self.counted_steps += 1
        if self.counted_steps % mp.interval:
            return
        self.counts = (self.counts * np.float32(mp.decay)).astype(np.float32)
        cold_ids = np.nonzero(self.cold)[0]
        warm_ids = np.nonzero(~self.cold)[0]
        if cold_ids.size == 0 or warm_ids.size == 0:
            return
        c = int(cold_ids[np.argmax(self.counts[cold_ids])])     # argmax / argmin: first = lowest id
        h = int(warm_ids[np.argmin(self.counts[warm_ids])])
        if not np.float32(self.counts[c] - self.counts[h]) > np.float32(mp.threshold):
            return
        self.cold[c] = False
        self.cold[h] = True
        freed = -1
        if h in self.expert_to_slot:
            freed = self.expert_to_slot.pop(h)
            self._remove(h)
            self.free.append(freed)
        self.stats["moves"] += 1
        rec.move = (c, h, freed)
