"""Parser for tests/golden/lru_traces.txt (hand-worked slot-pool traces)."""

import os
from dataclasses import dataclass, field

from oracle.slot_cache import SLOT_COLD, SLOT_POOL, SLOT_SCRATCH

HERE = os.path.dirname(os.path.abspath(__file__))


@dataclass
class Step:
    ids: list
    hits: list
    misses: list        # (expert, slot, evicted)
    bypass: bool
    slots: list         # encoded slot ids, one per id


@dataclass
class Trace:
    name: str
    cite: str = ""
    experts: int = 0
    slots: int = 0
    topk: int = 1
    cold: list = field(default_factory=list)
    steps: list = field(default_factory=list)
    totals: dict = field(default_factory=dict)


def _ints(tok: str) -> list:
    tok = tok.strip()
    if tok == "-":
        return []
    return [int(v) for v in tok.replace(",", " ").split()]


def _slot(tok: str) -> int:
    kind, idx = tok[0], int(tok[1:])
    return {"p": SLOT_POOL, "s": SLOT_SCRATCH, "c": SLOT_COLD}[kind] | idx


def load_traces(path: str = None) -> list:
    path = path or os.path.join(HERE, "golden", "lru_traces.txt")
    traces, cur = [], None
    with open(path) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            head, _, rest = line.partition(" ")
            if head == "trace":
                cur = Trace(rest.strip())
            elif head == "cite":
                cur.cite = rest
            elif head == "experts":
                tok = rest.split()
                cur.experts, cur.slots, cur.topk = int(tok[0]), int(tok[2]), int(tok[4])
                cur.cold = _ints(tok[6])
            elif head == "step":
                parts = [p.strip() for p in rest.split("|")]
                ids = _ints(parts[0])
                hits = _ints(parts[1].split(None, 1)[1])
                mtok = parts[2].split(None, 1)[1].strip()
                misses = [] if mtok == "-" else [tuple(int(v) for v in m.split(":")) for m in mtok.split()]
                bypass = bool(int(parts[3].split()[1]))
                slots = [_slot(t) for t in parts[4].split()[1:]]
                cur.steps.append(Step(ids, hits, misses, bypass, slots))
            elif head == "totals":
                tok = rest.split()
                cur.totals = {tok[i]: int(tok[i + 1]) for i in range(0, len(tok), 2)}
            elif head == "end":
                traces.append(cur)
                cur = None
    return traces
