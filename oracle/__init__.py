"""CPU oracle for the expert-slot-cache MoE forward — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of what the hot path computes,
written from the pages and kept independent of the CUDA path (no shared code,
headers, tables or constants beyond the documented interface encodings).
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import it; the product path never calls it.

Modules
-------
router       softmax over all experts + top-k selected on logits (ties -> lower id)
slot_cache   per-layer OrderedDict LRU slot pool, bypass rule, cold set, remap
expert_mlp   weight formats (f32, bf16, INT4 g128), dequantisation, SwiGLU expert
             MLP with top-k weighted combine, byte counts

Floating point runs in float64 throughout (the pages fix no precision); the
CUDA path is compared against it with the float tolerance the tests state.

Parity pins: every function here is pinned by tests under ``tests/`` marked
``not gpu`` (hand-worked traces in ``tests/golden``, brute force, closed forms,
page byte counts, invariants).  Nothing here is "parity unpinned".
"""

from .router import router_topk, softmax_f64
from .slot_cache import (LayerSlotCache, PrepareRecord, SLOT_KIND_SHIFT, SLOT_POOL,
                         SLOT_SCRATCH, SLOT_COLD, decode_slot_id)
from .expert_mlp import (expert_nbytes, split_block, dequant_expert, bf16_bits_to_f64,
                         swiglu_expert, moe_combine)

__all__ = [
    "router_topk", "softmax_f64", "LayerSlotCache", "PrepareRecord", "SLOT_KIND_SHIFT",
    "SLOT_POOL", "SLOT_SCRATCH", "SLOT_COLD", "decode_slot_id", "expert_nbytes",
    "split_block", "dequant_expert", "bf16_bits_to_f64", "swiglu_expert", "moe_combine",
]
