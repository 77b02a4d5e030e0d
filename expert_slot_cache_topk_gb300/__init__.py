"""GB300 expert-slot-cache MoE layer: C-ABI library binding and seeded inputs.

``import expert_slot_cache_topk_gb300`` is light; the CUDA library
(``libmoecache.so``) is loaded on first use by :mod:`._abi` and raises if it is
missing -- there is no CPU fallback.
"""
