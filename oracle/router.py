"""Router top-k (oracle).  Test infrastructure: see the package docstring.

What it follows
---------------
* The provider is handed ``topk_ids`` from the router and the fused MoE kernel
  takes the matching top-k weights (vLLM PR #37190 "Run MoE models exceeding
  VRAM via expert CPU offloading with GPU cache", section "How it works").
* On equal logits the lower expert id wins ("Running 125B MoE on Two 32 GB
  Cards", section 4.2 "One table that spans VRAM and host RAM").
* The pages fix no normalisation: weights are the softmax probabilities over
  all E experts of the chosen ones; ``renormalize`` divides them by their sum.

Selection is on the logits themselves, so ids do not depend on how exp() rounds.
NaN logits rank below every number (treated as -inf for selection).
"""

from __future__ import annotations

import numpy as np


def softmax_f64(logits: np.ndarray) -> np.ndarray:
    """Row softmax in float64: exp(l - max) / sum(exp(l - max))."""
    l = np.asarray(logits, dtype=np.float64)
    m = np.max(np.where(np.isnan(l), -np.inf, l), axis=-1, keepdims=True)
    e = np.exp(l - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def router_topk(logits: np.ndarray, k: int, renormalize: bool = False):
    """logits f32 [T, E] -> (ids int32 [T, k], weights float64 [T, k]).

    ids[t] lists the k largest logits in descending order, lower id first on
    equal logits; weights[t, j] = softmax(logits[t])[ids[t, j]], divided by
    their sum when ``renormalize``.
    """
    l = np.asarray(logits, dtype=np.float32)
    T, E = l.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    key = np.where(np.isnan(l), -np.inf, l).astype(np.float64)
    idx = np.broadcast_to(np.arange(E), (T, E))
    # lexsort: last key is primary -> ascending (-logit), then ascending id
    order = np.lexsort((idx, -key), axis=-1)
    ids = order[:, :k].astype(np.int32)
    p = softmax_f64(l)
    w = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    if renormalize:
        w = w / np.sum(w, axis=1, keepdims=True)
    return ids, w
