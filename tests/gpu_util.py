"""Helpers shared by the GPU parity tests: build a library handle for a
workload, fill its pinned backing store from the seeded generator, and run
the CPU oracle on the same inputs."""

from __future__ import annotations

import numpy as np

from expert_slot_cache_topk_gb300 import synth
from expert_slot_cache_topk_gb300._abi import MoECache
from oracle import LayerSlotCache, dequant_expert, expert_nbytes, moe_combine, router_topk

# float tolerance of the spec contract for bf16 / INT4 weights, applied
# elementwise as |gpu - oracle| <= ATOL + RTOL * |oracle|
ATOL, RTOL = 2e-2, 1e-2
# f32 weights (the tiny workload) compute and store in f32: the only error is
# f32 rounding of dot products of length <= 128 and of the exp in silu, far
# below 1e-5 relative; outputs there are ~3e-3, so the bf16 absolute bound
# would not see a wrong answer.
ATOL_F32, RTOL_F32 = 1e-7, 1e-4


def make_cache(w: synth.Workload, copy_mode="uva", slots=None, max_tokens=None, cold=None,
               fill=True, **kw) -> MoECache:
    L = w.layers
    if cold is None and w.cold_frac > 0:
        cold = np.stack([synth.cold_mask(w, l) for l in range(L)])
    c = MoECache(L, w.experts, w.top_k, w.hidden, w.inter, w.wdtype,
                 w.slots if slots is None else slots,
                 w.tokens if max_tokens is None else max_tokens,
                 cold_mask=cold, copy_mode=copy_mode, **kw)
    if fill:
        fill_weights(c, w)
    return c


def fill_weights(c: MoECache, w: synth.Workload):
    stride = c.info()["slot_stride"]
    for l in range(w.layers):
        synth.fill_layer_blocks(w, l, c.backing_view(l).reshape(-1), stride)


class OracleWeights:
    """Dequantised expert weights from the generator, computed on demand."""

    def __init__(self, w: synth.Workload):
        self.w = w
        self.cache = {}

    def __call__(self, layer: int, e: int):
        key = (layer, e)
        if key not in self.cache:
            blk = synth.expert_block(self.w, layer, e)
            self.cache[key] = dequant_expert(blk, self.w.wdtype, self.w.hidden, self.w.inter)
        return self.cache[key]


def x_to_f64(w: synth.Workload, x: np.ndarray) -> np.ndarray:
    if w.wdtype == "f32":
        return x.astype(np.float64)
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def y_to_f64(w: synth.Workload, y) -> np.ndarray:
    """GPU output tensor (f32, or bf16 stored as int16 / bfloat16) -> float64 numpy."""
    import torch
    if w.wdtype == "f32":
        return y.float().cpu().numpy().astype(np.float64)
    return y.to(torch.float32).cpu().numpy().astype(np.float64)


def oracle_y(w: synth.Workload, weights: OracleWeights, layer: int, x: np.ndarray,
             logits: np.ndarray, renorm=False) -> np.ndarray:
    ids, wts = router_topk(logits, w.top_k, renorm)
    return moe_combine(x_to_f64(w, x), ids, wts, lambda e: weights(layer, e))


def assert_close(got: np.ndarray, ref: np.ndarray, what="", f32=False):
    err = np.abs(got - ref)
    bound = (ATOL_F32 + RTOL_F32 * np.abs(ref)) if f32 else (ATOL + RTOL * np.abs(ref))
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance, "
                           f"max err {err.max():.3e}, worst at {np.unravel_index(np.argmax(err - bound), err.shape)}")


def oracle_slot_caches(w: synth.Workload, slots=None, cold=None):
    n = expert_nbytes(w.wdtype, w.hidden, w.inter)["total"]
    out = []
    for l in range(w.layers):
        cm = None
        if cold is not None:
            cm = cold[l]
        elif w.cold_frac > 0:
            cm = synth.cold_mask(w, l)
        out.append(LayerSlotCache(w.experts, w.slots if slots is None else slots, n, cm))
    return out


def torch_x(w: synth.Workload, x: np.ndarray, device="cuda"):
    import torch
    if w.wdtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(device).view(torch.bfloat16)


def empty_y(w: synth.Workload, T: int, device="cuda"):
    import torch
    dt = torch.float32 if w.wdtype == "f32" else torch.bfloat16
    return torch.empty((T, w.hidden), dtype=dt, device=device)
