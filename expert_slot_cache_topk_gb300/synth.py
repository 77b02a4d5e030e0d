"""Seeded synthetic inputs for the expert-slot-cache workloads.

This module only *generates inputs*: router logits, hidden states, expert
weight blocks in the canonical byte layout, and the cold-set choice.  It holds
none of the method's arithmetic (no top-k, softmax, LRU bookkeeping,
dequantisation or expert MLP), so the CUDA path and the CPU oracle can both
consume what it produces without sharing any computation.

Shapes follow the pages' models:

* OLMoE-1B-7B: 64 experts, 16 cached per layer, bf16
  (vLLM PR #37190, "Run MoE models exceeding VRAM via expert CPU offloading
  with GPU cache", section "Test results").
* Flash-Next INT4 g128: top-10 of 512 experts, w13 [1280, 2560] and
  w2 [2560, 640] with bf16 scales, 2.417 MiB per expert
  ("Running 125B MoE on Two 32 GB Cards", section 1 "What does not fit").
* Cold set = the least-selected 6.0% of experts per layer (same page,
  section 3.1 "How uneven the expert selection is").

Routing is Zipf-skewed; the pages' datasets are not available, and skewed
synthetic routing stands in for them.

Every stream is seeded by ``SeedSequence([1234, cfg_id, stream, ...])``.
"""

from __future__ import annotations

import statistics
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace
from typing import Optional

import numpy as np

MASTER_SEED = 1234

# stream ids inside one config
_S_ZIPF = 1       # per-layer expert permutation of the Zipf table
_S_ROUTE = 2      # decode routing
_S_PREFILL = 3    # prefill routing
_S_X = 4          # hidden states
_S_W = 5          # expert weights (per layer, expert)
_S_TOPIC = 6      # per-topic permutations (batched decode)

WEIGHT_STD = 0.02


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: model shape, cache size, routing recipe."""

    name: str
    cfg_id: int
    layers: int
    experts: int
    top_k: int
    hidden: int
    inter: int
    wdtype: str            # "f32" | "bf16" | "int4g128"
    slots: int             # N, pool slots per layer
    tokens: int            # tokens per decode step
    steps: int             # decode steps in the trace
    routing: str           # "zipf_logit" | "reuse" | "fresh" | "topics"
    zipf_s: float
    reuse_p: float = 0.0
    topics: int = 0
    prefill_tokens: int = 0
    cold_frac: float = 0.0

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def n_cold(self) -> int:
        return int(round(self.cold_frac * self.experts))


WORKLOADS = {
    "tiny": Workload("tiny", 1, layers=1, experts=8, top_k=2, hidden=64, inter=128,
                     wdtype="f32", slots=4, tokens=1, steps=64,
                     routing="zipf_logit", zipf_s=1.1),
    "olmoe": Workload("olmoe", 2, layers=16, experts=64, top_k=8, hidden=2048, inter=1024,
                      wdtype="bf16", slots=16, tokens=1, steps=512,
                      routing="reuse", zipf_s=1.2, reuse_p=0.8),
    "int4": Workload("int4", 3, layers=16, experts=512, top_k=10, hidden=2560, inter=640,
                     wdtype="int4g128", slots=64, tokens=1, steps=512,
                     routing="fresh", zipf_s=1.1),
    "batched": Workload("batched", 4, layers=16, experts=512, top_k=10, hidden=2560,
                        inter=640, wdtype="int4g128", slots=64, tokens=64, steps=512,
                        routing="topics", zipf_s=1.1, topics=4),
    "prefill_cold": Workload("prefill_cold", 5, layers=16, experts=512, top_k=10,
                             hidden=2560, inter=640, wdtype="int4g128", slots=64,
                             tokens=1, steps=512, routing="fresh", zipf_s=1.1,
                             prefill_tokens=2048, cold_frac=0.06),
}


def rng(cfg_id: int, *path: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([MASTER_SEED, cfg_id, *path])))


# --------------------------------------------------------------------------
# canonical expert byte layout (the interface the C header documents)
# --------------------------------------------------------------------------

def expert_layout(wdtype: str, hidden: int, inter: int) -> dict:
    """Byte offsets of one expert block: [w13 | w2 | s13 | s2].

    w13 is [2*inter, hidden] (rows [0, inter) gate, [inter, 2*inter) up),
    w2 is [hidden, inter], both row-major.  INT4: two weights per byte along
    the row, low nibble = even column; s13 [2*inter, hidden/128] and
    s2 [hidden, inter/128] bf16 scales.  FP8: one E4M3 byte per weight;
    s13 = float32 [gate scale, up scale] and s2 = float32 [down scale], each
    zero-padded to 16 bytes.
    """
    H, I = hidden, inter
    if wdtype == "f32":
        w13, w2, s13, s2 = 2 * I * H * 4, H * I * 4, 0, 0
    elif wdtype == "bf16":
        w13, w2, s13, s2 = 2 * I * H * 2, H * I * 2, 0, 0
    elif wdtype == "int4g128":
        if H % 128 or I % 128:
            raise ValueError("int4g128 needs hidden and inter divisible by 128")
        w13, w2 = 2 * I * H // 2, H * I // 2
        s13, s2 = 2 * I * (H // 128) * 2, H * (I // 128) * 2
    elif wdtype == "fp8":
        if H % 16 or I % 16:
            raise ValueError("fp8 needs hidden and inter divisible by 16")
        w13, w2, s13, s2 = 2 * I * H, H * I, 16, 16
    else:
        raise ValueError(wdtype)
    return {"w13": (0, w13), "w2": (w13, w2), "s13": (w13 + w2, s13),
            "s2": (w13 + w2 + s13, s2), "total": w13 + w2 + s13 + s2}


# --------------------------------------------------------------------------
# value tables
# --------------------------------------------------------------------------

def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + r) >> 16).astype(np.uint16)


_NORMAL_Q = None


def _normal_quantiles() -> np.ndarray:
    """65536 standard-normal quantiles at (u + 0.5) / 65536, float32."""
    global _NORMAL_Q
    if _NORMAL_Q is None:
        nd = statistics.NormalDist()
        _NORMAL_Q = np.array([nd.inv_cdf((u + 0.5) / 65536.0) for u in range(65536)],
                             dtype=np.float32)
    return _NORMAL_Q


def _normal_f32(g: np.random.Generator, n: int, std: float) -> np.ndarray:
    """n draws of N(0, std^2), resolved to 1/65536 quantiles, float32."""
    u = g.integers(0, 65536, size=n, dtype=np.uint16)
    return _normal_quantiles()[u] * np.float32(std)


# --------------------------------------------------------------------------
# expert weights
# --------------------------------------------------------------------------

def _quantize_int4_g128(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Symmetric offset-8 INT4 with one bf16 scale per 128 columns (generator only).

    s = bf16(max|w| / 7) per group, q = clip(rint(w / s), -8, 7) + 8, two
    nibbles per byte along the row, low nibble = even column.
    """
    rows, K = w.shape
    g = w.reshape(rows, K // 128, 128)
    amax = np.abs(g).max(axis=2)
    s_bits = _f32_to_bf16_bits(amax / np.float32(7.0))
    s = (s_bits.astype(np.uint32) << 16).view(np.float32)
    safe = np.where(s == 0, np.float32(1.0), s)
    q = np.clip(np.rint(g / safe[:, :, None]), -8, 7).astype(np.int16) + 8
    q = q.reshape(rows, K).astype(np.uint8)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return packed, s_bits


_E4M3_POS = None


def _e4m3_positive_values() -> np.ndarray:
    """Magnitudes of the finite E4M3 codes 0x00..0x7E (increasing with the code)."""
    global _E4M3_POS
    if _E4M3_POS is None:
        v = []
        for code in range(0x7F):
            exp, man = code >> 3, code & 7
            v.append(man * 2.0 ** -9 if exp == 0 else (8 + man) * 2.0 ** (exp - 10))
        _E4M3_POS = np.array(v, dtype=np.float64)
    return _E4M3_POS


def _quantize_fp8(w: np.ndarray) -> tuple[np.ndarray, np.float32]:
    """Per-tensor E4M3 (generator only): s = float32(max|w| / 448), each
    weight w / s rounded to the nearest E4M3 value, ties to the even code."""
    amax = float(np.abs(w).max())
    s = np.float32(amax / 448.0) if amax > 0 else np.float32(1.0)
    x = np.abs(w.astype(np.float64) / float(s)).reshape(-1)
    pos = _e4m3_positive_values()
    hi = np.clip(np.searchsorted(pos, x), 1, len(pos) - 1)
    lo = hi - 1
    dlo, dhi = x - pos[lo], pos[hi] - x
    code = np.where(dhi < dlo, hi, lo)
    code = np.where(dhi == dlo, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(x >= pos[-1], len(pos) - 1, code).astype(np.uint8)
    code |= np.where(w.reshape(-1) < 0, np.uint8(0x80), np.uint8(0))
    return code.reshape(w.shape), s


def expert_block(w: Workload, layer: int, expert: int, out: Optional[np.ndarray] = None) -> np.ndarray:
    """The canonical byte block of one expert (uint8, expert_layout(...)['total'] bytes)."""
    H, I = w.hidden, w.inter
    lay = expert_layout(w.wdtype, H, I)
    if out is None:
        out = np.empty(lay["total"], dtype=np.uint8)
    g = rng(w.cfg_id, _S_W, layer, expert)
    if w.wdtype == "f32":
        o, n = lay["w13"]
        out[o:o + n] = _normal_f32(g, 2 * I * H, WEIGHT_STD).view(np.uint8)
        o, n = lay["w2"]
        out[o:o + n] = _normal_f32(g, H * I, WEIGHT_STD).view(np.uint8)
    elif w.wdtype == "bf16":
        o, n = lay["w13"]
        out[o:o + n] = _f32_to_bf16_bits(_normal_f32(g, 2 * I * H, WEIGHT_STD)).view(np.uint8)
        o, n = lay["w2"]
        out[o:o + n] = _f32_to_bf16_bits(_normal_f32(g, H * I, WEIGHT_STD)).view(np.uint8)
    elif w.wdtype == "fp8":
        w13 = _normal_f32(g, 2 * I * H, WEIGHT_STD).reshape(2 * I, H)
        qg, sg = _quantize_fp8(w13[:I])
        qu, su = _quantize_fp8(w13[I:])
        qd, sd = _quantize_fp8(_normal_f32(g, H * I, WEIGHT_STD).reshape(H, I))
        o, n = lay["w13"]
        out[o:o + n] = np.concatenate([qg.reshape(-1), qu.reshape(-1)])
        o, n = lay["w2"]
        out[o:o + n] = qd.reshape(-1)
        for key, vals in (("s13", [sg, su]), ("s2", [sd])):
            o, n = lay[key]
            pad = np.zeros(n // 4, dtype=np.float32)
            pad[: len(vals)] = vals
            out[o:o + n] = pad.view(np.uint8)
    else:
        q13, s13 = _quantize_int4_g128(_normal_f32(g, 2 * I * H, WEIGHT_STD).reshape(2 * I, H))
        q2, s2 = _quantize_int4_g128(_normal_f32(g, H * I, WEIGHT_STD).reshape(H, I))
        for key, arr in (("w13", q13), ("w2", q2), ("s13", s13), ("s2", s2)):
            o, n = lay[key]
            out[o:o + n] = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
    return out


def fill_layer_blocks(w: Workload, layer: int, dest: np.ndarray, stride: int,
                      threads: int = 0) -> None:
    """Write every expert block of `layer` into dest[e*stride : e*stride + total]."""
    total = expert_layout(w.wdtype, w.hidden, w.inter)["total"]

    def job(e):
        expert_block(w, layer, e, out=dest[e * stride: e * stride + total])

    threads = threads or min(16, max(1, __import__("os").cpu_count() or 1))
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(job, range(w.experts)))


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------

def zipf_probs(w: Workload, layer: int, topic: Optional[int] = None) -> np.ndarray:
    """Per-layer Zipf(s) selection probabilities over a seeded permutation of experts.

    Rank r (1-based) gets weight r^-s; the permutation decides which expert holds
    which rank.  `topic` selects one of the batched-decode topic mixtures.
    """
    g = rng(w.cfg_id, _S_ZIPF, layer) if topic is None else rng(w.cfg_id, _S_TOPIC, layer, topic)
    perm = g.permutation(w.experts)
    ranks = np.arange(1, w.experts + 1, dtype=np.float64)
    pr = ranks ** (-w.zipf_s)
    pr /= pr.sum()
    p = np.empty(w.experts)
    p[perm] = pr
    return p


def cold_mask(w: Workload, layer: int) -> np.ndarray:
    """The round(cold_frac*E) experts with the lowest Zipf probability in this layer."""
    m = np.zeros(w.experts, dtype=np.uint8)
    if w.n_cold:
        p = zipf_probs(w, layer)
        m[np.argsort(p, kind="stable")[: w.n_cold]] = 1
    return m


def _gumbel_draw(g: np.random.Generator, logp: np.ndarray, k: int,
                 exclude: Optional[np.ndarray] = None) -> np.ndarray:
    """k distinct experts drawn without replacement with probabilities exp(logp)
    (Gumbel-top-k); `exclude` marks experts that may not be drawn.  logp is [.., E]."""
    keys = logp + g.gumbel(size=logp.shape)
    if exclude is not None:
        keys = np.where(exclude, -np.inf, keys)
    return np.argsort(-keys, axis=-1, kind="stable")[..., :k]


def _planted_logits(g: np.random.Generator, chosen: np.ndarray, E: int) -> np.ndarray:
    """clip(N(0,1), +-3) background plus 8 on the chosen experts ([T, k] -> [T, E])."""
    T = chosen.shape[0]
    lg = np.clip(g.standard_normal((T, E)), -3.0, 3.0)
    np.put_along_axis(lg, chosen, np.take_along_axis(lg, chosen, axis=1) + 8.0, axis=1)
    return lg.astype(np.float32)


def routing_logits(w: Workload, layer: int, steps: Optional[int] = None) -> np.ndarray:
    """Decode router logits [steps, tokens, E] float32 for one layer."""
    steps = w.steps if steps is None else steps
    E, k, T = w.experts, w.top_k, w.tokens
    g = rng(w.cfg_id, _S_ROUTE, layer)
    out = np.empty((steps, T, E), dtype=np.float32)
    if w.routing == "zipf_logit":
        logp = np.log(zipf_probs(w, layer))
        for s in range(steps):
            out[s] = (g.standard_normal((T, E)) + logp).astype(np.float32)
        return out
    if w.routing == "topics":
        logps = np.stack([np.log(zipf_probs(w, layer, topic=t)) for t in range(w.topics)])
        tok_topic = np.arange(T) % w.topics
        for s in range(steps):
            chosen = _gumbel_draw(g, logps[tok_topic], k)
            out[s] = _planted_logits(g, chosen, E)
        return out
    logp = np.log(zipf_probs(w, layer))
    if w.routing == "fresh":
        for s in range(steps):
            chosen = _gumbel_draw(g, np.broadcast_to(logp, (T, E)), k)
            out[s] = _planted_logits(g, chosen, E)
        return out
    if w.routing == "reuse":
        prev = [None] * T
        for s in range(steps):
            chosen = np.empty((T, k), dtype=np.int64)
            for t in range(T):
                if prev[t] is None:
                    keep = np.empty(0, dtype=np.int64)
                else:
                    keep = prev[t][g.random(k) < w.reuse_p]
                excl = np.zeros(E, dtype=bool)
                excl[keep] = True
                fill = _gumbel_draw(g, logp, k - keep.size, exclude=excl)
                chosen[t] = np.concatenate([keep, fill])
                prev[t] = chosen[t].copy()
            out[s] = _planted_logits(g, chosen, E)
        return out
    raise ValueError(w.routing)


def prefill_logits(w: Workload, layer: int) -> np.ndarray:
    """Prefill router logits [prefill_tokens, E]: independent Zipf draws per token."""
    g = rng(w.cfg_id, _S_PREFILL, layer)
    logp = np.log(zipf_probs(w, layer))
    chosen = _gumbel_draw(g, np.broadcast_to(logp, (w.prefill_tokens, w.experts)), w.top_k)
    return _planted_logits(g, chosen, w.experts)


# --------------------------------------------------------------------------
# hidden states
# --------------------------------------------------------------------------

def hidden_states(w: Workload, layer: int, steps: int, tokens: Optional[int] = None,
                  stream: int = 0) -> np.ndarray:
    """N(0,1) hidden states [steps, tokens, H]: float32 for f32 weights, else bf16 bits (uint16)."""
    T = w.tokens if tokens is None else tokens
    g = rng(w.cfg_id, _S_X, layer, stream)
    x = g.standard_normal((steps, T, w.hidden)).astype(np.float32)
    if w.wdtype == "f32":
        return x
    return _f32_to_bf16_bits(x).reshape(steps, T, w.hidden)
