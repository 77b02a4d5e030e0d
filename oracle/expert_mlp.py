"""Expert weight formats, dequantisation and the SwiGLU expert MLP (oracle).

Test infrastructure: see the package docstring.

What it follows
---------------
* The grouped expert computation is ``fused_experts(w1, w2, topk ids, ...)``:
  gate/up projection w13, SiLU-and-multiply, down projection w2, and the top-k
  weighted combine (vLLM PR #37190 "Run MoE models exceeding VRAM via expert CPU
  offloading with GPU cache", section "How it works").
* INT4 g128 expert: w13 [1280, 2560] + w2 [2560, 640] + BF16 scales, 2.417 MiB
  ("Running 125B MoE on Two 32 GB Cards", section 1 "What does not fit").

Readings where the pages are open
---------------------------------
* w13 rows [0, I) are the gate, rows [I, 2I) the up projection;
  h = silu(gate . x) * (up . x), silu(g) = g * sigmoid(g).
* INT4: two weights per byte along the row, low nibble = even column, value
  (q - 8) * scale with one bf16 scale per 128 consecutive columns and no zero
  point.  This is the reading that reproduces the page's 2.417 MiB exactly.
* y[t] = sum over j (in j order) of w[t, j] * W2_e (h_e), all in float64.
* FP8 per tensor (vLLM PR #37190 supports "BF16 + FP8 per-tensor" weights,
  with scale buffers copied into the slot together with the weights): one
  byte per weight in the OCP E4M3 encoding (sign, 4 exponent bits with bias 7,
  3 mantissa bits; exponent field 0 = subnormal 2^-6 * m / 8; no infinities;
  S.1111.111 = NaN), value = decoded byte * the tensor's float32 scale, with
  three tensors per expert: gate (w13 rows [0, I)), up (rows [I, 2I)) and
  down (w2).  s13 = [gate scale, up scale] and s2 = [down scale], each part
  zero-padded to 16 bytes.

Canonical block layout: [w13 | w2 | s13 | s2], each part row-major.
"""

from __future__ import annotations

import numpy as np


def expert_nbytes(wdtype: str, H: int, I: int) -> dict:
    """Part sizes in bytes of one expert and their total."""
    if wdtype == "f32":
        parts = {"w13": 2 * I * H * 4, "w2": H * I * 4, "s13": 0, "s2": 0}
    elif wdtype == "bf16":
        parts = {"w13": 2 * I * H * 2, "w2": H * I * 2, "s13": 0, "s2": 0}
    elif wdtype == "int4g128":
        parts = {"w13": (2 * I) * (H // 2), "w2": H * (I // 2),
                 "s13": (2 * I) * (H // 128) * 2, "s2": H * (I // 128) * 2}
    elif wdtype == "fp8":
        parts = {"w13": 2 * I * H, "w2": H * I, "s13": 16, "s2": 16}
    else:
        raise ValueError(wdtype)
    parts["total"] = parts["w13"] + parts["w2"] + parts["s13"] + parts["s2"]
    return parts


def split_block(block: np.ndarray, wdtype: str, H: int, I: int) -> dict:
    """Views of the parts of one expert block (uint8 array)."""
    n = expert_nbytes(wdtype, H, I)
    b = np.asarray(block, dtype=np.uint8).reshape(-1)
    out, off = {}, 0
    for key in ("w13", "w2", "s13", "s2"):
        out[key] = b[off: off + n[key]]
        off += n[key]
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def dequant_int4_g128(packed: np.ndarray, scale_bits: np.ndarray, rows: int, K: int) -> np.ndarray:
    """packed uint8 [rows, K/2] + bf16 scales [rows, K/128] -> float64 [rows, K]."""
    p = np.asarray(packed, dtype=np.uint8).reshape(rows, K // 2)
    q = np.empty((rows, K), dtype=np.int64)
    q[:, 0::2] = p & 0x0F          # low nibble -> even column
    q[:, 1::2] = p >> 4            # high nibble -> odd column
    s = bf16_bits_to_f64(np.asarray(scale_bits).reshape(rows, K // 128))
    col_group = np.arange(K) // 128
    return (q - 8).astype(np.float64) * s[:, col_group]


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP E4M3 bytes -> float64, from the format's definition (exact)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    out = sign * mag
    out[(c & 0x7F) == 0x7F] = np.nan
    return out


def dequant_fp8(codes: np.ndarray, scale: float, rows: int, K: int) -> np.ndarray:
    """E4M3 bytes [rows, K] times one per-tensor float32 scale -> float64 [rows, K]."""
    return e4m3_to_f64(np.asarray(codes).reshape(rows, K)) * float(np.float32(scale))


def dequant_expert(block: np.ndarray, wdtype: str, H: int, I: int):
    """One expert block -> (w13 float64 [2I, H], w2 float64 [H, I])."""
    parts = split_block(block, wdtype, H, I)
    if wdtype == "f32":
        w13 = parts["w13"].view(np.float32).astype(np.float64).reshape(2 * I, H)
        w2 = parts["w2"].view(np.float32).astype(np.float64).reshape(H, I)
    elif wdtype == "bf16":
        w13 = bf16_bits_to_f64(parts["w13"].view(np.uint16)).reshape(2 * I, H)
        w2 = bf16_bits_to_f64(parts["w2"].view(np.uint16)).reshape(H, I)
    elif wdtype == "fp8":
        s13 = parts["s13"].view(np.float32)
        s2 = parts["s2"].view(np.float32)
        w13 = np.concatenate([dequant_fp8(parts["w13"][: I * H], s13[0], I, H),
                              dequant_fp8(parts["w13"][I * H:], s13[1], I, H)])
        w2 = dequant_fp8(parts["w2"], s2[0], H, I)
    else:
        w13 = dequant_int4_g128(parts["w13"], parts["s13"].view(np.uint16), 2 * I, H)
        w2 = dequant_int4_g128(parts["w2"], parts["s2"].view(np.uint16), H, I)
    return w13, w2


def _sigmoid(g: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-g))


def swiglu_expert(x: np.ndarray, w13: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """One expert on one token: W2 (silu(Wg x) * (Wu x)); x [H] -> [H], float64."""
    I = w13.shape[0] // 2
    gate = w13[:I] @ x
    up = w13[I:] @ x
    h = gate * _sigmoid(gate) * up
    return w2 @ h


def moe_combine(x: np.ndarray, ids: np.ndarray, weights: np.ndarray, expert_weights) -> np.ndarray:
    """y[t] = sum_j weights[t, j] * expert_{ids[t, j]}(x[t]), summed in j order.

    x float [T, H]; ids [T, k]; weights [T, k]; ``expert_weights(e)`` returns
    the dequantised (w13, w2) of expert e.
    """
    x = np.asarray(x, dtype=np.float64)
    T, H = x.shape
    y = np.zeros((T, H), dtype=np.float64)
    cache = {}
    for t in range(T):
        for j in range(ids.shape[1]):
            e = int(ids[t, j])
            if e not in cache:
                cache[e] = expert_weights(e)
            w13, w2 = cache[e]
            y[t] += float(weights[t, j]) * swiglu_expert(x[t], w13, w2)
    return y
