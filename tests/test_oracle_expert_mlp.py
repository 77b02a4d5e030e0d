"""Pins for the expert-format and expert-MLP oracle: the pages' byte counts,
hand-built INT4 bytes, closed forms, a textbook SwiGLU via torch, a dense
one-hot brute force, and planted mistakes."""

import math

import numpy as np
import pytest

import oracle.expert_mlp as M
from oracle.expert_mlp import (bf16_bits_to_f64, dequant_expert, dequant_int4_g128,
                               expert_nbytes, moe_combine, swiglu_expert)

MiB, GiB = 2 ** 20, 2 ** 30


# ---------------------------------------------------------------------------
# byte counts printed on the pages
# ---------------------------------------------------------------------------

def test_int4_expert_is_2_417_mib():
    """"One expert is 2.417 MiB in INT4 g128 (w13 [1280, 2560] + w2 [2560, 640]
    + BF16 scales)" -- Running 125B MoE on Two 32 GB Cards, section 1."""
    n = expert_nbytes("int4g128", 2560, 640)
    assert n["total"] == 2_534_400
    assert round(n["total"] / MiB, 3) == 2.417
    # a zero-point per group would push it to 2.49 MiB: excluded by the page
    assert round((n["total"] + n["s13"] + n["s2"]) / MiB, 3) != 2.417


def test_routed_experts_58_01_gib():
    """48 layers x 512 routed experts = 58.01 GiB (same page, section 1)."""
    n = expert_nbytes("int4g128", 2560, 640)["total"]
    assert round(48 * 512 * n / GiB, 2) == 58.01


def test_cold_set_3_5_gib_is_1482_experts():
    """3.5 GiB = 1,482 experts = 6.0% of all (same page, section 3.1)."""
    n = expert_nbytes("int4g128", 2560, 640)["total"]
    assert round(1482 * n / GiB, 1) == 3.5
    assert round(100 * 1482 / (48 * 512), 1) == 6.0


def test_per_token_layer_bytes_and_whole_layer():
    """~24 MB per token per layer (top-10) and 1.2 GiB per layer (section 2)."""
    n = expert_nbytes("int4g128", 2560, 640)["total"]
    assert 24 <= 10 * n / MiB < 25
    assert round(512 * n / GiB, 1) == 1.2


def test_bf16_and_f32_sizes():
    assert expert_nbytes("bf16", 2048, 1024)["total"] == 12 * MiB
    assert expert_nbytes("f32", 64, 128)["total"] == 98_304


# ---------------------------------------------------------------------------
# formats
# ---------------------------------------------------------------------------

def test_bf16_known_bit_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x3E80, 0x4049, 0x7F80], dtype=np.uint16)
    vals = bf16_bits_to_f64(bits)
    assert vals[:5].tolist() == [1.0, -2.0, 0.0, -0.0, 0.25]
    assert vals[5] == 3.140625 and math.isinf(vals[6])


def test_int4_nibble_order_hand_bytes():
    """byte 0x21: low nibble 1 -> column 0 = (1-8)*s, high nibble 2 -> column 1."""
    K = 128
    packed = np.full((1, K // 2), 0x88, dtype=np.uint8)     # all zeros after the -8 offset
    packed[0, 0] = 0x21
    packed[0, 5] = 0xF0                                       # col 10 -> -8, col 11 -> +7
    scale = np.array([[0x4000]], dtype=np.uint16)            # 2.0
    w = dequant_int4_g128(packed, scale, 1, K)
    assert w[0, 0] == -14.0 and w[0, 1] == -12.0
    assert w[0, 10] == -16.0 and w[0, 11] == 14.0
    assert np.count_nonzero(w) == 4


def test_int4_scale_group_boundary():
    K = 384
    packed = np.full((2, K // 2), 0x99, dtype=np.uint8)      # every weight q=9 -> +1
    scales = np.array([[0x3F80, 0x4000, 0x4040], [0x3F00, 0x3E80, 0xBF80]], dtype=np.uint16)
    w = dequant_int4_g128(packed, scales, 2, K)
    assert (w[0, :128] == 1.0).all() and (w[0, 128:256] == 2.0).all() and (w[0, 256:] == 3.0).all()
    assert w[1, 127] == 0.5 and w[1, 128] == 0.25 and w[1, 383] == -1.0


def test_int4_exactly_representable_roundtrip():
    """Weights w = s*(q-8) with max |q-8| = 7 in each group survive the
    generator's quantiser and the oracle's dequantiser exactly."""
    from expert_slot_cache_topk_gb300.synth import _quantize_int4_g128
    g = np.random.default_rng(0)
    rows, K = 6, 512
    q = g.integers(-7, 8, size=(rows, K))
    q[:, ::128] = 7                                          # group max |q| = 7
    s = 2.0 ** g.integers(-9, -4, size=(rows, K // 128))
    w = (q * np.repeat(s, 128, axis=1)).astype(np.float32)
    packed, sbits = _quantize_int4_g128(w)
    back = dequant_int4_g128(packed, sbits, rows, K)
    assert (back == w.astype(np.float64)).all()


def test_block_layout_parts_in_order():
    """[w13 | w2 | s13 | s2]: fill each part with a marker and read it back."""
    H, I = 256, 128
    n = expert_nbytes("int4g128", H, I)
    blk = np.zeros(n["total"], np.uint8)
    o = 0
    for key, byte in (("w13", 0x99), ("w2", 0xAA), ("s13", None), ("s2", None)):
        if byte is not None:
            blk[o:o + n[key]] = byte
        else:
            blk[o:o + n[key]] = np.frombuffer(np.full(n[key] // 2, 0x3F80 if key == "s13" else 0x4000,
                                                      np.uint16).tobytes(), np.uint8)
        o += n[key]
    w13, w2 = dequant_expert(blk, "int4g128", H, I)
    assert w13.shape == (2 * I, H) and (w13 == 1.0).all()      # q=9, s=1
    assert w2.shape == (H, I) and (w2 == 4.0).all()           # q=10 -> +2, s=2


# ---------------------------------------------------------------------------
# expert MLP
# ---------------------------------------------------------------------------

def _f32_block(g, H, I):
    return g.standard_normal(3 * I * H).astype(np.float32) * np.float32(0.1)


def test_diagonal_weights_closed_form():
    """Wg = a*Id, Wu = b*Id, W2 = c*Id (H = I): y = c * silu(a x) * (b x) per element."""
    H = I = 16
    a, b, c = 0.7, -1.3, 0.5
    w13 = np.concatenate([a * np.eye(I), b * np.eye(I)])
    w2 = c * np.eye(H)
    x = np.linspace(-3, 3, H)
    y = swiglu_expert(x, w13, w2)
    for i in range(H):
        g = a * x[i]
        assert abs(y[i] - c * (g / (1 + math.exp(-g))) * (b * x[i])) < 1e-14
    # swapping gate and up gives a different answer (pins the row order)
    y_sw = swiglu_expert(x, np.concatenate([b * np.eye(I), a * np.eye(I)]), w2)
    assert np.abs(y - y_sw).max() > 0.1


def test_k1_w1_equals_textbook_swiglu_torch():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(1)
    H, I = 64, 128
    blk = _f32_block(g, H, I)
    w13, w2 = dequant_expert(blk.view(np.uint8), "f32", H, I)
    x = g.standard_normal((3, H))
    y = moe_combine(x, np.zeros((3, 1), np.int32), np.ones((3, 1)), lambda e: (w13, w2))
    tx, t13, t2 = (torch.from_numpy(v) for v in (x, w13, w2))
    ref = (torch.nn.functional.silu(tx @ t13[:I].T) * (tx @ t13[I:].T)) @ t2.T
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_dense_onehot_brute_force():
    """Gather-by-id combine equals a dense sum over all experts with a one-hot weight mask."""
    g = np.random.default_rng(2)
    E, H, I, T, k = 8, 64, 128, 7, 3
    experts = [dequant_expert(_f32_block(g, H, I).view(np.uint8), "f32", H, I) for _ in range(E)]
    x = g.standard_normal((T, H))
    ids = np.stack([g.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = g.random((T, k))
    y = moe_combine(x, ids, w, lambda e: experts[e])
    mask = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            mask[t, ids[t, j]] += w[t, j]
    dense = np.zeros((T, H))
    for e in range(E):
        w13, w2 = experts[e]
        gate, up = x @ w13[:I].T, x @ w13[I:].T
        dense += mask[:, e:e + 1] * ((gate / (1 + np.exp(-gate)) * up) @ w2.T)
    assert np.allclose(y, dense, rtol=1e-12, atol=1e-12)


def test_zero_input_gives_zero_and_linearity_in_weights():
    g = np.random.default_rng(3)
    H, I = 64, 128
    ex = [dequant_expert(_f32_block(g, H, I).view(np.uint8), "f32", H, I) for _ in range(2)]
    ids = np.array([[0, 1]], np.int32)
    assert (moe_combine(np.zeros((1, H)), ids, np.array([[0.3, 0.7]]), lambda e: ex[e]) == 0).all()
    x = g.standard_normal((1, H))
    y = moe_combine(x, ids, np.array([[0.3, 0.7]]), lambda e: ex[e])
    y0 = moe_combine(x, ids[:, :1], np.array([[1.0]]), lambda e: ex[e])
    y1 = moe_combine(x, ids[:, 1:], np.array([[1.0]]), lambda e: ex[e])
    assert np.allclose(y, 0.3 * y0 + 0.7 * y1, rtol=1e-13, atol=1e-13)


def test_planted_mistakes_are_caught(monkeypatch):
    # 1) nibble order swapped (high nibble read as the even column) -> hand-byte pin fails
    def swapped(packed, scale_bits, rows, K):
        p = np.asarray(packed, dtype=np.uint8)
        return dequant_int4_g128(((p >> 4) | (p << 4)).astype(np.uint8), scale_bits, rows, K)
    packed = np.full((1, 64), 0x88, np.uint8)
    packed[0, 0] = 0x21
    w = swapped(packed, np.array([[0x4000]], np.uint16), 1, 128)
    assert w[0, 0] != -14.0

    # 2) silu dropped (plain gate*up) -> diagonal closed form fails
    monkeypatch.setattr(M, "_sigmoid", lambda g: np.ones_like(g))
    H = I = 4
    y = M.swiglu_expert(np.ones(H), np.concatenate([np.eye(I), np.eye(I)]), np.eye(H))
    assert abs(y[0] - 1.0 / (1 + math.exp(-1.0))) > 0.1
