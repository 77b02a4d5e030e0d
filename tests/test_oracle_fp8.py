"""Pins for the oracle's FP8 per-tensor expert format (vLLM PR #37190 keeps
"BF16 + FP8 per-tensor" weights and copies their scale buffers into the slot
with the weights): the E4M3 decoder against torch's float8_e4m3fn for every
code and against closed forms of the encoding, the block layout, the
per-tensor scales on hand-built blocks, and planted mistakes."""

import numpy as np
import pytest

import oracle.expert_mlp as M
from oracle.expert_mlp import dequant_expert, e4m3_to_f64, expert_nbytes, swiglu_expert


def test_every_code_matches_torch_float8_e4m3fn():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], mine[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(mine[ok]))


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0x40, 2.0), (0xC0, -2.0), (0x3C, 1.5),
    (0x7E, 448.0),                 # largest finite: exponent 15, mantissa 6
    (0x08, 2.0 ** -6),             # smallest normal
    (0x07, 7 * 2.0 ** -9),         # largest subnormal
    (0x01, 2.0 ** -9),             # smallest subnormal
    (0x77, 240.0), (0x30, 0.5),
])
def test_closed_forms_of_the_encoding(code, value):
    assert e4m3_to_f64(np.array([code], np.uint8))[0] == value


def test_nan_codes_and_negative_zero():
    v = e4m3_to_f64(np.array([0x7F, 0xFF, 0x80], np.uint8))
    assert np.isnan(v[0]) and np.isnan(v[1])
    assert v[2] == 0.0 and np.signbit(v[2])


def test_block_size_and_parts():
    H, I = 2048, 1024
    n = expert_nbytes("fp8", H, I)
    assert (n["w13"], n["w2"], n["s13"], n["s2"]) == (2 * I * H, H * I, 16, 16)
    assert n["total"] == 3 * H * I + 32
    # a quarter of the f32 block and half of the bf16 block, plus the scales
    assert n["total"] - 32 == expert_nbytes("bf16", H, I)["total"] // 2


def _block(H, I, gate_code, up_code, down_code, sg, su, sd):
    w13 = np.concatenate([np.full(I * H, gate_code, np.uint8), np.full(I * H, up_code, np.uint8)])
    w2 = np.full(H * I, down_code, np.uint8)
    s13 = np.zeros(4, np.float32)
    s13[:2] = [sg, su]
    s2 = np.zeros(4, np.float32)
    s2[0] = sd
    return np.concatenate([w13, w2, s13.view(np.uint8), s2.view(np.uint8)])


def test_per_tensor_scales_on_a_hand_built_block():
    H, I = 32, 16
    blk = _block(H, I, 0x38, 0x40, 0xB8, 2.0, 0.25, 3.0)   # codes 1.0, 2.0, -1.0
    w13, w2 = dequant_expert(blk, "fp8", H, I)
    assert np.all(w13[:I] == 2.0) and np.all(w13[I:] == 0.5) and np.all(w2 == -3.0)


def test_expert_output_closed_form():
    # gate row i = a, up row i = b (constant), x = 1: g = a H, u = b H,
    # h = silu(g) u, y[n] = d * sum_i h = d * I * silu(a H) * b H
    H, I = 16, 16
    blk = _block(H, I, 0x30, 0x38, 0x38, 0.125, 1.0, 0.5)  # a = 1/16, b = 1, d = 1/2
    w13, w2 = dequant_expert(blk, "fp8", H, I)
    y = swiglu_expert(np.ones(H), w13, w2)
    g, u = H / 16.0, float(H)
    want = 0.5 * I * (g / (1.0 + np.exp(-g))) * u
    assert np.allclose(y, want, rtol=1e-14)


def test_planted_mistakes_are_caught(monkeypatch):
    H, I = 32, 16
    blk = _block(H, I, 0x38, 0x40, 0xB8, 2.0, 0.25, 3.0)
    # 1) one scale for all of w13 (the gate scale) -> the up rows come out 1.0, not 0.5
    real = M.dequant_fp8
    calls = []

    def first_scale_only(codes, scale, rows, K):
        calls.append(scale)
        return real(codes, calls[0], rows, K)
    monkeypatch.setattr(M, "dequant_fp8", first_scale_only)
    w13, _ = M.dequant_expert(blk, "fp8", H, I)
    assert not np.all(w13[I:] == 0.5)
    monkeypatch.setattr(M, "dequant_fp8", real)
    # 2) exponent bias 8 instead of 7 -> 1.0 decodes as 0.5
    c = np.array([0x38], np.uint8).astype(np.int64)
    wrong = (1.0 + (c & 7) / 8.0) * np.exp2(((c >> 3) & 0xF) - 8.0)
    assert wrong[0] != e4m3_to_f64(np.array([0x38], np.uint8))[0]
    # 3) subnormals read as normals with exponent 0 -> 0x01 decodes as (1 + 1/8) 2^-7
    assert e4m3_to_f64(np.array([0x01], np.uint8))[0] != (1.0 + 1 / 8) * 2.0 ** -7
