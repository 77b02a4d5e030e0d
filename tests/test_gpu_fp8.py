"""FP8 per-tensor experts (E4M3 weights, gate / up / down float32 scales) on the
GPU against the float64 oracle: one-token steps on the staged kernel in every
copy mode and on the cooperative kernel, multi-token steps on the tensor-core
grouped GEMM, bitwise stability across the homes of the expert bytes, and the
slots after churn."""

import numpy as np
import pytest

from expert_slot_cache_topk_gb300 import synth
from tests.gpu_util import OracleWeights, assert_close, make_cache, oracle_y, y_to_f64
from tests.test_gpu_forward import _forward_steps

pytestmark = pytest.mark.gpu
OLMOE8 = synth.WORKLOADS["olmoe"].with_(layers=1, wdtype="fp8")
TINY8 = synth.WORKLOADS["tiny"].with_(wdtype="fp8")


@pytest.mark.parametrize("w,steps", [(TINY8, 48), (OLMOE8, 10)], ids=["tiny", "olmoe"])
@pytest.mark.parametrize("mode", ["uva", "fused", "memcpy"])
@pytest.mark.parametrize("kernel", ["auto", "plain"])
def test_one_token_steps_match_oracle(w, steps, mode, kernel):
    lgs = synth.routing_logits(w, 0, steps)
    xs = synth.hidden_states(w, 0, steps)
    wt = OracleWeights(w)
    c = make_cache(w, slots=w.top_k + 2, copy_mode=mode, mlp_kernel=kernel)
    ys = _forward_steps(c, w, 0, xs, lgs)
    st = c.stats(0)
    assert st["misses"] > 0 and st["hits"] > 0
    assert c.verify_slots(0) == 0
    c.check()
    c.close()
    for s in range(steps):
        assert_close(y_to_f64(w, ys[s]), oracle_y(w, wt, 0, xs[s], lgs[s]), f"{mode} {kernel} step {s}")


def test_bitwise_equal_across_homes():
    import torch
    w = OLMOE8
    steps = 8
    lgs = synth.routing_logits(w, 0, steps)
    xs = synth.hidden_states(w, 0, steps)
    cold_all = np.ones((1, w.experts), np.uint8)
    variants = {
        "cached": dict(slots=w.top_k + 2),
        "resident": dict(slots=w.experts),
        "bypass": dict(slots=0),
        "cold": dict(slots=w.top_k, cold=cold_all),
        "fused": dict(slots=w.top_k + 2, copy_mode="fused"),
        "fused_bypass": dict(slots=0, copy_mode="fused"),
    }
    outs = {}
    for key, kw in variants.items():
        c = make_cache(w, **kw)
        outs[key] = [y.clone() for y in _forward_steps(c, w, 0, xs, lgs)]
        c.close()
    for key in variants:
        for s in range(steps):
            assert torch.equal(outs[key][s], outs["cached"][s]), (key, s)


@pytest.mark.parametrize("T,slots", [(16, 64), (16, 20), (48, 0)])
def test_multi_token_steps_on_the_tensor_cores(T, slots):
    w = OLMOE8.with_(tokens=T)
    steps = 2
    lgs = synth.routing_logits(w, 0, steps)
    xs = synth.hidden_states(w, 0, steps)
    wt = OracleWeights(w)
    c = make_cache(w, slots=slots)
    l0 = c.info()["kernel_launches"]
    ys = _forward_steps(c, w, 0, xs, lgs)
    assert (c.info()["kernel_launches"] - l0) / steps >= 5   # prepare, group, up, down, combine
    c.check()
    c.close()
    for s in range(steps):
        ref = oracle_y(w, wt, 0, xs[s], lgs[s])
        got = y_to_f64(w, ys[s])
        rows = np.random.default_rng(s).choice(T, 6, replace=False)
        assert_close(got[rows], ref[rows], f"T={T} slots={slots} step {s}")


def test_slots_hold_their_experts_after_churn():
    w = OLMOE8.with_(layers=2, hidden=256, inter=128)
    for mode in ("uva", "fused"):
        c = make_cache(w, slots=12, copy_mode=mode)
        for l in range(2):
            _forward_steps(c, w, l, synth.hidden_states(w, l, 30), synth.routing_logits(w, l, 30))
            assert c.verify_slots(l) == 0 and c.stats(l)["evictions"] > 0
        c.close()
