"""The whole layer on the GPU (router -> prepare -> copies -> grouped expert
MLP) against the float64 oracle, plus the invariants the pages state:
cached output == all-resident == bypass == cold (bitwise, same kernels),
copy modes agree, slots hold their expert's bytes, graph capture replays,
and bad input fails without faulting."""

import numpy as np
import pytest

from expert_slot_cache_topk_gb300 import synth
from expert_slot_cache_topk_gb300._abi import MoeError, MOE_EINVAL, MOE_ENOMEM, MOE_ESTATE, MOE_FWD_RESIDUAL
from oracle import router_topk
from tests.gpu_util import (OracleWeights, assert_close, empty_y, make_cache, oracle_slot_caches,
                            oracle_y, torch_x, x_to_f64, y_to_f64)

pytestmark = pytest.mark.gpu
W = synth.WORKLOADS


def _forward_steps(c, w, layer, xs, lgs, flags=0):
    import torch
    ys = []
    for x, lg in zip(xs, lgs):
        T = lg.shape[0]
        y = empty_y(w, T)
        c.forward(layer, torch_x(w, x), torch.from_numpy(lg).cuda(), T, y, flags)
        ys.append(y)
    torch.cuda.synchronize()
    return ys


@pytest.mark.parametrize("name,L,steps,slots,mode", [
    ("tiny", 1, 64, None, "uva"),
    ("tiny", 1, 64, None, "fused"),
    ("olmoe", 2, 10, None, "uva"),
    ("olmoe", 2, 10, None, "fused"),
    ("int4", 2, 10, 16, "fused"),
    ("int4", 1, 6, 0, "uva"),
    ("int4", 1, 6, 0, "fused"),
])
def test_forward_matches_oracle(name, L, steps, slots, mode):
    w = W[name].with_(layers=L)
    c = make_cache(w, slots=slots, copy_mode=mode)
    wt = OracleWeights(w)
    for l in range(L):
        lgs = synth.routing_logits(w, l, steps)
        xs = synth.hidden_states(w, l, steps)
        ys = _forward_steps(c, w, l, xs, lgs)
        for s in range(steps):
            ref = oracle_y(w, wt, l, xs[s], lgs[s])
            assert_close(y_to_f64(w, ys[s]), ref, f"{name} layer {l} step {s}", f32=w.wdtype == "f32")
    c.check()
    c.close()


def test_forward_batched_bypass_sampled_tokens():
    w = W["batched"].with_(layers=1)
    c = make_cache(w)
    wt = OracleWeights(w)
    lgs = synth.routing_logits(w, 0, 2)
    xs = synth.hidden_states(w, 0, 2)
    ys = _forward_steps(c, w, 0, xs, lgs)
    assert c.stats(0)["bypass_steps"] == 2
    g = np.random.default_rng(0)
    for s in range(2):
        toks = g.choice(w.tokens, 8, replace=False)
        ref = oracle_y(w, wt, 0, xs[s][toks], lgs[s][toks])
        assert_close(y_to_f64(w, ys[s])[toks], ref, f"batched step {s}")
    c.close()


def test_forward_prefill_with_cold_set_sampled_tokens():
    w = W["prefill_cold"].with_(layers=1, prefill_tokens=512)
    c = make_cache(w, max_tokens=512)
    wt = OracleWeights(w)
    lg = synth.prefill_logits(w, 0)
    x = synth.hidden_states(w, 0, 1, tokens=512)[0]
    (y,) = _forward_steps(c, w, 0, [x], [lg])
    st = c.stats(0)
    assert st["bypass_steps"] == 1 and st["misses"] == 0 and st["cold_reads"] > 0
    sm, _, _, nfree = c.get_state(0)
    assert (sm == -1).all() and nfree == w.slots          # prefill leaves the pool untouched
    g = np.random.default_rng(1)
    toks = g.choice(512, 24, replace=False)
    ref = oracle_y(w, wt, 0, x[toks], lg[toks])
    assert_close(y_to_f64(w, y)[toks], ref, "prefill")
    # decode after prefill, cold experts read in place
    lgs = synth.routing_logits(w, 0, 6)
    xs = synth.hidden_states(w, 0, 6)
    ys = _forward_steps(c, w, 0, xs, lgs)
    for s in range(6):
        assert_close(y_to_f64(w, ys[s]), oracle_y(w, wt, 0, xs[s], lgs[s]), f"decode {s}")
    c.close()


@pytest.mark.parametrize("name", ["tiny", "olmoe", "int4"])
def test_cached_resident_bypass_cold_bitwise_equal(name):
    """Same kernel, different homes for the expert bytes -> identical y.

    One-token steps run the staged-weight kernel by default and the
    cooperative kernel with mlp_kernel="plain"; each is bitwise stable across
    pool / scratch / host homes and copy modes, and the two agree within the
    float tolerance (their summation orders differ)."""
    import torch
    w = W[name].with_(layers=1)
    steps = 12
    lgs = synth.routing_logits(w, 0, steps)
    xs = synth.hidden_states(w, 0, steps)
    cold_all = np.ones((1, w.experts), np.uint8)
    groups = {
        "staged": {
            "cached": dict(slots=w.top_k + 2),
            "resident": dict(slots=w.experts),
            "bypass": dict(slots=0),
            "cold": dict(slots=w.top_k, cold=cold_all),
            "memcpy": dict(slots=w.top_k + 2, copy_mode="memcpy"),
            "fused": dict(slots=w.top_k + 2, copy_mode="fused"),
            "fused_bypass": dict(slots=0, copy_mode="fused"),
            "fused_resident": dict(slots=w.experts, copy_mode="fused"),
            "fused_cold": dict(slots=w.top_k, copy_mode="fused", cold=cold_all),
        },
        "plain": {
            "cached": dict(slots=w.top_k + 2, mlp_kernel="plain"),
            "resident": dict(slots=w.experts, mlp_kernel="plain"),
            "bypass": dict(slots=0, mlp_kernel="plain"),
            "cold": dict(slots=w.top_k, mlp_kernel="plain", cold=cold_all),
            "fused": dict(slots=w.top_k + 2, copy_mode="fused", mlp_kernel="plain"),
            "fused_cold": dict(slots=w.top_k, copy_mode="fused", mlp_kernel="plain", cold=cold_all),
        },
    }
    first = {}
    for gname, variants in groups.items():
        outs = {}
        for key, kw in variants.items():
            c = make_cache(w, **kw)
            outs[key] = [y.clone() for y in _forward_steps(c, w, 0, xs, lgs)]
            if key.endswith("cold"):
                assert c.stats(0)["cold_reads"] > 0 and c.stats(0)["misses"] == 0
            c.close()
        for key in variants:
            for s in range(steps):
                assert torch.equal(outs[key][s], outs["cached"][s]), (gname, key, s)
        first[gname] = outs["cached"]
    for s in range(steps):
        assert_close(y_to_f64(w, first["staged"][s]), y_to_f64(w, first["plain"][s]), f"staged vs plain {s}",
                     f32=w.wdtype == "f32")


@pytest.mark.parametrize("mode", ["uva", "fused", "memcpy"])
def test_slots_hold_their_experts_after_churn(mode):
    w = W["int4"].with_(layers=2, hidden=256, inter=128)
    c = make_cache(w, slots=12, copy_mode=mode)
    for l in range(2):
        _forward_steps(c, w, l, synth.hidden_states(w, l, 40), synth.routing_logits(w, l, 40))
        assert c.verify_slots(l) == 0
        st = c.stats(l)
        assert st["evictions"] > 0
    c.close()


def test_load_expert_refreshes_a_resident_slot():
    import torch
    w = W["tiny"]
    c = make_cache(w)
    lgs = synth.routing_logits(w, 0, 3)
    xs = synth.hidden_states(w, 0, 3)
    _forward_steps(c, w, 0, xs[:1], lgs[:1])
    ids, _ = router_topk(lgs[0], w.top_k)
    e = int(ids[0, 0])
    blk = synth.expert_block(w, 0, e).copy()
    blk.view(np.float32)[:] *= 2.0
    c.load_expert(0, e, blk)
    assert c.verify_slots(0) == 0
    (y,) = _forward_steps(c, w, 0, xs[:1], lgs[:1])
    wt = OracleWeights(w)
    from oracle import dequant_expert
    wt.cache[(0, e)] = dequant_expert(blk, w.wdtype, w.hidden, w.inter)
    assert_close(y_to_f64(w, y), oracle_y(w, wt, 0, xs[0], lgs[0]), "after reload", f32=True)
    c.close()


def test_residual_flag_and_expert_mlp_entry_point():
    import torch
    from expert_slot_cache_topk_gb300._abi import expert_mlp
    w = W["olmoe"].with_(layers=1)
    c = make_cache(w)
    lg = synth.routing_logits(w, 0, 1)[0]
    x = synth.hidden_states(w, 0, 1)[0]
    (y,) = _forward_steps(c, w, 0, [x], [lg])
    (yr,) = _forward_steps(c, w, 0, [x], [lg], flags=MOE_FWD_RESIDUAL)
    xt = torch_x(w, x)
    ref = xt.float() + y.float()
    assert ((yr.float() - ref).abs() <= 2e-2 + 1e-2 * ref.abs()).all()
    # standalone grouped MLP on the same pool slots
    ids, wts = router_topk(lg, w.top_k)
    sm, _, _, _ = c.get_state(0)
    pool, _ = c.pool_ptrs(0)
    stride = c.info()["slot_stride"]
    ptrs = torch.tensor([pool + int(sm[e]) * stride for e in ids[0]], dtype=torch.int64, device="cuda")
    wd = torch.tensor(wts.astype(np.float32), device="cuda")
    h = torch.empty((w.top_k, w.inter), dtype=torch.float32, device="cuda")
    y2 = empty_y(w, 1)
    expert_mlp("bf16", w.hidden, w.inter, w.top_k, xt, ptrs, wd, 1, h, y2)
    torch.cuda.synchronize()
    # the standalone entry point runs the cooperative kernel: bitwise equal to a
    # layer step on that kernel, within tolerance of the staged-weight kernel
    assert_close(y_to_f64(w, y2), y_to_f64(w, y), "expert_mlp vs staged forward")
    cp = make_cache(w, mlp_kernel="plain")
    (yp,) = _forward_steps(cp, w, 0, [x], [lg])
    assert torch.equal(y2, yp)          # same kernel, same bytes, same order
    cp.close()
    c.close()


@pytest.mark.parametrize("mode", ["uva", "fused"])
def test_graph_capture_replays_like_eager(mode):
    import torch
    w = W["olmoe"].with_(layers=2, hidden=512, inter=256)
    steps = 6
    lgs = [synth.routing_logits(w, l, steps) for l in range(2)]
    xs = [synth.hidden_states(w, l, steps) for l in range(2)]
    ref = make_cache(w, slots=10)
    ref_y = [[y.clone() for y in _forward_steps(ref, w, l, xs[l], lgs[l])] for l in range(2)]
    c = make_cache(w, slots=10, copy_mode=mode)
    x_st = [torch_x(w, xs[l][0]).clone() for l in range(2)]
    lg_st = [torch.from_numpy(lgs[l][0]).cuda() for l in range(2)]
    y_st = [empty_y(w, 1) for _ in range(2)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for l in range(2):
                c.forward(l, x_st[l], lg_st[l], 1, y_st[l], 0, torch.cuda.current_stream())
    torch.cuda.current_stream().wait_stream(s)
    for st in range(steps):
        for l in range(2):
            x_st[l].copy_(torch_x(w, xs[l][st]))
            lg_st[l].copy_(torch.from_numpy(lgs[l][st]).cuda())
        g.replay()
        torch.cuda.synchronize()
        for l in range(2):
            assert torch.equal(y_st[l], ref_y[l][st]), (st, l)
    for l in range(2):
        assert c.stats(l) == ref.stats(l)
    ref.close()
    c.close()


def test_memcpy_mode_refuses_capture():
    import torch
    w = W["tiny"]
    c = make_cache(w, copy_mode="memcpy")
    x = torch_x(w, synth.hidden_states(w, 0, 1)[0])
    lg = torch.from_numpy(synth.routing_logits(w, 0, 1)[0]).cuda()
    y = empty_y(w, 1)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(Exception):
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                c.forward(0, x, lg, 1, y, 0, torch.cuda.current_stream())
    torch.cuda.synchronize()
    c.close()


def test_model_step_host_matches_layer_chain():
    import torch
    w = W["olmoe"].with_(layers=3, hidden=512, inter=256)
    a = make_cache(w)
    b = make_cache(w)
    x0 = synth.hidden_states(w, 0, 1)[0]
    lg = np.stack([synth.routing_logits(w, l, 1)[0] for l in range(3)])
    y_h = np.zeros_like(x0)
    a.model_step_host(x0, lg, 1, y_h)
    x = torch_x(w, x0)
    for l in range(3):
        y = empty_y(w, 1)
        b.forward(l, x, torch.from_numpy(lg[l]).cuda(), 1, y, MOE_FWD_RESIDUAL)
        x = y
    torch.cuda.synchronize()
    assert (x.view(torch.int16).cpu().numpy() == y_h.view(np.int16)).all()
    a.close()
    b.close()


def test_counters_closed_forms():
    w = W["int4"].with_(layers=1, hidden=256, inter=128)
    c = make_cache(w, slots=16)
    oc = oracle_slot_caches(w, slots=16)[0]
    lgs = synth.routing_logits(w, 0, 30)
    _forward_steps(c, w, 0, synth.hidden_states(w, 0, 30), lgs)
    Be = c.info()["expert_bytes"]
    s = c.stats(0)
    D = 0
    for lg in lgs:
        ids, _ = router_topk(lg, w.top_k)
        oc.prepare(ids)
        D += len(set(ids.reshape(-1).tolist()))
    assert s["hits"] + s["misses"] == D
    assert s["bytes_h2d_miss"] == s["misses"] * Be == oc.stats["bytes_h2d_miss"]
    assert s == oc.stats
    c.close()


def test_errors_do_not_fault():
    import torch
    from expert_slot_cache_topk_gb300._abi import MoECache
    w = W["tiny"]
    with pytest.raises(MoeError) as ei:
        MoECache(1, 8, 2, 64, 128, "f32", 4, 1, hbm_budget_bytes=1000)
    assert ei.value.status == MOE_ENOMEM
    with pytest.raises(MoeError) as ei:
        MoECache(1, 8, 9, 64, 128, "f32", 4, 1)
    assert ei.value.status == MOE_EINVAL
    c = make_cache(w)
    lg = torch.from_numpy(synth.routing_logits(w, 0, 1)[0]).cuda()
    x = torch_x(w, synth.hidden_states(w, 0, 1)[0])
    y = empty_y(w, 2)
    with pytest.raises(MoeError) as ei:
        c.forward(0, x, lg, 2, y)                 # T > max_tokens
    assert ei.value.status == MOE_EINVAL
    with pytest.raises(MoeError):
        c.forward(1, x, lg, 1, y)                 # no such layer
    bad = torch.tensor([[3, 8]], dtype=torch.int32, device="cuda")
    out = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    c.prepare(0, bad, 1, out)
    with pytest.raises(MoeError) as ei:
        c.check()
    assert ei.value.status == MOE_ESTATE
    assert (out.cpu() == -1).all()
    c.reset()
    c.check()
    assert c.stats(0)["steps"] == 0
    c.close()


def test_staged_kernel_falls_back_for_shapes_it_cannot_take():
    """inter not a multiple of 8: the one-token step runs the cooperative kernel."""
    w = W["tiny"].with_(inter=12)
    c = make_cache(w)
    wt = OracleWeights(w)
    lgs = synth.routing_logits(w, 0, 8)
    xs = synth.hidden_states(w, 0, 8)
    ys = _forward_steps(c, w, 0, xs, lgs)
    for s in range(8):
        assert_close(y_to_f64(w, ys[s]), oracle_y(w, wt, 0, xs[s], lgs[s]), f"step {s}", f32=True)
    c.check()
    c.close()


# shapes: the workloads' own, and ones whose rows split into items of 128
# weight rows instead of 256 (hidden 384: 128-row down items; inter 192: 128-row
# up items), and 8 experts with 96 tokens each (two token tiles per expert)
@pytest.mark.parametrize("name,T,slots,over", [
    ("olmoe", 16, None, {}), ("olmoe", 16, 64, {}), ("int4", 24, 64, {}), ("int4", 24, 512, {}), ("int4", 3, 16, {}),
    ("olmoe", 12, None, {"wdtype": "fp8"}),
    ("olmoe", 12, None, {"hidden": 384, "inter": 192}),
    ("olmoe", 12, None, {"hidden": 384, "inter": 192, "wdtype": "fp8"}),
    ("int4", 12, None, {"hidden": 384, "inter": 384}),
    ("olmoe", 96, None, {"experts": 8, "slots": 8}),
    ("int4", 96, None, {"experts": 10, "slots": 10}),
])
def test_multi_token_steps_on_the_tensor_cores(name, T, slots, over):
    """Several tokens per step run the grouped tcgen05 GEMM (assignments
    grouped by expert): every token against the float64 oracle, and the
    per-token kernel (mlp_kernel="plain") within the same tolerance."""
    w = W[name].with_(layers=1, tokens=T, **over)
    steps = 3
    lgs = synth.routing_logits(w, 0, steps)
    xs = synth.hidden_states(w, 0, steps)
    wt = OracleWeights(w)
    c = make_cache(w, slots=slots)
    assert c.info()["gemm_kernel_name"] == "tma"   # weight rows on N, TMA-staged operands
    launches0 = c.info()["kernel_launches"]
    ys = _forward_steps(c, w, 0, xs, lgs)
    per_step = (c.info()["kernel_launches"] - launches0) / steps
    assert per_step >= 6          # prepare, group, gather, up GEMM, down GEMM, combine (+ copies)
    c.check()
    c.close()
    cp = make_cache(w, slots=slots, mlp_kernel="plain")
    yp = _forward_steps(cp, w, 0, xs, lgs)
    cp.close()
    for s in range(steps):
        ref = oracle_y(w, wt, 0, xs[s], lgs[s])
        assert_close(y_to_f64(w, ys[s]), ref, f"{name} T={T} step {s}")
        assert_close(y_to_f64(w, yp[s]), ref, f"{name} T={T} plain step {s}")


@pytest.mark.parametrize("name,T,over", [("olmoe", 16, {}), ("int4", 24, {}), ("olmoe", 12, {"wdtype": "fp8"})])
def test_multi_token_steps_on_the_cp_async_gemm(name, T, over):
    """gemm_kernel="tc" keeps the cp.async grouped GEMM in use (the kernel that
    runs where the driver provides no tensor-map encoder): every token against
    the float64 oracle."""
    w = W[name].with_(layers=1, tokens=T, **over)
    steps = 3
    lgs = synth.routing_logits(w, 0, steps)
    xs = synth.hidden_states(w, 0, steps)
    wt = OracleWeights(w)
    c = make_cache(w, gemm_kernel="tc")
    assert c.info()["gemm_kernel_name"] == "tc"
    ys = _forward_steps(c, w, 0, xs, lgs)
    c.check()
    c.close()
    for s in range(steps):
        assert_close(y_to_f64(w, ys[s]), oracle_y(w, wt, 0, xs[s], lgs[s]), f"{name} T={T} cp.async step {s}")
