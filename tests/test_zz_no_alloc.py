"""moe_expert_mlp_noalloc, the allocation-free grouped expert MLP.

Some callers of this library cannot allocate device memory where they call
it (a plugin inside a framework whose allocator owns all device memory, or a
loop that must not synchronise on cudaMalloc); this entry point keeps its
scratch in an array built into the library.  The tests call it through the
C ABI, several times in a row on different formats, shapes and inputs that
all share the built-in array, and check every output two ways: elementwise
against the float64 oracle at the tolerance of the other parity tests, and bit
for bit against the regular moe_expert_mlp, which takes a caller-provided
scratch buffer.  Buffers for inputs and outputs are made by the test; the
entry point itself allocates nothing.

Kept in a file that pytest collects last, so a run that stops at the first
failure has already run every other test.
"""

import numpy as np
import pytest

from expert_slot_cache_topk_gb300 import synth
from oracle import dequant_expert, moe_combine
from tests.gpu_util import assert_close, x_to_f64

pytestmark = pytest.mark.gpu

N_EXPERTS = 12

# (name, workload, tokens, seed): all four weight formats; the last FP8 shape has
# hidden and inter multiples of 16 but not of 32 (FP8 rows are 16-code chunks)
CASES = [
    ("f32", synth.WORKLOADS["tiny"], 3, 1),
    ("bf16", synth.WORKLOADS["olmoe"], 3, 2),
    ("int4", synth.WORKLOADS["int4"], 5, 3),
    ("fp8", synth.WORKLOADS["olmoe"].with_(wdtype="fp8"), 2, 4),
    ("fp8_h48", synth.WORKLOADS["tiny"].with_(wdtype="fp8", hidden=48, inter=80, top_k=3), 4, 5),
]


def _case(w, T, seed):
    import torch
    g = np.random.default_rng(seed)
    blocks = [synth.expert_block(w, 0, e) for e in range(N_EXPERTS)]
    stride = (blocks[0].nbytes + 255) // 256 * 256
    dev = torch.zeros(N_EXPERTS * stride, dtype=torch.uint8, device="cuda")
    for e, b in enumerate(blocks):
        dev[e * stride: e * stride + b.nbytes] = torch.from_numpy(b).cuda()
    ids = np.stack([g.choice(N_EXPERTS, w.top_k, replace=False) for _ in range(T)])
    wts = g.random((T, w.top_k)).astype(np.float32)
    ptrs = torch.tensor((dev.data_ptr() + ids * stride).reshape(-1), dtype=torch.int64, device="cuda")
    wt = torch.tensor(wts, device="cuda")
    x = synth.hidden_states(w, 0, 1, tokens=T)[0]
    if w.wdtype == "f32":
        xt = torch.from_numpy(x).cuda()
        y = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")
    else:
        xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        y = torch.empty((T, w.hidden), dtype=torch.bfloat16, device="cuda")
    return dict(w=w, T=T, blocks=blocks, dev=dev, ids=ids, wts=wts, ptrs=ptrs, wt=wt, x=x, xt=xt, y=y)


def _with_scratch(c):
    import torch
    from expert_slot_cache_topk_gb300._abi import expert_mlp
    w, T = c["w"], c["T"]
    h = torch.empty((T * w.top_k, w.inter), dtype=torch.float32, device="cuda")
    y = torch.empty_like(c["y"])
    expert_mlp(w.wdtype, w.hidden, w.inter, w.top_k, c["xt"], c["ptrs"], c["wt"], T, h, y)
    return y


def _oracle(c):
    w = c["w"]
    experts = {e: dequant_expert(c["blocks"][e], w.wdtype, w.hidden, w.inter)
               for e in np.unique(c["ids"])}
    return moe_combine(x_to_f64(w, c["x"]), c["ids"], c["wts"], lambda e: experts[e])


def test_noalloc_matches_oracle_and_expert_mlp_on_calls_in_a_row():
    import torch
    from expert_slot_cache_topk_gb300._abi import expert_mlp_noalloc
    cases = [(name, _case(w, T, seed)) for name, w, T, seed in CASES]
    for _, c in cases:          # back-to-back calls, every one sharing the built-in array
        w = c["w"]
        expert_mlp_noalloc(w.wdtype, w.hidden, w.inter, w.top_k, c["xt"], c["ptrs"], c["wt"], c["T"], c["y"])
    torch.cuda.synchronize()
    for name, c in cases:
        w = c["w"]
        got = c["y"].float().cpu().numpy().astype(np.float64)
        assert_close(got, _oracle(c), f"noalloc {name}", f32=(w.wdtype == "f32"))
        ref = _with_scratch(c)
        torch.cuda.synchronize()
        assert torch.equal(c["y"], ref), f"noalloc {name}: not bitwise equal to moe_expert_mlp"


def test_noalloc_second_call_on_same_inputs_is_identical():
    """The array keeps the previous call's contents; a repeat call must not depend on them."""
    import torch
    from expert_slot_cache_topk_gb300._abi import expert_mlp_noalloc
    c = _case(CASES[3][1], 3, 7)
    other = _case(CASES[2][1], 5, 8)
    w, wo = c["w"], other["w"]
    expert_mlp_noalloc(w.wdtype, w.hidden, w.inter, w.top_k, c["xt"], c["ptrs"], c["wt"], c["T"], c["y"])
    first = c["y"].clone()
    expert_mlp_noalloc(wo.wdtype, wo.hidden, wo.inter, wo.top_k, other["xt"], other["ptrs"], other["wt"],
                       other["T"], other["y"])
    expert_mlp_noalloc(w.wdtype, w.hidden, w.inter, w.top_k, c["xt"], c["ptrs"], c["wt"], c["T"], c["y"])
    torch.cuda.synchronize()
    assert torch.equal(first, c["y"])


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    from expert_slot_cache_topk_gb300._abi import (MOE_EINVAL, NOALLOC_MAX_SCRATCH_FLOATS, MoeError,
                                                  expert_mlp_noalloc)
    w = synth.WORKLOADS["olmoe"]
    T = NOALLOC_MAX_SCRATCH_FLOATS // (w.top_k * w.inter) + 1
    x = torch.zeros((T, w.hidden), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    ptrs = torch.zeros(T * w.top_k, dtype=torch.int64, device="cuda")
    wts = torch.zeros(T * w.top_k, dtype=torch.float32, device="cuda")
    with pytest.raises(MoeError) as ei:
        expert_mlp_noalloc(w.wdtype, w.hidden, w.inter, w.top_k, x, ptrs, wts, T, y)
    assert ei.value.status == MOE_EINVAL and "scratch" in str(ei.value)


def test_noalloc_on_a_second_device_after_the_first():
    """Kernel attributes are per device: configuring device 0 must not make device 1 skip its own."""
    import torch
    from expert_slot_cache_topk_gb300._abi import expert_mlp_noalloc
    if torch.cuda.device_count() < 2:
        pytest.skip("one GPU visible")
    outs = []
    for dev in (0, 1):
        with torch.cuda.device(dev):
            c = _case(CASES[1][1], 3, 2)
            w = c["w"]
            expert_mlp_noalloc(w.wdtype, w.hidden, w.inter, w.top_k, c["xt"], c["ptrs"], c["wt"], c["T"],
                               c["y"])
            torch.cuda.synchronize()
            outs.append(c["y"].cpu())
    assert torch.equal(outs[0], outs[1])
