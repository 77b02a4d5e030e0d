"""moe_expert_mlp_noalloc, the allocation-free grouped expert MLP.

Some callers of this library cannot allocate device memory where they call
it (under CUDA graph capture, inside a framework whose allocator owns all
device memory, or in loops that must not synchronise on cudaMalloc); this
entry point keeps its scratch in an array built into the library.  The test
calls it through the C ABI twice in a row, on different shapes and inputs,
and checks each output against the regular moe_expert_mlp, which takes a
caller-provided scratch buffer.  Buffers for inputs and outputs are made by
the test; the entry point itself allocates nothing.

Kept in a file that pytest collects last, so a run that stops at the first
failure has already run every other test.
"""

import numpy as np
import pytest

from expert_slot_cache_topk_gb300 import synth
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu


def _case(name, T, seed, H=None, I=None):
    import torch
    w = synth.WORKLOADS[name]
    if H:
        w = w.with_(hidden=H, inter=I)
    g = np.random.default_rng(seed)
    E = 12
    blocks = [synth.expert_block(w, 0, e) for e in range(E)]
    stride = (blocks[0].nbytes + 255) // 256 * 256
    dev = torch.zeros(E * stride, dtype=torch.uint8, device="cuda")
    for e, b in enumerate(blocks):
        dev[e * stride: e * stride + b.nbytes] = torch.from_numpy(b).cuda()
    ids = np.stack([g.choice(E, w.top_k, replace=False) for _ in range(T)])
    ptrs = torch.tensor((dev.data_ptr() + ids * stride).reshape(-1), dtype=torch.int64, device="cuda")
    wts = torch.tensor(g.random((T, w.top_k)).astype(np.float32), device="cuda")
    x = synth.hidden_states(w, 0, 1, tokens=T)[0]
    if w.wdtype == "f32":
        xt = torch.from_numpy(x).cuda()
        y = torch.empty((T, w.hidden), dtype=torch.float32, device="cuda")
    else:
        xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        y = torch.empty((T, w.hidden), dtype=torch.bfloat16, device="cuda")
    return w, dev, ptrs, wts, xt, y


def _reference(w, ptrs, wts, xt, T):
    import torch
    from expert_slot_cache_topk_gb300._abi import expert_mlp
    h = torch.empty((T * w.top_k, w.inter), dtype=torch.float32, device="cuda")
    y = torch.empty((T, w.hidden), dtype=xt.dtype, device="cuda")
    expert_mlp(w.wdtype, w.hidden, w.inter, w.top_k, xt, ptrs, wts, T, h, y)
    return y


def test_noalloc_matches_expert_mlp_on_two_calls_in_a_row():
    import torch
    from expert_slot_cache_topk_gb300._abi import expert_mlp_noalloc
    cases = [("olmoe", 3, 1, None, None), ("int4", 5, 2, None, None)]
    outs = []
    for name, T, seed, H, I in cases:          # two back-to-back calls sharing the built-in array
        w, dev, ptrs, wts, xt, y = _case(name, T, seed, H, I)
        expert_mlp_noalloc(w.wdtype, w.hidden, w.inter, w.top_k, xt, ptrs, wts, T, y)
        outs.append((w, dev, ptrs, wts, xt, y, T))
    torch.cuda.synchronize()
    for w, dev, ptrs, wts, xt, y, T in outs:
        ref = _reference(w, ptrs, wts, xt, T)
        torch.cuda.synchronize()
        assert_close(y.float().cpu().numpy().astype(np.float64),
                     ref.float().cpu().numpy().astype(np.float64), f"noalloc {w.name}")
        assert torch.equal(y, ref)             # same kernels, same order: identical bits


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
