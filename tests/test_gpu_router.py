"""Router top-k on the GPU vs the oracle: ids bit-exact (ties -> lower id,
NaN last), weights within 2e-5 relative of the float64 softmax."""

import numpy as np
import pytest

from oracle import router_topk

pytestmark = pytest.mark.gpu

W_ATOL, W_RTOL = 1e-7, 2e-5


def _cache(E, k, max_tokens, renorm=False):
    from expert_slot_cache_topk_gb300._abi import MoECache
    return MoECache(1, E, k, 64, 128, "f32", min(4, E), max_tokens, renormalize=renorm)


def _run(c, logits, k):
    import torch
    T, E = logits.shape
    lg = torch.from_numpy(logits).cuda()
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    c.router(lg, T, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("E,k,T", [(8, 2, 1), (8, 8, 5), (64, 8, 1), (64, 8, 65), (512, 10, 1),
                                   (512, 10, 200), (1000, 32, 33), (33, 1, 7), (1024, 10, 3)])
def test_router_ids_exact_weights_close(E, k, T):
    g = np.random.default_rng(E * 7 + k * 3 + T)
    logits = np.round(g.standard_normal((T, E)) * 2, 1).astype(np.float32)   # many exact ties
    c = _cache(E, k, T)
    ids, w = _run(c, logits, k)
    rids, rw = router_topk(logits, k)
    assert (ids == rids).all()
    assert np.all(np.abs(w - rw) <= W_ATOL + W_RTOL * np.abs(rw))
    c.close()


def test_router_renormalize():
    g = np.random.default_rng(1)
    logits = g.standard_normal((40, 64)).astype(np.float32)
    c = _cache(64, 8, 40, renorm=True)
    ids, w = _run(c, logits, 8)
    rids, rw = router_topk(logits, 8, renormalize=True)
    assert (ids == rids).all()
    assert np.all(np.abs(w - rw) <= W_ATOL + W_RTOL * np.abs(rw))
    assert np.allclose(w.sum(1), 1.0, atol=1e-5)
    c.close()


def test_router_all_equal_and_nan():
    E, k = 128, 6
    logits = np.zeros((3, E), np.float32)
    logits[1, [5, 9, 70]] = np.nan
    logits[2, :] = -np.inf
    logits[2, 100] = 1.0
    c = _cache(E, k, 3)
    ids, w = _run(c, logits, k)
    rids, rw = router_topk(logits, k)
    assert (ids == rids).all()
    assert ids[0].tolist() == list(range(k))
    assert np.allclose(w[0], 1.0 / E, rtol=1e-6)
    assert ids[2, 0] == 100 and abs(w[2, 0] - 1.0) < 1e-6 and (w[2, 1:] == 0).all()
    c.close()


def test_router_zero_tokens_is_noop():
    c = _cache(8, 2, 4)
    import torch
    ids = torch.full((1, 2), -7, dtype=torch.int32, device="cuda")
    c.router(torch.zeros((1, 8), device="cuda"), 0, ids, torch.zeros((1, 2), device="cuda"))
    torch.cuda.synchronize()
    assert (ids.cpu() == -7).all()
    c.close()
