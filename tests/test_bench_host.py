"""Host-side arithmetic of bench.py's measurement figures, on hand-built
records (no GPU): the copy-span bandwidth of missed experts, the least-squares
per-miss fit kept beside it, the copy-stream fallback, and the cache counts."""

import numpy as np
import pytest

import bench
from expert_slot_cache_topk_gb300 import synth

W = synth.WORKLOADS["olmoe"]
BE = synth.expert_layout(W.wdtype, W.hidden, W.inter)["total"]   # 12,582,912 B


def _record(spans, ms, miss, st0=None, st1=None, copy_ms=0.0):
    zero = {"bytes_h2d_miss": 0, "bytes_h2d_bypass": 0}
    return {"spans": np.asarray(spans, dtype=np.uint64).reshape(-1, 3),
            "mlp_ms": np.asarray(ms, dtype=np.float64), "mlp_miss": np.asarray(miss, dtype=np.int64),
            "st0": st0 or zero, "st1": st1 or zero, "tm": {"copy_ms": copy_ms}}


def test_expert_bytes_of_the_olmoe_block():
    assert BE == 3 * 2048 * 1024 * 2 == 12_582_912


def test_copy_span_bandwidth_by_hand():
    # two launches copied 1 and 2 experts over 60 us and 120 us; one launch
    # copied nothing (span fields zero) and must not count
    spans = [[1_000, 61_000, 1], [500_000, 620_000, 2], [0, 0, 0]]
    r = _record(spans, ms=[0.08, 0.14, 0.03], miss=[1, 2, 0],
                st1={"bytes_h2d_miss": 3 * BE, "bytes_h2d_bypass": 0})
    f = bench.h2d_figures(W, r, h2d_peak=210.0)
    want = 3 * BE / 180e-6 / 1e9                       # 3 experts over 180 us
    assert f["copy_launches"] == 2
    assert f["span_bytes"] == 3 * BE
    assert f["miss_gbs"] == pytest.approx(want, rel=1e-12)
    assert f["frac"] == pytest.approx(want / 210.0, rel=1e-12)
    assert f["span_us_per_launch"] == pytest.approx(90.0)
    assert f["miss_bytes"] == 3 * BE


def test_per_miss_fit_recovers_a_line():
    # launch time = 30 us + 55 us per miss, exactly
    miss = np.array([0, 0, 1, 2, 3, 1, 0, 2])
    ms = (30.0 + 55.0 * miss) * 1e-3
    base, per = bench._fit_per_miss(ms, miss)
    assert base == pytest.approx(30e-3, rel=1e-9)
    assert per == pytest.approx(55e-3, rel=1e-9)
    r = _record([[0, 0, 0]] * len(ms), ms, miss)
    f = bench.h2d_figures(W, r, h2d_peak=None)
    assert f["slope"]["per_miss_us"] == pytest.approx(55.0, rel=1e-9)
    assert f["slope"]["gbs"] == pytest.approx(BE / 55e-6 / 1e9, rel=1e-9)
    # no launch copied: no span figure
    assert f["miss_gbs"] is None and f["frac"] is None


def test_fit_needs_two_miss_counts():
    assert bench._fit_per_miss(np.array([0.03, 0.03]), np.array([1, 1])) == (None, None)


def test_copy_stream_fallback_uses_event_time():
    # copies on the copy stream (no copier spans): bytes / copy-stream event time
    r = _record([], ms=[], miss=[], st1={"bytes_h2d_miss": 2 * BE, "bytes_h2d_bypass": BE}, copy_ms=0.2)
    f = bench.h2d_figures(W, r, h2d_peak=200.0)
    want = 3 * BE / 0.2e-3 / 1e9
    assert f["miss_gbs"] == pytest.approx(want, rel=1e-12)
    assert f["frac"] == pytest.approx(want / 200.0, rel=1e-12)
    assert "event time" in f["how"]


def test_cache_counts_and_hit_rate():
    st0 = {"hits": 10, "misses": 5, "evictions": 1, "bypass_steps": 0, "cold_reads": 2}
    st1 = {"hits": 40, "misses": 15, "evictions": 6, "bypass_steps": 3, "cold_reads": 2}
    d = bench.cache_counts({"st0": st0, "st1": st1})
    assert d == {"hits": 30, "misses": 10, "evictions": 5, "bypass_steps": 3, "cold_reads": 0, "hit_rate": 0.75}
