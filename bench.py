"""Decode benchmark of the MoE layer through the GPU expert-slot cache.

One step = one decode token through every MoE layer of the OLMoE-shaped
workload (16 layers x 64 experts, top-8, H 2048, I 1024, bf16 weights, 16
pool slots per layer): router top-k, slot bookkeeping + remap, host->device
copies of missed experts, grouped expert MLP, residual add -- all in
libmoecache.so kernels.  Inputs (routing logits and hidden states of every
step) are resident in HBM before the timed region; every step reads 1.61 GB of
expert weights, far more than the 129 MB L2, so no flush is needed.

The same line carries the other workloads of the path, each measured the
same way (warm-up steps, then the timed steps replayed from an uploaded CUDA
graph from the warmed state):
  int4_decode     Flash-Next-shaped INT4 g128 decode (16 layers x 512 experts,
                  top-10) at pool sizes N = 0, 16, 32, 64, plus every expert
                  resident (the staged kernel's roofline without misses)
  batched_decode  64 sequences per step on the INT4 shapes, N = 64 (most steps
                  bypass the pool), and every expert resident (the grouped
                  tensor-core GEMM alone)
  prefill         a 2048-token prefill chunk (bypass) with the cold set read in
                  place, then batch-1 decode on the same cache

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line.  Under torchrun each rank runs an independent replica
on its own GPU (the path has no exchange step); value = all tokens / the
slowest rank's time.
"""

from __future__ import annotations

import argparse
import contextlib
import json
import os
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from expert_slot_cache_topk_gb300 import synth  # noqa: E402

METRIC = "MoE decode tok/s with slot cache; miss H2D GB/s and GEMM HBM GB/s vs roof"
UNIT = "tok/s"
DATA = "synthetic (seeded Zipf routing with reuse; N(0,0.02) weights)"


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def aggregate(seconds: float, units: float, world: int, device=None):
    """(max seconds over ranks, sum of units over ranks); identity at world 1."""
    if world <= 1:
        return seconds, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int, interval_ms: int = 500):
        self.gpu, self.proc, self.lines, self.interval_ms = gpu, None, [], interval_ms

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms), "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads, peaks, the profiled-traffic table
# ---------------------------------------------------------------------------

# arithmetic of the decode path per weight format
DTYPE_NAME = {"bf16": "bf16", "f32": "f32", "fp8": "fp8_e4m3 weights, bf16 activations",
              "int4g128": "int4_g128 weights, bf16 activations"}


def workload_desc(w) -> str:
    return (f"{w.name}-shaped decode: {w.layers} MoE layers x {w.experts} experts, top-{w.top_k}, "
            f"hidden {w.hidden}, expert inter {w.inter}, {w.wdtype} weights, {w.slots} slots/layer, "
            f"batch {w.tokens}, routing {w.routing} Zipf({w.zipf_s})"
            + (f" with p={w.reuse_p} reuse" if w.reuse_p else ""))


def run_config(w, world: int) -> dict:
    """The `config` of the JSON line: the workload only, identical in both arms."""
    lay = synth.expert_layout(w.wdtype, w.hidden, w.inter)
    return {"workload": workload_desc(w), "tokens_per_step": w.tokens,
            "l2": "inputs larger than L2: every step reads "
                  f"{w.layers * w.top_k * w.tokens * lay['total'] / 1e9:.2f} GB of expert weights",
            "parallelism": f"replicas x{world}"}


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# DRAM bytes (read + write) per launch of a staged-kernel launch without
# misses, from ncu captures of the source whose tag is the key (null once the
# kernel source differs from the profiled one).
MEASURED_TRAFFIC = {
    ("olmoe", "k_mlp_ring.cu:428978610526e72b"): 101_972_608,
}


def kernel_source_tag() -> str:
    """Hash of the staged kernel's code and the shared header it includes.

    Line comments and blank lines are left out, so that a change of wording
    in a comment keeps the tag of the measured traffic."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in ("k_mlp_ring.cu", "mlp_common.cuh"):
        with open(os.path.join(ROOT, "expert_slot_cache_topk_gb300", "csrc", name), encoding="utf-8") as f:
            code = re.sub(r"//[^\n]*", "", f.read())
        h.update("\n".join(ln.rstrip() for ln in code.splitlines() if ln.strip()).encode())
    return "k_mlp_ring.cu:" + h.hexdigest()[:16]


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline / reference arm) -- the one place bench runs it
# ---------------------------------------------------------------------------

class OracleSample:
    """The CPU oracle (router top-k, OrderedDict slot pool, float64 dequant +
    expert MLP, residual add) on a bounded sample of the decode workload:
    `tokens` decode tokens through every layer, one (token, layer) step per
    call.  Input generation happens here, outside any timed region."""

    def __init__(self, w, tokens: int = 2):
        from oracle import LayerSlotCache, expert_nbytes, router_topk
        self.w = w
        self.tokens = tokens
        Be = expert_nbytes(w.wdtype, w.hidden, w.inter)["total"]
        self.caches = [LayerSlotCache(w.experts, w.slots, Be) for _ in range(w.layers)]
        self.lgs = [synth.routing_logits(w, l, tokens) for l in range(w.layers)]
        x0 = synth.hidden_states(w, 0, tokens)
        self.x0 = (x0.astype(np.float64) if w.wdtype == "f32"
                   else (x0.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
        self.blocks = {}
        for l in range(w.layers):
            for s in range(tokens):
                for e in np.unique(router_topk(self.lgs[l][s], w.top_k)[0]):
                    if (l, int(e)) not in self.blocks:
                        self.blocks[(l, int(e))] = synth.expert_block(w, l, int(e))
        self.i = 0
        self.x = None

    def layer_step(self) -> float:
        """Run the next (token, layer) step; returns its seconds."""
        from oracle import dequant_expert, moe_combine, router_topk
        w = self.w
        n = self.tokens * w.layers
        s, l = divmod(self.i % n, w.layers)
        if l == 0:
            self.x = self.x0[s].copy()
        t0 = time.perf_counter()
        ids, wts = router_topk(self.lgs[l][s], w.top_k)
        self.caches[l].prepare(ids)
        self.x = self.x + moe_combine(
            self.x, ids, wts, lambda e: dequant_expert(self.blocks[(l, e)], w.wdtype, w.hidden, w.inter))
        dt = time.perf_counter() - t0
        self.i += 1
        return dt


def oracle_tokens_per_s(w, tokens: int = 2, budget_s: float = 20.0):
    """Oracle decode throughput on a bounded sample: (tok/s, layer steps, seconds)."""
    o = OracleSample(w, tokens)
    o.layer_step()                      # first call pays numpy/BLAS start-up; not counted
    o.i = 0
    o.caches = [type(cc)(cc.E, cc.N, cc.B, cc.cold) for cc in o.caches]
    done, spent = 0, 0.0
    while done < tokens * w.layers and spent < budget_s:
        spent += o.layer_step()
        done += 1
    return (done / w.layers) * w.tokens / spent, done, spent


def oracle_integer_trace(w, layers=None) -> dict:
    """The oracle's integer path alone (router top-k + the slot pool) over the
    workload's full decode trace: every step of `layers` (default: all).
    Logit generation is outside the timed part."""
    from oracle import LayerSlotCache, expert_nbytes, router_topk
    Be = expert_nbytes(w.wdtype, w.hidden, w.inter)["total"]
    ls = list(range(w.layers if layers is None else min(layers, w.layers)))
    spent = 0.0
    for l in ls:
        lg = synth.routing_logits(w, l, w.steps)
        cm = synth.cold_mask(w, l) if w.cold_frac > 0 else None
        c = LayerSlotCache(w.experts, w.slots, Be, cm)
        t0 = time.perf_counter()
        for s in range(w.steps):
            ids, _ = router_topk(lg[s], w.top_k)
            c.prepare(ids)
        spent += time.perf_counter() - t0
    n = len(ls) * w.steps
    return {"workload": w.name, "slots": w.slots, "steps": w.steps, "layers": len(ls),
            "layer_steps": n, "seconds": spent, "layer_steps_per_s": n / spent,
            "tokens_per_s": n / w.layers * w.tokens / spent}


def oracle_child(workload: str, budget: float):
    """Single-core oracle timing, run in a child process whose BLAS threads are
    pinned to 1 by the environment the parent sets before numpy loads."""
    try:
        os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
    except (AttributeError, OSError):
        pass
    w = synth.WORKLOADS[workload]
    v, n, dt = oracle_tokens_per_s(w, 2, budget_s=budget)
    print(json.dumps({"value": v, "layer_steps": n, "seconds": dt, "cores": cpu_cores()}), flush=True)


def oracle_single_core(workload: str, budget: float):
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", workload,
                            "--cpu-budget", str(budget)], env=env, capture_output=True, text=True,
                           timeout=budget * 6 + 120)
        for ln in r.stdout.splitlines():
            if ln.startswith("{"):
                return json.loads(ln)
    except (OSError, subprocess.TimeoutExpired):
        pass
    return None


def cpu_baseline(w, budget: float) -> dict:
    """The oracle as it stands on the host cores: the float path on a bounded
    sample with all cores (BLAS threads as installed) and on one core, and the
    integer path (router + slot pool) over the full 512-step traces."""
    v, n, dt = oracle_tokens_per_s(w, 2, budget_s=budget)
    one = oracle_single_core(w.name, budget)
    traces = [oracle_integer_trace(synth.WORKLOADS[name]) for name in ("tiny", "olmoe", "int4", "prefill_cold")]
    traces.append(oracle_integer_trace(synth.WORKLOADS["batched"], layers=2))
    return {"value": v, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{n} (token, layer) steps of the first 2 decode tokens in {dt:.1f} s "
                      f"(float64 numpy, BLAS threads as installed)",
            "single_core": (dict(one, unit=UNIT, cores=1,
                                 sample=f"{one['layer_steps']} (token, layer) steps in {one['seconds']:.1f} s, "
                                        "one core, BLAS threads 1") if one else None),
            "integer_trace": traces}


def run_reference(args, w):
    rank, _, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        if rank != 0:
            dist.barrier()
            return
    o = OracleSample(w, tokens=2)
    for _ in range(args.warmup):
        o.layer_step()
    total_s = sum(o.layer_step() for _ in range(args.steps))
    tokens = args.steps / w.layers * w.tokens
    value = tokens / total_s
    sample = (f"each step = one (token, layer) step of the decode workload, cycling over 2 tokens "
              f"x {w.layers} layers; value = (steps / {w.layers}) tokens / time")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": DATA, "config": run_config(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# weights
# ---------------------------------------------------------------------------

class Int4Weights:
    """The INT4 g128 expert blocks of the Flash-Next-shaped workload, generated
    once and copied into every INT4 handle of the run (the INT4 decode sweep,
    batched decode and the prefill chunk share these shapes; their routing is
    each workload's own)."""

    def __init__(self):
        self.w = synth.WORKLOADS["int4"]
        lay = synth.expert_layout(self.w.wdtype, self.w.hidden, self.w.inter)
        self.stride = (lay["total"] + 255) // 256 * 256
        self.layers = {}
        self.gen_s = 0.0

    def layer(self, l: int) -> np.ndarray:
        if l not in self.layers:
            t0 = time.time()
            buf = np.empty((self.w.experts, self.stride), np.uint8)
            synth.fill_layer_blocks(self.w, l, buf.reshape(-1), self.stride)
            self.layers[l] = buf
            self.gen_s += time.time() - t0
        return self.layers[l]

    def fill(self, c, layers: int):
        assert c.info()["slot_stride"] == self.stride

        def one(l):
            np.copyto(c.backing_view(l), self.layer(l))

        for l in range(layers):
            self.layer(l)
        with ThreadPoolExecutor(8) as ex:
            list(ex.map(one, range(layers)))


def fill_weights(c, w, int4src=None):
    if int4src is not None and (w.wdtype, w.experts, w.hidden, w.inter) == ("int4g128", 512, 2560, 640):
        int4src.fill(c, w.layers)
        return
    stride = c.info()["slot_stride"]
    for l in range(w.layers):
        synth.fill_layer_blocks(w, l, c.backing_view(l).reshape(-1), stride)


# ---------------------------------------------------------------------------
# one decode workload through the library, graph-replayed
# ---------------------------------------------------------------------------

def _fit_per_miss(ms: np.ndarray, misses: np.ndarray):
    """Least-squares fit ms = base + per_miss * misses over the timed MLP launches."""
    if len(ms) < 2 or misses.max() == misses.min():
        return None, None
    A = np.stack([np.ones(len(ms)), misses.astype(np.float64)], 1)
    base, per = np.linalg.lstsq(A, ms.astype(np.float64), rcond=None)[0]
    return float(base), float(per)


class DecodeRun:
    """Steps of one workload on one handle: inputs resident in HBM, each step
    writes its own output buffers, so the timed steps replay from one graph."""

    def __init__(self, c, w, dev, warmup: int, steps: int, graph: bool = True):
        import torch
        from expert_slot_cache_topk_gb300._abi import MOE_FWD_RESIDUAL
        self.c, self.w, self.dev = c, w, dev
        self.warmup, self.steps = warmup, steps
        S = warmup + steps
        self.lg = np.stack([synth.routing_logits(w, l, S) for l in range(w.layers)], axis=1)   # [S, L, T, E]
        self.x0 = synth.hidden_states(w, 0, S)                                                 # [S, T, H]
        self.lg_d = torch.from_numpy(self.lg).to(dev)
        if w.wdtype == "f32":
            self.x0_d = torch.from_numpy(self.x0).to(dev)
            ydt = torch.float32
        else:
            self.x0_d = torch.from_numpy(self.x0.view(np.int16)).to(dev).view(torch.bfloat16)
            ydt = torch.bfloat16
        self.ys = torch.empty((S, w.layers, w.tokens, w.hidden), dtype=ydt, device=dev)
        self.stream = torch.cuda.Stream(dev)
        self.flag = MOE_FWD_RESIDUAL
        # MEMCPY mode takes a host decision per layer step, so it cannot be captured
        self.use_graph = graph and c.info()["copy_mode_name"] != "memcpy"

    def step(self, s):
        x = self.x0_d[s]
        for l in range(self.w.layers):
            self.c.forward(l, x, self.lg_d[s, l], self.w.tokens, self.ys[s, l], self.flag, self.stream)
            x = self.ys[s, l]

    def warm(self):
        import torch
        self.c.reset()
        with torch.cuda.stream(self.stream):
            for s in range(self.warmup):
                self.step(s)
        self.stream.synchronize()

    def prime(self, timing: bool):
        """Empty the pools, run the warm-up steps, then capture (or not) the
        timed steps; returns (graph or None, kernel launches of the timed
        steps).  The uninstrumented graph is replayed once untimed (its first
        launch uploads it to the device), then the pools are emptied and warmed
        up again, so that the timed replay starts from the state the capture
        saw."""
        import torch
        self.warm()
        self.c.set_timing(timing, capacity=self.steps * self.w.layers + 64)
        l0 = self.c.info()["kernel_launches"]
        g = None
        if self.use_graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                with torch.cuda.graph(g, stream=self.stream):
                    for s in range(self.warmup, self.warmup + self.steps):
                        self.step(s)
            self.stream.synchronize()
            n = self.c.info()["kernel_launches"] - l0
            if not timing:
                with torch.cuda.stream(self.stream):
                    g.replay()
                self.stream.synchronize()
                self.warm()
            return g, n
        return g, 0

    def timed(self, g, world, sampler_ms=0, local_rank=0):
        """Run the timed steps once; (seconds, kernel launches, clock summary)."""
        import torch
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0 = self.c.info()["kernel_launches"]
        clk = ClockSampler(local_rank, sampler_ms)
        with (clk if sampler_ms > 0 else contextlib.nullcontext()):
            barrier(world)
            torch.cuda.synchronize(self.dev)
            with torch.cuda.stream(self.stream):
                ev0.record(self.stream)
                if g is not None:
                    g.replay()
                else:
                    for s in range(self.warmup, self.warmup + self.steps):
                        self.step(s)
                ev1.record(self.stream)
            torch.cuda.synchronize(self.dev)
            barrier(world)
        return (ev0.elapsed_time(ev1) / 1e3, self.c.info()["kernel_launches"] - l0,
                clk.summary() if sampler_ms > 0 else None)

    def measure(self, world, sampler_ms=0, local_rank=0) -> dict:
        """The uninstrumented timed replay (throughput, counters), then the same
        steps from the same state with per-launch events (kernel roofline,
        copy spans, phase split)."""
        g, launches = self.prime(False)
        st0 = self.c.stats(-1)
        sec, eager_launches, clocks = self.timed(g, world, sampler_ms, local_rank)
        st1 = self.c.stats(-1)
        del g
        gt, _ = self.prime(True)
        self.timed(gt, world)
        del gt
        tm = self.c.read_timing()
        mlp_ms, mlp_miss = self.c.read_timing_launches()
        spans = self.c.read_copy_spans()
        self.c.set_timing(False)
        return {"sec": sec, "launches": launches if self.use_graph else eager_launches, "clocks": clocks,
                "st0": st0, "st1": st1, "tm": tm, "mlp_ms": mlp_ms, "mlp_miss": mlp_miss, "spans": spans}


def kernel_roofline(w, r: dict, pk: dict) -> dict:
    """HBM roofline of the expert-MLP kernel over the launches that copied
    nothing (no miss, no bypass): every byte of the k experts' blocks is read
    from HBM once per launch."""
    lay = synth.expert_layout(w.wdtype, w.hidden, w.inter)
    bytes_hbm = w.tokens * w.top_k * lay["total"]
    ms, miss = r["mlp_ms"], r["mlp_miss"]
    sp = r["spans"]
    copied = sp[:, 2] if len(sp) == len(ms) else np.zeros(len(ms), np.uint64)   # bypass steps copy with 0 misses
    hit_ms = ms[(miss == 0) & (copied == 0) & (ms > 0)]
    hit_us = float(hit_ms.mean() * 1e3) if len(hit_ms) else None
    achieved = bytes_hbm / (hit_us * 1e-6) / 1e9 if hit_us else None
    return {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": (achieved / pk["hbm_gbs"]) if achieved else None, "peak_source": pk["source"],
            "bytes_per_launch": bytes_hbm, "avg_launch_us": hit_us, "launches": int(len(hit_ms))}


def h2d_figures(w, r: dict, h2d_peak) -> dict:
    """Host-link figures of the missed (or bypassed) expert copies.  Primary:
    bytes / copy span, where the span runs from the first chunk the staged
    kernel's copier warps issued to the last one landed, per launch (FUSED copy
    mode).  Secondary: the slope of MLP-launch time against its miss count."""
    lay = synth.expert_layout(w.wdtype, w.hidden, w.inter)
    Be = lay["total"]
    sp = r["spans"]
    ok = (sp[:, 2] > 0) & (sp[:, 1] > sp[:, 0]) if len(sp) else np.zeros(0, bool)
    span_s = float((sp[ok, 1] - sp[ok, 0]).astype(np.float64).sum()) * 1e-9 if ok.any() else 0.0
    span_bytes = float(sp[ok, 2].astype(np.float64).sum()) * Be if ok.any() else 0.0
    gbs = span_bytes / span_s / 1e9 if span_s > 0 else None
    ms, miss = r["mlp_ms"], r["mlp_miss"]
    base_ms, per_miss_ms = _fit_per_miss(ms[ms > 0], miss[ms > 0]) if len(ms) else (None, None)
    slope_gbs = Be / (per_miss_ms * 1e-3) / 1e9 if per_miss_ms and per_miss_ms > 0 else None
    st0, st1 = r["st0"], r["st1"]
    out = {"miss_gbs": gbs, "peak_gbs": h2d_peak,
           "frac": (gbs / h2d_peak) if (gbs and h2d_peak) else None,
           "how": "bytes copied / copy span (first chunk issued to last chunk landed) of the staged kernel's "
                  "copier warps, summed over the timed launches that copied",
           "copy_launches": int(ok.sum()), "span_bytes": span_bytes,
           "span_us_per_launch": (span_s * 1e6 / ok.sum()) if ok.any() else None,
           "miss_bytes": int(st1["bytes_h2d_miss"] - st0["bytes_h2d_miss"] + st1["bytes_h2d_bypass"]
                             - st0["bytes_h2d_bypass"]),
           "slope": {"per_miss_us": per_miss_ms * 1e3 if per_miss_ms else None,
                     "mlp_base_us": base_ms * 1e3 if base_ms is not None else None,
                     "gbs": slope_gbs,
                     "how": "marginal MLP-launch time per miss (least squares); overlap makes it exceed the link"}}
    if gbs is None and r["tm"]["copy_ms"] > 0:
        # copy kernel or cudaMemcpyAsync on the copy stream: event time of the copies
        out["miss_gbs"] = out["miss_bytes"] / (r["tm"]["copy_ms"] * 1e-3) / 1e9
        out["frac"] = out["miss_gbs"] / h2d_peak if h2d_peak else None
        out["how"] = "bytes copied / event time of the copy-stream launches"
    return out


def cache_counts(r: dict) -> dict:
    st0, st1 = r["st0"], r["st1"]
    d = {k: int(st1[k] - st0[k]) for k in ("hits", "misses", "evictions", "bypass_steps", "cold_reads")}
    d["hit_rate"] = d["hits"] / max(1, d["hits"] + d["misses"])
    return d


# ---------------------------------------------------------------------------
# the INT4 pool-size sweep and batched decode
# ---------------------------------------------------------------------------

def int4_decode(args, dev, world, src, pk) -> dict:
    """Flash-Next-shaped INT4 decode (batch 1, 16 layers) at N = 0, 16, 32, 64
    slots per layer, and with every expert resident (N = E)."""
    from expert_slot_cache_topk_gb300._abi import MoECache
    base = synth.WORKLOADS["int4"]
    if args.layers:
        base = base.with_(layers=args.layers)
    points = []
    for N in (0, 16, 32, 64, base.experts):
        w = base.with_(slots=N)
        c = MoECache(w.layers, w.experts, w.top_k, w.hidden, w.inter, w.wdtype, w.slots, w.tokens,
                     copy_mode="auto", device=dev.index)
        fill_weights(c, w, src)
        info = c.info()
        run = DecodeRun(c, w, dev, warmup=args.int4_warmup, steps=args.int4_steps)
        r = run.measure(world)
        c.close()
        max_sec, toks = aggregate(r["sec"], run.steps * w.tokens, world, dev)
        cc = cache_counts(r)
        p = {"slots": N, "value": toks / max_sec, "unit": UNIT, "ms_per_token": 1e3 * max_sec / run.steps,
             "hit_rate": cc["hit_rate"], "misses_per_token": cc["misses"] / run.steps,
             "bypass_steps_per_token": cc["bypass_steps"] / run.steps, "copy_mode": info["copy_mode_name"],
             "roofline": kernel_roofline(w, r, pk),
             "h2d": h2d_figures(w, r, max(info["memcpy_gbs"], info["uva_gbs"]) or None)}
        points.append(p)
    return {"workload": (f"int4-shaped decode: {base.layers} MoE layers x {base.experts} experts, top-{base.top_k}, "
                         f"hidden {base.hidden}, expert inter {base.inter}, int4 g128 (bf16 scales), batch 1, "
                         f"routing fresh Zipf({base.zipf_s})"),
            "warmup_steps": args.int4_warmup, "steps": args.int4_steps,
            "kernel": "k_mlp_ring (staged-weight expert MLP; copier warps move missed experts)",
            "points": points}


def batched_decode(args, dev, world, src, pk) -> dict:
    """64 sequences per step on the INT4 shapes: N = 64 (steps whose distinct
    experts exceed the pool bypass it) and every expert resident (the grouped
    tensor-core GEMM with no copy in flight)."""
    from expert_slot_cache_topk_gb300._abi import MoECache
    base = synth.WORKLOADS["batched"]
    if args.layers:
        base = base.with_(layers=args.layers)
    out = {"workload": (f"batched decode: {base.layers} MoE layers x {base.experts} experts, top-{base.top_k}, "
                        f"hidden {base.hidden}, expert inter {base.inter}, int4 g128, {base.tokens} sequences per "
                        f"step from {base.topics} Zipf({base.zipf_s}) topic mixtures"),
           "warmup_steps": args.batched_warmup, "steps": args.batched_steps, "points": []}
    for N in (base.slots, base.experts):
        w = base.with_(slots=N)
        c = MoECache(w.layers, w.experts, w.top_k, w.hidden, w.inter, w.wdtype, w.slots, w.tokens,
                     copy_mode="auto", device=dev.index)
        fill_weights(c, w, src)
        run = DecodeRun(c, w, dev, warmup=args.batched_warmup, steps=args.batched_steps)
        r = run.measure(world)
        c.close()
        max_sec, toks = aggregate(r["sec"], run.steps * w.tokens, world, dev)
        cc = cache_counts(r)
        tm = r["tm"]
        flops = run.steps * w.layers * w.tokens * w.top_k * 2 * 3 * w.hidden * w.inter
        gemm_s = tm["up_ms"] / 1e3
        tflops = flops / gemm_s / 1e12 if gemm_s > 0 else None
        copied = r["st1"]["bytes_h2d_miss"] - r["st0"]["bytes_h2d_miss"] + \
            r["st1"]["bytes_h2d_bypass"] - r["st0"]["bytes_h2d_bypass"]
        out["points"].append({
            "slots": N, "value": toks / max_sec, "unit": UNIT, "ms_per_step": 1e3 * max_sec / run.steps,
            "bypass_fraction": cc["bypass_steps"] / (run.steps * w.layers), "hit_rate": cc["hit_rate"],
            "grouped_gemm": {"kernel": "k_moe_gemm_tma (tcgen05, weight rows on N: group + gather + up + down + combine)", "bound": "tensor",
                             "achieved": tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": (tflops / pk["bf16_tflops"]) if tflops else None,
                             "ms_per_layer": 1e3 * gemm_s / (run.steps * w.layers),
                             "note": "event time of the GEMM launches; with copies in flight it includes "
                                     "waits for experts still crossing the host link"},
            "copy": {"bytes_per_step": copied / run.steps,
                     "gbs": copied / (tm["copy_ms"] * 1e-3) / 1e9 if tm["copy_ms"] > 0 else None}})
    return out


def gemm_bf16_resident(args, dev, world, pk, layers: int = 4, tokens: int = 256) -> dict:
    """The grouped GEMM on bf16 weights: OLMoE-shaped steps of 256 tokens with
    every expert resident (no copies), so each layer step reads the distinct
    experts' weight rows from HBM once per token tile."""
    from expert_slot_cache_topk_gb300._abi import MoECache
    w = synth.WORKLOADS["olmoe"].with_(layers=layers, tokens=tokens, slots=synth.WORKLOADS["olmoe"].experts)
    c = MoECache(w.layers, w.experts, w.top_k, w.hidden, w.inter, w.wdtype, w.slots, w.tokens,
                 copy_mode="auto", device=dev.index)
    fill_weights(c, w)
    run = DecodeRun(c, w, dev, warmup=args.batched_warmup, steps=args.batched_steps)
    r = run.measure(world)
    c.close()
    max_sec, toks = aggregate(r["sec"], run.steps * w.tokens, world, dev)
    tm = r["tm"]
    gemm_s = tm["up_ms"] / 1e3
    # weight bytes: the distinct experts of every timed layer step
    lg = run.lg[run.warmup:]                                       # [steps, L, T, E]
    top = np.argpartition(-lg, w.top_k - 1, axis=-1)[..., :w.top_k]
    distinct = sum(len(np.unique(top[s, l])) for s in range(lg.shape[0]) for l in range(lg.shape[1]))
    wbytes = distinct * synth.expert_layout(w.wdtype, w.hidden, w.inter)["total"]
    flops = run.steps * w.layers * w.tokens * w.top_k * 2 * 3 * w.hidden * w.inter
    gbs = wbytes / gemm_s / 1e9 if gemm_s > 0 else None
    return {"workload": (f"bf16 grouped GEMM: {w.layers} MoE layers x {w.experts} experts (all resident), "
                         f"top-{w.top_k}, hidden {w.hidden}, expert inter {w.inter}, {w.tokens} tokens per step"),
            "warmup_steps": run.warmup, "steps": run.steps, "value": toks / max_sec, "unit": UNIT,
            "ms_per_layer": 1e3 * gemm_s / (run.steps * w.layers),
            "distinct_experts_per_layer_step": distinct / (run.steps * w.layers),
            "roofline": {"kernel": "k_moe_gemm_tma (group + gather + up + down + combine)", "bound": "hbm",
                         "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"] if gbs else None,
                         "bytes": "distinct experts' weight rows per layer step, read once"},
            "tflops": flops / gemm_s / 1e12 if gemm_s > 0 else None}


# ---------------------------------------------------------------------------
# prefill chunk (bypass + cold set), then decode on the same cache
# ---------------------------------------------------------------------------

def _prefill_chunks(c, w, dev, reps: int, warm_chunks: int, world):
    import torch
    from expert_slot_cache_topk_gb300._abi import MOE_FWD_RESIDUAL
    T = w.prefill_tokens
    lg = torch.from_numpy(np.stack([synth.prefill_logits(w, l) for l in range(w.layers)])).to(dev)   # [L, T, E]
    x0 = torch.from_numpy(synth.hidden_states(w, 0, 1, tokens=T)[0].view(np.int16)).to(dev).view(torch.bfloat16)
    ys = torch.empty((w.layers, T, w.hidden), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)

    def chunk():
        x = x0
        for l in range(w.layers):
            c.forward(l, x, lg[l], T, ys[l], MOE_FWD_RESIDUAL, stream)
            x = ys[l]

    with torch.cuda.stream(stream):
        for _ in range(warm_chunks):
            chunk()
    stream.synchronize()
    st0 = c.stats(-1)
    c.set_timing(True, capacity=4 * w.layers * reps + 8)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            chunk()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    sec = ev0.elapsed_time(ev1) / 1e3
    tm = c.read_timing()
    c.set_timing(False)
    st1 = c.stats(-1)
    return sec, tm, st0, st1, stream


def run_prefill(args, dev, world, src, pk):
    """Prefill chunk of the prefill + cold-set workload: all layers of one
    2048-token chunk through moe_forward (the bypass path: every non-cold
    expert of the chunk is copied to scratch, cold experts are read in place,
    the grouped expert MLP runs on the tensor cores)."""
    from expert_slot_cache_topk_gb300._abi import MoECache
    w = synth.WORKLOADS["prefill_cold"]
    if args.layers:
        w = w.with_(layers=args.layers)
    if args.prefill_slots >= 0:
        w = w.with_(slots=args.prefill_slots)
    T = w.prefill_tokens
    cold = np.stack([synth.cold_mask(w, l) for l in range(w.layers)])
    c = MoECache(w.layers, w.experts, w.top_k, w.hidden, w.inter, w.wdtype, w.slots, T,
                 cold_mask=cold, copy_mode="auto", device=dev.index)
    fill_weights(c, w, src)
    reps = 2
    sec, tm, st0, st1, stream = _prefill_chunks(c, w, dev, reps, 1, world)
    dec = decode_after_prefill(c, w, dev, stream, world)
    c.close()
    max_sec, all_tok = aggregate(sec, reps * T, world, dev)
    flops = reps * w.layers * T * w.top_k * 2 * 3 * w.hidden * w.inter
    gemm_s = tm["up_ms"] / 1e3
    copy_s = tm["copy_ms"] / 1e3
    byp = st1["bytes_h2d_bypass"] - st0["bytes_h2d_bypass"]
    tflops = flops / gemm_s / 1e12 if gemm_s > 0 else None
    return {
        "workload": (f"prefill chunk: {w.layers} MoE layers x {w.experts} experts, top-{w.top_k}, hidden {w.hidden}, "
                     f"expert inter {w.inter}, int4 g128, {T} tokens, {w.slots} slots/layer"
                     f"{' (bypass)' if w.slots < w.experts - w.n_cold else ' (all non-cold resident)'}, "
                     f"{w.n_cold} cold experts/layer read in place"),
        "value": all_tok / max_sec, "unit": "tok/s", "ms_per_chunk": 1e3 * max_sec / reps, "chunks": reps,
        "grouped_gemm": {"kernel": "k_moe_gemm_tma (tcgen05, weight rows on N: group + gather + up + down + combine)",
                         "bound": "tensor", "achieved": tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": (tflops / pk["bf16_tflops"]) if tflops else None,
                         "flops_per_chunk": flops // reps, "ms_per_chunk": 1e3 * gemm_s / reps,
                         "note": "event time of the GEMM launches, which overlap the bypass copy and wait for "
                                 "experts still crossing the host link"},
        "bypass_copy": {"bytes_per_chunk": byp // reps, "ms_per_chunk": 1e3 * copy_s / reps,
                        "gbs": byp / copy_s / 1e9 if copy_s > 0 else None},
        "cold_reads_per_chunk": (st1["cold_reads"] - st0["cold_reads"]) // reps,
        "decode_after_prefill": dec,
        "grouped_gemm_resident": gemm_resident(args, dev, world, src, pk),
    }


def gemm_resident(args, dev, world, src, pk, layers=4):
    """The grouped GEMM alone: a prefill chunk on a few layers whose pools hold
    every non-cold expert (N = E - cold), after a first chunk has filled them,
    so no copy is in flight while the tensor cores run."""
    from expert_slot_cache_topk_gb300._abi import MoECache
    w = synth.WORKLOADS["prefill_cold"]
    w = w.with_(layers=min(layers, args.layers or layers), slots=w.experts - w.n_cold)
    T = w.prefill_tokens
    cold = np.stack([synth.cold_mask(w, l) for l in range(w.layers)])
    c = MoECache(w.layers, w.experts, w.top_k, w.hidden, w.inter, w.wdtype, w.slots, T,
                 cold_mask=cold, copy_mode="auto", device=dev.index)
    fill_weights(c, w, src)
    reps = 2
    sec, tm, st0, st1, _ = _prefill_chunks(c, w, dev, reps, 2, world)
    c.close()
    flops = reps * w.layers * T * w.top_k * 2 * 3 * w.hidden * w.inter
    gemm_s = tm["up_ms"] / 1e3
    tflops = flops / gemm_s / 1e12 if gemm_s > 0 else None
    max_sec, all_tok = aggregate(sec, reps * T, world, dev)
    return {"layers": w.layers, "slots": w.slots, "value": all_tok / max_sec, "unit": "tok/s",
            "misses": st1["misses"] - st0["misses"], "bound": "tensor", "achieved": tflops,
            "peak": pk["bf16_tflops"], "unit_gemm": "TFLOP/s",
            "frac": (tflops / pk["bf16_tflops"]) if tflops else None,
            "ms_per_layer_gemm": 1e3 * gemm_s / (reps * w.layers)}


def decode_after_prefill(c, w, dev, stream, world, warmup=32, steps=128):
    """Decode steps of the same workload on the same cache after its prefill
    chunks (batch 1, N slots, the cold set read in place): warm-up steps, then
    the timed steps replayed from an uploaded graph from the warmed state."""
    import torch
    from expert_slot_cache_topk_gb300._abi import MOE_FWD_RESIDUAL
    S = warmup + steps
    lg = torch.from_numpy(np.stack([synth.routing_logits(w.with_(tokens=1), l, S) for l in range(w.layers)], 1)).to(dev)
    x0 = torch.from_numpy(synth.hidden_states(w, 0, S, tokens=1).view(np.int16)).to(dev).view(torch.bfloat16)
    ys = torch.empty((S, w.layers, 1, w.hidden), dtype=torch.bfloat16, device=dev)

    def step(s):
        x = x0[s]
        for l in range(w.layers):
            c.forward(l, x, lg[s, l], 1, ys[s, l], MOE_FWD_RESIDUAL, stream)
            x = ys[s, l]

    with torch.cuda.stream(stream):
        for s in range(warmup):
            step(s)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for s in range(warmup, S):
                step(s)
    stream.synchronize()
    st_w = c.stats(-1)
    with torch.cuda.stream(stream):
        g.replay()                     # uploads the graph; the state moves on by `steps`
    stream.synchronize()
    st0 = c.stats(-1)
    # replaying from the state after the first replay: the same steps again,
    # the pool as those steps left it (the routing is stationary)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        g.replay()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    sec = ev0.elapsed_time(ev1) / 1e3
    st1 = c.stats(-1)
    del g
    max_sec, all_tok = aggregate(sec, steps, world, dev)
    hits, misses = st1["hits"] - st0["hits"], st1["misses"] - st0["misses"]
    return {"value": all_tok / max_sec, "unit": "tok/s", "steps": steps, "warmup_steps": warmup,
            "copy_mode": c.info()["copy_mode_name"],
            "misses_per_token": misses / steps, "cold_reads_per_token": (st1["cold_reads"] - st0["cold_reads"]) / steps,
            "hit_rate": hits / max(1, hits + misses), "warm_misses": st0["misses"] - st_w["misses"]}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, w):
    import torch
    from expert_slot_cache_topk_gb300 import _build
    from expert_slot_cache_topk_gb300._abi import MoECache

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    pk = peaks()

    c = MoECache(w.layers, w.experts, w.top_k, w.hidden, w.inter, w.wdtype, w.slots, w.tokens,
                 copy_mode=args.copy_mode, device=local_rank, table=args.table)
    info = c.info()
    t0 = time.time()
    fill_weights(c, w)
    fill_s = time.time() - t0
    run = DecodeRun(c, w, dev, warmup=args.warmup, steps=args.steps, graph=not args.no_graph)
    r = run.measure(world, args.clock_ms, local_rank)

    # cold start: every step from an empty pool (warm-up steps included),
    # replayed from a graph uploaded by one untimed replay
    cold_sec = None
    if run.use_graph:
        S = args.warmup + args.steps
        c.reset()
        gc = torch.cuda.CUDAGraph()
        with torch.cuda.stream(run.stream):
            with torch.cuda.graph(gc, stream=run.stream):
                for s in range(S):
                    run.step(s)
            gc.replay()
        run.stream.synchronize()
        c.reset()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(run.stream):
            e0.record(run.stream)
            gc.replay()
            e1.record(run.stream)
        torch.cuda.synchronize(dev)
        cold_sec = e0.elapsed_time(e1) / 1e3
        del gc

    tokens = args.steps * w.tokens
    max_sec, all_tokens = aggregate(r["sec"], tokens, world, dev)
    roof = kernel_roofline(w, r, pk)
    roof["kernel"] = "k_mlp_ring (staged-weight expert MLP: w13 + SiLU-mul + w2, launches with no miss)"
    roof["traffic"] = MEASURED_TRAFFIC.get((w.name, kernel_source_tag()))
    h2d_peak = max(info["memcpy_gbs"], info["uva_gbs"]) or None
    h2d = h2d_figures(w, r, h2d_peak)
    ms, miss = r["mlp_ms"], r["mlp_miss"]
    h2d["mlp_us_by_misses"] = {str(m): float(ms[(miss == m) & (ms > 0)].mean() * 1e3)
                               for m in range(4) if ((miss == m) & (ms > 0)).any()}

    # end-to-end through the C ABI with host buffers (copies inside the timed
    # region): the same warm-up, then the first timed steps
    e2e_steps = min(args.e2e_steps, args.steps)
    x_h = torch.from_numpy(run.x0.view(np.int16).copy()).pin_memory().numpy()
    lg_h = torch.from_numpy(np.ascontiguousarray(run.lg)).pin_memory().numpy()
    y_h = torch.empty((w.tokens, w.hidden), dtype=torch.int16).pin_memory().numpy()
    c.reset()
    for s in range(args.warmup):
        c.model_step_host(x_h[s], lg_h[s], w.tokens, y_h, 60000, run.stream)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for s in range(args.warmup, args.warmup + e2e_steps):
        c.model_step_host(x_h[s], lg_h[s], w.tokens, y_h, 60000, run.stream)
    e2e_s = time.perf_counter() - t0
    e2e_sec, e2e_tok = aggregate(e2e_s, e2e_steps * w.tokens, world, dev)
    c.close()
    del run

    line = {
        "metric": METRIC, "value": all_tokens / max_sec, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * max_sec / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[w.wdtype],
        "data": DATA, "config": run_config(w, world),
        "engine": {"copy_mode": info["copy_mode_name"], "graph": not args.no_graph, "table": args.table},
        "roofline": roof,
        "h2d": h2d,
        "phases_ms_per_step": {k[:-3]: r["tm"][k] / args.steps for k in ("route_ms", "copy_ms", "up_ms", "down_ms")},
        "cache": cache_counts(r),
        "cold_start": ({"value": (args.warmup + args.steps) * w.tokens / cold_sec, "unit": UNIT,
                        "steps": args.warmup + args.steps,
                        "note": "all steps from an empty pool, warm-up steps included"} if cold_sec else None),
        "e2e": {"value": (e2e_tok / e2e_sec) if e2e_steps > 0 else None, "unit": UNIT,
                "h2d_bytes_per_step": int(x_h[0].nbytes + lg_h[0].nbytes),
                "d2h_bytes_per_step": int(y_h.nbytes)},
        "gpu_launches": int(r["launches"]),
        "clocks": r["clocks"],
        "setup_s": {"fill_weights": fill_s},
    }
    # the other workloads of the path (INT4 weights generated once, shared)
    src = Int4Weights()
    if not args.no_int4:
        line["int4_decode"] = int4_decode(args, dev, world, src, pk)
    if not args.no_batched:
        line["batched_decode"] = batched_decode(args, dev, world, src, pk)
        line["gemm_bf16_resident"] = gemm_bf16_resident(args, dev, world, pk)
    if not args.no_prefill:
        line["prefill"] = run_prefill(args, dev, world, src, pk)
    line["setup_s"]["int4_weights"] = src.gen_s
    if (line.get("int4_decode") or line.get("batched_decode") or line.get("prefill")) and src.layers:
        line["setup_s"]["int4_note"] = ("the INT4 workloads (sweep, batched, prefill) share the int4 workload's "
                                        "generated expert weights; routing is each workload's own")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=480)
    ap.add_argument("--warmup", type=int, default=32)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="olmoe", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--copy-mode", default="auto", choices=["auto", "uva", "memcpy", "fused"])
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling case)")
    ap.add_argument("--slots", type=int, default=-1, help="override the pool slots per layer (N)")
    ap.add_argument("--table", default="split", choices=["split", "vmm"],
                    help="pool + backing store as two allocations, or one VMM table per layer")
    ap.add_argument("--wdtype", default="", choices=["", "f32", "bf16", "int4g128", "fp8"],
                    help="override the decode workload's weight format")
    ap.add_argument("--clock-ms", type=int, default=100, help="nvidia-smi sampling interval in ms")
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--int4-steps", type=int, default=128, help="timed steps per INT4 pool size")
    ap.add_argument("--int4-warmup", type=int, default=32)
    ap.add_argument("--batched-steps", type=int, default=16, help="timed 64-token steps of batched decode")
    ap.add_argument("--batched-warmup", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the timed steps eagerly")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill-chunk measurement")
    ap.add_argument("--no-int4", action="store_true", help="skip the INT4 pool-size sweep")
    ap.add_argument("--no-batched", action="store_true", help="skip batched decode")
    ap.add_argument("--prefill-slots", type=int, default=-1, help="pool slots per layer for the prefill chunk")
    ap.add_argument("--oracle-child", default="", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_child:
        oracle_child(args.oracle_child, args.cpu_budget)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = synth.WORKLOADS[args.workload]
    if args.layers:
        w = w.with_(layers=args.layers)
    if args.slots >= 0:
        w = w.with_(slots=args.slots)
    if args.wdtype:
        w = w.with_(wdtype=args.wdtype)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
