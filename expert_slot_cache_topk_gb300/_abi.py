"""ctypes binding of libmoecache.so (include/moe_cache.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  Device buffers may be passed as torch tensors (their
``data_ptr()``), numpy arrays (host buffers), or raw integer addresses.
Loading fails loudly when the library has not been built -- there is no CPU
fallback.
"""

from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoecache.so")

MOE_F32, MOE_BF16, MOE_INT4_G128, MOE_FP8_E4M3 = 0, 1, 2, 3
WDTYPE = {"f32": MOE_F32, "bf16": MOE_BF16, "int4g128": MOE_INT4_G128, "fp8": MOE_FP8_E4M3}
MOE_COPY_AUTO, MOE_COPY_MEMCPY, MOE_COPY_UVA, MOE_COPY_FUSED = 0, 1, 2, 3
COPY_MODE = {"auto": MOE_COPY_AUTO, "memcpy": MOE_COPY_MEMCPY, "uva": MOE_COPY_UVA,
             "fused": MOE_COPY_FUSED}
COPY_MODE_NAME = {v: k for k, v in COPY_MODE.items()}
MOE_MLP_AUTO, MOE_MLP_PLAIN = 0, 1
MLP_KERNEL = {"auto": MOE_MLP_AUTO, "plain": MOE_MLP_PLAIN}
MOE_EVICT_LRU, MOE_EVICT_LFU, MOE_EVICT_FIFO, MOE_EVICT_SLRU = 0, 1, 2, 3
EVICT_POLICY = {"lru": MOE_EVICT_LRU, "lfu": MOE_EVICT_LFU, "fifo": MOE_EVICT_FIFO, "slru": MOE_EVICT_SLRU}
MOE_TABLE_SPLIT, MOE_TABLE_VMM = 0, 1
TABLE_LAYOUT = {"split": MOE_TABLE_SPLIT, "vmm": MOE_TABLE_VMM}
MOE_OK, MOE_EINVAL, MOE_ENOMEM, MOE_ECUDA, MOE_ETIMEOUT, MOE_ESTATE = 0, -1, -2, -3, -4, -5
STATUS_NAME = {0: "MOE_OK", -1: "MOE_EINVAL", -2: "MOE_ENOMEM", -3: "MOE_ECUDA",
               -4: "MOE_ETIMEOUT", -5: "MOE_ESTATE"}
MOE_SLOT_KIND_SHIFT = 29
MOE_SLOT_POOL, MOE_SLOT_SCRATCH, MOE_SLOT_COLD = 0 << 29, 1 << 29, 2 << 29
MOE_FWD_RESIDUAL = 1
MOE_GEMM_NONE, MOE_GEMM_TC, MOE_GEMM_TMA = 0, 1, 2
GEMM_KERNEL_NAME = {MOE_GEMM_NONE: "none", MOE_GEMM_TC: "tc", MOE_GEMM_TMA: "tma"}
GEMM_KERNEL_PREF = {"auto": 0, "tc": MOE_GEMM_TC, "tma": MOE_GEMM_TMA}


class moe_cache_config(C.Structure):
    _fields_ = [("num_layers", C.c_int), ("num_experts", C.c_int), ("top_k", C.c_int),
                ("hidden", C.c_int), ("inter", C.c_int), ("wdtype", C.c_int),
                ("slots_per_layer", C.c_int), ("max_tokens", C.c_int), ("renormalize", C.c_int),
                ("cold_mask_h", C.POINTER(C.c_uint8)), ("copy_mode", C.c_int), ("device", C.c_int),
                ("hbm_budget_bytes", C.c_size_t), ("mlp_kernel", C.c_int),
                ("move_interval", C.c_int), ("move_decay", C.c_float), ("move_threshold", C.c_float),
                ("move_count_tokens", C.c_int), ("evict_policy", C.c_int), ("table_layout", C.c_int),
                ("gemm_kernel", C.c_int)]


class moe_cache_counters(C.Structure):
    _fields_ = [(n, C.c_uint64) for n in ("steps", "hits", "misses", "evictions", "bypass_steps",
                                          "cold_reads", "bytes_h2d_miss", "bytes_h2d_bypass",
                                          "bytes_uva_cold", "moves")]


class moe_prepare_info(C.Structure):
    _fields_ = [("n_ids", C.c_int), ("bypass", C.c_int), ("n_distinct", C.c_int),
                ("n_cold", C.c_int), ("n_noncold", C.c_int), ("n_hits", C.c_int),
                ("n_misses", C.c_int), ("n_evictions", C.c_int),
                ("hits_h", C.POINTER(C.c_int32)), ("miss_expert_h", C.POINTER(C.c_int32)),
                ("miss_slot_h", C.POINTER(C.c_int32)), ("miss_evicted_h", C.POINTER(C.c_int32)),
                ("cold_h", C.POINTER(C.c_int32)), ("noncold_h", C.POINTER(C.c_int32))]


class moe_cache_info(C.Structure):
    _fields_ = [("expert_bytes", C.c_size_t), ("slot_stride", C.c_size_t),
                ("pool_bytes", C.c_size_t), ("scratch_bytes", C.c_size_t),
                ("backing_bytes", C.c_size_t), ("copy_mode", C.c_int), ("memcpy_gbs", C.c_double),
                ("uva_gbs", C.c_double), ("kernel_launches", C.c_uint64),
                ("scratch_experts", C.c_int), ("table_layout", C.c_int), ("gemm_kernel", C.c_int)]


class moe_cache_timing(C.Structure):
    _fields_ = [("route_ms", C.c_double), ("copy_ms", C.c_double), ("up_ms", C.c_double),
                ("down_ms", C.c_double), ("route_n", C.c_uint64), ("copy_n", C.c_uint64),
                ("up_n", C.c_uint64), ("down_n", C.c_uint64)]


_H = C.c_void_p
_P = C.c_void_p
_I = C.c_int
_S = C.c_int

# name -> (restype, argtypes); every symbol include/moe_cache.h declares
SIGNATURES = {
    "moe_cache_create": (_S, [C.POINTER(moe_cache_config), C.POINTER(_H)]),
    "moe_cache_destroy": (None, [_H]),
    "moe_cache_last_error": (C.c_char_p, [_H]),
    "moe_cache_expert_bytes": (_S, [_I, _I, _I, C.POINTER(C.c_size_t)]),
    "moe_cache_get_info": (_S, [_H, C.POINTER(moe_cache_info)]),
    "moe_cache_backing_ptr": (_S, [_H, _I, _I, C.POINTER(_P), C.POINTER(C.c_size_t)]),
    "moe_cache_load_expert": (_S, [_H, _I, _I, _P, C.c_size_t]),
    "moe_cache_router": (_S, [_H, _P, _I, _P, _P, _P]),
    "moe_cache_prepare": (_S, [_H, _I, _P, _I, _P, _P]),
    "moe_cache_last_prepare": (_S, [_H, _I, C.POINTER(moe_prepare_info)]),
    "moe_forward": (_S, [_H, _I, _P, _P, _I, _P, _I, _P]),
    "moe_expert_mlp": (_S, [_I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _I, _P]),
    "moe_expert_mlp_noalloc": (_S, [_I, _I, _I, _I, _P, _P, _P, _I, _P, _I, _P]),
    "moe_model_step_host": (_S, [_H, _P, _P, _I, _P, _I, _P]),
    "moe_cache_stats": (_S, [_H, _I, C.POINTER(moe_cache_counters)]),
    "moe_cache_get_state": (_S, [_H, _I, _P, _P, _P, _P]),
    "moe_cache_verify_slots": (_S, [_H, _I, C.POINTER(_I)]),
    "moe_cache_get_cold": (_S, [_H, _I, _P]),
    "moe_cache_pool_ptrs": (_S, [_H, _I, C.POINTER(_P), C.POINTER(_P)]),
    "moe_cache_check": (_S, [_H]),
    "moe_cache_reset": (_S, [_H]),
    "moe_cache_set_timing": (_S, [_H, _I, _I]),
    "moe_cache_read_timing": (_S, [_H, C.POINTER(moe_cache_timing)]),
    "moe_cache_read_timing_launches": (_S, [_H, _P, _P, _I, C.POINTER(_I)]),
    "moe_cache_read_copy_spans": (_S, [_H, _P, _I, C.POINTER(_I)]),
}

_lib = None


def lib() -> C.CDLL:
    """Load libmoecache.so once; raise if it is missing (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAME.get(status, status)}: {msg}")
        self.status = status


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, handle=None):
    if st != MOE_OK:
        msg = lib().moe_cache_last_error(handle)
        raise MoeError(st, msg.decode() if msg else "")


def expert_bytes(wdtype: str, hidden: int, inter: int) -> int:
    n = C.c_size_t()
    _check(lib().moe_cache_expert_bytes(WDTYPE[wdtype], hidden, inter, C.byref(n)))
    return n.value


def expert_mlp(wdtype: str, hidden: int, inter: int, top_k: int, x, block_ptrs, w, T: int,
               h_scratch, y, flags: int = 0, stream=None):
    _check(lib().moe_expert_mlp(WDTYPE[wdtype], hidden, inter, top_k, _ptr(x), _ptr(block_ptrs),
                                _ptr(w), T, _ptr(h_scratch), _ptr(y), flags, _stream(stream)))


NOALLOC_MAX_SCRATCH_FLOATS = 1 << 19


def expert_mlp_noalloc(wdtype: str, hidden: int, inter: int, top_k: int, x, block_ptrs, w, T: int,
                       y, flags: int = 0, stream=None):
    """moe_expert_mlp without a scratch argument: the library's built-in array holds h."""
    _check(lib().moe_expert_mlp_noalloc(WDTYPE[wdtype], hidden, inter, top_k, _ptr(x),
                                        _ptr(block_ptrs), _ptr(w), T, _ptr(y), flags,
                                        _stream(stream)))


class MoECache:
    """One library handle: L layers of E experts with N pool slots each."""

    def __init__(self, num_layers, num_experts, top_k, hidden, inter, wdtype, slots, max_tokens,
                 renormalize=False, cold_mask=None, copy_mode="uva", device=0, hbm_budget_bytes=0,
                 mlp_kernel="auto", moves=None, policy="lru", table="split", gemm_kernel="auto"):
        """moves: None (off) or a dict with interval, decay, threshold, count_tokens
        (run-time moves between the cold set and the pool; see moe_cache_config).
        policy: the eviction policy, one of EVICT_POLICY's keys.
        table: "split" (device pool + pinned backing store) or "vmm" (one VMM table per layer).
        gemm_kernel: "auto" (the TMA grouped GEMM where it runs) or "tc" (the cp.async one)."""
        self.L, self.E, self.k, self.H, self.I = num_layers, num_experts, top_k, hidden, inter
        self.wdtype, self.N, self.max_tokens = wdtype, slots, max_tokens
        cfg = moe_cache_config()
        cfg.num_layers, cfg.num_experts, cfg.top_k = num_layers, num_experts, top_k
        cfg.hidden, cfg.inter, cfg.wdtype = hidden, inter, WDTYPE[wdtype]
        cfg.slots_per_layer, cfg.max_tokens, cfg.renormalize = slots, max_tokens, int(bool(renormalize))
        self._cold = None
        if cold_mask is not None:
            self._cold = np.ascontiguousarray(np.asarray(cold_mask, dtype=np.uint8).reshape(-1))
            if self._cold.size != num_layers * num_experts:
                raise ValueError("cold_mask must have num_layers * num_experts entries")
            cfg.cold_mask_h = self._cold.ctypes.data_as(C.POINTER(C.c_uint8))
        cfg.copy_mode = COPY_MODE[copy_mode]
        cfg.device = device
        cfg.hbm_budget_bytes = hbm_budget_bytes
        cfg.mlp_kernel = MLP_KERNEL[mlp_kernel]
        cfg.evict_policy = EVICT_POLICY[policy]
        cfg.table_layout = TABLE_LAYOUT[table]
        cfg.gemm_kernel = GEMM_KERNEL_PREF[gemm_kernel]
        if moves:
            cfg.move_interval = int(moves.get("interval", 8))
            cfg.move_decay = float(moves.get("decay", 2.0 ** (-1.0 / 64.0)))
            cfg.move_threshold = float(moves.get("threshold", 2.0))
            cfg.move_count_tokens = int(moves.get("count_tokens", 1))
        h = _H()
        _check(lib().moe_cache_create(C.byref(cfg), C.byref(h)))
        self._h = h

    # -- lifecycle ---------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None):
            lib().moe_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def _ck(self, st):
        _check(st, self._h)

    # -- info / weights ------------------------------------------------------
    def info(self) -> dict:
        i = moe_cache_info()
        self._ck(lib().moe_cache_get_info(self._h, C.byref(i)))
        d = {n: getattr(i, n) for n, _ in moe_cache_info._fields_}
        d["copy_mode_name"] = COPY_MODE_NAME[d["copy_mode"]]
        d["gemm_kernel_name"] = GEMM_KERNEL_NAME.get(d["gemm_kernel"], "?")
        return d

    def backing_view(self, layer: int) -> np.ndarray:
        """uint8 view [E, stride] of one layer's pinned backing store (write weights here)."""
        p, stride = _P(), C.c_size_t()
        self._ck(lib().moe_cache_backing_ptr(self._h, layer, 0, C.byref(p), C.byref(stride)))
        buf = (C.c_uint8 * (self.E * stride.value)).from_address(p.value)
        return np.frombuffer(buf, dtype=np.uint8).reshape(self.E, stride.value)

    def load_expert(self, layer: int, expert: int, block: np.ndarray):
        b = np.ascontiguousarray(block, dtype=np.uint8)
        self._ck(lib().moe_cache_load_expert(self._h, layer, expert, b.ctypes.data, b.nbytes))

    # -- hot path --------------------------------------------------------------
    def router(self, logits, T, ids, w, stream=None):
        self._ck(lib().moe_cache_router(self._h, _ptr(logits), T, _ptr(ids), _ptr(w), _stream(stream)))

    def prepare(self, layer, ids, T, slot_ids=None, stream=None):
        self._ck(lib().moe_cache_prepare(self._h, layer, _ptr(ids), T, _ptr(slot_ids), _stream(stream)))

    def forward(self, layer, x, logits, T, y, flags=0, stream=None):
        self._ck(lib().moe_forward(self._h, layer, _ptr(x), _ptr(logits), T, _ptr(y), flags,
                                   _stream(stream)))

    def model_step_host(self, x_h: np.ndarray, logits_h: np.ndarray, T: int, y_h: np.ndarray,
                        timeout_ms: int = 60000, stream=None):
        self._ck(lib().moe_model_step_host(self._h, _ptr(x_h), _ptr(logits_h), T, _ptr(y_h),
                                           timeout_ms, _stream(stream)))

    # -- inspection --------------------------------------------------------------
    def last_prepare(self, layer: int) -> dict:
        bufs = {n: np.zeros(self.E, dtype=np.int32) for n in
                ("hits_h", "miss_expert_h", "miss_slot_h", "miss_evicted_h", "cold_h", "noncold_h")}
        info = moe_prepare_info()
        for n, b in bufs.items():
            setattr(info, n, b.ctypes.data_as(C.POINTER(C.c_int32)))
        self._ck(lib().moe_cache_last_prepare(self._h, layer, C.byref(info)))
        nm = info.n_misses
        return {
            "n_ids": info.n_ids, "bypass": bool(info.bypass), "n_distinct": info.n_distinct,
            "hits": bufs["hits_h"][: info.n_hits].tolist(),
            "misses": list(zip(bufs["miss_expert_h"][:nm].tolist(), bufs["miss_slot_h"][:nm].tolist(),
                               bufs["miss_evicted_h"][:nm].tolist())),
            "cold": bufs["cold_h"][: info.n_cold].tolist(),
            "noncold": bufs["noncold_h"][: info.n_noncold].tolist(),
            "n_evictions": info.n_evictions,
        }

    def stats(self, layer: int = -1) -> dict:
        s = moe_cache_counters()
        self._ck(lib().moe_cache_stats(self._h, layer, C.byref(s)))
        return {n: getattr(s, n) for n, _ in moe_cache_counters._fields_}

    def get_state(self, layer: int):
        sm = np.zeros(self.E, np.int32)
        se = np.zeros(max(self.N, 1), np.int32)
        st = np.zeros(max(self.N, 1), np.int64)
        nf = C.c_int32()
        self._ck(lib().moe_cache_get_state(self._h, layer, sm.ctypes.data, se.ctypes.data,
                                           st.ctypes.data, C.addressof(nf)))
        return sm, se[: self.N], st[: self.N], nf.value

    def verify_slots(self, layer: int) -> int:
        n = C.c_int()
        self._ck(lib().moe_cache_verify_slots(self._h, layer, C.byref(n)))
        return n.value

    def get_cold(self, layer: int) -> np.ndarray:
        """Current cold set of a layer (bool [E])."""
        m = np.zeros(self.E, np.uint8)
        self._ck(lib().moe_cache_get_cold(self._h, layer, m.ctypes.data))
        return m.astype(bool)

    def pool_ptrs(self, layer: int):
        p, s = _P(), _P()
        self._ck(lib().moe_cache_pool_ptrs(self._h, layer, C.byref(p), C.byref(s)))
        return p.value, s.value

    def check(self):
        self._ck(lib().moe_cache_check(self._h))

    def reset(self):
        self._ck(lib().moe_cache_reset(self._h))

    def set_timing(self, on: bool, capacity: int = 0):
        self._ck(lib().moe_cache_set_timing(self._h, int(bool(on)), capacity))

    def read_timing_launches(self, cap: int = 1 << 16):
        """(ms per timed MLP launch, misses of that layer step) as numpy arrays."""
        ms = np.zeros(cap, np.float32)
        mi = np.zeros(cap, np.int32)
        n = C.c_int()
        self._ck(lib().moe_cache_read_timing_launches(self._h, ms.ctypes.data, mi.ctypes.data, cap,
                                                      C.byref(n)))
        return ms[: n.value], mi[: n.value]

    def read_copy_spans(self, cap: int = 1 << 16):
        """Per timed MLP launch: (first chunk issued ns, last chunk landed ns, experts copied), uint64 [n, 3]."""
        rec = np.zeros((cap, 3), np.uint64)
        n = C.c_int()
        self._ck(lib().moe_cache_read_copy_spans(self._h, rec.ctypes.data, cap, C.byref(n)))
        return rec[: n.value]

    def read_timing(self) -> dict:
        t = moe_cache_timing()
        self._ck(lib().moe_cache_read_timing(self._h, C.byref(t)))
        return {n: getattr(t, n) for n, _ in moe_cache_timing._fields_}
