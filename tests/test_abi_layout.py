"""The ctypes binding agrees with include/moe_cache.h byte for byte: every
struct's size and every field's offset, and every enum value and constant
the binding repeats.  A C probe compiled with the host compiler prints what
the header defines; no library call is made (runs without a GPU)."""

import ctypes
import os
import shutil
import subprocess

import pytest

from tests.conftest import ROOT

STRUCTS = ["moe_cache_config", "moe_cache_counters", "moe_prepare_info", "moe_cache_info", "moe_cache_timing"]

CONSTANTS = {
    "MOE_F32": "MOE_F32", "MOE_BF16": "MOE_BF16", "MOE_INT4_G128": "MOE_INT4_G128",
    "MOE_FP8_E4M3": "MOE_FP8_E4M3",
    "MOE_COPY_AUTO": "MOE_COPY_AUTO", "MOE_COPY_MEMCPY": "MOE_COPY_MEMCPY", "MOE_COPY_UVA": "MOE_COPY_UVA",
    "MOE_COPY_FUSED": "MOE_COPY_FUSED",
    "MOE_MLP_AUTO": "MOE_MLP_AUTO", "MOE_MLP_PLAIN": "MOE_MLP_PLAIN",
    "MOE_EVICT_LRU": "MOE_EVICT_LRU", "MOE_EVICT_LFU": "MOE_EVICT_LFU", "MOE_EVICT_FIFO": "MOE_EVICT_FIFO",
    "MOE_EVICT_SLRU": "MOE_EVICT_SLRU",
    "MOE_TABLE_SPLIT": "MOE_TABLE_SPLIT", "MOE_TABLE_VMM": "MOE_TABLE_VMM",
    "MOE_OK": "MOE_OK", "MOE_EINVAL": "MOE_EINVAL", "MOE_ENOMEM": "MOE_ENOMEM", "MOE_ECUDA": "MOE_ECUDA",
    "MOE_ETIMEOUT": "MOE_ETIMEOUT", "MOE_ESTATE": "MOE_ESTATE",
    "MOE_SLOT_KIND_SHIFT": "MOE_SLOT_KIND_SHIFT", "MOE_SLOT_POOL": "MOE_SLOT_POOL",
    "MOE_SLOT_SCRATCH": "MOE_SLOT_SCRATCH", "MOE_SLOT_COLD": "MOE_SLOT_COLD",
    "MOE_FWD_RESIDUAL": "MOE_FWD_RESIDUAL",
    "MOE_GEMM_NONE": "MOE_GEMM_NONE", "MOE_GEMM_TC": "MOE_GEMM_TC", "MOE_GEMM_TMA": "MOE_GEMM_TMA",
}


def _probe_source():
    from expert_slot_cache_topk_gb300 import _abi
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe_cache.h"', "int main(void) {"]
    for s in STRUCTS:
        lines.append(f'  printf("size {s} %zu\\n", sizeof({s}));')
        for name, _ in getattr(_abi, s)._fields_:
            lines.append(f'  printf("off {s}.{name} %zu\\n", offsetof({s}, {name}));')
    for c in CONSTANTS.values():
        lines.append(f'  printf("const {c} %lld\\n", (long long){c});')
    lines += ["  return 0;", "}"]
    return "\n".join(lines) + "\n"


@pytest.fixture(scope="module")
def header_facts(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    d = tmp_path_factory.mktemp("abi_probe")
    src, exe = d / "probe.c", d / "probe"
    src.write_text(_probe_source())
    subprocess.check_call([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           str(src), "-o", str(exe)])
    facts = {}
    for line in subprocess.check_output([str(exe)], text=True).splitlines():
        kind, key, val = line.split()
        facts[(kind, key)] = int(val)
    return facts


def test_struct_sizes_and_field_offsets_match_the_header(header_facts):
    from expert_slot_cache_topk_gb300 import _abi
    for s in STRUCTS:
        cls = getattr(_abi, s)
        assert ctypes.sizeof(cls) == header_facts[("size", s)], s
        for name, _ in cls._fields_:
            assert getattr(cls, name).offset == header_facts[("off", f"{s}.{name}")], f"{s}.{name}"


def test_every_header_field_is_bound(header_facts):
    """The last bound field ends where the C struct's padding allows: no C
    field is left out of a ctypes struct (an unbound trailing field would make
    the C struct larger than the end of the last bound field, rounded up to
    the struct's alignment)."""
    from expert_slot_cache_topk_gb300 import _abi
    for s in STRUCTS:
        cls = getattr(_abi, s)
        name, typ = cls._fields_[-1]
        end = getattr(cls, name).offset + ctypes.sizeof(typ)
        align = ctypes.alignment(cls)
        assert (end + align - 1) // align * align == header_facts[("size", s)], s


def test_enum_values_and_constants_match_the_header(header_facts):
    from expert_slot_cache_topk_gb300 import _abi
    for py_name, c_name in CONSTANTS.items():
        assert getattr(_abi, py_name) == header_facts[("const", c_name)], py_name
