"""The C-ABI library builds, loads and exports every entry point that
include/*.h declares; the Python binding covers exactly those names.
No compute calls (runs without a GPU)."""

import ctypes
import glob
import os
import re

import pytest

from tests.conftest import ROOT

HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))
_DECL = re.compile(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?([a-z_][a-z0-9_]*)\s*\(", re.M)


def declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in _DECL.finditer(src):
            if not m.group(0).lstrip().startswith(("typedef", "return", "#")):
                names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def built_lib():
    from expert_slot_cache_topk_gb300 import _build
    return _build.build()


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("moe_cache_create", "moe_cache_prepare", "moe_forward", "moe_cache_stats",
              "moe_cache_router", "moe_cache_destroy", "moe_expert_mlp"):
        assert n in names


def test_library_exports_every_declared_symbol(built_lib):
    L = ctypes.CDLL(built_lib)
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_signatures_cover_header(built_lib):
    from expert_slot_cache_topk_gb300 import _abi
    assert set(_abi.SIGNATURES) == declared_functions()
    _abi.lib()   # sets every restype/argtypes without calling into CUDA


def test_expert_bytes_without_gpu(built_lib):
    from expert_slot_cache_topk_gb300 import _abi
    assert _abi.expert_bytes("int4g128", 2560, 640) == 2_534_400
    assert _abi.expert_bytes("bf16", 2048, 1024) == 12 * 2 ** 20
    assert _abi.expert_bytes("fp8", 2048, 1024) == 3 * 2048 * 1024 + 32
    with pytest.raises(_abi.MoeError):
        _abi.expert_bytes("int4g128", 2560, 100)
