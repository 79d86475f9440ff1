"""CPU-side checks of the C ABI: the library loads and exports every entry
point that include/*.h declares; pure host helpers answer without a GPU."""
import ctypes
import glob
import os
import re

import pytest

from heterogeneous_adapters_lora_gb300 import lora as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        names |= set(re.findall(r"^LORA_API\s+[\w\s\*]+?\b(lora_\w+)\s*\(", txt, flags=re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from heterogeneous_adapters_lora_gb300 import build
        build.build()
    return L.lib()


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("lora_pool_create", "lora_set", "lora_reset", "lora_build_meta", "lora_shrink",
              "lora_expand", "lora_apply_slices", "lora_moe_apply"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(L.LIB_PATH)
    missing = [n for n in declared_symbols() if not hasattr(raw, n)]
    assert not missing, missing
    # and the binding wraps exactly that set
    assert set(L.EXPORTS) == set(declared_symbols())


def test_status_strings(lib):
    for code, name in L.STATUS.items():
        assert L.lora_status_string(code) == name


def test_meta_bytes_is_host_only(lib):
    a = L.lora_meta_bytes(256, 32)
    b = L.lora_meta_bytes(8192, 512)
    assert 0 < a < b
    assert L.lora_meta_bytes(16, 0) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        L.lib()
