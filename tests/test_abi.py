"""CPU-side checks of the C ABI: the library builds, loads and exports every
function include/*.h declares; host-only entry points and argument checks work
without a GPU (no compute is launched)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text, re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def so():
    from hbm_slot_cache_gb300 import build
    path = build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("moe_cache_create", "moe_cache_step", "moe_cache_stats", "moe_cache_destroy"):
        assert must in names
    assert len(names) >= 13


def test_library_exports_every_declared_symbol(so):
    missing = [n for n in _declared_functions() if not hasattr(so, n)]
    assert not missing, missing


def test_python_binding_names_match_header():
    import hbm_slot_cache_gb300._lib as L
    declared = set(_declared_functions())
    assert set(L.EXPORTS) == declared
    for n in declared - {"moe_cache_strerror"}:
        assert hasattr(L, n), n


def test_host_only_calls(so):
    from hbm_slot_cache_gb300 import _lib as L
    assert L.moe_expert_bytes(6144, 2048) == (18874368, 2359296)
    assert L.strerror(L.MOE_ERR_NOT_PINNED).startswith("host backing")
    # argument errors are reported before any device work
    with pytest.raises(L.MoeError) as e:
        L.moe_cache_create(0, 16, 4, 256, 128, 2, [])
    assert e.value.code == L.MOE_ERR_ARG
    h = ctypes.c_void_p()
    hl = (L.HostLayer * 1)(L.HostLayer(16, 16, 16))
    rc = L.lib().moe_cache_create(ctypes.byref(h), 1, 16, 4, 250, 128, 2,
                                  ctypes.cast(hl, ctypes.c_void_p), None)
    assert rc == L.MOE_ERR_UNSUPPORTED and not h.value
    rc = L.lib().moe_cache_create(ctypes.byref(h), 1, 16, 4, 256, 128, 17,
                                  ctypes.cast(hl, ctypes.c_void_p), None)
    assert rc == L.MOE_ERR_UNSUPPORTED
    assert L.lib().moe_cache_step(None, 0, 1, None, None, None, None) == L.MOE_ERR_ARG
    assert L.lib().moe_cache_destroy(None) == L.MOE_OK
