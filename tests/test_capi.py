"""The C ABI library loads and exports every symbol include/pagedkv.h declares;
host-side argument checks reject bad calls before any launch (CPU only: no
compute call reaches the GPU)."""

import ctypes
import os
import re

import pytest

from libbuild import ROOT, ensure_built

HEADER = os.path.join(ROOT, "include", "pagedkv.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*int\s+(\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported():
    kb = ensure_built()
    lib = kb.lib()
    names = declared_functions()
    assert len(names) >= 20
    for name in names:
        assert hasattr(lib, name), f"{name} is declared but not exported"
        assert name in kb.SIGNATURES, f"{name} has no binding signature"
    assert set(kb.SIGNATURES) == set(names)


def test_argument_checks_fail_before_launch():
    kb = ensure_built()
    lib = kb.lib()
    null = ctypes.c_void_p()
    assert lib.store_cache(null, 0, null, null, null, 4, null) == kb.KVP_ERR_INVALID_ARG
    assert lib.copy_pages(null, null, null, 1, null) == kb.KVP_ERR_INVALID_ARG
    assert lib.page_table_write(null, 1, 1, null, null, null, 1, 1, null, null) == kb.KVP_ERR_INVALID_ARG
    assert lib.page_table_write(ctypes.c_void_p(16), 1, 1, null, null, null, 1, 0, null, null) == kb.KVP_ERR_INVALID_ARG
    assert lib.paged_decode_attention(null, 0, null, 1, 1, null, 1, 1, 0, null, null, 0, 0, 1.0, null, null, 0,
                                      null) == kb.KVP_ERR_INVALID_ARG
    assert lib.gather_indices(null, null, 1, 1, 0, null, null, 1, 0, 0, null, 1, null) == kb.KVP_ERR_INVALID_ARG
    assert lib.kvp_selftest_wait(1000, 0, null, null) == kb.KVP_ERR_INVALID_ARG
    assert lib.kvp_selftest_wait(0, 0, ctypes.c_void_p(16), null) == kb.KVP_ERR_INVALID_ARG
    assert lib.kvp_selftest_wait(2_000_000_000, 0, ctypes.c_void_p(16), null) == kb.KVP_ERR_INVALID_ARG
    assert lib.kvp_selftest_wait(1000, 2, ctypes.c_void_p(16), null) == kb.KVP_ERR_INVALID_ARG
    BT = kb.KVP_BLOCK_TABLE
    assert lib.paged_prefill_attention(null, 0, null, 1, 1, 1, null, null, 1, 1, BT, null, null, 0, 0, 1.0, null,
                                       null) == kb.KVP_ERR_INVALID_ARG
    assert lib.paged_verify_attention(null, 0, null, 1, 1, 1, null, 1, 1, BT, null, null, 0, 0, 1.0, null, null, 0,
                                      null) == kb.KVP_ERR_INVALID_ARG
    assert lib.store_cache_and_attention(null, 0, null, null, null, null, 1, 1, null, 1, 1, BT, null, null, null,
                                         null, null, 0, 0, 0, 1.0, null, null, 0, null) == kb.KVP_ERR_INVALID_ARG
    assert lib.kvp_decode_step_device_io(null, null, null, 1, 1, BT, null, 1, 0, 0, 1, 1.0, null, null, null, null,
                                         null, null, null, null, null, 0, null, 0, null) == kb.KVP_ERR_INVALID_ARG
    out = ctypes.c_void_p()
    # misaligned buffer and bad dtype are rejected before any CUDA call
    assert lib.kv_pool_create(4, 4, 1, 16, 1, 1, ctypes.c_void_p(8), ctypes.c_void_p(64),
                              ctypes.byref(out)) == kb.KVP_ERR_INVALID_ARG
    assert lib.kv_pool_create(4, 4, 1, 16, 7, 1, ctypes.c_void_p(256), ctypes.c_void_p(64),
                              ctypes.byref(out)) == kb.KVP_ERR_INVALID_ARG
    # a row of kv_heads * head_dim * elem bytes must be a multiple of 16
    assert lib.kv_pool_create(4, 4, 1, 6, 1, 1, ctypes.c_void_p(256), ctypes.c_void_p(64),
                              ctypes.byref(out)) == kb.KVP_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    kb = ensure_built()
    monkeypatch.setattr(kb, "_lib", None)
    monkeypatch.setattr(kb, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError):
        kb.lib()


def test_tracing_accessors_live_only_in_the_tracing_build():
    """The prefill kernel's tracing build (KVP_PREFILL_TRACE) exports its two
    accessors; the product library exports neither, and neither library is
    the other."""
    kb = ensure_built()
    from paged_decode_attention_store_gb300 import build as kbuild

    traced = kbuild.build_traced()
    assert os.path.abspath(traced) != os.path.abspath(kb.LIB_PATH)
    t = ctypes.CDLL(traced)
    for name in ("kvp_prefill_trace_arm", "kvp_prefill_trace_read"):
        assert hasattr(t, name), f"the tracing build lacks {name}"
        assert not hasattr(kb.lib(), name), f"the product library exports {name}"
    for name in declared_functions():  # the tracing build is the whole library besides
        assert hasattr(t, name), f"the tracing build lacks {name}"
