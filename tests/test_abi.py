"""The C-ABI library loads on a machine without a GPU and exports every symbol include/mla.h
declares; host-only entry points answer without touching a device."""
import ctypes
import os
import re

import pytest

import mla_latent_kv_decode_gb300 as mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(mla.library_path()):
        import __graft_entry__
        __graft_entry__.build()
    return mla.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared("mla.h")
    assert "mla_decode" in names and "mla_cache_append" in names and "mla_combine" in names
    raw = ctypes.CDLL(mla.library_path())
    for n in names:
        assert hasattr(raw, n), f"{n} declared in include/mla.h but not exported"


def test_record_bytes_and_status_strings(lib):
    assert lib.mla_record_bytes(0) == 1152
    assert lib.mla_record_bytes(1) == 656
    assert lib.mla_record_bytes(7) == 0
    for code in range(6):
        assert lib.mla_status_string(code)
    assert mla.status_string(2) == "index outside the cache pool"


def test_host_validation_rejects_without_launching(lib):
    P = ctypes.c_void_p
    d = ctypes.c_void_p(0x1000)
    # H != 128
    rc = lib.mla_decode(0, d, 1, d, d, d, 1, d, 64, None, 0, 1, 64, 0.07, d, d, None, 0, None)
    assert rc == 1
    # unknown format, negative T, scale <= 0, topk without indices, max_seq_len beyond the table
    assert lib.mla_cache_append(3, d, 1, d, d, d, 1, None) == 1
    assert lib.mla_cache_append(0, d, 1, d, d, d, -1, None) == 1
    assert lib.mla_decode(0, d, 1, d, d, d, 1, d, 64, None, 0, 1, 128, 0.0, d, d, None, 0, None) == 1
    assert lib.mla_decode(0, d, 1, d, d, d, 1, d, 64, None, 5, 1, 128, 0.07, d, d, None, 0, None) == 1
    assert lib.mla_decode(0, d, 1, d, d, d, 1, d, 65, None, 0, 1, 128, 0.07, d, d, None, 0, None) == 1
    # misaligned pool
    assert lib.mla_cache_append(0, ctypes.c_void_p(0x1008), 1, d, d, d, 1, None) == 1
    # empty batch / no rows: nothing to do
    assert lib.mla_decode(0, None, 0, None, None, None, 0, None, 0, None, 0, 0, 128, 0.07, None,
                          None, None, 0, None) == 0
    assert lib.mla_cache_append(0, None, 0, None, None, None, 0, None) == 0


def test_synth_generator_library_loads():
    from mla_latent_kv_decode_gb300 import synth
    if not os.path.exists(os.path.join(os.path.dirname(mla.library_path()), "libmla_synth.so")):
        pytest.skip("not built")
    synth._load_gpu()
