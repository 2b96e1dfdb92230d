"""The C-ABI library loads on a machine without a GPU and exports every symbol include/mla.h
declares; host-only entry points answer without touching a device.

The host-validation tests hand the library made-up device addresses (0x1000, 0x1002) that every
call must refuse before it launches anything.  They run only where no CUDA device is visible, so
that a regression in a host check can never launch a kernel over such an address."""
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


def _no_device_visible():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


needs_no_device = pytest.mark.skipif(not _no_device_visible(),
                                     reason="made-up device addresses are passed only where no device exists")


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
    for code in range(7):
        assert lib.mla_status_string(code)
    assert mla.status_string(2) == "index outside the cache pool"


@needs_no_device
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


@needs_no_device
def test_host_validation_of_the_other_entry_points(lib):
    """Argument errors of the combine, indexer and top-k entry points are answered on the host
    (MLA_ERR_INVALID = 1), and empty work returns MLA_OK, without a device."""
    d = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1002)
    # mla_combine(o_part, lse_part, S, B, H, out, lse, stream)
    assert lib.mla_combine(d, d, 0, 1, 128, d, d, None) == 1          # S < 1
    assert lib.mla_combine(d, d, 2, 1, 0, d, d, None) == 1            # H < 1
    assert lib.mla_combine(d, d, 2, -1, 128, d, d, None) == 1         # B < 0
    assert lib.mla_combine(None, None, 2, 0, 128, None, None, None) == 0
    assert lib.mla_combine(d, d, 2, 1, 128, odd, d, None) == 1        # out misaligned
    assert lib.mla_combine(None, d, 2, 1, 128, d, d, None) == 1       # null partials
    # mla_index_append(pool, num_pages, k_index, slot, T, stream)
    assert lib.mla_index_append(d, 1, d, d, -1, None) == 1
    assert lib.mla_index_append(d, -1, d, d, 1, None) == 1
    assert lib.mla_index_append(None, 0, None, None, 0, None) == 0
    assert lib.mla_index_append(odd, 1, d, d, 1, None) == 1
    # mla_indexer_score(pool, num_pages, q, w, block_table, max_pages, seq_lens, B, max_seq_len,
    #                   scores, stream)
    assert lib.mla_indexer_score(d, 1, d, d, d, 1, d, -1, 64, d, None) == 1
    assert lib.mla_indexer_score(d, 1, d, d, d, 0, d, 1, 0, d, None) == 1     # max_pages < 1
    assert lib.mla_indexer_score(d, 1, d, d, d, 1, d, 1, 65, d, None) == 1    # beyond the table
    assert lib.mla_indexer_score(None, 0, None, None, None, 1, None, 0, 64, None, None) == 0
    assert lib.mla_indexer_score(d, 1, None, d, d, 1, d, 1, 64, d, None) == 1
    # mla_topk_select(scores, ld, seq_lens, B, K, topk_idx, stream)
    assert lib.mla_topk_select(d, 100, d, 1, 0, d, None) == 1          # K < 1
    assert lib.mla_topk_select(d, -1, d, 1, 8, d, None) == 1           # ld < 0
    assert lib.mla_topk_select(d, 100, d, -1, 8, d, None) == 1         # B < 0
    assert lib.mla_topk_select(None, 100, None, 0, 8, None, None) == 0
    assert lib.mla_topk_select(d, 100, d, 1, 8, odd, None) == 1        # misaligned output
    assert lib.mla_topk_select(d, 100, d, 1 << 30, 8, d, None) == 1    # 2 B would pass 2^31 - 1
    # mla_decode_noalloc: mla_decode's checks come first (H != 128, a misaligned output), an
    # empty batch returns at once, and an over-size batch is refused before its pointers are
    # looked at; none of these touches a device
    assert lib.mla_decode_noalloc(0, d, 1, d, d, d, 1, d, 64, None, 0, 1, 64, 0.07, d, d, None) == 1
    assert lib.mla_decode_noalloc(0, d, 1, d, d, d, 1, d, 64, None, 0, 1, 128, 0.07, odd, d, None) == 1
    assert lib.mla_decode_noalloc(0, None, 0, None, None, None, 0, None, 0, None, 0, 0, 128, 0.07,
                                  None, None, None) == 0
    assert lib.mla_decode_noalloc(0, d, 1, d, d, d, 1, d, 64, None, 0, 16_000_000, 128, 0.07, odd, d,
                                  None) == 5
