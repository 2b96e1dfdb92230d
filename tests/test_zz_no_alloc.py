"""mla_decode_noalloc: the decode entry point for callers that cannot allocate device memory while
they decode (a plug-in whose host application owns every device allocation, or a serving loop
that must not call cudaMalloc once running).  Its split-KV scratch is the library's static device
array instead of a caller workspace; its results must equal those of mla_decode with a
workspace, call after call.

This file is named to be collected last, so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import mla_latent_kv_decode_gb300 as mla
from mla_latent_kv_decode_gb300 import harness, synth
from parity_util import LSE_ABS, OUT_ABS

pytestmark = pytest.mark.gpu


def _noalloc_call(lib, torch, w, dw, out, lse):
    rc = lib.mla_decode_noalloc(
        w.fmt, ctypes.c_void_p(dw.pools[0].data_ptr()), w.num_pages,
        ctypes.c_void_p(dw.q_lat.data_ptr()), ctypes.c_void_p(dw.q_rope.data_ptr()),
        ctypes.c_void_p(dw.block_table.data_ptr()), w.max_pages,
        ctypes.c_void_p(dw.seq_lens.data_ptr()), w.max_seq_len,
        None if dw.topk_idx is None else ctypes.c_void_p(dw.topk_idx.data_ptr()),
        0 if dw.topk_idx is None else dw.topk_idx.shape[1], w.B, w.H, w.scale,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    import torch
    lib = mla.load()
    # a ragged batch long enough that the split-KV partials and their merge are exercised
    w = synth.make_workload("paged_batch", B=7, seq_len=5000)
    dw = harness.DeviceWorkload(w, gen="host")
    ref_out, ref_lse = mla.decode(w.fmt, dw.pools[0], w.num_pages, dw.q_lat, dw.q_rope,
                                  dw.block_table, dw.seq_lens, w.max_seq_len, w.scale)
    assert mla.check_status() == 0
    assert mla.decode_workspace_bytes(w.fmt, w.B, w.max_seq_len) > 0   # scratch really used
    ref_out = ref_out.float().cpu().numpy()
    ref_lse = ref_lse.cpu().numpy()
    for _ in range(2):
        out = torch.full((w.B, w.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.B, w.H), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc_call(lib, torch, w, dw, out, lse) == 0
        assert mla.check_status() == 0
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
        assert np.abs(o - ref_out).max() <= OUT_ABS
        assert np.abs(l - ref_lse).max() <= LSE_ABS


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    import torch
    lib = mla.load()
    # enough requests that the per-request table alone outgrows the static array
    B = 16_000_000
    need = mla.decode_workspace_bytes(0, B, 64)
    assert need > (48 << 20)
    dummy = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = lib.mla_decode_noalloc(0, p, 1, p, p, p, 1, p, 64, None, 0, B, 128, 0.07, p, p,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 5   # MLA_ERR_UNSUPPORTED, nothing launched
    assert mla.check_status() == 0
