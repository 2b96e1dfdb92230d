"""mla_decode_noalloc: the decode entry point for callers that cannot allocate device memory while
they decode (a plug-in whose host application owns every device allocation, or a serving loop
that must not call cudaMalloc once running).  Its split-KV scratch is the library's static device
array instead of a caller workspace; its results must equal those of mla_decode with a
workspace, call after call, and those of the oracle.

This file is named to be collected last, so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import mla_latent_kv_decode_gb300 as mla
from mla_latent_kv_decode_gb300 import harness, synth
from parity_util import LSE_ABS, OUT_ABS, assert_decode_close, oracle_decode_pairs

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


def _workspace_reference(w, dw):
    out, lse = mla.decode(w.fmt, dw.pools[0], w.num_pages, dw.q_lat, dw.q_rope, dw.block_table,
                          dw.seq_lens, w.max_seq_len, w.scale, topk_idx=dw.topk_idx)
    assert mla.check_status() == 0
    topk = 0 if dw.topk_idx is None else dw.topk_idx.shape[1]
    assert mla.decode_workspace_bytes(w.fmt, w.B, w.max_seq_len, topk) > 0   # scratch really used
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _noalloc_outputs(lib, torch, w, dw):
    out = torch.full((w.B, w.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.H), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc_call(lib, torch, w, dw, out, lse) == 0
    assert mla.check_status() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _check(w, o, l, ref_o, ref_l, oracle_pairs):
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    assert np.abs(o - ref_o).max() <= OUT_ABS
    assert np.abs(l - ref_l).max() <= LSE_ABS
    ro, rl = oracle_decode_pairs(w, oracle_pairs)
    assert_decode_close(np.stack([o[b, h] for b, h in oracle_pairs]),
                        np.array([l[b, h] for b, h in oracle_pairs]), ro, rl, f"noalloc {w.name}")


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    """Dense bf16 pages (the TMA decode kernel and its merge), two calls in a row, against
    mla_decode with a workspace and against the oracle on a few rows."""
    import torch
    lib = mla.load()
    # a ragged batch long enough that the split-KV partials and their merge are exercised
    w = synth.make_workload("paged_batch", B=7, seq_len=5000)
    dw = harness.DeviceWorkload(w, gen="host")
    ref_o, ref_l = _workspace_reference(w, dw)
    for _ in range(2):
        o, l = _noalloc_outputs(lib, torch, w, dw)
        _check(w, o, l, ref_o, ref_l, [(0, 0), (3, 77), (6, 127)])


def test_noalloc_gather_paths_with_a_smaller_plan_between():
    """FP8 pages and FP8 top-k rows (the gather kernel, whose partial slots and per-request merge
    table also live in the static array): a large call, a smaller call with a different plan,
    then the large call again, so that anything left from a larger plan would show."""
    import torch
    lib = mla.load()
    big_dense = synth.make_workload("fp8_batch", B=6, seq_len=6000)
    small_dense = synth.make_workload("fp8_batch", B=2, seq_len=700, seed=0x4D4C41 + 40)
    big_topk = synth.make_workload("topk_sparse", B=5, seq_len=9000, topk=1000)
    for big in (big_dense, big_topk):
        dwb = harness.DeviceWorkload(big, gen="host")
        dws = harness.DeviceWorkload(small_dense, gen="host")
        dwb.append()      # the tokens the workloads append (the FP8 batch's last 64 positions)
        dws.append()
        ref_b = _workspace_reference(big, dwb)
        ref_s = _workspace_reference(small_dense, dws)
        o, l = _noalloc_outputs(lib, torch, big, dwb)
        _check(big, o, l, *ref_b, [(0, 1), (big.B - 1, 100)])
        o, l = _noalloc_outputs(lib, torch, small_dense, dws)
        _check(small_dense, o, l, *ref_s, [(1, 64)])
        o, l = _noalloc_outputs(lib, torch, big, dwb)
        _check(big, o, l, *ref_b, [(2, 127)])


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    """An over-size call is refused with MLA_ERR_UNSUPPORTED before anything is looked at or
    launched.  Its output pointer is also misaligned, so that should the size check ever be
    lost, the host's pointer checks would still refuse the call (MLA_ERR_INVALID) rather than
    launch over buffers far too small for B."""
    import torch
    lib = mla.load()
    # enough requests that the per-request table alone outgrows the static array
    B = 16_000_000
    need = mla.decode_workspace_bytes(0, B, 64)
    assert need > (48 << 20)
    dummy = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    odd = ctypes.c_void_p(dummy.data_ptr() + 2)
    rc = lib.mla_decode_noalloc(0, p, 1, p, p, p, 1, p, 64, None, 0, B, 128, 0.07, odd, p,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 5   # MLA_ERR_UNSUPPORTED, nothing launched
    assert mla.check_status() == 0
