"""Failure detection on the GPU without a GPU fault: a bounded wait that is made to run out
returns an error status to the host and leaves the context usable."""
import numpy as np
import pytest

import oracle
import mla_latent_kv_decode_gb300 as mla
from mla_latent_kv_decode_gb300 import harness, synth
from parity_util import assert_decode_close, oracle_pool

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    import torch
    w = synth.make_workload("paged_batch", B=3, seq_len=2000)
    dw = harness.DeviceWorkload(w, gen="host")
    mla.set_wait_limit(1)                 # every bounded wait gives up after one poll
    try:
        dw.decode()
        rc = mla.check_status()
    finally:
        mla.set_wait_limit(0)             # back to the default cap
    assert rc == 3                        # MLA_ERR_TIMEOUT
    assert mla.check_status() == 0        # cleared
    out, lse = dw.decode()                # the context still works and results are right
    assert mla.check_status() == 0
    ql, qr = w.queries()
    pool = oracle_pool(w)
    pairs = [(b, h) for b in range(w.B) for h in (0, 64, 127)]
    ro, rl, _ = oracle.mla_decode(w.fmt, pool, ql, qr, w.block_table, w.seq_lens, w.scale,
                                  pairs=pairs)
    go = np.stack([out[b, h].float().cpu().numpy() for b, h in pairs])
    gl = np.array([float(lse[b, h]) for b, h in pairs])
    assert_decode_close(go, gl, ro, rl, "after timeout")


def _bf16(torch, x):
    return torch.tensor([x], dtype=torch.float32).to(torch.bfloat16).item()


def test_fp8_path_reports_values_outside_its_range():
    """The FP8 record path runs its latent products on f16 operands: a q_lat element that would
    overflow f16, or a visible record whose group scale is above 255 (so that P times the scale
    could overflow f16), is reported as MLA_ERR_RANGE instead of giving silent inf/NaN.  Values at
    the edge of the range are accepted, and the next call after an error is correct."""
    import torch
    for topk in (None, 64):
        w = synth.make_workload("fp8_batch", B=2, seq_len=300) if topk is None else \
            synth.make_workload("topk_sparse", B=2, seq_len=300, topk=topk)
        dw = harness.DeviceWorkload(w, gen="host")
        dw.append()                                    # the tokens the workload appends
        dw.decode()
        assert mla.check_status() == 0
        q0 = dw.q_lat[1, 5, 17].clone()
        # 65280 is the largest bf16 below f16's overflow threshold (65520); 65536 overflows
        dw.q_lat[1, 5, 17] = 65280.0
        dw.decode()
        assert mla.check_status() == 0
        dw.q_lat[1, 5, 17] = 65536.0
        dw.decode()
        assert mla.check_status() == 6                 # MLA_ERR_RANGE, then cleared
        assert mla.check_status() == 0
        dw.q_lat[1, 5, 17] = q0
        # one visible record of request 0 with a large group-1 element: amax 114,176 gives the
        # scale 254.86 (accepted), amax 114,688 the scale 256 (refused)
        t = 0 if topk is None else int(w.topk_idx[0, 0])
        c, r = dw.rows(0, t, t + 1)
        slot = dw.slots(0, t, t + 1)
        for big, want in ((114176.0, 0), (114688.0, 6)):
            assert _bf16(torch, big) == big
            cb = c.clone()
            cb[0, 130] = big
            mla.cache_append(w.fmt, dw.pools[0], w.num_pages, cb, r, slot)
            dw.decode()
            assert mla.check_status() == want
            assert mla.check_status() == 0
        mla.cache_append(w.fmt, dw.pools[0], w.num_pages, c, r, slot)   # the original record
        out, lse = dw.decode()
        assert mla.check_status() == 0
        pool = oracle_pool(w)
        assert np.array_equal(dw.pools[0].cpu().numpy(), pool)
        ql, qr = w.queries()
        pairs = [(b, h) for b in range(w.B) for h in (0, 5, 127)]
        ro, rl, _ = oracle.mla_decode(w.fmt, pool, ql, qr, w.block_table, w.seq_lens, w.scale,
                                      topk_idx=w.topk_idx, pairs=pairs)
        go = np.stack([out[b, h].float().cpu().numpy() for b, h in pairs])
        gl = np.array([float(lse[b, h]) for b, h in pairs])
        assert_decode_close(go, gl, ro, rl, f"after range errors topk={topk}")
