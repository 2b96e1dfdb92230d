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
