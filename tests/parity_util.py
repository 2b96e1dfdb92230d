"""Shared helpers of the parity tests: oracle-side set-up from the same seeded inputs, and the
comparison bar.

Tolerances (written here once, used by every decode parity test):
  out : max |gpu - oracle| <= 1e-2 over all elements (bf16 outputs, unit-variance inputs)
  lse : max |gpu - oracle| <= 1e-3
  and, per (request, head), ||gpu - oracle||_2 <= 1e-2 * ||oracle||_2 so that a near-zero
  output cannot pass the absolute bar at long context.
"""
from __future__ import annotations

import numpy as np

import oracle
from mla_latent_kv_decode_gb300 import synth

OUT_ABS = 1e-2
LSE_ABS = 1e-3
OUT_REL = 1e-2


def oracle_pool(w: synth.Workload, upto=None):
    """Host pool holding every request's rows at the workload's slots (small workloads only).
    ``upto[b]`` limits request b to positions < upto[b] (default: seq_lens)."""
    pool = oracle.new_pool(w.fmt, w.num_pages)
    for b in range(w.B):
        n = int(w.seq_lens[b] if upto is None else upto[b])
        if n <= 0:
            continue
        c, r = synth.kv_rows(w.seed, b, 0, n)
        bad = oracle.cache_append(w.fmt, pool, c, r, w.slots(b, 0, n))
        assert bad == 0
    return pool


def request_pool(w: synth.Workload, b: int, positions=None):
    """A one-request host pool with contiguous pages holding request b's rows (all positions
    below seq_lens[b], or only ``positions``; the rest of the pool stays zero)."""
    n = int(w.seq_lens[b])
    pages = (n + 63) // 64
    pool = oracle.new_pool(w.fmt, max(pages, 1))
    if positions is None:
        c, r = synth.kv_rows(w.seed, b, 0, n)
        slot = np.arange(n, dtype=np.int32)
    else:
        positions = np.asarray(positions, dtype=np.int64)
        c, r = synth.kv_rows_at(w.seed, b, positions)
        slot = positions.astype(np.int32)
    assert oracle.cache_append(w.fmt, pool, c, r, slot) == 0
    bt = np.arange(max(pages, 1), dtype=np.int32)[None]
    return pool, bt


def oracle_decode_pairs(w: synth.Workload, pairs, nthreads=0):
    """Oracle (out, lse) for sampled (b, h) pairs, each request rebuilt on its own pool."""
    ql, qr = w.queries()
    outs = np.empty((len(pairs), synth.D_C))
    lses = np.empty(len(pairs))
    by_b = {}
    for i, (b, h) in enumerate(pairs):
        by_b.setdefault(int(b), []).append((i, int(h)))
    for b, items in by_b.items():
        if w.topk_idx is not None:
            idx = w.topk_idx[b]
            vis = idx[(idx >= 0) & (idx < w.seq_lens[b])]
            pool, bt = request_pool(w, b, np.unique(vis))
            tk = w.topk_idx[b:b + 1]
        else:
            pool, bt = request_pool(w, b)
            tk = None
        hs = [h for _, h in items]
        o, l, _ = oracle.mla_decode(w.fmt, pool, ql[b:b + 1], qr[b:b + 1], bt,
                                    w.seq_lens[b:b + 1], w.scale, topk_idx=tk,
                                    pairs=[(0, h) for h in hs], nthreads=nthreads)
        for (i, _), oo, ll in zip(items, o, l):
            outs[i] = oo
            lses[i] = ll
    return outs, lses


def assert_decode_close(out_gpu: np.ndarray, lse_gpu: np.ndarray, out_ref: np.ndarray,
                        lse_ref: np.ndarray, what: str = ""):
    """out_*: [n, 512], lse_*: [n]; empty rows (lse = -inf) must be exactly zero / -inf."""
    out_gpu = np.asarray(out_gpu, dtype=np.float64).reshape(-1, synth.D_C)
    out_ref = np.asarray(out_ref, dtype=np.float64).reshape(-1, synth.D_C)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64).reshape(-1)
    lse_ref = np.asarray(lse_ref, dtype=np.float64).reshape(-1)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), empty), f"{what}: empty-set rows differ"
    assert np.all(out_gpu[empty] == 0), f"{what}: empty rows not zero"
    ne = ~empty
    if not ne.any():
        return
    err = np.abs(out_gpu[ne] - out_ref[ne])
    assert np.all(np.isfinite(out_gpu[ne])), f"{what}: non-finite outputs"
    assert err.max() <= OUT_ABS, f"{what}: max |out err| {err.max():.3e}"
    lerr = np.abs(lse_gpu[ne] - lse_ref[ne])
    assert lerr.max() <= LSE_ABS, f"{what}: max |lse err| {lerr.max():.3e}"
    rel = np.linalg.norm(out_gpu[ne] - out_ref[ne], axis=1) / np.linalg.norm(out_ref[ne], axis=1)
    assert rel.max() <= OUT_REL, f"{what}: max normwise rel err {rel.max():.3e}"


def twin_rows(w: synth.Workload, b: int, t0: int, t1: int):
    """bf16 bits (c_kv [n,512], k_rope [n,64]) of request b's positions t0..t1-1, drawn on the
    device by the generator's twin (bit-exact with synth.kv_rows) and copied to the host: the
    same inputs the host recipe gives, at a speed that suits the full-size workloads."""
    import torch
    n = t1 - t0
    c = torch.empty((n, synth.D_C), dtype=torch.bfloat16, device="cuda")
    r = torch.empty((n, synth.D_R), dtype=torch.bfloat16, device="cuda")
    base = (b * synth.KV_ROW_STRIDE + t0) * synth.D_K
    s = torch.cuda.current_stream().cuda_stream
    synth.gpu_normal_bf16(c.data_ptr(), n, w.seed, synth.STREAM_KV, base, synth.D_C, synth.D_K, s)
    synth.gpu_normal_bf16(r.data_ptr(), n, w.seed, synth.STREAM_KV, base + synth.D_C, synth.D_R,
                          synth.D_K, s)
    return (c.cpu().view(torch.int16).numpy().view(np.uint16),
            r.cpu().view(torch.int16).numpy().view(np.uint16))


def twin_rows_at(w: synth.Workload, b: int, positions: np.ndarray):
    """twin_rows at arbitrary sorted positions of request b (drawn in ranges, then picked)."""
    positions = np.asarray(positions, dtype=np.int64)
    c = np.empty((positions.size, synth.D_C), dtype=np.uint16)
    r = np.empty((positions.size, synth.D_R), dtype=np.uint16)
    if positions.size == 0:
        return c, r
    span = 1 << 15
    for t0 in range(0, int(positions.max()) + 1, span):
        sel = np.nonzero((positions >= t0) & (positions < t0 + span))[0]
        if sel.size == 0:
            continue
        t1 = int(positions[sel].max()) + 1
        cc, rr = twin_rows(w, b, t0, t1)
        c[sel] = cc[positions[sel] - t0]
        r[sel] = rr[positions[sel] - t0]
    return c, r


def custom_workload(name, fmt, seq_lens, seed, topk_idx=None, shuffle=True, appended=0, scale=None):
    """An MLA workload (bf16 or FP8 mixed records) of the given request lengths over a shuffled
    pool, optionally with top-k lists and a softmax scale of its own."""
    seq = np.asarray(seq_lens, dtype=np.int32)
    pages = int(((seq.astype(np.int64) + 63) // 64).sum())
    perm = synth.permutation(seed, synth.STREAM_PERM, pages) if shuffle else None
    bt, total = synth._block_table(seq, perm)
    return synth.Workload(name, fmt, len(seq), 128, seed, seq, bt, total,
                          topk_idx=None if topk_idx is None else np.asarray(topk_idx, np.int32),
                          appended=appended, scale=synth.SCALE if scale is None else scale)


def run_full_compare(w, what):
    """Append every request's rows and decode the batch through the C ABI, then compare every
    cache byte (bit-exact) and every output and log-sum-exp with the oracle."""
    import mla_latent_kv_decode_gb300 as mla
    from mla_latent_kv_decode_gb300 import harness
    dw = harness.DeviceWorkload(w, gen="host")
    dw.append()
    out, lse = dw.decode()
    assert mla.check_status() == 0
    ref_pool = oracle_pool(w)
    gpu_pool = dw.pools[0].cpu().numpy()
    assert np.array_equal(gpu_pool, ref_pool), f"{what}: pool bytes differ"
    ql, qr = w.queries()
    ro, rl, _ = oracle.mla_decode(w.fmt, ref_pool, ql, qr, w.block_table, w.seq_lens, w.scale,
                                  topk_idx=w.topk_idx)
    go = out.float().cpu().numpy().reshape(-1, 512)
    gl = lse.cpu().numpy().reshape(-1)
    assert_decode_close(go, gl, ro, rl, what)
    return dw


def shared_oracle_pool(w, upto=None):
    """Host pool of shared K = V entries (V4 or V4.1) holding every request's entries."""
    pool = oracle.new_shared_pool(w.fmt, w.num_pages)
    for b in range(w.B):
        n = int(w.seq_lens[b] if upto is None else upto[b])
        if n > 0:
            assert oracle.shared_append(w.fmt, pool, synth.shared_entries(w.seed, b, 0, n), w.slots(b, 0, n)) == 0
    return pool


def run_shared_compare(w, what):
    """The shared K = V path: entries appended and decoded through the C ABI, then every pool byte
    (bit-exact), output and log-sum-exp compared with the oracle; a request with nothing visible
    must give zeros and lse = z' (the sink)."""
    import mla_latent_kv_decode_gb300 as mla
    from mla_latent_kv_decode_gb300 import harness
    dw = harness.SharedDeviceWorkload(w, gen="host")
    dw.append()
    out, lse = dw.decode()
    assert mla.check_status() == 0
    pool = shared_oracle_pool(w)
    assert np.array_equal(dw.pools[0].cpu().numpy(), pool), f"{what}: pool bytes differ"
    ro, rl = oracle.shared_kv_decode(w.fmt, pool, w.queries(), w.block_table, w.seq_lens, w.scale,
                                     sink=w.sink(), rope_cs=w.rope_cs(), topk_idx=w.topk_idx)
    go = out.float().cpu().numpy().reshape(-1, 512)
    gl = lse.cpu().numpy().reshape(-1)
    if w.use_sink:
        sk = np.tile(w.sink(), w.B)
        empty = np.isclose(rl, sk) & np.all(ro == 0, axis=1)
        assert np.all(go[empty] == 0) and np.allclose(gl[empty], sk[empty])
        keep = ~empty
        assert_decode_close(go[keep], gl[keep], ro[keep], rl[keep], what)
    else:
        assert_decode_close(go, gl, ro, rl, what)
    return dw
