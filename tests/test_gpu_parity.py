"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on identical seeded inputs.

Bit-exact: cache bytes written by mla_cache_append (both formats) and the E4M3 conversion.
Tolerance (tests/parity_util.py): decode outputs and log-sum-exps.
"""
import numpy as np
import pytest

import oracle
import mla_latent_kv_decode_gb300 as mla
from mla_latent_kv_decode_gb300 import harness, synth
from parity_util import (assert_decode_close, custom_workload as _custom, oracle_decode_pairs,
                         oracle_pool, run_full_compare, twin_rows,
                         twin_rows_at)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    mla.load()
    t.cuda.init()
    return t


def test_tiny_dense_full(torch):
    """B=1, 4,096 tokens, contiguous pages (the whole small workload, every output)."""
    run_full_compare(synth.make_workload("tiny_dense"), "tiny_dense")


def test_ragged_paged_batch_edges(torch):
    """Ragged lengths around the 64-token page and tile edges, shuffled pages, one empty request."""
    w = _custom("ragged", 0, [1, 63, 64, 65, 127, 0, 1000, 3000], seed=21)
    run_full_compare(w, "ragged bf16")


def test_split_kv_long_request(torch):
    """One long request split across many work units and merged (split-KV + LSE merge)."""
    w = _custom("long", 0, [20000], seed=22)
    run_full_compare(w, "long bf16")


def test_fp8_mixed_batch_with_append(torch):
    w = _custom("fp8", 1, [300, 64, 1, 777], seed=23, appended=64)
    run_full_compare(w, "fp8 mixed")


def test_many_requests_mixed_lengths(torch):
    """40 requests (empty, one-token, page-edge and long ones interleaved): the tile stream with
    its per-request start cost, ranges that begin or end inside a request's start units, and
    the merge of requests cut into a few pieces (warp-per-head shape)."""
    rng = np.random.default_rng(27)
    seq = rng.integers(0, 6000, size=40)
    seq[::7] = 0
    seq[3::11] = 1
    seq[5::13] = 64
    for fmt in (0, 1):
        w = _custom(f"many{fmt}", fmt, seq, seed=27)
        run_full_compare(w, f"many requests fmt={fmt}")


def test_few_long_requests_deep_merge(torch):
    """Three long requests of different lengths: each is cut into many pieces, merged by the
    block-per-head shape, with one empty request between them."""
    for fmt in (0, 1):
        w = _custom(f"few{fmt}", fmt, [17000, 0, 9000, 25001], seed=28)
        run_full_compare(w, f"few long requests fmt={fmt}")


def test_running_max_growth(torch):
    """Scores spread wide (softmax scale 4 instead of 1/sqrt(192)): a head's running max grows by
    more than the kernels' lazy-max slack (2^16) on most pages (about 360 growth events over the
    128 heads of the 4,096-token request), so O rows are rescaled mid-segment on both CTAs of a
    pair, and requests split across clusters merge partials with very different maxima."""
    for fmt in (0, 1):
        w = _custom(f"growth{fmt}", fmt, [4096, 3000, 130, 8000, 65], seed=26, scale=4.0)
        run_full_compare(w, f"running-max growth fmt={fmt}")


def test_running_max_growth_topk_rows(torch):
    """The growth test of the dense paths, through top-k tiles of both formats: bf16 records use
    the double-buffered score and P layout, FP8 records the per-group one."""
    seq = [4096, 3000, 130, 8000, 65]
    K = 1024
    idx = np.stack([synth.sorted_distinct_sample(26, synth.STREAM_TOPK, b, n, min(K, n)).tolist() +
                    [-1] * (K - min(K, n)) for b, n in enumerate(seq)]).astype(np.int32)
    for fmt in (0, 1):
        w = _custom(f"growth_topk{fmt}", fmt, seq, seed=26, scale=4.0, topk_idx=idx)
        run_full_compare(w, f"running-max growth, top-k rows fmt={fmt}")


def test_topk_sparse_with_padding(torch):
    seed = 24
    seq = [5000, 700, 4097]
    K = 300
    idx = np.stack([synth.sorted_distinct_sample(seed, synth.STREAM_TOPK, b, n, K)
                    for b, n in enumerate(seq)])
    idx[1, -20:] = -1          # padding entries
    idx[2, -5:] = 4097 + np.arange(5)   # at/after seq_len: skipped
    for fmt in (0, 1):
        w = _custom(f"topk{fmt}", fmt, seq, seed=seed, topk_idx=idx)
        run_full_compare(w, f"topk fmt={fmt}")


def test_topk_all_padding_and_empty(torch):
    w = _custom("topk_empty", 1, [100, 0], seed=25, topk_idx=np.full((2, 64), -1, np.int32))
    run_full_compare(w, "topk all padding")


def test_combine_matches_oracle(torch):
    rng = np.random.default_rng(31)
    S, B, H = 5, 2, 128
    o = rng.normal(size=(S, B, H, 512)).astype(np.float32)
    l = rng.normal(size=(S, B, H)).astype(np.float32) * 3
    l[1, 0, :] = -np.inf            # one empty part
    l[:, 1, 7] = -np.inf            # one all-empty row
    out, lse = mla.combine(torch.from_numpy(o).cuda(), torch.from_numpy(l).cuda())
    go = out.float().cpu().numpy()
    gl = lse.cpu().numpy()
    for b in range(B):
        for h in range(H):
            ro, rl = oracle.combine(o[:, b, h], l[:, b, h])
            if np.isneginf(rl):
                assert np.isneginf(gl[b, h]) and np.all(go[b, h] == 0)
                continue
            assert abs(gl[b, h] - rl) <= 1e-5
            assert np.abs(go[b, h] - ro).max() <= 1e-2 * max(1.0, np.abs(ro).max())


def test_bounds_error_is_reported(torch):
    w = _custom("bounds", 0, [200], seed=26)
    dw = harness.DeviceWorkload(w, gen="host")
    bt = dw.block_table.clone()
    bt[0, 1] = w.num_pages + 5          # a page outside the pool
    mla.decode(w.fmt, dw.pools[0], w.num_pages, dw.q_lat, dw.q_rope, bt, dw.seq_lens,
               w.max_seq_len, w.scale)
    assert mla.check_status() == 2      # MLA_ERR_BOUNDS, and cleared
    assert mla.check_status() == 0
    # an append slot past the pool is reported and not written
    c, r = dw.rows(0, 0, 1)
    before = dw.pools[0].clone()
    mla.cache_append(w.fmt, dw.pools[0], w.num_pages, c, r,
                     torch.tensor([w.num_pages * 64], dtype=torch.int32, device="cuda"))
    assert mla.check_status() == 2
    assert torch.equal(before, dw.pools[0])


def test_generator_device_twin_is_bit_exact(torch):
    w = synth.make_workload("paged_batch", B=2, seq_len=1200)
    dw_host = harness.DeviceWorkload(w, gen="host")
    dw_dev = harness.DeviceWorkload(w, gen="device")
    assert torch.equal(dw_host.pools[0], dw_dev.pools[0])
    c1, r1 = dw_host.rows(1, 5, 300)
    c2, r2 = dw_dev.rows(1, 5, 300)
    assert torch.equal(c1, c2) and torch.equal(r1, r2)


def test_e4m3_conversion_exhaustive(torch):
    """Every fp32 value in [-512, 512]: the device conversion equals the oracle encoder."""
    limit = 0x44000000                     # bit pattern of 512.0
    chunk = 1 << 27
    nth = oracle.max_threads()
    for sign in (0, 0x80000000):
        for start in range(0, limit + 1, chunk):
            end = min(limit + 1, start + chunk)
            bits = np.arange(start, end, dtype=np.uint32) | np.uint32(sign)
            x = bits.view(np.float32)
            ref = oracle.e4m3_encode_array(x, nthreads=nth)
            got = mla.e4m3_encode(torch.from_numpy(x).cuda()).cpu().numpy()
            bad = np.nonzero(got != ref)[0]
            assert bad.size == 0, (f"first mismatch x={x[bad[0]]!r} gpu={got[bad[0]]:#x} "
                                   f"oracle={ref[bad[0]]:#x}")


# --------------------------------------------------------------------------------------------
# The five workloads at full size, in the launch configuration the benchmark times: every
# (request, head) output against the oracle, and the cache bytes bit-exact against the oracle's
# encoder (the whole pool for the dense workloads, every listed record for the top-k one).  The
# rows come from the input generator's device twin (bit-exact with the host recipe, checked by
# test_generator_device_twin_is_bit_exact) and are copied to the host for the oracle.
# --------------------------------------------------------------------------------------------

def _full_size(torch, name):
    w = synth.make_workload(name)
    dw = harness.DeviceWorkload(w)
    dw.append()
    out, lse = dw.decode()
    assert mla.check_status() == 0
    go = out.float().cpu().numpy().reshape(-1, 512)
    gl = lse.cpu().numpy().reshape(-1)
    assert np.isfinite(go).all() and np.isfinite(gl).all()   # every request sees positions
    ql, qr = w.queries()
    rb = mla.record_bytes(w.fmt)
    if w.topk_idx is None:
        ref_pool = oracle.new_pool(w.fmt, w.num_pages)
        for b in range(w.B):
            n = int(w.seq_lens[b])
            for t0 in range(0, n, 1 << 15):
                t1 = min(n, t0 + (1 << 15))
                c, r = twin_rows(w, b, t0, t1)
                assert oracle.cache_append(w.fmt, ref_pool, c, r, w.slots(b, t0, t1)) == 0
        assert np.array_equal(dw.pools[0].cpu().numpy(), ref_pool), f"{name}: pool bytes differ"
        del dw
        ro, rl, _ = oracle.mla_decode(w.fmt, ref_pool, ql, qr, w.block_table, w.seq_lens, w.scale)
        assert_decode_close(go, gl, ro, rl, name)
        return
    # top-k: each request's listed records (compared with the device pool's bytes at their slots)
    # on a compact oracle pool of their own
    pool_dev = dw.pools[0]
    for b in range(w.B):
        idx = w.topk_idx[b]
        vis = np.unique(idx[(idx >= 0) & (idx < w.seq_lens[b])]).astype(np.int64)
        c, r = twin_rows_at(w, b, vis)
        pages = (int(w.seq_lens[b]) + 63) // 64
        pool = oracle.new_pool(w.fmt, pages)
        assert oracle.cache_append(w.fmt, pool, c, r, vis.astype(np.int32)) == 0
        slots = torch.from_numpy(w.slots(b, 0, 0) if vis.size == 0 else
                                 (w.block_table[b, vis // 64].astype(np.int64) * 64 + vis % 64)).cuda()
        got = pool_dev.view(-1, rb)[slots].cpu().numpy()
        want = pool.reshape(-1, rb)[vis]
        assert np.array_equal(got, want), f"{name}: records of request {b} differ"
        bt = np.arange(pages, dtype=np.int32)[None]
        ro, rl, _ = oracle.mla_decode(w.fmt, pool, ql[b:b + 1], qr[b:b + 1], bt, w.seq_lens[b:b + 1],
                                      w.scale, topk_idx=w.topk_idx[b:b + 1])
        assert_decode_close(go[b * w.H:(b + 1) * w.H], gl[b * w.H:(b + 1) * w.H], ro, rl,
                            f"{name} request {b}")


def test_full_tiny_dense(torch):
    _full_size(torch, "tiny_dense")


def test_full_paged_batch(torch):
    _full_size(torch, "paged_batch")


def test_full_long_context(torch):
    _full_size(torch, "long_context")


def test_full_fp8_batch(torch):
    _full_size(torch, "fp8_batch")


def test_full_topk_sparse(torch):
    _full_size(torch, "topk_sparse")


def test_zero_queries_average_the_latents(torch):
    """q = 0: every visible position scores 0, so out is the plain mean of the visible latents and
    lse = ln N (the oracle's zero-query special case), through pages, splits and both formats."""
    for fmt in (0, 1):
        w = _custom(f"zeroq{fmt}", fmt, [1, 64, 3001, 9000], seed=29)
        dw = harness.DeviceWorkload(w, gen="host")
        dw.q_lat.zero_()
        dw.q_rope.zero_()
        out, lse = dw.decode()
        assert mla.check_status() == 0
        pool = oracle_pool(w)
        zl = np.zeros((w.B, 128, synth.D_C), dtype=np.uint16)
        zr = np.zeros((w.B, 128, synth.D_R), dtype=np.uint16)
        ro, rl, _ = oracle.mla_decode(w.fmt, pool, zl, zr, w.block_table, w.seq_lens, w.scale)
        assert np.allclose(rl.reshape(w.B, 128), np.log(w.seq_lens.astype(np.float64))[:, None], atol=1e-12)
        assert_decode_close(out.float().cpu().numpy().reshape(-1, 512), lse.cpu().numpy().reshape(-1),
                            ro, rl, f"zero queries fmt={fmt}")


def test_topk_listing_every_position_equals_dense(torch):
    """A top-k list holding every visible position (the top-k path's degenerate case) gives the
    dense result: both paths against the oracle, and against each other."""
    seq = [130, 1000, 64]
    K = 1024
    idx = np.full((len(seq), K), -1, np.int32)
    for b, n in enumerate(seq):
        idx[b, :n] = np.arange(n, dtype=np.int32)
    for fmt in (0, 1):
        wd = _custom(f"dense{fmt}", fmt, seq, seed=30)
        wk = _custom(f"all{fmt}", fmt, seq, seed=30, topk_idx=idx)
        dd = run_full_compare(wd, f"dense fmt={fmt}")
        dk = run_full_compare(wk, f"top-k of every position fmt={fmt}")
        od, ld = dd.decode()
        ok, lk = dk.decode()
        assert np.abs(od.float().cpu().numpy() - ok.float().cpu().numpy()).max() <= 1e-2
        assert np.abs(ld.cpu().numpy() - lk.cpu().numpy()).max() <= 1e-3


def _decode_into_offset_out(torch, dw):
    """Decode again into an output 16 bytes past a 32-byte boundary (the interface asks only for
    16-byte alignment); returns (out, lse)."""
    shape, n = dw.out.shape, dw.out.numel()
    buf = torch.empty(n + 32, dtype=torch.bfloat16, device="cuda")
    off = ((16 - buf.data_ptr() % 32) % 32) // 2
    dw.out = buf[off:off + n].view(shape)
    assert dw.out.data_ptr() % 32 == 16
    out, lse = dw.decode()
    assert mla.check_status() == 0
    return out, lse


def test_output_aligned_to_16_bytes_only(torch):
    """The epilogues store whole 32-byte pieces of a row when the output allows it and 16-byte
    ones otherwise: the same bits either way, for every kernel that writes rows of out (bf16
    pages, FP8 pages, FP8 and bf16 top-k rows, both shared K = V formats)."""
    seq = [300, 64, 1, 777]
    idx = np.stack([synth.sorted_distinct_sample(64, synth.STREAM_TOPK, b, n, 128) if n >= 128 else
                    np.concatenate([np.arange(n), np.full(128 - n, -1)]) for b, n in enumerate(seq)]).astype(np.int32)
    mla_cases = [_custom("al_bf16", 0, seq, seed=61), _custom("al_fp8", 1, seq, seed=62),
                 _custom("al_fp8_topk", 1, seq, seed=63, topk_idx=idx), _custom("al_bf16_topk", 0, seq, seed=64, topk_idx=idx)]
    shared_cases = [synth.make_shared_workload(f"al_shared{f}", fmt=f, seq_lens=seq, seed=65 + f) for f in (2, 3)]
    for w, shared in [(w, False) for w in mla_cases] + [(w, True) for w in shared_cases]:
        dw = (harness.SharedDeviceWorkload if shared else harness.DeviceWorkload)(w, gen="host")
        dw.append()
        ref_out, ref_lse = (t.clone() for t in dw.decode())
        assert mla.check_status() == 0
        assert dw.out.data_ptr() % 32 == 0
        out, lse = _decode_into_offset_out(torch, dw)
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), w.name
