"""Parity of the DSA lightning-indexer path (search-key append, indexer scores, top-k selection)
with the fp64 oracle, through the C ABI.

Bit-exact: the search-key pool bytes after mla_index_append, and the top-k indices, which are
compared with the oracle's selection applied to the kernel's own fp32 scores (where floating point
decides an integer, both sides decide it on the same values; ties go to the lower position).
Tolerance: the scores, against the fp64 oracle, within the fp32-accumulation bound derived in the
test.
"""
import numpy as np
import pytest

import oracle
import mla_latent_kv_decode_gb300 as mla
from mla_latent_kv_decode_gb300 import synth
from parity_util import assert_decode_close

pytestmark = pytest.mark.gpu

PAGE = 64


@pytest.fixture(scope="module")
def torch():
    import torch as t
    mla.load()
    t.cuda.init()
    return t


def _bits_tensor(torch, bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _index_case(torch, seq, seed, shuffle=True):
    """Host and device search-key pools of requests with lengths ``seq`` (pages shuffled)."""
    seq = np.asarray(seq, dtype=np.int32)
    pages_per = (seq.astype(np.int64) + PAGE - 1) // PAGE
    total = int(max(1, pages_per.sum()))
    perm = synth.permutation(seed, synth.STREAM_PERM, total) if shuffle else np.arange(total)
    max_pages = int(max(1, pages_per.max()))
    bt = np.full((seq.size, max_pages), -1, np.int32)
    off = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[off:off + n]
        off += n
    host = oracle.new_index_pool(total)
    dev = torch.zeros(mla.index_pool_bytes(total), dtype=torch.uint8, device="cuda")
    for b in range(seq.size):
        n = int(seq[b])
        if n == 0:
            continue
        keys = synth.index_keys(seed, b, 0, n)
        t = np.arange(n)
        slot = (bt[b, t // PAGE].astype(np.int64) * PAGE + t % PAGE).astype(np.int32)
        oracle.index_append(host, keys, slot)
        mla.index_append(dev, total, _bits_tensor(torch, keys), torch.from_numpy(slot).cuda())
    q = synth.index_queries(seed, seq.size)
    w = synth.index_weights(seed, seq.size)
    return host, dev, total, bt, seq, q, w


def _score_bound(host, q, w, bt, seq, ld):
    """Per position: 2^-15 sum_j |w_j| sum_d |q_jd| |k_d| (fp32 accumulation of 128 exact bf16
    products per head, the weighted sum over 64 heads, one scale product)."""
    qd = np.abs(oracle.bf16_to_f64(q).reshape(q.shape))
    bound = np.zeros((seq.size, ld))
    for b in range(seq.size):
        for t in range(int(seq[b])):
            k = np.abs(oracle.index_read(host, int(bt[b, t // PAGE]) * PAGE + t % PAGE))
            bound[b, t] = np.dot(np.abs(w[b]), qd[b] @ k)
    return 2.0 ** -15 * bound + 1e-30


def test_index_append_is_bit_exact(torch):
    rng = np.random.default_rng(51)
    T = 300
    x = rng.standard_normal((T, 128)).astype(np.float32) * rng.uniform(1e-3, 100, (T, 1)).astype(np.float32)
    x[7] = 0.0
    x[8, 5] = 1e30                    # one huge value: the rest flush to small codes
    bits = synth._bf16_rne(x)
    num_pages = 6
    slot = rng.permutation(num_pages * PAGE)[:T].astype(np.int32)
    slot[::50] = -1                   # skipped rows
    host = oracle.new_index_pool(num_pages)
    oracle.index_append(host, bits, slot)
    dev = torch.full((mla.index_pool_bytes(num_pages),), 0x5A, dtype=torch.uint8, device="cuda")
    ref = np.full(host.shape, 0x5A, np.uint8)
    # rows not written keep their bytes on both sides
    written = np.zeros(num_pages * PAGE, bool)
    written[slot[slot >= 0]] = True
    for s_ in np.flatnonzero(written):
        pg, row = divmod(int(s_), PAGE)
        base = pg * mla.INDEX_PAGE_BYTES
        ref[base + row * 128: base + row * 128 + 128] = host[base + row * 128: base + row * 128 + 128]
        ref[base + 8192 + 4 * row: base + 8192 + 4 * row + 4] = host[base + 8192 + 4 * row: base + 8192 + 4 * row + 4]
    mla.index_append(dev, num_pages, _bits_tensor(torch, bits), torch.from_numpy(slot).cuda())
    assert mla.check_status() == 0
    assert np.array_equal(dev.cpu().numpy(), ref)


@pytest.mark.parametrize("seq", [[1, 63, 64, 65, 127, 128, 129, 0, 700, 3000]])
def test_indexer_scores_and_topk(torch, seq):
    host, dev, total, bt, seq, q, w = _index_case(torch, seq, seed=52)
    ld = int(seq.max())
    scores = mla.indexer_score(dev, total, _bits_tensor(torch, q), torch.from_numpy(w).cuda(),
                               torch.from_numpy(bt).cuda(), torch.from_numpy(seq).cuda(), ld)
    assert mla.check_status() == 0
    gs = scores.cpu().numpy().astype(np.float64)
    ref = oracle.indexer_scores(host, q, w, bt, seq, ld)
    bound = _score_bound(host, q, w, bt, seq, ld)
    for b in range(seq.size):
        n = int(seq[b])
        err = np.abs(gs[b, :n] - ref[b, :n])
        assert np.all(err <= bound[b, :n]), (b, float(err.max()), float(bound[b, :n].min()))
    # top-k: bit-exact against the oracle's selection on the kernel's own scores
    sl = torch.from_numpy(seq).cuda()
    masked = np.where(np.arange(ld)[None, :] < seq[:, None], gs, -np.inf)
    for K in (1, 64, 129, 2048):
        got = mla.topk_select(scores, sl, K).cpu().numpy()
        exp = oracle.topk(masked, seq, K)
        assert np.array_equal(got, exp), K


def test_indexer_scores_subnormal_codes(torch):
    """Keys whose codes are almost all E4M3 subnormals (one dim holds the absmax, the others are
    ~1e-5 of it) against queries that give that dim no weight: the score is then the subnormal
    codes' contribution alone, so the bound below leaves no room for a code converted wrongly."""
    rng = np.random.default_rng(55)
    T, num_pages = 200, 4
    x = rng.uniform(-0.03, 0.03, (T, 128)).astype(np.float32)
    x[:, 0] = rng.uniform(500, 2000, T).astype(np.float32) * rng.choice([-1, 1], T)
    x[5, 1:] = 0.0
    bits = synth._bf16_rne(x)
    slot = np.arange(T, dtype=np.int32)
    host = oracle.new_index_pool(num_pages)
    oracle.index_append(host, bits, slot)
    k0 = oracle.index_read(host, 0)
    assert np.count_nonzero(np.abs(k0[1:]) < np.abs(k0[0]) * 2.0 ** -6 / 448 * 1.0001) > 100
    dev = torch.zeros(mla.index_pool_bytes(num_pages), dtype=torch.uint8, device="cuda")
    mla.index_append(dev, num_pages, _bits_tensor(torch, bits), torch.from_numpy(slot).cuda())
    q = synth._bf16_rne(rng.standard_normal((1, 64, 128)).astype(np.float32))
    q[:, :, 0] = 0
    w = rng.uniform(-1, 1, (1, 64)).astype(np.float32)
    bt = np.arange(num_pages, dtype=np.int32)[None]
    seq = np.array([T], np.int32)
    scores = mla.indexer_score(dev, num_pages, _bits_tensor(torch, q), torch.from_numpy(w).cuda(),
                               torch.from_numpy(bt).cuda(), torch.from_numpy(seq).cuda(), T)
    assert mla.check_status() == 0
    gs = scores.cpu().numpy().astype(np.float64)[0]
    ref = oracle.indexer_scores(host, q, w, bt, seq, T)[0]
    bound = _score_bound(host, q, w, bt, seq, T)[0]
    assert np.count_nonzero(ref) > T // 2
    assert np.all(np.abs(gs - ref) <= bound), float(np.max(np.abs(gs - ref) - bound))


def test_topk_ties_and_edges(torch):
    rng = np.random.default_rng(53)
    B, ld = 6, 9000
    s = rng.standard_normal((B, ld)).astype(np.float32)
    s[1] = np.round(s[1] * 4) / 4          # heavy ties
    s[2] = 1.5                              # all equal: the lowest positions win
    s[3, ::2] = -0.0                        # both zeros
    s[3, 1::2] = 0.0
    s[4] = np.linspace(-1, 1, ld, dtype=np.float32)[::-1].copy()
    seq = np.array([9000, 8191, 5000, 4097, 2048, 0], np.int32)
    sc = torch.from_numpy(s).cuda()
    sl = torch.from_numpy(seq).cuda()
    for K in (1, 100, 2048, 4096):
        got = mla.topk_select(sc, sl, K).cpu().numpy()
        exp = oracle.topk(s.astype(np.float64), seq, K)
        assert np.array_equal(got, exp), K


def test_topk_unaligned_rows(torch):
    """A row stride that is not a multiple of four scores, so that rows (and the second CTA's half)
    start off a 16-byte boundary: the loads' unaligned heads and tails."""
    rng = np.random.default_rng(59)
    B, ld = 4, 9001
    s = rng.standard_normal((B, ld)).astype(np.float32)
    s[2] = np.round(s[2] * 8) / 8            # ties
    seq = np.array([9001, 7777, 6003, 130], np.int32)
    sc = torch.from_numpy(s).cuda()
    sl = torch.from_numpy(seq).cuda()
    for K in (1, 100, 2048):
        got = mla.topk_select(sc, sl, K).cpu().numpy()
        exp = oracle.topk(s.astype(np.float64), seq, K)
        assert np.array_equal(got, exp), K


def test_topk_crowded_first_digit(torch):
    """Keys crowding one bin of the first digit (one exponent and two mantissa bits) beyond the
    8,192 candidates a CTA keeps in shared memory, in both halves or in the first only: both CTAs
    of the pair then take the later digits from the row; a spread row keeps the candidate path."""
    rng = np.random.default_rng(57)
    B, ld = 4, 40000
    s = np.empty((B, ld), np.float32)
    s[0] = rng.uniform(1.0, 1.25, ld)                        # every key in one first-digit bin
    s[1] = np.round(rng.uniform(1.0, 1.25, ld) * 64) / 64    # the same with heavy ties
    s[2, :20000] = rng.uniform(1.0, 1.25, 20000)             # first half crowded, second spread
    s[2, 20000:] = rng.standard_normal(20000)
    s[3] = rng.standard_normal(ld)                           # candidates fit
    seq = np.array([40000, 39999, 40000, 40000], np.int32)
    sc = torch.from_numpy(s).cuda()
    sl = torch.from_numpy(seq).cuda()
    for K in (2048, 8000):
        got = mla.topk_select(sc, sl, K).cpu().numpy()
        exp = oracle.topk(s.astype(np.float64), seq, K)
        assert np.array_equal(got, exp), K


def test_indexer_selection_feeds_sparse_decode(torch):
    """Search keys -> scores -> top-k -> sparse FP8 decode of the picked positions, against the
    oracle decode of the same picks (the DSA path of "MLA that reads only the picked positions",
    Fig. 10)."""
    from mla_latent_kv_decode_gb300 import harness
    seed = 54
    seq = np.array([5000, 300, 2100], np.int32)
    K = 256
    # the main cache and the search-key pool share the block table
    pages = int(((seq.astype(np.int64) + 63) // 64).sum())
    perm = synth.permutation(seed, synth.STREAM_PERM, pages)
    bt, total = synth._block_table(seq, perm)
    w_ = synth.Workload("dsa", 1, seq.size, 128, seed, seq, bt, total)
    dw = harness.DeviceWorkload(w_, gen="host")
    dw.append()
    host_idx = oracle.new_index_pool(total)
    dev_idx = torch.zeros(mla.index_pool_bytes(total), dtype=torch.uint8, device="cuda")
    for b in range(seq.size):
        n = int(seq[b])
        keys = synth.index_keys(seed, b, 0, n)
        slot = w_.slots(b, 0, n)
        oracle.index_append(host_idx, keys, slot)
        mla.index_append(dev_idx, total, _bits_tensor(torch, keys), torch.from_numpy(slot).cuda())
    q = synth.index_queries(seed, seq.size)
    w = synth.index_weights(seed, seq.size)
    ld = int(seq.max())
    scores = mla.indexer_score(dev_idx, total, _bits_tensor(torch, q), torch.from_numpy(w).cuda(),
                               dw.block_table, dw.seq_lens, ld)
    idx = mla.topk_select(scores, dw.seq_lens, K)
    dw.topk_idx = idx
    out, lse = mla.decode(1, dw.pools[0], total, dw.q_lat, dw.q_rope, dw.block_table, dw.seq_lens,
                          ld, w_.scale, topk_idx=idx)
    assert mla.check_status() == 0
    picks = idx.cpu().numpy()
    ql, qr = w_.queries()
    ro, rl, _ = oracle.mla_decode(1, dw.pools[0].cpu().numpy(), ql, qr, bt, seq, w_.scale, topk_idx=picks)
    assert_decode_close(out.float().cpu().numpy().reshape(-1, 512), lse.cpu().numpy().reshape(-1), ro, rl,
                        "indexer -> top-k -> sparse decode")
