"""Pins of the fp64 oracle to facts the source pages and mathematics fix (CPU only).

Each test names the passage it checks.  Together they are chosen so that a plausible slip in
the oracle (a dropped rope term, a wrong scale, a transposed operand, a wrong page/row index,
a wrong FP8 rounding or scale rule, a wrong merge weight) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from mla_latent_kv_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, *v = line.split()
            vals[k] = [float(x) for x in v]
    return vals


# ------------------------------------------------------------------------------------------
# Worked example: "What attention stores, and what DeepSeek changed",
# section "The four numbers attention works with".
# ------------------------------------------------------------------------------------------

def _worked():
    g = _golden("worked_example.txt")
    d = int(g["d_h"][0])
    K = np.array(g["K_flat"]).reshape(d, 3).T   # column-major: one column per token
    V = np.array(g["V_flat"]).reshape(d, 3).T
    return g, d, K, V, np.array(g["q3"])


def test_worked_example_scores_weights_output():
    g, d, K, V, q = _worked()
    out, lse, s = oracle.attend(q, K, V, 1.0 / math.sqrt(d), return_scores=True)
    np.testing.assert_allclose(s, g["scores"], atol=6e-4)
    np.testing.assert_allclose(out, g["out"], atol=6e-4)
    # weights: attending with V = identity returns the probability vector itself
    w, _ = oracle.attend(q, K, np.eye(3), 1.0 / math.sqrt(d))
    np.testing.assert_allclose(w, g["weights"], atol=6e-4)
    assert abs(w.sum() - 1.0) < 1e-15
    # lse is not printed; consistency: ln(sum exp(scores)) from the printed scores
    assert abs(lse - math.log(sum(math.exp(x) for x in g["scores"]))) < 2e-3


def test_worked_example_row_major_reading_does_not_match():
    """The alternative reading of the garbled matrices is rejected by the printed numbers."""
    g, d, _, _, q = _worked()
    K_rm = np.array(g["K_flat"]).reshape(3, d)
    w, _ = oracle.attend(q, K_rm, np.eye(3), 1.0 / math.sqrt(d))
    assert np.abs(w - np.array(g["weights"])).max() > 0.1


# ------------------------------------------------------------------------------------------
# Absorption = expansion ("DeepSeek's KV Cache", Fig. 5 (1)/(2) and Fig. 6 (1)/(2);
# "What attention stores", section "Two paths, one score")
# ------------------------------------------------------------------------------------------

def test_absorbed_equals_expanded_generic_core():
    rng = np.random.default_rng(1)
    d_h, d_c, d_r, n = 128, 512, 64, 97
    W_uk = rng.normal(0, 1 / math.sqrt(d_c), (d_c, d_h))
    W_uv = rng.normal(0, 1 / math.sqrt(d_c), (d_c, d_h))
    qc = rng.normal(size=d_h)
    qr = rng.normal(size=d_r)
    C = rng.normal(size=(n, d_c))
    KR = rng.normal(size=(n, d_r))
    scale = 1 / math.sqrt(d_h + d_r)
    # expanded: per-head key and value built from the latent at every position
    Kc = C @ W_uk
    Vh = C @ W_uv
    out_exp, lse_exp, s_exp = oracle.attend(np.concatenate([qc, qr]), np.hstack([Kc, KR]), Vh,
                                            scale, return_scores=True)
    # absorbed: W_uk folded into the query, latent used directly as key and as value
    q_lat = W_uk @ qc
    U, lse_abs, s_abs = oracle.attend(np.concatenate([q_lat, qr]), np.hstack([C, KR]), C, scale,
                                      return_scores=True)
    np.testing.assert_allclose(s_abs, s_exp, rtol=0, atol=1e-9)
    assert abs(lse_abs - lse_exp) < 1e-9
    np.testing.assert_allclose(U @ W_uv, out_exp, rtol=0, atol=1e-9)


def _pool_from_rows(fmt, c_rows, r_rows, seq_lens, perm_seed=7):
    """Build a shuffled paged pool + block table holding rows[b][t] at position t of request b."""
    B = len(seq_lens)
    pages_per = [(n + 63) // 64 for n in seq_lens]
    total = sum(pages_per)
    perm = np.random.default_rng(perm_seed).permutation(total)
    bt = np.full((B, max(pages_per)), -1, dtype=np.int32)
    pool = oracle.new_pool(fmt, total)
    off = 0
    for b in range(B):
        bt[b, :pages_per[b]] = perm[off:off + pages_per[b]]
        off += pages_per[b]
        t = np.arange(seq_lens[b])
        slot = (bt[b, t // 64].astype(np.int64) * 64 + t % 64).astype(np.int32)
        assert oracle.cache_append(fmt, pool, c_rows[b], r_rows[b], slot) == 0
    return pool, bt


def _bf16(x):
    return synth._bf16_rne(np.asarray(x, dtype=np.float32))


def test_absorbed_mla_decode_equals_expanded_heads_through_paged_pool():
    """MLA wrapper (paged reads, content + rope score, V = latent) vs an expanded-MHA brute force.

    W^UK and q^C are small integers so the absorbed query W^UK q^C is exact in bf16; the latent
    cache is bf16 N(0,1).  Scores and up-projected outputs agree to 1e-9.
    """
    rng = np.random.default_rng(3)
    H, d_h = 4, 128
    seq_lens = [130, 64, 1]
    c_rows = [_bf16(rng.normal(size=(n, 512))) for n in seq_lens]
    r_rows = [_bf16(rng.normal(size=(n, 64))) for n in seq_lens]
    pool, bt = _pool_from_rows(oracle.BF16, c_rows, r_rows, seq_lens)
    W_uk = rng.integers(-1, 2, size=(H, 512, d_h)).astype(np.float64)
    W_uv = rng.normal(size=(H, 512, d_h))
    qc = rng.integers(-1, 2, size=(len(seq_lens), H, d_h)).astype(np.float64)
    qr = _bf16(rng.normal(size=(len(seq_lens), H, 64)))
    q_lat = np.einsum("hkd,bhd->bhk", W_uk, qc)
    assert np.abs(q_lat).max() < 256        # integers below 256 are exact in bf16
    scale = synth.SCALE
    out, lse, _ = oracle.mla_decode(oracle.BF16, pool, _bf16(q_lat), qr, bt,
                                    np.array(seq_lens, dtype=np.int32), scale)
    out = out.reshape(len(seq_lens), H, 512)
    lse = lse.reshape(len(seq_lens), H)
    for b, n in enumerate(seq_lens):
        C = oracle.bf16_to_f64(c_rows[b])
        KR = oracle.bf16_to_f64(r_rows[b])
        for h in range(H):
            Kc = C @ W_uk[h]
            Vh = C @ W_uv[h]
            q = np.concatenate([qc[b, h], oracle.bf16_to_f64(qr[b, h])])
            o_exp, l_exp = oracle.attend(q, np.hstack([Kc, KR]), Vh, float(np.float32(scale)))
            assert abs(lse[b, h] - l_exp) < 1e-9
            np.testing.assert_allclose(out[b, h] @ W_uv[h], o_exp, rtol=0, atol=1e-9)


# ------------------------------------------------------------------------------------------
# Byte closed forms ("DeepSeek's KV Cache": "The baseline", "Calculating V2's KV cache",
# "Calculating V3.2's KV cache", "Looking at reads"; "What attention stores": "The cache table")
# ------------------------------------------------------------------------------------------

def test_byte_closed_forms():
    g = {k: int(v[0]) for k, v in _golden("byte_counts.txt").items()}
    rb16 = oracle.record_bytes(oracle.BF16)
    rb8 = oracle.record_bytes(oracle.FP8_MIXED)
    assert rb16 == g["bf16_record_bytes"]
    assert rb8 == g["fp8_mixed_record_bytes"]
    assert 60 * rb16 == g["v2_mla_bytes_per_token"]
    assert 61 * rb16 == g["v3_mla_bytes_per_token"]
    assert 60 * 131072 * rb16 == g["v2_read_bytes_131072_ctx"]
    assert 61 * (rb8 + 132) == g["v32_bytes_per_token"]
    assert 61 * 2048 * rb8 == g["v32_sparse_kv_read_bytes"]
    assert rb16 // 2 == g["mla_elements_per_token_layer"]
    assert 60 * g["mha_elements_per_token_layer"] * 2 == g["mha_v2_bytes_per_token"]
    # the hypothetical MHA is ~57x the MLA record ("about 1/57 of MHA")
    assert round(g["mha_v2_bytes_per_token"] / g["v2_mla_bytes_per_token"]) == 57
    assert oracle.new_pool(oracle.BF16, 3).size == 3 * 64 * 1152


# ------------------------------------------------------------------------------------------
# Special cases of the decode definition
# ------------------------------------------------------------------------------------------

def _small_case(fmt=oracle.BF16, seq_lens=(70, 1, 128), H=3, seed=11):
    rng = np.random.default_rng(seed)
    c_rows = [_bf16(rng.normal(size=(n, 512))) for n in seq_lens]
    r_rows = [_bf16(rng.normal(size=(n, 64))) for n in seq_lens]
    pool, bt = _pool_from_rows(fmt, c_rows, r_rows, list(seq_lens))
    q_lat = _bf16(rng.normal(size=(len(seq_lens), H, 512)))
    q_rope = _bf16(rng.normal(size=(len(seq_lens), H, 64)))
    return pool, bt, np.array(seq_lens, dtype=np.int32), q_lat, q_rope, c_rows, r_rows


def test_single_position_returns_that_latent_and_its_score():
    pool, bt, sl, ql, qr, c_rows, r_rows = _small_case(seq_lens=(1,))
    out, lse, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, sl, synth.SCALE)
    c = oracle.bf16_to_f64(c_rows[0][0])
    kr = oracle.bf16_to_f64(r_rows[0][0])
    for h in range(ql.shape[1]):
        np.testing.assert_array_equal(out[h], c)        # exactly the cached latent
        s = float(np.float32(synth.SCALE)) * (oracle.bf16_to_f64(ql[0, h]) @ c +
                                              oracle.bf16_to_f64(qr[0, h]) @ kr)
        assert abs(lse[h] - s) < 1e-12


def test_zero_scale_gives_mean_latent_and_log_n():
    pool, bt, sl, ql, qr, c_rows, _ = _small_case()
    out, lse, pairs = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, sl, 0.0)
    for i, (b, h) in enumerate(pairs):
        np.testing.assert_allclose(out[i], oracle.bf16_to_f64(c_rows[b]).mean(0), atol=1e-13)
        assert abs(lse[i] - math.log(sl[b])) < 1e-13


def test_identical_rows_give_that_row():
    rng = np.random.default_rng(5)
    row_c = _bf16(rng.normal(size=512))
    row_r = _bf16(rng.normal(size=64))
    n = 150
    pool, bt = _pool_from_rows(oracle.BF16, [np.tile(row_c, (n, 1))], [np.tile(row_r, (n, 1))], [n])
    ql = _bf16(rng.normal(size=(1, 2, 512)))
    qr = _bf16(rng.normal(size=(1, 2, 64)))
    out, _, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, np.array([n], np.int32), synth.SCALE)
    np.testing.assert_allclose(out, np.tile(oracle.bf16_to_f64(row_c), (2, 1)), atol=1e-13)


def test_page_permutation_invariance():
    pool, bt, sl, ql, qr, c_rows, r_rows = _small_case()
    pool2, bt2 = _pool_from_rows(oracle.BF16, c_rows, r_rows, list(sl), perm_seed=99)
    assert not np.array_equal(bt, bt2)
    o1, l1, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, sl, synth.SCALE)
    o2, l2, _ = oracle.mla_decode(oracle.BF16, pool2, ql, qr, bt2, sl, synth.SCALE)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_position_order_matters_through_block_table():
    """A wrong page/row index would read another token: swapping two pages' table entries must
    change the result of a request that spans them."""
    pool, bt, sl, ql, qr, _, _ = _small_case(seq_lens=(128,))
    o1, _, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, sl, synth.SCALE)
    bt_sw = bt.copy()
    bt_sw[0, 0], bt_sw[0, 1] = bt[0, 1], bt[0, 0]
    o2, _, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt_sw, sl, synth.SCALE)
    np.testing.assert_allclose(o1, o2, atol=1e-12)      # full pages: a permutation of the set
    sl_short = np.array([100], np.int32)                # partial second page: set changes
    o3, _, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, sl_short, synth.SCALE)
    o4, _, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt_sw, sl_short, synth.SCALE)
    assert np.abs(o3 - o4).max() > 1e-3


def test_topk_all_positions_equals_dense():
    pool, bt, sl, ql, qr, _, _ = _small_case(seq_lens=(70, 128))
    idx = np.full((2, 128), -1, dtype=np.int32)
    idx[0, :70] = np.arange(70)
    idx[1, :] = np.arange(128)
    od, ld, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, sl, synth.SCALE)
    os_, ls, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, sl, synth.SCALE, topk_idx=idx)
    np.testing.assert_allclose(os_, od, atol=1e-13)
    np.testing.assert_allclose(ls, ld, atol=1e-13)


def test_topk_subset_equals_dense_over_compacted_cache():
    """Renormalisation on the picked subset ("DeepSeek's KV Cache", Fig. 10)."""
    pool, bt, sl, ql, qr, c_rows, r_rows = _small_case(seq_lens=(200,))
    pick = np.array([3, 17, 64, 65, 130, 199], dtype=np.int32)
    idx = np.concatenate([pick, [-1, 250, 200]]).astype(np.int32)[None]   # padding skipped
    o_s, l_s, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, sl, synth.SCALE, topk_idx=idx)
    pool_c, bt_c = _pool_from_rows(oracle.BF16, [c_rows[0][pick]], [r_rows[0][pick]], [len(pick)])
    o_c, l_c, _ = oracle.mla_decode(oracle.BF16, pool_c, ql, qr, bt_c,
                                    np.array([len(pick)], np.int32), synth.SCALE)
    np.testing.assert_allclose(o_s, o_c, atol=1e-13)
    np.testing.assert_allclose(l_s, l_c, atol=1e-13)


def test_empty_visible_set():
    pool, bt, sl, ql, qr, _, _ = _small_case(seq_lens=(64,))
    o, l, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, np.array([0], np.int32), synth.SCALE)
    assert np.all(o == 0) and np.all(np.isneginf(l))
    idx = np.full((1, 4), -1, np.int32)
    o, l, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, sl, synth.SCALE, topk_idx=idx)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_sparse_truncation_bound():
    """|o_S - o| <= 2 delta max|v| with delta the omitted dense mass (restricted-support bound,
    "Shared KV Memory", section "What is lost by restricting the support?")."""
    pool, bt, sl, ql, qr, c_rows, _ = _small_case(seq_lens=(256,), H=4)
    pick = np.sort(np.random.default_rng(2).choice(256, 40, replace=False)).astype(np.int32)
    o_d, l_d, pairs = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, sl, synth.SCALE)
    o_s, l_s, _ = oracle.mla_decode(oracle.BF16, pool, ql, qr, bt, sl, synth.SCALE, topk_idx=pick[None])
    vmax = np.linalg.norm(oracle.bf16_to_f64(c_rows[0]), axis=1).max()
    for i in range(len(pairs)):
        delta = 1.0 - math.exp(l_s[i] - l_d[i])      # omitted share of the dense mass
        assert 0.0 <= delta < 1.0
        assert np.linalg.norm(o_s[i] - o_d[i]) <= 2 * delta * vmax + 1e-12


# ------------------------------------------------------------------------------------------
# Split-KV merge
# ------------------------------------------------------------------------------------------

def test_combine_equals_unsplit_for_any_boundaries():
    rng = np.random.default_rng(8)
    n, dk, dv = 301, 20, 12
    q = rng.normal(size=dk)
    K = rng.normal(size=(n, dk))
    V = rng.normal(size=(n, dv))
    full, lfull = oracle.attend(q, K, V, 0.4)
    for cuts in ([0, 301], [0, 1, 301], [0, 64, 65, 200, 301], [0, 150, 150, 301]):
        parts, lses = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            o, l = oracle.attend(q, K[a:b], V[a:b], 0.4)
            parts.append(o)
            lses.append(l)
        o, l = oracle.combine(np.array(parts, np.float32), np.array(lses, np.float32))
        # inputs are rounded to fp32 (the partial format), so compare at fp32 accuracy
        np.testing.assert_allclose(o, full, atol=2e-6)
        assert abs(l - lfull) < 2e-6


def test_combine_single_split_and_all_empty():
    o_in = np.random.default_rng(0).normal(size=(1, 7)).astype(np.float32)
    o, l = oracle.combine(o_in, np.array([1.25], np.float32))
    np.testing.assert_array_equal(o, o_in[0].astype(np.float64))
    assert l == 1.25
    o, l = oracle.combine(np.full((3, 7), np.nan, np.float32), np.full(3, -np.inf, np.float32))
    assert np.all(o == 0) and np.isneginf(l)


# ------------------------------------------------------------------------------------------
# OCP E4M3 codec and the FP8 mixed record ("DeepSeek's KV Cache", "Calculating V3.2's KV cache")
# ------------------------------------------------------------------------------------------

def test_e4m3_known_codes():
    assert oracle.e4m3_decode(0x7E) == 448.0            # largest finite
    assert oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x38) == 1.0              # exponent 7 = bias
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6        # smallest normal
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9        # smallest subnormal
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_decode(0x00) == 0.0
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    vals = [oracle.e4m3_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))    # strictly increasing codes
    assert sum(1 for c in range(256) if math.isnan(oracle.e4m3_decode(c))) == 2   # no infinities


def test_e4m3_encode_round_trip_ties_and_saturation():
    vals = [oracle.e4m3_decode(c) for c in range(0x7F)]
    for c, v in enumerate(vals):
        assert oracle.e4m3_encode(v) == c
        assert oracle.e4m3_encode(-v) == (c | 0x80)
    for c in range(0x7E):
        lo, hi = vals[c], vals[c + 1]
        mid = (lo + hi) / 2                              # exact in fp32 for all E4M3 neighbours
        assert np.float32(mid) == mid
        want = c if c % 2 == 0 else c + 1                # ties to even mantissa
        assert oracle.e4m3_encode(mid) == want
        assert oracle.e4m3_encode(np.nextafter(np.float32(mid), np.float32(0))) == c
        assert oracle.e4m3_encode(np.nextafter(np.float32(mid), np.float32(1e9))) == c + 1
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(463.9) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E               # saturate, never NaN
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00          # half the smallest subnormal: tie to 0
    assert oracle.e4m3_encode(np.float32(2.0 ** -10) * np.float32(1.0000001)) == 0x01


def test_e4m3_error_bounds_random():
    rng = np.random.default_rng(4)
    x = (rng.normal(size=20000) * np.exp(rng.uniform(-12, 6, 20000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    codes = oracle.e4m3_encode_array(x)
    xh = np.array([oracle.e4m3_decode(c) for c in codes])
    normal = np.abs(x) >= 2.0 ** -6
    assert np.all(np.abs(xh[normal] - x[normal]) <= 2.0 ** -4 * np.abs(x[normal]))
    assert np.all(np.abs(xh[~normal] - x[~normal]) <= 2.0 ** -10)


def test_fp8_record_layout_and_scale_rule():
    rng = np.random.default_rng(6)
    T = 5
    c = _bf16(rng.normal(size=(T, 512)) * np.array([1.0, 3.0, 0.01, 100.0]).repeat(128))
    c[4, 128:256] = 0                                    # an all-zero group
    r = _bf16(rng.normal(size=(T, 64)))
    pool = oracle.new_pool(oracle.FP8_MIXED, 1)
    slot = np.array([0, 5, 63, 17, -1], dtype=np.int32)
    assert oracle.cache_append(oracle.FP8_MIXED, pool, c, r, slot) == 0
    rec = pool.reshape(64, 656)
    for i in range(4):
        row = rec[slot[i]]
        xf = synth.bf16_bits_to_f32(c[i])
        for g in range(4):
            grp = xf[g * 128:(g + 1) * 128]
            amax = np.float32(np.abs(grp).max())
            s = np.frombuffer(row[512 + 4 * g:516 + 4 * g].tobytes(), np.float32)[0]
            assert s == np.float32(amax / np.float32(448.0))
            codes = row[g * 128:(g + 1) * 128]
            j = int(np.argmax(np.abs(grp)))
            assert codes[j] in (0x7E, 0xFE)               # absmax element maps to +-448
        assert row[528:656].tobytes() == r[i].tobytes()   # rope kept bit-for-bit in bf16
        cd, krd = oracle.read_record(oracle.FP8_MIXED, pool, int(slot[i]))
        np.testing.assert_array_equal(krd, oracle.bf16_to_f64(r[i]))
        s_all = np.repeat(np.frombuffer(row[512:528].tobytes(), np.float32), 128).astype(np.float64)
        assert np.all(np.abs(cd - xf) <= 2.0 ** -4 * np.abs(xf) + 2.0 ** -10 * s_all + 0.0)
    # the skipped row (slot -1) wrote nothing; the untouched slots stay zero
    touched = set(int(s) for s in slot[:4])
    for sl in range(64):
        if sl not in touched:
            assert not rec[sl].any()


def test_fp8_zero_group_gives_zero_scale_and_codes():
    c = np.zeros((1, 512), np.uint16)
    c[0, 300] = _bf16(np.array([2.5]))[0]
    r = np.zeros((1, 64), np.uint16)
    pool = oracle.new_pool(oracle.FP8_MIXED, 1)
    oracle.cache_append(oracle.FP8_MIXED, pool, c, r, np.array([9], np.int32))
    row = pool.reshape(64, 656)[9]
    scales = np.frombuffer(row[512:528].tobytes(), np.float32)
    assert scales[0] == 0 and scales[1] == 0 and scales[3] == 0
    assert scales[2] == np.float32(np.float32(2.5) / np.float32(448))
    assert not row[:256].any() and not row[384:512].any()
    assert row[300] == 0x7E


def test_append_leaves_other_slots_unchanged():
    """Appending a token does not change earlier cached state ("Shared KV Memory", section 3,
    the proposition that appending a token leaves earlier causal states unchanged)."""
    rng = np.random.default_rng(12)
    for fmt in (oracle.BF16, oracle.FP8_MIXED):
        pool = np.frombuffer(rng.bytes(oracle.new_pool(fmt, 2).size), np.uint8).copy()
        before = pool.copy()
        c = _bf16(rng.normal(size=(2, 512)))
        r = _bf16(rng.normal(size=(2, 64)))
        slot = np.array([70, 3], np.int32)
        oracle.cache_append(fmt, pool, c, r, slot)
        rb = oracle.record_bytes(fmt)
        a = pool.reshape(128, rb)
        b = before.reshape(128, rb)
        for s in range(128):
            if s not in (70, 3):
                assert np.array_equal(a[s], b[s])
            else:
                assert not np.array_equal(a[s], b[s])


def test_append_out_of_pool_slot_is_reported():
    pool = oracle.new_pool(oracle.BF16, 1)
    c = np.zeros((2, 512), np.uint16)
    r = np.zeros((2, 64), np.uint16)
    assert oracle.cache_append(oracle.BF16, pool, c, r, np.array([64, 2], np.int32)) == 1


def test_fp8_decode_through_pool_matches_dequantised_expansion():
    """FP8 path of the wrapper: the decoded latent c = code * scale enters both score and value."""
    pool, bt, sl, ql, qr, c_rows, r_rows = _small_case(fmt=oracle.FP8_MIXED, seq_lens=(90,), H=2)
    out, lse, _ = oracle.mla_decode(oracle.FP8_MIXED, pool, ql, qr, bt, sl, synth.SCALE)
    C = np.empty((90, 512))
    KR = np.empty((90, 64))
    for t in range(90):
        C[t], KR[t] = oracle.read_record(oracle.FP8_MIXED, pool, int(bt[0, t // 64]) * 64 + t % 64)
    np.testing.assert_array_equal(KR, oracle.bf16_to_f64(r_rows[0]))
    assert np.abs(C - oracle.bf16_to_f64(c_rows[0])).max() < 0.07 * np.abs(C).max()
    for h in range(2):
        q = np.concatenate([oracle.bf16_to_f64(ql[0, h]), oracle.bf16_to_f64(qr[0, h])])
        o, l = oracle.attend(q, np.hstack([C, KR]), C, float(np.float32(synth.SCALE)))
        np.testing.assert_allclose(out[h], o, atol=1e-12)
        assert abs(lse[h] - l) < 1e-12


# ------------------------------------------------------------------------------------------
# Input generator (shared by both sides; holds no method arithmetic)
# ------------------------------------------------------------------------------------------

def test_generator_is_deterministic_and_unit_variance():
    a = synth.normal_f32(123, synth.STREAM_KV, 1000, 200000)
    b = synth.normal_f32(123, synth.STREAM_KV, 1000, 200000)
    assert np.array_equal(a, b)
    assert abs(a.mean()) < 0.01 and abs(a.var() - 1.0) < 0.01
    assert a.min() >= -6 and a.max() <= 6
    # counter-based: any window equals the slice of a larger draw
    c = synth.normal_f32(123, synth.STREAM_KV, 1100, 50)
    assert np.array_equal(c, a[100:150])
    bits = synth.normal_bf16(123, synth.STREAM_KV, 0, 1000)
    f = synth.bf16_bits_to_f32(bits)
    assert np.all(np.abs(f - synth.normal_f32(123, synth.STREAM_KV, 0, 1000)) <= 2 ** -8 * 6)


def test_workload_recipes():
    w = synth.make_workload("paged_batch")
    assert w.B == 32 and w.seq_lens.min() >= 1024 and w.seq_lens.max() <= 8192
    pages = w.block_table[w.block_table >= 0]
    assert sorted(pages.tolist()) == list(range(w.num_pages))   # a permutation of the pool
    w5 = synth.make_workload("topk_sparse", B=2, seq_len=4096, topk=256)
    for b in range(2):
        idx = w5.topk_idx[b]
        assert len(set(idx.tolist())) == 256 and np.all(np.diff(idx) > 0)
        assert idx.min() >= 0 and idx.max() < 4096


# ------------------------------------------------------------------------------------------
# DSA lightning indexer and top-k selection: "DeepSeek's KV Cache: From 3.9 MB to 890 B per
# Token", sections "DSA: three things the indexer builds" (Fig. 8), "The score that picks
# positions" (Fig. 9) and "Calculating V3.2's KV cache" (search key, 132 B).
# ------------------------------------------------------------------------------------------

def _bf16_bits(x):
    return synth._bf16_rne(np.asarray(x, dtype=np.float32))


def test_index_page_bytes_closed_form():
    # "Search key, 132 B": 128 FP8 values + one fp32 scale, per token; 64 tokens per page
    assert oracle.index_page_bytes() == 64 * (128 + 4) == 8448


def test_index_score_hand_example():
    # two heads, three dims: head 0's dot is 2 - 2 + 0 = 0 (ReLU keeps 0), head 1's is
    # 0 + 1 + 3 = 4, so I = 0.5 * 0 + 2 * 4 = 8; a key that makes both dots negative scores 0
    q = np.array([[1.0, -2.0, 0.0], [0.0, 1.0, 1.0]])
    w = np.array([0.5, 2.0])
    assert oracle.index_score(q, w, np.array([2.0, 1.0, 3.0])) == 8.0
    assert oracle.index_score(q, w, np.array([-1.0, 1.0, -2.0])) == 0.0
    # a negative head weight counts against the position (the score is not a probability)
    assert oracle.index_score(q, np.array([0.5, -2.0]), np.array([2.0, 1.0, 3.0])) == -8.0


def test_index_score_invariants():
    rng = np.random.default_rng(41)
    q = rng.standard_normal((64, 128))
    k = rng.standard_normal(128)
    w1, w2 = rng.standard_normal(64), rng.standard_normal(64)
    I = lambda qq, ww, kk: oracle.index_score(qq, ww, kk)
    # linear in the head weights
    assert abs(I(q, w1 + w2, k) - (I(q, w1, k) + I(q, w2, k))) < 1e-9
    # positively homogeneous in the query (ReLU commutes with a positive factor)
    assert abs(I(2.5 * q, w1, k) - 2.5 * I(q, w1, k)) < 1e-9
    # ReLU(x) + ReLU(-x) = |x|: the scores of k and -k add up to the weighted absolute dots
    dots = q @ k
    assert abs(I(q, w1, k) + I(q, w1, -k) - float(np.sum(w1 * np.abs(dots)))) < 1e-9


def test_index_append_codec_and_layout():
    rng = np.random.default_rng(42)
    T = 40
    x = rng.standard_normal((T, 128)).astype(np.float32) * rng.uniform(0.01, 30, (T, 1)).astype(np.float32)
    x[3] = 0.0                                   # an all-zero key
    bits = _bf16_bits(x)
    xf = oracle.bf16_to_f64(bits).reshape(T, 128)
    pool = oracle.new_index_pool(2)
    slot = np.arange(T, dtype=np.int32) * 3 % 128  # rows scattered over both pages
    assert oracle.index_append(pool, bits, slot) == 0
    page_bytes = oracle.index_page_bytes()
    for i in range(T):
        k = oracle.index_read(pool, int(slot[i]))
        amax = np.float32(np.max(np.abs(xf[i].astype(np.float32))))
        s = np.float32(amax / np.float32(448.0))
        # the scale sits after the page's 64 x 128 codes, row-major
        pg, row = divmod(int(slot[i]), 64)
        stored = np.frombuffer(pool[pg * page_bytes + 8192 + 4 * row: pg * page_bytes + 8192 + 4 * row + 4].tobytes(),
                               dtype=np.float32)[0]
        assert stored == s
        if amax == 0:
            assert np.all(k == 0.0)
            continue
        j = int(np.argmax(np.abs(xf[i])))
        assert abs(k[j]) == 448.0 * float(s)         # the largest magnitude maps to +-448
        nz = np.abs(xf[i]) >= 2.0 ** -6 * float(s)   # normal E4M3 range
        assert np.all(np.abs(k[nz] - xf[i][nz]) <= 2.0 ** -4 * np.abs(xf[i][nz]) + 1e-30)
        assert np.all(np.abs(k[~nz] - xf[i][~nz]) <= 2.0 ** -10 * float(s) + 1e-30)
    # other rows untouched, an out-of-pool slot reported
    untouched = np.setdiff1d(np.arange(128), slot)
    for t in untouched[:5]:
        assert np.all(oracle.index_read(pool, int(t)) == 0.0)
    assert oracle.index_append(pool, bits[:1], np.array([128], np.int32)) == 1


def test_indexer_scores_through_pages_and_visibility():
    rng = np.random.default_rng(43)
    B, heads, n_pages = 2, 64, 5
    keys = _bf16_bits(rng.standard_normal((n_pages * 64, 128)).astype(np.float32))
    pool = oracle.new_index_pool(n_pages)
    oracle.index_append(pool, keys, np.arange(n_pages * 64, dtype=np.int32))
    q = _bf16_bits(rng.standard_normal((B, heads, 128)).astype(np.float32))
    w = rng.standard_normal((B, heads)).astype(np.float32)
    bt = np.array([[3, 0, 4], [1, 2, -1]], np.int32)
    seq = np.array([150, 70], np.int32)
    sc = oracle.indexer_scores(pool, q, w, bt, seq, ld=192)
    qd = oracle.bf16_to_f64(q).reshape(B, heads, 128)
    for b in range(B):
        for t in (0, 63, 64, int(seq[b]) - 1):
            k = oracle.index_read(pool, int(bt[b, t // 64]) * 64 + t % 64)
            assert sc[b, t] == oracle.index_score(qd[b], w[b].astype(np.float64), k)
        assert np.all(np.isneginf(sc[b, seq[b]:]))
    # permuting the pages together with the block table leaves every score unchanged
    perm = np.array([4, 2, 0, 1, 3])
    pool2 = oracle.new_index_pool(n_pages)
    pb = oracle.index_page_bytes()
    for new, old in enumerate(perm):
        pool2[new * pb:(new + 1) * pb] = pool[old * pb:(old + 1) * pb]
    inv = np.argsort(perm)
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1).astype(np.int32)
    assert np.array_equal(oracle.indexer_scores(pool2, q, w, bt2, seq, ld=192), sc)


def _topk_lexsort(scores, n, K):
    # independent statement of the selection: order by (score descending, position ascending)
    t = np.arange(n)
    order = np.lexsort((t, -scores[:n]))
    pick = np.sort(order[:min(K, n)])
    return np.concatenate([pick, -np.ones(K - pick.size, dtype=np.int64)]).astype(np.int32)


def test_topk_selection():
    rng = np.random.default_rng(44)
    ld = 300
    sc = rng.standard_normal((5, ld))
    sc[1, ::3] = 0.5            # many ties at the cut
    sc[2, :] = 1.0              # all tied: the lowest positions win
    seq = np.array([300, 250, 100, 7, 0], np.int32)
    for K in (1, 16, 64, 120, 300):
        idx = oracle.topk(sc, seq, K)
        for b in range(5):
            ref = _topk_lexsort(sc[b], int(seq[b]), K)
            assert np.array_equal(idx[b], ref), (K, b)
            picks = idx[b][idx[b] >= 0]
            assert np.all(np.diff(picks) > 0) and np.all(picks < seq[b])
            assert picks.size == min(K, int(seq[b]))
    assert np.array_equal(oracle.topk(sc, seq, 64)[2], np.arange(64))


# ------------------------------------------------------------------------------------------
# Value up-projection and output projection ("DeepSeek's KV Cache", section "Computing without
# expanding Key and Value", Fig. 6 (1), (2), (3))
# ------------------------------------------------------------------------------------------

def test_value_project_hand_example():
    """Two heads, dc = 2, dv = 1, D = 2, worked by hand:
    U_0 = [1, 2], U_1 = [3, -1]; W^UV_0 = [[1], [1]], W^UV_1 = [[2], [0]]
      -> Z_0 = 1 + 2 = 3, Z_1 = 6 + 0 = 6;
    W^O_0 = [[1, 0]], W^O_1 = [[0, -1]] -> Y = 3 [1, 0] + 6 [0, -1] = [3, -6].
    Pre-merged: What^O_0 = [[1, 0], [1, 0]], What^O_1 = [[0, -2], [0, 0]]."""
    u = np.array([[[1.0, 2.0], [3.0, -1.0]]])
    w_uv = np.array([[[1.0], [1.0]], [[2.0], [0.0]]])
    w_o = np.array([[1.0, 0.0], [0.0, -1.0]])
    z, y = oracle.value_project(u, w_uv, w_o)
    assert z.reshape(-1).tolist() == [3.0, 6.0]
    assert y.reshape(-1).tolist() == [3.0, -6.0]
    w_hat = oracle.merge_value_output(w_uv, w_o)
    assert w_hat.tolist() == [[[1.0, 0.0], [1.0, 0.0]], [[0.0, -2.0], [0.0, 0.0]]]
    assert oracle.project_merged(u, w_hat).reshape(-1).tolist() == [3.0, -6.0]


def test_value_project_three_orders_agree():
    """Fig. 6: (1) expand V_h = C W^UV_h and weight it by the probabilities, (2) weight the
    latent rows first (U_h) and multiply by W^UV_h and W^O_h, (3) multiply U_h by the pre-merged
    What^O_h -- the same layer output (1e-9 relative in fp64).  (1) goes through the attention
    core with the expanded values; the output weight of each head is its block of rows of W^O."""
    rng = np.random.default_rng(61)
    H, dc, dv, D, n, B = 3, 16, 4, 10, 9, 2
    C = rng.normal(size=(n, dc))
    w_uv = rng.normal(size=(H, dc, dv)) / 4
    w_o = rng.normal(size=(H * dv, D)) / 2
    q = rng.normal(size=(B, H, dc))
    U = np.empty((B, H, dc))
    Zx = np.empty((B, H, dv))
    for b in range(B):
        for h in range(H):
            U[b, h], _ = oracle.attend(q[b, h], C, C, 0.3)
            Zx[b, h], _ = oracle.attend(q[b, h], C, C @ w_uv[h], 0.3)
    Y1 = np.stack([sum(Zx[b, h] @ w_o[h * dv:(h + 1) * dv] for h in range(H)) for b in range(B)])
    z2, Y2 = oracle.value_project(U, w_uv, w_o)
    Y3 = oracle.project_merged(U, oracle.merge_value_output(w_uv, w_o))
    scale = np.abs(Y1).max()
    assert np.abs(z2 - Zx).max() <= 1e-9 * np.abs(Zx).max()
    assert np.abs(Y2 - Y1).max() <= 1e-9 * scale
    assert np.abs(Y3 - Y1).max() <= 1e-9 * scale
    # a head's rows of W^O taken from the wrong block change the result
    w_o_swapped = np.concatenate([w_o[dv:2 * dv], w_o[:dv], w_o[2 * dv:]])
    _, Yw = oracle.value_project(U, w_uv, w_o_swapped)
    assert np.abs(Yw - Y1).max() > 1e-3 * scale


def test_value_project_of_the_worked_example_output():
    """With identity up-projection and output weights, the layer output is the worked example's
    attention output ("What attention stores, and what DeepSeek changed", section "The four
    numbers attention works with": out_3 = [0.610, 1.171, 0.610])."""
    g, d, K, V, q = _worked()
    out, _ = oracle.attend(q, K, V, 1.0 / math.sqrt(d))
    _, y = oracle.value_project(out.reshape(1, 1, d), np.eye(d).reshape(1, d, d), np.eye(d))
    np.testing.assert_allclose(y.reshape(-1), g["out"], atol=6e-4)
