"""Pins of the shared K = V oracle ("DeepSeek's KV Cache: From 3.9 MB to 890 B per Token",
section "HCA: 128 tokens into one", Fig. 15; the V4 and V4.1 entry formats of "Calculating
V4-Flash's KV cache" and "Calculating V4.1-Flash's KV cache") to facts the pages and the format
definitions fix (CPU only)."""
import math
import os

import numpy as np

import oracle
from mla_latent_kv_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *v = line.split()
                vals[k] = [float(x) for x in v]
    return vals


def _bf16(x):
    return synth._bf16_rne(np.asarray(x, dtype=np.float32))


def test_entry_byte_closed_forms():
    g = {k: int(v[0]) for k, v in _golden("byte_counts.txt").items()}
    assert oracle.shared_record_bytes(oracle.V4_FP8) == g["v4_entry_bytes"] == 448 + 64 * 2 + 7 + 1
    assert oracle.shared_record_bytes(oracle.V41_FP4) == g["v41_entry_bytes"] == 512 // 2 + 512 // 16
    assert g["v4_search_key_bytes"] == 128 // 2 + 128 // 32
    assert (3 * (g["v41_entry_bytes"] + g["v4_search_key_bytes"]) + 2 * (g["v41_entry_bytes"] +
            g["v4_search_key_bytes"])) // 2 == g["v41_bytes_per_token"]
    assert 21 * (g["v4_entry_bytes"] + g["v4_search_key_bytes"]) + 20 * g["v4_entry_bytes"] // 32 == \
        g["v4_flash_bytes_per_token_x4"]
    assert round(g["v4_flash_bytes_per_token_x4"] / 4) == 3514
    # a whole page of each format
    assert oracle.new_shared_pool(oracle.V4_FP8, 1).size == 64 * 584 == 37376
    assert oracle.new_shared_pool(oracle.V41_FP4, 1).size == 64 * 288


def test_e2m1_codec_from_its_definition():
    """OCP MX E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; ties to the even mantissa; saturation."""
    mags = [oracle.e2m1_decode(c) for c in range(8)]
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [oracle.e2m1_decode(c | 8) for c in range(8)] == [-m for m in mags]
    for c in range(16):
        v = oracle.e2m1_decode(c)
        assert oracle.e2m1_decode(oracle.e2m1_encode(v)) == v
    # midpoints go to the code whose mantissa bit is 0
    for x, want in [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0), (5.0, 4.0)]:
        assert oracle.e2m1_decode(oracle.e2m1_encode(x)) == want, x
        assert oracle.e2m1_decode(oracle.e2m1_encode(-x)) == -want, x
    for x, want in [(0.26, 0.5), (0.74, 0.5), (5.01, 6.0), (7.0, 6.0), (1e9, 6.0)]:
        assert oracle.e2m1_decode(oracle.e2m1_encode(x)) == want, x


def test_v4_entry_layout_and_scale_rule():
    """One entry at slot 67 (page 1, row 3).  Group 0 holds powers of two only (exact), group 1 is
    all zero, the RoPE dims are copied; the scale byte is e + 127 for the smallest e with
    448 * 2^e >= amax, so the largest magnitude's code lies in (224, 448]."""
    rng = np.random.default_rng(71)
    x = rng.normal(size=512).astype(np.float32) * 3
    x[0:64] = np.ldexp(1.0, rng.integers(-5, 5, size=64)) * rng.choice([-1, 1], size=64)
    x[64:128] = 0.0
    bits = _bf16(x)
    pool = oracle.new_shared_pool(oracle.V4_FP8, 2)
    assert oracle.shared_append(oracle.V4_FP8, pool, bits[None], np.array([67], np.int32)) == 0
    page = pool[37376:2 * 37376]
    codes = page[3 * 448:4 * 448]
    rope = page[64 * 448 + 3 * 128:64 * 448 + 4 * 128]
    scales = page[64 * 576 + 3 * 8:64 * 576 + 4 * 8]
    assert np.array_equal(rope.view(np.uint16), bits[448:])
    assert scales[1] == 0 and np.all(codes[64:128] == 0) and scales[7] == 0
    xv = synth.bf16_bits_to_f32(bits).astype(np.float64)
    for g in (0, 2, 3, 4, 5, 6):
        amax = np.abs(xv[64 * g:64 * g + 64]).max()
        e = int(scales[g]) - 127
        assert 448 * 2.0 ** e >= amax > 448 * 2.0 ** (e - 1)
    e = oracle.shared_read(oracle.V4_FP8, pool, 67)
    assert np.array_equal(e[:64], xv[:64])                       # powers of two survive exactly
    assert np.all(e[64:128] == 0)
    assert np.array_equal(e[448:], xv[448:])                     # RoPE dims stay bf16
    nz = np.abs(xv[128:448]) >= 2.0 ** -6 * np.abs(xv[128:448]).max()
    assert np.all(np.abs(e[128:448] - xv[128:448])[nz] <= 2.0 ** -4 * np.abs(xv[128:448])[nz])
    # no other byte of the pool was written
    touched = np.zeros(pool.size, bool)
    touched[37376 + 3 * 448:37376 + 4 * 448] = True
    touched[37376 + 64 * 448 + 3 * 128:37376 + 64 * 448 + 4 * 128] = True
    touched[37376 + 64 * 576 + 3 * 8:37376 + 64 * 576 + 4 * 8] = True
    assert np.all(pool[~touched] == 0)


def test_v41_entry_layout_and_scale_rule():
    """One entry at slot 5: byte i holds dims 2i (low nibble) and 2i + 1 (high nibble); scale g is
    E4M3(amax_g / 6).  A group whose values are E2M1 magnitudes times 2^k round-trips exactly."""
    rng = np.random.default_rng(72)
    x = rng.normal(size=512).astype(np.float32)
    grid = np.array([0.5, 1, 1.5, 2, 3, 4, 6])
    x[0:16] = rng.choice(grid, size=16) * rng.choice([-1, 1], size=16) * 0.25
    x[0] = 6 * 0.25                                              # amax / 6 = 0.25 exactly
    x[16:32] = 0.0
    bits = _bf16(x)
    pool = oracle.new_shared_pool(oracle.V41_FP4, 1)
    assert oracle.shared_append(oracle.V41_FP4, pool, bits[None], np.array([5], np.int32)) == 0
    rec = pool[5 * 288:6 * 288]
    assert oracle.e4m3_decode(int(rec[256])) == 0.25 and rec[257] == 0
    e = oracle.shared_read(oracle.V41_FP4, pool, 5)
    xv = synth.bf16_bits_to_f32(bits).astype(np.float64)
    assert np.array_equal(e[:16], xv[:16]) and np.all(e[16:32] == 0)
    lo, hi = rec[0] & 0xF, rec[0] >> 4
    assert oracle.e2m1_decode(lo) * 0.25 == xv[0] and oracle.e2m1_decode(hi) * 0.25 == xv[1]
    for g in range(2, 32):
        s = oracle.e4m3_decode(int(rec[256 + g]))
        amax = np.abs(xv[16 * g:16 * g + 16]).max()
        assert s == oracle.e4m3_decode(oracle.e4m3_encode(np.float32(amax) / np.float32(6)))
        # every element within half an E2M1 step of its code, or saturated at 6 s
        err = np.abs(e[16 * g:16 * g + 16] - xv[16 * g:16 * g + 16])
        assert np.all(err <= 1.0 * s + 1e-12)
    assert np.all(pool[:5 * 288] == 0) and np.all(pool[6 * 288:] == 0)


def test_sink_softmax_closed_forms():
    """Fig. 15 (2): exp(z') joins the denominator.  No sink (-inf) is plain attention (the worked
    example of "What attention stores, and what DeepSeek changed", section "The four numbers
    attention works with"); one entry: out = v e^s / (e^s + e^z'), lse = ln(e^s + e^z'); the
    weights sum to 1 - e^(z' - lse); nothing visible: out = 0, lse = z'."""
    g = _golden("worked_example.txt")
    K = np.array(g["K_flat"]).reshape(3, 3).T
    V = np.array(g["V_flat"]).reshape(3, 3).T
    q = np.array(g["q3"])
    out, lse = oracle.attend_sink(q, K, V, 1 / math.sqrt(3))
    np.testing.assert_allclose(out, g["out"], atol=6e-4)
    ref, ref_lse = oracle.attend(q, K, V, 1 / math.sqrt(3))
    assert np.abs(out - ref).max() < 1e-15 and abs(lse - ref_lse) < 1e-15
    z = 2.0
    w, lse_z = oracle.attend_sink(q, K, np.eye(3), 1 / math.sqrt(3), z)
    assert abs(lse_z - math.log(math.exp(ref_lse) + math.exp(z))) < 1e-12
    assert abs(w.sum() - (1 - math.exp(z - lse_z))) < 1e-14
    np.testing.assert_allclose(w, np.array(g["weights"]) * math.exp(ref_lse - lse_z), atol=6e-4)
    k1 = np.array([[0.5, -1.0]])
    v1 = np.array([[3.0, 4.0]])
    o1, l1 = oracle.attend_sink(np.array([2.0, 1.0]), k1, v1, 1.0, 0.3)
    s = 2 * 0.5 - 1.0
    assert abs(l1 - math.log(math.exp(s) + math.exp(0.3))) < 1e-14
    np.testing.assert_allclose(o1, v1[0] * math.exp(s) / (math.exp(s) + math.exp(0.3)), rtol=1e-14)
    o0, l0 = oracle.attend_sink(np.array([2.0, 1.0]), np.zeros((0, 2)), np.zeros((0, 2)), 1.0, 0.3)
    assert np.all(o0 == 0) and l0 == 0.3


def _rot_cs(theta):
    return np.concatenate([np.cos(theta), np.sin(theta)]).astype(np.float32)


def test_inverse_rotation_gives_relative_position():
    """Fig. 15 (3): an entry stored at position s carries its RoPE dims rotated by s; rotating the
    output back by the query position t leaves that entry's contribution rotated by s - t (the
    relative distance).  Checked for one entry (its output is the entry itself) against a rotation
    by the angle difference computed directly."""
    rng = np.random.default_rng(73)
    freqs = 10000.0 ** (-np.arange(32) / 32.0)
    k = rng.normal(size=64)
    s_pos, t_pos = 37, 1000
    def rotate(v, ang):
        out = v.copy()
        c, sn = np.cos(ang), np.sin(ang)
        out[0::2] = v[0::2] * c - v[1::2] * sn
        out[1::2] = v[0::2] * sn + v[1::2] * c
        return out
    # the stored entry: its rope dims rotated by s (fp32 angles, as a caller passes them)
    ang_s = (np.float32(s_pos) * freqs.astype(np.float32)).astype(np.float64)
    ang_t = (np.float32(t_pos) * freqs.astype(np.float32)).astype(np.float64)
    e = np.concatenate([rng.normal(size=448), rotate(k, ang_s)])
    out, _ = oracle.attend_sink(rng.normal(size=512), e[None], e[None], 0.05)
    assert np.abs(out - e).max() < 1e-14
    back = oracle.unrotate(out, _rot_cs(ang_t))
    cs = _rot_cs(ang_t).astype(np.float64)
    want = rotate(k, ang_s - np.arctan2(cs[32:], cs[:32]))
    assert np.abs(back[448:] - want).max() < 1e-6
    assert np.array_equal(back[:448], out[:448])
    # rotating back by the entry's own position restores the unrotated key
    assert np.abs(oracle.unrotate(out, _rot_cs(ang_s))[448:] - k).max() < 1e-6


def _exact_v4_entries(rng, n):
    """Entries the V4 format holds exactly: per 64-dim group, E4M3 values times a power of two whose
    largest magnitude is a code in (224, 448]; bf16 RoPE dims."""
    x = np.empty((n, 512), np.float32)
    codes = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    for i in range(n):
        for g in range(7):
            v = rng.choice(codes, size=64) * rng.choice([-1, 1], size=64)
            v[rng.integers(64)] = 448.0 * rng.choice([-1, 1])
            x[i, 64 * g:64 * g + 64] = v * 2.0 ** int(rng.integers(-12, -4))
        x[i, 448:] = rng.normal(size=64)
    return _bf16(x)


def _exact_v41_entries(rng, n):
    grid = np.array([0.0, 0.5, 1, 1.5, 2, 3, 4, 6])
    x = np.empty((n, 512), np.float32)
    for i in range(n):
        for g in range(32):
            v = rng.choice(grid, size=16) * rng.choice([-1, 1], size=16)
            v[rng.integers(16)] = 6.0
            x[i, 16 * g:16 * g + 16] = v * 2.0 ** int(rng.integers(-6, 0))
    return _bf16(x)


def test_shared_kv_decode_equals_attention_over_the_entries():
    """Entries the formats hold exactly, written through shuffled pages: the decode equals the sink
    attention over the original bf16 values with K = V = E (then rotated back), for every pair;
    a top-k list of every position equals the dense decode; permuting the pages changes nothing."""
    rng = np.random.default_rng(74)
    for fmt, gen in ((oracle.V4_FP8, _exact_v4_entries), (oracle.V41_FP4, _exact_v41_entries)):
        seq = np.array([70, 1, 0, 130], np.int32)
        pages = int(((seq + 63) // 64).sum())
        perm = rng.permutation(pages)
        bt = np.full((4, 3), -1, np.int32)
        off = 0
        for b, n in enumerate(seq):
            k = (n + 63) // 64
            bt[b, :k] = perm[off:off + k]
            off += k
        pool = oracle.new_shared_pool(fmt, pages)
        entries = {}
        for b, n in enumerate(seq):
            if n:
                ent = gen(rng, int(n))
                t = np.arange(n)
                slot = (bt[b, t // 64].astype(np.int64) * 64 + t % 64).astype(np.int32)
                assert oracle.shared_append(fmt, pool, ent, slot) == 0
                entries[b] = synth.bf16_bits_to_f32(ent).astype(np.float64)
        H = 4
        q = _bf16(rng.normal(size=(4, H, 512)).astype(np.float32))
        sink = rng.normal(size=H).astype(np.float32)
        cs = np.stack([_rot_cs(rng.uniform(0, 6, size=32)) for _ in range(4)])
        scale = 1 / math.sqrt(512)
        out, lse = oracle.shared_kv_decode(fmt, pool, q, bt, seq, scale, sink=sink, rope_cs=cs)
        qd = synth.bf16_bits_to_f32(q).astype(np.float64)
        for b in range(4):
            for h in range(H):
                E = entries.get(b, np.zeros((0, 512)))
                o, l = oracle.attend_sink(qd[b, h], E, E, float(np.float32(scale)), float(sink[h]))
                o = oracle.unrotate(o, cs[b])
                i = b * H + h
                assert np.abs(out[i] - o).max() < 1e-12 and abs(lse[i] - l) < 1e-12
        # top-k of every position == dense; another page permutation == the same
        tk = np.full((4, 200), -1, np.int32)
        for b, n in enumerate(seq):
            tk[b, :n] = np.arange(n)
        out_k, lse_k = oracle.shared_kv_decode(fmt, pool, q, bt, seq, scale, sink=sink, rope_cs=cs, topk_idx=tk)
        assert np.abs(out_k - out).max() < 1e-12 and np.abs(lse_k - lse).max() < 1e-12
        # empty request: zeros and lse = z'
        assert np.all(out[2 * H:3 * H] == 0) and np.allclose(lse[2 * H:3 * H], sink)
