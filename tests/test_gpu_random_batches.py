"""Seeded random batches through every decode path, each compared in full with the fp64 oracle.

A case draws one batch for one record format (bf16 or FP8 mixed records of "DeepSeek's KV Cache:
From 3.9 MB to 890 B per Token", section "Calculating V3.2's KV cache"; V4 584-B or V4.1 288-B
shared K = V entries of its sections "Calculating V4-Flash's KV cache" and "Calculating
V4.1-Flash's KV cache") over a shuffled pool:
  * dense: 1-20 requests whose lengths mix the edges the kernels treat apart (empty, one
    position, the page edges 63/64/65 and 127/128/129, 4095/4096/4097) with lengths of 32 to
    6,000;
  * top-k: the same kind of batch with lists (Fig. 10) of a length that is not a multiple of the
    64-entry tile, holding -1 padding, entries at or past the request's length, unsorted and
    repeated entries (each listed entry counts once, as the oracle takes them);
  * long: two to four requests of 8,000 to 24,000 positions (one of them sometimes empty), cut
    across many clusters and merged.
Every cache byte, output and log-sum-exp is compared (the bar of parity_util).

Every request sees no position, one position (its output is that row, exactly) or at least 32,
at the workloads' softmax scale, so the weight spreads over many rows.  Where it sits on two or
three positions, the bf16 rounding of P (2^-9 of a weight) moves the output by up to about
2^-10 of the rows' difference, which on top of the output's own rounding can pass 1e-2 (mla_decode's
arithmetic in include/mla.h states that bound); this test does not cover that case.
"""
import numpy as np
import pytest

import mla_latent_kv_decode_gb300 as mla
from mla_latent_kv_decode_gb300 import synth
from parity_util import custom_workload, run_full_compare, run_shared_compare

pytestmark = pytest.mark.gpu

EDGES = [0, 1, 63, 64, 65, 127, 128, 129, 4095, 4096, 4097]
KINDS = ["dense", "topk", "long"]
CASES = [(kind, fmt) for kind in KINDS for fmt in (0, 1, 2, 3)]


@pytest.fixture(scope="module")
def torch():
    import torch as t
    mla.load()
    t.cuda.init()
    return t


def _lengths(rng, kind):
    if kind == "long":
        seq = rng.integers(8000, 24001, size=int(rng.integers(2, 5)))
        if rng.random() < 0.5:
            seq[int(rng.integers(0, seq.size))] = 0
        return seq.astype(np.int32)
    B = int(rng.integers(1, 21))
    seq = rng.integers(32, 6001, size=B)
    edge = rng.random(B) < 0.4
    seq[edge] = rng.choice(EDGES, size=int(edge.sum()))
    return seq.astype(np.int32)


def _topk_lists(rng, seq):
    """Per request a visible set of no position, one position (listed up to four times) or at
    least 32 distinct positions, some of them listed again; the rest of the row is -1, at or past
    the request's length, or the largest int32, and the row is shuffled."""
    K = int(rng.choice([1, 37, 64, 200, 513]))
    idx = np.empty((seq.size, K), dtype=np.int32)
    for b, n in enumerate(seq):
        n = int(n)
        mode = rng.random()
        if n == 0 or mode < 0.15:
            inside = np.empty(0, dtype=np.int64)
        elif n == 1 or K < 32 or mode < 0.3:
            inside = np.full(int(rng.integers(1, min(K, 4) + 1)), int(rng.integers(0, n)), dtype=np.int64)
        else:
            nd = int(rng.integers(32, min(n, K) + 1))
            inside = rng.choice(n, size=nd, replace=False).astype(np.int64)
            inside = np.concatenate([inside, rng.choice(inside, size=int(rng.integers(0, K - nd + 1)) // 4)])
        rest = K - inside.size
        kind = rng.integers(0, 3, size=rest)
        outside = np.where(kind == 0, -1, np.where(kind == 1, n + rng.integers(0, 100, size=rest),
                                                   np.iinfo(np.int32).max))
        row = np.concatenate([inside, outside]).astype(np.int64)
        rng.shuffle(row)
        idx[b] = row.astype(np.int32)
    return idx


@pytest.mark.parametrize("kind,fmt", CASES, ids=[f"{k}-fmt{f}" for k, f in CASES])
def test_random_batch_matches_oracle(torch, kind, fmt):
    seed = 0x5EED00 + 16 * KINDS.index(kind) + fmt
    rng = np.random.default_rng(seed)
    seq = _lengths(rng, kind)
    idx = _topk_lists(rng, seq) if kind == "topk" else None
    what = f"random {kind} fmt={fmt} B={seq.size} lens={seq.tolist()[:8]}"
    if fmt in (0, 1):
        # the workloads' softmax scale: a steeper one can put almost all the weight on one latent
        # row, and an output of magnitude 4 or more then rounds to bf16 with an error of up to
        # 2^-6, above the 1e-2 bar whatever the kernel does (the growth tests steepen the softmax
        # so far that the output is one stored row, which bf16 holds exactly)
        run_full_compare(custom_workload(f"rand_{kind}{fmt}", fmt, seq, seed, topk_idx=idx), what)
    else:
        use_sink = bool(rng.random() < 0.75)
        w = synth.make_shared_workload(f"rand_{kind}{fmt}", fmt=fmt, seq_lens=seq, seed=seed, topk_idx=idx,
                                       use_sink=use_sink, use_rope=bool(rng.random() < 0.75))
        run_shared_compare(w, what)
