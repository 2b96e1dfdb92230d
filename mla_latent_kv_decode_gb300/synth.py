"""Seeded synthetic inputs for absorbed-MLA decode: the one input recipe both the CUDA path and
the fp64 oracle consume.

This module holds no attention, quantisation or cache-layout arithmetic.  It draws numbers:

* ``u64(seed, stream, i)`` -- a counter-based generator: the splitmix64 output function
  (Steele, Lea & Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014)
  applied to ``key(seed, stream) + (i + 1) * 0x9E3779B97F4A7C15``.
* ``normal`` values -- Irwin-Hall with twelve terms: value i sums the twelve 16-bit fields of
  the three words ``u64(seed, stream, 3i + j)``, j = 0, 1, 2, and maps the integer sum S to
  ``(S - 393210) / 65536``: mean 0, variance (2^32 - 1) / 2^32, support [-6, 6].  Every step is
  integer arithmetic or an exact division by a power of two, so the fp32 value is exact and
  the same on any machine; it is then rounded to bf16 (round to nearest even).
* permutations (argsort of 64-bit keys), uniform integers (modulo) and distinct sorted samples
  (the smallest keys of a random key per candidate).

The same recipe exists as a CUDA kernel (``gpu_normal_bf16``) for inputs too large to draw on
the host; a test checks the two agree bit for bit.

Workloads (one MLA layer each; H = 128 heads, 64-token pages, scale = 1/sqrt(192)):

  tiny_dense    B=1,  4,096 cached tokens, contiguous pages, bf16 cache
  paged_batch   B=32, seq_lens uniform in [1024, 8192], pages in a seeded random permutation
                of a shared pool, bf16 cache
  long_context  B=1,  131,072 tokens in shuffled pages, bf16 cache (split-KV over all SMs)
  fp8_batch     B=64, 32,768 tokens each (32,704 prefilled + 64 appended), FP8 mixed cache
  topk_sparse   B=64, 131,072 tokens each, FP8 mixed cache, 2,048 distinct sorted positions
                per request drawn uniformly from [0, seq_len)

DSA lightning-indexer inputs (64 indexer heads x 128 dims): search keys, queries and head
weights from their own streams (``index_keys``, ``index_queries``, ``index_weights``).
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass, field

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
STREAM_MUL = 0xD1B54A32D192ED03

STREAM_Q = 1
STREAM_KV = 2
STREAM_SEQ = 4
STREAM_PERM = 5
STREAM_TOPK = 6
STREAM_IDX_K = 7          # DSA indexer search keys
STREAM_IDX_Q = 8          # DSA indexer queries
STREAM_IDX_W = 9          # DSA indexer head weights
STREAM_U = 10             # value projection: decode outputs U
STREAM_WUV = 11           # value projection: W^UV
STREAM_WO = 12            # value projection: W^O (or the merged weight)
STREAM_SINK = 13          # shared K = V decode: per-head sinks
STREAM_ANGLE = 14         # shared K = V decode: the query positions' RoPE angles

D_C = 512
D_R = 64
D_K = D_C + D_R
H_DEFAULT = 128
PAGE = 64
KV_ROW_STRIDE = 1 << 20          # index space reserved per request for its token rows
SCALE = float(np.float32(1.0 / math.sqrt(192.0)))

_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def key(seed: int, stream: int) -> int:
    z = np.array([(seed ^ ((stream * STREAM_MUL) & MASK64)) & MASK64], dtype=np.uint64)
    return int(_mix(z)[0])


def u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Words i = start .. start+count-1 of the counter-based generator."""
    k = np.uint64(key(seed, stream))
    i = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(k + i * np.uint64(GOLDEN))


def _bf16_rne(f: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def normal_f32(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Irwin-Hall(12) values i = start .. start+count-1 as exact fp32."""
    w = u64(seed, stream, 3 * start, 3 * count).reshape(count, 3)
    s = np.zeros(count, dtype=np.int64)
    for j in range(3):
        x = w[:, j]
        for f in range(4):
            s += ((x >> np.uint64(16 * f)) & np.uint64(0xFFFF)).astype(np.int64)
    return ((s - 393210).astype(np.float32) / np.float32(65536.0)).astype(np.float32)


def normal_bf16(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """bf16 bit patterns (uint16) of the Irwin-Hall(12) values, rounded to nearest even."""
    return _bf16_rne(normal_f32(seed, stream, start, count))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------------------------
# Structured inputs
# ----------------------------------------------------------------------------------------------

def queries(seed: int, B: int, H: int = H_DEFAULT):
    """q_lat bf16[B,H,512] and q_rope bf16[B,H,64] (bit patterns)."""
    v = normal_bf16(seed, STREAM_Q, 0, B * H * D_K).reshape(B, H, D_K)
    return np.ascontiguousarray(v[:, :, :D_C]), np.ascontiguousarray(v[:, :, D_C:])


def kv_rows(seed: int, b: int, t0: int, t1: int):
    """Latent rows of request b, positions t0..t1-1: c_kv bf16[n,512], k_rope bf16[n,64]."""
    n = t1 - t0
    v = normal_bf16(seed, STREAM_KV, (b * KV_ROW_STRIDE + t0) * D_K, n * D_K).reshape(n, D_K)
    return np.ascontiguousarray(v[:, :D_C]), np.ascontiguousarray(v[:, D_C:])


def kv_rows_at(seed: int, b: int, positions: np.ndarray):
    """Latent rows of request b at arbitrary positions (for sampled parity checks)."""
    positions = np.asarray(positions, dtype=np.int64)
    c = np.empty((positions.size, D_C), dtype=np.uint16)
    r = np.empty((positions.size, D_R), dtype=np.uint16)
    for i, t in enumerate(positions):
        ci, ri = kv_rows(seed, b, int(t), int(t) + 1)
        c[i], r[i] = ci[0], ri[0]
    return c, r


def uniform_int(seed: int, stream: int, count: int, lo: int, hi: int) -> np.ndarray:
    """count integers uniform in [lo, hi] (inclusive), by modulo of the 64-bit words."""
    w = u64(seed, stream, 0, count)
    return (lo + (w % np.uint64(hi - lo + 1)).astype(np.int64)).astype(np.int64)


IDX_HEADS = 64
IDX_DIM = 128


def index_keys(seed: int, b: int, t0: int, t1: int) -> np.ndarray:
    """Search keys of request b, positions t0..t1-1: bf16 bits [n, 128]."""
    n = t1 - t0
    return normal_bf16(seed, STREAM_IDX_K, (b * KV_ROW_STRIDE + t0) * IDX_DIM, n * IDX_DIM).reshape(n, IDX_DIM)


def index_queries(seed: int, B: int) -> np.ndarray:
    """Indexer queries: bf16 bits [B, 64, 128]."""
    return normal_bf16(seed, STREAM_IDX_Q, 0, B * IDX_HEADS * IDX_DIM).reshape(B, IDX_HEADS, IDX_DIM)


def index_weights(seed: int, B: int) -> np.ndarray:
    """Indexer head weights: fp32 [B, 64] (both signs)."""
    return normal_f32(seed, STREAM_IDX_W, 0, B * IDX_HEADS).reshape(B, IDX_HEADS)


@dataclass
class IndexWorkload:
    """DSA lightning-indexer workload: B queries over their own search-key pools."""
    name: str
    B: int
    seed: int
    seq_lens: np.ndarray          # int32[B]
    block_table: np.ndarray       # int32[B, max_pages]
    num_pages: int
    K: int
    description: str = ""

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0

    def slots(self, b: int, t0: int, t1: int) -> np.ndarray:
        t = np.arange(t0, t1, dtype=np.int64)
        return (self.block_table[b, t // PAGE].astype(np.int64) * PAGE + t % PAGE).astype(np.int32)


def make_index_workload(name: str = "indexer_topk", seed: int | None = None, B: int | None = None,
                        seq_len: int | None = None, K: int = 2048) -> IndexWorkload:
    """indexer_topk: B=64 queries, 131,072 cached search keys each (2,048 shuffled pages per
    request, 132 B per key), top-2,048 selection -- the step that produces topk_sparse's lists."""
    seed = 0x4D4C41 + 6 if seed is None else seed
    B = B or 64
    N = seq_len or 131072
    seq = np.full(B, N, dtype=np.int32)
    pages = int(((seq.astype(np.int64) + PAGE - 1) // PAGE).sum())
    bt, total = _block_table(seq, permutation(seed, STREAM_PERM, pages))
    return IndexWorkload(name, B, seed, seq, bt, total, K,
                         f"B={B}, {N} search keys each (FP8, 132 B), 64 indexer heads x 128 dims, top-{K}")


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """A seeded random permutation of 0..n-1 (stable argsort of 64-bit keys)."""
    return np.argsort(u64(seed, stream, 0, n), kind="stable").astype(np.int64)


def sorted_distinct_sample(seed: int, stream: int, b: int, n: int, k: int) -> np.ndarray:
    """k distinct positions of [0, n), uniform without replacement, sorted ascending."""
    keys = u64(seed, stream, b * KV_ROW_STRIDE, n)
    if k >= n:
        return np.arange(n, dtype=np.int32)
    pick = np.argpartition(keys, k - 1)[:k]
    return np.sort(pick).astype(np.int32)


# ----------------------------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    fmt: int                      # 0 = bf16 record (1,152 B), 1 = FP8 mixed record (656 B)
    B: int
    H: int
    seed: int
    seq_lens: np.ndarray          # int32[B]
    block_table: np.ndarray       # int32[B, max_pages]
    num_pages: int
    scale: float = SCALE
    topk_idx: np.ndarray | None = None   # int32[B, topk] or None
    appended: int = 0             # tokens per request written by the timed append
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0

    def slots(self, b: int, t0: int, t1: int) -> np.ndarray:
        t = np.arange(t0, t1, dtype=np.int64)
        return (self.block_table[b, t // PAGE].astype(np.int64) * PAGE + t % PAGE).astype(np.int32)

    def attended(self) -> int:
        """Positions entering the softmax, summed over requests."""
        if self.topk_idx is None:
            return int(self.seq_lens.astype(np.int64).sum())
        n = 0
        for b in range(self.B):
            idx = self.topk_idx[b]
            n += int(((idx >= 0) & (idx < self.seq_lens[b])).sum())
        return n

    def queries(self):
        return queries(self.seed, self.B, self.H)


def _block_table(seq_lens: np.ndarray, perm: np.ndarray | None):
    pages_per = (seq_lens.astype(np.int64) + PAGE - 1) // PAGE
    total = int(pages_per.sum())
    max_pages = int(max(1, pages_per.max()))
    order = perm if perm is not None else np.arange(total, dtype=np.int64)
    bt = np.full((seq_lens.size, max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = order[off:off + n]
        off += n
    return bt, total


def make_workload(name: str, seed: int | None = None, B: int | None = None,
                  seq_len: int | None = None, topk: int | None = None) -> Workload:
    """Build one of the five workloads (optionally shrunk via B / seq_len / topk for tests)."""
    cfg_id = {"tiny_dense": 1, "paged_batch": 2, "long_context": 3, "fp8_batch": 4,
              "topk_sparse": 5}[name]
    if seed is None:
        seed = 0x4D4C41 + cfg_id
    H = H_DEFAULT
    if name == "tiny_dense":
        B = B or 1
        N = seq_len or 4096
        seq = np.full(B, N, dtype=np.int32)
        bt, total = _block_table(seq, None)
        return Workload(name, 0, B, H, seed, seq, bt, total,
                        description=f"B={B}, {N} cached tokens, contiguous 64-token pages, bf16")
    if name == "paged_batch":
        B = B or 32
        hi = seq_len or 8192
        lo = min(1024, hi)
        seq = uniform_int(seed, STREAM_SEQ, B, lo, hi).astype(np.int32)
        pages = int(((seq.astype(np.int64) + PAGE - 1) // PAGE).sum())
        bt, total = _block_table(seq, permutation(seed, STREAM_PERM, pages))
        return Workload(name, 0, B, H, seed, seq, bt, total,
                        description=f"B={B}, seq_lens uniform in [{lo}, {hi}], shuffled shared pool, bf16")
    if name == "long_context":
        B = B or 1
        N = seq_len or 131072
        seq = np.full(B, N, dtype=np.int32)
        pages = B * ((N + PAGE - 1) // PAGE)
        bt, total = _block_table(seq, permutation(seed, STREAM_PERM, pages))
        return Workload(name, 0, B, H, seed, seq, bt, total,
                        description=f"B={B}, {N} tokens in shuffled pages, bf16, split-KV")
    if name == "fp8_batch":
        B = B or 64
        N = seq_len or 32768
        seq = np.full(B, N, dtype=np.int32)
        pages = B * ((N + PAGE - 1) // PAGE)
        bt, total = _block_table(seq, permutation(seed, STREAM_PERM, pages))
        return Workload(name, 1, B, H, seed, seq, bt, total, appended=min(64, N),
                        description=f"B={B}, {N} tokens each ({N - min(64, N)} prefilled + "
                                    f"{min(64, N)} appended), FP8 mixed cache")
    # topk_sparse
    B = B or 64
    N = seq_len or 131072
    K = topk or 2048
    seq = np.full(B, N, dtype=np.int32)
    pages = B * ((N + PAGE - 1) // PAGE)
    bt, total = _block_table(seq, permutation(seed, STREAM_PERM, pages))
    idx = np.stack([sorted_distinct_sample(seed, STREAM_TOPK, b, N, K) for b in range(B)])
    return Workload(name, 1, B, H, seed, seq, bt, total, topk_idx=idx.astype(np.int32),
                    description=f"B={B}, {N} tokens each, FP8 mixed cache, {K} sorted distinct "
                                f"positions per request")


# ----------------------------------------------------------------------------------------------
# GPU twin of the generator (for inputs too large to draw on the host)
# ----------------------------------------------------------------------------------------------

_synth_lib = None


def _load_gpu():
    global _synth_lib
    if _synth_lib is None:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla_synth.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        lib.synth_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_void_p]
        lib.synth_normal_bf16.restype = ctypes.c_int
        _synth_lib = lib
    return _synth_lib


def gpu_normal_bf16(dst_ptr: int, rows: int, seed: int, stream: int, first_index: int,
                    row_len: int, row_stride_index: int, cuda_stream: int = 0) -> None:
    """Fill ``rows`` x ``row_len`` bf16 values on the device: element (r, j) is generator value
    ``first_index + r * row_stride_index + j`` of (seed, stream)."""
    rc = _load_gpu().synth_normal_bf16(ctypes.c_void_p(dst_ptr), rows, key(seed, stream), 0,
                                       first_index, row_len, row_stride_index,
                                       ctypes.c_void_p(cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16 failed with CUDA error {rc}")


# ----------------------------------------------------------------------------------------------
# Shared K = V entries (V4 / V4.1 formats): 512-dim entries, queries, sinks, RoPE angles
# ----------------------------------------------------------------------------------------------
E_DIM = 512


def shared_entries(seed: int, b: int, t0: int, t1: int) -> np.ndarray:
    """Entries of request b, positions t0..t1-1: bf16 bits [n, 512] (unit normal)."""
    n = t1 - t0
    return normal_bf16(seed, STREAM_KV, (b * KV_ROW_STRIDE + t0) * E_DIM, n * E_DIM).reshape(n, E_DIM)


def shared_queries(seed: int, B: int, H: int = H_DEFAULT) -> np.ndarray:
    """Queries bf16 bits [B, H, 512]."""
    return normal_bf16(seed, STREAM_Q, 0, B * H * E_DIM).reshape(B, H, E_DIM)


def sinks(seed: int, H: int = H_DEFAULT) -> np.ndarray:
    """Per-head sink values z' (fp32 [H], unit normal)."""
    return normal_f32(seed, STREAM_SINK, 0, H)


def rope_cos_sin(seed: int, B: int) -> np.ndarray:
    """Per request the cos and sin of 32 angles drawn uniformly in [0, 2 pi): fp32 [B, 64] (cos
    first).  The decode only rotates by the angles it is given, so uniform angles exercise it as
    well as any position's."""
    w = u64(seed, STREAM_ANGLE, 0, B * 32).reshape(B, 32)
    ang = (w >> np.uint64(11)).astype(np.float64) * (2.0 * math.pi / float(1 << 53))
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


@dataclass
class SharedWorkload:
    """B requests over a pool of shared K = V entries (format V4 = 2 or V4.1 = 3)."""
    name: str
    fmt: int
    B: int
    H: int
    seed: int
    seq_lens: np.ndarray
    block_table: np.ndarray
    num_pages: int
    scale: float = float(np.float32(1.0 / math.sqrt(512.0)))
    topk_idx: np.ndarray | None = None
    use_sink: bool = True
    use_rope: bool = True
    description: str = ""

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0

    def slots(self, b: int, t0: int, t1: int) -> np.ndarray:
        t = np.arange(t0, t1, dtype=np.int64)
        return (self.block_table[b, t // PAGE].astype(np.int64) * PAGE + t % PAGE).astype(np.int32)

    def attended(self) -> int:
        if self.topk_idx is None:
            return int(self.seq_lens.astype(np.int64).sum())
        n = 0
        for b in range(self.B):
            idx = self.topk_idx[b]
            n += int(((idx >= 0) & (idx < self.seq_lens[b])).sum())
        return n

    def queries(self):
        return shared_queries(self.seed, self.B, self.H)

    def sink(self):
        return sinks(self.seed, self.H) if self.use_sink else None

    def rope_cs(self):
        return rope_cos_sin(self.seed, self.B) if self.use_rope else None


def make_shared_workload(name: str, fmt: int | None = None, seq_lens=None, seed: int | None = None,
                         topk_idx=None, shuffle: bool = True, use_sink: bool = True,
                         use_rope: bool = True) -> SharedWorkload:
    """v4_batch / v41_batch: B=64 requests of 32,768 entries each (V4 584-B or V4.1 288-B entries),
    shuffled pages, per-head sinks, RoPE rotated back; or a custom batch (seq_lens, top-k lists)."""
    if fmt is None:
        fmt = {"v4_batch": 2, "v41_batch": 3}[name]
    if seed is None:
        seed = 0x4D4C41 + 10 + fmt
    if seq_lens is None:
        seq_lens = np.full(64, 32768, dtype=np.int32)
    seq = np.asarray(seq_lens, dtype=np.int32)
    pages = int(((seq.astype(np.int64) + PAGE - 1) // PAGE).sum())
    perm = permutation(seed, STREAM_PERM, pages) if shuffle else None
    bt, total = _block_table(seq, perm)
    label = "V4 584-B" if fmt == 2 else "V4.1 288-B"
    return SharedWorkload(name, fmt, len(seq), H_DEFAULT, seed, seq, bt, total,
                          topk_idx=None if topk_idx is None else np.asarray(topk_idx, np.int32),
                          use_sink=use_sink, use_rope=use_rope,
                          description=f"B={len(seq)}, {int(seq.max()) if len(seq) else 0} entries max, {label} "
                                      f"shared K = V entries, shuffled pages")
