"""fp64 CPU oracle for absorbed MLA decode over a paged latent cache.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / ``--impl reference`` legs are the only callers.  The product package never
imports this module, and this module imports nothing from the product package.

The arithmetic lives in ``mla_oracle.c`` (plain C, fp64, optional OpenMP over heads); this file
only compiles it with gcc and marshals numpy arrays through ctypes.  Each function cites the
web-page passage it follows; see the C source for the definitions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
FP8_MIXED = 1
D_C = 512
D_R = 64
D_K = D_C + D_R
PAGE = 64


def build(force: bool = False) -> str:
    """Compile ``mla_oracle.c`` into ``liboracle.so`` next to it (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = f64
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = f64
            lib.oracle_e4m3_encode.argtypes = [f32]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode_array.argtypes = [P, P, i64, ctypes.c_int]
            lib.oracle_e4m3_encode_array.restype = None
            lib.oracle_attend.argtypes = [P, P, i64, P, i64, i64, ctypes.c_int, ctypes.c_int, f64, P, P, P]
            lib.oracle_attend.restype = None
            lib.oracle_record_bytes.argtypes = [ctypes.c_int]
            lib.oracle_record_bytes.restype = i64
            lib.oracle_cache_append.argtypes = [ctypes.c_int, P, i64, P, P, P, i64, ctypes.c_int]
            lib.oracle_cache_append.restype = i64
            lib.oracle_read_record.argtypes = [ctypes.c_int, P, i64, P, P]
            lib.oracle_read_record.restype = None
            lib.oracle_mla_decode.argtypes = [ctypes.c_int, P, i64, P, P, P, i32, P, P, i32, i32, i32,
                                              f32, P, i64, P, P, ctypes.c_int]
            lib.oracle_mla_decode.restype = ctypes.c_int
            lib.oracle_combine.argtypes = [P, P, i32, i64, P, P]
            lib.oracle_combine.restype = None
            lib.oracle_index_page_bytes.argtypes = []
            lib.oracle_index_page_bytes.restype = i64
            lib.oracle_index_append.argtypes = [P, i64, P, P, i64]
            lib.oracle_index_append.restype = i64
            lib.oracle_index_read.argtypes = [P, i64, P]
            lib.oracle_index_read.restype = None
            lib.oracle_index_score.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int]
            lib.oracle_index_score.restype = f64
            lib.oracle_indexer_scores.argtypes = [P, i64, P, P, ctypes.c_int, P, i32, P, i32, i64, P,
                                                  ctypes.c_int]
            lib.oracle_indexer_scores.restype = ctypes.c_int
            lib.oracle_topk.argtypes = [P, i64, P, i32, i32, P, ctypes.c_int]
            lib.oracle_topk.restype = None
            lib.oracle_value_project.argtypes = [P, P, P] + [ctypes.c_int] * 5 + [P, P, ctypes.c_int]
            lib.oracle_value_project.restype = None
            lib.oracle_merge_value_output.argtypes = [P, P] + [ctypes.c_int] * 4 + [P, ctypes.c_int]
            lib.oracle_merge_value_output.restype = None
            lib.oracle_project_merged.argtypes = [P, P] + [ctypes.c_int] * 4 + [P, ctypes.c_int]
            lib.oracle_project_merged.restype = None
            lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_decode.restype = f64
            lib.oracle_e2m1_encode.argtypes = [f32]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint8
            lib.oracle_shared_record_bytes.argtypes = [ctypes.c_int]
            lib.oracle_shared_record_bytes.restype = i64
            lib.oracle_shared_append.argtypes = [ctypes.c_int, P, i64, P, P, i64]
            lib.oracle_shared_append.restype = i64
            lib.oracle_shared_read.argtypes = [ctypes.c_int, P, i64, P]
            lib.oracle_shared_read.restype = None
            lib.oracle_attend_sink.argtypes = [P, P, i64, P, i64, i64, ctypes.c_int, ctypes.c_int, f64, f64, P, P]
            lib.oracle_attend_sink.restype = None
            lib.oracle_unrotate.argtypes = [P, P]
            lib.oracle_unrotate.restype = None
            lib.oracle_shared_kv_decode.argtypes = [ctypes.c_int, P, i64, P, P, i32, P, P, i32, i32, i32, f32, P, P,
                                                    P, i64, P, P, ctypes.c_int]
            lib.oracle_shared_kv_decode.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_decode(code: int) -> float:
    """OCP OFP8 E4M3 value of one code (exact)."""
    return float(_load().oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    """OCP OFP8 E4M3 round-to-nearest-even, saturating at +-448, of one fp32 value."""
    return int(_load().oracle_e4m3_encode(float(np.float32(x))))


def e4m3_encode_array(x: np.ndarray, nthreads: int = 0) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(x), _ptr(out), x.size, nthreads)
    return out


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, return_scores: bool = False):
    """Scaled dot-product attention of one query (fp64): returns (out[dv], lse[, scores[n]]).

    s_t = scale * q.K_t ; lse = ln sum exp(s_t) ; out = sum exp(s_t - lse) V_t
    ("What attention stores, and what DeepSeek changed", section "The four numbers attention
    works with").
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    n, dk = K.shape
    nv, dv = V.shape
    assert nv == n and q.shape == (dk,)
    out = np.empty(dv, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    s = np.empty(max(n, 1), dtype=np.float64)
    _load().oracle_attend(_ptr(q), _ptr(K), dk, _ptr(V), dv, n, dk, dv, float(scale),
                          _ptr(out), _ptr(lse), _ptr(s))
    if return_scores:
        return out, float(lse[0]), s[:n]
    return out, float(lse[0])


def record_bytes(fmt: int) -> int:
    return int(_load().oracle_record_bytes(int(fmt)))


def new_pool(fmt: int, num_pages: int) -> np.ndarray:
    """A zero-filled host pool of ``num_pages`` 64-token pages (uint8)."""
    return np.zeros(num_pages * PAGE * record_bytes(fmt), dtype=np.uint8)


def cache_append(fmt: int, pool: np.ndarray, c_kv: np.ndarray, k_rope: np.ndarray,
                 slot: np.ndarray, nthreads: int = 0) -> int:
    """Write T tokens (bf16 bits c_kv[T,512], k_rope[T,64]) into ``pool`` at ``slot``.

    Returns the number of rows whose slot lies outside the pool (not written).  Large appends
    whose non-negative slots are all distinct are spread over ``nthreads`` threads (all host
    threads for 0); otherwise rows are written one after another, in order.
    """
    c_kv = np.ascontiguousarray(c_kv, dtype=np.uint16)
    k_rope = np.ascontiguousarray(k_rope, dtype=np.uint16)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    T = slot.shape[0]
    assert c_kv.shape == (T, D_C) and k_rope.shape == (T, D_R)
    num_pages = pool.size // (PAGE * record_bytes(fmt))
    nth = 1
    if T >= 4096:
        live = slot[slot >= 0]
        if np.unique(live).size == live.size:
            nth = nthreads if nthreads > 0 else max_threads()
    return int(_load().oracle_cache_append(fmt, _ptr(pool), num_pages, _ptr(c_kv), _ptr(k_rope),
                                           _ptr(slot), T, nth))


def read_record(fmt: int, pool: np.ndarray, slot: int):
    """(c[512], k_rope[64]) of one cached token as exact doubles."""
    c = np.empty(D_C, dtype=np.float64)
    kr = np.empty(D_R, dtype=np.float64)
    _load().oracle_read_record(fmt, _ptr(pool), int(slot), _ptr(c), _ptr(kr))
    return c, kr


def mla_decode(fmt: int, pool: np.ndarray, q_lat: np.ndarray, q_rope: np.ndarray,
               block_table: np.ndarray, seq_lens: np.ndarray, scale: float,
               topk_idx: np.ndarray | None = None, pairs=None, nthreads: int = 0):
    """Absorbed MLA decode in fp64 for the (b, h) pairs given (all pairs by default).

    q_lat: bf16 bits [B,H,512]; q_rope: bf16 bits [B,H,64]; block_table int32 [B,max_pages];
    seq_lens int32 [B]; topk_idx int32 [B,topk] or None.
    Returns (out float64[n_pairs,512], lse float64[n_pairs], pairs int32[n_pairs,2]).
    """
    q_lat = np.ascontiguousarray(q_lat, dtype=np.uint16)
    q_rope = np.ascontiguousarray(q_rope, dtype=np.uint16)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, H, _ = q_lat.shape
    if pairs is None:
        pairs = np.stack(np.meshgrid(np.arange(B), np.arange(H), indexing="ij"), -1).reshape(-1, 2)
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    order = np.argsort(pairs[:, 0], kind="stable")
    sp = np.ascontiguousarray(pairs[order])
    n = sp.shape[0]
    out = np.empty((n, D_C), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    topk = 0
    if topk_idx is not None:
        topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
        topk = topk_idx.shape[1]
    num_pages = pool.size // (PAGE * record_bytes(fmt))
    rc = _load().oracle_mla_decode(fmt, _ptr(pool), num_pages, _ptr(q_lat), _ptr(q_rope),
                                   _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                   _ptr(topk_idx), topk, B, H, float(np.float32(scale)),
                                   _ptr(sp), n, _ptr(out), _ptr(lse), nthreads)
    if rc != 0:
        raise ValueError("oracle_mla_decode: a visible position maps outside the pool")
    res_out = np.empty_like(out)
    res_lse = np.empty_like(lse)
    res_out[order] = out
    res_lse[order] = lse
    return res_out, res_lse, pairs


def combine(o_part: np.ndarray, lse_part: np.ndarray):
    """Merge split-KV partials: o_part float32[S,D], lse_part float32[S] -> (out[D], lse)."""
    o_part = np.ascontiguousarray(o_part, dtype=np.float32)
    lse_part = np.ascontiguousarray(lse_part, dtype=np.float32)
    S, D = o_part.shape
    out = np.empty(D, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    _load().oracle_combine(_ptr(o_part), _ptr(lse_part), S, D, _ptr(out), _ptr(lse))
    return out, float(lse[0])


# ------------------------------------------------------------------------------------------
# DSA lightning indexer and top-k selection ("DeepSeek's KV Cache: From 3.9 MB to 890 B per
# Token", "DSA: three things the indexer builds" (Fig. 8), "The score that picks positions"
# (Fig. 9), "Calculating V3.2's KV cache" (search key, 132 B)).
# ------------------------------------------------------------------------------------------
IDX_DIM = 128
IDX_HEADS = 64


def index_page_bytes() -> int:
    """Bytes of one 64-token page of the index-key pool (64 x (128 codes + 4-byte scale))."""
    return int(_load().oracle_index_page_bytes())


def new_index_pool(num_pages: int) -> np.ndarray:
    return np.zeros(num_pages * index_page_bytes(), dtype=np.uint8)


def index_append(pool: np.ndarray, k: np.ndarray, slot: np.ndarray) -> int:
    """Quantise T search keys (bf16 bits k[T,128]) into ``pool`` at ``slot``; returns the number of
    rows whose slot lies outside the pool."""
    k = np.ascontiguousarray(k, dtype=np.uint16)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    T = slot.shape[0]
    assert k.shape == (T, IDX_DIM)
    num_pages = pool.size // index_page_bytes()
    return int(_load().oracle_index_append(_ptr(pool), num_pages, _ptr(k), _ptr(slot), T))


def index_read(pool: np.ndarray, slot: int) -> np.ndarray:
    """The search key of one cached token, exact doubles [128]."""
    k = np.empty(IDX_DIM, dtype=np.float64)
    _load().oracle_index_read(_ptr(pool), int(slot), _ptr(k))
    return k


def index_score(q: np.ndarray, w: np.ndarray, k: np.ndarray) -> float:
    """sum_j w[j] ReLU(q[j] . k) for one query q[heads, dim] (fp64) and one key k[dim]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    heads, dim = q.shape
    assert w.shape == (heads,) and k.shape == (dim,)
    return float(_load().oracle_index_score(_ptr(q), _ptr(w), _ptr(k), heads, dim))


def indexer_scores(pool: np.ndarray, q: np.ndarray, w: np.ndarray, block_table: np.ndarray,
                   seq_lens: np.ndarray, ld: int, nthreads: int = 0) -> np.ndarray:
    """Scores float64[B, ld] of each request's query (bf16 bits q[B,heads,128], fp32 w[B,heads])
    at every visible position; -inf from seq_lens[b] on."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, heads, dim = q.shape
    assert dim == IDX_DIM and w.shape == (B, heads)
    out = np.empty((B, ld), dtype=np.float64)
    num_pages = pool.size // index_page_bytes()
    rc = _load().oracle_indexer_scores(_ptr(pool), num_pages, _ptr(q), _ptr(w), heads, _ptr(block_table),
                                       block_table.shape[1], _ptr(seq_lens), B, ld, _ptr(out), nthreads)
    if rc != 0:
        raise ValueError("oracle_indexer_scores: a visible position maps outside the pool")
    return out


def topk(scores: np.ndarray, seq_lens: np.ndarray, K: int, nthreads: int = 0) -> np.ndarray:
    """int32[B, K]: per row, the K highest scores among positions < seq_lens[b] (a tie goes to the
    lower position), in increasing position order, -1 past the picks."""
    scores = np.ascontiguousarray(scores, dtype=np.float64)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, ld = scores.shape
    idx = np.empty((B, K), dtype=np.int32)
    _load().oracle_topk(_ptr(scores), ld, _ptr(seq_lens), B, K, _ptr(idx), nthreads)
    return idx


# ------------------------------------------------------------------------------------------
# Value up-projection and output projection ("DeepSeek's KV Cache: From 3.9 MB to 890 B per
# Token", section "Computing without expanding Key and Value", Fig. 6 (2) and (3)).
# ------------------------------------------------------------------------------------------

def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def value_project(u: np.ndarray, w_uv: np.ndarray, w_o: np.ndarray, nthreads: int = 0):
    """Fig. 6 (2): Z_h = U_h W^UV_h and Y = sum_h Z_h W^O_h, in fp64.

    u [B,H,dc], w_uv [H,dc,dv] (W^UV_h: dc rows, dv columns), w_o [H*dv, D] (W^O; rows h*dv ..
    h*dv + dv - 1 are W^O_h).  Returns (z [B,H,dv], y [B,D])."""
    u, w_uv, w_o = _f64(u), _f64(w_uv), _f64(w_o)
    B, H, dc = u.shape
    dv = w_uv.shape[2]
    D = w_o.shape[1]
    assert w_uv.shape == (H, dc, dv) and w_o.shape == (H * dv, D)
    z = np.empty((B, H, dv))
    y = np.empty((B, D))
    _load().oracle_value_project(_ptr(u), _ptr(w_uv), _ptr(w_o), B, H, dc, dv, D, _ptr(z), _ptr(y), nthreads)
    return z, y


def merge_value_output(w_uv: np.ndarray, w_o: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """Fig. 6 (3): the pre-merged weight What^O_h = W^UV_h W^O_h, [H, dc, D] in fp64."""
    w_uv, w_o = _f64(w_uv), _f64(w_o)
    H, dc, dv = w_uv.shape
    D = w_o.shape[1]
    assert w_o.shape == (H * dv, D)
    w_hat = np.empty((H, dc, D))
    _load().oracle_merge_value_output(_ptr(w_uv), _ptr(w_o), H, dc, dv, D, _ptr(w_hat), nthreads)
    return w_hat


def project_merged(u: np.ndarray, w_hat: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """Y = sum_h U_h What^O_h (Fig. 6 (3)); u [B,H,dc], w_hat [H,dc,D] -> y [B,D]."""
    u, w_hat = _f64(u), _f64(w_hat)
    B, H, dc = u.shape
    D = w_hat.shape[2]
    assert w_hat.shape == (H, dc, D)
    y = np.empty((B, D))
    _load().oracle_project_merged(_ptr(u), _ptr(w_hat), B, H, dc, D, _ptr(y), nthreads)
    return y


# ------------------------------------------------------------------------------------------
# Shared K = V decode over V4 / V4.1 main-KV entries ("DeepSeek's KV Cache: From 3.9 MB to 890 B
# per Token", section "HCA: 128 tokens into one" (Fig. 15), "Calculating V4-Flash's KV cache",
# "Calculating V4.1-Flash's KV cache").
# ------------------------------------------------------------------------------------------
V4_FP8 = 2       # 584 B: 448 E4M3 (one UE8M0 scale per 64) + 64 bf16 RoPE + 7 scales + 1 pad
V41_FP4 = 3      # 288 B: 512 E2M1 (one E4M3 scale per 16)
E_DIM = 512


def e2m1_decode(code: int) -> float:
    """OCP MX E2M1 value of one 4-bit code (exact)."""
    return float(_load().oracle_e2m1_decode(int(code) & 0xF))


def e2m1_encode(x: float) -> int:
    """E2M1 round-to-nearest-even, saturating at +-6, of one fp32 value."""
    return int(_load().oracle_e2m1_encode(float(np.float32(x))))


def shared_record_bytes(fmt: int) -> int:
    return int(_load().oracle_shared_record_bytes(int(fmt)))


def new_shared_pool(fmt: int, num_pages: int) -> np.ndarray:
    return np.zeros(num_pages * PAGE * shared_record_bytes(fmt), dtype=np.uint8)


def shared_append(fmt: int, pool: np.ndarray, entry: np.ndarray, slot: np.ndarray) -> int:
    """Quantise T entries (bf16 bits [T,512]) into ``pool`` at ``slot``; returns the number of rows
    whose slot lies outside the pool."""
    entry = np.ascontiguousarray(entry, dtype=np.uint16)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    T = slot.shape[0]
    assert entry.shape == (T, E_DIM)
    num_pages = pool.size // (PAGE * shared_record_bytes(fmt))
    return int(_load().oracle_shared_append(int(fmt), _ptr(pool), num_pages, _ptr(entry), _ptr(slot), T))


def shared_read(fmt: int, pool: np.ndarray, slot: int) -> np.ndarray:
    """One cached entry as exact doubles [512]."""
    e = np.empty(E_DIM, dtype=np.float64)
    _load().oracle_shared_read(int(fmt), _ptr(pool), int(slot), _ptr(e))
    return e


def attend_sink(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, sink: float = -np.inf):
    """Attention of one query with the sink exp(sink) in the softmax denominator (fp64):
    returns (out[dv], lse) with lse = ln(sum_t exp(s_t) + exp(sink))."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    n, dk = K.shape
    dv = V.shape[1]
    out = np.empty(dv)
    lse = np.empty(1)
    _load().oracle_attend_sink(_ptr(q), _ptr(K), dk, _ptr(V), dv, n, dk, dv, float(scale), float(sink),
                               _ptr(out), _ptr(lse))
    return out, float(lse[0])


def unrotate(o: np.ndarray, cos_sin: np.ndarray) -> np.ndarray:
    """The last 64 dims of a 512-dim head output rotated back by the angles whose cosines and
    sines cos_sin[0:32], cos_sin[32:64] gives (pairs 448 + 2i, 448 + 2i + 1)."""
    o = _f64(o).copy()
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    assert o.shape == (E_DIM,) and cs.shape == (64,)
    _load().oracle_unrotate(_ptr(o), _ptr(cs))
    return o


def shared_kv_decode(fmt: int, pool: np.ndarray, q: np.ndarray, block_table: np.ndarray,
                     seq_lens: np.ndarray, scale: float, sink: np.ndarray | None = None,
                     rope_cs: np.ndarray | None = None, topk_idx: np.ndarray | None = None, pairs=None,
                     nthreads: int = 0):
    """Shared K = V decode in fp64 for the (b, h) pairs given (all by default).  q bf16 bits
    [B,H,512]; sink fp32 [H] or None; rope_cs fp32 [B,64] (cos then sin of the query position's
    32 angles) or None.  Returns (out float64[n,512], lse float64[n])."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, H, _ = q.shape
    if pairs is None:
        pairs = np.stack(np.meshgrid(np.arange(B), np.arange(H), indexing="ij"), -1).reshape(-1, 2)
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    order = np.argsort(pairs[:, 0], kind="stable")
    sp = np.ascontiguousarray(pairs[order])
    n = sp.shape[0]
    out = np.empty((n, E_DIM))
    lse = np.empty(n)
    topk = 0
    if topk_idx is not None:
        topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
        topk = topk_idx.shape[1]
    sk = None if sink is None else np.ascontiguousarray(sink, dtype=np.float32)
    cs = None if rope_cs is None else np.ascontiguousarray(rope_cs, dtype=np.float32)
    num_pages = pool.size // (PAGE * shared_record_bytes(fmt))
    rc = _load().oracle_shared_kv_decode(int(fmt), _ptr(pool), num_pages, _ptr(q), _ptr(block_table),
                                         block_table.shape[1], _ptr(seq_lens), _ptr(topk_idx), topk, B, H,
                                         float(np.float32(scale)), _ptr(sk), _ptr(cs), _ptr(sp), n, _ptr(out),
                                         _ptr(lse), nthreads)
    if rc != 0:
        raise ValueError("oracle_shared_kv_decode: a visible position maps outside the pool")
    res_out = np.empty_like(out)
    res_lse = np.empty_like(lse)
    res_out[order] = out
    res_lse[order] = lse
    return res_out, res_lse
