"""GB300-native absorbed MLA decode over a paged latent cache.

A thin ctypes binding over the C ABI of ``libmla.so`` (declared in ``include/mla.h``): every call
only checks tensor dtypes/shapes/devices, marshals pointers and the current CUDA stream, and
forwards to the library; all computation happens in the library's kernels.  PyTorch provides
device memory and streams.  The library is loaded lazily on first use and its absence is an
error (there is no fallback path).

Entry points (same names as the C ABI, without the ``mla_`` prefix):
  record_bytes(fmt), cache_append(...), decode_workspace_bytes(...), decode(...), combine(...),
  check_status(), status_string(code), set_wait_limit(n), e4m3_encode(x)
"""
from __future__ import annotations

import ctypes
import os
import threading

BF16 = 0          # 1,152-byte record: [c_KV 512 bf16 | k_rope 64 bf16]
FP8_MIXED = 1     # 656-byte record: [512 E4M3 | 4 fp32 scales | 64 bf16 rope]
V4_FP8 = 2        # 584-byte shared K = V entry: 448 E4M3 (UE8M0 per 64) + 64 bf16 RoPE dims
V41_FP4 = 3       # 288-byte shared K = V entry: 512 E2M1 + one E4M3 scale per 16 dims
D_C = 512
D_R = 64
HEADS = 128
PAGE = 64

STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID", 2: "MLA_ERR_BOUNDS", 3: "MLA_ERR_TIMEOUT",
          4: "MLA_ERR_CUDA", 5: "MLA_ERR_UNSUPPORTED", 6: "MLA_ERR_RANGE"}

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla.so")
_lock = threading.Lock()
_lib = None


class MlaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({status_string(code)})")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libmla.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
        lib.mla_record_bytes.argtypes = [i32]
        lib.mla_record_bytes.restype = sz
        lib.mla_cache_append.argtypes = [i32, P, i64, P, P, P, i64, P]
        lib.mla_cache_append.restype = ctypes.c_int
        lib.mla_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        lib.mla_decode_workspace_bytes.restype = sz
        lib.mla_decode_launches.argtypes = [i32, i32, i32, i32, i32]
        lib.mla_decode_launches.restype = i32
        lib.mla_decode.argtypes = [i32, P, i64, P, P, P, i32, P, i32, P, i32, i32, i32, f32, P, P,
                                   P, sz, P]
        lib.mla_decode.restype = ctypes.c_int
        lib.mla_decode_noalloc.argtypes = [i32, P, i64, P, P, P, i32, P, i32, P, i32, i32, i32, f32,
                                           P, P, P]
        lib.mla_decode_noalloc.restype = ctypes.c_int
        lib.mla_combine.argtypes = [P, P, i32, i32, i32, P, P, P]
        lib.mla_combine.restype = ctypes.c_int
        lib.mla_check_status.argtypes = [P]
        lib.mla_check_status.restype = ctypes.c_int
        lib.mla_status_string.argtypes = [ctypes.c_int]
        lib.mla_status_string.restype = ctypes.c_char_p
        lib.mla_set_wait_limit.argtypes = [ctypes.c_uint32]
        lib.mla_set_wait_limit.restype = ctypes.c_int
        lib.mla_e4m3_encode.argtypes = [P, P, i64, P]
        lib.mla_e4m3_encode.restype = ctypes.c_int
        lib.mla_index_append.argtypes = [P, i64, P, P, i64, P]
        lib.mla_index_append.restype = ctypes.c_int
        lib.mla_indexer_score.argtypes = [P, i64, P, P, P, i32, P, i32, i32, P, P]
        lib.mla_indexer_score.restype = ctypes.c_int
        lib.mla_topk_select.argtypes = [P, i64, P, i32, i32, P, P]
        lib.mla_topk_select.restype = ctypes.c_int
        lib.mla_shared_kv_append.argtypes = [i32, P, i64, P, P, i64, P]
        lib.mla_shared_kv_append.restype = ctypes.c_int
        lib.mla_shared_kv_decode.argtypes = [i32, P, i64, P, P, i32, P, i32, P, i32, i32, i32, f32, P, P, P, P,
                                             P, sz, P]
        lib.mla_shared_kv_decode.restype = ctypes.c_int
        lib.mla_value_project.argtypes = [P, P, P, i32, i32, i32, P, P, P]
        lib.mla_value_project.restype = ctypes.c_int
        lib.mla_value_project_merged.argtypes = [P, P, i32, i32, i32, P, P]
        lib.mla_value_project_merged.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(code: int) -> str:
    try:
        return load().mla_status_string(int(code)).decode()
    except Exception:
        return STATUS.get(code, "unknown")


def _torch():
    import torch
    return torch


def _stream_ptr(stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _dev_ptr(t, name: str, dtype=None, shape=None) -> int | None:
    if t is None:
        return None
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return int(t.data_ptr())


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise MlaError(rc, what)


def record_bytes(fmt: int) -> int:
    return int(load().mla_record_bytes(int(fmt)))


def pool_bytes(fmt: int, num_pages: int) -> int:
    return num_pages * PAGE * record_bytes(fmt)


def cache_append(fmt: int, pool, num_pages: int, c_kv, k_rope, slot, stream=None) -> None:
    """Write T tokens (bf16 c_kv[T,512], k_rope[T,64]) into the pool at int32 ``slot[T]``."""
    torch = _torch()
    T = int(slot.shape[0])
    rc = load().mla_cache_append(
        int(fmt), _dev_ptr(pool, "pool", torch.uint8), int(num_pages),
        _dev_ptr(c_kv, "c_kv", torch.bfloat16, (T, D_C)),
        _dev_ptr(k_rope, "k_rope", torch.bfloat16, (T, D_R)),
        _dev_ptr(slot, "slot", torch.int32), T, _stream_ptr(stream))
    _check(rc, "mla_cache_append")


def decode_workspace_bytes(fmt: int, B: int, max_seq_len: int, topk: int = 0, H: int = HEADS) -> int:
    return int(load().mla_decode_workspace_bytes(int(fmt), int(B), int(H), int(max_seq_len), int(topk)))


def decode(fmt: int, pool, num_pages: int, q_lat, q_rope, block_table, seq_lens,
           max_seq_len: int, scale: float, topk_idx=None, out=None, lse=None, workspace=None,
           stream=None):
    """Absorbed MLA decode; returns (out bf16[B,H,512], lse fp32[B,H])."""
    torch = _torch()
    B, H, _ = q_lat.shape
    if out is None:
        out = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=q_lat.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q_lat.device)
    topk = 0 if topk_idx is None else int(topk_idx.shape[1])
    if workspace is None:   # (a caller's workspace is checked against the need by the library)
        need = decode_workspace_bytes(fmt, B, max_seq_len, topk, H)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q_lat.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().mla_decode(
        int(fmt), _dev_ptr(pool, "pool", torch.uint8), int(num_pages),
        _dev_ptr(q_lat, "q_lat", torch.bfloat16, (B, H, D_C)),
        _dev_ptr(q_rope, "q_rope", torch.bfloat16, (B, H, D_R)),
        _dev_ptr(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev_ptr(seq_lens, "seq_lens", torch.int32, (B,)), int(max_seq_len),
        _dev_ptr(topk_idx, "topk_idx", torch.int32), topk, int(B), int(H), float(scale),
        _dev_ptr(out, "out", torch.bfloat16, (B, H, D_C)),
        _dev_ptr(lse, "lse", torch.float32, (B, H)),
        _dev_ptr(workspace, "workspace"), ws_bytes, _stream_ptr(stream))
    _check(rc, "mla_decode")
    return out, lse


def decode_noalloc(fmt: int, pool, num_pages: int, q_lat, q_rope, block_table, seq_lens,
                   max_seq_len: int, scale: float, topk_idx=None, out=None, lse=None, stream=None):
    """decode() for callers that cannot allocate device memory while decoding: the split-KV
    scratch is the library's static device array (include/mla.h, mla_decode_noalloc) instead of a
    workspace tensor.  Outputs must be passed in by such callers; calls must not overlap."""
    torch = _torch()
    B, H, _ = q_lat.shape
    if out is None:
        out = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=q_lat.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q_lat.device)
    topk = 0 if topk_idx is None else int(topk_idx.shape[1])
    rc = load().mla_decode_noalloc(
        int(fmt), _dev_ptr(pool, "pool", torch.uint8), int(num_pages),
        _dev_ptr(q_lat, "q_lat", torch.bfloat16, (B, H, D_C)),
        _dev_ptr(q_rope, "q_rope", torch.bfloat16, (B, H, D_R)),
        _dev_ptr(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev_ptr(seq_lens, "seq_lens", torch.int32, (B,)), int(max_seq_len),
        _dev_ptr(topk_idx, "topk_idx", torch.int32), topk, int(B), int(H), float(scale),
        _dev_ptr(out, "out", torch.bfloat16, (B, H, D_C)),
        _dev_ptr(lse, "lse", torch.float32, (B, H)), _stream_ptr(stream))
    _check(rc, "mla_decode_noalloc")
    return out, lse


def combine(o_part, lse_part, out=None, lse=None, stream=None):
    """Merge split partials o_part fp32[S,B,H,512], lse_part fp32[S,B,H] -> (out, lse)."""
    torch = _torch()
    S, B, H, _ = o_part.shape
    if out is None:
        out = torch.empty((B, H, D_C), dtype=torch.bfloat16, device=o_part.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=o_part.device)
    rc = load().mla_combine(_dev_ptr(o_part, "o_part", torch.float32),
                            _dev_ptr(lse_part, "lse_part", torch.float32, (S, B, H)), int(S),
                            int(B), int(H), _dev_ptr(out, "out", torch.bfloat16, (B, H, D_C)),
                            _dev_ptr(lse, "lse", torch.float32, (B, H)), _stream_ptr(stream))
    _check(rc, "mla_combine")
    return out, lse


def check_status(stream=None) -> int:
    """Synchronise and return (then clear) the first error a kernel recorded (0 if none)."""
    return int(load().mla_check_status(_stream_ptr(stream)))


def set_wait_limit(iterations: int) -> None:
    _check(load().mla_set_wait_limit(int(iterations)), "mla_set_wait_limit")


def e4m3_encode(x, codes=None, stream=None):
    torch = _torch()
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    rc = load().mla_e4m3_encode(_dev_ptr(x, "x", torch.float32), _dev_ptr(codes, "codes", torch.uint8),
                                int(x.numel()), _stream_ptr(stream))
    _check(rc, "mla_e4m3_encode")
    return codes


# DSA lightning indexer: search-key pool, indexer scores, top-k selection (include/mla.h).
INDEX_HEADS = 64
INDEX_DIM = 128
INDEX_PAGE_BYTES = 8448


def index_pool_bytes(num_pages: int) -> int:
    return num_pages * INDEX_PAGE_BYTES


def index_append(pool, num_pages: int, k_index, slot, stream=None) -> None:
    """Quantise T search keys (bf16 k_index[T,128]) into the search-key pool at int32 ``slot[T]``."""
    torch = _torch()
    T = int(slot.shape[0])
    rc = load().mla_index_append(_dev_ptr(pool, "pool", torch.uint8), int(num_pages),
                                 _dev_ptr(k_index, "k_index", torch.bfloat16, (T, INDEX_DIM)),
                                 _dev_ptr(slot, "slot", torch.int32), T, _stream_ptr(stream))
    _check(rc, "mla_index_append")


def indexer_score(pool, num_pages: int, q_index, w_index, block_table, seq_lens, max_seq_len: int,
                  scores=None, stream=None):
    """fp32 scores[B, max_seq_len] of the queries (bf16 q_index[B,64,128], fp32 w_index[B,64])."""
    torch = _torch()
    B = int(q_index.shape[0])
    if scores is None:
        scores = torch.empty((B, max_seq_len), dtype=torch.float32, device=q_index.device)
    rc = load().mla_indexer_score(_dev_ptr(pool, "pool", torch.uint8), int(num_pages),
                                  _dev_ptr(q_index, "q_index", torch.bfloat16, (B, INDEX_HEADS, INDEX_DIM)),
                                  _dev_ptr(w_index, "w_index", torch.float32, (B, INDEX_HEADS)),
                                  _dev_ptr(block_table, "block_table", torch.int32), int(block_table.shape[1]),
                                  _dev_ptr(seq_lens, "seq_lens", torch.int32, (B,)), B, int(max_seq_len),
                                  _dev_ptr(scores, "scores", torch.float32, (B, max_seq_len)), _stream_ptr(stream))
    _check(rc, "mla_indexer_score")
    return scores


def topk_select(scores, seq_lens, K: int, topk_idx=None, stream=None):
    """int32 topk_idx[B, K]: per row the K highest scores among positions < seq_lens[b], in
    increasing position order, -1 past the picks."""
    torch = _torch()
    B, ld = scores.shape
    if topk_idx is None:
        topk_idx = torch.empty((B, K), dtype=torch.int32, device=scores.device)
    rc = load().mla_topk_select(_dev_ptr(scores, "scores", torch.float32), int(ld),
                                _dev_ptr(seq_lens, "seq_lens", torch.int32, (B,)), int(B), int(K),
                                _dev_ptr(topk_idx, "topk_idx", torch.int32, (B, K)), _stream_ptr(stream))
    _check(rc, "mla_topk_select")
    return topk_idx


# Value up-projection and output projection of the decode output (include/mla.h).
D_V = 128


def value_project(u, w_uv_t, w_o_t, z=None, y=None, stream=None):
    """Y = sum_h (U_h W^UV_h) W^O_h: u bf16[B,H,512], w_uv_t bf16[H,128,512] (W^UV_h transposed),
    w_o_t bf16[D,H*128] (W^O transposed).  Returns (y bf16[B,D], z bf16[2,B,H*128]: Z as hi and lo
    planes)."""
    torch = _torch()
    B, H, _ = u.shape
    D = int(w_o_t.shape[0])
    if z is None:
        z = torch.empty((2, B, H * D_V), dtype=torch.bfloat16, device=u.device)
    if y is None:
        y = torch.empty((B, D), dtype=torch.bfloat16, device=u.device)
    rc = load().mla_value_project(_dev_ptr(u, "u", torch.bfloat16, (B, H, D_C)),
                                  _dev_ptr(w_uv_t, "w_uv_t", torch.bfloat16, (H, D_V, D_C)),
                                  _dev_ptr(w_o_t, "w_o_t", torch.bfloat16, (D, H * D_V)), int(B), int(H), D,
                                  _dev_ptr(z, "z", torch.bfloat16, (2, B, H * D_V)),
                                  _dev_ptr(y, "y", torch.bfloat16, (B, D)), _stream_ptr(stream))
    _check(rc, "mla_value_project")
    return y, z


def value_project_merged(u, w_hat_t, y=None, stream=None):
    """Y = sum_h U_h What^O_h with the pre-merged weight: u bf16[B,H,512], w_hat_t bf16[D,H*512]."""
    torch = _torch()
    B, H, _ = u.shape
    D = int(w_hat_t.shape[0])
    if y is None:
        y = torch.empty((B, D), dtype=torch.bfloat16, device=u.device)
    rc = load().mla_value_project_merged(_dev_ptr(u, "u", torch.bfloat16, (B, H, D_C)),
                                         _dev_ptr(w_hat_t, "w_hat_t", torch.bfloat16, (D, H * D_C)), int(B),
                                         int(H), D, _dev_ptr(y, "y", torch.bfloat16, (B, D)), _stream_ptr(stream))
    _check(rc, "mla_value_project_merged")
    return y


# Shared K = V decode over V4 / V4.1 entries (include/mla.h).
E_DIM = 512


def shared_kv_append(fmt: int, pool, num_pages: int, entry, slot, stream=None) -> None:
    """Quantise T entries (bf16 entry[T,512]) into a V4 / V4.1 pool at int32 ``slot[T]``."""
    torch = _torch()
    T = int(slot.shape[0])
    rc = load().mla_shared_kv_append(int(fmt), _dev_ptr(pool, "pool", torch.uint8), int(num_pages),
                                     _dev_ptr(entry, "entry", torch.bfloat16, (T, E_DIM)),
                                     _dev_ptr(slot, "slot", torch.int32), T, _stream_ptr(stream))
    _check(rc, "mla_shared_kv_append")


def shared_kv_decode(fmt: int, pool, num_pages: int, q, block_table, seq_lens, max_seq_len: int,
                     scale: float, sink=None, rope_cs=None, topk_idx=None, out=None, lse=None, workspace=None,
                     stream=None):
    """Shared K = V decode; returns (out bf16[B,H,512], lse fp32[B,H])."""
    torch = _torch()
    B, H, _ = q.shape
    if out is None:
        out = torch.empty((B, H, E_DIM), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    topk = 0 if topk_idx is None else int(topk_idx.shape[1])
    if workspace is None:
        need = decode_workspace_bytes(fmt, B, max_seq_len, topk, H)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().mla_shared_kv_decode(
        int(fmt), _dev_ptr(pool, "pool", torch.uint8), int(num_pages),
        _dev_ptr(q, "q", torch.bfloat16, (B, H, E_DIM)),
        _dev_ptr(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev_ptr(seq_lens, "seq_lens", torch.int32, (B,)), int(max_seq_len),
        _dev_ptr(topk_idx, "topk_idx", torch.int32), topk, int(B), int(H), float(scale),
        _dev_ptr(sink, "sink", torch.float32, (H,)), _dev_ptr(rope_cs, "rope_cs", torch.float32, (B, 64)),
        _dev_ptr(out, "out", torch.bfloat16, (B, H, E_DIM)), _dev_ptr(lse, "lse", torch.float32, (B, H)),
        _dev_ptr(workspace, "workspace"), ws_bytes, _stream_ptr(stream))
    _check(rc, "mla_shared_kv_decode")
    return out, lse
