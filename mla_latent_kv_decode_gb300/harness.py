"""Device-side set-up of a synthetic workload through the public API.

Draws the seeded inputs of ``synth`` (on the host for small workloads, with the generator's
device twin for large ones), writes the cache through ``cache_append`` and keeps the decode
arguments as device tensors.  Used by the benchmark, the smoke check and the GPU tests.
"""
from __future__ import annotations

import numpy as np

import mla_latent_kv_decode_gb300 as mla
from mla_latent_kv_decode_gb300 import synth

HOST_GEN_LIMIT = 4_000_000     # values drawn on the host below this size, else on the device


def _t(torch, a, device, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


def bf16_tensor(torch, bits: np.ndarray, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


class DeviceWorkload:
    """The device tensors of one workload: a pool (or several identical replicas), queries,
    block table, seq_lens, optional top-k indices, and the rows each step appends."""

    def __init__(self, w: synth.Workload, device="cuda", replicas: int = 1, gen: str = "auto",
                 prefill_skip_last: int | None = None):
        import torch
        self.torch = torch
        self.w = w
        self.device = torch.device(device)
        self.replicas = replicas
        self.pool_bytes = mla.pool_bytes(w.fmt, w.num_pages)
        self.pools = [torch.zeros(self.pool_bytes, dtype=torch.uint8, device=self.device)
                      for _ in range(replicas)]
        ql, qr = w.queries()
        self.q_lat = bf16_tensor(torch, ql, self.device)
        self.q_rope = bf16_tensor(torch, qr, self.device)
        self.block_table = _t(torch, w.block_table, self.device, torch.int32)
        self.seq_lens = _t(torch, w.seq_lens, self.device, torch.int32)
        self.topk_idx = None if w.topk_idx is None else _t(torch, w.topk_idx, self.device, torch.int32)
        total = int(w.seq_lens.astype(np.int64).sum()) * synth.D_K
        self.gen = gen if gen != "auto" else ("host" if total <= HOST_GEN_LIMIT else "device")
        # tokens appended by each timed step: the last `appended` positions of every request
        self.appended = w.appended if prefill_skip_last is None else prefill_skip_last
        self._fill()
        self._make_step_rows()

    # -- input drawing ------------------------------------------------------------------------
    def rows(self, b: int, t0: int, t1: int):
        """(c_kv bf16[n,512], k_rope bf16[n,64]) device tensors of request b, positions t0..t1-1."""
        torch = self.torch
        n = t1 - t0
        if self.gen == "host":
            c, r = synth.kv_rows(self.w.seed, b, t0, t1)
            return bf16_tensor(torch, c, self.device), bf16_tensor(torch, r, self.device)
        c = torch.empty((n, synth.D_C), dtype=torch.bfloat16, device=self.device)
        r = torch.empty((n, synth.D_R), dtype=torch.bfloat16, device=self.device)
        base = (b * synth.KV_ROW_STRIDE + t0) * synth.D_K
        s = torch.cuda.current_stream().cuda_stream
        synth.gpu_normal_bf16(c.data_ptr(), n, self.w.seed, synth.STREAM_KV, base, synth.D_C, synth.D_K, s)
        synth.gpu_normal_bf16(r.data_ptr(), n, self.w.seed, synth.STREAM_KV, base + synth.D_C,
                              synth.D_R, synth.D_K, s)
        return c, r

    def slots(self, b: int, t0: int, t1: int):
        return _t(self.torch, self.w.slots(b, t0, t1), self.device, self.torch.int32)

    def _fill(self):
        w = self.w
        chunk = 1 << 16
        for b in range(w.B):
            n = int(w.seq_lens[b]) - self.appended
            for t0 in range(0, max(n, 0), chunk):
                t1 = min(n, t0 + chunk)
                c, r = self.rows(b, t0, t1)
                sl = self.slots(b, t0, t1)
                for pool in self.pools:
                    mla.cache_append(w.fmt, pool, w.num_pages, c, r, sl)
        rc = mla.check_status()
        if rc != 0:
            raise mla.MlaError(rc, "cache fill")

    def _make_step_rows(self):
        torch = self.torch
        w = self.w
        cs, rs, ss = [], [], []
        for b in range(w.B):
            n = int(w.seq_lens[b])
            t0 = max(0, n - self.appended)
            if t0 < n:
                c, r = self.rows(b, t0, n)
                cs.append(c)
                rs.append(r)
                ss.append(self.slots(b, t0, n))
        if cs:
            self.new_c = torch.cat(cs).contiguous()
            self.new_r = torch.cat(rs).contiguous()
            self.new_slot = torch.cat(ss).contiguous()
        else:
            self.new_c = self.new_r = self.new_slot = None

    # -- the hot path -------------------------------------------------------------------------
    def append(self, replica: int = 0, stream=None):
        if self.new_slot is not None:
            mla.cache_append(self.w.fmt, self.pools[replica], self.w.num_pages, self.new_c,
                             self.new_r, self.new_slot, stream=stream)

    def alloc_outputs(self):
        torch = self.torch
        w = self.w
        self.out = torch.empty((w.B, w.H, synth.D_C), dtype=torch.bfloat16, device=self.device)
        self.lse = torch.empty((w.B, w.H), dtype=torch.float32, device=self.device)
        need = mla.decode_workspace_bytes(w.fmt, w.B, w.max_seq_len,
                                          0 if w.topk_idx is None else w.topk_idx.shape[1])
        self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        return self.out, self.lse

    def decode(self, replica: int = 0, stream=None):
        w = self.w
        if not hasattr(self, "out"):
            self.alloc_outputs()
        return mla.decode(w.fmt, self.pools[replica], w.num_pages, self.q_lat, self.q_rope,
                          self.block_table, self.seq_lens, w.max_seq_len, w.scale,
                          topk_idx=self.topk_idx, out=self.out, lse=self.lse,
                          workspace=self.workspace, stream=stream)

    def step(self, replica: int = 0, stream=None):
        """One pass of the hot path: append this step's new tokens, then decode the batch."""
        self.append(replica, stream)
        return self.decode(replica, stream)

    # -- accounting ---------------------------------------------------------------------------
    def algorithmic_bytes(self) -> int:
        """Bytes the method must move per decode: attended records, q, out, lse, indices."""
        w = self.w
        rb = mla.record_bytes(w.fmt)
        n = w.attended()
        b = n * rb + w.B * w.H * (synth.D_K * 2 + synth.D_C * 2 + 4)
        b += w.B * 4 + w.block_table.size * 4
        if w.topk_idx is not None:
            b += w.topk_idx.size * 4
        return int(b)

    def kv_bytes(self) -> int:
        return int(self.w.attended() * mla.record_bytes(self.w.fmt))

    def flops(self) -> int:
        """2 * H * (576 + 512) per attended position (scores + weighted sum)."""
        return int(2 * self.w.H * (synth.D_K + synth.D_C) * self.w.attended())


class ProjInputs:
    """Seeded inputs of the value up-projection and output projection on the device: U (unit
    normal bf16), W^UV_h transposed (unit normal times 2^-4) and W^O transposed (unit normal
    times 2^-7), drawn by the generator's device twin; the power-of-two factors are exact in
    bf16 and give Z and Y a variance of about 2.  With merged=True the weight is instead a
    stand-in for What^O transposed [D, H*512] (unit normal times 2^-8), for timing."""

    def __init__(self, B: int, H: int = 128, D: int = 5120, seed: int = 0x4D4C41 + 7, merged: bool = False,
                 device="cuda"):
        import torch
        self.B, self.H, self.D, self.seed = B, H, D, seed
        dev = torch.device(device)
        s = torch.cuda.current_stream().cuda_stream

        def draw(shape, stream, scale):
            t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
            n = t.numel()
            row = shape[-1]
            synth.gpu_normal_bf16(t.data_ptr(), n // row, seed, stream, 0, row, row, s)
            if scale != 1.0:
                t.mul_(scale)
            return t

        self.u = draw((B, H, synth.D_C), synth.STREAM_U, 1.0)
        if merged:
            self.w_hat_t = draw((D, H * synth.D_C), synth.STREAM_WO, 2.0 ** -8)
        else:
            self.w_uv_t = draw((H, mla.D_V, synth.D_C), synth.STREAM_WUV, 2.0 ** -4)
            self.w_o_t = draw((D, H * mla.D_V), synth.STREAM_WO, 2.0 ** -7)
        torch.cuda.synchronize()

    def weight_bytes(self) -> int:
        if hasattr(self, "w_hat_t"):
            return self.w_hat_t.numel() * 2
        return (self.w_uv_t.numel() + self.w_o_t.numel()) * 2

    def algorithmic_bytes(self) -> int:
        """Weights, U and Y: what one call must move (the intermediate Z is not counted)."""
        return self.weight_bytes() + self.u.numel() * 2 + self.B * self.D * 2

    def flops(self) -> int:
        if hasattr(self, "w_hat_t"):
            return 2 * self.B * self.H * synth.D_C * self.D
        return 2 * self.B * self.H * mla.D_V * (synth.D_C + self.D)


class SharedDeviceWorkload:
    """The device tensors of a shared K = V workload (synth.SharedWorkload): pool replicas filled
    through shared_kv_append, queries, sinks, RoPE cos/sin, tables; the entries each step appends
    (the newest of every request)."""

    def __init__(self, w: synth.SharedWorkload, device="cuda", replicas: int = 1, gen: str = "auto",
                 appended: int = 1):
        import torch
        self.torch = torch
        self.w = w
        self.device = torch.device(device)
        self.replicas = replicas
        self.pool_bytes = w.num_pages * synth.PAGE * mla.record_bytes(w.fmt)
        self.pools = [torch.zeros(self.pool_bytes, dtype=torch.uint8, device=self.device) for _ in range(replicas)]
        self.q = bf16_tensor(torch, w.queries(), self.device)
        sk = w.sink()
        cs = w.rope_cs()
        self.sink = None if sk is None else torch.from_numpy(sk).to(self.device)
        self.rope_cs = None if cs is None else torch.from_numpy(cs).to(self.device)
        self.block_table = _t(torch, w.block_table, self.device, torch.int32)
        self.seq_lens = _t(torch, w.seq_lens, self.device, torch.int32)
        self.topk_idx = None if w.topk_idx is None else _t(torch, w.topk_idx, self.device, torch.int32)
        total = int(w.seq_lens.astype(np.int64).sum()) * synth.E_DIM
        self.gen = gen if gen != "auto" else ("host" if total <= HOST_GEN_LIMIT else "device")
        self.appended = appended
        self._fill()
        cs_, ss = [], []
        for b in range(w.B):
            n = int(w.seq_lens[b])
            t0 = max(0, n - appended)
            if t0 < n:
                cs_.append(self.entries(b, t0, n))
                ss.append(_t(torch, w.slots(b, t0, n), self.device, torch.int32))
        self.new_e = torch.cat(cs_).contiguous() if cs_ else None
        self.new_slot = torch.cat(ss).contiguous() if ss else None

    def entries(self, b: int, t0: int, t1: int):
        torch = self.torch
        if self.gen == "host":
            return bf16_tensor(torch, synth.shared_entries(self.w.seed, b, t0, t1), self.device)
        n = t1 - t0
        e = torch.empty((n, synth.E_DIM), dtype=torch.bfloat16, device=self.device)
        synth.gpu_normal_bf16(e.data_ptr(), n, self.w.seed, synth.STREAM_KV, (b * synth.KV_ROW_STRIDE + t0) * synth.E_DIM,
                              synth.E_DIM, synth.E_DIM, torch.cuda.current_stream().cuda_stream)
        return e

    def _fill(self):
        w = self.w
        chunk = 1 << 16
        for b in range(w.B):
            n = int(w.seq_lens[b]) - self.appended
            for t0 in range(0, max(n, 0), chunk):
                t1 = min(n, t0 + chunk)
                e = self.entries(b, t0, t1)
                sl = _t(self.torch, w.slots(b, t0, t1), self.device, self.torch.int32)
                for pool in self.pools:
                    mla.shared_kv_append(w.fmt, pool, w.num_pages, e, sl)
        rc = mla.check_status()
        if rc != 0:
            raise mla.MlaError(rc, "entry fill")

    def append(self, replica: int = 0, stream=None):
        if self.new_slot is not None:
            mla.shared_kv_append(self.w.fmt, self.pools[replica], self.w.num_pages, self.new_e, self.new_slot,
                                 stream=stream)

    def alloc_outputs(self):
        torch = self.torch
        w = self.w
        self.out = torch.empty((w.B, w.H, synth.E_DIM), dtype=torch.bfloat16, device=self.device)
        self.lse = torch.empty((w.B, w.H), dtype=torch.float32, device=self.device)
        need = mla.decode_workspace_bytes(w.fmt, w.B, w.max_seq_len, 0 if w.topk_idx is None else w.topk_idx.shape[1])
        self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        return self.out, self.lse

    def decode(self, replica: int = 0, stream=None):
        w = self.w
        if not hasattr(self, "out"):
            self.alloc_outputs()
        return mla.shared_kv_decode(w.fmt, self.pools[replica], w.num_pages, self.q, self.block_table,
                                    self.seq_lens, w.max_seq_len, w.scale, sink=self.sink, rope_cs=self.rope_cs,
                                    topk_idx=self.topk_idx, out=self.out, lse=self.lse, workspace=self.workspace,
                                    stream=stream)

    def step(self, replica: int = 0, stream=None):
        self.append(replica, stream)
        return self.decode(replica, stream)

    def kv_bytes(self) -> int:
        return int(self.w.attended() * mla.record_bytes(self.w.fmt))

    def algorithmic_bytes(self) -> int:
        """Attended entries, q, out, lse, sinks, cos/sin, tables."""
        w = self.w
        b = self.kv_bytes() + w.B * w.H * (synth.E_DIM * 2 * 2 + 4) + w.H * 4 + w.B * 64 * 4
        b += w.B * 4 + w.block_table.size * 4
        if w.topk_idx is not None:
            b += w.topk_idx.size * 4
        return int(b)

    def flops(self) -> int:
        """2 * H * (512 + 512) per attended entry (scores + weighted sum)."""
        return int(2 * self.w.H * 2 * synth.E_DIM * self.w.attended())
