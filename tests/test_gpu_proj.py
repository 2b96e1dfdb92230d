"""Parity of the value up-projection and output projection ("DeepSeek's KV Cache: From 3.9 MB to
890 B per Token", section "Computing without expanding Key and Value", Fig. 6 (2) and (3)) with
the fp64 oracle, through the C ABI.

Tolerance, from the arithmetic: Y is rounded once to bf16 (relative error at most 2^-9) after
fp32 accumulation of products of bf16 values, with Z carried to about 16 significant bits; so
every element within 2^-8 |Y| + 2^-12 of the oracle (twice the rounding bound, plus room for the
accumulation), and per request ||gpu - oracle|| <= 1e-2 ||oracle||.  Z's two bf16 planes:
|hi + lo - Z| <= 2^-14 |Z| + 2^-16 sum_k |U_k W_kj| per element (16-bit planes plus the fp32
accumulation), and |lo| at most half a bf16 step of hi.
"""
import numpy as np
import pytest

import oracle
import mla_latent_kv_decode_gb300 as mla
from mla_latent_kv_decode_gb300 import harness

pytestmark = pytest.mark.gpu

Y_REL = 1e-2


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _check_y(y, ref, what):
    err = np.abs(y - ref)
    assert np.isfinite(y).all(), what
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -12
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), f"{what}: |y err| {err.flat[worst]:.3e} at |y| {np.abs(ref).flat[worst]:.3e}"
    rel = np.linalg.norm(y - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    assert rel.max() <= Y_REL, f"{what}: normwise {rel.max():.3e}"


def _two_stage(B, H, D, seed):
    p = harness.ProjInputs(B, H, D, seed=seed)
    y, z = mla.value_project(p.u, p.w_uv_t, p.w_o_t)
    assert mla.check_status() == 0
    u = _np(p.u)
    w_uv = _np(p.w_uv_t).transpose(0, 2, 1)          # [H, 512, 128]: W^UV_h as in Fig. 6
    w_o = _np(p.w_o_t).T                             # [H*128, D]: W^O
    zr, yr = oracle.value_project(u, w_uv, w_o)
    _check_y(_np(y), yr, f"value_project B={B} H={H} D={D}")
    zz = _np(z)
    zsum = zz[0] + zz[1]
    zref = zr.reshape(B, H * mla.D_V)
    # fp32 accumulation of 512 products: an error bound relative to the sum of |products|
    zabs, _ = oracle.value_project(np.abs(u), np.abs(w_uv), np.zeros((H * mla.D_V, 128)))
    bound = 2.0 ** -14 * np.abs(zref) + 2.0 ** -16 * zabs.reshape(B, H * mla.D_V)
    assert np.all(np.abs(zsum - zref) <= bound), "Z planes"
    # the lo plane is what the hi plane's rounding left: at most half a bf16 step of hi
    assert np.all(np.abs(zz[1]) <= 2.0 ** -8 * np.abs(zz[0]) + 1e-30)
    return p, y


def test_value_project_full_size():
    """DeepSeek-V2's shapes: 128 heads, d_v = 128, hidden size 5,120, a batch of 64."""
    _two_stage(64, 128, 5120, seed=0x4D4C41 + 7)


@pytest.mark.parametrize("B,H,D", [(1, 2, 128), (7, 3, 256), (130, 5, 384), (33, 128, 640)])
def test_value_project_ragged_shapes(B, H, D):
    """Batches that are not a multiple of the tile (one request, 7, 130 across two batch tiles),
    head counts whose reduction splits unevenly across a cluster, several output tiles."""
    _two_stage(B, H, D, seed=0x4D4C41 + 8 + B)


def test_value_project_merged_weight():
    """Fig. 6 (3): the pre-merged What^O_h = W^UV_h W^O_h (merged in fp64 by the oracle, rounded to
    bf16 as the caller would store it); the GPU product against the oracle's on that same bf16
    weight, and the two GPU forms against each other."""
    import torch
    B, H, D = 48, 128, 1024
    p = harness.ProjInputs(B, H, D, seed=0x4D4C41 + 9)
    u = _np(p.u)
    w_uv = _np(p.w_uv_t).transpose(0, 2, 1)
    w_o = _np(p.w_o_t).T
    w_hat = oracle.merge_value_output(w_uv, w_o)                       # [H, 512, D]
    w_hat_t = torch.from_numpy(np.ascontiguousarray(w_hat.transpose(2, 0, 1).reshape(D, H * 512))).to(
        torch.float32).to(torch.bfloat16).cuda()
    y3 = mla.value_project_merged(p.u, w_hat_t)
    assert mla.check_status() == 0
    w_hat_b = _np(w_hat_t).reshape(D, H, 512).transpose(1, 2, 0)       # the bf16 weight, as doubles
    _check_y(_np(y3), oracle.project_merged(u, w_hat_b), "merged")
    y2, _ = mla.value_project(p.u, p.w_uv_t, p.w_o_t)
    assert mla.check_status() == 0
    _, yr = oracle.value_project(u, w_uv, w_o)
    # the two GPU forms against the unrounded fp64 result: the merged weight's own bf16 rounding
    # (2^-9 relative per element, averaging out over 65,536 terms) adds a little to the first
    _check_y(_np(y2), yr, "two products vs fp64")
    rel = np.linalg.norm(_np(y3) - yr) / np.linalg.norm(yr)
    assert rel <= 1e-2, f"merged vs fp64 normwise {rel:.3e}"


def test_value_project_empty_batch_and_bad_sizes():
    import torch
    p = harness.ProjInputs(4, 2, 256)
    lib = mla.load()
    s = torch.cuda.current_stream().cuda_stream
    # B = 0: nothing to do
    assert lib.mla_value_project(p.u.data_ptr(), p.w_uv_t.data_ptr(), p.w_o_t.data_ptr(), 0, 2, 256,
                                 p.u.data_ptr(), p.u.data_ptr(), s) == 0
    # D not a multiple of 128, H < 1: refused before launch
    y = torch.empty((4, 256), dtype=torch.bfloat16, device="cuda")
    z = torch.empty((2, 4, 256), dtype=torch.bfloat16, device="cuda")
    assert lib.mla_value_project(p.u.data_ptr(), p.w_uv_t.data_ptr(), p.w_o_t.data_ptr(), 4, 2, 200,
                                 z.data_ptr(), y.data_ptr(), s) == 1
    assert lib.mla_value_project(p.u.data_ptr(), p.w_uv_t.data_ptr(), p.w_o_t.data_ptr(), 4, 0, 256,
                                 z.data_ptr(), y.data_ptr(), s) == 1
    assert mla.check_status() == 0
