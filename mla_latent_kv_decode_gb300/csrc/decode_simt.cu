// decode_simt.cu -- first correct CUDA-core path of absorbed MLA decode (fp32 FMA, no tensor
// cores).  It exists to validate the boundary, the split-KV plan and the merge end to end; the
// tensor-core kernel replaces it on the hot path.
//
// Per head h and visible position t ("DeepSeek's KV Cache: From 3.9 MB to 890 B per Token",
// Fig. 4 (1), Fig. 5 (2), Fig. 6 (2), Fig. 10):
//   s_t = scale * (q_lat[h] . c_t + q_rope[h] . k_rope_t),  out = sum_t softmax(s)_t c_t,
//   lse = ln sum_t exp(s_t), streamed over 32-position tiles with a running max (online softmax).
//
// Grid: (split, request, head group of 8).  The 32 x 576 tile is widened to fp32 in shared
// memory (FP8 codes times their group scale), each thread scores one (head, position) pair and
// accumulates 2 latent dims x 8 heads of the output.
#include <cfloat>
#include <cuda_fp8.h>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kTile = 32;
constexpr int kHG = 8;             // heads per block
constexpr int kThreads = 256;
constexpr int kKStride = kDk + 1;  // padded row: conflict-free column reads

struct SimtSmem {
    float q[kHG][kDk];
    float k[kTile][kKStride];
    float p[kHG][kTile];
    float alpha[kHG];
    float l[kHG];
    float m[kHG];
    const uint8_t* rec[kTile];
    int valid[kTile];
};

__device__ __forceinline__ float bf16_at(const uint8_t* p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}

__global__ void __launch_bounds__(kThreads) decode_simt_kernel(DecodeArgs a, int chunk, int splits) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SimtSmem& sm = *reinterpret_cast<SimtSmem*>(smem_raw);
    const int split = blockIdx.x;
    const int b = blockIdx.y;
    const int h0 = blockIdx.z * kHG;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    int n_b = a.seq_lens[b];
    if (n_b < 0 || n_b > a.max_seq_len) {
        if (tid == 0) record_error(a.ctl, MLA_ERR_BOUNDS, b);
        n_b = n_b < 0 ? 0 : a.max_seq_len;
    }
    const int n_entries = a.topk_idx ? a.topk : n_b;
    const int e0 = split * chunk;
    const int e1 = min(n_entries, e0 + chunk);
    const int rb = a.fmt == MLA_KV_BF16 ? kBf16RecordBytes : kFp8RecordBytes;

    for (int i = tid; i < kHG * kDk; i += kThreads) {
        const int h = i / kDk, d = i % kDk;
        const size_t qrow = (size_t)b * kHeads + h0 + h;
        sm.q[h][d] = d < kDc ? __bfloat162float(a.q_lat[qrow * kDc + d])
                             : __bfloat162float(a.q_rope[qrow * kDr + d - kDc]);
    }
    float acc[kHG][2];
#pragma unroll
    for (int h = 0; h < kHG; ++h) acc[h][0] = acc[h][1] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;   // per warp = per head (warp w owns head h0 + w)

    for (int t0 = e0; t0 < e1; t0 += kTile) {
        __syncthreads();
        if (tid < kTile) {
            const int e = t0 + tid;
            int valid = 0;
            const uint8_t* rec = nullptr;
            if (e < e1) {
                int pos = a.topk_idx ? a.topk_idx[(size_t)b * a.topk + e] : e;
                if (pos >= 0 && pos < n_b) {
                    const int page = a.block_table[(size_t)b * a.max_pages + pos / kPage];
                    if (page >= 0 && page < a.num_pages) {
                        valid = 1;
                        rec = a.pool + ((size_t)page * kPage + pos % kPage) * rb;
                    } else {
                        record_error(a.ctl, MLA_ERR_BOUNDS, page);
                    }
                }
            }
            sm.valid[tid] = valid;
            sm.rec[tid] = rec;
        }
        __syncthreads();
        for (int i = tid; i < kTile * kDk; i += kThreads) {
            const int t = i / kDk, d = i % kDk;
            const uint8_t* rec = sm.rec[t];
            float v = 0.f;
            if (rec) {
                if (a.fmt == MLA_KV_BF16) {
                    v = bf16_at(rec + 2 * d);
                } else if (d < kDc) {
                    const float sc = reinterpret_cast<const float*>(rec + kFp8ScaleOff)[d / kFp8Group];
                    __nv_fp8_storage_t code = rec[d];
                    __half_raw hr = __nv_cvt_fp8_to_halfraw(code, __NV_E4M3);
                    v = __half2float(__half(hr)) * sc;
                } else {
                    v = bf16_at(rec + kFp8RopeOff + 2 * (d - kDc));
                }
            }
            sm.k[t][d] = v;
        }
        __syncthreads();
        {
            const int h = warp, t = lane;
            float dot = 0.f;
#pragma unroll 8
            for (int d = 0; d < kDk; ++d) dot = fmaf(sm.q[h][d], sm.k[t][d], dot);
            float s = sm.valid[t] ? dot * a.scale : -INFINITY;
            float mt = s;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
            const float m_new = fmaxf(m_run, mt);
            float p = 0.f, alpha = 1.f;
            if (m_new != -INFINITY) {
                p = expf(s - m_new);
                alpha = expf(m_run - m_new);
            }
            float ps = p;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            l_run = l_run * alpha + ps;
            m_run = m_new;
            sm.p[h][t] = p;
            if (lane == 0) sm.alpha[h] = alpha;
        }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < kHG; ++h) {
            const float al = sm.alpha[h];
            float a0 = acc[h][0] * al, a1 = acc[h][1] * al;
#pragma unroll 8
            for (int t = 0; t < kTile; ++t) {
                const float p = sm.p[h][t];
                a0 = fmaf(p, sm.k[t][tid], a0);
                a1 = fmaf(p, sm.k[t][tid + 256], a1);
            }
            acc[h][0] = a0;
            acc[h][1] = a1;
        }
    }
    if (lane == 0) {
        sm.l[warp] = l_run;
        sm.m[warp] = m_run;
    }
    __syncthreads();
    const size_t BH = (size_t)a.B * kHeads;
#pragma unroll
    for (int h = 0; h < kHG; ++h) {
        const float l = sm.l[h];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t row = (size_t)b * kHeads + h0 + h;
        const float o0 = acc[h][0] * inv, o1 = acc[h][1] * inv;
        const float L = l > 0.f ? sm.m[h] + logf(l) : -INFINITY;
        if (splits == 1) {
            a.out[row * kDc + tid] = __float2bfloat16_rn(o0);
            a.out[row * kDc + tid + 256] = __float2bfloat16_rn(o1);
            if (tid == 0) a.lse[row] = L;
        } else {
            float* op = a.o_part + ((size_t)split * BH + row) * kDc;
            op[tid] = o0;
            op[tid + 256] = o1;
            if (tid == 0) a.lse_part[(size_t)split * BH + row] = L;
        }
    }
}

}  // namespace

DecodePlan plan_decode_simt(int fmt, int B, int max_seq_len, int topk, int sms) {
    (void)fmt;
    DecodePlan p;
    const int L = topk > 0 ? topk : max_seq_len;
    const int blocks_per_split = B * (kHeads / kHG);
    int S = (2 * sms + blocks_per_split - 1) / blocks_per_split;
    const int max_s = (L + 63) / 64;
    if (S > max_s) S = max_s;
    if (S < 1) S = 1;
    int chunk = (L + S - 1) / S;
    chunk = (chunk + 63) / 64 * 64;
    if (chunk < 64) chunk = 64;
    S = (L + chunk - 1) / chunk;
    if (S < 1) S = 1;
    p.splits = S;
    p.chunk = chunk;
    p.workspace = S > 1 ? (size_t)S * B * kHeads * (kDc + 1) * sizeof(float) : 0;
    p.launches = S > 1 ? 2 : 1;
    return p;
}

cudaError_t launch_decode_simt(const DecodeArgs& args, const DecodePlan& p, cudaStream_t st) {
    DecodeArgs a = args;
    if (p.splits > 1) {
        a.o_part = static_cast<float*>(a.workspace);
        a.lse_part = a.o_part + (size_t)p.splits * a.B * kHeads * kDc;
    }
    const int smem = (int)sizeof(SimtSmem);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {   // set once per device, outside any stream capture
        e = cudaFuncSetAttribute(decode_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    dim3 grid(p.splits, a.B, kHeads / kHG);
    decode_simt_kernel<<<grid, kThreads, smem, st>>>(a, p.chunk, p.splits);
    e = cudaGetLastError();
    if (e != cudaSuccess || p.splits == 1) return e;
    return launch_combine(a.o_part, a.lse_part, p.splits, a.B, kHeads, a.out, a.lse, st);
}

}  // namespace mla
