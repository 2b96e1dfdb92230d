// combine.cu -- merge split-KV partials of absorbed MLA decode.
//
// Part i covers a disjoint subset of the visible positions and holds its normalised output o_i
// and lse_i = ln sum exp(s_t) over the subset.  The softmax over the union renormalises each
// part by its share of the mass (the renormalisation on a subset of "DeepSeek's KV Cache",
// Fig. 10):  lse = ln sum_i exp(lse_i),  out = sum_i exp(lse_i - lse) o_i.
//
// One 128-thread block per (request, head); each thread owns 4 of the 512 latent dims (one
// 16-byte load per part), so a part's 2 KB row is read with fully coalesced 512-byte warps.
// HBM-bound: S x 2 KB read + 1 KB written per (request, head).
#include "mla_internal.cuh"

namespace mla {
namespace {

__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ o_part,
                                                      const float* __restrict__ lse_part, int S,
                                                      int BH, __nv_bfloat16* __restrict__ out,
                                                      float* __restrict__ lse) {
    const int bh = blockIdx.x;
    const int t = threadIdx.x;
    float m = -INFINITY;
    for (int i = 0; i < S; ++i) m = fmaxf(m, lse_part[(size_t)i * BH + bh]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = -INFINITY;
    if (m != -INFINITY) {
        float l = 0.f;
        for (int i = 0; i < S; ++i) l += expf(lse_part[(size_t)i * BH + bh] - m);
        L = m + logf(l);
        for (int i = 0; i < S; ++i) {
            const float w = expf(lse_part[(size_t)i * BH + bh] - L);
            if (w == 0.f) continue;
            const float4 o = reinterpret_cast<const float4*>(o_part + ((size_t)i * BH + bh) * kDc)[t];
            acc.x += w * o.x;
            acc.y += w * o.y;
            acc.z += w * o.z;
            acc.w += w * o.w;
        }
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(out + (size_t)bh * kDc)[t] = packed;
    if (t == 0) lse[bh] = L;
}

}  // namespace

cudaError_t launch_combine(const float* o_part, const float* lse_part, int S, int B, int H,
                           __nv_bfloat16* out, float* lse, cudaStream_t st) {
    const int64_t BH = (int64_t)B * H;
    if (BH > 0x7fffffff) return cudaErrorInvalidValue;
    combine_kernel<<<(unsigned)BH, 128, 0, st>>>(o_part, lse_part, S, (int)BH, out, lse);
    return cudaGetLastError();
}

}  // namespace mla
