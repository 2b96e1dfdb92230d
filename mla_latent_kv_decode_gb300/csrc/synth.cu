// synth.cu -- device twin of the seeded input generator of mla_latent_kv_decode_gb300/synth.py.
//
// Not part of libmla: it only draws synthetic inputs too large to draw on the host.  Word i of
// a (seed, stream) sequence is the splitmix64 output function applied to key + (i + 1) * golden
// (Steele, Lea & Flood, OOPSLA 2014); value i is the Irwin-Hall sum of the twelve 16-bit fields
// of words 3i, 3i+1, 3i+2, mapped to (S - 393210) / 65536 (exact in fp32) and rounded to bf16.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__global__ void normal_bf16_kernel(__nv_bfloat16* __restrict__ dst, int64_t rows, uint64_t key,
                                   int64_t first_index, int64_t row_len, int64_t row_stride_index) {
    const int64_t n = rows * row_len;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
        const int64_t r = e / row_len, j = e % row_len;
        const uint64_t idx = (uint64_t)(first_index + r * row_stride_index + j);
        int32_t s = 0;
#pragma unroll
        for (int w = 0; w < 3; ++w) {
            const uint64_t x = mix64(key + (3 * idx + w + 1) * 0x9E3779B97F4A7C15ull);
            s += (int32_t)(x & 0xFFFF) + (int32_t)((x >> 16) & 0xFFFF) +
                 (int32_t)((x >> 32) & 0xFFFF) + (int32_t)(x >> 48);
        }
        const float z = (float)(s - 393210) / 65536.0f;   // exact: |s - 393210| < 2^20
        dst[e] = __float2bfloat16_rn(z);
    }
}

}  // namespace

extern "C" int synth_normal_bf16(void* dst, int64_t rows, uint64_t key, uint64_t unused,
                                 int64_t first_index, int64_t row_len, int64_t row_stride_index,
                                 cudaStream_t stream) {
    (void)unused;
    if (rows <= 0 || row_len <= 0) return 0;
    int64_t n = rows * row_len;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    normal_bf16_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<__nv_bfloat16*>(dst), rows,
                                                           key, first_index, row_len,
                                                           row_stride_index);
    return (int)cudaGetLastError();
}
