// append.cu -- write new latent tokens into the paged pool (BF16 record or FP8 mixed record), and
// new shared K = V entries (V4 or V4.1 entry).
//
// BF16 record (1,152 B): [c_KV 512 bf16 | k_rope 64 bf16]
//   ("DeepSeek's KV Cache: From 3.9 MB to 890 B per Token", "Calculating V2's KV cache").
// FP8 mixed record (656 B): [512 E4M3 codes | 4 fp32 scales, one per 128 dims | 64 bf16 rope]
//   (same page, "Calculating V3.2's KV cache"); scale = absmax / 448 so the largest magnitude of
//   each group lands on the largest finite E4M3 value.
//
// One warp per token row.  Lane l owns latent dims [16 l, 16 l + 16) and rope dims [2 l, 2 l + 2):
// reads are 32 B (latent) + 4 B (rope) per lane, fully coalesced; an FP8 group of 128 dims is
// owned by 8 consecutive lanes, so its absmax is three xor-shuffles.  The row is HBM-bound and
// tiny next to decode.
#include "mla_internal.cuh"

namespace mla {
namespace {

__device__ __forceinline__ uint16_t e4m3x2(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;   // byte 1 = E4M3(hi), byte 0 = E4M3(lo)
}

__global__ void __launch_bounds__(256) cache_append_kernel(
    int fmt, uint8_t* __restrict__ pool, int64_t num_pages, const __nv_bfloat16* __restrict__ c_kv,
    const __nv_bfloat16* __restrict__ k_rope, const int32_t* __restrict__ slot, int64_t T,
    DevCtl* ctl) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= T) return;
    const int64_t s = slot[row];
    if (s < 0) return;
    if (s >= num_pages * kPage) {
        if (lane == 0) record_error(ctl, MLA_ERR_BOUNDS, (int)(s / kPage));
        return;
    }
    // 16 latent values (32 B) and 2 rope values (4 B) per lane
    const uint4* src = reinterpret_cast<const uint4*>(c_kv + row * kDc) + lane * 2;
    uint4 v0 = __ldg(src);
    uint4 v1 = __ldg(src + 1);
    uint32_t rope = __ldg(reinterpret_cast<const uint32_t*>(k_rope + row * kDr) + lane);

    if (fmt == MLA_KV_BF16) {
        uint8_t* rec = pool + s * kBf16RecordBytes;
        uint4* dst = reinterpret_cast<uint4*>(rec) + lane * 2;
        dst[0] = v0;
        dst[1] = v1;
        reinterpret_cast<uint32_t*>(rec + kDc * 2)[lane] = rope;
        return;
    }

    uint8_t* rec = pool + s * kFp8RecordBytes;
    float x[16];
    const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&v0);
    const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&v1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 a = __bfloat1622float2(h0[i]);
        float2 b = __bfloat1622float2(h1[i]);
        x[2 * i] = a.x;
        x[2 * i + 1] = a.y;
        x[8 + 2 * i] = b.x;
        x[8 + 2 * i + 1] = b.y;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const float sg = __fdiv_rn(amax, 448.0f);
    uint32_t packed[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t w = 0;
        if (amax != 0.0f) {
            uint16_t lo = e4m3x2(__fdiv_rn(x[4 * i + 1], sg), __fdiv_rn(x[4 * i], sg));
            uint16_t hi = e4m3x2(__fdiv_rn(x[4 * i + 3], sg), __fdiv_rn(x[4 * i + 2], sg));
            w = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        packed[i] = w;
    }
    // 656-byte records are only 16-byte aligned: 16 codes per lane go out as one 16-byte store.
    *reinterpret_cast<uint4*>(rec + lane * 16) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if ((lane & 7) == 0) reinterpret_cast<float*>(rec + kFp8ScaleOff)[lane >> 3] = sg;
    reinterpret_cast<uint32_t*>(rec + kFp8RopeOff)[lane] = rope;
}

// Shared K = V entries ("DeepSeek's KV Cache", section "HCA: 128 tokens into one", Fig. 15), one
// warp per entry, lane l owning dims [16 l, 16 l + 16).
//   V4 (584 B, "Calculating V4-Flash's KV cache"): dims 0..447 in E4M3 with one UE8M0 scale per 64
//   dims (4 lanes: two xor-shuffles for the group's absmax), the scale the smallest power of two
//   2^e with 448 * 2^e >= amax, stored as the byte e + 127; dims 448..511 (lanes 28..31) copied as
//   bf16.  The page holds codes [64][448], RoPE [64][128 B], scale bytes [64][8] (the 8th is 0).
//   V4.1 (288 B, "Calculating V4.1-Flash's KV cache"): dims in E2M1 with one E4M3 scale per 16
//   dims (one lane per group), s = E4M3(amax / 6); dims 2i, 2i + 1 share a byte, 2i in the low
//   nibble; the 32 scale bytes follow the 256 code bytes.
__device__ __forceinline__ uint32_t e2m1x2(float hi, float lo) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;   // high nibble = E2M1(hi), low nibble = E2M1(lo)
}

__global__ void __launch_bounds__(256) shared_append_kernel(
    int fmt, uint8_t* __restrict__ pool, int64_t num_pages, const __nv_bfloat16* __restrict__ entry,
    const int32_t* __restrict__ slot, int64_t T, DevCtl* ctl) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= T) return;
    const int64_t s = slot[row];
    if (s < 0) return;
    if (s >= num_pages * kPage) {
        if (lane == 0) record_error(ctl, MLA_ERR_BOUNDS, (int)(s / kPage));
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(entry + row * kE) + lane * 2;
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    float x[16];
    const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&v0);
    const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&v1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 a = __bfloat1622float2(h0[i]), b = __bfloat1622float2(h1[i]);
        x[2 * i] = a.x;
        x[2 * i + 1] = a.y;
        x[8 + 2 * i] = b.x;
        x[8 + 2 * i + 1] = b.y;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    if (fmt == MLA_KV_V4_FP8) {
        uint8_t* base = pool + (s / kPage) * kV4PageBytes;
        const int prow = (int)(s % kPage);
        if (lane >= kENope / 16) {   // RoPE dims: stored as given
            uint4* dst = reinterpret_cast<uint4*>(base + kV4RopeOff + prow * 128 + (lane - kENope / 16) * 32);
            dst[0] = v0;
            dst[1] = v1;
            if (lane == kENope / 16) base[kV4ScaleOff + prow * 8 + 7] = 0;   // pad byte
            amax = 0.0f;
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        if (lane >= kENope / 16) return;
        // smallest e with 448 * 2^e >= amax: amax = f 2^k with f in [0.5, 1) and 448 = 0.875 2^9
        int e = -127;
        if (amax > 0.0f) {
            int k;
            const float f = frexpf(amax, &k);
            e = k - 9 + (f > 0.875f ? 1 : 0);
            e = e < -127 ? -127 : (e > 127 ? 127 : e);
        }
        const float inv = ldexpf(1.0f, -e);   // exact: 2^-e is a float for e in [-127, 127]
        uint32_t packed[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t w = 0;
            if (amax > 0.0f) {
                const uint16_t lo = e4m3x2(x[4 * i + 1] * inv, x[4 * i] * inv);
                const uint16_t hi = e4m3x2(x[4 * i + 3] * inv, x[4 * i + 2] * inv);
                w = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            packed[i] = w;
        }
        *reinterpret_cast<uint4*>(base + prow * kENope + lane * 16) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        if ((lane & 3) == 0) base[kV4ScaleOff + prow * 8 + (lane >> 2)] = amax > 0.0f ? (uint8_t)(e + 127) : 0;
        return;
    }
    // V4.1: lane = one group of 16 dims
    uint8_t* rec = pool + s * kV41EntryBytes;
    const uint32_t sc = e4m3x2(0.0f, __fdiv_rn(amax, 6.0f)) & 0xFFu;
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)sc));
    const float sv = __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
    uint32_t w0 = 0, w1 = 0;
    if (sv != 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            w0 |= e2m1x2(__fdiv_rn(x[2 * i + 1], sv), __fdiv_rn(x[2 * i], sv)) << (8 * i);
            w1 |= e2m1x2(__fdiv_rn(x[8 + 2 * i + 1], sv), __fdiv_rn(x[8 + 2 * i], sv)) << (8 * i);
        }
    }
    *reinterpret_cast<uint2*>(rec + lane * 8) = make_uint2(w0, w1);
    rec[kV41ScaleOff + lane] = (uint8_t)sc;
}

__global__ void e4m3_encode_kernel(const float* __restrict__ x, uint8_t* __restrict__ codes,
                                   int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        codes[i] = (uint8_t)(e4m3x2(0.0f, x[i]) & 0xFF);
}

}  // namespace

cudaError_t launch_cache_append(int fmt, uint8_t* pool, int64_t num_pages,
                                const __nv_bfloat16* c_kv, const __nv_bfloat16* k_rope,
                                const int32_t* slot, int64_t T, DevCtl* ctl, cudaStream_t st) {
    const int rows_per_block = 8;
    int64_t blocks = (T + rows_per_block - 1) / rows_per_block;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    cache_append_kernel<<<(unsigned)blocks, 32 * rows_per_block, 0, st>>>(fmt, pool, num_pages, c_kv,
                                                                          k_rope, slot, T, ctl);
    return cudaGetLastError();
}

cudaError_t launch_shared_append(int fmt, uint8_t* pool, int64_t num_pages, const __nv_bfloat16* entry,
                                 const int32_t* slot, int64_t T, DevCtl* ctl, cudaStream_t st) {
    const int rows_per_block = 8;
    int64_t blocks = (T + rows_per_block - 1) / rows_per_block;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    shared_append_kernel<<<(unsigned)blocks, 32 * rows_per_block, 0, st>>>(fmt, pool, num_pages, entry, slot, T, ctl);
    return cudaGetLastError();
}

cudaError_t launch_e4m3_encode(const float* x, uint8_t* codes, int64_t n, cudaStream_t st) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    e4m3_encode_kernel<<<(unsigned)blocks, 256, 0, st>>>(x, codes, n);
    return cudaGetLastError();
}

}  // namespace mla
