// decode_common.cuh -- pieces shared by the tensor-core decode kernels: the balanced tile
// schedule over a batch, the cursor that walks a cluster's tiles request by request, and small
// device helpers.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "mla_internal.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace dc {

constexpr int kT = 64;                  // positions per tile (a cache page, or 64 top-k entries)
constexpr int kMinTilesPerCluster = 4;

__device__ __forceinline__ void fail(DevCtl* ctl, volatile int* abort_flag, int where) {
    *abort_flag = 1;
    record_error(ctl, MLA_ERR_TIMEOUT, where);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ int clamp_len(int n, int max_len) {
    return n < 0 ? 0 : (n > max_len ? max_len : n);
}

// Tiles of request b: its visible positions in pages of 64 (dense), or its top-k list in groups
// of 64 entries (sparse: the list length is the same for every request).
__device__ __forceinline__ int tiles_of(int n, int topk) {
    return topk > 0 ? (topk + kT - 1) / kT : (n + kT - 1) / kT;
}

// Walks the tiles of one cluster's range: request b, tile t of that request, local tile index j
// of n_loc.  Six ints (the request table and limits are passed in), as several copies stay live in
// the softmax warps' registers.
struct Cursor {
    int b, t, nt, n;   // request, its tile, its tiles, its visible positions
    int j, n_loc;      // local tile index, tiles in the range
    __device__ __forceinline__ void load_req(const int32_t* seq_lens, int max_len, int topk) {
        n = clamp_len(seq_lens[b], max_len);
        nt = tiles_of(n, topk);
    }
    __device__ __forceinline__ void init(const int32_t* seq_lens, int max_len, int topk, int b0, int t0,
                                         int n_local) {
        b = b0, t = t0, j = 0, n_loc = n_local;
        if (n_loc > 0) load_req(seq_lens, max_len, topk);
        else n = nt = 0;
    }
    __device__ __forceinline__ bool first() const { return t == 0 || j == 0; }
    __device__ __forceinline__ bool last() const { return t == nt - 1 || j == n_loc - 1; }
    __device__ __forceinline__ void next(const int32_t* seq_lens, int max_len, int B, int topk) {
        ++j;
        ++t;
        if (j >= n_loc) return;
        while (t >= nt && b + 1 < B) {
            ++b;
            t = 0;
            load_req(seq_lens, max_len, topk);
        }
    }
};

// Cluster of stream index x when cluster c of C owns [floor(c W / C), floor((c + 1) W / C)).
__device__ __forceinline__ int cluster_of(long long x, long long W, int C) {
    long long c = ((x + 1) * C + W - 1) / W - 1;
    return (int)(c < 0 ? 0 : (c > C - 1 ? C - 1 : c));
}

// The balanced schedule, run by one warp of every CTA.  The requests form one stream in which
// request b > 0 takes seg_cost "start" units followed by its tiles (a request with no tiles takes
// none; request 0 starts with the kernel): the units stand for the fixed cost of starting a
// segment inside a cluster's range (the epilogue of the one before, the new request's first
// page), so that a cluster whose range holds more request starts gets fewer tiles.  With W units in all, cluster c takes units [c W / C, (c + 1) W / C) and processes
// the tiles among them.  Returns this cluster's tile count and first tile (request, tile).
// Cluster 0's rank-0 CTA also records, per request, where its partials are: meta[2b] = the first
// partial slot (2 c_lo if the request is that cluster's first segment, else 2 c_lo + 1; -1 for a
// request with no tiles), meta[2b + 1] = the last cluster whose range holds one of its tiles.
__device__ __forceinline__ void schedule_warp(const int32_t* seq_lens, int max_len, int B, int topk,
                                              int seg_cost, int c, int C, bool record, int32_t* meta,
                                              DevCtl* ctl, int* n_local, int* start_b, int* start_t) {
    const int lane = threadIdx.x & 31;
    const int per = (B + 31) / 32;
    const int b_lo = min(B, lane * per), b_hi = min(B, b_lo + per);
    long long mine = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        const int raw = seq_lens[b];
        if ((raw < 0 || raw > max_len) && record) record_error(ctl, MLA_ERR_BOUNDS, b);
        const int nt = tiles_of(clamp_len(raw, max_len), topk);
        mine += nt > 0 ? nt + (b > 0 ? seg_cost : 0) : 0;
    }
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const long long W = __shfl_sync(0xffffffffu, incl, 31);
    const long long g0 = (long long)c * W / C, g1 = (long long)(c + 1) * W / C;
    long long v = incl - mine;   // start unit of request b
    int cnt = 0, fb = B, ft = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        const int nt = tiles_of(clamp_len(seq_lens[b], max_len), topk);
        if (nt == 0) {
            if (record) {
                meta[2 * b] = -1;
                meta[2 * b + 1] = -1;
            }
            continue;
        }
        const int sc = b > 0 ? seg_cost : 0;
        const long long t0 = v + sc;   // unit of the request's tile 0
        // tiles t with t0 + t in [g0, g1)
        const long long lo_t = g0 - t0 < 0 ? 0 : (g0 - t0 > nt ? nt : g0 - t0);
        const long long hi_t = g1 - t0 < 0 ? 0 : (g1 - t0 > nt ? nt : g1 - t0);
        if (hi_t > lo_t) {
            if (fb == B) {
                fb = b;
                ft = (int)lo_t;
            }
            cnt += (int)(hi_t - lo_t);
        }
        if (record) {
            const int clo = cluster_of(t0, W, C), chi = cluster_of(t0 + nt - 1, W, C);
            // the request is cluster clo's first segment iff clo's range starts at or after the
            // request's start units (the unit before them is the previous request's last tile)
            const bool starts = (long long)clo * W / C >= v;
            meta[2 * b] = 2 * clo + (starts ? 0 : 1);
            meta[2 * b + 1] = chi;
        }
        v += nt + sc;
    }
    // the first request (lowest b) with tiles in range, and the total
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const int ob = __shfl_xor_sync(0xffffffffu, fb, o);
        const int ot = __shfl_xor_sync(0xffffffffu, ft, o);
        if (ob < fb) {
            fb = ob;
            ft = ot;
        }
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    }
    if (lane == 0) {
        *n_local = cnt;
        *start_b = fb;
        *start_t = ft;
    }
}

// 4 bytes into the peer's shared memory, completing tx-bytes on its barrier.
__device__ __forceinline__ void st_async_b32(uint32_t remote_addr, uint32_t remote_bar, uint32_t v) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                     remote_addr),
                 "r"(v), "r"(remote_bar)
                 : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

// Two fp32 values to an f16 pair (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// A bf16 pair to an f16 pair: exact for magnitudes in the f16 normal range.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// non-zero when either f16 half is an infinity or a NaN (exponent field all ones)
__device__ __forceinline__ uint32_t f16x2_inf_or_nan(uint32_t v) {
    return ((v & 0x7C00u) == 0x7C00u) | ((v & 0x7C000000u) == 0x7C000000u);
}

// 16 e4m3 codes (OCP 8-bit floating point, bias 7) to 16 f16 values, exactly: every e4m3 value
// (normal or subnormal, at most 448) is an f16 value.
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 c, uint32_t (&o)[8]) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int j = 0; j < 2; ++j)
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o[2 * k + j]) : "h"((uint16_t)(w[k] >> (16 * j))));
}

// Clusters for a batch: at most one per SM pair, at least kMinTilesPerCluster tiles each.
inline int clusters_for_tiles(long long w_max, int sms) {
    long long c = sms / 2;
    const long long by_work = (w_max + kMinTilesPerCluster - 1) / kMinTilesPerCluster;
    if (by_work < c) c = by_work;
    return c < 1 ? 1 : (int)c;
}

// One E4M3 code (the low byte of `code`) as a float, exactly.
__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)(code & 0xFFu)));
    return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// 16 e4m3 codes times a power-of-two scale to 16 bf16 values (pairs, low half first), exactly:
// an E4M3 value has at most 4 significant bits and the scale only moves its exponent.
__device__ __forceinline__ void e4m3x16_scaled_bf16(const uint4 c, float s, uint32_t (&o)[8]) {
    uint32_t h[8];
    e4m3x16_to_f16(c, h);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[k]));
        o[k] = pack_bf16x2(f.x * s, f.y * s);
    }
}

// 32 E2M1 codes (16 bytes; byte i holds dims 2i in its low and 2i + 1 in its high nibble) times an
// E4M3 scale value (s0 for bytes 0-7, s1 for bytes 8-15) to 32 bf16 values, exactly: an E2M1 value
// times an E4M3 value has at most 5 significant bits, well inside bf16's range.
__device__ __forceinline__ void e2m1x32_scaled_bf16(const uint4 c, float s0, float s1, uint32_t (&o)[16]) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t h;
            asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
                : "=r"(h)
                : "r"((w[k] >> (8 * j)) & 0xFFu));
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
            const float sc = k < 2 ? s0 : s1;
            o[4 * k + j] = pack_bf16x2(f.x * sc, f.y * sc);
        }
}

}  // namespace dc

// Shared by the tensor-core decode kernels (defined in decode_tc.cu): the merge of split
// requests' partial slots into the output (B requests, C clusters), on stream st.
cudaError_t launch_merge_slots(const float* o_part, const float* lse_part, const int32_t* meta,
                               __nv_bfloat16* out, float* lse, int B, int C, cudaStream_t st,
                               const float* sink = nullptr);
bool encode_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
               uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw,
               CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
// 3D tiled tensor map (dims innermost first, byte strides of dims 1 and 2).
bool encode_3d(CUtensorMap* m, const void* base, const uint64_t dims[3], const uint64_t strides_bytes[2],
               const uint32_t box[3], CUtensorMapSwizzle sw, CUtensorMapDataType dt);

}  // namespace mla
