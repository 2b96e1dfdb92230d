// indexer.cu -- DSA lightning indexer: search-key cache append, per-position indexer scores and
// top-k selection ("DeepSeek's KV Cache: From 3.9 MB to 890 B per Token", sections "DSA: three
// things the indexer builds" (Fig. 8), "The score that picks positions" (Fig. 9) and
// "Calculating V3.2's KV cache", search key 132 B).
//
//   I(t, s) = sum_j w(t, j) ReLU(q(t, j) . k(s)),  j < 64 indexer heads, 128 dims;
//   each query keeps the (up to) K highest-scoring positions it can see.
//
// Search-key pool: 64-token pages of 8,448 B = the 64 tokens' 128 E4M3 codes (token-major) then
// their 64 fp32 scales (one per key, absmax / 448, the main cache's rule); the codes of a page are
// kept together so that every key starts on a 16-byte boundary.
//
// Scores: the keys of 128 positions (two pages) against one request's 64 head queries are one
// tensor-core contraction D[128 x 64] = codes[128 x 128] . q^T (bf16, fp32 accumulation in TMEM;
// E4M3 codes convert to bf16 exactly), and since a key's scale s >= 0,
//   I = s * sum_j w_j max(D_j, 0).
// One CTA per SM walks a balanced range of (request, 128-position) tiles: 8 converter warps load
// and convert each tile's codes and the request's q into a 3-stage ring, one warp issues the MMAs
// into two TMEM accumulators, 4 warps (thread = position = TMEM lane) finish the scores.  The pass
// is HBM-bound on the keys (132 B per position).
//
// Top-k: one CTA per request; a radix select on order-preserving keys of the fp32 scores (four
// 8-bit digits, most significant first) finds the K-th largest, then an ordered compaction writes
// the positions above it and, of those equal to it, the lowest ones, in increasing position order.
#include <cuda.h>

#include "decode_common.cuh"

namespace mla {
namespace {

using namespace ptx;
using namespace dc;

constexpr int kIdxDim = MLA_INDEX_DIM;           // 128
constexpr int kIdxHeads = MLA_INDEX_HEADS;       // 64
constexpr int kIdxPageBytes = MLA_INDEX_PAGE_BYTES;   // 8448
constexpr int kIdxScaleOff = kPage * kIdxDim;    // 8192: scales after the page's codes
constexpr int kTile = 128;                       // positions per tile (two pages)

// ------------------------------------------------------------------------------------ append

__device__ __forceinline__ uint16_t e4m3x2_rn(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;   // byte 1 = E4M3(hi), byte 0 = E4M3(lo)
}

// One warp per key: lane l owns dims 4 l .. 4 l + 3.
__global__ void __launch_bounds__(256) index_append_kernel(uint8_t* __restrict__ pool, int64_t num_pages,
                                                           const __nv_bfloat16* __restrict__ k,
                                                           const int32_t* __restrict__ slot, int64_t T,
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
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(k + row * kIdxDim) + lane);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
    float amax = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y)));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sg = __fdiv_rn(amax, 448.0f);
    uint32_t w = 0;
    if (amax != 0.0f) {
        const uint16_t lo = e4m3x2_rn(__fdiv_rn(a.y, sg), __fdiv_rn(a.x, sg));
        const uint16_t hi = e4m3x2_rn(__fdiv_rn(b.y, sg), __fdiv_rn(b.x, sg));
        w = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    uint8_t* page = pool + (s / kPage) * kIdxPageBytes;
    const int r = (int)(s % kPage);
    reinterpret_cast<uint32_t*>(page + r * kIdxDim)[lane] = w;
    if (lane == 0) reinterpret_cast<float*>(page + kIdxScaleOff)[r] = sg;
}

// ------------------------------------------------------------------------------------ scores

constexpr int kSNS = 3;                          // stages
constexpr int kConvWarps = 8;
constexpr int kSThreads = 32 * (kConvWarps + 4 + 1);   // converters, epilogue, MMA issuer
constexpr int kAChunk = kTile * 128;             // [128 positions x 64 dims] bf16, SW128
constexpr int kQChunk = kIdxHeads * 128;         // [64 heads x 64 dims] bf16, SW128
constexpr int kOffA = 0;                         // 2 chunks
constexpr int kOffQ = 2 * kAChunk;               // 32768: 2 chunks
constexpr int kOffScale = kOffQ + 2 * kQChunk;   // 49152: 128 fp32 key scales
constexpr int kOffW = kOffScale + kTile * 4;     // 49664: 64 fp32 head weights
constexpr int kOffMeta = kOffW + kIdxHeads * 4;  // 49920: request, first position, valid count
constexpr int kSStage = 50176;                   // (49920 + 16) rounded to 1 KB
constexpr int kSOffBar = kSNS * kSStage;
constexpr int kSSmem = kSOffBar + 8 * (2 * kSNS + 4 + 1) + 1024;
constexpr uint32_t kSTmemCols = 128;             // two [128 x 64] fp32 accumulators
static_assert(kOffMeta + 16 <= kSStage && kSStage % 1024 == 0, "stage layout");

struct ScoreParams {
    const uint8_t* pool;
    int64_t num_pages;
    const __nv_bfloat16* q;    // [B][64][128]
    const float* w;            // [B][64]
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* scores;             // [B][ld]
    int64_t ld;
    DevCtl* ctl;
    int max_pages;
    int max_seq_len;
    int B;
};

__device__ __forceinline__ int tiles128(int n) { return (n + kTile - 1) / kTile; }

// Balanced contiguous range of the (request, 128-position tile) stream for CTA c of C; run by one
// warp.  Returns the first tile and the tile count through shared memory.
__device__ void score_schedule(const ScoreParams& p, int c, int C, int* s_b, int* s_t, int* s_n) {
    const int lane = threadIdx.x & 31;
    const int per = (p.B + 31) / 32;
    const int b_lo = min(p.B, lane * per), b_hi = min(p.B, b_lo + per);
    long long mine = 0;
    for (int b = b_lo; b < b_hi; ++b) mine += tiles128(clamp_len(p.seq_lens[b], p.max_seq_len));
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const long long W = __shfl_sync(0xffffffffu, incl, 31);
    const long long g0 = (long long)c * W / C, g1 = (long long)(c + 1) * W / C;
    long long pre = incl - mine;
    for (int b = b_lo; b < b_hi; ++b) {
        const int nt = tiles128(clamp_len(p.seq_lens[b], p.max_seq_len));
        if (g0 < W && g0 >= pre && g0 < pre + nt) {
            *s_b = b;
            *s_t = (int)(g0 - pre);
        }
        pre += nt;
    }
    if (lane == 0) *s_n = (int)(g1 - g0);
}

struct TileCursor {
    int b, t, nt, n;
    __device__ __forceinline__ void load(const ScoreParams& p) {
        n = clamp_len(p.seq_lens[b], p.max_seq_len);
        nt = tiles128(n);
    }
    __device__ __forceinline__ void next(const ScoreParams& p) {
        ++t;
        while (t >= nt && b + 1 < p.B) {
            ++b;
            t = 0;
            load(p);
        }
    }
};

__global__ void __launch_bounds__(kSThreads, 1) indexer_score_kernel(ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_b0, s_t0, s_n;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar0 = sbase + kSOffBar;
    auto full = [&](int s) { return bar0 + 8 * s; };             // converters -> issuer
    auto empty = [&](int s) { return bar0 + 8 * (kSNS + s); };   // MMA done + epilogue done
    auto dfull = [&](int i) { return bar0 + 8 * (2 * kSNS + i); };
    auto dfree = [&](int i) { return bar0 + 8 * (2 * kSNS + 2 + i); };
    const uint32_t drain = bar0 + 8 * (2 * kSNS + 4);
    const uint32_t wait_limit = p.ctl->wait_limit;

    if (tid == 0) {
        s_abort = 0;
        s_b0 = p.B;
        s_t0 = 0;
        s_n = 0;
    }
    __syncthreads();
    if (warp == 0) score_schedule(p, blockIdx.x, gridDim.x, &s_b0, &s_t0, &s_n);
    const int iss = kConvWarps + 4;   // the MMA issuer warp
    if (tid == 32) {
        for (int s = 0; s < kSNS; ++s) {
            mbar_init(full(s), kConvWarps);
            mbar_init(empty(s), 1 + 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(dfull(i), 1);
            mbar_init(dfree(i), 4);
        }
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == iss) {
        tmem_alloc(smem_u32(&s_tmem), kSTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int n_local = s_n;
    TileCursor cur;
    cur.b = s_b0;
    cur.t = s_t0;
    if (n_local > 0) cur.load(p);

    auto fail = [&](int where) {
        s_abort = 1;
        record_error(p.ctl, MLA_ERR_TIMEOUT, 40 + where);
    };

    if (warp < kConvWarps) {
        // ------------------------------------------------------------ converters
        const int ct = tid;                 // 0 .. 255
        const int pp = ct >> 1, hf = ct & 1;   // codes: position pp, dims 64 hf .. 64 hf + 63
        const int qh = ct >> 2, qq = ct & 3;   // q: head qh, dims 32 qq .. 32 qq + 31
        for (int i = 0; i < n_local; ++i, cur.next(p)) {
            if (s_abort) break;
            const int s = i % kSNS;
            uint8_t* st = sm + s * kSStage;
            const int pos = cur.t * kTile + pp;
            const bool valid = pos < cur.n;
            // the loads go out before the wait for the stage
            uint4 raw[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                            make_uint4(0, 0, 0, 0)};
            float scale = 0.f;
            if (valid) {
                const int page = p.block_table[(size_t)cur.b * p.max_pages + (pos >> 6)];
                if (page >= 0 && page < p.num_pages) {
                    const uint8_t* pg = p.pool + (size_t)page * kIdxPageBytes;
                    const uint4* src = reinterpret_cast<const uint4*>(pg + (pos & 63) * kIdxDim + 64 * hf);
#pragma unroll
                    for (int k = 0; k < 4; ++k) raw[k] = __ldg(src + k);
                    scale = __ldg(reinterpret_cast<const float*>(pg + kIdxScaleOff) + (pos & 63));
                } else if (hf == 0) {
                    record_error(p.ctl, MLA_ERR_BOUNDS, page);
                }
            }
            uint4 qv[4];
            {
                const uint4* qs = reinterpret_cast<const uint4*>(p.q + ((size_t)cur.b * kIdxHeads + qh) * kIdxDim + 32 * qq);
#pragma unroll
                for (int k = 0; k < 4; ++k) qv[k] = __ldg(qs + k);
            }
            const float wj = ct < kIdxHeads ? __ldg(p.w + (size_t)cur.b * kIdxHeads + ct) : 0.f;
            if (i >= kSNS && !mbar_wait(empty(s), ((i / kSNS) - 1) & 1, wait_limit)) {
                if (lane == 0) fail(1);
                break;
            }
            // codes of position pp, dims 64 hf + 16 k ..: 16-byte units 2k, 2k + 1 of row pp of
            // chunk hf (unit u at u ^ (pp % 8): 128-byte swizzle)
            uint8_t* arow = st + kOffA + hf * kAChunk + pp * 128;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t o[8];
                e4m3x16_to_bf16(raw[k], o);
                st_shared_v4(arow + (((2 * k) ^ (pp & 7)) << 4), o[0], o[1], o[2], o[3]);
                st_shared_v4(arow + (((2 * k + 1) ^ (pp & 7)) << 4), o[4], o[5], o[6], o[7]);
            }
            // q of head qh, dims 32 qq ..: units 4 (qq % 2) .. + 3 of row qh of chunk qq / 2
            uint8_t* qrow = st + kOffQ + (qq >> 1) * kQChunk + qh * 128;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                st_shared_v4(qrow + (((4 * (qq & 1) + k) ^ (qh & 7)) << 4), qv[k].x, qv[k].y, qv[k].z, qv[k].w);
            if (hf == 0) reinterpret_cast<float*>(st + kOffScale)[pp] = scale;
            if (ct < kIdxHeads) reinterpret_cast<float*>(st + kOffW)[ct] = wj;
            if (ct == 0) {
                int* meta = reinterpret_cast<int*>(st + kOffMeta);
                meta[0] = cur.b;
                meta[1] = cur.t * kTile;
                meta[2] = min(kTile, cur.n - cur.t * kTile);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(full(s));
        }
    } else if (warp == iss) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_bf16(128, kIdxHeads, 0, 0);
        const uint64_t hi = smem_desc(0, 16, 1024, kSw128) & 0xFFFFFFFF00000000ull;
        const uint32_t lo = (uint32_t)smem_desc(0, 16, 1024, kSw128);
        for (int i = 0; i < n_local; ++i) {
            if (__any_sync(0xffffffffu, s_abort)) break;
            const int s = i % kSNS, d = i & 1;
            bool ok = mbar_wait(full(s), (i / kSNS) & 1, wait_limit);
            ok = ok && (i < 2 || mbar_wait(dfree(d), ((i >> 1) - 1) & 1, wait_limit));
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail(2);
                break;
            }
            tc_fence_after();
            const uint32_t a_lo = ((sbase + s * kSStage + kOffA) >> 4) & 0x3FFF;
            const uint32_t b_lo = ((sbase + s * kSStage + kOffQ) >> 4) & 0x3FFF;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kIdxDim / 16; ++kk) {
                    const uint32_t off_a = ((kk >> 2) * kAChunk + (kk & 3) * 32) >> 4;
                    const uint32_t off_b = ((kk >> 2) * kQChunk + (kk & 3) * 32) >> 4;
                    mma_bf16_ss(tmem + 64 * d, hi | (a_lo + lo + off_a), hi | (b_lo + lo + off_b), idesc,
                                kk > 0 ? 1u : 0u);
                }
                mma_commit(dfull(d));
                mma_commit(empty(s));
            }
            __syncwarp();
        }
        __syncwarp();
        if (elect_one()) {
            mma_commit(drain);
            mbar_wait(drain, 0, wait_limit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q4 = warp & 3;            // TMEM lanes 32 q4 .. 32 q4 + 31
        const int pp = q4 * 32 + lane;      // position within the tile
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        for (int i = 0; i < n_local; ++i) {
            const int s = i % kSNS, d = i & 1;
            bool ok = !s_abort && mbar_wait(dfull(d), (i >> 1) & 1, wait_limit);
            ok = ok && mbar_wait(full(s), (i / kSNS) & 1, wait_limit);   // the stage's scales, weights
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail(3);
                break;
            }
            tc_fence_after();
            uint32_t a[32], b[32];
            tmem_ld32(tmem + lane_off + 64 * d, a);
            tmem_ld32(tmem + lane_off + 64 * d + 32, b);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dfree(d));
            const uint8_t* st = sm + s * kSStage;
            const float* wv = reinterpret_cast<const float*>(st + kOffW);
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) acc = fmaf(wv[j], fmaxf(__uint_as_float(a[j]), 0.f), acc);
#pragma unroll
            for (int j = 0; j < 32; ++j) acc = fmaf(wv[32 + j], fmaxf(__uint_as_float(b[j]), 0.f), acc);
            const float score = reinterpret_cast<const float*>(st + kOffScale)[pp] * acc + 0.0f;   // (-0 -> +0)
            const int* meta = reinterpret_cast<const int*>(st + kOffMeta);
            const int rb = meta[0], base = meta[1], cnt = meta[2];
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
            if (pp < cnt) p.scores[(size_t)rb * p.ld + base + pp] = score;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == iss) tmem_dealloc(tmem, kSTmemCols);
}

// ------------------------------------------------------------------------------------ top-k

constexpr int kKThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float x) {
    const uint32_t u = __float_as_uint(x + 0.0f);        // -0 -> +0: the two zeros tie
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);   // larger float, larger key
}

// Block-wide exclusive scan of v (1024 threads); returns the prefix, *total the sum.
__device__ __forceinline__ int block_scan(int v, int* total, int* sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = sh[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        sh[32 + lane] = s;
    }
    __syncthreads();
    *total = sh[32 + 31];
    const int r = (warp > 0 ? sh[32 + warp - 1] : 0) + x - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kKThreads) topk_select_kernel(const float* __restrict__ scores, int64_t ld,
                                                                const int32_t* __restrict__ seq_lens,
                                                                int K, int32_t* __restrict__ idx) {
    __shared__ uint32_t hist[256];
    __shared__ int sh[64];
    __shared__ uint32_t s_prefix, s_mask;
    __shared__ int s_krem;
    const int b = blockIdx.x, tid = threadIdx.x;
    int64_t n = seq_lens[b];
    n = n < 0 ? 0 : (n > ld ? ld : n);
    const float* row = scores + (size_t)b * ld;
    int32_t* out = idx + (size_t)b * K;
    if (n <= K) {
        for (int t = tid; t < K; t += kKThreads) out[t] = t < n ? t : -1;
        return;
    }
    if (tid == 0) {
        s_prefix = 0;
        s_mask = 0;
        s_krem = K;
    }
    // the K-th largest key, one 8-bit digit at a time (most significant first): krem counts the
    // keys still to take among those matching the prefix
    for (int level = 0; level < 4; ++level) {
        const int shift = 24 - 8 * level;
        for (int j = tid; j < 256; j += kKThreads) hist[j] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix, mask = s_mask;
        for (int64_t t = tid; t < n; t += kKThreads) {
            const uint32_t key = order_key(row[t]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid == 0) {
            int krem = s_krem;
            int dsel = 0;
            for (int dg = 255; dg >= 0; --dg) {
                const int c = (int)hist[dg];
                if (c >= krem) {
                    dsel = dg;
                    break;
                }
                krem -= c;
            }
            s_krem = krem;
            s_prefix = prefix | ((uint32_t)dsel << shift);
            s_mask = mask | (255u << shift);
        }
        __syncthreads();
    }
    const uint32_t T = s_prefix;
    const int krem = s_krem;   // keys equal to T to take, lowest positions first
    // ordered compaction, 4 consecutive positions per thread per round
    int base = 0, eq_seen = 0;
    for (int64_t c0 = 0; c0 < n; c0 += 4 * kKThreads) {
        const int64_t t0 = c0 + 4 * tid;
        uint32_t key[4];
        int n_eq = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            key[e] = t0 + e < n ? order_key(row[t0 + e]) : 0u;
            n_eq += (t0 + e < n && key[e] == T) ? 1 : 0;
        }
        int eq_total;
        const int eq_before = eq_seen + block_scan(n_eq, &eq_total, sh);
        int take[4], n_take = 0, r = eq_before;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool in = t0 + e < n;
            const bool gt = in && key[e] > T;
            const bool eq = in && key[e] == T;
            take[e] = gt || (eq && r < krem);
            r += eq ? 1 : 0;
            n_take += take[e];
        }
        int take_total;
        int w = base + block_scan(n_take, &take_total, sh);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (take[e]) out[w++] = (int32_t)(t0 + e);
        base += take_total;
        eq_seen += eq_total;
    }
}

}  // namespace

cudaError_t launch_index_append(uint8_t* pool, int64_t num_pages, const __nv_bfloat16* k, const int32_t* slot,
                                int64_t T, DevCtl* ctl, cudaStream_t st) {
    const int64_t blocks = (T + 7) / 8;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    index_append_kernel<<<(unsigned)blocks, 256, 0, st>>>(pool, num_pages, k, slot, T, ctl);
    return cudaGetLastError();
}

cudaError_t launch_indexer_score(const uint8_t* pool, int64_t num_pages, const __nv_bfloat16* q, const float* w,
                                 const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                                 int max_seq_len, float* scores, DevCtl* ctl, cudaStream_t st) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(indexer_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    ScoreParams p;
    p.pool = pool;
    p.num_pages = num_pages;
    p.q = q;
    p.w = w;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.scores = scores;
    p.ld = max_seq_len;
    p.ctl = ctl;
    p.max_pages = max_pages;
    p.max_seq_len = max_seq_len;
    p.B = B;
    const long long max_tiles = (long long)B * ((max_seq_len + kTile - 1) / kTile);
    int sms = num_sms();
    if (sms <= 0) sms = 152;
    const int C = (int)(max_tiles < sms ? (max_tiles < 1 ? 1 : max_tiles) : sms);
    indexer_score_kernel<<<C, kSThreads, kSSmem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_topk_select(const float* scores, int64_t ld, const int32_t* seq_lens, int B, int K,
                               int32_t* idx, cudaStream_t st) {
    topk_select_kernel<<<B, kKThreads, 0, st>>>(scores, ld, seq_lens, K, idx);
    return cudaGetLastError();
}

}  // namespace mla
