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
// tensor-core contraction D[128 x 64] = codes[128 x 128] . q^T (f16 operands, exact products,
// fp32 accumulation in TMEM), and since a key's scale s >= 0,
//   I = s * sum_j w_j max(D_j, 0).
// One CTA per SM walks a balanced range of (request, 128-position) tiles.  A producer thread
// loads whole pages into an 8-deep shared-memory ring by TMA; converter warps turn the E4M3 codes
// into f16 straight in tensor memory (the MMA's A operand); one warp issues the MMAs; 4 warps
// (thread = position = TMEM lane) finish the scores.  The pass is HBM-bound on the keys (132 B per
// position).
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

// Warp roles: 8 converter warps in two groups of 4 (group g converts the tiles i = g mod 2; warp
// w of a group owns TMEM lanes 32 (w % 4) ..), 4 epilogue warps, the MMA issuer, the producer.
constexpr int kConvWarps = 8;
constexpr int kIssWarp = kConvWarps + 4;
constexpr int kProdWarp = kConvWarps + 5;
constexpr int kSThreads = 32 * (kConvWarps + 6);
constexpr int kNR = 8;                           // raw page slots (tiles in flight)
constexpr int kNS = 4;                           // q / scale / weight stages
constexpr int kNA = 4;                           // A operands in tensor memory
constexpr int kND = 2;                           // accumulators in tensor memory
constexpr int kLookup = 8;                       // tiles whose pages the producer looks up together
// raw slot: the tile's two pages' codes (64 rows x 128 B each, 128-byte swizzle) then their scales
constexpr int kSlotScales = 2 * kPage * kIdxDim;       // 16384
constexpr int kSlot = 17408;                            // 16384 + 2 x 256 rounded to 1 KB
// stage: q as the MMA's B operand ([64 heads x 64 dims] f16 per chunk, two chunks, SW128),
// the tile's 128 key scales, the 64 head weights, request / first position / count
constexpr int kQChunk = kIdxHeads * 128;
constexpr int kStQ = 0;
constexpr int kStScale = 2 * kQChunk;                   // 16384
constexpr int kStW = kStScale + kTile * 4;              // 16896
constexpr int kStMeta = kStW + kIdxHeads * 4;           // 17152
constexpr int kStage = 17408;
constexpr int kSOffStage = kNR * kSlot;                 // 139264
constexpr int kSOffEntry = kSOffStage + kNS * kStage;   // 208896: per raw slot {b, base, cnt, -}
constexpr int kSOffBar = kSOffEntry + kNR * 16;
constexpr int kNBars = 2 * kNR + 2 * kNS + kNA + 2 * kND + 1;
constexpr int kSSmem = kSOffBar + 8 * kNBars + 1024;
constexpr uint32_t kSTmemCols = 512;                    // A: 4 x 64 columns, D: 2 x 64 columns
constexpr uint32_t kTmemD = 64 * kNA;
static_assert(kSlotScales + 2 * 256 <= kSlot && kSlot % 1024 == 0, "raw slot");
static_assert(kStMeta + 16 <= kStage && kStage % 1024 == 0, "stage layout");
static_assert(kSSmem <= 232448, "shared memory");
static_assert(kNR % 2 == 0 && kNS % 2 == 0 && kNA % 2 == 0, "rings shared by two converter groups");
static_assert(kTmemD + 64 * kND <= kSTmemCols, "tensor memory");

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

// Two E4M3 codes (bits 15:8 and 7:0) to f16x2 (high half, low half), exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)v));
    return r;
}

__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// Scores of a balanced range of (request, 128-position) tiles per CTA.
//   producer: looks up each tile's two pages (checked) and loads them whole into a raw slot (the
//             codes by a 3D tensor map with a 128-byte swizzle, the scales by a bulk copy);
//   converters: E4M3 codes -> f16 (exact) straight into tensor memory as the MMA's A operand
//             (row = position, two dims per column), key scales into the stage, and on a request
//             change the request's q (scaled per head by 2^e into [2^14, 2^15) of f16, the head
//             weight by 2^-e: the products w ReLU(q . k) are unchanged, and every bf16 q element
//             not 2^31 below its head's largest is exact in f16);
//   issuer:   D[128 x 64] = A[128 x 128] . q^T, eight K=16 MMAs;
//   epilogue: thread = position = TMEM lane: I = s * sum_j w_j max(D_j, 0).
__global__ void __launch_bounds__(kSThreads, 1)
    indexer_score_kernel(const __grid_constant__ CUtensorMap tm_codes, ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_b0, s_t0, s_n;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar0 = sbase + kSOffBar;
    auto raw_full = [&](int r) { return bar0 + 8 * r; };
    auto raw_empty = [&](int r) { return bar0 + 8 * (kNR + r); };
    auto full = [&](int s) { return bar0 + 8 * (2 * kNR + s); };
    auto empty = [&](int s) { return bar0 + 8 * (2 * kNR + kNS + s); };
    auto afree = [&](int a) { return bar0 + 8 * (2 * kNR + 2 * kNS + a); };
    auto dfull = [&](int d) { return bar0 + 8 * (2 * kNR + 2 * kNS + kNA + d); };
    auto dfree = [&](int d) { return bar0 + 8 * (2 * kNR + 2 * kNS + kNA + kND + d); };
    const uint32_t drain = bar0 + 8 * (kNBars - 1);
    int4* entry = reinterpret_cast<int4*>(sm + kSOffEntry);
    const uint32_t wait_limit = p.ctl->wait_limit;

    if (tid == 0) {
        s_abort = 0;
        s_b0 = p.B;
        s_t0 = 0;
        s_n = 0;
    }
    __syncthreads();
    if (warp == 0) score_schedule(p, blockIdx.x, gridDim.x, &s_b0, &s_t0, &s_n);
    if (tid == 32) {
        for (int r = 0; r < kNR; ++r) {
            mbar_init(raw_full(r), 1);
            mbar_init(raw_empty(r), 4);
        }
        for (int s = 0; s < kNS; ++s) {
            mbar_init(full(s), 4);
            mbar_init(empty(s), 1 + 4);
        }
        for (int a = 0; a < kNA; ++a) mbar_init(afree(a), 1);
        for (int d = 0; d < kND; ++d) {
            mbar_init(dfull(d), 1);
            mbar_init(dfree(d), 4);
        }
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == kIssWarp) {
        tmem_alloc(smem_u32(&s_tmem), kSTmemCols);
        tmem_relinquish();
    }
    if (tid == kProdWarp * 32) tma_prefetch_desc(&tm_codes);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int n_local = s_n;

    auto fail = [&](int where) {
        s_abort = 1;
        record_error(p.ctl, MLA_ERR_TIMEOUT, 40 + where);
    };

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n_local > 0) {
            TileCursor pf;
            pf.b = s_b0;
            pf.t = s_t0;
            pf.load(p);
            int issued = 0;
            for (int j0 = 0; j0 < n_local && !s_abort; j0 += kLookup) {
                const int jn = min(kLookup, n_local - j0);
                int eb[kLookup], ebase[kLookup], ecnt[kLookup], pg0[kLookup], pg1[kLookup];
#pragma unroll
                for (int k = 0; k < kLookup; ++k) {
                    eb[k] = pf.b;
                    ebase[k] = pf.t * kTile;
                    ecnt[k] = min(kTile, pf.n - ebase[k]);
                    if (k + 1 < jn) pf.next(p);
                }
#pragma unroll
                for (int k = 0; k < kLookup; ++k) {   // the lookups go out together
                    pg0[k] = pg1[k] = -1;
                    if (k < jn) {
                        const int32_t* row = p.block_table + (size_t)eb[k] * p.max_pages + (ebase[k] >> 6);
                        pg0[k] = row[0];
                        if (ecnt[k] > 64) pg1[k] = row[1];
                    }
                }
                bool ok = true;
#pragma unroll
                for (int k = 0; k < kLookup; ++k) {
                    if (k >= jn || !ok) continue;
                    const int j = j0 + k, r = j % kNR;
                    if (j >= kNR && !mbar_wait(raw_empty(r), ((j / kNR) - 1) & 1, wait_limit)) {
                        fail(4);
                        ok = false;
                        continue;
                    }
                    int pg[2] = {pg0[k], pg1[k]};
                    uint32_t bytes = 0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h == 1 && ecnt[k] <= 64) continue;
                        if (pg[h] < 0 || pg[h] >= p.num_pages) {
                            record_error(p.ctl, MLA_ERR_BOUNDS, pg[h]);
                            pg[h] = -1;
                        } else {
                            bytes += kPage * kIdxDim + kPage * 4;
                        }
                    }
                    entry[r] = make_int4(eb[k], ebase[k], ecnt[k], 0);
                    const uint32_t slot = sbase + r * kSlot;
                    mbar_arrive_expect_tx(raw_full(r), bytes);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (pg[h] < 0) continue;
                        tma_load_3d(slot + h * kPage * kIdxDim, &tm_codes, raw_full(r), 0, 0, pg[h]);
                        bulk_load(slot + kSlotScales + h * 256, p.pool + (size_t)pg[h] * kIdxPageBytes + kIdxScaleOff,
                                  kPage * 4, raw_full(r));
                    }
                    issued = j + 1;
                }
                if (!ok) break;
                if (j0 + jn < n_local) pf.next(p);
            }
            // nothing of this CTA's copies is left in flight when it exits
            for (int j = max(0, issued - kNR); j < issued; ++j)
                if (!mbar_wait(raw_full(j % kNR), (j / kNR) & 1, wait_limit)) fail(6);
        }
        __syncwarp();
    } else if (warp < kConvWarps) {
        // ------------------------------------------------------------ converters
        const int g = warp >> 2, q4 = warp & 3;
        const int gt = tid & 127;             // thread within the group
        const int pp = q4 * 32 + lane;        // position = TMEM lane
        const int h = pp >> 6, rr = pp & 63;  // page of the tile, row of the page
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        int qh1 = -1, qh2 = -1;               // requests of this group's previous two tiles
        for (int i = g; i < n_local; i += 2) {
            if (s_abort) break;
            const int s = i % kNS, r = i % kNR, a = i % kNA;
            if (!mbar_wait(raw_full(r), (i / kNR) & 1, wait_limit)) {
                if (lane == 0) fail(1);
                break;
            }
            const int4 en = entry[r];
            const uint32_t rowa = sbase + r * kSlot + h * kPage * kIdxDim + rr * kIdxDim;
            uint4 u[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) u[c] = ld_shared_v4(rowa + ((c ^ (rr & 7)) << 4));
            const float sc = *reinterpret_cast<const float*>(sm + r * kSlot + kSlotScales + h * 256 + rr * 4);
            __syncwarp();
            if (lane == 0) mbar_arrive(raw_empty(r));
            const bool new_q = qh2 != en.x;
            qh2 = qh1;
            qh1 = en.x;
            if (i >= kNA && !mbar_wait(afree(a), ((i / kNA) - 1) & 1, wait_limit)) {
                if (lane == 0) fail(2);
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t o[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = u[4 * half + c];
                    o[8 * c + 0] = e4m3x2_to_f16x2(v.x);
                    o[8 * c + 1] = e4m3x2_to_f16x2(v.x >> 16);
                    o[8 * c + 2] = e4m3x2_to_f16x2(v.y);
                    o[8 * c + 3] = e4m3x2_to_f16x2(v.y >> 16);
                    o[8 * c + 4] = e4m3x2_to_f16x2(v.z);
                    o[8 * c + 5] = e4m3x2_to_f16x2(v.z >> 16);
                    o[8 * c + 6] = e4m3x2_to_f16x2(v.w);
                    o[8 * c + 7] = e4m3x2_to_f16x2(v.w >> 16);
                }
                tmem_st32(tmem + lane_off + 64 * a + 32 * half, o);
            }
            uint4 qv[8];
            if (new_q) {
                const uint4* qs = reinterpret_cast<const uint4*>(p.q + (size_t)en.x * kIdxHeads * kIdxDim);
#pragma unroll
                for (int k = 0; k < 8; ++k) qv[k] = __ldg(qs + gt + 128 * k);
            }
            if (i >= kNS && !mbar_wait(empty(s), ((i / kNS) - 1) & 1, wait_limit)) {
                if (lane == 0) fail(3);
                break;
            }
            uint8_t* st = sm + kSOffStage + s * kStage;
            if (new_q) {
                // q unit gq (of 1024): head gq / 16, dims 8 (gq % 16) ..: chunk (gq % 16) / 8,
                // unit gq % 8; the 16 units of a head sit in 16 consecutive lanes
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int gq = gt + 128 * k;
                    const int hd = gq >> 4, uq = gq & 15;
                    const uint32_t qw[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
                    float f[8];
                    float amax = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        f[2 * m] = __uint_as_float(qw[m] << 16);
                        f[2 * m + 1] = __uint_as_float(qw[m] & 0xFFFF0000u);
                        amax = fmaxf(amax, fmaxf(fabsf(f[2 * m]), fabsf(f[2 * m + 1])));
                    }
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                    const int eb = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
                    const int e = amax == 0.f ? 0 : max(-64, min(64, 141 - eb));
                    const float up = __uint_as_float((uint32_t)(127 + e) << 23);
                    uint32_t o[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) o[m] = f32x2_to_f16x2(f[2 * m] * up, f[2 * m + 1] * up);
                    st_shared_v4(st + kStQ + (uq >> 3) * kQChunk + hd * 128 + (((uq & 7) ^ (hd & 7)) << 4), o[0],
                                 o[1], o[2], o[3]);
                    if (uq == 0) {
                        const float down = __uint_as_float((uint32_t)(127 - e) << 23);
                        reinterpret_cast<float*>(st + kStW)[hd] = __ldg(p.w + (size_t)en.x * kIdxHeads + hd) * down;
                    }
                }
            }
            reinterpret_cast<float*>(st + kStScale)[pp] = sc;
            if (gt == 0) *reinterpret_cast<int4*>(st + kStMeta) = en;
            tmem_wait_st();
            tc_fence_before();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(full(s));
        }
    } else if (warp == kIssWarp) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_f16(128, kIdxHeads, 0, 0);
        const uint64_t hi = smem_desc(0, 16, 1024, kSw128) & 0xFFFFFFFF00000000ull;
        const uint32_t lo = (uint32_t)smem_desc(0, 16, 1024, kSw128);
        for (int i = 0; i < n_local; ++i) {
            if (__any_sync(0xffffffffu, s_abort)) break;
            const int s = i % kNS, a = i % kNA, d = i % kND;
            bool ok = mbar_wait(full(s), (i / kNS) & 1, wait_limit);
            ok = ok && (i < kND || mbar_wait(dfree(d), ((i / kND) - 1) & 1, wait_limit));
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail(5);
                break;
            }
            tc_fence_after();
            const uint32_t b_lo = ((sbase + kSOffStage + s * kStage + kStQ) >> 4) & 0x3FFF;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kIdxDim / 16; ++kk) {
                    const uint32_t off_b = ((kk >> 2) * kQChunk + (kk & 3) * 32) >> 4;
                    mma_bf16_ts(tmem + kTmemD + 64 * d, tmem + 64 * a + 8 * kk, hi | (b_lo + lo + off_b), idesc,
                                kk > 0 ? 1u : 0u);
                }
                mma_commit(dfull(d));
                mma_commit(empty(s));
                mma_commit(afree(a));
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
            const int s = i % kNS, d = i % kND;
            bool ok = !s_abort && mbar_wait(dfull(d), (i / kND) & 1, wait_limit);
            ok = ok && mbar_wait(full(s), (i / kNS) & 1, wait_limit);   // the stage's scales, weights
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail(7);
                break;
            }
            tc_fence_after();
            uint32_t a[32], b[32];
            tmem_ld32(tmem + lane_off + kTmemD + 64 * d, a);
            tmem_ld32(tmem + lane_off + kTmemD + 64 * d + 32, b);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dfree(d));
            const uint8_t* st = sm + kSOffStage + s * kStage;
            const float4* wv = reinterpret_cast<const float4*>(st + kStW);
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 wa = wv[j], wb = wv[8 + j];
                acc0 = fmaf(wa.x, fmaxf(__uint_as_float(a[4 * j]), 0.f), acc0);
                acc0 = fmaf(wa.y, fmaxf(__uint_as_float(a[4 * j + 1]), 0.f), acc0);
                acc0 = fmaf(wa.z, fmaxf(__uint_as_float(a[4 * j + 2]), 0.f), acc0);
                acc0 = fmaf(wa.w, fmaxf(__uint_as_float(a[4 * j + 3]), 0.f), acc0);
                acc1 = fmaf(wb.x, fmaxf(__uint_as_float(b[4 * j]), 0.f), acc1);
                acc1 = fmaf(wb.y, fmaxf(__uint_as_float(b[4 * j + 1]), 0.f), acc1);
                acc1 = fmaf(wb.z, fmaxf(__uint_as_float(b[4 * j + 2]), 0.f), acc1);
                acc1 = fmaf(wb.w, fmaxf(__uint_as_float(b[4 * j + 3]), 0.f), acc1);
            }
            const float score = reinterpret_cast<const float*>(st + kStScale)[pp] * (acc0 + acc1) + 0.0f;   // (-0 -> +0)
            const int4 meta = *reinterpret_cast<const int4*>(st + kStMeta);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
            if (pp < meta.z) p.scores[(size_t)meta.x * p.ld + meta.y + pp] = score;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kIssWarp) tmem_dealloc(tmem, kSTmemCols);
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
    // codes of page z, row y, byte x: pool + z * 8448 + y * 128 + x
    CUtensorMap tm;
    const uint64_t dims[3] = {(uint64_t)kIdxDim, (uint64_t)kPage, (uint64_t)(num_pages > 0 ? num_pages : 1)};
    const uint64_t strides[2] = {(uint64_t)kIdxDim, (uint64_t)kIdxPageBytes};
    const uint32_t box[3] = {(uint32_t)kIdxDim, (uint32_t)kPage, 1u};
    if (!encode_3d(&tm, pool, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_UINT8))
        return cudaErrorInvalidValue;
    indexer_score_kernel<<<C, kSThreads, kSSmem, st>>>(tm, p);
    return cudaGetLastError();
}

cudaError_t launch_topk_select(const float* scores, int64_t ld, const int32_t* seq_lens, int B, int K,
                               int32_t* idx, cudaStream_t st) {
    topk_select_kernel<<<B, kKThreads, 0, st>>>(scores, ld, seq_lens, K, idx);
    return cudaGetLastError();
}

}  // namespace mla
