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
// Scores: the keys of 256 positions (four pages) against one request's 64 head queries are two
// tensor-core contractions D[128 x 64] = codes[128 x 128] . q^T (f16 operands, exact products,
// fp32 accumulation in TMEM), and since a key's scale s >= 0,
//   I = s * sum_j w_j max(D_j, 0).
// One CTA per SM walks a balanced range of (request, 256-position) tiles.  Two producer threads
// load whole pages into an 8-deep shared-memory ring by TMA; converter warps turn the E4M3 codes
// into f16 straight in tensor memory (the MMA's A operand); one warp issues the MMAs; epilogue
// warps (thread = position = TMEM lane) finish the scores.  The pass is HBM-bound on the keys
// (132 B per position).
//
// Top-k: one cluster of two CTAs per request, each holding half the row; a radix select on
// order-preserving keys of the fp32 scores (digits of 11, 11 and 10 bits, most significant first,
// the two halves' histograms summed through distributed shared memory) finds the K-th largest,
// then each warp writes the positions of its range of a half that are above it and, of those
// equal to it, the lowest ones, in increasing position order.
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
constexpr int kTile = 256;                       // positions per tile (four pages)
constexpr int kMH = kTile / 128;                 // its 128-position halves (one MMA row block each)
constexpr int kTP = kTile / 64;                  // its pages

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

// Warp roles: 8 converter warps and 8 epilogue warps, each in two groups of 4 (group g takes the
// tiles i = g mod 2; warp w of a group owns TMEM lanes 32 (w % 4) ..), two MMA issuers (warps 16
// and 19) and two producers (warps 17, 18), issuer / producer g for the tiles i = g mod 2.  A warp
// runs on sub-partition warp % 4, so each sub-partition carries one single-thread role.
constexpr int kConvWarps = 8;
constexpr int kEpiWarps = 8;
constexpr int kIssWarp = kConvWarps + kEpiWarps;   // even tiles; kIssWarp + 3: odd tiles
constexpr int kProdWarp = kIssWarp + 1;
constexpr int kSThreads = 32 * (kIssWarp + 4);
constexpr int kNR = 4;                           // raw page slots (tiles in flight)
constexpr int kNS = 8;                           // per-tile stages (scales, weights, tile info)
constexpr int kNA = 2;                           // A operands in tensor memory
constexpr int kND = 2;                           // accumulators in tensor memory
constexpr int kLookup = 2;                       // tiles whose pages a producer looks up together
// raw slot: the tile's four pages whole, each as 66 rows of 128 B (64 rows of codes, then the 64
// scales) with the 128-byte swizzle, at 9 KB apart
constexpr int kPageRows = kIdxPageBytes / 128;          // 66
constexpr int kSlotPage = 9216;
constexpr int kSlot = kTP * kSlotPage;
// q slot (one per request in flight, two): q as the MMA's B operand ([64 heads x 64 dims] f16
// per chunk, two chunks, SW128), then the 64 rescaled head weights
constexpr int kQChunk = kIdxHeads * 128;
constexpr int kQW = 2 * kQChunk;                        // 16384
constexpr int kQSlot = 17408;
// stage: the tile's 256 key scales, its 64 head weights, {request, first position, count, flags}
constexpr int kStScale = 0;
constexpr int kStW = kTile * 4;                         // 1024
constexpr int kStMeta = kStW + kIdxHeads * 4;           // 1280
constexpr int kStage = 1296;
constexpr int kSOffQ = kNR * kSlot;                     // 147456
constexpr int kSOffStage = kSOffQ + 2 * kQSlot;         // 182272
constexpr int kSOffEntry = kSOffStage + kNS * kStage;   // per raw slot {b, base, cnt, flags}
constexpr int kSOffBar = kSOffEntry + kNR * 16;
constexpr int kNBars = 2 * kNR + 2 * kNS + kNA + 2 * kND + 4 + 2;
constexpr int kSSmem = kSOffBar + 8 * kNBars + 1024;
constexpr uint32_t kSTmemCols = 512;                    // A: 2 x 128 columns, D: 2 x 128 columns
constexpr uint32_t kTmemD = 64 * kMH * kNA;
// tile flags: request ordinal within the CTA's range (bits 0..27), first / last tile of the request
constexpr int kFirst = 1 << 28, kLast = 1 << 29, kOrdMask = (1 << 28) - 1;
static_assert(kPageRows * 128 == kIdxPageBytes && kIdxPageBytes <= kSlotPage && kSlotPage % 1024 == 0, "raw slot");
static_assert(kQW + kIdxHeads * 4 <= kQSlot && kQSlot % 1024 == 0 && kSOffQ % 1024 == 0, "q slot");
static_assert(kStMeta + 16 <= kStage && kStage % 16 == 0, "stage layout");
static_assert(kSSmem <= 232448, "shared memory");
static_assert(kNR % 2 == 0 && kNS % 2 == 0 && kNA % 2 == 0 && kND % 2 == 0, "rings shared by two groups");
static_assert(kTmemD + 64 * kMH * kND <= kSTmemCols, "tensor memory");

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

__device__ __forceinline__ int tiles_n(int n) { return (n + kTile - 1) / kTile; }

// Balanced contiguous range of the (request, 256-position tile) stream for CTA c of C; run by one
// warp.  Returns the first tile and the tile count through shared memory.
__device__ void score_schedule(const ScoreParams& p, int c, int C, int* s_b, int* s_t, int* s_n) {
    const int lane = threadIdx.x & 31;
    const int per = (p.B + 31) / 32;
    const int b_lo = min(p.B, lane * per), b_hi = min(p.B, b_lo + per);
    long long mine = 0;
    for (int b = b_lo; b < b_hi; ++b) mine += tiles_n(clamp_len(p.seq_lens[b], p.max_seq_len));
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
        const int nt = tiles_n(clamp_len(p.seq_lens[b], p.max_seq_len));
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
        nt = tiles_n(n);
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

// Scores of a balanced range of (request, 256-position) tiles per CTA.
//   producers: look up each tile's four pages (checked) and load each whole into a raw slot by one
//             TMA copy (a 3D tensor map: 66 rows of 128 B per page, 128-byte swizzle); they walk
//             the whole tile stream, so they also number the requests and mark each request's
//             first and last tile;
//   converters: E4M3 codes -> f16 (exact) straight into tensor memory as the MMA's A operand
//             (row = position, two dims per column); key scales, head weights and tile info into
//             the tile's stage; on a request's first tile, that request's q into a q slot (scaled
//             per head by 2^e into [2^14, 2^15) of f16, the head weight by 2^-e: the products
//             w ReLU(q . k) are unchanged, and every bf16 q element not 2^31 below its head's
//             largest is exact in f16);
//   issuers:  D[128 x 64] = A[128 x 128] . q^T for each half of the tile, eight K=16 MMAs each; each walks the tile
//             stream and, at the end of each request, commits the release of its q slot (the slot
//             is free once both issuers' MMAs up to there are done);
//   epilogue: thread = position = TMEM lane: I = s * sum_j w_j max(D_j, 0), two groups of 4 warps
//             on alternate tiles.
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
    auto raw_full = [&](int r) { return bar0 + 8 * r; };                   // producer -> converters
    auto raw_empty = [&](int r) { return bar0 + 8 * (kNR + r); };          // converters -> producer
    auto full = [&](int s) { return bar0 + 8 * (2 * kNR + s); };           // converters -> issuer, epilogue
    auto sempty = [&](int s) { return bar0 + 8 * (2 * kNR + kNS + s); };   // epilogue -> converters
    auto afree = [&](int a) { return bar0 + 8 * (2 * kNR + 2 * kNS + a); };            // MMA -> converters
    auto dfull = [&](int d) { return bar0 + 8 * (2 * kNR + 2 * kNS + kNA + d); };      // MMA -> epilogue
    auto dfree = [&](int d) { return bar0 + 8 * (2 * kNR + 2 * kNS + kNA + kND + d); };   // epilogue -> MMA
    auto qfull = [&](int q) { return bar0 + 8 * (2 * kNR + 2 * kNS + kNA + 2 * kND + q); };     // q slot written
    auto qempty = [&](int q) { return bar0 + 8 * (2 * kNR + 2 * kNS + kNA + 2 * kND + 2 + q); };   // q slot free
    int4* entry = reinterpret_cast<int4*>(sm + kSOffEntry);
    const uint32_t wait_limit = p.ctl->wait_limit;
    auto swait = [](uint32_t bar, uint32_t parity, uint32_t limit) { return mbar_wait(bar, parity, limit); };

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
            mbar_init(sempty(s), 4);
        }
        for (int a = 0; a < kNA; ++a) mbar_init(afree(a), 1);
        for (int d = 0; d < kND; ++d) {
            mbar_init(dfull(d), 1);
            mbar_init(dfree(d), 4);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(qfull(q), 4);
            mbar_init(qempty(q), 2);   // both issuers, at the request's end
        }
        mbar_init(bar0 + 8 * (kNBars - 2), 1);   // the issuers' drains
        mbar_init(bar0 + 8 * (kNBars - 1), 1);
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

    if (warp == kProdWarp || warp == kProdWarp + 1) {
        // ------------------------------------------------------------ producers
        // Producer pw loads the tiles j = pw, pw + 2, ..; its cursor walks every tile, counting
        // request changes.  The block-table lookups of its next kLookup tiles are in flight while
        // the current ones are issued.
        const int pw = warp - kProdWarp;
        if (lane == 0 && pw < n_local) {
            TileCursor pf;
            pf.b = s_b0;
            pf.t = s_t0;
            pf.load(p);
            int ord = 0, prev_b = -1;   // request ordinal of the cursor's tile; request before it
            auto step = [&](int j) {    // cursor from tile j to tile j + 1 (j + 1 < n_local)
                prev_b = pf.b;
                pf.next(p);
                if (pf.b != prev_b) ++ord;
            };
            if (pw == 1) step(0);
            struct Batch {
                int b[kLookup], base[kLookup], cnt[kLookup], flags[kLookup], pg[kLookup][kTP];
            };
            // tiles j0, j0 + 2, .. of this producer (cursor at tile j0; left at the tile after)
            auto fill = [&](Batch& x, int j0) {
#pragma unroll
                for (int k = 0; k < kLookup; ++k) {
                    const int j = j0 + 2 * k;
#pragma unroll
                    for (int h = 0; h < kTP; ++h) x.pg[k][h] = -1;
                    x.b[k] = pf.b;
                    x.base[k] = pf.t * kTile;
                    x.cnt[k] = min(kTile, pf.n - x.base[k]);
                    x.flags[k] = ord | (prev_b != pf.b ? kFirst : 0);
                    if (j < n_local) {
                        const int32_t* row = p.block_table + (size_t)x.b[k] * p.max_pages + (x.base[k] >> 6);
#pragma unroll
                        for (int h = 0; h < kTP; ++h)
                            if (x.cnt[k] > 64 * h) x.pg[k][h] = row[h];
                        if (j + 1 < n_local) {
                            step(j);
                            if (pf.b != x.b[k]) x.flags[k] |= kLast;
                            if (j + 2 < n_local) step(j + 1);
                        } else {
                            x.flags[k] |= kLast;
                        }
                    }
                }
            };
            Batch cur, nxt;
            int issued_hi = -1;   // the last tile issued
            fill(cur, pw);
            bool ok = true;
            for (int j0 = pw; ok && j0 < n_local && !s_abort; j0 += 2 * kLookup) {
                if (j0 + 2 * kLookup < n_local) fill(nxt, j0 + 2 * kLookup);
#pragma unroll
                for (int k = 0; k < kLookup; ++k) {
                    const int j = j0 + 2 * k, r = j % kNR;
                    if (j >= n_local || !ok) continue;
                    if (j >= kNR && !swait(raw_empty(r), ((j / kNR) - 1) & 1, wait_limit)) {
                        fail(4);
                        ok = false;
                        continue;
                    }
                    int pg[kTP];
                    uint32_t bytes = 0;
#pragma unroll
                    for (int h = 0; h < kTP; ++h) {
                        pg[h] = cur.pg[k][h];
                        if (cur.cnt[k] <= 64 * h) continue;
                        if (pg[h] < 0 || pg[h] >= p.num_pages) {
                            record_error(p.ctl, MLA_ERR_BOUNDS, pg[h]);
                            pg[h] = -1;
                        } else {
                            bytes += kIdxPageBytes;
                        }
                    }
                    entry[r] = make_int4(cur.b[k], cur.base[k], cur.cnt[k], cur.flags[k]);
                    const uint32_t slot = sbase + r * kSlot;
                    mbar_arrive_expect_tx(raw_full(r), bytes);
#pragma unroll
                    for (int h = 0; h < kTP; ++h)
                        if (pg[h] >= 0) tma_load_3d(slot + h * kSlotPage, &tm_codes, raw_full(r), 0, 0, pg[h]);
                    issued_hi = j;
                }
                cur = nxt;
            }
            // nothing of this CTA's copies is left in flight when it exits
            for (int j = issued_hi; j >= 0 && j > issued_hi - kNR; j -= 2)
                if (!swait(raw_full(j % kNR), (j / kNR) & 1, wait_limit)) fail(6);
        }
        __syncwarp();
    } else if (warp < kConvWarps) {
        // ------------------------------------------------------------ converters
        const int g = warp >> 2, q4 = warp & 3;
        const int gt = tid & 127;             // thread within the group
        const int pp = q4 * 32 + lane;        // position within each half = TMEM lane
        const int rr = pp & 63;               // row of the page
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        for (int i = g; i < n_local; i += 2) {
            if (s_abort) break;
            const int s = i % kNS, r = i % kNR, a = i % kNA;
            if (!swait(raw_full(r), (i / kNR) & 1, wait_limit)) {
                if (lane == 0) fail(1);
                break;
            }
            const int4 en = entry[r];
            if (i >= kNA && !swait(afree(a), ((i / kNA) - 1) & 1, wait_limit)) {
                if (lane == 0) fail(2);
                break;
            }
            tc_fence_after();
            float sc[kMH];
#pragma unroll
            for (int m = 0; m < kMH; ++m) {
                // position 128 m + pp: page 2 m + pp / 64, row rr
                const int pgo = r * kSlot + (2 * m + (pp >> 6)) * kSlotPage;
                const uint32_t rowa = sbase + pgo + rr * 128;
                uint4 u[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) u[c] = ld_shared_v4(rowa + ((c ^ (rr & 7)) << 4));
                // scale rr: byte 4 rr of rows 64, 65 (unit (rr % 32) / 4, swizzled by the row)
                sc[m] = *reinterpret_cast<const float*>(
                    sm + pgo + (64 + (rr >> 5)) * 128 + ((((rr & 31) >> 2) ^ (rr >> 5)) << 4) + (rr & 3) * 4);
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
                    tmem_st32(tmem + lane_off + 64 * (kMH * a + m) + 32 * half, o);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(raw_empty(r));
            const int ord = en.w & kOrdMask, qs = ord & 1;
            uint8_t* qslot = sm + kSOffQ + qs * kQSlot;
            if (en.w & kFirst) {
                // this request's q into its slot, once the request two before has left it
                uint4 qv[8];
                const uint4* qsrc = reinterpret_cast<const uint4*>(p.q + (size_t)en.x * kIdxHeads * kIdxDim);
#pragma unroll
                for (int k = 0; k < 8; ++k) qv[k] = __ldg(qsrc + gt + 128 * k);
                if (ord >= 2 && !swait(qempty(qs), ((ord >> 1) - 1) & 1, wait_limit)) {
                    if (lane == 0) fail(8);
                    break;
                }
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
                    st_shared_v4(qslot + (uq >> 3) * kQChunk + hd * 128 + (((uq & 7) ^ (hd & 7)) << 4), o[0], o[1],
                                 o[2], o[3]);
                    if (uq == 0) {
                        const float down = __uint_as_float((uint32_t)(127 - e) << 23);
                        reinterpret_cast<float*>(qslot + kQW)[hd] = __ldg(p.w + (size_t)en.x * kIdxHeads + hd) * down;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(qfull(qs));
            }
            if (i >= kNS && !swait(sempty(s), ((i / kNS) - 1) & 1, wait_limit)) {
                if (lane == 0) fail(3);
                break;
            }
            if (!swait(qfull(qs), (ord >> 1) & 1, wait_limit)) {   // the request's weights
                if (lane == 0) fail(9);
                break;
            }
            uint8_t* st = sm + kSOffStage + s * kStage;
#pragma unroll
            for (int m = 0; m < kMH; ++m) reinterpret_cast<float*>(st + kStScale)[128 * m + pp] = sc[m];
            if (gt < kIdxHeads)
                reinterpret_cast<float*>(st + kStW)[gt] = reinterpret_cast<const float*>(qslot + kQW)[gt];
            if (gt == 0) *reinterpret_cast<int4*>(st + kStMeta) = en;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(full(s));
        }
    } else if (warp == kIssWarp || warp == kIssWarp + 3) {
        // ------------------------------------------------------------ MMA issuers
        constexpr uint32_t idesc = idesc_f16(128, kIdxHeads, 0, 0);
        const uint64_t hi = smem_desc(0, 16, 1024, kSw128) & 0xFFFFFFFF00000000ull;
        const uint32_t lo = (uint32_t)smem_desc(0, 16, 1024, kSw128);
        const int ig = warp == kIssWarp ? 0 : 1;
        const uint32_t drain = bar0 + 8 * (kNBars - 2 + ig);
        TileCursor ic;
        ic.b = s_b0;
        ic.t = s_t0;
        if (n_local > 0) ic.load(p);
        int ord = 0, ready_ord = -1;   // request ordinal of tile i; the last one whose q was seen
        for (int i = 0; i < n_local; ++i) {
            if (__any_sync(0xffffffffu, s_abort)) break;
            if ((i & 1) == ig) {
                const int s = i % kNS, a = i % kNA, d = i % kND, qs = ord & 1;
                bool ok = swait(full(s), (i / kNS) & 1, wait_limit);
                if (ord != ready_ord) {
                    ok = ok && swait(qfull(qs), (ord >> 1) & 1, wait_limit);
                    ready_ord = ord;
                }
                ok = ok && (i < kND || swait(dfree(d), ((i / kND) - 1) & 1, wait_limit));
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) fail(5);
                    break;
                }
                tc_fence_after();
                const uint32_t b_lo = ((sbase + kSOffQ + qs * kQSlot) >> 4) & 0x3FFF;
                if (elect_one()) {
#pragma unroll
                    for (int m = 0; m < kMH; ++m)
#pragma unroll
                        for (int kk = 0; kk < kIdxDim / 16; ++kk) {
                            const uint32_t off_b = ((kk >> 2) * kQChunk + (kk & 3) * 32) >> 4;
                            mma_bf16_ts(tmem + kTmemD + 64 * (kMH * d + m), tmem + 64 * (kMH * a + m) + 8 * kk,
                                        hi | (b_lo + lo + off_b), idesc, kk > 0 ? 1u : 0u);
                        }
                    mma_commit(dfull(d));
                    mma_commit(afree(a));
                }
                __syncwarp();
            }
            const int b = ic.b;
            if (i + 1 < n_local) ic.next(p);
            if (i + 1 == n_local || ic.b != b) {   // the request of tile i ends here
                if (elect_one()) mma_commit(qempty(ord & 1));
                __syncwarp();
                ++ord;
            }
        }
        __syncwarp();
        if (elect_one()) {
            mma_commit(drain);
            swait(drain, 0, wait_limit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int eg = (warp - kConvWarps) >> 2, q4 = warp & 3;   // group; TMEM lanes 32 q4 ..
        const int pp = q4 * 32 + lane;                            // position within the tile
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        for (int i = eg; i < n_local; i += 2) {
            const int s = i % kNS, d = i % kND;
            bool ok = !s_abort && swait(dfull(d), (i / kND) & 1, wait_limit);
            ok = ok && swait(full(s), (i / kNS) & 1, wait_limit);   // the stage's scales, weights
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail(7);
                break;
            }
            tc_fence_after();
            const uint8_t* st = sm + kSOffStage + s * kStage;
            const float4* wv = reinterpret_cast<const float4*>(st + kStW);
            const int4 meta = *reinterpret_cast<const int4*>(st + kStMeta);
            float score[kMH];
#pragma unroll
            for (int m = 0; m < kMH; ++m) {
                uint32_t a[32], b[32];
                tmem_ld32(tmem + lane_off + kTmemD + 64 * (kMH * d + m), a);
                tmem_ld32(tmem + lane_off + kTmemD + 64 * (kMH * d + m) + 32, b);
                tmem_wait_ld();
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 wa = wv[j], wb = wv[8 + j];
                    acc[0] = fmaf(wa.x, fmaxf(__uint_as_float(a[4 * j]), 0.f), acc[0]);
                    acc[1] = fmaf(wa.y, fmaxf(__uint_as_float(a[4 * j + 1]), 0.f), acc[1]);
                    acc[2] = fmaf(wa.z, fmaxf(__uint_as_float(a[4 * j + 2]), 0.f), acc[2]);
                    acc[3] = fmaf(wa.w, fmaxf(__uint_as_float(a[4 * j + 3]), 0.f), acc[3]);
                    acc[0] = fmaf(wb.x, fmaxf(__uint_as_float(b[4 * j]), 0.f), acc[0]);
                    acc[1] = fmaf(wb.y, fmaxf(__uint_as_float(b[4 * j + 1]), 0.f), acc[1]);
                    acc[2] = fmaf(wb.z, fmaxf(__uint_as_float(b[4 * j + 2]), 0.f), acc[2]);
                    acc[3] = fmaf(wb.w, fmaxf(__uint_as_float(b[4 * j + 3]), 0.f), acc[3]);
                }
                score[m] = reinterpret_cast<const float*>(st + kStScale)[128 * m + pp] *
                               ((acc[0] + acc[1]) + (acc[2] + acc[3])) +
                           0.0f;   // (-0 -> +0)
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(dfree(d));
                mbar_arrive(sempty(s));
            }
#pragma unroll
            for (int m = 0; m < kMH; ++m)
                if (128 * m + pp < meta.z) p.scores[(size_t)meta.x * p.ld + meta.y + 128 * m + pp] = score[m];
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

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

constexpr int kKWarps = kKThreads / 32;

// f(key) for every order key of x[0, cnt), in no particular order, with 16-byte loads where x is
// aligned (the unaligned head and the tail one value at a time).
template <typename F>
__device__ __forceinline__ void for_each_key(const float* __restrict__ x, int cnt, F f) {
    const int tid = threadIdx.x;
    int head = (int)(((16u - ((uint32_t)(uintptr_t)x & 15u)) & 15u) >> 2);
    head = head < cnt ? head : cnt;
    if (tid < head) f(order_key(x[tid]));
    const float4* xv = reinterpret_cast<const float4*>(x + head);
    const int nv = (cnt - head) >> 2;
    constexpr int kV = 4;   // 16-byte loads in flight per thread
    for (int base = 0; base < nv; base += kV * kKThreads) {
        float4 v[kV];
#pragma unroll
        for (int u = 0; u < kV; ++u) {
            const int i = base + u * kKThreads + tid;
            v[u] = i < nv ? __ldg(xv + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kV; ++u) {
            if (base + u * kKThreads + tid < nv) {
                f(order_key(v[u].x));
                f(order_key(v[u].y));
                f(order_key(v[u].z));
                f(order_key(v[u].w));
            }
        }
    }
    const int t = head + 4 * nv + tid;
    if (t < cnt) f(order_key(x[t]));
}
constexpr int kKU = 8;   // loads in flight per thread in the passes over the row

// One request per cluster of two CTAs; CTA q holds positions [q h, min(n, (q + 1) h)), h = the
// row's first half rounded up.  The K-th largest key T is found one digit at a time (11, 11 and
// 10 bits, most significant first) from the sum of the two CTAs' histograms of their halves
// (the peer's read through distributed shared memory; two histogram buffers, so one cluster
// barrier per digit suffices).  The first digit's keys crowd into few bins (their exponents), so
// its histogram is counted in eight private copies (warp w into copy w % 8) that are then summed.
// The digit is chosen by all threads at once: thread t holds bins [p t, p t + p) (p = bins / 1024)
// of both halves' sum, one block-wide suffix sum gives each thread the keys in the bins above its
// own, and the thread whose bins hold the krem-th largest key writes the digit.  The histograms
// also give how many keys above T and equal to T the first half holds, which places the second
// CTA's output.  After the first digit, one pass over the row keeps the keys of its bin (with their
// positions) in shared memory and counts, per warp range, the keys above it; the later digits and
// the counts of keys above and equal to T then come from those candidates alone.  If either CTA's
// candidates do not fit, both take the later digits and the counts from the row.  Each warp of a CTA then owns a
// contiguous range of its half: one pass counts the range's keys above and equal to T, and a
// second writes its positions in order (the keys above T, and of the krem keys equal to T the
// lowest positions).
constexpr int kKPriv = 8;                                        // private copies of the first histogram
constexpr int kKSmem = kKPriv * 2048 * (int)sizeof(uint32_t);    // dynamic shared memory: those copies,
constexpr int kKCand = kKSmem / 8;                                // then up to 8,192 candidates (key, position)

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kKThreads)
    topk_select_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ seq_lens, int K,
                       int32_t* __restrict__ idx) {
    static_assert(kKWarps == 32, "the suffix sum over warps takes one warp");
    extern __shared__ uint32_t priv[];   // [kKPriv][2048]
    __shared__ uint32_t hist[2][2048];
    __shared__ int wgt[kKWarps], weq[kKWarps];
    __shared__ uint32_t wsum[kKWarps], wsum0[kKWarps], wab[kKWarps], wab0[kKWarps];
    __shared__ uint32_t s_prefix, s_mask;
    __shared__ int s_krem, s_above0, s_eq0, s_ncand;
    const uint32_t q = cluster_rank();
    const int b = blockIdx.x >> 1, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int64_t n64 = seq_lens[b];
    n64 = n64 < 0 ? 0 : (n64 > ld ? ld : n64);
    const int n = (int)n64;
    const float* row = scores + (size_t)b * ld;
    int32_t* out = idx + (size_t)b * K;
    if (n <= K) {
        if (q == 0)
            for (int t = tid; t < K; t += kKThreads) out[t] = t < n ? t : -1;
        return;   // both CTAs of the cluster leave here
    }
    const int h = (n + 1) / 2;
    const int lo = (int)q * h, hi = q == 0 ? h : n;
    const uint32_t peer_hist = mapa(smem_u32(&hist[0][0]), q ^ 1u);
    const uint32_t peer_ncand = mapa(smem_u32(&s_ncand), q ^ 1u);
    if (tid == 0) {
        s_prefix = 0;
        s_mask = 0;
        s_krem = K;
        s_above0 = 0;
        s_eq0 = 0;
        s_ncand = 0;
    }
    // each warp's contiguous range of this half (candidates, counts and the ordered write)
    const unsigned lt = (1u << lane) - 1u;
    const int L = (hi - lo + kKU * kKThreads - 1) / (kKU * kKThreads) * (kKU * 32);
    const int r0 = lo + warp * L, r1 = min(hi, r0 + L);
    uint2* cand = reinterpret_cast<uint2*>(priv);   // after the first digit: (key, position) of its bin
    bool from_cand = false;                         // digits 2 and 3 over the candidates
    int ncand = 0;
    for (int level = 0; level < 3; ++level) {
        if (level == 1) {
            // The keys of the first digit's bin d0 (the candidates) into shared memory in one pass
            // over the row, and per warp range the keys above that bin (all above T).  If either
            // CTA's candidates do not fit, both take digits 2 and 3 and the counts from the row.
            const uint32_t d0 = s_prefix >> 21;
            int g = 0;
            for (int c0 = r0; c0 < r0 + L; c0 += 32 * kKU) {
                uint32_t key[kKU];
#pragma unroll
                for (int u = 0; u < kKU; ++u) {
                    const int t = c0 + 32 * u + lane;
                    key[u] = t < r1 ? order_key(row[t]) : 0u;
                }
                // one shared-counter update per warp and chunk
                unsigned cb[kKU];
                int total = 0;
#pragma unroll
                for (int u = 0; u < kKU; ++u) {
                    const bool in = c0 + 32 * u + lane < r1;
                    g += (in && (key[u] >> 21) > d0) ? 1 : 0;
                    cb[u] = __ballot_sync(0xffffffffu, in && (key[u] >> 21) == d0);
                    total += __popc(cb[u]);
                }
                if (total > 0) {
                    int base = 0;
                    if (lane == 0) base = atomicAdd(&s_ncand, total);
                    base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
                    for (int u = 0; u < kKU; ++u) {
                        const int at = base + __popc(cb[u] & lt);
                        if (((cb[u] >> lane) & 1u) && at < kKCand)
                            cand[at] = make_uint2(key[u], (uint32_t)(c0 + 32 * u + lane));
                        base += __popc(cb[u]);
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
            if (lane == 0) {
                wgt[warp] = g;
                weq[warp] = 0;
            }
            cluster_sync();   // both CTAs' candidate counts are final
            ncand = s_ncand;
            from_cand = ncand <= kKCand && (int)ld_cluster_u32(peer_ncand) <= kKCand;
        }
        const int shift = level == 0 ? 21 : (level == 1 ? 10 : 0);
        const int nb = level == 2 ? 1024 : 2048;
        const int hb = level & 1;
        if (level == 0) {
            for (int j = tid; j < kKPriv * 2048; j += kKThreads) priv[j] = 0;
        } else {
            for (int j = tid; j < 2048; j += kKThreads) hist[hb][j] = 0;
        }
        __syncthreads();
        const uint32_t prefix = s_prefix, mask = s_mask;
        const int krem = s_krem;
        uint32_t* hdst = level == 0 ? priv + (warp % kKPriv) * 2048 : hist[hb];
        if (from_cand) {
            for (int i = tid; i < ncand; i += kKThreads) {
                const uint32_t key = cand[i].x;
                if ((key & mask) == prefix) atomicAdd(&hist[hb][(key >> shift) & (uint32_t)(nb - 1)], 1u);
            }
        }
        if (!from_cand)
            for_each_key(row + lo, hi - lo, [&](uint32_t key) {
                if ((key & mask) == prefix) atomicAdd(&hdst[(key >> shift) & (uint32_t)(nb - 1)], 1u);
            });
        if (level == 0) {
            __syncthreads();
            for (int j = tid; j < 2048; j += kKThreads) {
                uint32_t sum = 0;
#pragma unroll
                for (int c = 0; c < kKPriv; ++c) sum += priv[c * 2048 + j];
                hist[0][j] = sum;
            }
        }
        cluster_sync();   // both halves' histograms of this digit are complete
        // this thread's bins: counts over both halves (c) and over the first half (f)
        const int per = nb / kKThreads;   // 2 or 1
        uint32_t c[2] = {0u, 0u}, f[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (i < per) {
                const int j = per * tid + i;
                const uint32_t own = hist[hb][j];
                const uint32_t oth = ld_cluster_u32(peer_hist + 4u * (uint32_t)(hb * 2048 + j));
                c[i] = own + oth;
                f[i] = q == 0 ? own : oth;
            }
        }
        const uint32_t ct = c[0] + c[1], ft = f[0] + f[1];
        // suffix sums: within the warp (a higher lane holds higher bins), then over the warps
        uint32_t x = ct, x0 = ft;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_down_sync(0xffffffffu, x, o), y0 = __shfl_down_sync(0xffffffffu, x0, o);
            if (lane + o < 32) {
                x += y;
                x0 += y0;
            }
        }
        if (lane == 0) {
            wsum[warp] = x;
            wsum0[warp] = x0;
        }
        __syncthreads();
        if (warp == 0) {
            const uint32_t v = wsum[lane], v0 = wsum0[lane];
            uint32_t sx = v, sx0 = v0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_down_sync(0xffffffffu, sx, o), y0 = __shfl_down_sync(0xffffffffu, sx0, o);
                if (lane + o < 32) {
                    sx += y;
                    sx0 += y0;
                }
            }
            wab[lane] = sx - v;     // keys in the bins of the warps above
            wab0[lane] = sx0 - v0;
        }
        __syncthreads();
        const uint32_t above = wab[warp] + (x - ct);   // keys in every bin above this thread's
        if (above < (uint32_t)krem && (uint32_t)krem <= above + ct) {   // exactly one thread
            uint32_t rem = (uint32_t)krem - above;
            uint32_t a0 = wab0[warp] + (x0 - ft);      // the first half's keys above
#pragma unroll
            for (int i = 1; i >= 0; --i) {
                if (i >= per) continue;
                if (rem <= c[i]) {
                    const uint32_t d = (uint32_t)(per * tid + i);
                    // the first half's keys in bins above d (all above T), and at the last digit in bin d
                    s_above0 += (int)a0;
                    if (level == 2) s_eq0 = (int)f[i];
                    s_krem = (int)rem;
                    s_prefix = prefix | (d << shift);
                    s_mask = mask | ((uint32_t)(nb - 1) << shift);
                    break;
                }
                rem -= c[i];
                a0 += f[i];
            }
        }
        __syncthreads();
    }
    cluster_sync();   // no CTA reads the other's histograms any more (it may exit)
    const uint32_t T = s_prefix;
    const int krem = s_krem;   // keys equal to T to take, lowest positions first

    // per warp range of this half: keys above T and equal to T (from the candidates: the range's
    // keys above the first digit's bin, counted before, plus its candidates above / equal to T)
    if (from_cand) {
        for (int i = tid; i < ncand; i += kKThreads) {
            const uint2 c = cand[i];
            const int w = ((int)c.y - lo) / L;
            if (c.x > T) atomicAdd(&wgt[w], 1);
            else if (c.x == T) atomicAdd(&weq[w], 1);
        }
    } else {
        int g = 0, e = 0;
        for (int c0 = r0; c0 < r0 + L; c0 += 32 * kKU) {
            uint32_t key[kKU];
#pragma unroll
            for (int u = 0; u < kKU; ++u) {
                const int t = c0 + 32 * u + lane;
                key[u] = t < r1 ? order_key(row[t]) : 0u;
            }
#pragma unroll
            for (int u = 0; u < kKU; ++u) {
                const bool in = c0 + 32 * u + lane < r1;
                g += (in && key[u] > T) ? 1 : 0;
                e += (in && key[u] == T) ? 1 : 0;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            g += __shfl_xor_sync(0xffffffffu, g, o);
            e += __shfl_xor_sync(0xffffffffu, e, o);
        }
        if (lane == 0) {
            wgt[warp] = g;
            weq[warp] = e;
        }
    }
    __syncthreads();
    int above = q == 0 ? 0 : s_above0, eq_before = q == 0 ? 0 : s_eq0;
    for (int v = 0; v < warp; ++v) {
        above += wgt[v];
        eq_before += weq[v];
    }
    // ordered write: the keys above T before this range, and the equal ones (at most krem)
    int o = above + min(krem, eq_before);
    for (int c0 = r0; c0 < r0 + L; c0 += 32 * kKU) {
        uint32_t key[kKU];
#pragma unroll
        for (int u = 0; u < kKU; ++u) {
            const int t = c0 + 32 * u + lane;
            key[u] = t < r1 ? order_key(row[t]) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kKU; ++u) {
            const int t = c0 + 32 * u + lane;
            const bool in = t < r1;
            const bool is_eq = in && key[u] == T;
            const unsigned eb = __ballot_sync(0xffffffffu, is_eq);
            const bool take = (in && key[u] > T) || (is_eq && eq_before + __popc(eb & lt) < krem);
            const unsigned tb = __ballot_sync(0xffffffffu, take);
            if (take) out[o + __popc(tb & lt)] = t;
            o += __popc(tb);
            eq_before += __popc(eb);
        }
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
    // page z as 66 rows y of 128 bytes x (64 rows of codes, then the scales): pool + z * 8448 +
    // y * 128 + x
    CUtensorMap tm;
    const uint64_t dims[3] = {128u, (uint64_t)kPageRows, (uint64_t)(num_pages > 0 ? num_pages : 1)};
    const uint64_t strides[2] = {128u, (uint64_t)kIdxPageBytes};
    const uint32_t box[3] = {128u, (uint32_t)kPageRows, 1u};
    if (!encode_3d(&tm, pool, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_UINT8))
        return cudaErrorInvalidValue;
    indexer_score_kernel<<<C, kSThreads, kSSmem, st>>>(tm, p);
    return cudaGetLastError();
}

cudaError_t launch_topk_select(const float* scores, int64_t ld, const int32_t* seq_lens, int B, int K,
                               int32_t* idx, cudaStream_t st) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    topk_select_kernel<<<dim3(2u * (unsigned)B), kKThreads, kKSmem, st>>>(scores, ld, seq_lens, K, idx);
    return cudaGetLastError();
}

}  // namespace mla
