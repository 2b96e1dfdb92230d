// decode_tc.cu -- tensor-core absorbed MLA decode for sm_103a (tcgen05 + TMA + 2-CTA clusters).
//
// What it computes, per request b, head h and visible position t ("DeepSeek's KV Cache: From
// 3.9 MB to 890 B per Token", Fig. 4 (1), Fig. 5 (2), Fig. 6 (2)):
//     s_t = scale * (q_lat[h] . c_t + q_rope[h] . k_rope_t)
//     out[h] = sum_t softmax(s)_t c_t,   lse[h] = ln sum_t exp(s_t).
// All 128 heads share each cached latent row, so per 64-position tile (one cache page) the work is
// two dense contractions: S[128 x 64] = Q[128 x 576] K^T and O[128 x 512] += P[128 x 64] V[64 x 512],
// V being the first 512 columns of the same rows.
//
// Capacity drives the design.  O (128 x 512 fp32) fills all 512 columns of one SM's tensor memory
// and Q (128 x 576 bf16, 144 KB) most of its shared memory, so the work runs on clusters of two
// CTAs, r = 0, 1.  CTA r owns latent dims [256 r, 256 r + 256) and rope dims [32 r, 32 r + 32):
//   * it streams only its 288 columns of every cached row (576 B per position) through a 3-page
//     TMA ring, and holds only its half of Q: the latent part in tensor memory (written by the
//     softmax warps, which read it from global memory once per request), the rope part in shared
//     memory;
//   * S_r = Q_r K_r^T is a partial score over its 288 dims, for all 128 heads (16 MMAs of
//     128x64x16 with Q from tensor memory and 2 with Q from shared memory per page);
//   * O_r[128 x 256] += P V_r (4 MMAs of 128x256x16, P and V from shared memory), V_r being the
//     latent half already in the stage: nothing is loaded twice and no FLOP is repeated.
// The softmax is split by heads: CTA r finishes heads [64 r, 64 r + 64) ("owned" heads).  Per page
// it receives the peer's partial scores of its owned heads (16 KB fp32) through distributed shared
// memory, computes P for them into its own P buffer and copies those rows (8 KB bf16, one bulk
// copy per 32 heads) into the peer's, so that each CTA ends up with P for all 128 heads.  That
// halves both the exchange and the exponentials against exchanging all scores.  Each CTA's MMA
// issuer signals the completion of its PV to both CTAs (the buffer is free once both are done).
// The online softmax runs in the log2 domain with a lazily updated running max: the max of a
// segment's first page is kept until a later score exceeds it by 2^16, so the common page needs
// no row reduction and never touches O; a vote among the warps sharing a head detects the rare
// page that does.  Its rescale factors travel with P; the peer's MMA issuer reads them and, when
// one differs from 1, has that CTA's receiver warps rescale those O rows before the page's PV.
// O is normalised by the sum of the bf16 P values the PV multiplied (the weights sum to one
// exactly), the log-sum-exp uses the sum of the fp32 values.
//
// Tensor memory (512 columns): O_r [0, 256), two score buffers [256 + 64 k), Q_r latent
// [384, 512) (two bf16 per column).
//
// Scheduling: the grid is a fixed set of C clusters (at most one per SM pair).  The pages of all
// requests form one stream of W tiles; cluster c takes tiles [c W / C, (c + 1) W / C), so every
// cluster gets the same work whatever the length mix.  A cluster walks its range request by
// request ("segments"); a segment that covers a whole request writes the final output, one cut
// by a range boundary writes a partial (normalised output + lse) into slot 2c (the range's first
// segment) or 2c + 1 (its last), and a merge kernel combines the partials of cut requests.
//
// Warp roles (576 threads): warp 0 TMA producer; warp 1 MMA issuer (+ TMEM owner); warps 2-17:
// thread = head = TMEM lane, four warps per 32-lane group, 16 positions of a page each.  The 8
// warps on the owned heads' lanes run the softmax ("owners"); on the other heads' lanes four
// "forwarders" send this CTA's partial scores of those heads to the peer and four "receivers"
// apply the rare rescales and finish those O rows.  Every wait is bounded: on expiry the
// kernel records MLA_ERR_TIMEOUT, stops issuing, drains its copies and MMAs, frees TMEM, returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "decode_common.cuh"

namespace mla {
namespace {

using namespace ptx;
using namespace dc;

constexpr int kNS = 3;                 // KV ring stages (pages)
constexpr int kNSB = 2;                // score buffers in TMEM (read early in a page's chain)
constexpr int kNP = 2;                 // P buffers in shared memory (held until both PVs are done)
constexpr int kNX = 2;                 // partial-score exchange buffers
constexpr int kSegCost = 4;           // a segment start costs about four pages (schedule units)
constexpr int kQKAhead = kNS - 1;      // QK may run this many tiles ahead of PV
constexpr int kSoftmaxThreads = 512;   // 16 warps: 8 owners, 4 forwarders, 4 receivers
constexpr int kScoreReaders = 12;      // owners and forwarders read each score buffer
constexpr int kOwnerWarps = 8;         // write P and finish the owned heads' O rows
constexpr int kORowWarps = 12;         // owners and receivers finish O rows
constexpr int kSlice = kT / 4;         // positions per warp
constexpr int kThreads = 64 + kSoftmaxThreads;
constexpr float kLazySlack = 16.0f;    // running max kept until a row max exceeds it by 2^16
constexpr int kHalfLat = 256;          // latent dims per CTA
constexpr int kHalfRope = 32;          // rope dims per CTA
constexpr int kOwned = 64;             // heads whose softmax a CTA finishes
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;         // O_r: columns [0, 256)
constexpr uint32_t kTmemS = 256;       // score buffer k: columns [256 + 64 k, 320 + 64 k)
constexpr uint32_t kTmemQ = 384;       // Q_r latent: columns [384, 512), two bf16 per column
constexpr uint32_t kDrainLimit = 1u << 20;

// shared-memory layout (bytes from a 1024-aligned base)
constexpr int kQRopeBytes = 128 * 64;                  // [128 heads x 32 dims] bf16, SW64
constexpr int kKvLatChunk = kT * 128;                  // [64 pos x 64 dims], SW128
constexpr int kKvRope = kT * 64;                       // [64 pos x 32 dims], SW64
constexpr int kStageBytes = 4 * kKvLatChunk + kKvRope;  // 36864
constexpr int kXBytes = kOwned * kT * 4;               // peer partial scores of owned heads, fp32
constexpr int kPBytes = 128 * kT * 2;                  // P [128 heads x 64 pos] bf16, SW128
constexpr int kPMsgBytes = 2 * (32 * 128 + 32 * 4);    // the peer's P rows and rescale factors
constexpr int kOffQRope = 0;
constexpr int kOffKv = kOffQRope + kQRopeBytes;        // 8192
constexpr int kOffX = kOffKv + kNS * kStageBytes;      // 118784: 2 buffers [16][64][16 B]
constexpr int kOffP = kOffX + kNX * kXBytes;           // kNP P buffers
constexpr int kOffAlphaIn = kOffP + kNP * kPBytes;     // kNP x alpha[64] of the peer's heads
constexpr int kOffAlphaOut = kOffAlphaIn + kNP * kOwned * 4;   // kNP x alpha[64], owned heads
constexpr int kOffLIn = kOffAlphaOut + kNP * kOwned * 4;  // 2 x l[64] of the peer's heads
// epilogue staging, 2 KB per softmax warp: [32 rows x 64 B], 64-byte swizzle (the TMA store box)
constexpr int kOffStage = (kOffLIn + 2 * kOwned * 4 + 1023) / 1024 * 1024;
constexpr int kStageOut = 2048;
constexpr int kOffBar = kOffStage + 12 * kStageOut;   // owners and receivers
constexpr int kNumBars = 2 * kNS + 2 * kNSB + 2 * kNP + 2 * kNX + 2 + 5 + 2;
constexpr int kOffRed = kOffBar + 8 * kNumBars;        // per-head exchange between slices [4][128]
constexpr int kSmemBytes = kOffRed + 4 * 128 * 4 + 1024;   // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(kOffP % 1024 == 0 && kPBytes % 1024 == 0, "P buffers on 128-byte swizzle atoms");


struct TcParams {
    const __nv_bfloat16* q_lat;   // [B][128][512]
    const int32_t* block_table;
    const int32_t* seq_lens;
    __nv_bfloat16* out;
    float* lse;
    float* o_part;          // [2C][128][512]
    float* lse_part;        // [2C][128]
    int32_t* meta;          // per request: first partial slot, last cluster (2 x int32)
    DevCtl* ctl;
    int64_t num_pages;
    int max_pages;
    int max_seq_len;
    int B;
    float scale_log2;       // scale * log2(e)
};

struct Bars {
    uint32_t kv_full, kv_empty;   // arrays of kNS
    uint32_t s_full, s_empty;     // arrays of kNSB
    uint32_t p_full, p_empty;     // arrays of kNP
    uint32_t x_full, x_free;      // arrays of kNX
    uint32_t l_full;              // array of 2
    uint32_t q_full, q_empty, o_full, o_free, mma_drain;
    uint32_t resc_req, resc;      // a rescale of the peer's heads' O rows: asked, done
    __device__ __forceinline__ uint32_t kvf(int i) const { return kv_full + 8 * i; }
    __device__ __forceinline__ uint32_t kve(int i) const { return kv_empty + 8 * i; }
    __device__ __forceinline__ uint32_t sf(int i) const { return s_full + 8 * i; }
    __device__ __forceinline__ uint32_t se(int i) const { return s_empty + 8 * i; }
    __device__ __forceinline__ uint32_t pf(int i) const { return p_full + 8 * i; }
    __device__ __forceinline__ uint32_t pe(int i) const { return p_empty + 8 * i; }
    __device__ __forceinline__ uint32_t xf(int i) const { return x_full + 8 * i; }
    __device__ __forceinline__ uint32_t xe(int i) const { return x_free + 8 * i; }
    __device__ __forceinline__ uint32_t lf(int i) const { return l_full + 8 * i; }
};

__device__ __forceinline__ Bars make_bars(uint32_t a) {
    Bars b;
    b.kv_full = a; a += 8 * kNS;
    b.kv_empty = a; a += 8 * kNS;
    b.s_full = a; a += 8 * kNSB;
    b.s_empty = a; a += 8 * kNSB;
    b.p_full = a; a += 8 * kNP;
    b.p_empty = a; a += 8 * kNP;
    b.x_full = a; a += 8 * kNX;
    b.x_free = a; a += 8 * kNX;
    b.l_full = a; a += 16;
    b.q_full = a; a += 8;
    b.q_empty = a; a += 8;
    b.o_full = a; a += 8;
    b.o_free = a; a += 8;
    b.mma_drain = a; a += 8;
    b.resc_req = a; a += 8;
    b.resc = a; a += 8;
    return b;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_qlat,
                     const __grid_constant__ CUtensorMap tm_qrope,
                     const __grid_constant__ CUtensorMap tm_kv_lat,
                     const __grid_constant__ CUtensorMap tm_kv_rope,
                     const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_opart,
                     TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ uint32_t s_tmem_base;
    __shared__ volatile int s_abort;
    __shared__ int s_start_b, s_start_t;
    __shared__ int s_n_local;
    __shared__ volatile int s_resc_page;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t r = cluster_rank();
    const uint32_t peer = r ^ 1u;
    const int c = blockIdx.x >> 1;
    const int C = gridDim.x >> 1;
    const uint32_t wait_limit = p.ctl->wait_limit;

    const uint32_t sbase = smem_u32(sm);
    const Bars bars = make_bars(sbase + kOffBar);

    // ---- schedule (warp 0): W = sum_b ceil(n_b / 64); this cluster's tiles [g_begin, g_end).
    // Cluster 0 also records, per request, where its partials are: the first slot and the last
    // cluster of the ranges it touches (first slot -1: no tiles).
    if (tid == 0) {
        s_abort = 0;
        s_start_b = p.B;
        s_start_t = 0;
        s_n_local = 0;
    }
    __syncthreads();
    if (warp == 0)
        schedule_warp(p.seq_lens, p.max_seq_len, p.B, 0, kSegCost, c, C, c == 0 && r == 0, p.meta, p.ctl,
                      &s_n_local, &s_start_b, &s_start_t);

    if (tid == 32) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(bars.kvf(i), 1);
            mbar_init(bars.kve(i), 1);
        }
        for (int i = 0; i < kNSB; ++i) {
            mbar_init(bars.sf(i), 1);
            mbar_init(bars.se(i), kScoreReaders);   // one arrive per warp reading scores
        }
        for (int i = 0; i < kNP; ++i) {
            // P ready: one arrive per owner warp (one of them with the peer's bytes)
            mbar_init(bars.pf(i), kOwnerWarps);
            mbar_init(bars.pe(i), 2);    // the PV completion of both CTAs of the pair
        }
        for (int i = 0; i < kNX; ++i) {
            mbar_init(bars.xf(i), 1);
            mbar_init(bars.xe(i), 8);    // one remote arrive per peer owner warp
        }
        for (int i = 0; i < 2; ++i) mbar_init(bars.lf(i), 1);
        // per segment: the producer's rope copy (with its bytes) and every score-reading warp's
        // share of the latent half in tensor memory
        mbar_init(bars.q_full, 1 + kScoreReaders);
        mbar_init(bars.q_empty, 1);
        mbar_init(bars.o_full, 1);
        mbar_init(bars.o_free, kORowWarps);   // one arrive per warp finishing O rows
        mbar_init(bars.mma_drain, 1);
        mbar_init(bars.resc_req, 1);
        mbar_init(bars.resc, 4);             // one arrive per receiver warp
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&s_tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();   // the peer's barriers are initialised before any remote arrive / st.async
    const uint32_t tmem = s_tmem_base;
    const int n_local = s_n_local;   // tiles of this cluster
    const int start_b = s_start_b, start_t = s_start_t;

    if (n_local == 0 && warp >= 2) {
        // an empty range: its partial slots must not contribute to any merge
        const int h = tid - 64;
        if (r == 0 && h < kHeads) {
            p.lse_part[(size_t)(2 * c) * kHeads + h] = -INFINITY;
            p.lse_part[(size_t)(2 * c + 1) * kHeads + h] = -INFINITY;
        }
    }

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0 && n_local > 0) {
            tma_prefetch_desc(&tm_qlat);
            tma_prefetch_desc(&tm_qrope);
            tma_prefetch_desc(&tm_kv_lat);
            tma_prefetch_desc(&tm_kv_rope);
            Cursor cu;
            cu.init(p.seq_lens, p.max_seq_len, 0, start_b, start_t, n_local);
            int seg = 0, issued = 0;
            for (int i = 0; i < n_local; ++i, cu.next(p.seq_lens, p.max_seq_len, p.B, 0)) {
                if (s_abort) break;
                if (cu.first()) {
                    if (seg > 0 && !mbar_wait(bars.q_empty, (seg - 1) & 1, wait_limit)) {
                        fail(p.ctl, &s_abort, 1);
                        break;
                    }
                    const int qrow = cu.b * kHeads;
                    mbar_arrive_expect_tx(bars.q_full, kQRopeBytes);
                    tma_load_2d(sbase + kOffQRope, &tm_qrope, bars.q_full, (int)r * kHalfRope, qrow);
                    ++seg;
                }
                const int s = i % kNS;
                if (!mbar_wait(bars.kve(s), ((i / kNS) & 1) ^ 1, wait_limit)) {
                    fail(p.ctl, &s_abort, 2);
                    break;
                }
                const int page = p.block_table[(size_t)cu.b * p.max_pages + cu.t];
                int row = -2 * kPage;   // outside the pool: the tile reads as zeros
                if (page >= 0 && page < p.num_pages) row = page * kPage;
                else if (r == 0) record_error(p.ctl, MLA_ERR_BOUNDS, page);
                const uint32_t st = sbase + kOffKv + s * kStageBytes;
                mbar_arrive_expect_tx(bars.kvf(s), kStageBytes);
                for (int k = 0; k < 4; ++k)
                    tma_load_2d(st + k * kKvLatChunk, &tm_kv_lat, bars.kvf(s),
                                (int)r * kHalfLat + 64 * k, row);
                tma_load_2d(st + 4 * kKvLatChunk, &tm_kv_rope, bars.kvf(s), kDc + (int)r * kHalfRope,
                            row);
                issued = i + 1;
                if (cu.last() && i + 1 < n_local) {
                    // the next request's latent Q, which the softmax warps read into tensor memory
                    // once this segment's QKs are done, into L2
                    Cursor cn = cu;
                    cn.next(p.seq_lens, p.max_seq_len, p.B, 0);
                    for (int k = 0; k < 4; ++k)
                        tma_prefetch_l2_2d(&tm_qlat, (int)r * kHalfLat + 64 * k, cn.b * kHeads);
                }
            }
            // drain: every load issued lands before this CTA may exit
            for (int j = max(0, issued - kNS); j < issued; ++j)
                mbar_wait(bars.kvf(j % kNS), (j / kNS) & 1, kDrainLimit);
            if (seg > 0) mbar_wait(bars.q_full, (seg - 1) & 1, kDrainLimit);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop so that its operands stay warp-uniform (cheap to issue);
        // one elected lane issues each MMA and commit.
        if (n_local > 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, kT, 0, 0);
            constexpr uint32_t id_pv = idesc_bf16(128, kHalfLat, 0, 1);
            // descriptor words: the low word carries the start address (bits 4..17 of the shared
            // address), so an offset inside a buffer is a 32-bit add to a masked base; the high
            // word (stride, version, swizzle) is constant
            const uint64_t lat_hi = smem_desc(0, 16, 1024, kSw128) & 0xFFFFFFFF00000000ull;
            const uint64_t rope_hi = smem_desc(0, 16, 512, kSw64) & 0xFFFFFFFF00000000ull;
            const uint64_t v_hi = smem_desc(0, kKvLatChunk, 1024, kSw128) & 0xFFFFFFFF00000000ull;
            const uint32_t lat_lo = (uint32_t)smem_desc(0, 16, 1024, kSw128);
            const uint32_t rope_lo = (uint32_t)smem_desc(0, 16, 512, kSw64);
            const uint32_t v_lo = (uint32_t)smem_desc(0, kKvLatChunk, 1024, kSw128);
            const uint32_t qr_lo = rope_lo + (((sbase + kOffQRope) >> 4) & 0x3FFF);
            Cursor cq, cp;
            cq.init(p.seq_lens, p.max_seq_len, 0, start_b, start_t, n_local);
            cp = cq;
            int iq = 0, ip = 0, seg_q = 0, seg_p = 0;
            int asked = -1, n_resc = 0;
            bool grow = false;
            uint32_t polls = 0;
            // Poll both queues: issue the next QK (up to kQKAhead tiles ahead of PV) when its
            // inputs are ready, else the next PV when its P is ready, so that neither a late KV
            // stage nor the next request's Q can hold back a PV.  Lane 0's view of the barriers
            // decides for the warp.
            while (ip < n_local && !__any_sync(0xffffffffu, s_abort)) {
                if (iq < n_local && iq <= ip + kQKAhead) {
                    const int s = iq % kNS, sb = iq % kNSB;
                    const bool ready = __shfl_sync(
                        0xffffffffu,
                        (!cq.first() || mbar_test(bars.q_full, seg_q & 1)) &&
                            mbar_test(bars.kvf(s), (iq / kNS) & 1) &&
                            mbar_test(bars.se(sb), ((iq / kNSB) & 1) ^ 1),
                        0);
                    if (ready) {
                        tc_fence_after();
                        const uint32_t st_lo = ((sbase + kOffKv + s * kStageBytes) >> 4) & 0x3FFF;
                        const uint32_t d = tmem + kTmemS + sb * kT;
                        if (elect_one()) {
#pragma unroll
                            for (int k = 0; k < 4; ++k)
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    mma_bf16_ts(d, tmem + kTmemQ + 32 * k + 8 * kk,
                                                lat_hi | (st_lo + lat_lo + ((k * kKvLatChunk + kk * 32) >> 4)),
                                                id_qk, (k | kk) != 0 ? 1u : 0u);
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk)
                                mma_bf16_ss(d, rope_hi | (qr_lo + kk * 2),
                                            rope_hi | (st_lo + rope_lo + ((4 * kKvLatChunk + kk * 32) >> 4)),
                                            id_qk, 1u);
                            mma_commit(bars.sf(sb));
                            if (cq.last()) mma_commit(bars.q_empty);
                        }
                        __syncwarp();
                        if (cq.last()) ++seg_q;
                        cq.next(p.seq_lens, p.max_seq_len, p.B, 0);
                        ++iq;
                        polls = 0;
                        continue;
                    }
                }
                // PV of tile ip: O_r += P (shared memory, K-major) x V_r (stage, MN-major)
                const bool seg_first = cp.first();
                const int pb = ip % kNP;
                bool pv_ready = __shfl_sync(
                    0xffffffffu,
                    (!seg_first || seg_p == 0 || mbar_test(bars.o_free, (seg_p - 1) & 1)) &&
                        mbar_test(bars.pf(pb), (ip / kNP) & 1),
                    0);
                if (pv_ready) {
                    if (asked != ip) {
                        // a running max of the peer's heads grew on this page (rescale factor
                        // != 1): the receivers rescale those O rows here before this PV
                        const float* al = reinterpret_cast<const float*>(sm + kOffAlphaIn) + pb * kOwned;
                        grow = __any_sync(0xffffffffu, al[lane] != 1.0f || al[lane + 32] != 1.0f);
                        if (grow && lane == 0) {
                            s_resc_page = ip;
                            mbar_arrive(bars.resc_req);
                        }
                        asked = ip;
                    }
                    if (grow) pv_ready = __shfl_sync(0xffffffffu, mbar_test(bars.resc, n_resc & 1), 0);
                }
                if (!pv_ready) {
                    if (++polls > wait_limit) {
                        if (lane == 0) fail(p.ctl, &s_abort, 6);
                        break;
                    }
                    continue;
                }
                polls = 0;
                if (grow) {
                    ++n_resc;
                    grow = false;
                }
                tc_fence_after();
                const uint32_t v = ((sbase + kOffKv + (ip % kNS) * kStageBytes) >> 4) & 0x3FFF;
                const uint32_t pa = ((sbase + kOffP + pb * kPBytes) >> 4) & 0x3FFF;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kT / 16; ++kk)
                        mma_bf16_ss(tmem + kTmemO, lat_hi | (pa + lat_lo + ((kk * 32) >> 4)),
                                    v_hi | (v + v_lo + ((kk * 16 * 128) >> 4)), id_pv,
                                    (!seg_first || kk > 0) ? 1u : 0u);
                    // P buffer pb is free once both CTAs' PV of this page is done (each CTA's
                    // owners write their rows into both)
                    mma_commit_mc(bars.pe(pb), 0x3);
                    mma_commit(bars.kve(ip % kNS));
                    if (cp.last()) mma_commit(bars.o_full);
                }
                __syncwarp();
                if (cp.last()) ++seg_p;
                cp.next(p.seq_lens, p.max_seq_len, p.B, 0);
                ++ip;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ owners and agents
        // Lane group lg = warp % 4 (the TMEM lanes this warp may access: heads 32 lg .. 32 lg + 31,
        // thread = head), slice ts = (warp - 2) / 4 (positions 16 ts .. 16 ts + 15 of a page, and
        // O columns 64 ts .. 64 ts + 63 in corrections and epilogues).  Lane groups 2r, 2r + 1
        // hold the owned heads.
        //
        // The four owner warps of a lane group meet at named barriers (ids 1 + lg, 5 + lg, 128
        // threads), which cannot time out, so these loops never leave early: after a failed
        // (bounded) wait they keep executing every barrier but skip the work, and waits return at
        // once.  Wait results are made warp-uniform before any warp-collective tcgen05 instruction.
        const int lg = warp & 3;
        const int ts = (warp - 2) >> 2;
        const int h = lg * 32 + lane;
        const bool owner = (lg >> 1) == (int)r;
        const int hh = h & (kOwned - 1);   // index among the owning CTA's heads
        const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
        float* red = reinterpret_cast<float*>(sm + kOffRed);   // [4 slices][128 heads]

        auto wwait = [&](uint32_t bar, uint32_t parity, int where) -> bool {
            // common case first: the phase is complete by the first try
            if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
            bool ok = !s_abort && mbar_wait(bar, parity, wait_limit);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0) fail(p.ctl, &s_abort, where);
            return ok;
        };

        // Q_r latent of request b into tensor memory: columns [c0, c0 + 32 n) of this warp's 32
        // lanes (two bf16 per column, lower dim in the low half: the order of the dims in memory),
        // then this warp's share of the segment's Q is in place
        auto load_q = [&](int b, int c0, int n) {
            if (__any_sync(0xffffffffu, s_abort)) return;
            const uint4* src = reinterpret_cast<const uint4*>(
                p.q_lat + ((size_t)b * kHeads + h) * kDc + (int)r * kHalfLat + 2 * c0);
#pragma unroll 1
            for (int half = 0; half < n; ++half) {
                uint32_t q[32];   // 64 dims: all eight loads in flight before the store
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint4 v = __ldg(src + 8 * half + k);
                    q[4 * k] = v.x;
                    q[4 * k + 1] = v.y;
                    q[4 * k + 2] = v.z;
                    q[4 * k + 3] = v.w;
                }
                tmem_st32(tmem + lane_off + kTmemQ + c0 + 32 * half, q);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.q_full);
        };

        // this CTA's partial scores of page i for the warp's 16 positions (TMEM -> registers)
        auto load_s = [&](int i, uint32_t (&v)[16]) -> bool {
            const int sb = i % kNSB;
            if (!wwait(bars.sf(sb), (i / kNSB) & 1, 7)) return false;
            tc_fence_after();
            tmem_ld16(tmem + lane_off + kTmemS + sb * kT + kSlice * ts, v);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.se(sb));
            return true;
        };

        // O rows of this warp (columns [col0, col0 + 32 n)) times alpha, once PV of page i - 1
        // has completed
        auto rescale_o = [&](int i, float alpha, int col0, int n) {
            if (!wwait(bars.pe((i - 1) % kNP), ((i - 1) / kNP) & 1, 10)) return;
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < n; ++cc) {
                const uint32_t col = kTmemO + col0 + 32 * cc;
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + col, o);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                tmem_st32(tmem + lane_off + col, o);
            }
            tmem_wait_st();
        };

        // O rows of this warp (columns [col0, col0 + 32 n)) normalised by l (row sum) into the
        // output (bf16) or a partial slot (fp32).  The rows go out through the warp's staging
        // buffer and TMA stores of [32 rows x 64 B] boxes (a thread holds one row, so direct
        // stores would touch 32 lines per instruction); O is released to the next segment's PV
        // once its last columns are in registers.
        auto epilogue_rows = [&](int seg, const Cursor& cu, bool partial, float l_row, int col0, int n) {
            const int slot = 2 * c + (seg == 0 ? 0 : 1);
            const bool ok = wwait(bars.o_full, seg & 1, 12);
            if (ok) {
                tc_fence_after();
                const float inv = l_row > 0.f ? 1.0f / l_row : 0.0f;
                const int si = owner ? (lg & 1) * 4 + ts : 8 + (lg & 1) * 2 + (ts - 2);   // staging buffer
                uint8_t* stg = sm + kOffStage + si * kStageOut;
                const uint32_t stg_s = sbase + kOffStage + si * kStageOut;
                uint8_t* srow = stg + lane * 64;
                const int sw = (lane >> 1) & 3;   // 64-byte swizzle: chunk j at j ^ sw
                const int row0 = (partial ? slot : cu.b) * kHeads + lg * 32;
                auto put = [&](const CUtensorMap* m, int x, const uint32_t (&w)[16]) {
                    if (lane == 0) bulk_wait_read0();   // the previous box has left the buffer
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        st_shared_v4(srow + ((j ^ sw) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tma_store_2d(m, stg_s, x, row0);
                };
#pragma unroll 1
                for (int cc = 0; cc < n; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_off + kTmemO + col0 + 32 * cc, o);
                    tmem_wait_ld();
                    if (cc == n - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bars.o_free);
                    }
                    const int col = (int)r * kHalfLat + col0 + 32 * cc;
                    uint32_t w[16];
                    if (!partial) {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            w[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv);
                        put(&tm_out, col, w);
                    } else {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                            for (int k = 0; k < 16; ++k) w[k] = __float_as_uint(__uint_as_float(o[16 * hf + k]) * inv);
                            put(&tm_opart, col + 16 * hf, w);
                        }
                    }
                }
            } else {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.o_free);
            }
        };

        Cursor cu;
        cu.init(p.seq_lens, p.max_seq_len, 0, start_b, start_t, n_local);
        int seg = 0;
        bool cut_front = false;

        if (!owner && ts < 2) {
            // ------------------------------------------------------------ forwarders
            // this CTA's partial scores of the peer's heads to the peer, 32 positions per warp
            const uint32_t x_remote = mapa(sbase + kOffX, peer);
            const uint32_t xfull_remote = mapa(bars.x_full, peer);
            if (n_local > 0) load_q(cu.b, 64 * ts, 2);
            for (int i = 0; i < n_local; ++i, cu.next(p.seq_lens, p.max_seq_len, p.B, 0)) {
                const int sb = i % kNSB;
                if (!wwait(bars.sf(sb), (i / kNSB) & 1, 7)) continue;
                uint32_t v[32];
                tc_fence_after();
                tmem_ld32(tmem + lane_off + kTmemS + sb * kT + 32 * ts, v);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.se(sb));
                const int xb = i % kNX;
                // already in log2 units (times scale log2(e)): the owner adds its own part with an FMA
#pragma unroll
                for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * p.scale_log2);
                if (wwait(bars.xe(xb), ((i / kNX) & 1) ^ 1, 8)) {
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        st_async_v4(x_remote + xb * kXBytes + ((8 * ts + g) * kOwned + hh) * 16,
                                    xfull_remote + 8 * xb, v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
                }
                if (cu.last() && i + 1 < n_local) {
                    // the segment's QKs are done: the next request's Q, this warp's 64 columns
                    Cursor cn = cu;
                    cn.next(p.seq_lens, p.max_seq_len, p.B, 0);
                    load_q(cn.b, 64 * ts, 2);
                }
            }
        } else if (!owner) {
            // ------------------------------------------------------------ receivers
            // this CTA's O rows of the peer's heads: the rare rescales the MMA issuer asks for (a
            // running max of those heads grew by more than the slack) and each segment's
            // epilogue, 128 columns per warp
            const int rts = ts - 2;
            const bool lead = (rts == 0 && lg == 2 * (int)peer && lane == 0);
            int n_req = 0;
            for (int i = 0; i < n_local; ++i, cu.next(p.seq_lens, p.max_seq_len, p.B, 0)) {
                if (cu.first()) cut_front = cu.t > 0;
                if (!cu.last()) continue;
                // until the segment's last PV completes, its rescales in page order (a request
                // always names a page of this segment: its PV waits for the rescale, and the
                // next segment's PVs wait for this segment's epilogue)
                uint32_t polls = 0;
                while (!__any_sync(0xffffffffu, s_abort)) {
                    if (__shfl_sync(0xffffffffu, mbar_test(bars.o_full, seg & 1), 0)) break;
                    if (__shfl_sync(0xffffffffu, mbar_test(bars.resc_req, n_req & 1), 0)) {
                        const int ir = s_resc_page;
                        ++n_req;
                        const float alpha =
                            reinterpret_cast<const float*>(sm + kOffAlphaIn)[(ir % kNP) * kOwned + hh];
                        rescale_o(ir, alpha, 128 * rts, 4);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bars.resc);
                        polls = 0;
                        continue;
                    }
                    if (++polls > wait_limit) {
                        if (lane == 0) fail(p.ctl, &s_abort, 13);
                        break;
                    }
                    __nanosleep(32);
                }
                const bool partial = cut_front || cu.t < cu.nt - 1;
                // the row sums of these heads, sent by the peer's owners
                if (lead && !s_abort) mbar_arrive_expect_tx(bars.lf(seg & 1), kOwned * 4);
                const bool lok = wwait(bars.lf(seg & 1), (seg >> 1) & 1, 14);
                const float l_row = lok ? reinterpret_cast<const float*>(sm + kOffLIn)[(seg & 1) * kOwned + hh] : 0.f;
                epilogue_rows(seg, cu, partial, l_row, 128 * rts, 4);
                ++seg;
            }
        } else {
            // ------------------------------------------------------------ owners
            const uint32_t p_remote = mapa(sbase + kOffP, peer);
            const uint32_t ain_remote = mapa(sbase + kOffAlphaIn, peer);
            const uint32_t pfull_remote = mapa(bars.p_full, peer);
            const uint32_t xfree_remote = mapa(bars.x_free, peer);
            const uint32_t lin_remote = mapa(sbase + kOffLIn, peer);
            const uint32_t lfull_remote = mapa(bars.l_full, peer);
            const bool lead = (ts == 0 && lg == 2 * (int)r && lane == 0);
            const uint32_t bar_vote = 1 + lg, bar_sync = 5 + lg;
            // row sums of P: l_part of the fp32 values (the log-sum-exp), lr_part of the bf16 values
            // the PV multiplies (the output's normaliser, so that the weights applied to the rows
            // sum to one exactly; with a running max below the true max the dominant P carries a
            // bf16 rounding that would otherwise show in the output)
            float m_used = -INFINITY, l_part = 0.f, lr_part = 0.f;
            if (n_local > 0) load_q(cu.b, 32 * ts, 1);
            for (int i = 0; i < n_local; ++i, cu.next(p.seq_lens, p.max_seq_len, p.B, 0)) {
                const int xb = i % kNX;
                const bool first = cu.first();
                if (first) {
                    m_used = -INFINITY;
                    l_part = 0.f;
                    lr_part = 0.f;
                    cut_front = cu.t > 0;   // the request started before this cluster's range
                }
                uint32_t v[16];
                const bool sok = load_s(i, v);
                if (cu.last() && i + 1 < n_local) {
                    // the segment's QKs are done: the next request's Q, this warp's 32 columns
                    Cursor cn = cu;
                    cn.next(p.seq_lens, p.max_seq_len, p.B, 0);
                    load_q(cn.b, 32 * ts, 1);
                }
                // the peer's partial scores of these heads for page i
                if (lead && !s_abort) mbar_arrive_expect_tx(bars.xf(xb), kXBytes);
                const bool xok = wwait(bars.xf(xb), (i / kNX) & 1, 9);
                const int nv = min(kT, cu.n - cu.t * kT) - kSlice * ts;   // valid positions here
                float x[16];
                const uint8_t* xp = sm + kOffX + xb * kXBytes;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float4 q = *reinterpret_cast<const float4*>(xp + ((4 * ts + g) * kOwned + hh) * 16);
                    x[4 * g] = fmaf(__uint_as_float(v[4 * g]), p.scale_log2, q.x);
                    x[4 * g + 1] = fmaf(__uint_as_float(v[4 * g + 1]), p.scale_log2, q.y);
                    x[4 * g + 2] = fmaf(__uint_as_float(v[4 * g + 2]), p.scale_log2, q.z);
                    x[4 * g + 3] = fmaf(__uint_as_float(v[4 * g + 3]), p.scale_log2, q.w);
                }
                // positions past the end of the request take no weight
                if (nv < 16) {
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if (t >= nv) x[t] = -INFINITY;
                }
                // every loaded value has been consumed: hand the exchange buffer back to the peer
                __syncwarp();
                if (lane == 0 && xok) mbar_arrive_remote_relaxed(xfree_remote + 8 * xb);
                // P = 2^(x - m) for this warp's positions, packed to bf16, with the running max m.
                // m is kept while every P of a row stays at most 2^16, so the common page needs no
                // row max: a thread whose 16 P sum past 2^16 (or not to a finite value) votes for
                // the rare path, as does every segment start.  There the exact page row max over
                // the four slices raises m where it exceeds m by more than the slack, O is rescaled
                // here and, through alpha sent with P, in the peer, and P is computed again.
                const int pb = i % kNP;
                bool pok = true;   // P buffer pb is free (checked once P is computed)
                float alpha = 1.0f;
                float psum, prsum;
                uint32_t pk[8];
                // this warp's 16 P of its lane's row: 16-byte chunks 2 ts, 2 ts + 1 of the 128-byte
                // row (chunk c stored at c ^ (row % 8): 128-byte swizzle), and the rescale factor
                const int lrow = lg * 32 + lane;   // P row = TMEM lane
                uint8_t* prow = sm + kOffP + pb * kPBytes + lrow * 128;
                auto write_p = [&]() {
                    if (!pok) return;
                    st_shared_v4(prow + (((2 * ts) ^ (lrow & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
                    st_shared_v4(prow + (((2 * ts + 1) ^ (lrow & 7)) << 4), pk[4], pk[5], pk[6], pk[7]);
                    if (ts == 0) reinterpret_cast<float*>(sm + kOffAlphaOut)[pb * kOwned + hh] = alpha;
                    fence_proxy_async_smem();
                };
                // (m = -inf only before a segment's first page has set it: P is then recomputed)
                auto exp_page = [&]() {
                    const float m = m_used == -INFINITY ? INFINITY : m_used;
                    float s0 = 0.f, s1 = 0.f, r0 = 0.f, r1 = 0.f;
#pragma unroll
                    for (int t = 0; t < 16; t += 2) {
                        const float p0 = ex2(x[t] - m), p1 = ex2(x[t + 1] - m);
                        s0 += p0;
                        s1 += p1;
                        pk[t / 2] = pack_bf16x2(p0, p1);
                        r0 += __uint_as_float(pk[t / 2] << 16);
                        r1 += __uint_as_float(pk[t / 2] & 0xFFFF0000u);
                    }
                    psum = s0 + s1;
                    prsum = r0 + r1;
                };
                exp_page();
                // both CTAs' PV of page i - kNP has completed: P buffer pb is free here and there
                pok = i < kNP || wwait(bars.pe(pb), ((i - kNP) / kNP) & 1, 11);
                write_p();
                const bool need = first || !(psum <= 65536.0f);
                if (bar_red_or(bar_vote, 128, need)) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int t = 0; t < 16; ++t) mx = fmaxf(mx, x[t]);
                    red[ts * 128 + h] = mx;
                    named_bar_sync(bar_sync, 128);
                    const float tmax = fmaxf(fmaxf(red[h], red[128 + h]), fmaxf(red[256 + h], red[384 + h]));
                    const bool grow = first || tmax > m_used + kLazySlack;
                    const float m_new = grow ? (first ? tmax : fmaxf(tmax, m_used)) : m_used;
                    if (!first) {
                        alpha = grow ? ex2(m_used - m_new) : 1.0f;
                        if (__any_sync(0xffffffffu, grow)) rescale_o(i, alpha, 64 * ts, 2);
                        l_part *= alpha;
                        lr_part *= alpha;
                    }
                    m_used = m_new;
                    exp_page();
                    write_p();
                    // red[] rows of this lane group are free again, its final P rows in place
                    named_bar_sync(bar_sync, 128);
                }
                l_part += psum;
                lr_part += prsum;
                // positions past the end of the request: zero their V rows so that
                // 0 * (stale bytes) cannot poison O (QK of this page has completed, PV has not
                // started); the owner warps of both lane groups share the rows
                const int nvalid = min(kT, cu.n - cu.t * kT);
                if (nvalid < kT && sok) {
                    uint8_t* st = sm + kOffKv + (i % kNS) * kStageBytes;
                    const int nrows = kT - nvalid;
                    const int ot = (lg & 1) * 128 + ts * 32 + lane;   // 0 .. 255 over the owners
                    for (int e = ot; e < nrows * 4 * 8; e += 256) {
                        const int row = nvalid + e / 32, k = (e / 8) % 4, part = e % 8;
                        *reinterpret_cast<uint4*>(st + k * kKvLatChunk + row * 128 + part * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                // the lane group's P rows and rescale factors (all four warps wrote theirs before
                // the vote or the barrier after the recompute) into the peer's P buffer
                if (ts == 0 && lane == 0 && pok && !s_abort) {
                    const uint32_t off = pb * kPBytes + lg * 32 * 128;
                    bulk_copy_s2c(p_remote + off, sbase + kOffP + off, 32 * 128, pfull_remote + 8 * pb);
                    const uint32_t aoff = (pb * kOwned + (lg & 1) * 32) * 4;
                    bulk_copy_s2c(ain_remote + aoff, sbase + kOffAlphaOut + aoff, 32 * 4, pfull_remote + 8 * pb);
                }
                // P ready for this CTA's PV (the lead arrival also expects the peer's bytes)
                __syncwarp();
                if (lane == 0 && pok && !s_abort) {
                    if (lead) mbar_arrive_expect_tx(bars.pf(pb), kPMsgBytes);
                    else mbar_arrive(bars.pf(pb));
                }

                if (cu.last()) {
                    // ------------------------------------------------------ segment epilogue
                    const bool partial = cut_front || cu.t < cu.nt - 1;
                    // (the other CTA's heads' entries of red[] hold the second sum)
                    red[ts * 128 + h] = l_part;
                    red[ts * 128 + (h ^ kOwned)] = lr_part;
                    named_bar_sync(bar_sync, 128);
                    const float l_row = (red[h] + red[128 + h]) + (red[256 + h] + red[384 + h]);
                    const int hr = h ^ kOwned;
                    const float lr_row = (red[hr] + red[128 + hr]) + (red[256 + hr] + red[384 + hr]);
                    named_bar_sync(bar_sync, 128);
                    // the normalisers of these heads to the peer, which finishes its O rows of them
                    if (ts == 0 && !s_abort)
                        st_async_b32(lin_remote + ((seg & 1) * kOwned + hh) * 4,
                                     lfull_remote + 8 * (seg & 1), __float_as_uint(lr_row));
                    const float L = l_row > 0.f ? (m_used + log2f(l_row)) * 0.6931471805599453f : -INFINITY;
                    if (ts == 0) {
                        const size_t row = (size_t)cu.b * kHeads + h;
                        if (!partial) p.lse[row] = L;
                        else p.lse_part[(size_t)(2 * c + (seg == 0 ? 0 : 1)) * kHeads + h] = L;
                    }
                    epilogue_rows(seg, cu, partial, lr_row, 64 * ts, 2);
                    ++seg;
                }
            }
        }
    }

    // ---------------------------------------------------------------------- teardown
    bulk_wait_read0();   // this thread's epilogue stores have read their staging buffers
    if (warp == 1 && n_local > 0) {
        __syncwarp();
        // all MMAs issued by the elected lane (the lowest active one, as in the loop) are complete
        // once this barrier flips
        if (elect_one()) {
            mma_commit(bars.mma_drain);
            if (!mbar_wait(bars.mma_drain, 0, kDrainLimit)) record_error(p.ctl, MLA_ERR_TIMEOUT, 16);
            // the peer's PV completion signals of the last kNP pages have landed here
            if (!s_abort)
                for (int j = max(0, n_local - kNP); j < n_local; ++j)
                    mbar_wait(bars.pe(j % kNP), (j / kNP) & 1, kDrainLimit);
        }
    }
    __syncwarp();
    if (s_abort) __nanosleep(100000);   // let any in-flight distributed-shared-memory stores land
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();   // the peer no longer writes into this CTA's shared memory
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

// Finish of mla_decode: requests cut by cluster range boundaries get their partials merged,
// requests with no visible position get zeros and lse = -inf; the rest were finished by the
// decode kernel.  Request b's partials sit in slot first (2 c_lo or 2 c_lo + 1) and slots 2c for
// the following clusters c up to c_hi.  Two shapes, both built so that the loads of a step are
// independent (a few memory latencies in all rather than one per slot):
//   * wide (few slots per request, many requests): block (b, heads 8 g .. 8 g + 7), warp = head;
//     lanes take slots for the log-sum-exp, then columns for the weighted row sum;
//   * deep (many slots, few requests): block (b, h); every warp forms the log-sum-exp, warp w
//     accumulates slots w, w + 8, ... over the whole row and shared memory sums the eight rows.
__device__ __forceinline__ float merge_lse(const float* __restrict__ lse_part, int first, int c_lo, int n,
                                           int h, int lane, float z) {
    // z: the head's sink (shared K = V entries; -inf for none), one more term of the sum
    float m = z;
    for (int k = lane; k < n; k += 32)
        m = fmaxf(m, __ldg(lse_part + (size_t)(k == 0 ? first : 2 * (c_lo + k)) * kHeads + h));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (m == -INFINITY) return -INFINITY;
    float l = lane == 0 && z != -INFINITY ? expf(z - m) : 0.f;
    for (int k = lane; k < n; k += 32)
        l += expf(__ldg(lse_part + (size_t)(k == 0 ? first : 2 * (c_lo + k)) * kHeads + h) - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    return m + logf(l);
}

// acc (this lane's columns 4 lane + 128 j of row h) += the weighted rows of slots k0, k0 + dk, ...
__device__ __forceinline__ void merge_rows(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                                           int first, int c_lo, int n, int k0, int dk, int h, int lane,
                                           float L, float4 (&acc)[4]) {
#pragma unroll 4
    for (int k = k0; k < n; k += dk) {
        const int slot = k == 0 ? first : 2 * (c_lo + k);
        const float w = expf(__ldg(lse_part + (size_t)slot * kHeads + h) - L);
        const float4* src = reinterpret_cast<const float4*>(o_part + ((size_t)slot * kHeads + h) * kDc) + lane;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 o = __ldg(src + 32 * j);
            acc[j].x += w * o.x;
            acc[j].y += w * o.y;
            acc[j].z += w * o.z;
            acc[j].w += w * o.w;
        }
    }
}

__global__ void __launch_bounds__(256) merge_wide_kernel(const float* __restrict__ o_part,
                                                         const float* __restrict__ lse_part,
                                                         const int32_t* __restrict__ meta,
                                                         __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                                         const float* __restrict__ sink) {
    const int b = blockIdx.x >> 4;
    const int lane = threadIdx.x & 31;
    const int h = (blockIdx.x & 15) * 8 + (threadIdx.x >> 5);
    const int first = __ldg(meta + 2 * b), c_hi = __ldg(meta + 2 * b + 1);
    const int c_lo = first >> 1;
    if (first >= 0 && c_hi == c_lo) return;   // inside one range: already final
    float4 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float z = sink != nullptr ? __ldg(sink + h) : -INFINITY;
    float L = z;   // no visible position: lse = ln exp(z') (-inf without a sink)
    if (first >= 0) {
        const int n = c_hi - c_lo + 1;
        L = merge_lse(lse_part, first, c_lo, n, h, lane, z);
        if (L != -INFINITY) merge_rows(o_part, lse_part, first, c_lo, n, 0, 1, h, lane, L, acc);
    }
    uint2* dst = reinterpret_cast<uint2*>(out + ((size_t)b * kHeads + h) * kDc) + lane;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint2 packed;
        packed.x = pack_bf16x2(acc[j].x, acc[j].y);
        packed.y = pack_bf16x2(acc[j].z, acc[j].w);
        dst[32 * j] = packed;
    }
    if (lane == 0) lse[(size_t)b * kHeads + h] = L;
}

__global__ void __launch_bounds__(256) merge_deep_kernel(const float* __restrict__ o_part,
                                                         const float* __restrict__ lse_part,
                                                         const int32_t* __restrict__ meta,
                                                         __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                                         const float* __restrict__ sink) {
    __shared__ float4 red[8][kDc / 4];
    const int b = blockIdx.x / kHeads, h = blockIdx.x % kHeads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int first = __ldg(meta + 2 * b), c_hi = __ldg(meta + 2 * b + 1);
    const int c_lo = first >> 1;
    if (first >= 0 && c_hi == c_lo) return;   // inside one range: already final (whole block)
    float4 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float z = sink != nullptr ? __ldg(sink + h) : -INFINITY;
    float L = z;   // no visible position: lse = ln exp(z') (-inf without a sink)
    if (first >= 0) {
        const int n = c_hi - c_lo + 1;
        L = merge_lse(lse_part, first, c_lo, n, h, lane, z);
        if (L != -INFINITY) merge_rows(o_part, lse_part, first, c_lo, n, warp, 8, h, lane, L, acc);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) red[warp][lane + 32 * j] = acc[j];
    __syncthreads();
    if (threadIdx.x < kDc / 4) {
        float4 t = red[0][threadIdx.x];
#pragma unroll
        for (int w = 1; w < 8; ++w) {
            const float4 u = red[w][threadIdx.x];
            t.x += u.x;
            t.y += u.y;
            t.z += u.z;
            t.w += u.w;
        }
        uint2 packed;
        packed.x = pack_bf16x2(t.x, t.y);
        packed.y = pack_bf16x2(t.z, t.w);
        reinterpret_cast<uint2*>(out + ((size_t)b * kHeads + h) * kDc)[threadIdx.x] = packed;
    }
    if (threadIdx.x == 0) lse[(size_t)b * kHeads + h] = L;
}

cudaError_t launch_merge_slots(const float* o_part, const float* lse_part, const int32_t* meta,
                               __nv_bfloat16* out, float* lse, int B, int C, cudaStream_t st, const float* sink) {
    if (B <= 0) return cudaSuccess;
    // a request spans about C / B + 1 cluster ranges
    if ((C + B - 1) / B + 1 <= 8) {
        const int64_t blocks = (int64_t)B * (kHeads / 8);
        if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
        merge_wide_kernel<<<(unsigned)blocks, 256, 0, st>>>(o_part, lse_part, meta, out, lse, sink);
    } else {
        const int64_t blocks = (int64_t)B * kHeads;
        if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
        merge_deep_kernel<<<(unsigned)blocks, 256, 0, st>>>(o_part, lse_part, meta, out, lse, sink);
    }
    return cudaGetLastError();
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &f, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

bool encode_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
               uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw, CUtensorMapDataType dt) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d(CUtensorMap* m, const void* base, const uint64_t dims[3], const uint64_t strides_bytes[2],
               const uint32_t box[3], CUtensorMapSwizzle sw, CUtensorMapDataType dt) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
    cuuint32_t bx[3] = {box[0], box[1], box[2]};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Workspace of the tensor-core path: 2 partial slots per cluster (fp32 [128][512] + lse [128]),
// then per request its first partial slot and last cluster (int32 [B][2]).
DecodePlan plan_decode_tc(int fmt, int B, int max_seq_len, int topk, int sms) {
    (void)fmt;
    (void)topk;
    DecodePlan p;
    const int C = clusters_for_tiles((long long)B * ((max_seq_len + kT - 1) / kT), sms);
    p.splits = C;
    p.workspace = (size_t)2 * C * kHeads * (kDc + 1) * sizeof(float) + (size_t)2 * B * sizeof(int32_t);
    p.workspace = (p.workspace + 255) / 256 * 256;
    p.launches = 2;
    return p;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t st) {
    if (a.fmt != MLA_KV_BF16 || a.topk_idx != nullptr) return cudaErrorNotSupported;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    CUtensorMap tm_qlat, tm_qrope, tm_kv_lat, tm_kv_rope, tm_out, tm_opart;
    const uint64_t qrows = (uint64_t)a.B * kHeads;
    const uint64_t kv_rows = (uint64_t)a.num_pages * kPage;
    if (!encode_2d(&tm_qlat, a.q_lat, kDc, qrows, kDc * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tm_qrope, a.q_rope, kDr, qrows, kDr * 2, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_2d(&tm_kv_lat, a.pool, kDk, kv_rows, kBf16RecordBytes, 64, kT,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tm_kv_rope, a.pool, kDk, kv_rows, kBf16RecordBytes, 32, kT,
                   CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    const int C = plan.splits;
    float* o_part = static_cast<float*>(a.workspace);
    float* lse_part = o_part + (size_t)2 * C * kHeads * kDc;
    int32_t* meta = reinterpret_cast<int32_t*>(lse_part + (size_t)2 * C * kHeads);
    // epilogue boxes: 32 rows x 32 bf16 of the output, 32 rows x 16 fp32 of a partial slot
    if (!encode_2d(&tm_out, a.out, kDc, qrows, kDc * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_2d(&tm_opart, o_part, kDc, (uint64_t)2 * C * kHeads, kDc * 4, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
        return cudaErrorInvalidValue;
    TcParams p;
    p.q_lat = a.q_lat;
    p.block_table = a.block_table;
    p.seq_lens = a.seq_lens;
    p.out = a.out;
    p.lse = a.lse;
    p.o_part = o_part;
    p.lse_part = lse_part;
    p.meta = meta;
    p.ctl = a.ctl;
    p.num_pages = a.num_pages;
    p.max_pages = a.max_pages;
    p.max_seq_len = a.max_seq_len;
    p.B = a.B;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    decode_tc_kernel<<<2 * C, kThreads, kSmemBytes, st>>>(tm_qlat, tm_qrope, tm_kv_lat, tm_kv_rope, tm_out,
                                                         tm_opart, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_merge_slots(o_part, lse_part, meta, a.out, a.lse, a.B, C, st);
}

}  // namespace mla
