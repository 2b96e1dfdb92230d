// decode_tc.cu -- tensor-core absorbed MLA decode for sm_103a (tcgen05 + TMA + 2-CTA clusters).
//
// What it computes, per request b, head h and visible position t ("DeepSeek's KV Cache: From
// 3.9 MB to 890 B per Token", Fig. 4 (1), Fig. 5 (2), Fig. 6 (2)):
//     s_t = scale * (q_lat[h] . c_t + q_rope[h] . k_rope_t)
//     out[h] = sum_t softmax(s)_t c_t,   lse[h] = ln sum_t exp(s_t).
// All 128 heads share each cached latent row, so per 32-position tile the work is two dense
// contractions: S[128 x 32] = Q[128 x 576] K^T and O[128 x 512] += P[128 x 32] V[32 x 512], with
// V = the first 512 columns of the same rows.
//
// Capacity drives the design.  O (128 x 512 fp32) fills all 512 columns of one SM's tensor memory
// and Q (128 x 576 bf16, 144 KB) most of its shared memory, so one work unit runs on a cluster of
// two CTAs, r = 0, 1.  CTA r owns latent dims [256 r, 256 r + 256) and rope dims [32 r, 32 r + 32):
//   * it streams only its 288 columns of every cached row (576 B per position) through a
//     5-stage TMA ring, and holds only its half of Q (72 KB);
//   * S_r = Q_r K_r^T is a partial score over its 288 dims (18 MMAs of 128x32x16 per tile);
//   * the 128 softmax threads (one per head) send S_r to the peer CTA through distributed shared
//     memory (st.async, 16 KB per tile), add the peer's part: both CTAs then hold the same fp32
//     scores, bit for bit, and take identical softmax decisions;
//   * P (bf16) goes to shared memory and O_r[128 x 256] += P V_r (2 MMAs of 128x256x16), V_r being
//     the latent half already in the stage: nothing is loaded twice and no FLOP is repeated.
// The online softmax runs in the log2 domain with a lazily updated running max (O is rescaled only
// when a row max grows by more than 2^8), so the common tile never touches O.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer (+ TMEM owner), warps 2-5
// softmax / exchange / epilogue (thread = head = TMEM lane).  Every wait is bounded: on expiry the
// kernel records MLA_ERR_TIMEOUT, stops issuing, drains its copies and MMAs, frees TMEM, returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "mla_internal.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kT = 32;                 // positions per tile
constexpr int kNS = 5;                 // KV ring stages
constexpr int kThreads = 192;
constexpr int kHalfLat = 256;          // latent dims per CTA
constexpr int kHalfRope = 32;          // rope dims per CTA
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;         // O_r: columns [0, 256)
constexpr uint32_t kTmemS = 256;       // S buffers: [256 + 32 k, 256 + 32 k + 32), k = 0, 1
constexpr uint32_t kDrainLimit = 1u << 20;

// shared-memory layout (bytes from a 1024-aligned base)
constexpr int kQLatChunk = 128 * 128;                  // [128 heads x 64 dims] bf16, SW128
constexpr int kQRopeBytes = 128 * 64;                  // [128 heads x 32 dims] bf16, SW64
constexpr int kKvLatChunk = kT * 128;                  // [32 pos x 64 dims], SW128
constexpr int kKvRope = kT * 64;                       // [32 pos x 32 dims], SW64
constexpr int kStageBytes = 4 * kKvLatChunk + kKvRope;  // 18432
constexpr int kXBytes = 128 * kT * 4;                  // peer partial scores, fp32 [8][128][4]
constexpr int kPBytes = 128 * kT * 2;                  // P [128 heads x 32 pos] bf16, SW64
constexpr int kOffQ = 0;
constexpr int kOffQRope = kOffQ + 4 * kQLatChunk;      // 65536
constexpr int kOffKv = kOffQRope + kQRopeBytes;        // 73728
constexpr int kOffX = kOffKv + kNS * kStageBytes;      // 165888
constexpr int kOffP = kOffX + 2 * kXBytes;             // 198656
constexpr int kOffBar = kOffP + 2 * kPBytes;           // 215040
constexpr int kNumBars = 2 * kNS + 2 + 2 * 6;
constexpr int kSmemBytes = kOffBar + 8 * kNumBars + 64 + 1024;   // + alignment slack

constexpr uint32_t kQBytes = 4 * kQLatChunk + kQRopeBytes;       // 73728 per CTA

struct TcParams {
    const int32_t* block_table;
    const int32_t* seq_lens;
    __nv_bfloat16* out;
    float* lse;
    float* o_part;
    float* lse_part;
    DevCtl* ctl;
    int64_t num_pages;
    int max_pages;
    int max_seq_len;
    int B;
    int chunk;
    int splits;
    float scale_log2;     // scale * log2(e)
};

struct Bars {
    uint32_t kv_full[kNS], kv_empty[kNS], q_full, mma_drain;
    uint32_t s_full[2], s_empty[2], p_full[2], p_empty[2], x_full[2], x_free[2];
};

__device__ __forceinline__ Bars make_bars(uint32_t base) {
    Bars b;
    uint32_t a = base;
    for (int i = 0; i < kNS; ++i) b.kv_full[i] = a, a += 8;
    for (int i = 0; i < kNS; ++i) b.kv_empty[i] = a, a += 8;
    b.q_full = a, a += 8;
    b.mma_drain = a, a += 8;
    for (int i = 0; i < 2; ++i) b.s_full[i] = a, a += 8;
    for (int i = 0; i < 2; ++i) b.s_empty[i] = a, a += 8;
    for (int i = 0; i < 2; ++i) b.p_full[i] = a, a += 8;
    for (int i = 0; i < 2; ++i) b.p_empty[i] = a, a += 8;
    for (int i = 0; i < 2; ++i) b.x_full[i] = a, a += 8;
    for (int i = 0; i < 2; ++i) b.x_free[i] = a, a += 8;
    return b;
}

__device__ __forceinline__ void fail(DevCtl* ctl, volatile int* abort_flag, int where) {
    *abort_flag = 1;
    record_error(ctl, MLA_ERR_TIMEOUT, where);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_qlat,
                     const __grid_constant__ CUtensorMap tm_qrope,
                     const __grid_constant__ CUtensorMap tm_kv_lat,
                     const __grid_constant__ CUtensorMap tm_kv_rope, TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ uint32_t s_tmem_base;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t r = cluster_rank();
    const uint32_t peer = r ^ 1u;
    const int unit = blockIdx.x >> 1;
    const int b = unit / p.splits;
    const int split = unit % p.splits;
    const uint32_t wait_limit = p.ctl->wait_limit;

    const uint32_t sbase = smem_u32(sm);
    const Bars bars = make_bars(sbase + kOffBar);

    int n_b = p.seq_lens[b];
    if (n_b < 0 || n_b > p.max_seq_len) {
        if (tid == 0 && r == 0) record_error(p.ctl, MLA_ERR_BOUNDS, b);
        n_b = n_b < 0 ? 0 : p.max_seq_len;
    }
    const int e0 = split * p.chunk;
    const int e1 = min(n_b, e0 + p.chunk);
    const int n_tiles = e1 > e0 ? (e1 - e0 + kT - 1) / kT : 0;

    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < kNS; ++i) {
            mbar_init(bars.kv_full[i], 1);
            mbar_init(bars.kv_empty[i], 1);
        }
        mbar_init(bars.q_full, 1);
        mbar_init(bars.mma_drain, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bars.s_full[i], 1);
            mbar_init(bars.s_empty[i], 128);
            mbar_init(bars.p_full[i], 128);
            mbar_init(bars.p_empty[i], 1);
            mbar_init(bars.x_full[i], 1);
            mbar_init(bars.x_free[i], 4);   // one remote arrive per peer softmax warp
        }
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

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0 && n_tiles > 0) {
            tma_prefetch_desc(&tm_qlat);
            tma_prefetch_desc(&tm_qrope);
            tma_prefetch_desc(&tm_kv_lat);
            tma_prefetch_desc(&tm_kv_rope);
            const int qrow = b * kHeads;
            mbar_arrive_expect_tx(bars.q_full, kQBytes);
            for (int k = 0; k < 4; ++k)
                tma_load_2d(sbase + kOffQ + k * kQLatChunk, &tm_qlat, bars.q_full,
                            (int)r * kHalfLat + 64 * k, qrow);
            tma_load_2d(sbase + kOffQRope, &tm_qrope, bars.q_full, (int)r * kHalfRope, qrow);
            int issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                if (s_abort) break;
                const int s = j % kNS;
                if (!mbar_wait(bars.kv_empty[s], ((j / kNS) & 1) ^ 1, wait_limit)) {
                    fail(p.ctl, &s_abort, 1);
                    break;
                }
                const int pos0 = e0 + j * kT;
                const int page = p.block_table[(size_t)b * p.max_pages + pos0 / kPage];
                int row = -2 * kPage;   // outside the pool: the tile reads as zeros
                if (page >= 0 && page < p.num_pages) row = page * kPage + pos0 % kPage;
                else if (r == 0) record_error(p.ctl, MLA_ERR_BOUNDS, page);
                const uint32_t st = sbase + kOffKv + s * kStageBytes;
                mbar_arrive_expect_tx(bars.kv_full[s], kStageBytes);
                for (int k = 0; k < 4; ++k)
                    tma_load_2d(st + k * kKvLatChunk, &tm_kv_lat, bars.kv_full[s],
                                (int)r * kHalfLat + 64 * k, row);
                tma_load_2d(st + 4 * kKvLatChunk, &tm_kv_rope, bars.kv_full[s],
                            kDc + (int)r * kHalfRope, row);
                issued = j + 1;
            }
            // drain: the last (up to kNS) loads must land before this CTA may exit
            for (int j = max(0, issued - kNS); j < issued; ++j)
                mbar_wait(bars.kv_full[j % kNS], (j / kNS) & 1, kDrainLimit);
            if (!mbar_wait(bars.q_full, 0, kDrainLimit)) record_error(p.ctl, MLA_ERR_TIMEOUT, 9);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, kT, 0, 0);
            constexpr uint32_t id_pv = idesc_bf16(128, kHalfLat, 0, 1);
            const uint32_t q_lat = sbase + kOffQ, q_rope = sbase + kOffQRope;
            bool ok = mbar_wait(bars.q_full, 0, wait_limit);
            if (!ok) fail(p.ctl, &s_abort, 2);
            auto issue_pv = [&](int i) -> bool {
                const int pb = i & 1;
                if (!mbar_wait(bars.p_full[pb], (i >> 1) & 1, wait_limit)) {
                    fail(p.ctl, &s_abort, 3);
                    return false;
                }
                tc_fence_after();
                const uint32_t pa = sbase + kOffP + pb * kPBytes;
                const uint32_t v = sbase + kOffKv + (i % kNS) * kStageBytes;
#pragma unroll
                for (int kk = 0; kk < kT / 16; ++kk)
                    mma_bf16_ss(tmem + kTmemO, smem_desc(pa + kk * 32, 16, 512, kSw64),
                                smem_desc(v + kk * 16 * 128, kKvLatChunk, 1024, kSw128), id_pv,
                                (i > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bars.p_empty[pb]);
                mma_commit(bars.kv_empty[i % kNS]);
                return true;
            };
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (s_abort) break;
                const int s = j % kNS, sb = j & 1;
                if (!mbar_wait(bars.kv_full[s], (j / kNS) & 1, wait_limit)) {
                    fail(p.ctl, &s_abort, 4);
                    break;
                }
                if (j >= 2 && !mbar_wait(bars.s_empty[sb], ((j >> 1) & 1) ^ 1, wait_limit)) {
                    fail(p.ctl, &s_abort, 5);
                    break;
                }
                tc_fence_after();
                const uint32_t st = sbase + kOffKv + s * kStageBytes;
                const uint32_t d = tmem + kTmemS + sb * kT;
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ss(d, smem_desc(q_lat + k * kQLatChunk + kk * 32, 16, 1024, kSw128),
                                    smem_desc(st + k * kKvLatChunk + kk * 32, 16, 1024, kSw128),
                                    id_qk, (k | kk) != 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    mma_bf16_ss(d, smem_desc(q_rope + kk * 32, 16, 512, kSw64),
                                smem_desc(st + 4 * kKvLatChunk + kk * 32, 16, 512, kSw64), id_qk, 1u);
                mma_commit(bars.s_full[sb]);
                if (j >= 1 && !issue_pv(j - 1)) break;
                if (j == n_tiles - 1) issue_pv(j);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ softmax warps
        const int lg = warp & 3;                 // TMEM lane group this warp may access
        const int h = lg * 32 + lane;            // head = TMEM lane
        const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
        const uint32_t x_local = sbase + kOffX;
        const uint32_t x_remote = mapa(x_local, peer);
        const uint32_t xfull_remote[2] = {mapa(bars.x_full[0], peer), mapa(bars.x_full[1], peer)};
        const uint32_t xfree_remote[2] = {mapa(bars.x_free[0], peer), mapa(bars.x_free[1], peer)};
        const bool leader = (tid == 64);
        float m_used = -INFINITY, l_run = 0.f;
        float s_own[kT], s_next[kT];

        // read S_j of this CTA from TMEM and send it to the peer
        auto load_and_send = [&](int j, float (&dst)[kT]) -> bool {
            const int sb = j & 1;
            if (!mbar_wait(bars.s_full[sb], (j >> 1) & 1, wait_limit)) {
                fail(p.ctl, &s_abort, 6);
                return false;
            }
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + kTmemS + sb * kT, v);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bars.s_empty[sb]);
#pragma unroll
            for (int t = 0; t < kT; ++t) dst[t] = __uint_as_float(v[t]);
            if (!mbar_wait(bars.x_free[sb], ((j >> 1) & 1) ^ 1, wait_limit)) {
                fail(p.ctl, &s_abort, 7);
                return false;
            }
#pragma unroll
            for (int g = 0; g < kT / 4; ++g)
                st_async_v4(x_remote + sb * kXBytes + (g * 128 + h) * 16, xfull_remote[sb],
                            v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
            return true;
        };

        bool ok = true;
        if (n_tiles > 0) ok = load_and_send(0, s_own);
        for (int j = 0; ok && j < n_tiles; ++j) {
            if (s_abort) break;
            const int sb = j & 1;
            if (j + 1 < n_tiles && !load_and_send(j + 1, s_next)) break;
            // peer's partial scores of tile j
            if (leader) mbar_arrive_expect_tx(bars.x_full[sb], kXBytes);
            if (!mbar_wait(bars.x_full[sb], (j >> 1) & 1, wait_limit)) {
                fail(p.ctl, &s_abort, 8);
                break;
            }
            float x[kT];
            const uint8_t* xp = sm + kOffX + sb * kXBytes;
#pragma unroll
            for (int g = 0; g < kT / 4; ++g) {
                const float4 q = *reinterpret_cast<const float4*>(xp + (g * 128 + h) * 16);
                x[4 * g] = s_own[4 * g] + q.x;
                x[4 * g + 1] = s_own[4 * g + 1] + q.y;
                x[4 * g + 2] = s_own[4 * g + 2] + q.z;
                x[4 * g + 3] = s_own[4 * g + 3] + q.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(xfree_remote[sb]);

            // visibility of the tile's positions
            const int pos0 = e0 + j * kT;
            const int page = p.block_table[(size_t)b * p.max_pages + pos0 / kPage];
            const bool page_ok = page >= 0 && page < p.num_pages;
            const int nvalid = page_ok ? min(kT, e1 - pos0) : 0;
            float mt = -INFINITY;
#pragma unroll
            for (int t = 0; t < kT; ++t) {
                x[t] = t < nvalid ? x[t] * p.scale_log2 : -INFINITY;
                mt = fmaxf(mt, x[t]);
            }
            // lazy running max: rescale O only when the row max grows by more than 2^8
            const bool need = mt > m_used + 8.0f;
            const float m_new = need ? mt : m_used;
            if (__any_sync(0xffffffffu, need) && j > 0) {
                if (!mbar_wait(bars.p_empty[(j - 1) & 1], ((j - 1) >> 1) & 1, wait_limit)) {
                    fail(p.ctl, &s_abort, 10);
                    break;
                }
                tc_fence_after();
                const float alpha = need ? exp2f(m_used - m_new) : 1.0f;
#pragma unroll 1
                for (int c = 0; c < kHalfLat / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_off + kTmemO + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tmem + lane_off + kTmemO + 32 * c, o);
                }
                tmem_wait_st();
                l_run *= alpha;
            } else if (need) {
                l_run = 0.f;    // first tile: nothing accumulated yet
            }
            m_used = m_new;
            float psum = 0.f;
            uint32_t pk[kT / 2];
#pragma unroll
            for (int t = 0; t < kT; t += 2) {
                const float p0 = m_used == -INFINITY ? 0.f : exp2f(x[t] - m_used);
                const float p1 = m_used == -INFINITY ? 0.f : exp2f(x[t + 1] - m_used);
                psum += p0 + p1;
                pk[t / 2] = pack_bf16x2(p0, p1);
            }
            l_run += psum;
            // positions past the end of the unit in a live page: zero their V rows so that
            // 0 * (stale bytes) cannot poison O
            if (page_ok && nvalid < kT) {
                uint8_t* st = sm + kOffKv + (j % kNS) * kStageBytes;
                const int nrows = kT - nvalid;
                for (int i = tid - 64; i < nrows * 4 * 8; i += 128) {
                    const int row = nvalid + i / 32, k = (i / 8) % 4, part = i % 8;
                    *reinterpret_cast<uint4*>(st + k * kKvLatChunk + row * 128 + part * 16) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            // P row h (64 bytes) into the SW64 K-major buffer once PV_{j-2} has released it
            if (j >= 2 && !mbar_wait(bars.p_empty[sb], ((j - 2) >> 1) & 1, wait_limit)) {
                fail(p.ctl, &s_abort, 11);
                break;
            }
            uint8_t* pbuf = sm + kOffP + sb * kPBytes;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int pc = c ^ ((h >> 1) & 3);
                *reinterpret_cast<uint4*>(pbuf + h * 64 + pc * 16) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bars.p_full[sb]);
#pragma unroll
            for (int t = 0; t < kT; ++t) s_own[t] = s_next[t];
        }

        // ---------------------------------------------------------------- epilogue
        if (n_tiles > 0 && !s_abort) {
            const int jl = n_tiles - 1;
            if (!mbar_wait(bars.p_empty[jl & 1], (jl >> 1) & 1, wait_limit)) fail(p.ctl, &s_abort, 12);
            tc_fence_after();
        }
        const float inv = l_run > 0.f ? 1.0f / l_run : 0.0f;
        const float L = l_run > 0.f ? (m_used + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
        const size_t row = (size_t)b * kHeads + h;
        const size_t BH = (size_t)p.B * kHeads;
#pragma unroll 1
        for (int c = 0; c < kHalfLat / 32; ++c) {
            uint32_t o[32];
            if (n_tiles > 0 && !s_abort) {
                tmem_ld32(tmem + lane_off + kTmemO + 32 * c, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = 0u;
            }
            const int col = (int)r * kHalfLat + 32 * c;
            if (p.splits == 1) {
                uint4* dst = reinterpret_cast<uint4*>(p.out + row * kDc + col);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * i]) * inv, __uint_as_float(o[8 * i + 1]) * inv),
                                        pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv),
                                        pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv),
                                        pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv));
            } else {
                float4* dst = reinterpret_cast<float4*>(p.o_part + ((size_t)split * BH + row) * kDc + col);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                         __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
            }
        }
        if (r == 0) {
            if (p.splits == 1) p.lse[row] = L;
            else p.lse_part[(size_t)split * BH + row] = L;
        }
    }

    // ---------------------------------------------------------------------- teardown
    if (warp == 1 && lane == 0 && n_tiles > 0) {
        // all MMAs issued by this thread are complete once this barrier flips
        mma_commit(bars.mma_drain);
        if (!mbar_wait(bars.mma_drain, 0, kDrainLimit)) record_error(p.ctl, MLA_ERR_TIMEOUT, 13);
    }
    __syncwarp();
    if (s_abort) __nanosleep(100000);   // let any in-flight distributed-shared-memory stores land
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();   // the peer no longer writes into this CTA's shared memory
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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
               uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Split plan of the tensor-core path: a work unit is (request, chunk of positions) and runs on
// one 2-CTA cluster; units per request are chosen so that the grid fills the SM pairs.
DecodePlan plan_decode_tc(int fmt, int B, int max_seq_len, int topk, int sms) {
    (void)fmt;
    DecodePlan p;
    const int L = topk > 0 ? topk : max_seq_len;
    const int pairs = sms / 2 > 0 ? sms / 2 : 1;
    int S = (pairs + B - 1) / B;
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
    CUtensorMap tm_qlat, tm_qrope, tm_kv_lat, tm_kv_rope;
    const uint64_t qrows = (uint64_t)a.B * kHeads;
    const uint64_t kv_rows = (uint64_t)a.num_pages * kPage;
    if (!encode_2d(&tm_qlat, a.q_lat, kDc, qrows, kDc * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tm_qrope, a.q_rope, kDr, qrows, kDr * 2, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_2d(&tm_kv_lat, a.pool, kDk, kv_rows, kBf16RecordBytes, 64, kT,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tm_kv_rope, a.pool, kDk, kv_rows, kBf16RecordBytes, 32, kT,
                   CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    TcParams p;
    p.block_table = a.block_table;
    p.seq_lens = a.seq_lens;
    p.out = a.out;
    p.lse = a.lse;
    p.o_part = a.o_part;
    p.lse_part = a.lse_part;
    p.ctl = a.ctl;
    p.num_pages = a.num_pages;
    p.max_pages = a.max_pages;
    p.max_seq_len = a.max_seq_len;
    p.B = a.B;
    p.chunk = plan.chunk;
    p.splits = plan.splits;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    const int64_t ctas = 2LL * a.B * plan.splits;
    if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
    decode_tc_kernel<<<(unsigned)ctas, kThreads, kSmemBytes, st>>>(tm_qlat, tm_qrope, tm_kv_lat,
                                                                    tm_kv_rope, p);
    e = cudaGetLastError();
    if (e != cudaSuccess || plan.splits == 1) return e;
    return launch_combine(a.o_part, a.lse_part, plan.splits, a.B, kHeads, a.out, a.lse, st);
}

}  // namespace mla
