// proj.cu -- the value up-projection and output projection of the decode output on the tensor
// cores ("DeepSeek's KV Cache: From 3.9 MB to 890 B per Token", section "Computing without
// expanding Key and Value", Fig. 6 (2) and (3)).
//
// Fig. 6 (2): the decode gives per head the weighted latent sum U_h (512); the layer output is
// Y = sum_h (U_h W^UV_h) W^O_h.  Two products:
//   stage 1  Z_h = U_h W^UV_h        per head: [B x 512] x [512 x 128]       (128 heads)
//   stage 2  Y   = Z W^O             [B x H*128] x [H*128 x D]              (Z = heads side by side)
// Fig. 6 (3): with the pre-merged weight What^O_h = W^UV_h W^O_h, Y = U What^O: one product
// [B x H*512] x [H*512 x D].
//
// Decode batches are small, so every product is "weight times a few activation rows": the
// weight is the MMA's M side (128 output rows per tile, read from HBM once), the batch is its N
// side (up to 128 requests per tile), and the reduction dimension K is long.  One kernel does
// all three products:
//   * a cluster of S CTAs owns one 128-row tile of outputs; CTA r of the cluster takes the r-th
//     share of the K range, so that about one CTA per SM streams weight rows;
//   * warp 0 streams [128 x 64] weight boxes and [N x 64] activation boxes by TMA (128-byte
//     swizzle) into a ring of stages; warp 1 issues tcgen05.mma kind::f16 (bf16 in, fp32
//     accumulators in tensor memory: lane = output row, column = request); warps 2-5 finish;
//   * the S partial accumulators are summed in rank 0 through distributed shared memory, 16
//     columns a round, in a fixed order (deterministic);
//   * stage 1 writes Z as two bf16 planes, hi = bf16(Z) and lo = bf16(Z - hi), so that Z reaches
//     stage 2 with about 16 significant bits instead of 8: stage 2 multiplies both planes (its N
//     side holds the hi and the lo rows of each request) and adds the two columns of a request
//     in fp32.  The weights and U are bf16 values already; only Z is an intermediate.
// Every wait is bounded: on expiry the kernel records MLA_ERR_TIMEOUT, stops issuing, drains its
// copies and MMAs, keeps the cluster barriers, frees tensor memory and returns.
#include <cuda.h>
#include <cstring>

#include "decode_common.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kBM = 128;              // output rows (weight rows) per tile
constexpr int kBK = 64;               // K per stage: one 128-byte swizzle row of bf16
constexpr int kMaxNB = 128;           // requests per tile
constexpr int kPThreads = 192;        // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kMaxStages = 8;
constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KB
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kDrainLimit = 1u << 20;
constexpr int kRingBudget = 104 * 1024;   // two CTAs fit on an SM (tensor memory: 2 x 256 columns)
constexpr int kPrefetchChunks = 12;   // stage-2 weight chunks (16 KB each) per CTA prefetched by stage 1

enum Epi : int { kEpiZ = 0, kEpiYPair = 1, kEpiY = 2 };

struct ProjParams {
    int k_chunks;        // K / 64
    int nb;              // requests per tile (rows of each activation box)
    int n_mma;           // MMA N: nb (kEpiZ, kEpiY) or 2 nb (kEpiYPair)
    int stages;
    uint32_t stage_bytes;
    int B;
    int a_rows_per_z;    // weight-row offset per blockIdx.z (stage 1: one head's 128 rows)
    int b_cols_per_z;    // activation-column offset per blockIdx.z (stage 1: one head's 512)
    int out_cols_per_z;  // output-column offset per blockIdx.z (stage 1: one head's 128)
    int64_t out_ld;      // output row stride (elements)
    int64_t out_plane;   // kEpiZ: elements from the hi plane to the lo plane
    __nv_bfloat16* out;
    DevCtl* ctl;
    // kEpiZ: the next product's weight boxes to prefetch into L2 while this one runs (one CTA per
    // CTA of the next launch: its output tile and the first chunks of its K share)
    int pf_tiles;        // output tiles of the next product (0: no prefetch)
    int pf_split;        // its cluster size
    int pf_k_chunks;     // its K / 64
    int pf_chunks;       // chunks to prefetch per CTA
    bool wait_prior;     // this launch depends on the previous one (programmatic): wait before
                         // reading the activations
};

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int kEpi>
__global__ void __launch_bounds__(kPThreads, 2)
    proj_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_next, ProjParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t s_bar[2 * kMaxStages + 2];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t S = cluster_size();
    const uint32_t r = cluster_rank();
    const int mt = blockIdx.x / S;
    const int z = blockIdx.z;
    const int b0 = blockIdx.y * kMaxNB;
    const int per = p.k_chunks / (int)S, extra = p.k_chunks % (int)S;
    const int c0 = (int)r * per + ((int)r < extra ? (int)r : extra);
    const int nck = per + ((int)r < extra ? 1 : 0);
    const int a_row = mt * kBM + z * p.a_rows_per_z;
    const int b_col0 = z * p.b_cols_per_z;
    const uint32_t wait_limit = p.ctl->wait_limit;

    const uint32_t sbase = smem_u32(sm);
    auto full = [&](int s) { return smem_u32(&s_bar[s]); };
    auto empty = [&](int s) { return smem_u32(&s_bar[kMaxStages + s]); };
    const uint32_t acc_full = smem_u32(&s_bar[2 * kMaxStages]);
    const uint32_t mma_drain = smem_u32(&s_bar[2 * kMaxStages + 1]);
    auto a_dst = [&](int s) { return sbase + (uint32_t)s * p.stage_bytes; };
    auto b_dst = [&](int s) { return sbase + (uint32_t)s * p.stage_bytes + kABytes; };

    if (tid == 0) {
        s_abort = 0;
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(mma_drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        int issued = 0;
        if (lane == 0) {
            tma_prefetch_desc(&tm_a);
            tma_prefetch_desc(&tm_b);
            // the weights of the first ring's worth of chunks go out at once; when this launch
            // depends on the one before (its activations are that launch's output), the
            // activations wait for it, the weights do not
            const int first = nck < p.stages ? nck : p.stages;
            for (int i = 0; i < first; ++i) {
                mbar_arrive_expect_tx(full(i), p.stage_bytes);
                tma_load_2d(a_dst(i), &tm_a, full(i), (c0 + i) * kBK, a_row);
            }
            if (p.wait_prior) grid_dependency_wait();
            for (int i = 0; i < nck; ++i) {
                const int s = i % p.stages;
                if (i >= p.stages && !mbar_wait(empty(s), ((i / p.stages) - 1) & 1, wait_limit)) {
                    s_abort = 1;
                    record_error(p.ctl, MLA_ERR_TIMEOUT, 60);
                }
                if (s_abort) {
                    // the weight boxes already issued still land on their barriers: count them in
                    issued = i > first ? i : first;
                    break;
                }
                const int kx = (c0 + i) * kBK;
                if (i >= first) {
                    mbar_arrive_expect_tx(full(s), p.stage_bytes);
                    tma_load_2d(a_dst(s), &tm_a, full(s), kx, a_row);
                }
                if (kEpi == kEpiYPair) {
                    tma_load_3d(b_dst(s), &tm_b, full(s), b_col0 + kx, b0, 0);
                    tma_load_3d(b_dst(s) + (uint32_t)p.nb * 128u, &tm_b, full(s), b_col0 + kx, b0, 1);
                } else {
                    tma_load_2d(b_dst(s), &tm_b, full(s), b_col0 + kx, b0);
                }
                ++issued;
            }
            // the next product's first weight chunks into L2 (its launch waits for this one)
            if (kEpi == kEpiZ && p.pf_tiles > 0) {
                const int cta = (int)(blockIdx.z * gridDim.y + blockIdx.y) * (int)gridDim.x + (int)blockIdx.x;
                const int n_next = p.pf_tiles * p.pf_split;
                const int per_cta_z = (n_next + (int)(gridDim.x * gridDim.y * gridDim.z) - 1) /
                                      (int)(gridDim.x * gridDim.y * gridDim.z);
                for (int q = cta * per_cta_z; q < (cta + 1) * per_cta_z && q < n_next; ++q) {
                    const int tile = q / p.pf_split, rr = q % p.pf_split;
                    const int per2 = p.pf_k_chunks / p.pf_split, ex2 = p.pf_k_chunks % p.pf_split;
                    const int k0 = rr * per2 + (rr < ex2 ? rr : ex2);
                    for (int c = 0; c < p.pf_chunks && c < per2; ++c)
                        tma_prefetch_l2_2d(&tm_next, (k0 + c) * kBK, tile * kBM);
                }
            }
            grid_launch_dependents();
            // drain: every issued copy lands before the ring is reused or the CTA exits
            for (int i = issued - 1; i >= 0 && i >= issued - p.stages; --i)
                mbar_wait(full(i % p.stages), (i / p.stages) & 1, kDrainLimit);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        const uint32_t idesc = idesc_bf16(kBM, (uint32_t)p.n_mma, 0, 0);
        const uint64_t d_hi = smem_desc(0, 16, 1024, kSw128) & 0xFFFFFFFF00000000ull;
        const uint32_t d_lo = (uint32_t)smem_desc(0, 16, 1024, kSw128);
        int done = 0;
        for (int i = 0; i < nck; ++i) {
            const int s = i % p.stages;
            bool ok = !s_abort && mbar_wait(full(s), (i / p.stages) & 1, wait_limit);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) {
                    s_abort = 1;
                    record_error(p.ctl, MLA_ERR_TIMEOUT, 61);
                }
                break;
            }
            tc_fence_after();
            const uint32_t a_lo = d_lo + ((a_dst(s) >> 4) & 0x3FFF);
            const uint32_t b_lo = d_lo + ((b_dst(s) >> 4) & 0x3FFF);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    mma_bf16_ss(tmem, d_hi | (a_lo + kk * 2), d_hi | (b_lo + kk * 2), idesc,
                                (i > 0 || kk > 0) ? 1u : 0u);
                mma_commit(empty(s));
                if (i == nck - 1) mma_commit(acc_full);
            }
            __syncwarp();
            ++done;
        }
        // all issued MMAs complete before tensor memory is read back or freed
        if (elect_one()) {
            mma_commit(mma_drain);
            if (!mbar_wait(mma_drain, 0, kDrainLimit)) record_error(p.ctl, MLA_ERR_TIMEOUT, 62);
        }
        __syncwarp();
        (void)done;
    }

    // ---------------------------------------------------------------------- epilogue
    // Warps 2-5: warp w reads tensor-memory lanes 32 (w % 4) .. + 31; thread = output row m.
    const bool epi = warp >= 2;
    const int lg = warp & 3;
    const int m = lg * 32 + lane;
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    bool have_acc = false;
    if (epi) {
        bool ok = !s_abort && nck > 0 && mbar_wait(acc_full, 0, wait_limit);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0 && nck > 0) {
            s_abort = 1;
            record_error(p.ctl, MLA_ERR_TIMEOUT, 63);
        }
        have_acc = ok;
        tc_fence_after();
    }

    // The cluster's partial sums, in one exchange: the accumulator's columns are cut into units of
    // 16 requests (for kEpiYPair a unit is its hi column block and its lo column block), CTA q of
    // the cluster owns units [u_of(q), u_of(q + 1)); every CTA writes its partials of the other
    // CTAs' units into their slot buffers through distributed shared memory (slot: the sender's
    // rank among the others), all threads of the cluster meet, and each CTA adds, in rank order,
    // the partials of its own units to its own and writes those outputs.  The first barrier: every
    // CTA's main loop is over (the ring, where the slots live, is no longer written by TMA).
    const int units = (kEpi == kEpiYPair ? p.nb : p.n_mma) / 16;
    auto u_of = [&](int q) { return q * units / (int)S; };
    const int blocks = kEpi == kEpiYPair ? 2 : 1;                  // column blocks per unit
    const int max_units = (units + (int)S - 1) / (int)S;
    const int slot_stride = blocks * 16 * max_units + 4;          // floats per slot row (+4: banks)
    const int slot_floats = kBM * slot_stride;
    auto col_of = [&](int u, int blk) { return blk == 0 ? 16 * u : p.nb + 16 * u; };
    if (S > 1) {
        tc_fence_before();
        __syncthreads();
        cluster_sync();
        if (epi && have_acc) {
            for (int q = 0; q < (int)S; ++q) {
                if (q == (int)r) continue;
                const int slot = (int)r < q ? (int)r : (int)r - 1;
                const uint32_t base = mapa(sbase, (uint32_t)q) +
                                      (uint32_t)((slot * slot_floats + m * slot_stride) * 4);
                for (int u = u_of(q); u < u_of(q + 1); ++u)
                    for (int blk = 0; blk < blocks; ++blk) {
                        uint32_t v[16];
                        tmem_ld16(tmem + lane_off + col_of(u, blk), v);
                        tmem_wait_ld();
                        const uint32_t dst = base + (uint32_t)(((blk * max_units + (u - u_of(q))) * 16) * 4);
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            st_cluster_v4(dst + 16 * t, __uint_as_float(v[4 * t]), __uint_as_float(v[4 * t + 1]),
                                          __uint_as_float(v[4 * t + 2]), __uint_as_float(v[4 * t + 3]));
                    }
            }
        }
        __syncwarp();
        cluster_sync();
    }

    if (epi && have_acc) {
        const int64_t col = (int64_t)z * p.out_cols_per_z + (int64_t)mt * kBM + m;
        __nv_bfloat16* out = p.out + (int64_t)b0 * p.out_ld + col;
        const int nvalid = min(p.nb, p.B - b0);
        for (int u = u_of((int)r); u < u_of((int)r + 1); ++u) {
            if (16 * u >= nvalid) break;
            float acc[2][16];
            for (int blk = 0; blk < blocks; ++blk) {
                uint32_t v[16];
                tmem_ld16(tmem + lane_off + col_of(u, blk), v);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 16; ++t) acc[blk][t] = __uint_as_float(v[t]);
                for (int q = 1; q < (int)S; ++q) {
                    const float4* src = reinterpret_cast<const float4*>(
                        sm + ((q - 1) * slot_floats + m * slot_stride + (blk * max_units + (u - u_of((int)r))) * 16) * 4);
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float4 x = src[t];
                        acc[blk][4 * t] += x.x;
                        acc[blk][4 * t + 1] += x.y;
                        acc[blk][4 * t + 2] += x.z;
                        acc[blk][4 * t + 3] += x.w;
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const int b = 16 * u + t;
                if (b >= nvalid) break;
                __nv_bfloat16* o = out + (int64_t)b * p.out_ld;
                if (kEpi == kEpiYPair) {
                    *o = __float2bfloat16_rn(acc[0][t] + acc[1][t]);
                } else if (kEpi == kEpiZ) {
                    const __nv_bfloat16 hi = __float2bfloat16_rn(acc[0][t]);
                    *o = hi;
                    o[p.out_plane] = __float2bfloat16_rn(acc[0][t] - __bfloat162float(hi));
                } else {
                    *o = __float2bfloat16_rn(acc[0][t]);
                }
            }
        }
    }

    // ---------------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (S > 1) cluster_sync();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Cluster size along K: about 1.35 CTAs per SM for the tiles given (two fit on an SM, and a sweep
// of the merged product at 40 tiles ran best with clusters of 5: 5.9 TB/s, against 4.5 TB/s with
// one CTA per SM and 3.9 TB/s at 7), at most 8, at most one share per K chunk.
int pick_split(int tiles, int k_chunks, int sms) {
    int s = tiles > 0 ? (27 * sms) / (20 * tiles) : 1;
    if (s < 1) s = 1;
    if (s > 8) s = 8;
    if (s > k_chunks) s = k_chunks;
    return s < 1 ? 1 : s;
}

// Shared memory of the reduction's slots for a cluster of S (they reuse the ring).
size_t slot_bytes(bool pair, int units, int S) {
    const int max_units = (units + S - 1) / S;
    return (size_t)(S - 1) * kBM * ((pair ? 2 : 1) * 16 * max_units + 4) * 4 + 1024;
}

// The cluster size of a launch: pick_split, lowered until the reduction's slots fit.
int split_of(int tiles, int k_chunks, bool pair, int units) {
    int sms = num_sms();
    if (sms <= 0) sms = 152;
    int S = pick_split(tiles, k_chunks, sms);
    while (S > 1 && slot_bytes(pair, units, S) > (size_t)kRingBudget + 1024) --S;
    return S;
}

template <int kEpi>
cudaError_t launch_proj(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_next, ProjParams p,
                        int m_tiles, int n_tiles, int zdim, bool programmatic, cudaStream_t st) {
    auto* kernel = proj_gemm_kernel<kEpi>;
    const int b_rows = kEpi == kEpiYPair ? 2 * p.nb : p.n_mma;
    p.stage_bytes = kABytes + (uint32_t)b_rows * 128u;
    p.stages = kRingBudget / (int)p.stage_bytes;
    if (p.stages > kMaxStages) p.stages = kMaxStages;
    if (p.stages < 2) return cudaErrorInvalidValue;
    const int units = (kEpi == kEpiYPair ? p.nb : p.n_mma) / 16;
    const int S = split_of(m_tiles * n_tiles * zdim, p.k_chunks, kEpi == kEpiYPair, units);
    size_t smem = (size_t)p.stages * p.stage_bytes + 1024;
    // the reduction's slots (they reuse the ring once the main loop is over)
    const size_t slot_need = slot_bytes(kEpi == kEpiYPair, units, S);
    if (slot_need > smem) smem = slot_need;
    if (smem > (size_t)kRingBudget + 2048) return cudaErrorInvalidValue;
    p.wait_prior = programmatic;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kRingBudget + 2048));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(m_tiles * S), (unsigned)n_tiles, (unsigned)zdim);
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // the launch may begin before the previous one on the stream ends; its producer waits for that
    // one (griddepcontrol.wait) before it reads the activations the previous launch wrote
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tm_a, tm_b, tm_next, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int round_up(int x, int a) { return (x + a - 1) / a * a; }

}  // namespace

// Fig. 6 (2): stage 1 (per head, Z into the hi/lo planes), then stage 2 (Y from both planes).
cudaError_t launch_value_project(const __nv_bfloat16* u, const __nv_bfloat16* w_uv_t, const __nv_bfloat16* w_o_t,
                                 int B, int H, int D, __nv_bfloat16* z, __nv_bfloat16* y, DevCtl* ctl,
                                 cudaStream_t st) {
    const int nt = (B + kMaxNB - 1) / kMaxNB;
    const int bt = B < kMaxNB ? B : kMaxNB;
    const uint64_t hk = (uint64_t)H * kDv;   // stage 2 K: the heads' outputs side by side
    CUtensorMap tm_w_o;                       // stage 2's weight: W^O^T [D x H*128]
    if (!encode_2d(&tm_w_o, w_o_t, hk, (uint64_t)D, hk * 2, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    {
        // stage 1: A = W^UV_h^T rows [h*128, h*128 + 128) of [H*128 x 512]; B = U [B x H*512]
        CUtensorMap tm_a, tm_b;
        const int nb = round_up(bt, 16);
        if (!encode_2d(&tm_a, w_uv_t, kDc, (uint64_t)H * kDv, kDc * 2, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&tm_b, u, (uint64_t)H * kDc, (uint64_t)B, (uint64_t)H * kDc * 2, kBK, (uint32_t)nb,
                       CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        ProjParams p = {};
        p.k_chunks = kDc / kBK;
        p.nb = nb;
        p.n_mma = nb;
        p.B = B;
        p.a_rows_per_z = kDv;
        p.b_cols_per_z = kDc;
        p.out_cols_per_z = kDv;
        p.out_ld = (int64_t)hk;
        p.out_plane = (int64_t)B * (int64_t)hk;
        p.out = z;
        p.ctl = ctl;
        // while it runs (it is latency-bound), the stage-2 CTAs' first weight chunks go into L2
        p.pf_tiles = (D / kBM) * nt;
        p.pf_split = split_of(p.pf_tiles, (int)(hk / kBK), true, round_up(bt, 16) / 16);
        p.pf_k_chunks = (int)(hk / kBK);
        p.pf_chunks = kPrefetchChunks;
        cudaError_t e = launch_proj<kEpiZ>(tm_a, tm_b, tm_w_o, p, 1, nt, H, false, st);
        if (e != cudaSuccess) return e;
    }
    {
        // stage 2: A = W^O^T [D x H*128]; B = the hi and lo planes of Z, [2][B][H*128] (each plane's
        // box a multiple of 16 rows, so that the lo columns start on a 16-column boundary); launched
        // so that it may start while stage 1 finishes
        CUtensorMap tm_b;
        const int nb = round_up(bt, 16);
        const uint64_t dims[3] = {hk, (uint64_t)B, 2};
        const uint64_t strides[2] = {hk * 2, (uint64_t)B * hk * 2};
        const uint32_t box[3] = {(uint32_t)kBK, (uint32_t)nb, 1};
        if (!encode_3d(&tm_b, z, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
            return cudaErrorInvalidValue;
        ProjParams p = {};
        p.k_chunks = (int)(hk / kBK);
        p.nb = nb;
        p.n_mma = 2 * nb;
        p.B = B;
        p.out_ld = D;
        p.out = y;
        p.ctl = ctl;
        return launch_proj<kEpiYPair>(tm_w_o, tm_b, tm_w_o, p, D / kBM, nt, 1, true, st);
    }
}

// Fig. 6 (3): Y = U What^O with What^O^T [D x H*512].
cudaError_t launch_value_project_merged(const __nv_bfloat16* u, const __nv_bfloat16* w_hat_t, int B, int H, int D,
                                        __nv_bfloat16* y, DevCtl* ctl, cudaStream_t st) {
    const int nt = (B + kMaxNB - 1) / kMaxNB;
    const int bt = B < kMaxNB ? B : kMaxNB;
    const uint64_t hk = (uint64_t)H * kDc;
    CUtensorMap tm_a, tm_b;
    const int nb = round_up(bt, 16);
    if (!encode_2d(&tm_a, w_hat_t, hk, (uint64_t)D, hk * 2, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tm_b, u, hk, (uint64_t)B, hk * 2, kBK, (uint32_t)nb, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    ProjParams p = {};
    p.k_chunks = (int)(hk / kBK);
    p.nb = nb;
    p.n_mma = nb;
    p.B = B;
    p.out_ld = D;
    p.out = y;
    p.ctl = ctl;
    return launch_proj<kEpiY>(tm_a, tm_b, tm_a, p, D / kBM, nt, 1, false, st);
}

}  // namespace mla
