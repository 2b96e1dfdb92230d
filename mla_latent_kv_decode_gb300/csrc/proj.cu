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
constexpr int kSlotStride = 20;       // floats per row of a reduction slot (16 + 4: no bank conflicts)
constexpr int kSlotBytes = kBM * kSlotStride * 4;
constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KB
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kDrainLimit = 1u << 20;
constexpr int kRingBudget = 200 * 1024;

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

template <int kEpi>
__global__ void __launch_bounds__(kPThreads, 1)
    proj_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     ProjParams p) {
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
            for (int i = 0; i < nck; ++i) {
                const int s = i % p.stages;
                if (i >= p.stages && !mbar_wait(empty(s), ((i / p.stages) - 1) & 1, wait_limit)) {
                    s_abort = 1;
                    record_error(p.ctl, MLA_ERR_TIMEOUT, 60);
                }
                if (s_abort) break;
                const int kx = (c0 + i) * kBK;
                mbar_arrive_expect_tx(full(s), p.stage_bytes);
                tma_load_2d(a_dst(s), &tm_a, full(s), kx, a_row);
                if (kEpi == kEpiYPair) {
                    tma_load_3d(b_dst(s), &tm_b, full(s), b_col0 + kx, b0, 0);
                    tma_load_3d(b_dst(s) + (uint32_t)p.nb * 128u, &tm_b, full(s), b_col0 + kx, b0, 1);
                } else {
                    tma_load_2d(b_dst(s), &tm_b, full(s), b_col0 + kx, b0);
                }
                ++issued;
            }
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

    // Partial sums of the cluster into rank 0, 16 columns a round through two slot buffers:
    // ranks 1 .. S-1 write their columns into their own slot of rank 0's buffer (j & 1), then
    // every thread of the cluster meets; rank 0 adds the slots, in rank order, to its own
    // columns in tensor memory.  The barrier of round j + 1 follows rank 0's reads of round j,
    // so round j + 2 may overwrite that buffer.  The first barrier: every CTA's main loop is
    // over (rank 0's ring is no longer written by TMA).
    if (S > 1) {
        const int rounds = (p.n_mma + 15) / 16;
        const uint32_t slots = sbase;   // the ring, free once the main loop is over
        const uint32_t slots_remote = mapa(slots, 0);
        tc_fence_before();
        __syncthreads();
        cluster_sync();
        for (int j = 0; j <= rounds; ++j) {
            if (epi && have_acc && j < rounds && r != 0) {
                uint32_t v[16];
                tmem_ld16(tmem + lane_off + 16 * j, v);
                tmem_wait_ld();
                const uint32_t dst = slots_remote + (uint32_t)(((j & 1) * (int)(S - 1) + (int)r - 1) * kSlotBytes) +
                                     (uint32_t)(m * kSlotStride * 4);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st_cluster_v4(dst + 16 * q, __uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                  __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
            if (epi && have_acc && j >= 1 && r == 0) {
                const int jj = j - 1;
                uint32_t v[16];
                tmem_ld16(tmem + lane_off + 16 * jj, v);
                tmem_wait_ld();
                float acc[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) acc[t] = __uint_as_float(v[t]);
                for (int q = 1; q < (int)S; ++q) {
                    const float4* src = reinterpret_cast<const float4*>(
                        sm + ((jj & 1) * (int)(S - 1) + q - 1) * kSlotBytes + m * kSlotStride * 4);
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float4 x = src[t];
                        acc[4 * t] += x.x;
                        acc[4 * t + 1] += x.y;
                        acc[4 * t + 2] += x.z;
                        acc[4 * t + 3] += x.w;
                    }
                }
#pragma unroll
                for (int t = 0; t < 16; ++t) v[t] = __float_as_uint(acc[t]);
                tmem_st16(tmem + lane_off + 16 * jj, v);
                tmem_wait_st();
            }
            __syncwarp();
            cluster_sync();
        }
    }

    if (epi && have_acc && r == 0) {
        const int nvalid = min(p.nb, p.B - b0);
        const int64_t col = (int64_t)z * p.out_cols_per_z + (int64_t)mt * kBM + m;
        __nv_bfloat16* out = p.out + (int64_t)b0 * p.out_ld + col;
        for (int c = 0; c < nvalid; c += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + lane_off + c, v);
            tmem_wait_ld();
            if (kEpi == kEpiYPair) {
                uint32_t w[16];
                tmem_ld16(tmem + lane_off + p.nb + c, w);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    if (c + t < nvalid)
                        out[(int64_t)(c + t) * p.out_ld] =
                            __float2bfloat16_rn(__uint_as_float(v[t]) + __uint_as_float(w[t]));
            } else if (kEpi == kEpiZ) {
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    if (c + t < nvalid) {
                        const float x = __uint_as_float(v[t]);
                        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
                        out[(int64_t)(c + t) * p.out_ld] = hi;
                        out[p.out_plane + (int64_t)(c + t) * p.out_ld] = lo;
                    }
            } else {
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    if (c + t < nvalid) out[(int64_t)(c + t) * p.out_ld] = __float2bfloat16_rn(__uint_as_float(v[t]));
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

// Cluster size along K: about one CTA per SM for the tiles given, at most 8, at most one share
// per K chunk.
int pick_split(int tiles, int k_chunks, int sms) {
    int s = tiles > 0 ? sms / tiles : 1;
    if (s < 1) s = 1;
    if (s > 8) s = 8;
    if (s > k_chunks) s = k_chunks;
    return s < 1 ? 1 : s;
}

template <int kEpi>
cudaError_t launch_proj(const CUtensorMap& tm_a, const CUtensorMap& tm_b, ProjParams p, int m_tiles, int n_tiles,
                        int zdim, cudaStream_t st) {
    auto* kernel = proj_gemm_kernel<kEpi>;
    const int b_rows = kEpi == kEpiYPair ? 2 * p.nb : p.n_mma;
    p.stage_bytes = kABytes + (uint32_t)b_rows * 128u;
    p.stages = kRingBudget / (int)p.stage_bytes;
    if (p.stages > kMaxStages) p.stages = kMaxStages;
    if (p.stages < 2) return cudaErrorInvalidValue;
    int sms = num_sms();
    if (sms <= 0) sms = 152;
    const int S = pick_split(m_tiles * n_tiles * zdim, p.k_chunks, sms);
    size_t smem = (size_t)p.stages * p.stage_bytes + 1024;
    const size_t slot_need = (size_t)2 * (S - 1) * kSlotBytes + 1024;
    if (slot_need > smem) smem = slot_need;
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
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tm_a, tm_b, p);
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
        cudaError_t e = launch_proj<kEpiZ>(tm_a, tm_b, p, 1, nt, H, st);
        if (e != cudaSuccess) return e;
    }
    {
        // stage 2: A = W^O^T [D x H*128]; B = the hi and lo planes of Z, [2][B][H*128] (each plane's
        // box a multiple of 16 rows, so that the lo columns start on a 16-column boundary)
        CUtensorMap tm_a, tm_b;
        const int nb = round_up(bt, 16);
        const uint64_t dims[3] = {hk, (uint64_t)B, 2};
        const uint64_t strides[2] = {hk * 2, (uint64_t)B * hk * 2};
        const uint32_t box[3] = {(uint32_t)kBK, (uint32_t)nb, 1};
        if (!encode_2d(&tm_a, w_o_t, hk, (uint64_t)D, hk * 2, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_3d(&tm_b, z, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
            return cudaErrorInvalidValue;
        ProjParams p = {};
        p.k_chunks = (int)(hk / kBK);
        p.nb = nb;
        p.n_mma = 2 * nb;
        p.B = B;
        p.out_ld = D;
        p.out = y;
        p.ctl = ctl;
        return launch_proj<kEpiYPair>(tm_a, tm_b, p, D / kBM, nt, 1, st);
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
    return launch_proj<kEpiY>(tm_a, tm_b, p, D / kBM, nt, 1, st);
}

}  // namespace mla
