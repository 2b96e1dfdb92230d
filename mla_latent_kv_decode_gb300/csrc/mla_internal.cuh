// mla_internal.cuh -- definitions shared by the libmla translation units (not installed).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/mla.h"

namespace mla {

constexpr int kDc = MLA_D_C;                 // latent width
constexpr int kDr = MLA_D_R;                 // rope width
constexpr int kDk = kDc + kDr;               // 576 = score contraction length
constexpr int kDv = MLA_D_V;                 // value width of one head (value up-projection)
constexpr int kHeads = MLA_HEADS;
constexpr int kPage = MLA_PAGE_TOKENS;
constexpr int kBf16RecordBytes = kDk * 2;    // 1152
constexpr int kFp8RecordBytes = kDc + 16 + kDr * 2;   // 656
constexpr int kFp8Group = 128;
constexpr int kFp8ScaleOff = kDc;            // 4 fp32 scales after the 512 codes
constexpr int kFp8RopeOff = kDc + 16;        // 64 bf16 rope after the scales
// Shared K = V entries (512 dims, the last 64 carry RoPE)
constexpr int kE = 512;
constexpr int kENope = 448;                  // V4: E4M3 dims, one UE8M0 scale per 64
constexpr int kV4EntryBytes = 584;
constexpr int kV4PageBytes = kPage * kV4EntryBytes;          // 37,376: codes, RoPE, scales by field
constexpr int kV4RopeOff = kPage * kENope;                   // 28,672: RoPE [64][128 B]
constexpr int kV4ScaleOff = kPage * (kENope + 128);          // 36,864: scale bytes [64][8]
constexpr int kV41EntryBytes = 288;          // V4.1: 256 B of E2M1 pairs, 32 E4M3 scales
constexpr int kV41ScaleOff = 256;

// Per-device control block living in device global memory (one per device; its address is
// taken with cudaGetSymbolAddress and passed to every kernel).
struct DevCtl {
    int32_t status;        // first error recorded (mla_status), 0 = none
    int32_t detail;        // kernel-specific detail of that error (e.g. offending page)
    uint32_t wait_limit;   // iteration cap of bounded waits
    uint32_t pad;
};

constexpr uint32_t kDefaultWaitLimit = 1u << 20;   // far above any real wait; bounds a lost signal

__device__ __forceinline__ void record_error(DevCtl* ctl, int code, int detail) {
    if (atomicCAS(&ctl->status, 0, code) == 0) ctl->detail = detail;
}

// Host helpers implemented in mla_api.cu.
DevCtl* device_ctl();          // control block of the current device (nullptr on failure)
int num_sms();                 // SM count of the current device
int device_cc();               // compute capability major*10+minor of the current device

// Launchers (one per translation unit).
cudaError_t launch_cache_append(int fmt, uint8_t* pool, int64_t num_pages,
                                const __nv_bfloat16* c_kv, const __nv_bfloat16* k_rope,
                                const int32_t* slot, int64_t T, DevCtl* ctl, cudaStream_t st);
cudaError_t launch_e4m3_encode(const float* x, uint8_t* codes, int64_t n, cudaStream_t st);
cudaError_t launch_shared_append(int fmt, uint8_t* pool, int64_t num_pages, const __nv_bfloat16* entry,
                                 const int32_t* slot, int64_t T, DevCtl* ctl, cudaStream_t st);
cudaError_t launch_combine(const float* o_part, const float* lse_part, int S, int B, int H,
                           __nv_bfloat16* out, float* lse, cudaStream_t st);

// DSA lightning indexer (indexer.cu).
cudaError_t launch_index_append(uint8_t* pool, int64_t num_pages, const __nv_bfloat16* k, const int32_t* slot,
                                int64_t T, DevCtl* ctl, cudaStream_t st);
cudaError_t launch_indexer_score(const uint8_t* pool, int64_t num_pages, const __nv_bfloat16* q, const float* w,
                                 const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                                 int max_seq_len, float* scores, DevCtl* ctl, cudaStream_t st);
cudaError_t launch_topk_select(const float* scores, int64_t ld, const int32_t* seq_lens, int B, int K,
                               int32_t* idx, cudaStream_t st);

// Value up-projection and output projection (proj.cu).
cudaError_t launch_value_project(const __nv_bfloat16* u, const __nv_bfloat16* w_uv_t, const __nv_bfloat16* w_o_t,
                                 int B, int H, int D, __nv_bfloat16* z, __nv_bfloat16* y, DevCtl* ctl,
                                 cudaStream_t st);
cudaError_t launch_value_project_merged(const __nv_bfloat16* u, const __nv_bfloat16* w_hat_t, int B, int H, int D,
                                        __nv_bfloat16* y, DevCtl* ctl, cudaStream_t st);

// Split-KV plan of one decode call.
struct DecodePlan {
    int splits;            // C: clusters of the launch (two partial slots each)
    size_t workspace;      // bytes of the partial slots and the per-request merge table
    int launches;          // kernels one decode call launches
};

struct DecodeArgs {
    int fmt;
    const uint8_t* pool;
    int64_t num_pages;
    const __nv_bfloat16* q_lat;
    const __nv_bfloat16* q_rope;
    const int32_t* block_table;
    int max_pages;
    const int32_t* seq_lens;
    int max_seq_len;
    const int32_t* topk_idx;
    int topk;
    int B;
    float scale;
    __nv_bfloat16* out;
    float* lse;
    void* workspace;       // caller scratch of at least plan.workspace bytes
    DevCtl* ctl;
    const float* sink = nullptr;      // shared K = V entries: per-head sink z' [128] (or null)
    const float* rope_cs = nullptr;   // shared K = V entries: [B][64] cos, sin of the query angles (or null)
};

// Tensor-core paths: bf16 dense pages (decode_tc.cu), FP8 records and top-k lists (decode_gather.cu).
DecodePlan plan_decode_tc(int fmt, int B, int max_seq_len, int topk, int sms);
cudaError_t launch_decode_tc(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st);

DecodePlan plan_decode_gather(int fmt, int B, int max_seq_len, int topk, int sms);
cudaError_t launch_decode_gather(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st);
cudaError_t launch_decode_shared(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st);   // decode_shared.cu

// bf16 dense pages: TMA-fed tensor-core kernel; FP8 records or a top-k list: the tensor-core
// kernel that gathers and converts rows itself.
inline bool use_tma_path(int fmt, int topk) { return fmt == MLA_KV_BF16 && topk == 0; }
inline DecodePlan plan_decode(int fmt, int B, int max_seq_len, int topk, int sms) {
    return use_tma_path(fmt, topk) ? plan_decode_tc(fmt, B, max_seq_len, topk, sms)
                                   : plan_decode_gather(fmt, B, max_seq_len, topk, sms);
}
inline cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st) {
    return use_tma_path(a.fmt, a.topk) ? launch_decode_tc(a, p, st) : launch_decode_gather(a, p, st);
}

}  // namespace mla
