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
constexpr int kHeads = MLA_HEADS;
constexpr int kPage = MLA_PAGE_TOKENS;
constexpr int kBf16RecordBytes = kDk * 2;    // 1152
constexpr int kFp8RecordBytes = kDc + 16 + kDr * 2;   // 656
constexpr int kFp8Group = 128;
constexpr int kFp8ScaleOff = kDc;            // 4 fp32 scales after the 512 codes
constexpr int kFp8RopeOff = kDc + 16;        // 64 bf16 rope after the scales

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
cudaError_t launch_combine(const float* o_part, const float* lse_part, int S, int B, int H,
                           __nv_bfloat16* out, float* lse, cudaStream_t st);

// Split-KV plan of one decode call.
struct DecodePlan {
    int splits;            // S: work units per request along the visible positions
    int chunk;             // positions per unit (multiple of 64 for dense, of 32 for sparse)
    size_t workspace;      // bytes of (o_part, lse_part) needed; 0 when splits == 1
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
    float* o_part;         // simt path: [S, B, H, 512] when splits > 1
    float* lse_part;       // simt path: [S, B, H]
    void* workspace;       // caller scratch of at least plan.workspace bytes
    DevCtl* ctl;
};

// Tensor-core path (bf16 dense) and CUDA-core path (FP8 mixed and top-k for now).
DecodePlan plan_decode_tc(int fmt, int B, int max_seq_len, int topk, int sms);
cudaError_t launch_decode_tc(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st);
DecodePlan plan_decode_simt(int fmt, int B, int max_seq_len, int topk, int sms);
cudaError_t launch_decode_simt(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st);

inline bool use_tc(int fmt, int topk) { return fmt == MLA_KV_BF16 && topk == 0; }
inline DecodePlan plan_decode(int fmt, int B, int max_seq_len, int topk, int sms) {
    return use_tc(fmt, topk) ? plan_decode_tc(fmt, B, max_seq_len, topk, sms)
                             : plan_decode_simt(fmt, B, max_seq_len, topk, sms);
}
inline cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st) {
    return use_tc(a.fmt, a.topk) ? launch_decode_tc(a, p, st) : launch_decode_simt(a, p, st);
}

}  // namespace mla
