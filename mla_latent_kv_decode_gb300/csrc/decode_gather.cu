// decode_gather.cu -- instantiations of the gather decode kernel (decode_gather.cuh) for the MLA
// record formats: FP8 mixed pages, FP8 mixed top-k rows and bf16 top-k rows; its plan and launch.
#include "decode_gather.cuh"

namespace mla {

// Same workspace as the dense bf16 kernel: 2 partial slots per cluster (fp32 [128][512] + lse
// [128]), then per request its first partial slot and last cluster (int32 [B][2]).
DecodePlan plan_decode_gather(int fmt, int B, int max_seq_len, int topk, int sms) {
    (void)fmt;
    DecodePlan p;
    const long long per_req = topk > 0 ? (topk + kT - 1) / kT : (max_seq_len + kT - 1) / kT;
    const int C = clusters_for_tiles((long long)B * per_req, sms);
    p.splits = C;
    p.workspace = (size_t)2 * C * kHeads * (kDc + 1) * sizeof(float) + (size_t)2 * B * sizeof(int32_t);
    p.workspace = (p.workspace + 255) / 256 * 256;
    p.launches = 2;
    return p;
}

cudaError_t launch_decode_gather(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t st) {
    const bool topk = a.topk_idx != nullptr && a.topk > 0;
    if (a.fmt == MLA_KV_V4_FP8 || a.fmt == MLA_KV_V41_FP4) return launch_decode_shared(a, plan, st);
    if (a.fmt == MLA_KV_FP8_MIXED)
        return topk ? launch_gather_instance<MLA_KV_FP8_MIXED, true>(a, plan, st)
                    : launch_gather_instance<MLA_KV_FP8_MIXED, false>(a, plan, st);
    if (!topk) return cudaErrorInvalidValue;   // dense bf16 pages: decode_tc_kernel
    return launch_gather_instance<MLA_KV_BF16, true>(a, plan, st);
}

}  // namespace mla
