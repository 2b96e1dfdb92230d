// decode_shared.cu -- instantiations of the gather decode kernel (decode_gather.cuh) for the shared
// K = V entry formats ("DeepSeek's KV Cache: From 3.9 MB to 890 B per Token", section "HCA: 128
// tokens into one", Fig. 15): V4 entries (584 B) and V4.1 entries (288 B), pages and top-k rows.
#include "decode_gather.cuh"

namespace mla {

cudaError_t launch_decode_shared(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t st) {
    const bool topk = a.topk_idx != nullptr && a.topk > 0;
    if (a.fmt == MLA_KV_V4_FP8)
        return topk ? launch_gather_instance<MLA_KV_V4_FP8, true>(a, plan, st)
                    : launch_gather_instance<MLA_KV_V4_FP8, false>(a, plan, st);
    if (a.fmt == MLA_KV_V41_FP4)
        return topk ? launch_gather_instance<MLA_KV_V41_FP4, true>(a, plan, st)
                    : launch_gather_instance<MLA_KV_V41_FP4, false>(a, plan, st);
    return cudaErrorInvalidValue;
}

}  // namespace mla
