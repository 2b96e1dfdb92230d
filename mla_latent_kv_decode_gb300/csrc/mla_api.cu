// mla_api.cu -- the C ABI of libmla: argument validation, per-device state, launches.
#include <cmath>
#include <cstring>
#include <mutex>

#include "mla_internal.cuh"

namespace mla {

__device__ DevCtl g_ctl = {0, 0, kDefaultWaitLimit, 0};

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DevCtl* g_ctl_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
int g_cc[kMaxDevices] = {};

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

bool init_device(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_ctl_ptr[dev]) return true;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ctl) != cudaSuccess) return false;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return false;
    g_sms[dev] = prop.multiProcessorCount;
    g_cc[dev] = prop.major * 10 + prop.minor;
    g_ctl_ptr[dev] = static_cast<DevCtl*>(p);
    return true;
}
}  // namespace

DevCtl* device_ctl() {
    int dev = current_device();
    if (dev < 0 || !init_device(dev)) return nullptr;
    return g_ctl_ptr[dev];
}

int num_sms() {
    int dev = current_device();
    if (dev < 0 || !init_device(dev)) return 0;
    return g_sms[dev];
}

int device_cc() {
    int dev = current_device();
    if (dev < 0 || !init_device(dev)) return 0;
    return g_cc[dev];
}

}  // namespace mla

using namespace mla;

namespace {
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool fmt_ok(int32_t fmt) { return fmt == MLA_KV_BF16 || fmt == MLA_KV_FP8_MIXED; }
bool shared_fmt_ok(int32_t fmt) { return fmt == MLA_KV_V4_FP8 || fmt == MLA_KV_V41_FP4; }
mla_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }
// The kernels are built for sm_103a only; any other device would fail at launch.
bool device_supported() { return device_cc() == 103; }

// mla_decode's checks of its sizes and scale (no pointer is looked at)
mla_status decode_shape_status(int32_t fmt, int64_t num_pages, int32_t max_pages, int32_t max_seq_len,
                               int32_t topk, int32_t B, int32_t H, float scale, bool shared = false) {
    if (!(shared ? shared_fmt_ok(fmt) : fmt_ok(fmt)) || B < 0 || H != kHeads || num_pages < 0 || max_pages < 0 ||
        max_seq_len < 0 || topk < 0)
        return MLA_ERR_INVALID;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return MLA_ERR_INVALID;
    if ((int64_t)max_seq_len > (int64_t)max_pages * kPage) return MLA_ERR_INVALID;
    return MLA_OK;
}

// mla_decode's checks of its pointers (null, alignment, top-k list given iff topk > 0)
mla_status decode_pointer_status(const void* pool, const void* q_lat, const void* q_rope,
                                 const int32_t* block_table, const int32_t* seq_lens,
                                 const int32_t* topk_idx, int32_t topk, const void* out,
                                 const float* lse) {
    if (!pool || !q_lat || !q_rope || !block_table || !seq_lens || !out || !lse)
        return MLA_ERR_INVALID;
    if ((topk_idx == nullptr) != (topk == 0)) return MLA_ERR_INVALID;
    if (!aligned(pool, 128) || !aligned(q_lat, 16) || !aligned(q_rope, 16) || !aligned(out, 16) ||
        !aligned(lse, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
        (topk_idx && !aligned(topk_idx, 4)))
        return MLA_ERR_INVALID;
    return MLA_OK;
}
}  // namespace

extern "C" {

size_t mla_record_bytes(int32_t fmt) {
    if (fmt == MLA_KV_BF16) return kBf16RecordBytes;
    if (fmt == MLA_KV_FP8_MIXED) return kFp8RecordBytes;
    if (fmt == MLA_KV_V4_FP8) return kV4EntryBytes;
    if (fmt == MLA_KV_V41_FP4) return kV41EntryBytes;
    return 0;
}

mla_status mla_cache_append(int32_t fmt, void* pool, int64_t num_pages, const void* c_kv,
                            const void* k_rope, const int32_t* slot, int64_t T,
                            cudaStream_t stream) {
    if (!fmt_ok(fmt) || T < 0 || num_pages < 0) return MLA_ERR_INVALID;
    if (T == 0) return MLA_OK;
    if (!pool || !c_kv || !k_rope || !slot) return MLA_ERR_INVALID;
    if (!aligned(pool, 128) || !aligned(c_kv, 16) || !aligned(k_rope, 16) || !aligned(slot, 4))
        return MLA_ERR_INVALID;
    DevCtl* ctl = device_ctl();
    if (!ctl) return MLA_ERR_CUDA;
    if (!device_supported()) return MLA_ERR_UNSUPPORTED;
    return from_cuda(launch_cache_append(fmt, static_cast<uint8_t*>(pool), num_pages,
                                         static_cast<const __nv_bfloat16*>(c_kv),
                                         static_cast<const __nv_bfloat16*>(k_rope), slot, T, ctl,
                                         stream));
}

mla_status mla_index_append(void* pool, int64_t num_pages, const void* k_index, const int32_t* slot,
                            int64_t T, cudaStream_t stream) {
    if (T < 0 || num_pages < 0) return MLA_ERR_INVALID;
    if (T == 0) return MLA_OK;
    if (!pool || !k_index || !slot) return MLA_ERR_INVALID;
    if (!aligned(pool, 16) || !aligned(k_index, 16) || !aligned(slot, 4)) return MLA_ERR_INVALID;
    DevCtl* ctl = device_ctl();
    if (!ctl) return MLA_ERR_CUDA;
    if (!device_supported()) return MLA_ERR_UNSUPPORTED;
    return from_cuda(launch_index_append(static_cast<uint8_t*>(pool), num_pages,
                                         static_cast<const __nv_bfloat16*>(k_index), slot, T, ctl, stream));
}

mla_status mla_indexer_score(const void* pool, int64_t num_pages, const void* q_index, const float* w_index,
                             const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                             int32_t B, int32_t max_seq_len, float* scores, cudaStream_t stream) {
    if (B < 0 || num_pages < 0 || max_pages < 1 || max_seq_len < 0 ||
        (int64_t)max_seq_len > (int64_t)max_pages * kPage)
        return MLA_ERR_INVALID;
    if (B == 0 || max_seq_len == 0) return MLA_OK;
    if (!pool || !q_index || !w_index || !block_table || !seq_lens || !scores) return MLA_ERR_INVALID;
    if (!aligned(pool, 16) || !aligned(q_index, 16) || !aligned(w_index, 4) || !aligned(block_table, 4) ||
        !aligned(seq_lens, 4) || !aligned(scores, 4))
        return MLA_ERR_INVALID;
    DevCtl* ctl = device_ctl();
    if (!ctl) return MLA_ERR_CUDA;
    if (!device_supported()) return MLA_ERR_UNSUPPORTED;
    return from_cuda(launch_indexer_score(static_cast<const uint8_t*>(pool), num_pages,
                                          static_cast<const __nv_bfloat16*>(q_index), w_index, block_table,
                                          max_pages, seq_lens, B, max_seq_len, scores, ctl, stream));
}

mla_status mla_topk_select(const float* scores, int64_t ld, const int32_t* seq_lens, int32_t B, int32_t K,
                           int32_t* topk_idx, cudaStream_t stream) {
    // two CTAs a request: 2 B must stay below 2^31 (a grid dimension and an int)
    if (B < 0 || B >= (1 << 30) || K < 1 || ld < 0) return MLA_ERR_INVALID;
    if (B == 0) return MLA_OK;
    if (!scores || !seq_lens || !topk_idx) return MLA_ERR_INVALID;
    if (!aligned(scores, 4) || !aligned(seq_lens, 4) || !aligned(topk_idx, 4)) return MLA_ERR_INVALID;
    if (!device_supported()) return MLA_ERR_UNSUPPORTED;
    return from_cuda(launch_topk_select(scores, ld, seq_lens, B, K, topk_idx, stream));
}

size_t mla_decode_workspace_bytes(int32_t fmt, int32_t B, int32_t H, int32_t max_seq_len,
                                  int32_t topk) {
    if (!(fmt_ok(fmt) || shared_fmt_ok(fmt)) || B <= 0 || H != kHeads || max_seq_len < 0 || topk < 0) return 0;
    int sms = num_sms();
    if (sms <= 0) sms = 152;
    return plan_decode(fmt, B, max_seq_len, topk, sms).workspace;
}

int32_t mla_decode_launches(int32_t fmt, int32_t B, int32_t H, int32_t max_seq_len,
                            int32_t topk) {
    if (!(fmt_ok(fmt) || shared_fmt_ok(fmt)) || B <= 0 || H != kHeads || max_seq_len < 0 || topk < 0) return 0;
    int sms = num_sms();
    if (sms <= 0) sms = 152;
    return plan_decode(fmt, B, max_seq_len, topk, sms).launches;
}

mla_status mla_decode(int32_t fmt, const void* pool, int64_t num_pages, const void* q_lat,
                      const void* q_rope, const int32_t* block_table, int32_t max_pages,
                      const int32_t* seq_lens, int32_t max_seq_len, const int32_t* topk_idx,
                      int32_t topk, int32_t B, int32_t H, float scale, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    mla_status st = decode_shape_status(fmt, num_pages, max_pages, max_seq_len, topk, B, H, scale);
    if (st != MLA_OK || B == 0) return st;
    st = decode_pointer_status(pool, q_lat, q_rope, block_table, seq_lens, topk_idx, topk, out, lse);
    if (st != MLA_OK) return st;
    DevCtl* ctl = device_ctl();
    if (!ctl) return MLA_ERR_CUDA;
    if (!device_supported()) return MLA_ERR_UNSUPPORTED;
    DecodePlan plan = plan_decode(fmt, B, max_seq_len, topk, num_sms());
    DecodeArgs a;
    a.fmt = fmt;
    a.pool = static_cast<const uint8_t*>(pool);
    a.num_pages = num_pages;
    a.q_lat = static_cast<const __nv_bfloat16*>(q_lat);
    a.q_rope = static_cast<const __nv_bfloat16*>(q_rope);
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.seq_lens = seq_lens;
    a.max_seq_len = max_seq_len;
    a.topk_idx = topk_idx;
    a.topk = topk;
    a.B = B;
    a.scale = scale;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.workspace = workspace;
    a.ctl = ctl;
    if (plan.workspace > 0 &&
        (!workspace || workspace_bytes < plan.workspace || !aligned(workspace, 256)))
        return MLA_ERR_INVALID;
    return from_cuda(launch_decode(a, plan, stream));
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// Decode with a static scratch array, for callers that cannot allocate device memory (see mla.h).
// ------------------------------------------------------------------------------------------------
namespace {
// The split-KV scratch of mla_decode_noalloc.  In host code this name is only a stand-in for the
// device array: its device address comes from cudaGetSymbolAddress, once per device.
__device__ __align__(256) unsigned char g_static_workspace[MLA_STATIC_WORKSPACE_BYTES];
std::mutex g_static_mu;
void* g_static_ptr[64] = {};

void* static_workspace_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess) return nullptr;
        g_static_ptr[dev] = p;
    }
    return g_static_ptr[dev];
}
}  // namespace

extern "C" {

mla_status mla_decode_noalloc(int32_t fmt, const void* pool, int64_t num_pages, const void* q_lat,
                              const void* q_rope, const int32_t* block_table, int32_t max_pages,
                              const int32_t* seq_lens, int32_t max_seq_len,
                              const int32_t* topk_idx, int32_t topk, int32_t B, int32_t H,
                              float scale, void* out, float* lse, cudaStream_t stream) {
    // the checks of mla_decode first, and the size limit before the pointers, so that an
    // over-size call is refused whatever it points at; the array is looked up only when a
    // launch follows
    mla_status st = decode_shape_status(fmt, num_pages, max_pages, max_seq_len, topk, B, H, scale);
    if (st != MLA_OK || B == 0) return st;
    if (mla_decode_workspace_bytes(fmt, B, H, max_seq_len, topk) > MLA_STATIC_WORKSPACE_BYTES)
        return MLA_ERR_UNSUPPORTED;
    st = decode_pointer_status(pool, q_lat, q_rope, block_table, seq_lens, topk_idx, topk, out, lse);
    if (st != MLA_OK) return st;
    void* ws = static_workspace_for_current_device();
    if (!ws) return MLA_ERR_CUDA;
    return mla_decode(fmt, pool, num_pages, q_lat, q_rope, block_table, max_pages, seq_lens,
                      max_seq_len, topk_idx, topk, B, H, scale, out, lse, ws,
                      MLA_STATIC_WORKSPACE_BYTES, stream);
}

mla_status mla_combine(const float* o_part, const float* lse_part, int32_t S, int32_t B, int32_t H,
                       void* out, float* lse, cudaStream_t stream) {
    if (S <= 0 || B < 0 || H <= 0) return MLA_ERR_INVALID;
    if (B == 0) return MLA_OK;
    if (!o_part || !lse_part || !out || !lse) return MLA_ERR_INVALID;
    if (!aligned(o_part, 16) || !aligned(lse_part, 4) || !aligned(out, 16) || !aligned(lse, 4))
        return MLA_ERR_INVALID;
    if (!device_ctl()) return MLA_ERR_CUDA;
    if (!device_supported()) return MLA_ERR_UNSUPPORTED;
    return from_cuda(launch_combine(o_part, lse_part, S, B, H, static_cast<__nv_bfloat16*>(out),
                                    lse, stream));
}

mla_status mla_shared_kv_append(int32_t fmt, void* pool, int64_t num_pages, const void* entry,
                                const int32_t* slot, int64_t T, cudaStream_t stream) {
    if (!shared_fmt_ok(fmt) || T < 0 || num_pages < 0) return MLA_ERR_INVALID;
    if (T == 0) return MLA_OK;
    if (!pool || !entry || !slot) return MLA_ERR_INVALID;
    if (!aligned(pool, 128) || !aligned(entry, 16) || !aligned(slot, 4)) return MLA_ERR_INVALID;
    DevCtl* ctl = device_ctl();
    if (!ctl) return MLA_ERR_CUDA;
    if (!device_supported()) return MLA_ERR_UNSUPPORTED;
    return from_cuda(launch_shared_append(fmt, static_cast<uint8_t*>(pool), num_pages,
                                          static_cast<const __nv_bfloat16*>(entry), slot, T, ctl, stream));
}

mla_status mla_shared_kv_decode(int32_t fmt, const void* pool, int64_t num_pages, const void* q,
                                const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                                int32_t max_seq_len, const int32_t* topk_idx, int32_t topk, int32_t B,
                                int32_t H, float scale, const float* sink, const float* rope_cs, void* out,
                                float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    mla_status st = decode_shape_status(fmt, num_pages, max_pages, max_seq_len, topk, B, H, scale, true);
    if (st != MLA_OK || B == 0) return st;
    // (q takes the place of q_lat; there is no separate rotary query)
    st = decode_pointer_status(pool, q, q, block_table, seq_lens, topk_idx, topk, out, lse);
    if (st != MLA_OK) return st;
    if ((sink && !aligned(sink, 4)) || (rope_cs && !aligned(rope_cs, 4))) return MLA_ERR_INVALID;
    DevCtl* ctl = device_ctl();
    if (!ctl) return MLA_ERR_CUDA;
    if (!device_supported()) return MLA_ERR_UNSUPPORTED;
    DecodePlan plan = plan_decode_gather(fmt, B, max_seq_len, topk, num_sms());
    DecodeArgs a;
    a.fmt = fmt;
    a.pool = static_cast<const uint8_t*>(pool);
    a.num_pages = num_pages;
    a.q_lat = static_cast<const __nv_bfloat16*>(q);
    a.q_rope = nullptr;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.seq_lens = seq_lens;
    a.max_seq_len = max_seq_len;
    a.topk_idx = topk_idx;
    a.topk = topk;
    a.B = B;
    a.scale = scale;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.workspace = workspace;
    a.ctl = ctl;
    a.sink = sink;
    a.rope_cs = rope_cs;
    if (plan.workspace > 0 &&
        (!workspace || workspace_bytes < plan.workspace || !aligned(workspace, 256)))
        return MLA_ERR_INVALID;
    return from_cuda(launch_decode_gather(a, plan, stream));
}

namespace {
mla_status value_project_status(const void* u, const void* w1, const void* w2, int32_t B, int32_t H, int32_t D,
                                const void* y) {
    if (B < 0 || H < 1 || H > 65535 || D < kDv || D % 128 != 0 || (int64_t)B > 65535LL * 128)
        return MLA_ERR_INVALID;
    if (B == 0) return MLA_OK;
    if (!u || !w1 || !y) return MLA_ERR_INVALID;
    if (!aligned(u, 16) || !aligned(w1, 16) || !aligned(y, 16) || (w2 && !aligned(w2, 16)))
        return MLA_ERR_INVALID;
    return MLA_OK;
}
}  // namespace

mla_status mla_value_project(const void* u, const void* w_uv_t, const void* w_o_t, int32_t B, int32_t H,
                             int32_t D, void* z, void* y, cudaStream_t stream) {
    mla_status st = value_project_status(u, w_uv_t, w_o_t, B, H, D, y);
    if (st != MLA_OK || B == 0) return st;
    if (!w_o_t || !z || !aligned(z, 16)) return MLA_ERR_INVALID;
    DevCtl* ctl = device_ctl();
    if (!ctl) return MLA_ERR_CUDA;
    if (!device_supported()) return MLA_ERR_UNSUPPORTED;
    return from_cuda(launch_value_project(static_cast<const __nv_bfloat16*>(u),
                                          static_cast<const __nv_bfloat16*>(w_uv_t),
                                          static_cast<const __nv_bfloat16*>(w_o_t), B, H, D,
                                          static_cast<__nv_bfloat16*>(z), static_cast<__nv_bfloat16*>(y), ctl,
                                          stream));
}

mla_status mla_value_project_merged(const void* u, const void* w_hat_t, int32_t B, int32_t H, int32_t D,
                                    void* y, cudaStream_t stream) {
    mla_status st = value_project_status(u, w_hat_t, nullptr, B, H, D, y);
    if (st != MLA_OK || B == 0) return st;
    DevCtl* ctl = device_ctl();
    if (!ctl) return MLA_ERR_CUDA;
    if (!device_supported()) return MLA_ERR_UNSUPPORTED;
    return from_cuda(launch_value_project_merged(static_cast<const __nv_bfloat16*>(u),
                                                 static_cast<const __nv_bfloat16*>(w_hat_t), B, H, D,
                                                 static_cast<__nv_bfloat16*>(y), ctl, stream));
}

mla_status mla_check_status(cudaStream_t stream) {
    DevCtl* ctl = device_ctl();
    if (!ctl) return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    DevCtl h;
    if (cudaMemcpy(&h, ctl, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
    if (h.status != 0) {
        int32_t zero[2] = {0, 0};
        if (cudaMemcpy(ctl, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return MLA_ERR_CUDA;
    }
    return static_cast<mla_status>(h.status);
}

const char* mla_status_string(mla_status s) {
    switch (s) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID: return "invalid argument";
        case MLA_ERR_BOUNDS: return "index outside the cache pool";
        case MLA_ERR_TIMEOUT: return "bounded wait ran out inside a kernel";
        case MLA_ERR_CUDA: return "CUDA error";
        case MLA_ERR_UNSUPPORTED: return "unsupported device or size";
        case MLA_ERR_RANGE: return "value outside the range of the format's arithmetic";
    }
    return "unknown status";
}

mla_status mla_set_wait_limit(uint32_t iterations) {
    DevCtl* ctl = device_ctl();
    if (!ctl) return MLA_ERR_CUDA;
    uint32_t v = iterations ? iterations : kDefaultWaitLimit;
    return from_cuda(cudaMemcpy(&ctl->wait_limit, &v, sizeof v, cudaMemcpyHostToDevice));
}

mla_status mla_e4m3_encode(const float* x, uint8_t* codes, int64_t n, cudaStream_t stream) {
    if (n < 0) return MLA_ERR_INVALID;
    if (n == 0) return MLA_OK;
    if (!x || !codes || !aligned(x, 4)) return MLA_ERR_INVALID;
    if (!device_ctl()) return MLA_ERR_CUDA;
    if (!device_supported()) return MLA_ERR_UNSUPPORTED;
    return from_cuda(launch_e4m3_encode(x, codes, n, stream));
}

}  // extern "C"
