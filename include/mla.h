/*
 * mla.h -- libmla: absorbed Multi-head Latent Attention decode over a paged latent cache,
 * for NVIDIA GB300 (sm_103a).
 *
 * What is computed.  Each cached token of one layer is a latent record [c_KV (512) | k_rope (64)]
 * ("DeepSeek's KV Cache: From 3.9 MB to 890 B per Token", Fig. 3: the cache keeps only the
 * 512-dim latent C^KV and the 64-dim rotary key K^R of each token).  For a new token, every
 * head h brings a query already absorbed into the latent space, q_lat[h] = Q^C_h (W^UK_h)^T
 * (512), and a rotary query q_rope[h] (64) (same page, Fig. 5 (2) "Absorb").  Decode scores every visible position t,
 *     s_t = scale * (q_lat[h] . c_t + q_rope[h] . k_rope_t)              (Fig. 4 (1); scale is
 *                                                                        1/sqrt(d_k + d_r))
 * and returns the absorbed value path U_h = sum_t softmax(s)_t c_t (Fig. 6 (2)) together with
 * lse_h = ln sum_t exp(s_t).  Optionally only listed positions are visible (the DSA selection
 * mask of Fig. 10, "MLA that reads only the picked positions").
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller; libmla allocates nothing.
 *    Calls are asynchronous on the caller's stream; host-side validation failures return a
 *    non-zero status and launch nothing.
 *  - bf16 arrays hold IEEE bfloat16 values; every array is dense, row-major, C-contiguous.
 *  - Errors the kernels detect (a page index outside the pool, a wait that ran out) are recorded
 *    in a per-device error word and reported, then cleared, by mla_check_status().  The outputs
 *    of a call that recorded an error are undefined.
 *  - Outputs must not alias inputs.  A token must be written by mla_cache_append before an
 *    mla_decode reads it; ordering on one stream is enough.
 *  - Device buffers must be 16-byte aligned; the cache pool must be 128-byte aligned.
 *
 * Geometry fixed by the format: D_C = 512 latent dims, D_R = 64 rope dims, H = 128 heads,
 * 64 tokens per page.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID = 1,      /* bad argument (null pointer, size, alignment, format)        */
    MLA_ERR_BOUNDS = 2,       /* a kernel met a page/slot index outside the pool             */
    MLA_ERR_TIMEOUT = 3,      /* a bounded wait inside a kernel ran out; the kernel returned */
    MLA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed                           */
    MLA_ERR_UNSUPPORTED = 5,  /* the device is not sm_103 / sm_100-family, or a size limit   */
    MLA_ERR_RANGE = 6         /* a kernel met a value outside the range its format's arithmetic
                                 carries (see the FP8 notes of mla_decode)                   */
} mla_status;

typedef enum {
    /* 1,152 B per token: 512 bf16 latent then 64 bf16 rope ("DeepSeek's KV Cache",
     * "Calculating V2's KV cache": (C^KV 512 + K^R 64) x 2 B). */
    MLA_KV_BF16 = 0,
    /* 656 B per token: 512 E4M3 latent codes, 4 fp32 scales (one per 128 latent dims),
     * 64 bf16 rope, in that order and without padding ("DeepSeek's KV Cache",
     * "Calculating V3.2's KV cache": 512 + 16 + 128 = 656 B). */
    MLA_KV_FP8_MIXED = 1,
    /* Shared K = V entries ("DeepSeek's KV Cache", section "HCA: 128 tokens into one", Fig. 15: one
     * 512-dim entry E per position serves as both Key and Value; its last 64 dims carry RoPE).
     * Written by mla_shared_kv_append and read by mla_shared_kv_decode only.
     * 584 B per entry ("Calculating V4-Flash's KV cache"): 448 E4M3 codes with one UE8M0 scale
     * per 64 dims, 64 bf16 RoPE dims, 7 scale bytes + 1 pad byte.  A 64-entry page (37,376 B)
     * holds its entries field by field: codes [64][448], then RoPE [64][64] bf16, then scale
     * bytes [64][8], so that each field starts on a 16-byte boundary. */
    MLA_KV_V4_FP8 = 2,
    /* 288 B per entry ("Calculating V4.1-Flash's KV cache"): 512 E2M1 codes, two per byte (dim 2i
     * in the low nibble), then 32 E4M3 scales, one per 16 dims; entries one after another. */
    MLA_KV_V41_FP4 = 3
} mla_kv_format;

#define MLA_D_C 512
#define MLA_D_R 64
#define MLA_HEADS 128
#define MLA_PAGE_TOKENS 64

/* Bytes of one token's record: 1152 (MLA_KV_BF16), 656 (MLA_KV_FP8_MIXED), 584 (MLA_KV_V4_FP8)
 * or 288 (MLA_KV_V41_FP4); 0 for an unknown format.  Host only. */
size_t mla_record_bytes(int32_t fmt);

/* Write T new tokens into the paged pool ("DeepSeek's KV Cache", Fig. 3: C^KV and K^R are what
 * is cached; "Calculating V3.2's KV cache" for the FP8 mixed record).
 *   pool       : device, num_pages * 64 * mla_record_bytes(fmt) bytes; slot s lives at byte
 *                s * mla_record_bytes(fmt) (page = s / 64, row = s % 64).
 *   c_kv       : device bf16 [T, 512]  latent of each new token.
 *   k_rope     : device bf16 [T, 64]   rotary key of each new token (already rotated).
 *   slot       : device int32 [T]      destination slot; a negative slot skips the row; a slot
 *                >= num_pages * 64 is not written and records MLA_ERR_BOUNDS.
 * BF16: the 576 values are stored as given.  FP8 mixed, per 128-dim group g: amax = max |x|,
 * s_g = amax / 448 (fp32, correctly rounded), code = E4M3(x / s_g) rounded to nearest even and
 * saturated to +-448; amax = 0 gives s_g = 0 and zero codes; rope is stored as bf16.
 * Only the listed slots change.  Returns MLA_ERR_INVALID for null pointers, T < 0, an unknown
 * format or a misaligned pool. */
mla_status mla_cache_append(int32_t fmt, void* pool, int64_t num_pages, const void* c_kv,
                            const void* k_rope, const int32_t* slot, int64_t T,
                            cudaStream_t stream);

/* Workspace bytes mla_decode needs for these sizes (0 when no split-KV partials are needed).
 * max_seq_len is an upper bound of seq_lens; topk is 0 for dense decode. Host only. */
size_t mla_decode_workspace_bytes(int32_t fmt, int32_t B, int32_t H, int32_t max_seq_len,
                                  int32_t topk);

/* Number of kernels one mla_decode call with these sizes launches (1, or 2 when split-KV
 * partials are merged by a separate kernel).  Host only. */
int32_t mla_decode_launches(int32_t fmt, int32_t B, int32_t H, int32_t max_seq_len, int32_t topk);

/* Absorbed MLA decode of one layer for B requests (the per-head computation in the file
 * comment; "DeepSeek's KV Cache", Fig. 4 (1), Fig. 5 (2), Fig. 6 (2), Fig. 10).
 *   fmt, pool, num_pages : the cache written by mla_cache_append.
 *   q_lat      : device bf16 [B, H, 512]  absorbed content queries.
 *   q_rope     : device bf16 [B, H, 64]   rotary queries.
 *   block_table: device int32 [B, max_pages]; position t of request b is row t % 64 of page
 *                block_table[b][t / 64].
 *   seq_lens   : device int32 [B]; request b sees positions 0 .. seq_lens[b]-1 (the newest
 *                token included).  Every seq_lens[b] must be <= max_seq_len <= max_pages * 64.
 *   max_seq_len: host-side upper bound of seq_lens, used to size the split-KV grid.
 *   topk_idx   : NULL for dense decode, or device int32 [B, topk]: request b sees only the
 *                listed positions p with 0 <= p < seq_lens[b] (others, e.g. -1 padding, are
 *                skipped).  Listed positions are expected distinct; a repeated one is counted
 *                as often as it is listed.
 *   B >= 0, H == 128, scale > 0 finite (normally 1/sqrt(192)).
 *   out        : device bf16 [B, H, 512] = sum_t softmax(s)_t c_t (zeros if nothing is visible).
 *   lse        : device fp32 [B, H] = ln sum_t exp(s_t) (-inf if nothing is visible).
 *   workspace  : device scratch of at least mla_decode_workspace_bytes(...) bytes (may be NULL
 *                when that is 0); 256-byte aligned; its contents are clobbered.
 * A page index outside [0, num_pages) met while reading records MLA_ERR_BOUNDS.
 * Arithmetic: scores and outputs accumulate in fp32 on the tensor cores.  bf16 records: bf16
 * operands, P rounded once to bf16 (2^-9 of each weight; O is divided by the sum of the rounded
 * P, so the weights still sum to one).  Where the weight sits on two or three positions, that
 * rounding moves an output element by up to about 2^-10 of the rows' difference, on top of the
 * bf16 output's own rounding (up to 2^-9 of its magnitude).  FP8 records: the E4M3 codes enter as f16 (exact), and so
 * does q_lat, converted once per request (exact for |q| in [2^-14, 65504); smaller magnitudes
 * lose low bits).  Each 128-dim group's scale multiplies in fp32: on that group's partial score,
 * and on P as f16(P * scale), which stays finite for group scales up to 255 (absmax up to
 * 114,240) because the running max is kept within 2^8 of every P.  Outside those two ranges the
 * FP8 path does not compute: a q_lat element of magnitude 65520 or more (it would overflow f16),
 * or a visible record with a group scale above 255 (or not finite), records MLA_ERR_RANGE. */
mla_status mla_decode(int32_t fmt, const void* pool, int64_t num_pages, const void* q_lat,
                      const void* q_rope, const int32_t* block_table, int32_t max_pages,
                      const int32_t* seq_lens, int32_t max_seq_len, const int32_t* topk_idx,
                      int32_t topk, int32_t B, int32_t H, float scale, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* mla_decode without a caller-provided workspace (this entry point has no counterpart in the
 * pages; it is a convenience of this library).
 *
 * For callers that cannot allocate device memory at the point where they decode: a plug-in
 * running inside a host application that owns every device allocation, or a serving loop that
 * must not allocate (cudaMalloc synchronises the device and may fail under memory pressure)
 * once it is running.  Such a caller still owns and passes all inputs and outputs; the split-KV
 * scratch comes from a static device array of MLA_STATIC_WORKSPACE_BYTES that every GPU holds
 * from the first use of this library until the process exits.  Nothing is allocated: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Arguments, results and errors are those of mla_decode (without workspace/workspace_bytes).
 * Additionally returns MLA_ERR_UNSUPPORTED, before launching anything, when
 * mla_decode_workspace_bytes(fmt, B, H, max_seq_len, topk) exceeds MLA_STATIC_WORKSPACE_BYTES.
 * The order of the host checks: sizes and scale (MLA_ERR_INVALID), then B == 0 (MLA_OK, nothing
 * touched), then the size limit (MLA_ERR_UNSUPPORTED), then the pointers (MLA_ERR_INVALID).
 *
 * The first call on a device that passes those checks, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and keeps it; make that first call before any
 * stream capture.  All
 * calls on a device share the one array, which keeps whatever the last call left in it (the
 * decode writes every scratch byte it reads, so nothing has to start at zero).  Calls whose
 * executions overlap on the GPU (on different streams, or from different threads) race on the
 * array: order them, e.g. on one stream. */
#define MLA_STATIC_WORKSPACE_BYTES ((size_t)48 << 20)
mla_status mla_decode_noalloc(int32_t fmt, const void* pool, int64_t num_pages, const void* q_lat,
                              const void* q_rope, const int32_t* block_table, int32_t max_pages,
                              const int32_t* seq_lens, int32_t max_seq_len,
                              const int32_t* topk_idx, int32_t topk, int32_t B, int32_t H,
                              float scale, void* out, float* lse, cudaStream_t stream);

/* Split-KV merge: S partial results of the same queries over disjoint position sets.
 *   o_part  : device fp32 [S, B, H, 512] normalised partial outputs.
 *   lse_part: device fp32 [S, B, H] partial log-sum-exps (-inf for an empty part).
 *   out     : device bf16 [B, H, 512] = sum_i exp(lse_i - lse) o_i;  lse: device fp32 [B, H]
 *             = ln sum_i exp(lse_i).  All parts empty: out = 0, lse = -inf.
 * This is the renormalisation of a softmax restricted to parts of the visible set ("DeepSeek's
 * KV Cache", Fig. 10; "Shared KV Memory", "What is lost by restricting the support?"). */
mla_status mla_combine(const float* o_part, const float* lse_part, int32_t S, int32_t B,
                       int32_t H, void* out, float* lse, cudaStream_t stream);

/* Synchronise `stream`, then return and clear the first error a kernel recorded on the current
 * device (MLA_OK if none); a pending CUDA error is returned as MLA_ERR_CUDA. */
mla_status mla_check_status(cudaStream_t stream);

/* Static description of a status code. */
const char* mla_status_string(mla_status status);

/* Iteration cap of every bounded wait inside libmla kernels on the current device (0 restores
 * the default).  When a wait runs out the kernel records MLA_ERR_TIMEOUT, drains its own
 * copies in flight, frees its tensor memory and returns.  Meant for tests of that path. */
mla_status mla_set_wait_limit(uint32_t iterations);

/* E4M3 encoding of n fp32 values with the device conversion mla_cache_append uses (round to
 * nearest even, saturating to +-448): codes[i] = E4M3(x[i]).  Device pointers; for checking
 * the conversion against an independent encoder (OCP OFP8 specification, format E4M3). */
mla_status mla_e4m3_encode(const float* x, uint8_t* codes, int64_t n, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * DSA lightning indexer ("DeepSeek's KV Cache: From 3.9 MB to 890 B per Token", sections "DSA:
 * three things the indexer builds" (Fig. 8), "The score that picks positions" (Fig. 9) and
 * "Calculating V3.2's KV cache" (search key)).  The indexer ranks the positions a query may read:
 *     I(t, s) = sum_j w(t, j) * ReLU(q(t, j) . k(s)),  j < 64 indexer heads, 128 dims,
 * and each query keeps its (up to) K highest-scoring visible positions; the result is the
 * topk_idx of mla_decode.
 * ------------------------------------------------------------------------------------------ */
#define MLA_INDEX_HEADS 64
#define MLA_INDEX_DIM 128
/* One 64-token page of the search-key pool: the 64 keys' 128 E4M3 codes (token-major, 8,192 B)
 * followed by their 64 fp32 scales (256 B): 132 B per token, "128 FP8 values with one FP32 scale
 * for all 128 dimensions". */
#define MLA_INDEX_PAGE_BYTES 8448

/* Write T search keys into the search-key pool.
 *   pool       : device, num_pages * MLA_INDEX_PAGE_BYTES bytes, 16-byte aligned; slot s is row
 *                s % 64 of page s / 64 (the pages can share the main cache's block_table).
 *   k_index    : device bf16 [T, 128]  search key of each new token.
 *   slot       : device int32 [T]      destination slot; negative skips the row; a slot >=
 *                num_pages * 64 is not written and records MLA_ERR_BOUNDS.
 * Per key: amax = max |x|, s = amax / 448 (fp32, correctly rounded), code = E4M3(x / s) rounded
 * to nearest even and saturated to +-448; amax = 0 gives s = 0 and zero codes.  Only the listed
 * slots change.  MLA_ERR_INVALID for null pointers, T < 0 or a misaligned pointer. */
mla_status mla_index_append(void* pool, int64_t num_pages, const void* k_index, const int32_t* slot,
                            int64_t T, cudaStream_t stream);

/* Indexer scores of B queries at every visible position.
 *   pool, num_pages : the search-key pool written by mla_index_append.
 *   q_index    : device bf16 [B, 64, 128]  indexer query of each head.
 *   w_index    : device fp32 [B, 64]       head weights (any sign; not a probability).
 *   block_table, max_pages, seq_lens, max_seq_len : as in mla_decode (position t of request b is
 *                row t % 64 of page block_table[b][t / 64]; positions t < seq_lens[b] are visible).
 *   scores     : device fp32 [B, max_seq_len]; scores[b][t] = I(b, t) for t < seq_lens[b]; the
 *                rest of each row is not written.
 * The dot products have exact products and fp32 accumulation (E4M3 codes convert to f16 exactly;
 * per head, q is scaled by a power of two into f16 range and the head weight by its inverse, so
 * every bf16 q element within 2^31 of its head's largest magnitude is exact); the key scale
 * multiplies after the ReLU (it is >= 0).  A visible position whose page is outside the pool
 * records MLA_ERR_BOUNDS (its score is then unspecified; no memory outside the pool is read).  MLA_ERR_INVALID for
 * null or misaligned pointers, B < 0, max_pages < 1 or max_seq_len > max_pages * 64. */
mla_status mla_indexer_score(const void* pool, int64_t num_pages, const void* q_index, const float* w_index,
                             const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                             int32_t B, int32_t max_seq_len, float* scores, cudaStream_t stream);

/* Top-k selection per row: among positions t < seq_lens[b] (clamped to [0, ld]) of row b of
 * `scores` (device fp32 [B, ld]), the K highest scores, a tie going to the lower position
 * (section "The score that picks positions": every query keeps at most 2,048 of the positions
 * visible to it, those with the largest scores), written to topk_idx[b] (device int32
 * [B, K]) in increasing position order and padded with -1 past the min(K, seq_lens[b]) picks: directly the topk_idx of mla_decode.  Scores must
 * not be NaN.  MLA_ERR_INVALID for null pointers, B < 0, B >= 2^30, K < 1 or ld < 0. */
mla_status mla_topk_select(const float* scores, int64_t ld, const int32_t* seq_lens, int32_t B, int32_t K,
                           int32_t* topk_idx, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Shared K = V decode over compressed V4 / V4.1 entries ("DeepSeek's KV Cache: From 3.9 MB to
 * 890 B per Token", section "HCA: 128 tokens into one", Fig. 15).  Each visible entry E (512
 * dims, the last 64 carrying RoPE) serves as both Key and Value; the softmax adds a per-head sink
 * exp(z'_h) to its denominator (so the weights may sum to less than one); the output's last 64
 * dims are rotated back by the query position (each entry's contribution then carries the
 * relative rotation s - t):
 *     s_t = scale * (q[h] . E_t)        L_h = sum_t exp(s_t) + exp(z'_h)
 *     o[h] = sum_t (exp(s_t) / L_h) E_t,  then dims (448 + 2i, 448 + 2i + 1) rotated by -theta_i
 *     lse[h] = ln L_h
 * ------------------------------------------------------------------------------------------ */

/* Write T entries into a pool of format MLA_KV_V4_FP8 or MLA_KV_V41_FP4.
 *   pool  : device, num_pages * 64 * mla_record_bytes(fmt) bytes, 128-byte aligned (the page
 *           layouts are given with the formats).
 *   entry : device bf16 [T, 512]  the entries (dims 448..511: the RoPE part, already rotated).
 *   slot  : device int32 [T]  page * 64 + row; negative skips the row; >= num_pages * 64 is not
 *           written and records MLA_ERR_BOUNDS.
 * V4: per 64-dim group of dims 0..447, amax = max |x| and the scale 2^e with the smallest integer e
 * (clamped to [-127, 127]) such that 448 * 2^e >= amax, stored as the byte e + 127 (UE8M0); code =
 * E4M3(x * 2^-e) rounded to nearest even (saturating); amax = 0 stores byte 0 and zero codes;
 * dims 448..511 are stored as bf16; the pad byte is 0.
 * V4.1: per 16-dim group, s = E4M3(amax / 6) (fp32 division correctly rounded, then rounded to
 * nearest even, saturating); code = E2M1(x / value(s)) rounded to nearest even, saturating at 6
 * (all zero when value(s) = 0).
 * Only the listed slots change.  MLA_ERR_INVALID for another format, null or misaligned pointers or
 * T < 0. */
mla_status mla_shared_kv_append(int32_t fmt, void* pool, int64_t num_pages, const void* entry,
                                const int32_t* slot, int64_t T, cudaStream_t stream);

/* Shared K = V decode of B requests (the computation above).
 *   fmt, pool, num_pages : the entries written by mla_shared_kv_append.
 *   q          : device bf16 [B, H, 512]  queries (already normalised and rotated by the caller).
 *   block_table, max_pages, seq_lens, max_seq_len, topk_idx, topk, B, H (== 128), scale : as in
 *                mla_decode (scale is normally 1/sqrt(512)); top-k lists pick the visible entries.
 *   sink       : device fp32 [128]  z'_h, or NULL for none (then L_h has no extra term).
 *   rope_cs    : device fp32 [B, 64]  per request cos(theta_i) (i < 32) then sin(theta_i) of the
 *                query position's RoPE angles, or NULL for no rotation.
 *   out        : device bf16 [B, H, 512];  lse : device fp32 [B, H] (a request with no visible entry:
 *                out = 0 and lse = z'_h, or -inf without a sink).
 *   workspace  : mla_decode_workspace_bytes(fmt, B, H, max_seq_len, topk) bytes, 256-byte aligned.
 * Arithmetic: every stored code converts exactly to bf16 (an E4M3 value times a power of two; an
 * E2M1 value times an E4M3 value); q . E and P E accumulate in fp32 on the tensor cores with bf16
 * operands and P rounded once to bf16.  Errors as mla_decode. */
mla_status mla_shared_kv_decode(int32_t fmt, const void* pool, int64_t num_pages, const void* q,
                                const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                                int32_t max_seq_len, const int32_t* topk_idx, int32_t topk, int32_t B,
                                int32_t H, float scale, const float* sink, const float* rope_cs, void* out,
                                float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Value up-projection and output projection of the decode output ("DeepSeek's KV Cache: From
 * 3.9 MB to 890 B per Token", section "Computing without expanding Key and Value", Fig. 6).
 * mla_decode returns per head the weighted latent sum U_h (512); what the layer adds to the
 * residual stream is Y = sum_h (U_h W^UV_h) W^O_h, where W^UV_h (512 x 128) rebuilds head h's
 * value width and W^O_h is head h's block of 128 rows of the output weight W^O (Fig. 6 (2)), or
 * Y = sum_h U_h What^O_h with the pre-merged What^O_h = W^UV_h W^O_h (512 x D, Fig. 6 (3)).
 * Weights are passed transposed, in the [output, input] layout, bf16.
 * ------------------------------------------------------------------------------------------ */
#define MLA_D_V 128

/* Fig. 6 (2).
 *   u      : device bf16 [B, H, 512]    U, e.g. mla_decode's out.
 *   w_uv_t : device bf16 [H, 128, 512]  row j of head h is column j of W^UV_h.
 *   w_o_t  : device bf16 [D, H * 128]   row n is column n of W^O (columns h * 128 .. h * 128 + 127
 *                                        of a row belong to head h).
 *   z      : device bf16 [2, B, H * 128], written: Z_h = U_h W^UV_h of every head, heads side by
 *            side, as two planes whose sum carries Z: z[0] = bf16(Z), z[1] = bf16(Z - z[0]) (about
 *            16 significant bits).  It is the intermediate of the two products.
 *   y      : device bf16 [B, D]  Y.
 * Products: bf16 operands, fp32 accumulation on the tensor cores; Z enters the second product as
 * its two planes, whose two fp32 results are added; Y is rounded once to bf16.  The second
 * product's reduction over H * 128 is split across up to 8 CTAs whose fp32 partial sums are added
 * in a fixed order.  B >= 0 (B = 0 does nothing), 1 <= H <= 65535, D a positive multiple of 128,
 * B <= 8,388,480; pointers 16-byte aligned; otherwise MLA_ERR_INVALID. */
mla_status mla_value_project(const void* u, const void* w_uv_t, const void* w_o_t, int32_t B, int32_t H,
                             int32_t D, void* z, void* y, cudaStream_t stream);

/* Fig. 6 (3), with the merged weight.
 *   u       : device bf16 [B, H, 512].
 *   w_hat_t : device bf16 [D, H * 512]  row n, columns h * 512 .. h * 512 + 511, is column n of
 *             What^O_h.
 *   y       : device bf16 [B, D].
 * Same arithmetic, limits and errors as mla_value_project (one product, no intermediate). */
mla_status mla_value_project_merged(const void* u, const void* w_hat_t, int32_t B, int32_t H, int32_t D,
                                    void* y, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
