#pragma once
// decode_gather.cuh -- the tensor-core decode kernel over rows it gathers itself (included by
// decode_gather.cu and decode_shared.cu, which instantiate it for their record formats).
//
// Tensor-core absorbed MLA decode over rows the kernel gathers itself: the FP8 mixed cache
// (pages and top-k rows), bf16 top-k rows, and the shared K = V entry formats.
//
// It computes what decode_tc.cu computes ("DeepSeek's KV Cache: From 3.9 MB to 890 B per Token",
// Fig. 4 (1), Fig. 5 (2), Fig. 6 (2)) and shares its organisation: clusters of two CTAs that
// split the latent and rope dims (CTA r: latent [256 r, 256 r + 256), rope [32 r, 32 r + 32)),
// the softmax split by heads between the pair (owners finish heads [64 r, 64 r + 64), agents
// forward this CTA's partial scores of the other heads and place the P the peer sends back), the
// lazily updated running max, the balanced tile schedule and the partial merge.  What differs is
// where a tile's rows come from and how FP8 scales enter:
//   * a tile is 64 rows: the positions of one cache page (dense), or 64 consecutive entries of a
//     request's top-k list (sparse: only listed positions enter the softmax, same page, Fig. 8
//     and the DSA description on that page).  Rows outside the request (past its length, padding
//     entries, entries >= N_b) are masked and their latent rows read as zeros;
//   * raw record formats: a producer warp copies each tile's bytes of this CTA's half (a page:
//     TMA boxes; top-k rows: 16-byte cp.async pieces, one row per lane) and each is converted
//     into the MMA operand layouts, latent [64 x 256] (128-byte swizzle) and rope [64 x 32]
//     (64-byte swizzle, straight from the copy).  Two ways, one per instantiation:
//       - FP8 pages: the codes land in the conversion slot with the rope, the four group scales
//         and a 64-bit mask of valid rows once PV has released the slot, and the agent warps
//         convert them in place;
//       - FP8 top-k rows and the shared K = V formats ("converter instantiations"): the codes of
//         the next tile land in a staging buffer, and four converter warps write each piece
//         converted into the slot once PV has released it (its rope and scales land there);
//   * bf16 records (top-k only) are loaded by the agents from global memory straight into those
//     layouts;
//   * FP8 records (512 e4m3 codes, one fp32 scale per 128 dims, 64 bf16 rope dims; the 656-byte
//     layout of the same page's FP8 section) convert exactly to f16: every e4m3 value is an f16
//     value, and the MMAs of the latent dims run on f16 operands (this CTA's half of the latent
//     query is converted from bf16 to f16 in place once per request, exact for |q| in the f16
//     normal range).  The scale of each 128-dim group is applied in fp32 where the group meets
//     the other factor: on the scores, S = s_a S_a + s_b S_b + S_rope with one tensor-memory
//     accumulator per group, and on P, O_g += (P s_g) V_g for the PV of group g, with P s_g
//     rounded once to f16 (2^-11).  The running max is kept within 2^8 of every P here, so P s_g
//     stays finite for group scales below 255 (absmax below 114,000).  BF16 records take scale 1
//     and bf16 operands throughout; shared K = V entries convert exactly to bf16 with their
//     scales applied.
//
// Tensor memory (all 512 columns): O_r [0, 256), S_a [256, 320), S_b [320, 384),
// S_rope [384, 448), P_a [448, 480), P_b [480, 512) (64 16-bit values per lane in 32 columns);
// other formats two score buffers and two P buffers in [256, 512).
// Shared memory: Q half (72 KB, TMA), three conversion slots (36 KB each), the staging buffer
// (16 KB; the second exchange buffer where nothing is staged), exchange buffers.
//
// Warp roles: warps 0-3: Q loads (TMA) and the f16 conversion of Q (FP8 records: warps 0 and 3, a
// half each), the MMA issuer (+ TMEM owner), the producer; warps 4-19: thread = head = TMEM lane, four warps per 32-lane
// group, 16 positions of a tile each; the 8 warps on the owned heads' lanes run the softmax, the
// other 8 ("agents") forward partial scores, place the peer's P and finish those O rows (and
// convert FP8 pages, or load bf16 rows); warps 20-23 (converter instantiations): the converters.
// Every wait is bounded: on expiry the kernel records MLA_ERR_TIMEOUT, stops issuing, drains its
// MMAs, frees TMEM and returns.
//
// The kernel is a template over (record format, tile kind) so that each instantiation holds only
// its own paths: at 640 threads a thread has 96 registers; converter instantiations launch 768
// threads with 80 a thread and move registers from warps 0-3 and the converters to the owners and
// agents (setmaxnreg).
#include <cuda.h>
#include <cstring>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "decode_common.cuh"

namespace mla {
namespace {

using namespace ptx;
using namespace dc;

// Per-warpgroup register budget (all four warps of a warpgroup execute the same instruction):
// reg_dealloc lowers this warpgroup's registers a thread to N, returning the rest to the CTA's
// pool; reg_alloc raises them to N, waiting until the pool holds enough.
template <uint32_t N>
__device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Eight 32-bit words to global memory in one 256-bit store (the address 32-byte aligned).  A
// thread's O row goes out this way in the epilogue: each store instruction touches a line per
// thread, so halving the instructions of a row halves the lines an epilogue touches.
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

constexpr int kSegCost = 1;           // a segment start costs about one tile (schedule units)
constexpr int kNC = 3;                 // converted tile slots
constexpr int kSoftmaxThreads = 512;   // 16 warps: 8 owners + 8 agents
constexpr int kSlice = kT / 4;         // positions per warp
constexpr int kProducerWarp = 2;       // raw tile loads
constexpr int kSoftWarp0 = 4;          // warps 4-19: owners and agents
constexpr int kConvWarp0 = kSoftWarp0 + kSoftmaxThreads / 32;   // warps 20-23: conversion of raw tiles
constexpr int kConvWarps = 4;
constexpr uint32_t kBarAgents = 9;     // named barrier of the 8 agent warps (in-place conversion)
// Instantiations whose raw tiles are converted by converter warps (FP8 top-k rows and the shared
// K = V formats) rather than in place by the agents (FP8 pages; bf16 top-k rows are loaded by the
// agents): they stage each tile's codes, and add four warps.
constexpr bool gather_conv(int fmt, bool topk) { return fmt != MLA_KV_BF16 && (topk || fmt != MLA_KV_FP8_MIXED); }
constexpr int gather_threads(int fmt, bool topk) {
    return 32 * kSoftWarp0 + kSoftmaxThreads + (gather_conv(fmt, topk) ? 32 * kConvWarps : 0);
}
// Registers a thread in converter instantiations: 768 threads launch with 80 a thread; each
// warpgroup then sets its own, kRegsW0 for warps 0-3, kRegsConv for the converters and
// kRegsSoftmax for each of the four warpgroups of owners and agents, at most the launch's 6 x 80
// per sub-partition lane; all return to 80 before the common teardown.  A raise waits until other warpgroups have
// released enough: the releases come first (warps 0-3 and the converters, at the start of their
// roles) and the returns to 80 last.
constexpr int kRegsLaunch = 80;
constexpr int kRegsW0 = 64;
constexpr int kRegsConv = 64;
constexpr int kRegsSoftmax = 88;
// every warp meets here after its warpgroup's first register change, so that no warpgroup takes
// registers back (at its end) before the owners' and agents' raise has been granted
constexpr uint32_t kBarRegs = 15;
static_assert(kRegsW0 + kRegsConv + 4 * kRegsSoftmax <= 6 * kRegsLaunch, "register split above the launch's registers");
// the running max is kept until a row max exceeds it by 2^slack: 2^15 keeps P within the fp16
// range of the exchange (bf16 and shared K = V records); 2^8 keeps P s_g within f16 range for
// s_g < 255 (FP8 mixed records)
constexpr float kLazySlackBf16 = 15.0f;
constexpr float kLazySlackFp8 = 8.0f;
constexpr float kMaxGroupScale = 255.0f;   // 2^8 * 255 = 65280: P s_g stays a finite f16
constexpr int kHalfLat = 256;          // latent dims per CTA
constexpr int kHalfRope = 32;          // rope dims per CTA
constexpr int kOwned = 64;             // heads whose softmax a CTA finishes
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;         // O_r: columns [0, 256); group a [0, 128), group b [128, 256)
// Tensor memory.  bf16 and shared K = V records: two score accumulators of 64 columns (tile i uses
// i & 1) and two P buffers of 32 columns (64 16-bit values a lane), so that QK of the next tiles
// overlaps the softmax of this one.  FP8 mixed records keep the scores of their two 128-dim scale
// groups and of the rope dims apart (each group's scale multiplies its partial score in fp32,
// exactly), and P times each group's scale: one set of three accumulators and two P buffers.
constexpr uint32_t kTmemS = 256;
constexpr uint32_t kTmemP = 384;
constexpr uint32_t kTmemSa = 256;
constexpr uint32_t kTmemSb = 320;
constexpr uint32_t kTmemSr = 384;
constexpr uint32_t kTmemPa = 448;
constexpr uint32_t kTmemPb = 480;
constexpr uint32_t kDrainLimit = 1u << 20;

// shared-memory layout (bytes from a 1024-aligned base)
constexpr int kQLatChunk = 128 * 128;                  // [128 heads x 64 dims] bf16, SW128
constexpr int kQRopeBytes = 128 * 64;                  // [128 heads x 32 dims] bf16, SW64
constexpr int kKvLatChunk = kT * 128;                  // [64 rows x 64 dims], SW128
constexpr int kConvBytes = 4 * kKvLatChunk + kT * 64;  // latent + rope [64 rows x 32 dims], SW64
constexpr int kXBytes = kOwned * kT * 4;               // peer partial scores of owned heads, fp32
constexpr int kPInBytes = kOwned * kT * 2;             // peer's P of its owned heads, fp16
constexpr int kPInMsg = kPInBytes + kOwned * 4;        // + one rescale factor per head
constexpr int kOffQ = 0;
constexpr int kOffQRope = kOffQ + 4 * kQLatChunk;      // 65536
constexpr int kOffConv = kOffQRope + kQRopeBytes;      // 73728
constexpr int kScaleBytes = kT * 16;                   // per slot: [64 rows][4 groups] fp32
constexpr int kStageBytes = kT * kHalfLat;             // converter instantiations: raw codes of the next
                                                       // tile [64][256 B]; otherwise the second X buffer
constexpr int kOffStage = kOffConv + kNC * kConvBytes; // 184320
constexpr int kOffScale = kOffStage + kStageBytes;     // 200704: [kNC][64 rows][16 B]
constexpr int kOffMask = kOffScale + kNC * kScaleBytes; // 203776: [kNC][2] uint32 valid rows + staging's [2]
constexpr int kOffX = kOffMask + 32;                   // 203808: [16][64][16 B] (X buffer 0)
constexpr int kOffPIn = kOffX + kXBytes;               // 220192: [8][64][16 B] + alpha[64]
constexpr int kOffLIn = kOffPIn + kPInMsg;             // 228640: 2 x l[64] of the peer's heads
constexpr int kOffBar = kOffLIn + 2 * kOwned * 4;      // 229152
constexpr int kNumBars = 3 * kNC + 8 + 2 + 2 + 2 + 2 + 6 + 2;
constexpr int kOffRed = (kOffBar + 8 * kNumBars + 15) & ~15;   // owned heads' exchange between slices [4][64]
constexpr int kSmemBytes = kOffRed + 4 * kOwned * 4 + 1024;    // + alignment slack

constexpr uint32_t kQBytes = 4 * kQLatChunk + kQRopeBytes;     // 73728 per CTA
static_assert(kSmemBytes + 64 <= 232448, "shared memory above the 227 KB a CTA may use");

struct GatherParams {
    const uint8_t* pool;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* topk_idx;   // [B][topk] or null (dense)
    __nv_bfloat16* out;
    float* lse;
    float* o_part;             // [2C][128][512]
    float* lse_part;           // [2C][128]
    int32_t* meta;             // per request: first partial slot, last cluster (2 x int32)
    DevCtl* ctl;
    int64_t num_pages;
    int max_pages;
    int max_seq_len;
    int topk;
    int B;
    float scale_log2;          // scale * log2(e)
    const float* sink;         // shared K = V entries: per head z' ([128]) or null
    const float* rope_cs;      // shared K = V entries: per request cos, sin of 32 angles ([B][64]) or null
};

struct Bars {
    uint32_t c_full, c_empty;     // arrays of kNC
    uint32_t r_full;              // array of kNC: the slot's raw rope and scales landed
    uint32_t stage_full, stage_empty;   // the staging buffer holds the next tile's raw codes / was read
    uint32_t s_full, s_empty, p_full, p_empty;   // arrays of 2 (score and P buffers)
    uint32_t x_full, x_free;      // arrays of 2
    uint32_t pin_full, pin_free;
    uint32_t l_full;              // array of 2
    uint32_t q_full, q_ready, q_empty, o_full, o_free, mma_drain;
    __device__ __forceinline__ uint32_t cf(int i) const { return c_full + 8 * i; }
    __device__ __forceinline__ uint32_t ce(int i) const { return c_empty + 8 * i; }
    __device__ __forceinline__ uint32_t rf(int i) const { return r_full + 8 * i; }
    __device__ __forceinline__ uint32_t xf(int i) const { return x_full + 8 * i; }
    __device__ __forceinline__ uint32_t xe(int i) const { return x_free + 8 * i; }
    __device__ __forceinline__ uint32_t lf(int i) const { return l_full + 8 * i; }
    __device__ __forceinline__ uint32_t sf(int i) const { return s_full + 8 * i; }
    __device__ __forceinline__ uint32_t se(int i) const { return s_empty + 8 * i; }
    __device__ __forceinline__ uint32_t pf(int i) const { return p_full + 8 * i; }
    __device__ __forceinline__ uint32_t pe(int i) const { return p_empty + 8 * i; }
};

__device__ __forceinline__ Bars make_bars(uint32_t a) {
    Bars b;
    b.c_full = a; a += 8 * kNC;
    b.c_empty = a; a += 8 * kNC;
    b.r_full = a; a += 8 * kNC;
    b.stage_full = a; a += 8;
    b.stage_empty = a; a += 8;
    b.s_full = a; a += 16;
    b.s_empty = a; a += 16;
    b.p_full = a; a += 16;
    b.p_empty = a; a += 16;
    b.x_full = a; a += 16;
    b.x_free = a; a += 16;
    b.pin_full = a; a += 8;
    b.pin_free = a; a += 8;
    b.l_full = a; a += 16;
    b.q_full = a; a += 8;
    b.q_ready = a; a += 8;
    b.q_empty = a; a += 8;
    b.o_full = a; a += 8;
    b.o_free = a; a += 8;
    b.mma_drain = a; a += 8;
    return b;
}

// One instantiation per (record format, tile kind) in use: FP8 pages, FP8 top-k rows, bf16 top-k
// rows (dense bf16 pages take decode_tc_kernel), and pages and top-k rows of each shared K = V
// entry format, so that each holds only its own paths.
template <int kFmt, bool kTopk>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gather_threads(kFmt, kTopk), 1)
    decode_gather_kernel(const __grid_constant__ CUtensorMap tm_qlat,
                         const __grid_constant__ CUtensorMap tm_qrope,
                         const __grid_constant__ CUtensorMap tm_codes,    // pool fields as bytes
                         const __grid_constant__ CUtensorMap tm_krope,    // (FP8 mixed: boxes of 64
                         const __grid_constant__ CUtensorMap tm_scl,      // rows x 256, 64, 16 B)
                         GatherParams p) {
    constexpr bool kFp8 = kFmt == MLA_KV_FP8_MIXED;
    constexpr bool kV4 = kFmt == MLA_KV_V4_FP8;
    constexpr bool kV41 = kFmt == MLA_KV_V41_FP4;
    constexpr bool kShared = kV4 || kV41;     // K = V = the 512-dim entry; no separate rope
    constexpr bool kRaw = kFp8 || kShared;    // the producer warp stages raw record bytes
    constexpr bool kConv = gather_conv(kFmt, kTopk);   // converter warps (else in-place conversion)
    constexpr bool kQSplit = kFp8;   // warps 0 and 3 share the f16 conversion of a request's Q half
    constexpr int kNX = kConv ? 1 : 2;        // X buffers (the second one shares the staging buffer)
    // converter warps that convert: FP8 top-k rows use only the two on the agents' sub-partitions,
    // leaving the owners' to the softmax (measured faster there; the shared K = V formats, whose
    // conversion is heavier, need all four)
    constexpr int kConvActive = (kFp8 && kTopk) ? 2 : kConvWarps;
    constexpr int kCT = 32 * kConvActive;     // converting threads
    constexpr int kSB = kFp8 ? 1 : 2;         // score buffers (and P buffers)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ uint32_t s_tmem_base;
    __shared__ volatile int s_abort;
    __shared__ int s_start_b, s_start_t;
    __shared__ int s_n_local;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t r = cluster_rank();
    const uint32_t peer = r ^ 1u;
    const int c = blockIdx.x >> 1;
    const int C = gridDim.x >> 1;
    const uint32_t wait_limit = p.ctl->wait_limit;

    const uint32_t sbase = smem_u32(sm);
    const Bars bars = make_bars(sbase + kOffBar);

    if (tid == 0) {
        s_abort = 0;
        s_start_b = p.B;
        s_start_t = 0;
        s_n_local = 0;
    }
    __syncthreads();
    if (warp == 0)
        schedule_warp(p.seq_lens, p.max_seq_len, p.B, p.topk, kSegCost, c, C, c == 0 && r == 0, p.meta,
                      p.ctl, &s_n_local, &s_start_b, &s_start_t);

    if (tid == 32) {
        for (int i = 0; i < kNC; ++i) {
            // one arrive per converter warp (converter instantiations) or agent warp (FP8 pages, bf16
            // rows) once its rows are written
            mbar_init(bars.cf(i), kConv ? kConvActive : 8);
            mbar_init(bars.ce(i), 1);
            // pages: the producer's one arrival with the TMA bytes; top-k rows: one arrival per
            // producer lane once its copies land
            mbar_init(bars.rf(i), kTopk ? 32 : 1);
        }
        // the staging buffer: as rf, plus (top-k) one arrival after the mask is written; emptied
        // by one arrive per converter warp
        mbar_init(bars.stage_full, kTopk ? 33 : 1);
        mbar_init(bars.stage_empty, kConvActive);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bars.sf(i), 1);
            mbar_init(bars.se(i), kSoftmaxThreads / 32);   // one arrive per softmax warp
            mbar_init(bars.pf(i), kSoftmaxThreads / 32);
            mbar_init(bars.pe(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bars.xf(i), 1);
            mbar_init(bars.xe(i), 8);    // one remote arrive per peer owner warp
            mbar_init(bars.lf(i), 1);
        }
        mbar_init(bars.pin_full, 1);
        mbar_init(bars.pin_free, 8);     // one remote arrive per peer agent warp
        mbar_init(bars.q_full, 1);
        mbar_init(bars.q_ready, kQSplit ? 2 : 1);   // warps 0 and 3 convert a half each
        mbar_init(bars.q_empty, 1);
        mbar_init(bars.o_full, 1);
        mbar_init(bars.o_free, kSoftmaxThreads / 32);
        mbar_init(bars.mma_drain, 1);
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

    // the record of row `row` of the tile at cursor cj, or null when the row is outside the
    // request (it then reads as zeros); an out-of-pool page is recorded as MLA_ERR_BOUNDS
    // (two stages, so that several rows' index loads, then their page loads, can be in flight)
    // (V4 pages hold their entries field by field: a "record" address there only encodes the
    // slot, pool + slot * 584, from which the fields are found)
    constexpr int rec_bytes = kFp8 ? kFp8RecordBytes : kV4 ? kV4EntryBytes : kV41 ? kV41EntryBytes : kBf16RecordBytes;
    auto row_pos = [&](const Cursor& cj, int row) -> int {   // visible position of the row, or -1
        int pos = cj.t * kT + row;
        if (kTopk) pos = pos < p.topk ? __ldg(p.topk_idx + (size_t)cj.b * p.topk + pos) : -1;
        return pos >= 0 && pos < cj.n ? pos : -1;
    };
    auto page_of = [&](const Cursor& cj, int pos) -> int {
        return pos >= 0 ? __ldg(p.block_table + (size_t)cj.b * p.max_pages + (pos >> 6)) : 0;
    };
    auto record_at = [&](int pos, int page) -> const uint8_t* {
        if (pos < 0) return nullptr;
        if (page < 0 || page >= p.num_pages) {
            if (r == 0) record_error(p.ctl, MLA_ERR_BOUNDS, page);
            return nullptr;
        }
        return p.pool + ((size_t)page * kPage + (pos & (kPage - 1))) * rec_bytes;
    };
    auto pos_record = [&](const Cursor& cj, int pos) -> const uint8_t* { return record_at(pos, page_of(cj, pos)); };
    auto row_record = [&](const Cursor& cj, int row) -> const uint8_t* { return pos_record(cj, row_pos(cj, row)); };

    if (n_local == 0 && warp >= kSoftWarp0 && warp < kConvWarp0) {
        // an empty range: its partial slots must not contribute to any merge
        const int h = tid - 32 * kSoftWarp0;
        if (r == 0 && h < kHeads) {
            p.lse_part[(size_t)(2 * c) * kHeads + h] = -INFINITY;
            p.lse_part[(size_t)(2 * c + 1) * kHeads + h] = -INFINITY;
        }
    }

    if (warp < kSoftWarp0) {
        // warps 0-3: Q loads, MMA issuer, raw tile loads, and (FP8 records) the Q conversion in warps 0 and 3
        if constexpr (kConv) {
            reg_dealloc<kRegsW0>();
            named_bar_sync(kBarRegs, gather_threads(kFmt, kTopk));
        }
        if (warp == 0 || (kQSplit && warp == 3)) {
            // ------------------------------------------------------------------ Q loads (TMA) + f16
            // Warp 0 loads a request's Q half by TMA.  FP8 records: once it has landed, warps 0 and 3
            // (two sub-partitions) convert its latent part from bf16 to f16 in place, half each (the
            // swizzle permutes whole 16-byte chunks, so each chunk keeps its place), and release it to
            // the MMA issuer.  Warp 0 then prefetches the next segment's Q half into L2.
            const bool qlead = warp == 0;
            Cursor cu;
            if (qlead && lane == 0 && n_local > 0) {
                tma_prefetch_desc(&tm_qlat);
                if (!kShared) tma_prefetch_desc(&tm_qrope);
            }
            cu.init(p.seq_lens, p.max_seq_len, p.topk, start_b, start_t, n_local);
            int seg = 0;
            for (int i = 0; i < n_local; ++i, cu.next(p.seq_lens, p.max_seq_len, p.B, p.topk)) {
                if (!cu.first()) continue;
                bool ok = !s_abort;
                if (qlead && ok && seg > 0) ok = mbar_wait(bars.q_empty, (seg - 1) & 1, wait_limit);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    if (lane == 0) fail(p.ctl, &s_abort, 1);
                    break;
                }
                if (qlead && lane == 0) {
                    const int qrow = cu.b * kHeads;
                    mbar_arrive_expect_tx(bars.q_full, kShared ? 4 * kQLatChunk : kQBytes);
                    for (int k = 0; k < 4; ++k)
                        tma_load_2d(sbase + kOffQ + k * kQLatChunk, &tm_qlat, bars.q_full,
                                    (int)r * kHalfLat + 64 * k, qrow);
                    if (!kShared) tma_load_2d(sbase + kOffQRope, &tm_qrope, bars.q_full, (int)r * kHalfRope, qrow);
                }
                // warp 3 waits for the whole segment: sleeping polls leave its sub-partition's issue
                // slots to the softmax warps there
                ok = __all_sync(0xffffffffu, qlead ? mbar_wait(bars.q_full, seg & 1, wait_limit)
                                                   : mbar_wait_sleep(bars.q_full, seg & 1, wait_limit, 256));
                if (!ok) {
                    if (lane == 0) fail(p.ctl, &s_abort, 19);
                    break;
                }
                if (kFp8) {
                    // an element that overflows f16 (|q| >= 65520) is outside this path's range.  bf16
                    // holds nothing in [65504, 65536), so that is a magnitude field of 0x4780 or more,
                    // which (field + 0x3880) marks in bit 15 (two fields a word, no carry between
                    // them; infinities and NaNs included)
                    uint32_t big = 0;
    #pragma unroll 8
                    for (int u = lane + (qlead ? 0 : 32); u < 4 * kQLatChunk / 16; u += kQSplit ? 64 : 32) {
                        uint4* q = reinterpret_cast<uint4*>(sm + kOffQ) + u;
                        const uint4 v = *q;
                        big |= ((v.x & 0x7FFF7FFFu) + 0x38803880u) | ((v.y & 0x7FFF7FFFu) + 0x38803880u) |
                               ((v.z & 0x7FFF7FFFu) + 0x38803880u) | ((v.w & 0x7FFF7FFFu) + 0x38803880u);
                        *q = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                                        bf16x2_to_f16x2(v.w));
                    }
                    fence_proxy_async_smem();
                    if (__any_sync(0xffffffffu, (big & 0x80008000u) != 0) && lane == 0)
                        record_error(p.ctl, MLA_ERR_RANGE, cu.b);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.q_ready);
                if (qlead && lane == 0 && i + (cu.nt - cu.t) < n_local) {
                    // the range goes on with the next request that has tiles: its Q half into L2
                    int b = cu.b + 1;
                    while (b + 1 < p.B && tiles_of(clamp_len(p.seq_lens[b], p.max_seq_len), p.topk) == 0) ++b;
                    for (int k = 0; k < 4; ++k) tma_prefetch_l2_2d(&tm_qlat, (int)r * kHalfLat + 64 * k, b * kHeads);
                    if (!kShared) tma_prefetch_l2_2d(&tm_qrope, (int)r * kHalfRope, b * kHeads);
                }
                ++seg;
            }
            // drain: the last Q load lands before this CTA may exit
            if (qlead && lane == 0 && seg > 0) mbar_wait(bars.q_full, (seg - 1) & 1, kDrainLimit);
            __syncwarp();
        } else if (warp == 1) {
            // ------------------------------------------------------------------ MMA issuer
            // The whole warp runs this loop so that its operands stay warp-uniform; one elected lane
            // issues each MMA and commit.  QK of a tile: 8 MMAs per latent group into that group's
            // accumulator (f16 operands for FP8 records), 2 rope MMAs (bf16); PV: per group, 4 MMAs
            // of 128x128x16 with P times the group's scales from tensor memory.  One score set and
            // one P set in tensor memory: QK of tile i + 1 follows the softmax's reads of tile i's
            // scores, P of tile i + 1 follows PV of tile i.
            if (n_local > 0) {
                constexpr uint32_t id_qk = kFp8 ? idesc_f16(128, kT, 0, 0) : idesc_bf16(128, kT, 0, 0);
                constexpr uint32_t id_qr = idesc_bf16(128, kT, 0, 0);
                constexpr uint32_t id_pv = kFp8 ? idesc_f16(128, 128, 0, 1) : idesc_bf16(128, 128, 0, 1);
                const uint64_t lat_hi = smem_desc(0, 16, 1024, kSw128) & 0xFFFFFFFF00000000ull;
                const uint64_t rope_hi = smem_desc(0, 16, 512, kSw64) & 0xFFFFFFFF00000000ull;
                const uint64_t v_hi = smem_desc(0, kKvLatChunk, 1024, kSw128) & 0xFFFFFFFF00000000ull;
                const uint32_t lat_lo = (uint32_t)smem_desc(0, 16, 1024, kSw128);
                const uint32_t rope_lo = (uint32_t)smem_desc(0, 16, 512, kSw64);
                const uint32_t v_lo = (uint32_t)smem_desc(0, kKvLatChunk, 1024, kSw128);
                const uint32_t ql_lo = lat_lo + (((sbase + kOffQ) >> 4) & 0x3FFF);
                const uint32_t qr_lo = rope_lo + (((sbase + kOffQRope) >> 4) & 0x3FFF);
                Cursor cq, cp;
                cq.init(p.seq_lens, p.max_seq_len, p.topk, start_b, start_t, n_local);
                cp = cq;
                int iq = 0, ip = 0, seg_q = 0, seg_p = 0;
                uint32_t polls = 0;
                while (ip < n_local && !__any_sync(0xffffffffu, s_abort)) {
                    if (iq < n_local && iq <= ip + kSB) {   // QK up to kSB tiles ahead of PV (its score buffers)
                        const int s = iq % kNC;
                        const int sb = iq % kSB;
                        const bool ready = __shfl_sync(
                            0xffffffffu,
                            (!cq.first() || mbar_test(bars.q_ready, seg_q & 1)) &&
                                mbar_test(bars.cf(s), (iq / kNC) & 1) &&
                                mbar_test(bars.se(sb), ((iq / kSB) & 1) ^ 1),
                            0);
                        if (ready) {
                            tc_fence_after();
                            const uint32_t st_lo = ((sbase + kOffConv + s * kConvBytes) >> 4) & 0x3FFF;
                            if (elect_one()) {
                                // FP8 records: one accumulator per scale group and one for the rope
                                // dims; otherwise everything into score buffer sb
                                const uint32_t sacc = tmem + kTmemS + 64 * sb;
    #pragma unroll
                                for (int k = 0; k < 4; ++k)
    #pragma unroll
                                    for (int kk = 0; kk < 4; ++kk)
                                        mma_bf16_ss(kFp8 ? tmem + (k < 2 ? kTmemSa : kTmemSb) : sacc,
                                                    lat_hi | (ql_lo + ((k * kQLatChunk + kk * 32) >> 4)),
                                                    lat_hi | (st_lo + lat_lo + ((k * kKvLatChunk + kk * 32) >> 4)),
                                                    id_qk, (kFp8 ? ((k & 1) | kk) : (k | kk)) != 0 ? 1u : 0u);
                                if (!kShared) {
    #pragma unroll
                                    for (int kk = 0; kk < 2; ++kk)
                                        mma_bf16_ss(kFp8 ? tmem + kTmemSr : sacc, rope_hi | (qr_lo + kk * 2),
                                                    rope_hi | (st_lo + rope_lo + ((4 * kKvLatChunk + kk * 32) >> 4)),
                                                    id_qr, (kFp8 && kk == 0) ? 0u : 1u);
                                }
                                mma_commit(bars.sf(sb));
                                if (cq.last()) mma_commit(bars.q_empty);
                            }
                            __syncwarp();
                            if (cq.last()) ++seg_q;
                            cq.next(p.seq_lens, p.max_seq_len, p.B, p.topk);
                            ++iq;
                            polls = 0;
                            continue;
                        }
                    }
                    const bool seg_first = cp.first();
                    const bool pv_ready = __shfl_sync(
                        0xffffffffu,
                        (!seg_first || seg_p == 0 || mbar_test(bars.o_free, (seg_p - 1) & 1)) &&
                            mbar_test(bars.pf(ip % kSB), (ip / kSB) & 1),
                        0);
                    if (!pv_ready) {
                        if (++polls > wait_limit) {
                            if (lane == 0) fail(p.ctl, &s_abort, 6);
                            break;
                        }
                        continue;
                    }
                    polls = 0;
                    tc_fence_after();
                    const uint32_t v = ((sbase + kOffConv + (ip % kNC) * kConvBytes) >> 4) & 0x3FFF;
                    if (elect_one()) {
    #pragma unroll
                        for (int g = 0; g < 2; ++g)
    #pragma unroll
                            for (int kk = 0; kk < kT / 16; ++kk) {
                                const uint64_t vd = v_hi | (v + v_lo + ((2 * g * kKvLatChunk + kk * 16 * 128) >> 4));
                                mma_bf16_ts(tmem + kTmemO + 128 * g,
                                            tmem + (kFp8 ? (g == 0 ? kTmemPa : kTmemPb) : kTmemP + 32 * (ip % kSB)) + 8 * kk,
                                            vd, id_pv, (!seg_first || kk > 0) ? 1u : 0u);
                            }
                        mma_commit(bars.pe(ip % kSB));
                        mma_commit(bars.ce(ip % kNC));
                        if (cp.last()) mma_commit(bars.o_full);
                    }
                    __syncwarp();
                    if (cp.last()) ++seg_p;
                    cp.next(p.seq_lens, p.max_seq_len, p.B, p.topk);
                    ++ip;
                }
            }
            __syncwarp();
        } else if (warp == kProducerWarp) {
            // ------------------------------------------------------------------ FP8 tile loads
            // Tile j's raw bytes into conversion slot j % kNC once PV of tile j - kNC has released it,
            // with the mask of valid rows (written before the arrival the agents wait on).  A dense
            // tile is one page: three TMA boxes of its 64 rows (rows past the request's end are
            // loaded and then zeroed by the agents).  A top-k tile: each lane copies its two rows with
            // 16-byte cp.async (21 pieces per row: 16 of codes, the scales, 4 of rope) and arrives
            // once they have landed.  Pages: the next tile's rows are looked up after a tile is
            // issued, and the page kPfAhead tiles ahead is prefetched into L2.  Top-k rows: index
            // loads, page loads and records run as a three-stage pipeline (see below), and each
            // tile's rows are prefetched into L2 one tile ahead of their copies.
            if (kRaw && n_local > 0) {
                constexpr int kPfAhead = 3;
                constexpr bool dense = !kTopk;
                if (dense && lane == 0) {
                    tma_prefetch_desc(&tm_codes);
                    tma_prefetch_desc(&tm_krope);
                    tma_prefetch_desc(&tm_scl);
                }
                Cursor cj, cpf;   // the next tile to load, and (dense) the next tile to prefetch into L2
                cj.init(p.seq_lens, p.max_seq_len, p.topk, start_b, start_t, n_local);
                cpf = cj;
                int j_pf = 0;
                // L2 prefetch of the rows of the records given (dense: lane 0 holds the page's row 0)
                auto prefetch = [&](const uint8_t* f0, const uint8_t* f1) {
                    if (dense) {
                        if (f0) {
                            const int y = (int)((f0 - p.pool) / rec_bytes);   // slot of the page's row 0
                            if (kFp8) {
                                tma_prefetch_l2_2d(&tm_codes, kHalfLat * (int)r, y);
                                tma_prefetch_l2_2d(&tm_krope, kFp8RopeOff + 2 * kHalfRope * (int)r, y);
                                tma_prefetch_l2_2d(&tm_scl, kFp8ScaleOff, y);
                            } else if (kV4) {
                                tma_prefetch_l2_3d(&tm_codes, kHalfLat * (int)r, 0, y / kPage);
                                if (r == 1) tma_prefetch_l2_3d(&tm_krope, 0, 0, y / kPage);
                                prefetch_l2(p.pool + (size_t)(y / kPage) * kV4PageBytes + kV4ScaleOff, kPage * 8);
                            } else {
                                tma_prefetch_l2_2d(&tm_codes, 128 * (int)r, y);
                                tma_prefetch_l2_2d(&tm_scl, kV41ScaleOff + 16 * (int)r, y);
                            }
                        }
                    } else {
                        // the lines of the row's codes half and of its scales and rope
                        const uint8_t* pq[2] = {f0, f1};
    #pragma unroll
                        for (int q = 0; q < 2; ++q)
                            if (pq[q]) {
                                if (kFp8) {
                                    prefetch_line_l2(pq[q] + kHalfLat * (int)r);
                                    prefetch_line_l2(pq[q] + kHalfLat * (int)r + 128);
                                    prefetch_line_l2(pq[q] + kFp8ScaleOff);
                                    prefetch_line_l2(pq[q] + kFp8RecordBytes - 16);
                                } else if (kV4) {
                                    const size_t sl = (size_t)(pq[q] - p.pool) / kV4EntryBytes;
                                    const uint8_t* base = p.pool + (sl / kPage) * kV4PageBytes;
                                    const int row = (int)(sl % kPage);
                                    prefetch_l2(base + row * kENope + kHalfLat * (int)r, r == 0 ? 256 : 192);
                                    if (r == 1) prefetch_l2(base + kV4RopeOff + row * 128, 128);
                                    prefetch_line_l2(base + kV4ScaleOff + row * 8);
                                } else {
                                    prefetch_l2(pq[q] + 128 * (int)r, 128);
                                    prefetch_line_l2(pq[q] + kV41ScaleOff + 16 * (int)r);
                                }
                            }
                    }
                };
                // Dense tiles: at the start of each iteration the page of tile j_pf (looked up by lane 0
                // the iteration before) is prefetched and the page of the next tile to prefetch looked
                // up; after a tile is issued, rows lane, lane + 32 of the next one are looked up.
                const uint8_t* rec0 = nullptr;
                const uint8_t* rec1 = nullptr;
                const uint8_t* pf_page = nullptr;
                auto prefetch_dense = [&]() {
                    prefetch(pf_page, nullptr);
                    pf_page = nullptr;
                    if (j_pf < n_local) {
                        if (lane == 0) pf_page = row_record(cpf, 0);
                        ++j_pf;
                        cpf.next(p.seq_lens, p.max_seq_len, p.B, p.topk);
                    }
                };
                // Top-k tiles: a three-stage pipeline in which every load is consumed one iteration
                // after it is issued: index loads of tile j + 3, page loads of tile j + 2, records of
                // tile j + 1 (whose rows are then prefetched into L2), run after tile j is issued.
                Cursor cB = cj, cA = cj;   // the tiles of the page and index stages
                int jB = 0, jA = 0;
                int ia0 = -1, ia1 = -1;    // index stage results (raw list entries)
                int pb0 = -1, pb1 = -1, gb0 = 0, gb1 = 0;   // page stage results: positions, pages
                auto stage_a = [&]() {
                    ia0 = ia1 = -1;
                    if (jA < n_local) {
                        const int e0 = cA.t * kT + lane, e1 = e0 + 32;
                        const size_t base = (size_t)cA.b * p.topk;
                        ia0 = e0 < p.topk ? __ldg(p.topk_idx + base + e0) : -1;
                        ia1 = e1 < p.topk ? __ldg(p.topk_idx + base + e1) : -1;
                    }
                };
                auto stage_b = [&]() {   // consumes the index stage of the same tile, then advances it
                    pb0 = pb1 = -1;
                    if (jB < n_local) {
                        pb0 = ia0 >= 0 && ia0 < cB.n ? ia0 : -1;
                        pb1 = ia1 >= 0 && ia1 < cB.n ? ia1 : -1;
                        gb0 = page_of(cB, pb0);
                        gb1 = page_of(cB, pb1);
                        ++jB;
                        cB.next(p.seq_lens, p.max_seq_len, p.B, p.topk);
                    }
                    if (jA < n_local) {
                        ++jA;
                        cA.next(p.seq_lens, p.max_seq_len, p.B, p.topk);
                    }
                    stage_a();
                };
                auto lookups_topk = [&](bool load_next) {   // records of the tile the page stage holds
                    rec0 = load_next ? record_at(pb0, gb0) : nullptr;
                    rec1 = load_next ? record_at(pb1, gb1) : nullptr;
                    prefetch(rec0, rec1);
                    stage_b();
                };
                if (dense) {
                    for (int k = 0; k < kPfAhead; ++k) prefetch_dense();
                    rec0 = row_record(cj, lane);
                    rec1 = row_record(cj, lane + 32);
                } else {
                    stage_a();    // tile 0
                    stage_b();    // tile 0 pages, tile 1 indices
                    lookups_topk(true);
                }
                int issued = 0, staged = 0;
                const uint32_t stage = sbase + kOffStage;
                constexpr int stage_row = kV41 ? 128 : kHalfLat;   // bytes of a row's codes in the staging buffer
                for (int j = 0; j < n_local; ++j) {
                    if (dense) prefetch_dense();
                    const int slot = j % kNC;
                    const uint32_t m0 = __ballot_sync(0xffffffffu, rec0 != nullptr);
                    const uint32_t m1 = __ballot_sync(0xffffffffu, rec1 != nullptr);
                    // (a) converter instantiations: tile j's codes into the staging buffer once the
                    // converters have read tile j - 1's, with the mask of valid rows (written before the
                    // arrival the converters wait on)
                    bool ok = !s_abort;
                    if (kConv && ok && j >= 1) ok = mbar_wait(bars.stage_empty, (j - 1) & 1, wait_limit);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) {
                        if (lane == 0) fail(p.ctl, &s_abort, 20);
                        break;
                    }
                    if (kConv && lane == 0) {
                        uint32_t* mk = reinterpret_cast<uint32_t*>(sm + kOffMask) + 2 * kNC;
                        mk[0] = m0;
                        mk[1] = m1;
                        if (dense) {
                            if (m0 & 1u) {   // row 0 of a dense tile is visible unless its page is not
                                const int y = (int)((rec0 - p.pool) / rec_bytes);
                                mbar_arrive_expect_tx(bars.stage_full, kT * stage_row);
                                if (kFp8) tma_load_2d(stage, &tm_codes, bars.stage_full, kHalfLat * (int)r, y);
                                // V4: codes [64 x 256 B] of this half (CTA 1: dims 448.. read as zeros)
                                else if (kV4) tma_load_3d(stage, &tm_codes, bars.stage_full, kHalfLat * (int)r, 0, y / kPage);
                                else tma_load_2d(stage, &tm_codes, bars.stage_full, 128 * (int)r, y);
                            } else {
                                mbar_arrive(bars.stage_full);
                            }
                        }
                    }
                    // top-k rows: each lane copies its rows' 16-byte pieces starting at piece `lane`, so
                    // that the 32 lanes of one copy instruction write different banks
                    auto copy_codes = [&](const uint8_t* rec, int row) {
                        if (!rec) return;
                        if (kFp8) {
                            const uint8_t* cs = rec + kHalfLat * (int)r;
    #pragma unroll
                            for (int k = 0; k < kHalfLat / 16; ++k) {
                                const int q = (k + lane) & (kHalfLat / 16 - 1);
                                cp_async16(stage + row * kHalfLat + 16 * q, cs + 16 * q);
                            }
                        } else if (kV4) {
                            // codes of this half (CTA 1: its 192; the rest of the row is never read)
                            const size_t sl = (size_t)(rec - p.pool) / kV4EntryBytes;
                            const uint8_t* cs = p.pool + (sl / kPage) * kV4PageBytes + (int)(sl % kPage) * kENope + kHalfLat * (int)r;
                            const int pieces = r == 0 ? 16 : 12;
    #pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                if (k >= pieces) break;
                                const int q = (k + lane) % pieces;
                                cp_async16(stage + row * kHalfLat + 16 * q, cs + 16 * q);
                            }
                        } else {
                            const uint8_t* cs = rec + 128 * (int)r;
    #pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const int q = (k + lane) & 7;
                                cp_async16(stage + row * 128 + 16 * q, cs + 16 * q);
                            }
                        }
                    };
                    if (kConv && !dense) {
                        copy_codes(rec0, lane);
                        copy_codes(rec1, lane + 32);
                        cp_async_arrive_noinc(bars.stage_full);
                        if (lane == 0) mbar_arrive(bars.stage_full);
                    }
                    if (kConv) ++staged;
                    // (b) the tile's rope (FP8 mixed: straight into its 64-byte-swizzled operand; V4:
                    // CTA 1's RoPE dims into operand chunk 3) and scales into slot j % kNC once PV of tile
                    // j - kNC has released it; FP8 pages (converted in place) also take their codes there,
                    // and the mask of valid rows
                    if (ok && j >= kNC) ok = mbar_wait(bars.ce(slot), ((j / kNC) - 1) & 1, wait_limit);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) {
                        if (lane == 0) fail(p.ctl, &s_abort, 21);
                        break;
                    }
                    const uint32_t dst = sbase + kOffConv + slot * kConvBytes;
                    const uint32_t dst_rope = dst + 4 * kKvLatChunk;
                    const uint32_t dst_scl = sbase + kOffScale + slot * kScaleBytes;
                    const uint32_t bar = bars.rf(slot);
                    if (dense && lane == 0) {
                        if (!kConv) {
                            uint32_t* mk = reinterpret_cast<uint32_t*>(sm + kOffMask) + 2 * slot;
                            mk[0] = m0;
                            mk[1] = m1;
                        }
                        if (m0 & 1u) {
                            const int y = (int)((rec0 - p.pool) / rec_bytes);
                            if (kFp8) {
                                mbar_arrive_expect_tx(bar, kT * ((kConv ? 0 : kHalfLat) + 2 * kHalfRope + 16));
                                if (!kConv) tma_load_2d(dst, &tm_codes, bar, kHalfLat * (int)r, y);
                                tma_load_2d(dst_rope, &tm_krope, bar, kFp8RopeOff + 2 * kHalfRope * (int)r, y);
                                tma_load_2d(dst_scl, &tm_scl, bar, kFp8ScaleOff, y);
                            } else if (kV4) {
                                const int z = y / kPage;
                                mbar_arrive_expect_tx(bar, (r == 1 ? kT * 128 : 0) + kT * 8);
                                if (r == 1) tma_load_3d(dst + 3 * kKvLatChunk, &tm_krope, bar, 0, 0, z);
                                bulk_load(dst_scl, p.pool + (size_t)z * kV4PageBytes + kV4ScaleOff, kT * 8, bar);
                            } else {
                                mbar_arrive_expect_tx(bar, kT * 16);
                                tma_load_2d(dst_scl, &tm_scl, bar, kV41ScaleOff + 16 * (int)r, y);
                            }
                        } else {
                            mbar_arrive(bar);
                        }
                    }
                    if (!dense) {
                        auto copy_side = [&](const uint8_t* rec, int row) {
                            if (!rec) return;
                            if (kFp8) {
                                cp_async16(dst_scl + row * 16, rec + kFp8ScaleOff);
                                const uint8_t* rs = rec + kFp8RopeOff + 2 * kHalfRope * (int)r;
    #pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const int q = (k + lane) & 3;
                                    cp_async16(dst_rope + row * 64 + ((q ^ ((row >> 1) & 3)) << 4), rs + 16 * q);
                                }
                            } else if (kV4) {
                                const size_t sl = (size_t)(rec - p.pool) / kV4EntryBytes;
                                const uint8_t* base = p.pool + (sl / kPage) * kV4PageBytes;
                                const int prow = (int)(sl % kPage);
                                if (r == 1) {
                                    const uint8_t* rs = base + kV4RopeOff + prow * 128;
    #pragma unroll
                                    for (int k = 0; k < 8; ++k) {
                                        const int q = (k + lane) & 7;
                                        cp_async16(dst + 3 * kKvLatChunk + row * 128 + ((q ^ (row & 7)) << 4), rs + 16 * q);
                                    }
                                }
                                cp_async8(dst_scl + row * 8, base + kV4ScaleOff + prow * 8);
                            } else {
                                cp_async16(dst_scl + row * 16, rec + kV41ScaleOff + 16 * (int)r);
                            }
                        };
                        copy_side(rec0, lane);
                        copy_side(rec1, lane + 32);
                        cp_async_arrive_noinc(bar);
                    }
                    __syncwarp();
                    ++issued;
                    cj.next(p.seq_lens, p.max_seq_len, p.B, p.topk);
                    if (dense) {
                        rec0 = rec1 = nullptr;
                        if (j + 1 < n_local) {
                            rec0 = row_record(cj, lane);
                            rec1 = row_record(cj, lane + 32);
                        }
                    } else {
                        lookups_topk(j + 1 < n_local);
                    }
                }
                // drain: the copies of the last tiles (one per slot, and the staging buffer's) land
                // before this CTA may exit
                if (dense) {
                    if (lane == 0) {
                        for (int j = issued - 1; j >= 0 && j >= issued - kNC; --j)
                            mbar_wait(bars.rf(j % kNC), (j / kNC) & 1, kDrainLimit);
                        if (staged > 0) mbar_wait(bars.stage_full, (staged - 1) & 1, kDrainLimit);
                    }
                } else {
                    cp_async_wait_all();
                }
            }
            __syncwarp();
        }
        __syncwarp();
        if constexpr (kConv) reg_alloc<kRegsLaunch>();
    } else if (warp >= kConvWarp0) {
        // ------------------------------------------------------------------ converters
        // Tile j: once its codes have landed in the staging buffer, PV of tile j - kNC has freed
        // slot j % kNC and the slot's rope and scales have landed, each 16-byte piece of codes is
        // read and written converted into the MMA operand layout: latent chunks [64 rows x 64 dims]
        // (128-byte swizzle), zeros for rows outside the request; the staging buffer is then
        // released for tile j + 1.  FP8 mixed: E4M3 to f16 (exact); V4: E4M3 times 2^(UE8M0 - 127)
        // to bf16 (exact), CTA 1's RoPE dims already in place (zeroed for rows outside); V4.1: E2M1
        // times the E4M3 scale of its 16 dims to bf16 (exact).
        if constexpr (kConv) {
            reg_dealloc<kRegsConv>();
            named_bar_sync(kBarRegs, gather_threads(kFmt, kTopk));
        }
        const int cw = warp - kConvWarp0;   // this converter's sub-partition
        const bool converts = kConvActive == kConvWarps || (cw >> 1) == (int)(1u - r);
        if (kConv && n_local > 0 && converts) {
            const int ct = (kConvActive == kConvWarps ? cw : (cw & 1)) * 32 + lane;   // 0 .. kCT - 1
            Cursor cc;
            cc.init(p.seq_lens, p.max_seq_len, p.topk, start_b, start_t, n_local);
            for (int j = 0; j < n_local; ++j, cc.next(p.seq_lens, p.max_seq_len, p.B, p.topk)) {
                const int slot = j % kNC;
                bool ok = !s_abort && mbar_wait(bars.stage_full, j & 1, wait_limit);
                ok = ok && (j < kNC || mbar_wait(bars.ce(slot), ((j / kNC) - 1) & 1, wait_limit));
                ok = ok && mbar_wait(bars.rf(slot), (j / kNC) & 1, wait_limit);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    if (lane == 0) fail(p.ctl, &s_abort, 22);
                    break;
                }
                const uint32_t* smk = reinterpret_cast<const uint32_t*>(sm + kOffMask) + 2 * kNC;
                const uint32_t mk0 = smk[0], mk1 = smk[1];
                auto valid = [&](int row) -> bool { return ((row < 32 ? mk0 : mk1) >> (row & 31)) & 1u; };
                uint8_t* lat = sm + kOffConv + slot * kConvBytes;
                const uint8_t* scl = sm + kOffScale + slot * kScaleBytes;
                const uint8_t* stg = sm + kOffStage;
                // piece e = ct + kCT k: FP8 mixed and V4 [64 rows][16 x 16 B] (row e >> 4, dims 16 ch ..
                // 16 ch + 15 of this half, ch = e & 15 = ct & 15); V4.1 [64 rows][8 x 16 B] (row e >> 3,
                // dims 32 ch .. 32 ch + 31, ch = ct & 7)
                if (!kV41) {
                    const int ch = ct & 15;
                    const bool rope_piece = kV4 && r == 1 && ch >= 12;   // V4, CTA 1: dims 448 .. 511
                    const int s0 = 2 * (ch & 3);
#pragma unroll 2
                    for (int k = 0; k < 1024 / kCT; ++k) {
                        const int row = (ct + kCT * k) >> 4;
                        uint8_t* dst = lat + (ch >> 2) * kKvLatChunk + row * 128;
                        if (rope_piece && valid(row)) continue;
                        uint32_t o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                        if (valid(row) && !rope_piece) {
                            const uint4 raw = *reinterpret_cast<const uint4*>(stg + (ct + kCT * k) * 16);
                            if (kFp8) {
                                e4m3x16_to_f16(raw, o);
                            } else {
                                const uint32_t byte = scl[row * 8 + 4 * (int)r + (ch >> 2)];
                                e4m3x16_scaled_bf16(raw, __uint_as_float(byte ? byte << 23 : 0x00400000u), o);   // 2^(byte - 127)
                            }
                        }
                        st_shared_v4(dst + ((s0 ^ (row & 7)) << 4), o[0], o[1], o[2], o[3]);
                        st_shared_v4(dst + (((s0 + 1) ^ (row & 7)) << 4), o[4], o[5], o[6], o[7]);
                    }
                } else {
                    const int ch = ct & 7;
#pragma unroll 1
                    for (int k = 0; k < 512 / kCT; ++k) {
                        const int row = (ct + kCT * k) >> 3;
                        uint32_t o[16];
#pragma unroll
                        for (int t = 0; t < 16; ++t) o[t] = 0;
                        if (valid(row))
                            e2m1x32_scaled_bf16(*reinterpret_cast<const uint4*>(stg + (ct + kCT * k) * 16),
                                                e4m3_to_float(scl[row * 16 + 2 * ch]),
                                                e4m3_to_float(scl[row * 16 + 2 * ch + 1]), o);
                        uint8_t* dst = lat + (ch >> 1) * kKvLatChunk + row * 128;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int part = 4 * (ch & 1) + q;
                            st_shared_v4(dst + ((part ^ (row & 7)) << 4), o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                        }
                    }
                }
                // every piece of the staging buffer read: it may take tile j + 1
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.stage_empty);
                if (kFp8 && ct < kT) {
                    // scales of rows outside the request: zero (their P is zero); a visible row whose
                    // group scale is above 255 (or not finite) would overflow f16(P s_g)
                    uint4* sc = reinterpret_cast<uint4*>(sm + kOffScale + slot * kScaleBytes + ct * 16);
                    if (!valid(ct)) {
                        *sc = make_uint4(0, 0, 0, 0);
                    } else {
                        const uint4 q = *sc;   // (a NaN fails every comparison)
                        if (!(__uint_as_float(q.x) <= kMaxGroupScale) || !(__uint_as_float(q.y) <= kMaxGroupScale) ||
                            !(__uint_as_float(q.z) <= kMaxGroupScale) || !(__uint_as_float(q.w) <= kMaxGroupScale))
                            record_error(p.ctl, MLA_ERR_RANGE, cc.b);
                    }
                }
                if (ct == 0) {
                    uint32_t* mk = reinterpret_cast<uint32_t*>(sm + kOffMask) + 2 * slot;
                    mk[0] = mk0;
                    mk[1] = mk1;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.cf(slot));
            }
        }
        __syncwarp();
        if constexpr (kConv) reg_alloc<kRegsLaunch>();
    } else {
        // ------------------------------------------------------------------ owners and agents
        // Lane group lg = warp % 4 (the TMEM lanes this warp may access: heads 32 lg .. 32 lg + 31,
        // thread = head), slice ts = (warp - 4) / 4 (positions 16 ts .. 16 ts + 15 of a tile, and
        // O columns 64 ts .. 64 ts + 63 in corrections and epilogues).  Lane groups 2r, 2r + 1
        // hold the owned heads.
        //
        // The four owner warps of a lane group meet at named barriers (ids 1 + lg, 5 + lg, 128
        // threads), which cannot time out, so these loops never leave early: after a failed
        // (bounded) wait they keep executing every barrier but skip the work, and waits return at
        // once.  Wait results are made warp-uniform before any warp-collective tcgen05 instruction.
        if constexpr (kConv) {
            reg_alloc<kRegsSoftmax>();
            named_bar_sync(kBarRegs, gather_threads(kFmt, kTopk));
        }
        const int lg = warp & 3;
        const int ts = (warp - kSoftWarp0) >> 2;
        const int h = lg * 32 + lane;
        const bool owner = (lg >> 1) == (int)r;
        const int hh = h & (kOwned - 1);   // index among the owning CTA's heads
        const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
        float* red = reinterpret_cast<float*>(sm + kOffRed);   // [4 slices][64 owned heads]

        auto wwait = [&](uint32_t bar, uint32_t parity, int where) -> bool {
            bool ok = !s_abort && mbar_wait(bar, parity, wait_limit);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0) fail(p.ctl, &s_abort, where);
            return ok;
        };

        // group scales of the warp's 16 positions of tile i (FP8 records): element 2 t is (s_a, s_b)
        // of position 16 ts + t (each row holds the scales of all four groups)
        auto scales_of = [&](int i) -> const float2* {
            return reinterpret_cast<const float2*>(sm + kOffScale + (i % kNC) * kScaleBytes) + 32 * ts + (int)r;
        };

        // this CTA's partial scores of tile i for the warp's 16 positions: score buffer i % kSB, or
        // for FP8 records s_a S_a + s_b S_b + S_rope (the tile's scales and mask, written with its
        // slot, are read once the slot is complete)
        auto load_s = [&](int i, float (&v)[16]) -> bool {
            if (!wwait(bars.cf(i % kNC), (i / kNC) & 1, 18)) return false;
            if (!wwait(bars.sf(i % kSB), (i / kSB) & 1, 7)) return false;
            tc_fence_after();
            if (kFp8) {
                const float2* sc = scales_of(i);
                uint32_t a[16], b[16];
                tmem_ld16(tmem + lane_off + kTmemSa + kSlice * ts, a);
                tmem_ld16(tmem + lane_off + kTmemSb + kSlice * ts, b);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const float2 q = sc[2 * t];
                    v[t] = fmaf(q.x, __uint_as_float(a[t]), q.y * __uint_as_float(b[t]));
                }
                uint32_t e[16];
                tmem_ld16(tmem + lane_off + kTmemSr + kSlice * ts, e);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 16; ++t) v[t] += __uint_as_float(e[t]);
            } else {
                uint32_t a[16];
                tmem_ld16(tmem + lane_off + kTmemS + 64 * (i % kSB) + kSlice * ts, a);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 16; ++t) v[t] = __uint_as_float(a[t]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.se(i % kSB));
            return true;
        };

        // O rows of this warp (its 64 columns) times alpha, once PV of tile i - 1 has completed
        auto rescale_o = [&](int i, float alpha) {
            if (!wwait(bars.pe((i - 1) % kSB), ((i - 1) / kSB) & 1, 10)) return;
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                const uint32_t col = kTmemO + 64 * ts + 32 * cc;
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + col, o);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                tmem_st32(tmem + lane_off + col, o);
            }
            tmem_wait_st();
        };

        // the warp's 16 P values of tile i (fp16 pairs from the softmax) into tensor memory, once
        // PV of tile i - kSB (the last reader of that P buffer) has completed, then P ready for the
        // MMA: f16 (P s_g) per scale group for FP8 records, bf16 P otherwise
        auto store_p = [&](int i, const uint32_t (&pk)[8]) {
            if (i >= kSB && !wwait(bars.pe(i % kSB), ((i / kSB) & 1) ^ 1, 11)) return;
            if (kFp8) {
                uint32_t pa[8], pb[8];
                const float2* sc = scales_of(i);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 q0 = sc[4 * k], q1 = sc[4 * k + 2];
                    __half2 h2;
                    *reinterpret_cast<uint32_t*>(&h2) = pk[k];
                    const float2 pf = __half22float2(h2);
                    pa[k] = pack_f16x2(pf.x * q0.x, pf.y * q1.x);
                    pb[k] = pack_f16x2(pf.x * q0.y, pf.y * q1.y);
                }
                tmem_st8(tmem + lane_off + kTmemPa + 8 * ts, pa);
                tmem_st8(tmem + lane_off + kTmemPb + 8 * ts, pb);
            } else {
                uint32_t pa[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    __half2 h2;
                    *reinterpret_cast<uint32_t*>(&h2) = pk[k];
                    const float2 pf = __half22float2(h2);
                    pa[k] = pack_bf16x2(pf.x, pf.y);
                }
                tmem_st8(tmem + lane_off + kTmemP + 32 * (i % kSB) + 8 * ts, pa);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && !s_abort) mbar_arrive(bars.pf(i % kSB));
        };

        // O rows of this warp normalised by l (row sum) into the output or a partial slot
        auto epilogue_rows = [&](int seg, const Cursor& cu, bool partial, float l_row) {
            const int slot = 2 * c + (seg == 0 ? 0 : 1);
            if (!wwait(bars.o_full, seg & 1, 12)) return;
            tc_fence_after();
            const float inv = l_row > 0.f ? 1.0f / l_row : 0.0f;
            const size_t row = (size_t)cu.b * kHeads + h;
            const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + kTmemO + 64 * ts + 32 * cc, o);
                tmem_wait_ld();
                const int col = (int)r * kHalfLat + 64 * ts + 32 * cc;
                if (kShared && r == 1 && ts == 3 && p.rope_cs != nullptr) {
                    // dims 448 .. 511 carry RoPE: rotate the pairs (448 + 2i, 448 + 2i + 1), i = 16 cc
                    // + k, back by the query position's angle (a partial too: the merge is linear)
                    const float* cs = p.rope_cs + (size_t)cu.b * 64 + 16 * cc;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float cv = __ldg(cs + k), sv = __ldg(cs + 32 + k);
                        const float x0 = __uint_as_float(o[2 * k]), x1 = __uint_as_float(o[2 * k + 1]);
                        o[2 * k] = __float_as_uint(x0 * cv + x1 * sv);
                        o[2 * k + 1] = __float_as_uint(x1 * cv - x0 * sv);
                    }
                }
                if (!partial) {
                    // 32 bf16 (64 bytes at a 64-byte offset in the row): 256-bit stores when the
                    // output is 32-byte aligned (the interface promises 16)
                    uint32_t w[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        w[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv);
                    uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + row * kDc + col);
                    if (out32) {
                        st_global_v8(dst, reinterpret_cast<const uint32_t(&)[8]>(w[0]));
                        st_global_v8(dst + 8, reinterpret_cast<const uint32_t(&)[8]>(w[8]));
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            reinterpret_cast<uint4*>(dst)[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                    }
                } else {
                    // 32 fp32 (128 bytes at a 128-byte offset in a partial slot of the 256-byte
                    // aligned workspace)
                    uint32_t* dst = reinterpret_cast<uint32_t*>(p.o_part + ((size_t)slot * kHeads + h) * kDc + col);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(__uint_as_float(o[8 * k + e]) * inv);
                        st_global_v8(dst + 8 * k, w);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.o_free);
        };

        Cursor cu;
        cu.init(p.seq_lens, p.max_seq_len, p.topk, start_b, start_t, n_local);
        int seg = 0;
        bool cut_front = false;

        // Tile preparation by the agents (converter instantiations have their tiles prepared by the
        // converter warps): thread `at` of the 256 agent threads puts tile j (cursor cj) into
        // conversion slot j % kNC, this CTA's half of every row in the MMA layouts with zeros for
        // rows outside the request: FP8 pages converted in place from the raw bytes the producer
        // warp loaded there; bf16 top-k rows loaded from global memory once PV of tile j - kNC has
        // freed the slot, with the mask of valid rows.
        const int at = ((lg & 1) * 4 + ts) * 32 + lane;
        auto prepare = [&](int j, const Cursor& cj) {
            const int slot = j % kNC;
            uint8_t* lat = sm + kOffConv + slot * kConvBytes;
            uint8_t* rope = lat + 4 * kKvLatChunk;
            const uint4 zero = make_uint4(0, 0, 0, 0);
            if (kFp8 && !kConv) {
                // FP8 pages: the producer warp has put the raw codes [64][256] at the slot's start
                // (the rope dims, already in their operand layout, the scales and the mask of valid
                // rows beside them); each agent thread reads its 16-byte pieces, all agents meet, and
                // each writes its pieces converted (zeros for rows outside the request)
                const bool ok = wwait(bars.rf(slot), (j / kNC) & 1, 17);
                const uint32_t* mk = reinterpret_cast<const uint32_t*>(sm + kOffMask) + 2 * slot;
                const uint32_t mk0 = mk[0], mk1 = mk[1];
                auto valid = [&](int row) -> bool { return ((row < 32 ? mk0 : mk1) >> (row & 31)) & 1u; };
                uint4 raw[4];
                if (ok) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) raw[k] = *reinterpret_cast<const uint4*>(lat + (at + 256 * k) * 16);
                }
                named_bar_sync(kBarAgents, kSoftmaxThreads / 2);   // every raw piece read
                if (ok) {
                    // 64 rows x 16 chunks of 16 codes; piece at + 256 k is chunk ch of row `row`
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int e = at + 256 * k, row = e >> 4, ch = e & 15;
                        uint32_t o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                        if (valid(row)) e4m3x16_to_f16(raw[k], o);
                        // dims 16 ch .. 16 ch + 15 of this half: 64-dim chunk ch / 4, 16-byte parts
                        // 2 (ch % 4) and 2 (ch % 4) + 1 of the row, 128-byte swizzle
                        uint8_t* dst = lat + (ch >> 2) * kKvLatChunk + row * 128;
                        const int s0 = 2 * (ch & 3);
                        st_shared_v4(dst + ((s0 ^ (row & 7)) << 4), o[0], o[1], o[2], o[3]);
                        st_shared_v4(dst + (((s0 + 1) ^ (row & 7)) << 4), o[4], o[5], o[6], o[7]);
                    }
                    // scales of rows outside the request: zero (their P is zero); a visible row
                    // whose group scale is above 255 (or not finite) would overflow f16(P s_g)
                    if (at < kT) {
                        uint4* sc = reinterpret_cast<uint4*>(sm + kOffScale + slot * kScaleBytes + at * 16);
                        if (!valid(at)) {
                            *sc = zero;
                        } else {
                            const uint4 q = *sc;   // (a NaN fails every comparison)
                            if (!(__uint_as_float(q.x) <= kMaxGroupScale) || !(__uint_as_float(q.y) <= kMaxGroupScale) ||
                                !(__uint_as_float(q.z) <= kMaxGroupScale) || !(__uint_as_float(q.w) <= kMaxGroupScale))
                                record_error(p.ctl, MLA_ERR_RANGE, cj.b);
                        }
                    }
                }
            } else if (!kRaw) {
                // 64 rows x 32 chunks of 8 bf16 dims; this thread copies chunks at + 256 k
                // (the first half loaded before the wait)
                const int rope_off = 2 * kDc + 2 * kHalfRope * (int)r;
                const uint8_t* rrec = row_record(cj, at >> 2);
                const uint4 rraw = rrec ? __ldg(reinterpret_cast<const uint4*>(rrec + rope_off + 16 * (at & 3))) : zero;
                const uint8_t* srec = at < kT ? row_record(cj, at) : nullptr;
                uint4 raw[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int e = at + 256 * k, row = e >> 5, ch = e & 31;
                    const uint8_t* rec = row_record(cj, row);
                    raw[k] = rec ? __ldg(reinterpret_cast<const uint4*>(rec + 2 * kHalfLat * (int)r + 16 * ch)) : zero;
                }
                if (j >= kNC && !wwait(bars.ce(slot), ((j / kNC) - 1) & 1, 17)) return;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (half == 1) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int e = at + 256 * (4 + k), row = e >> 5, ch = e & 31;
                            const uint8_t* rec = row_record(cj, row);
                            raw[k] = rec ? __ldg(reinterpret_cast<const uint4*>(rec + 2 * kHalfLat * (int)r + 16 * ch)) : zero;
                        }
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int e = at + 256 * (4 * half + k), row = e >> 5, ch = e & 31;
                        st_shared_v4(lat + (ch >> 3) * kKvLatChunk + row * 128 + (((ch & 7) ^ (row & 7)) << 4),
                                     raw[k].x, raw[k].y, raw[k].z, raw[k].w);
                    }
                }
                {
                    // rope: 64 rows x 4 chunks of 8 dims, 64-byte swizzle
                    const int row = at >> 2, c4 = at & 3;
                    st_shared_v4(rope + row * 64 + ((c4 ^ ((row >> 1) & 3)) << 4), rraw.x, rraw.y, rraw.z, rraw.w);
                }
                if (at < kT) {
                    // the valid-row mask
                    const uint32_t m = __ballot_sync(0xffffffffu, srec != nullptr);
                    if (lane == 0) reinterpret_cast<uint32_t*>(sm + kOffMask)[2 * slot + (at >> 5)] = m;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.cf(slot));
        };

        Cursor cpr = cu;   // next tile to prepare
        int i_pr = 0;
        auto prepare_until = [&](int upto) {
            for (; i_pr < upto && i_pr < n_local; ++i_pr, cpr.next(p.seq_lens, p.max_seq_len, p.B, p.topk)) prepare(i_pr, cpr);
        };
        // bf16 records: L2 prefetch of the rows of tile i + 5 during iteration i (tile i + 2 is
        // prepared in iteration i, so prefetches run three iterations ahead): thread `at` covers
        // part at / 64 (latent bytes, rope) of row at % 64.  Its address comes from the index
        // loads of the iteration before, so their latency overlaps an iteration.  (FP8 tiles are
        // prefetched by warp 18.)
        const int pf_row = at & (kT - 1), pf_part = at >> 6;
        const uint32_t pf_bytes = pf_part == 0 ? (kFp8 ? kHalfLat : 2 * kHalfLat) : (pf_part == 1 ? 64 : 16);
        const int pf_off = pf_part == 0 ? (kFp8 ? kHalfLat : 2 * kHalfLat) * (int)r
                                        : (pf_part == 1 ? (kFp8 ? kFp8RopeOff : 2 * kDc) + 64 * (int)r : kFp8ScaleOff);
        const bool pf_on = !kRaw && pf_part < 2;   // FP8 and shared entries: the producer warp prefetches
        Cursor cpf = cu;   // the tile whose prefetch address is computed next (tiles 0, 1 are
        int i_pf = 0;      // prepared at once)
        for (; i_pf < 2 && i_pf < n_local; ++i_pf) cpf.next(p.seq_lens, p.max_seq_len, p.B, p.topk);
        const uint8_t* pf_rec = nullptr;
        auto prefetch_step = [&]() {
            if (pf_rec) prefetch_l2(pf_rec + pf_off, pf_bytes);
            pf_rec = nullptr;
            if (i_pf < n_local) {
                if (pf_on) pf_rec = row_record(cpf, pf_row);
                ++i_pf;
                cpf.next(p.seq_lens, p.max_seq_len, p.B, p.topk);
            }
        };
        if (!owner) {
            // ------------------------------------------------------------ agents
            const uint32_t x_remote = mapa(sbase + kOffX, peer);
            const uint32_t x1_remote = mapa(sbase + kOffStage, peer);
            const uint32_t xfull_remote = mapa(bars.x_full, peer);
            const uint32_t pinfree_remote = mapa(bars.pin_free, peer);
            const bool lead = (ts == 0 && lg == 2 * (int)peer && lane == 0);

            // forward this CTA's partial scores of tile i (the peer's heads) to the peer
            auto forward = [&](int i) {
                float v[16];
                if (!load_s(i, v)) return;
                // buffer i % kNX (converter instantiations have one: the staging buffer takes the
                // second) once the peer's owners have read the scores it held
                const int xb = i % kNX;
                if (!wwait(bars.xe(xb), ((i / kNX) & 1) ^ 1, 8)) return;
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    st_async_v4((xb == 0 ? x_remote : x1_remote) + ((4 * ts + g) * kOwned + hh) * 16, xfull_remote + 8 * xb, __float_as_uint(v[4 * g]), __float_as_uint(v[4 * g + 1]),
                                __float_as_uint(v[4 * g + 2]), __float_as_uint(v[4 * g + 3]));
            };

            if (!kConv) {
                for (int k = 0; k < 4; ++k) prefetch_step();   // tiles 2, 3, 4 prefetched, 5 addressed
                prepare_until(2);
            }
            if (n_local > 0) forward(0);
            // Iteration i: converter instantiations send this CTA's scores of tile i + 1 to the
            // peer as soon as QK of tile i + 1 has completed (it does not wait for P of tile i),
            // then place the peer's P of tile i in tensor memory (PV of tile i can then go).  The
            // others place P of tile i first, then send the scores of tile i + 1, then prepare tile
            // i + 2.
            for (int i = 0; i < n_local; ++i, cu.next(p.seq_lens, p.max_seq_len, p.B, p.topk)) {
                if (kConv && i + 1 < n_local) forward(i + 1);
                const bool first = cu.first();
                if (first) cut_front = cu.t > 0;
                // the peer's P of its heads for tile i, and its rescale factors
                if (lead && !s_abort) mbar_arrive_expect_tx(bars.pin_full, kPInMsg);
                const bool ok = wwait(bars.pin_full, i & 1, 13);
                uint32_t pk[8];
                const uint8_t* pin = sm + kOffPIn;
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const uint4 q = *reinterpret_cast<const uint4*>(pin + ((2 * ts + g) * kOwned + hh) * 16);
                    pk[4 * g] = q.x;
                    pk[4 * g + 1] = q.y;
                    pk[4 * g + 2] = q.z;
                    pk[4 * g + 3] = q.w;
                }
                const float alpha = reinterpret_cast<const float*>(pin + kPInBytes)[hh];
                __syncwarp();
                if (lane == 0 && ok) mbar_arrive_remote_relaxed(pinfree_remote);
                if (!first && __any_sync(0xffffffffu, ok && alpha != 1.0f)) rescale_o(i, alpha);
                store_p(i, pk);
                if (cu.last()) {
                    const bool partial = cut_front || cu.t < cu.nt - 1;
                    // the row sums of these heads, sent by the peer's owners
                    if (lead && !s_abort) mbar_arrive_expect_tx(bars.lf(seg & 1), kOwned * 4);
                    const bool lok = wwait(bars.lf(seg & 1), (seg >> 1) & 1, 14);
                    const float l_row = lok ? reinterpret_cast<const float*>(sm + kOffLIn)[(seg & 1) * kOwned + hh] : 0.f;
                    epilogue_rows(seg, cu, partial, l_row);
                    ++seg;
                }
                if (!kConv) {
                    if (i + 1 < n_local) forward(i + 1);
                    prepare_until(i + 3);
                    prefetch_step();
                }
            }
        } else {
            // ------------------------------------------------------------ owners
            const uint32_t pin_remote = mapa(sbase + kOffPIn, peer);
            const uint32_t pinfull_remote = mapa(bars.pin_full, peer);
            const uint32_t xfree_remote = mapa(bars.x_free, peer);
            const uint32_t lin_remote = mapa(sbase + kOffLIn, peer);
            const uint32_t lfull_remote = mapa(bars.l_full, peer);
            const bool lead = (ts == 0 && lg == 2 * (int)r && lane == 0);
            const uint32_t bar_vote = 1 + lg, bar_sync = 5 + lg;
            constexpr float slack = kFp8 ? kLazySlackFp8 : kLazySlackBf16;
            const float p_max = exp2f(slack);
            // l_part sums the P values PV multiplies (it normalises O); lx_part the unrounded ones
            // (it gives the log-sum-exp); they differ only for bf16 P
            float m_used = -INFINITY, l_part = 0.f, lx_part = 0.f;
            for (int i = 0; i < n_local; ++i, cu.next(p.seq_lens, p.max_seq_len, p.B, p.topk)) {
                const bool first = cu.first();
                if (first) {
                    m_used = -INFINITY;
                    l_part = 0.f;
                    lx_part = 0.f;
                    cut_front = cu.t > 0;   // the request started before this cluster's range
                }
                float v[16];
                load_s(i, v);
                // valid rows of this warp's 16 positions
                const uint32_t vmask =
                    (reinterpret_cast<const uint32_t*>(sm + kOffMask)[2 * (i % kNC) + (ts >> 1)] >> (16 * (ts & 1))) & 0xFFFFu;
                // the peer's partial scores of these heads for tile i
                const int xb = i % kNX;
                if (lead && !s_abort) mbar_arrive_expect_tx(bars.xf(xb), kXBytes);
                const bool xok = wwait(bars.xf(xb), (i / kNX) & 1, 9);
                float x[16];
                const uint8_t* xp = sm + (xb == 0 ? kOffX : kOffStage);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float4 q = *reinterpret_cast<const float4*>(xp + ((4 * ts + g) * kOwned + hh) * 16);
                    x[4 * g] = (v[4 * g] + q.x) * p.scale_log2;
                    x[4 * g + 1] = (v[4 * g + 1] + q.y) * p.scale_log2;
                    x[4 * g + 2] = (v[4 * g + 2] + q.z) * p.scale_log2;
                    x[4 * g + 3] = (v[4 * g + 3] + q.w) * p.scale_log2;
                }
                // every loaded value has been consumed: hand the exchange buffer back to the peer
                __syncwarp();
                if (lane == 0 && xok) mbar_arrive_remote_relaxed(xfree_remote + 8 * xb);
                // P = 2^(x - m) with the running max m (rows outside the request give 0).  m is
                // kept while every P of a row stays at most 2^slack: a thread whose 16 P sum past
                // 2^slack (or not to a finite value) votes for the rare path, as does every segment
                // start and a row with no visible position yet.  There the exact row max over the
                // four slices raises m where it exceeds m by more than the slack, O is rescaled
                // here and, through alpha sent with P, in the peer, and P is computed again.
                float alpha = 1.0f;
                float psum, pxsum;
                uint32_t pk[8];
                auto exp_tile = [&]() {
                    psum = 0.f;
                    pxsum = 0.f;
#pragma unroll
                    for (int t = 0; t < 16; t += 2) {
                        const bool live = m_used != -INFINITY;
                        float p0 = (live && ((vmask >> t) & 1)) ? ex2(x[t] - m_used) : 0.f;
                        float p1 = (live && ((vmask >> (t + 1)) & 1)) ? ex2(x[t + 1] - m_used) : 0.f;
                        pxsum += p0 + p1;
                        if (!kFp8) {
                            // bf16 P: the row sum adds the values PV multiplies (each bf16 value,
                            // at most 2^15, travels exactly as fp16), so the weights sum to one
                            p0 = __bfloat162float(__float2bfloat16_rn(p0));
                            p1 = __bfloat162float(__float2bfloat16_rn(p1));
                        }
                        psum += p0 + p1;
                        const __half2 h2 = __floats2half2_rn(p0, p1);
                        pk[t / 2] = *reinterpret_cast<const uint32_t*>(&h2);
                    }
                };
                exp_tile();
                const bool need = first || m_used == -INFINITY || !(psum <= p_max);
                if (bar_red_or(bar_vote, 128, need)) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if ((vmask >> t) & 1) mx = fmaxf(mx, x[t]);
                    red[ts * kOwned + hh] = mx;
                    named_bar_sync(bar_sync, 128);
                    const float tmax = fmaxf(fmaxf(red[hh], red[kOwned + hh]), fmaxf(red[2 * kOwned + hh], red[3 * kOwned + hh]));
                    const bool grow = first || tmax > m_used + slack;
                    const float m_new = grow ? (first ? tmax : fmaxf(tmax, m_used)) : m_used;
                    if (!first) {
                        alpha = grow ? ex2(m_used - m_new) : 1.0f;
                        if (__any_sync(0xffffffffu, grow)) rescale_o(i, alpha);
                        l_part *= alpha;
                        lx_part *= alpha;
                    }
                    m_used = m_new;
                    named_bar_sync(bar_sync, 128);   // red[] rows of this lane group are free again
                    exp_tile();
                }
                l_part += psum;
                lx_part += pxsum;
                // P of these heads (fp16, before the group scales) to the peer, once it has taken
                // the previous one; both CTAs apply their group scales to these values
                if (wwait(bars.pin_free, (i & 1) ^ 1, 15)) {
#pragma unroll
                    for (int g = 0; g < 2; ++g)
                        st_async_v4(pin_remote + ((2 * ts + g) * kOwned + hh) * 16, pinfull_remote,
                                    pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
                    if (ts == 0)
                        st_async_b32(pin_remote + kPInBytes + hh * 4, pinfull_remote, __float_as_uint(alpha));
                }
                store_p(i, pk);

                if (cu.last()) {
                    // ------------------------------------------------------ segment epilogue
                    const bool partial = cut_front || cu.t < cu.nt - 1;
                    red[ts * kOwned + hh] = l_part;
                    named_bar_sync(bar_sync, 128);
                    const float l_row = (red[hh] + red[kOwned + hh]) + (red[2 * kOwned + hh] + red[3 * kOwned + hh]);
                    named_bar_sync(bar_sync, 128);
                    float lx_row = l_row;
                    if (!kFp8) {
                        red[ts * kOwned + hh] = lx_part;
                        named_bar_sync(bar_sync, 128);
                        lx_row = (red[hh] + red[kOwned + hh]) + (red[2 * kOwned + hh] + red[3 * kOwned + hh]);
                        named_bar_sync(bar_sync, 128);
                    }
                    // shared K = V entries with a sink, request finished here: exp(z') joins the
                    // denominator, 2^(z' log2 e - m) in the units of l (the merge adds it otherwise)
                    float l_fin = l_row;
                    float L = lx_row > 0.f ? (m_used + log2f(lx_row)) * 0.6931471805599453f : -INFINITY;
                    if (kShared && p.sink != nullptr && !partial) {
                        const float zl = __ldg(p.sink + h);
                        if (l_row > 0.f) {
                            const float a = m_used + log2f(lx_row), z2 = zl * 1.4426950408889634f;
                            const float hi = fmaxf(a, z2), lo = fminf(a, z2);
                            L = (hi + log2f(1.0f + exp2f(lo - hi))) * 0.6931471805599453f;
                            l_fin = l_row + exp2f(z2 - m_used);   // inf when the sink dominates: O / inf = 0
                        } else {
                            L = zl;
                        }
                    }
                    // the row sums of these heads to the peer, which finishes its O rows of them
                    if (ts == 0 && !s_abort)
                        st_async_b32(lin_remote + ((seg & 1) * kOwned + hh) * 4,
                                     lfull_remote + 8 * (seg & 1), __float_as_uint(l_fin));
                    if (ts == 0) {
                        const size_t row = (size_t)cu.b * kHeads + h;
                        if (!partial) p.lse[row] = L;
                        else p.lse_part[(size_t)(2 * c + (seg == 0 ? 0 : 1)) * kHeads + h] = L;
                    }
                    epilogue_rows(seg, cu, partial, l_fin);
                    ++seg;
                }
            }
        }
        __syncwarp();
        if constexpr (kConv) reg_dealloc<kRegsLaunch>();
    }

    // ---------------------------------------------------------------------- teardown
    if (warp == 1 && n_local > 0) {
        __syncwarp();
        // all MMAs issued by the elected lane (the lowest active one, as in the loop) are complete
        // once this barrier flips
        if (elect_one()) {
            mma_commit(bars.mma_drain);
            if (!mbar_wait(bars.mma_drain, 0, kDrainLimit)) record_error(p.ctl, MLA_ERR_TIMEOUT, 16);
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


// One launch of instantiation <kFmt, kTopk>: tensor maps of the queries and (pages) of the pool's
// fields, the kernel over plan.splits clusters, then the merge of the requests cut by cluster ranges.
template <int kFmt, bool kTopk>
cudaError_t launch_gather_instance(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t st) {
    auto* kernel = decode_gather_kernel<kFmt, kTopk>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        if (gather_conv(kFmt, kTopk)) {
            // the warpgroups' register split adds up to 80 a thread at launch: a build that launches
            // with fewer would leave a reg_alloc waiting forever, so it is refused here
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, kernel);
            if (e != cudaSuccess) return e;
            if (fa.numRegs < kRegsLaunch) return cudaErrorInvalidConfiguration;
        }
        attr_set[dev] = true;
    }
    constexpr bool shared = kFmt == MLA_KV_V4_FP8 || kFmt == MLA_KV_V41_FP4;
    CUtensorMap tm_qlat, tm_qrope, tm_codes, tm_krope, tm_scl;
    const uint64_t qrows = (uint64_t)a.B * kHeads;
    if (!encode_2d(&tm_qlat, a.q_lat, kDc, qrows, kDc * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (shared) {
        std::memset(&tm_qrope, 0, sizeof(tm_qrope));
    } else if (!encode_2d(&tm_qrope, a.q_rope, kDr, qrows, kDr * 2, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B)) {
        return cudaErrorInvalidValue;
    }
    std::memset(&tm_codes, 0, sizeof(tm_codes));
    std::memset(&tm_krope, 0, sizeof(tm_krope));
    std::memset(&tm_scl, 0, sizeof(tm_scl));
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t rows = (uint64_t)a.num_pages * kPage;
    if (kFmt == MLA_KV_FP8_MIXED && !kTopk) {
        // the pool as rows of 656 bytes; a box is 64 rows (one page) of a record's byte range (the
        // rope box lands in its operand layout, 64-byte swizzle)
        if (!encode_2d(&tm_codes, a.pool, kFp8RecordBytes, rows, kFp8RecordBytes, kHalfLat, kT,
                       CU_TENSOR_MAP_SWIZZLE_NONE, u8) ||
            !encode_2d(&tm_krope, a.pool, kFp8RecordBytes, rows, kFp8RecordBytes, 2 * kHalfRope, kT,
                       CU_TENSOR_MAP_SWIZZLE_64B, u8) ||
            !encode_2d(&tm_scl, a.pool, kFp8RecordBytes, rows, kFp8RecordBytes, 16, kT,
                       CU_TENSOR_MAP_SWIZZLE_NONE, u8))
            return cudaErrorInvalidValue;
    } else if (kFmt == MLA_KV_V4_FP8 && !kTopk) {
        // page z: codes [64 rows][448 B] (a box of 256 B, read past 448 as zeros), RoPE [64][128 B]
        // into the 128-byte-swizzled operand layout
        const uint64_t np = (uint64_t)(a.num_pages > 0 ? a.num_pages : 1);
        const uint64_t cd[3] = {(uint64_t)kENope, (uint64_t)kPage, np};
        const uint64_t cs[2] = {(uint64_t)kENope, (uint64_t)kV4PageBytes};
        const uint32_t cb[3] = {(uint32_t)kHalfLat, (uint32_t)kT, 1u};
        const uint64_t rd[3] = {128u, (uint64_t)kPage, np};
        const uint64_t rs[2] = {128u, (uint64_t)kV4PageBytes};
        const uint32_t rb[3] = {128u, (uint32_t)kT, 1u};
        if (!encode_3d(&tm_codes, a.pool, cd, cs, cb, CU_TENSOR_MAP_SWIZZLE_NONE, u8) ||
            !encode_3d(&tm_krope, a.pool + kV4RopeOff, rd, rs, rb, CU_TENSOR_MAP_SWIZZLE_128B, u8))
            return cudaErrorInvalidValue;
    } else if (kFmt == MLA_KV_V41_FP4 && !kTopk) {
        // the pool as rows of 288 bytes: codes [64 x 128 B] and scales [64 x 16 B] of this half
        if (!encode_2d(&tm_codes, a.pool, kV41EntryBytes, rows, kV41EntryBytes, 128, kT,
                       CU_TENSOR_MAP_SWIZZLE_NONE, u8) ||
            !encode_2d(&tm_scl, a.pool, kV41EntryBytes, rows, kV41EntryBytes, 16, kT,
                       CU_TENSOR_MAP_SWIZZLE_NONE, u8))
            return cudaErrorInvalidValue;
    }
    const int C = plan.splits;
    float* o_part = static_cast<float*>(a.workspace);
    float* lse_part = o_part + (size_t)2 * C * kHeads * kDc;
    int32_t* meta = reinterpret_cast<int32_t*>(lse_part + (size_t)2 * C * kHeads);
    GatherParams p;
    p.pool = a.pool;
    p.block_table = a.block_table;
    p.seq_lens = a.seq_lens;
    p.topk_idx = a.topk > 0 ? a.topk_idx : nullptr;
    p.out = a.out;
    p.lse = a.lse;
    p.o_part = o_part;
    p.lse_part = lse_part;
    p.meta = meta;
    p.ctl = a.ctl;
    p.num_pages = a.num_pages;
    p.max_pages = a.max_pages;
    p.max_seq_len = a.max_seq_len;
    p.topk = a.topk_idx != nullptr ? a.topk : 0;
    p.B = a.B;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.sink = shared ? a.sink : nullptr;
    p.rope_cs = shared ? a.rope_cs : nullptr;
    kernel<<<2 * C, gather_threads(kFmt, kTopk), kSmemBytes, st>>>(tm_qlat, tm_qrope, tm_codes, tm_krope, tm_scl, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_merge_slots(o_part, lse_part, meta, a.out, a.lse, a.B, C, st, p.sink);
}

}  // namespace
}  // namespace mla
