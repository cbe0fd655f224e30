// decode.cuh -- MLA decode over the paged latent cache, absorbed form, on a CTA pair.
//
// What it computes (page 1, "撕開 DeepSeek MLA 源碼", sections 1, 3, 4): for every work item
// (sequence b, page range) and all 128 heads h,
//   s[h,t] = (q_abs[b,h] . c_KV[t] + q_R[b,h] . k_R[t]) * softmax_scale
// with an online softmax over t, and the latent output o[h] = sum_t p[h,t] c_KV[t] (512-d).
// All heads share the cache row, so per 64-token page QK is a dense [128 x 576] x [576 x 64]
// contraction and PV a dense [128 x 64] x [64 x 512] one: both run on tcgen05.
//
// Why two CTAs.  The fp32 accumulator O[128 x 512] takes all 512 columns of one SM's tensor
// memory, and the scores need 64 more; the bf16 query [128 x 576] is 144 KB.  So a cluster of
// two CTAs on two SMs splits the work by role instead of recomputing anything:
//   rank 0, the score CTA: q_abs lives in TMEM (256 columns, the A operand of "TS" MMAs) and
//     q_R in shared memory (16 KB); the scores of two pages at a time go to one of two
//     128-column TMEM buffers (one N=128 MMA covers both pages, which halves the MMA count:
//     a tcgen05.mma costs about the same to issue at N=64 as at N=128).  Pages stream through
//     a ring of K-chunks (one 64-column box of both pages, 16 KB).  Four warps run the softmax,
//     write P (bf16, 16 KB per page) into local shared memory, and ship it to the value CTA
//     with asynchronous bulk copies that complete the peer's barrier by byte count.
//   rank 1, the value CTA: O lives in TMEM (512 columns); per page it runs PV from P and its
//     own copy of the page's 512 latent columns; four warps apply the (rare) rescales, zero
//     the unused slots of a sequence's last page, and write the normalised output.
// Both CTAs stream the same pages with their own TMA ring; the score CTA reads first with
// normal L2 priority and the value CTA second with evict-first, so HBM sees each page once.
//
// Online softmax with lazy rescaling: the running max m used for exp2 only moves when a tile's
// max exceeds it by more than 8 (log2 units); then l and O are scaled by exp2(m_old - m_new).
// P values stay <= 2^8, and the final division by l makes the result exact whatever m is.
//
// Pipelines (all waits bounded; see ptx.cuh):
//   kv_full/kv_empty[S]   TMA rings: 10 K-chunk stages in the score CTA, 3 page stages in the
//                         value CTA
//   s_full/s_free[2]      two-page score buffers (score CTA)
//   q_ready               query loaded into TMEM for an item (score CTA)
//   msg_full[2]           P + per-row statistics landed in the value CTA (bulk copies; armed
//                         by the value CTA's MMA thread)
//   msg_free[2]           PV using that P finished (value CTA's MMA commit, multicast to rank 0)
//                         and the value CTA's four correction warps have read the statistics
//   o_drain[2]            every PV issued before a flagged tile has finished (value CTA's MMA
//                         commit right before it waits o_ready)
//   o_ready[2]            value CTA's correction warps finished a flagged tile (rescale O, zero
//                         a tail, or write the previous item's output before the next item's
//                         first PV overwrites O)
#pragma once
#include "plan.h"
#include "ptx.cuh"

namespace mla {
namespace decode {

constexpr int kThreads = 192;
constexpr int kChunkStages = 10;
constexpr int kValueStages = 3;
constexpr int kMaxStages = 10;
constexpr int kBoxBytes = 64 * 128;               // 64 tokens x 64 bf16 columns
constexpr int kBoxesPerRow = 9;                   // c_KV: 8 boxes, k_R: 1 box
constexpr int kGroupPages = 2;                    // pages per score MMA (N = 128)
constexpr int kChunkBytes = kGroupPages * kBoxBytes;  // one box column of a two-page group
constexpr int kValueStageBytes = 8 * kBoxBytes;   // 65,536: c_KV only
constexpr int kPBytes = 128 * 128;                // P: 128 heads x 64 tokens bf16
// Per message statistics, one 272-byte block per softmax warp (32 heads): factor[32] (rescale
// of those O rows), inv_l[32] (1/l, last tile of an item), then a 16-byte flags slot (bit 0:
// one of the rows rescales, bit 1: the page has slots past the sequence end).  Each warp ships
// its 4 KB slice of P and its block with its own bulk copies.
constexpr int kStatsWarpBytes = 128 + 128 + 16;
constexpr int kStatsBytes = 4 * kStatsWarpBytes;
constexpr int kPWarpBytes = kPBytes / 4;
constexpr int kMsgBytes = kPBytes + kStatsBytes;
// score CTA: q_R (K-major, 128-byte swizzle), the K-chunk ring, two local P staging buffers
constexpr int kOffQR = 0;
constexpr int kOffChunks = kOffQR + 128 * 128;
constexpr int kOffScoreStaging = kOffChunks + kChunkStages * kChunkBytes;
// value CTA: stages, then two P buffers (1024-aligned, the MMA reads them)
constexpr int kOffP = kValueStages * kValueStageBytes;
// both CTAs: statistics (staging in the score CTA, destination in the value CTA)
constexpr int kOffStats = kOffP + 2 * kPBytes;
constexpr int kOffBars = kOffStats + 2 * kStatsBytes;

enum Bar : int {
    kFull0 = 0,
    kEmpty0 = kFull0 + kMaxStages,
    kSFull0 = kEmpty0 + kMaxStages,
    kSFree0 = kSFull0 + 2,
    kQReady = kSFree0 + 2,
    kMsgFree0 = kQReady + 1,
    kMsgFull0 = kMsgFree0 + 2,
    kOReady0 = kMsgFull0 + 2,
    kODrain0 = kOReady0 + 2,
    kDrain = kODrain0 + 2,
    kNumBars = kDrain + 1
};

constexpr int kOffTmemHolder = kOffBars + 8 * kNumBars;
constexpr int kOffAbort = kOffTmemHolder + 4;
constexpr int kSmemBytes = ((kOffAbort + 4 + 127) / 128) * 128;
static_assert(kOffScoreStaging + 2 * kPBytes <= kOffStats, "score staging overlaps the statistics");
static_assert(kChunkStages <= kMaxStages && kValueStages <= kMaxStages, "barrier slots per ring");
static_assert(kOffBars % 8 == 0, "barriers need 8-byte alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kStatsWarpBytes % 16 == 0 && kPWarpBytes % 16 == 0, "bulk copies move multiples of 16 bytes");

// TMEM columns
constexpr uint32_t kQCol = 0;      // score CTA: q_abs, 256 columns (512 bf16 per lane)
constexpr uint32_t kSCol = 256;    // score CTA: two 128-column score buffers (two pages each)
constexpr uint32_t kTmemCols = 512;

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8

// Wait-cycle accounting for performance work, compiled only with MLA_DECODE_TRACE: each role
// adds the SM cycles it spends in each wait to a local array and writes it to
// trace[blockIdx.x * kTraceSlots + slot] at the end.  Normal builds compile it away.
constexpr int kTraceSlots = 16;
#ifdef MLA_DECODE_TRACE
#define MLA_TIMED(slot, expr)                              \
    ([&]() {                                               \
        const long long t0_ = clock64();                   \
        const auto r_ = (expr);                            \
        tr_[(slot)] += clock64() - t0_;                    \
        return r_;                                         \
    }())
#define MLA_TRACE_DECL long long tr_[kTraceSlots] = {0}; const long long tstart_ = clock64()
#define MLA_TRACE_ADD(slot, v) (tr_[(slot)] += (v))
#define MLA_TRACE_NOW() clock64()
#define MLA_TRACE_FLUSH(first, last, total_slot)                                                    \
    do {                                                                                            \
        tr_[(total_slot)] = clock64() - tstart_;                                                    \
        if (p.trace)                                                                                \
            for (int s_ = (first); s_ <= (last); ++s_) p.trace[blockIdx.x * kTraceSlots + s_] = tr_[s_]; \
    } while (0)
#else
#define MLA_TIMED(slot, expr) (expr)
#define MLA_TRACE_DECL do { } while (0)
#define MLA_TRACE_ADD(slot, v) do { } while (0)
#define MLA_TRACE_NOW() 0LL
#define MLA_TRACE_FLUSH(first, last, total_slot) do { } while (0)
#endif

struct Params {
    const int32_t* plan;
    const __nv_bfloat16* q_abs;  // [B][128][512]
    const __nv_bfloat16* q_r;    // [B][128][64]
    const int32_t* block_table;  // [B][max_pages]
    int32_t max_pages;
    int32_t num_pool_pages;
    float scale_log2;            // softmax_scale * log2(e)
    __nv_bfloat16* o_lat;        // [B][128][512]
    float* lse;                  // [B][128]
    float* ws_o;                 // [partials][128][512]
    float* ws_lse;               // [partials][128]
    uint32_t* dev_error;
    uint64_t timeout_ns;
    long long* trace;            // wait-cycle accounting (MLA_DECODE_TRACE builds only), else null
};

struct Item {
    int seq, page_begin, page_end, seq_len, slot;
};

__device__ __forceinline__ Item load_item(const int32_t* plan, int items_off, int i)
{
    const int4 a = *reinterpret_cast<const int4*>(plan + items_off + kItemWords * i);
    const int4 b = *reinterpret_cast<const int4*>(plan + items_off + kItemWords * i + 4);
    return Item{a.x, a.y, a.z, a.w, b.x};
}

// ---------------------------------------------------------------------------- TMA producer

// Streams the pages of this cluster's items into a `stages`-deep ring; `boxes` 64-column boxes
// per page (9 for the score CTA: latent + RoPE key, 8 for the value CTA: latent only).
__device__ __forceinline__ void run_producer(const CUtensorMap* tm, const Params& p, int item_begin, int item_end,
                                             int items_off, uint32_t sbase, uint32_t bars, int boxes, int stages,
                                             int stage_bytes, uint64_t policy, const dev::WaitCtx& w, int lane)
{
    using namespace dev;
    MLA_TRACE_DECL;
    if (lane == 0) tma_prefetch_desc(tm);
    int g = 0;
    bool ok = true;
    for (int i = item_begin; i < item_end && ok; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        const int32_t* bt = p.block_table + (int64_t)it.seq * p.max_pages;
        for (int pg0 = it.page_begin; pg0 < it.page_end && ok; pg0 += 32) {
            const int n = min(32, it.page_end - pg0);
            int page = 0;
            if (lane < n) {
                page = __ldg(bt + pg0 + lane);
                if (page < 0 || page >= p.num_pool_pages) raise_error(p.dev_error, MLA_DEVERR_BAD_PAGE);
            }
            for (int j = 0; j < n; ++j) {
                const int pj = __shfl_sync(0xffffffffu, page, j);
                if (lane == 0) {
                    const int s = g % stages;
                    if (g >= stages) ok = MLA_TIMED(1, wait_phase(bars + 8 * (kEmpty0 + s), g / stages - 1, w));
                    if (ok) {
                        const uint32_t full = bars + 8 * (kFull0 + s);
                        const uint32_t dst = sbase + s * stage_bytes;
                        mbar_arrive_expect_tx(full, boxes * kBoxBytes);
                        // an out-of-range page id reads as zeros (TMA fills outside the tensor)
                        for (int x = 0; x < boxes; ++x) tma_load_3d(dst + x * kBoxBytes, tm, full, 64 * x, 0, pj, policy);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                ++g;
            }
        }
    }
    if (lane == 0 && *w.abort) {  // loads still in flight must land before the CTA exits
        for (int k = (g > stages ? g - stages : 0); k < g; ++k)
            drain_phase(bars + 8 * (kFull0 + k % stages), k / stages, w.timeout_ns);
    }
    if (lane == 0) MLA_TRACE_FLUSH(0, 1, 0);
}

// ---------------------------------------------------------------------------- score CTA

// Streams this cluster's pages as K-chunks: chunk j of a two-page group holds 64-column box j
// (boxes 0-7: c_KV, box 8: k_R) of the first page in rows 0-63 and of the second in rows 64-127.
__device__ __forceinline__ void score_producer(const CUtensorMap* tm, const Params& p, int item_begin, int item_end,
                                               int items_off, uint32_t sbase, uint32_t bars, const dev::WaitCtx& w,
                                               int lane)
{
    using namespace dev;
    MLA_TRACE_DECL;
    const uint64_t policy = l2_policy_evict_normal();  // the value CTA reads these pages next
    if (lane == 0) tma_prefetch_desc(tm);
    int c = 0;
    bool ok = true;
    for (int i = item_begin; i < item_end && ok; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        const int32_t* bt = p.block_table + (int64_t)it.seq * p.max_pages;
        for (int pg0 = it.page_begin; pg0 < it.page_end && ok; pg0 += 32) {
            const int n = min(32, it.page_end - pg0);  // even unless it ends the item
            int page = 0;
            if (lane < n) {
                page = __ldg(bt + pg0 + lane);
                if (page < 0 || page >= p.num_pool_pages) raise_error(p.dev_error, MLA_DEVERR_BAD_PAGE);
            }
            for (int j = 0; j < n && ok; j += kGroupPages) {
                const int npg = min(kGroupPages, n - j);
                const int pa = __shfl_sync(0xffffffffu, page, j);
                const int pb = __shfl_sync(0xffffffffu, page, min(j + 1, 31));
                if (lane == 0) {
                    for (int box = 0; box < kBoxesPerRow && ok; ++box, ++c) {
                        const int s = c % kChunkStages;
                        if (c >= kChunkStages)
                            ok = MLA_TIMED(1, wait_phase(bars + 8 * (kEmpty0 + s), c / kChunkStages - 1, w));
                        if (!ok) break;
                        const uint32_t full = bars + 8 * (kFull0 + s);
                        const uint32_t dst = sbase + kOffChunks + s * kChunkBytes;
                        mbar_arrive_expect_tx(full, npg * kBoxBytes);
                        // an out-of-range page id reads as zeros (TMA fills outside the tensor)
                        tma_load_3d(dst, tm, full, 64 * box, 0, pa, policy);
                        if (npg == 2) tma_load_3d(dst + kBoxBytes, tm, full, 64 * box, 0, pb, policy);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
        }
    }
    if (lane == 0 && *w.abort) {  // loads still in flight must land before the CTA exits
        for (int k = (c > kChunkStages ? c - kChunkStages : 0); k < c; ++k)
            drain_phase(bars + 8 * (kFull0 + k % kChunkStages), k / kChunkStages, w.timeout_ns);
    }
    if (lane == 0) MLA_TRACE_FLUSH(0, 1, 0);
}

// QK of a two-page group: S[128 heads x N tokens] (N = 64 per page) accumulated over the nine
// K-chunks: chunks 0-7 take q_abs from TMEM ("TS"), chunk 8 takes q_R from shared memory.
// One thread issues everything, so the loop is kept to a handful of instructions per MMA:
// descriptors are built once and advanced by constants (16-byte units in the low bits),
// the ring position is a wrapping counter, and the nine chunks are unrolled.
__device__ __forceinline__ void score_mma(const Params& p, int item_begin, int item_end, int items_off, uint32_t sbase,
                                          uint32_t bars, uint32_t tmem, const dev::WaitCtx& w)
{
    using namespace dev;
    constexpr uint32_t idesc2 = idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc1 = idesc_bf16(128, 64, false, false);
    const uint64_t chunk_desc0 = smem_desc(sbase + kOffChunks, 16, 1024);
    const uint64_t qr_desc = smem_desc(sbase + kOffQR, 16, 1024);
    const uint32_t full0 = bars + 8 * kFull0, empty0 = bars + 8 * kEmpty0;
    MLA_TRACE_DECL;
    int s = 0, phase = 0, G = 0, n_item = 0;
    for (int i = item_begin; i < item_end; ++i, ++n_item) {
        const Item it = load_item(p.plan, items_off, i);
        if (!MLA_TIMED(5, wait_phase(bars + 8 * kQReady, n_item, w))) goto out;
        tc_fence_after();
        for (int pg = it.page_begin; pg < it.page_end; pg += kGroupPages, ++G) {
            const uint32_t idesc = (it.page_end - pg >= 2) ? idesc2 : idesc1;
            const int buf = G & 1;
            if (G >= 2 && !MLA_TIMED(4, wait_phase(bars + 8 * (kSFree0 + buf), (G >> 1) - 1, w))) goto out;
            const uint32_t d = tmem + kSCol + 128 * buf;
#pragma unroll
            for (int box = 0; box < kBoxesPerRow; ++box) {
                if (!MLA_TIMED(3, wait_phase(full0 + 8 * s, phase, w))) goto out;
                tc_fence_after();
                const uint64_t b0 = chunk_desc0 + (uint64_t)(s * (kChunkBytes >> 4));
                if (box < 8) {
                    const uint32_t a0 = tmem + kQCol + 32 * box;
                    mma_ts(d, a0, b0, idesc, box != 0 ? 1u : 0u);
                    mma_ts(d, a0 + 8, b0 + 2, idesc, 1u);
                    mma_ts(d, a0 + 16, b0 + 4, idesc, 1u);
                    mma_ts(d, a0 + 24, b0 + 6, idesc, 1u);
                } else {
                    mma_ss(d, qr_desc, b0, idesc, 1u);
                    mma_ss(d, qr_desc + 2, b0 + 2, idesc, 1u);
                    mma_ss(d, qr_desc + 4, b0 + 4, idesc, 1u);
                    mma_ss(d, qr_desc + 6, b0 + 6, idesc, 1u);
                }
                mma_commit(empty0 + 8 * s);
                if (++s == kChunkStages) {
                    s = 0;
                    ++phase;
                }
            }
            mma_commit(bars + 8 * (kSFull0 + buf));
        }
    }
out:
    mma_commit(bars + 8 * kDrain);
    drain_phase(bars + 8 * kDrain, 0, w.timeout_ns);
    MLA_TRACE_ADD(12, G);
    MLA_TRACE_FLUSH(2, 5, 2);
    MLA_TRACE_FLUSH(12, 12, 2);
}

// Query row of this thread: q_abs -> TMEM lane `row`, columns 0..255 (two bf16 per column, K
// order); q_R -> row `row` of the K-major, 128-byte-swizzled q_R tile in shared memory.
__device__ __forceinline__ void load_query(const Params& p, int seq, int row, uint32_t taddr, uint8_t* qr_smem)
{
    using namespace dev;
    const uint4* qa = reinterpret_cast<const uint4*>(p.q_abs + ((int64_t)seq * 128 + row) * 512);
    const uint4* qr = reinterpret_cast<const uint4*>(p.q_r + ((int64_t)seq * 128 + row) * 64);
    uint4 r8[8];
#pragma unroll
    for (int v = 0; v < 8; ++v) r8[v] = __ldg(qr + v);
#pragma unroll
    for (int c0 = 0; c0 < 8; c0 += 2) {
        uint4 x[16];
#pragma unroll
        for (int v = 0; v < 16; ++v) x[v] = __ldg(qa + 8 * c0 + v);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            uint32_t r[32];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                r[4 * v + 0] = x[8 * cc + v].x;
                r[4 * v + 1] = x[8 * cc + v].y;
                r[4 * v + 2] = x[8 * cc + v].z;
                r[4 * v + 3] = x[8 * cc + v].w;
            }
            tmem_st32(taddr + kQCol + 32 * (c0 + cc), r);
        }
    }
    uint8_t* dst = qr_smem + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
    for (int v = 0; v < 8; ++v) *reinterpret_cast<uint4*>(dst + ((v ^ (row & 7)) << 4)) = r8[v];
    fence_proxy_async_cta();  // read by the MMA (async proxy)
    tmem_wait_st();
}

__device__ __forceinline__ void score_softmax(const Params& p, int item_begin, int item_end, int items_off,
                                              uint8_t* smem, uint32_t sbase, uint32_t bars, uint32_t tmem,
                                              const dev::WaitCtx& w, int warp, int lane)
{
    using namespace dev;
    const int q4 = warp & 3, row = 32 * q4 + lane;
    const bool leader = (warp == 2 && lane == 0);  // writes the wait-cycle trace, if enabled
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    // addresses in the value CTA (rank 1)
    const uint32_t r_p = map_to_cta(sbase + kOffP, 1);
    const uint32_t r_stats = map_to_cta(sbase + kOffStats, 1);
    const uint32_t r_msg_full = map_to_cta(bars + 8 * kMsgFull0, 1);
    const uint32_t p_row_off = (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
    MLA_TRACE_DECL;
    int g = 0, G = 0;  // pages (messages) and two-page groups
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        [[maybe_unused]] const long long tq0 = MLA_TRACE_NOW();
        load_query(p, it.seq, row, tmem + lane_off, smem + kOffQR);
        tc_fence_before();
        mbar_arrive(bars + 8 * kQReady);
        MLA_TRACE_ADD(9, MLA_TRACE_NOW() - tq0);
        float m_used = -INFINITY, l = 0.f;
        for (int pg = it.page_begin; pg < it.page_end; pg += kGroupPages, ++G) {
            const int npg = min(kGroupPages, it.page_end - pg);
            const int sbuf = G & 1;
            if (!MLA_TIMED(7, wait_warp(bars + 8 * (kSFull0 + sbuf), G >> 1, w))) return;
            tc_fence_after();
            for (int pp = 0; pp < npg; ++pp, ++g) {
                const int t = pg + pp;
                const int buf = g & 1;
                const int valid = min(64, it.seq_len - 64 * t);
                const bool last = (t == it.page_end - 1);
                [[maybe_unused]] const long long tc0 = MLA_TRACE_NOW();
                uint32_t sr[64];
                const uint32_t scol = tmem + lane_off + kSCol + 128 * sbuf + 64 * pp;
                tmem_ld32(scol, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                tmem_wait_ld();
                MLA_TRACE_ADD(11, MLA_TRACE_NOW() - tc0);
                if (pp == npg - 1) {  // both pages of the group are in registers or done
                    [[maybe_unused]] const long long ta0 = MLA_TRACE_NOW();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars + 8 * (kSFree0 + sbuf));
                    MLA_TRACE_ADD(13, MLA_TRACE_NOW() - ta0);
                }

                // slots past the sequence end score -inf (their p is exactly 0)
                if (valid < 64) {
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        if (j >= valid) sr[j] = __float_as_uint(-INFINITY);
                }
                // row max of the raw scores (softmax_scale > 0 commutes with max), 8-way tree
                float m8[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) m8[a] = __uint_as_float(sr[a]);
#pragma unroll
                for (int j = 8; j < 64; ++j) m8[j & 7] = fmaxf(m8[j & 7], __uint_as_float(sr[j]));
                const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * p.scale_log2;
                float factor = 1.f;
                if (mx > m_used + kRescaleThreshold) {
                    if (t != it.page_begin) {
                        factor = ex2_approx(m_used - mx);
                        l *= factor;
                    }
                    m_used = mx;
                }
                // p = 2^(s * scale * log2(e) - m): one FMA and one MUFU.EX2 per score
                uint32_t pk[32];
                float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * j]), p.scale_log2, -m_used));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * j + 1]), p.scale_log2, -m_used));
                    pk[j] = pack_bf16x2(p0, p1);
                    l8[j & 7] += p0 + p1;
                }
                l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
                MLA_TRACE_ADD(14, MLA_TRACE_NOW() - tc0);

                // the staging buffer and the peer's P buffer `buf` are free once PV(g-2) finished
                if (g >= 2 && !MLA_TIMED(8, wait_warp<true>(bars + 8 * (kMsgFree0 + buf), (g >> 1) - 1, w))) return;
                [[maybe_unused]] const long long tw0 = MLA_TRACE_NOW();
                uint8_t* stage_p = smem + kOffScoreStaging + buf * kPBytes + p_row_off;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(stage_p + ((c ^ (row & 7)) << 4)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                const uint32_t stats_off = kOffStats + buf * kStatsBytes + q4 * kStatsWarpBytes;
                float* stats = reinterpret_cast<float*>(smem + stats_off);
                stats[lane] = factor;
                if (last) stats[32 + lane] = 1.f / l;
                const bool any_rescale = __any_sync(0xffffffffu, factor != 1.f);
                if (lane == 0)
                    reinterpret_cast<uint32_t*>(stats)[64] = (any_rescale ? 1u : 0u) | (valid < 64 ? 2u : 0u);
                fence_proxy_async_cta();  // these generic writes are read by the bulk copies
                __syncwarp();
                if (lane == 0) {
                    const uint32_t bar = r_msg_full + 8 * buf;
                    // rows 32*q4 .. 32*q4+31 of P are one contiguous 4 KB slice of the swizzled tile
                    bulk_copy_to_cta(r_p + buf * kPBytes + q4 * kPWarpBytes,
                                     sbase + kOffScoreStaging + buf * kPBytes + q4 * kPWarpBytes, kPWarpBytes, bar);
                    bulk_copy_to_cta(r_stats + (stats_off - kOffStats), sbase + stats_off, kStatsWarpBytes, bar);
                }
                MLA_TRACE_ADD(10, MLA_TRACE_NOW() - tw0);
            }
        }
        const float lse_val = (m_used + log2f(l)) * 0.69314718055994531f;
        if (it.slot < 0)
            p.lse[(int64_t)it.seq * 128 + row] = lse_val;
        else
            p.ws_lse[(int64_t)it.slot * 128 + row] = lse_val;
    }
    // the value CTA's last commits arrive here, and the last bulk copies read this CTA's
    // staging buffers: wait for both before this CTA can finish
    for (int k = (g > 2 ? g - 2 : 0); k < g; ++k)
        if (!wait_warp<true>(bars + 8 * (kMsgFree0 + (k & 1)), k >> 1, w)) return;
    if (leader) MLA_TRACE_FLUSH(6, 11, 6);
    if (leader) MLA_TRACE_FLUSH(13, 14, 6);
}

// ---------------------------------------------------------------------------- value CTA

__device__ __forceinline__ uint32_t msg_flags(const uint8_t* smem, int buf)
{
    const volatile uint32_t* f = reinterpret_cast<const volatile uint32_t*>(smem + kOffStats + buf * kStatsBytes);
    const int w = kStatsWarpBytes / 4;
    return f[64] | f[w + 64] | f[2 * w + 64] | f[3 * w + 64];
}

__device__ __forceinline__ void value_mma(const Params& p, int item_begin, int item_end, int items_off,
                                          const uint8_t* smem, uint32_t sbase, uint32_t bars, uint32_t tmem,
                                          const dev::WaitCtx& w)
{
    using namespace dev;
    constexpr uint32_t idesc = idesc_bf16(128, 256, false, true);
    const uint64_t p_desc0 = smem_desc(sbase + kOffP, 16, 1024);
    const uint64_t v_desc0 = smem_desc(sbase, kBoxBytes, 1024);
    MLA_TRACE_DECL;
    int g = 0, n_flagged = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int s = g % kValueStages, buf = g & 1;
            if (!MLA_TIMED(3, wait_phase(bars + 8 * (kFull0 + s), g / kValueStages, w))) goto out;
            // expect this message's bytes (the copies may land before or after this)
            mbar_arrive_expect_tx(bars + 8 * (kMsgFull0 + buf), kMsgBytes);
            if (!MLA_TIMED(4, wait_phase<true>(bars + 8 * (kMsgFull0 + buf), g >> 1, w))) goto out;
            // The correction warps go first on flagged tiles (rescale O, zero a tail) and on the
            // first tile of every item after the first (their epilogue still reads O, which this
            // PV overwrites).  Both sides apply the same rule, so o_ready phases stay paired.
            if (msg_flags(smem, buf) != 0 || (t == it.page_begin && i != item_begin)) {
                const int e = n_flagged & 1;
                mma_commit(bars + 8 * (kODrain0 + e));  // arrives once every earlier PV is done
                if (!MLA_TIMED(5, wait_phase(bars + 8 * (kOReady0 + e), n_flagged >> 1, w))) goto out;
                ++n_flagged;
            }
            tc_fence_after();
            {
                // A = P [128 heads x 16 tokens] K-major; B = page [16 tokens x 256 dims] MN-major
                const uint64_t a0 = p_desc0 + (uint64_t)(buf * (kPBytes >> 4));
                const uint64_t b0 = v_desc0 + (uint64_t)(s * (kValueStageBytes >> 4));
                const uint32_t acc0 = (t == it.page_begin) ? 0u : 1u;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint64_t bh = b0 + (uint64_t)(half * ((4 * kBoxBytes) >> 4));
                    mma_ss(tmem + 256 * half, a0, bh, idesc, acc0);
                    mma_ss(tmem + 256 * half, a0 + 2, bh + (2048 >> 4), idesc, 1u);
                    mma_ss(tmem + 256 * half, a0 + 4, bh + (4096 >> 4), idesc, 1u);
                    mma_ss(tmem + 256 * half, a0 + 6, bh + (6144 >> 4), idesc, 1u);
                }
            }
            mma_commit(bars + 8 * (kEmpty0 + s));
            mma_commit_multicast(bars + 8 * (kMsgFree0 + buf), 0x1);
        }
    }
out:
    mma_commit(bars + 8 * kDrain);
    drain_phase(bars + 8 * kDrain, 0, w.timeout_ns);
    MLA_TRACE_ADD(12, g);
    MLA_TRACE_FLUSH(2, 5, 2);
    MLA_TRACE_FLUSH(12, 12, 2);
}

// Normalised output of an item: O / l to o_lat (bf16, sole item of its sequence) or to the
// item's split partial (fp32).  Thread `row` owns TMEM lane `row`.
__device__ __forceinline__ void write_output(const Params& p, const Item& it, float inv_l, uint32_t tmem,
                                             uint32_t lane_off, int row)
{
    using namespace dev;
#pragma unroll 1
    for (int j = 0; j < 16; ++j) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + 32 * j, r);
        tmem_wait_ld();
        if (it.slot < 0) {
            uint4* d4 = reinterpret_cast<uint4*>(p.o_lat + ((int64_t)it.seq * 128 + row) * 512 + 32 * j);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                uint4 o;
                o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv_l, __uint_as_float(r[8 * v + 1]) * inv_l);
                o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv_l, __uint_as_float(r[8 * v + 3]) * inv_l);
                o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv_l, __uint_as_float(r[8 * v + 5]) * inv_l);
                o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv_l, __uint_as_float(r[8 * v + 7]) * inv_l);
                d4[v] = o;
            }
        } else {
            float4* d4 = reinterpret_cast<float4*>(p.ws_o + ((int64_t)it.slot * 128 + row) * 512 + 32 * j);
#pragma unroll
            for (int v = 0; v < 8; ++v)
                d4[v] = make_float4(__uint_as_float(r[4 * v + 0]) * inv_l, __uint_as_float(r[4 * v + 1]) * inv_l,
                                    __uint_as_float(r[4 * v + 2]) * inv_l, __uint_as_float(r[4 * v + 3]) * inv_l);
        }
    }
}

__device__ __forceinline__ void value_correction(const Params& p, int item_begin, int item_end, int items_off,
                                                 uint8_t* smem, uint32_t bars, uint32_t tmem, const dev::WaitCtx& w,
                                                 int warp, int lane, int tid128)
{
    using namespace dev;
    const int q4 = warp & 3, row = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const uint32_t r_msg_free = dev::map_to_cta(dev::smem_u32(smem) + kOffBars + 8 * kMsgFree0, 0);
    MLA_TRACE_DECL;
    int g = 0, n_flagged = 0;
    Item prev{};
    float prev_inv_l = 0.f;
    bool have_prev = false;  // an item whose output is still in TMEM
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        float inv_l = 0.f;
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int buf = g & 1;
            if (!MLA_TIMED(7, wait_warp<true>(bars + 8 * (kMsgFull0 + buf), g >> 1, w))) goto done;
            const float* stats =
                reinterpret_cast<const float*>(smem + kOffStats + buf * kStatsBytes + q4 * kStatsWarpBytes);
            if (t == it.page_end - 1) inv_l = stats[32 + lane];
            const float factor = stats[lane];
            const uint32_t flags = msg_flags(smem, buf);
            // statistics read: the score CTA may reuse this buffer once PV(g) is done too
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(r_msg_free + 8 * buf);
            const bool boundary = (t == it.page_begin) && have_prev;
            if (flags == 0 && !boundary) continue;

            // flagged tile: the MMA thread committed o_drain and waits o_ready before this PV
            [[maybe_unused]] const long long tc0 = MLA_TRACE_NOW();
            const int e = n_flagged & 1;
            if (!MLA_TIMED(10, wait_warp(bars + 8 * (kODrain0 + e), n_flagged >> 1, w))) goto done;
            tc_fence_after();
            if (boundary) {  // the previous item's output leaves TMEM before this PV overwrites it
                [[maybe_unused]] const long long te0 = MLA_TRACE_NOW();
                write_output(p, prev, prev_inv_l, tmem, lane_off, row);
                have_prev = false;
                MLA_TRACE_ADD(9, MLA_TRACE_NOW() - te0);
            }
            if (flags & 2u) {
                // slots past the sequence end may hold anything (NaN): zero them so that
                // p = 0 times them stays 0 in the PV contraction
                const int valid = min(64, it.seq_len - 64 * t);
                const int s = g % kValueStages;
                if (!wait_warp(bars + 8 * (kFull0 + s), g / kValueStages, w)) goto done;
                uint8_t* stage = smem + s * kValueStageBytes;
                const int chunks = (64 - valid) * 64;  // rows x (8 boxes x 8 chunks of 16 B)
                for (int c = tid128; c < chunks; c += 128) {
                    const int r = valid + (c >> 6), box = (c >> 3) & 7, ch = c & 7;
                    *reinterpret_cast<uint4*>(stage + box * kBoxBytes + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_cta();
            }
            if ((flags & 1u) && t != it.page_begin && __any_sync(0xffffffffu, factor != 1.f)) {
#pragma unroll 1
                for (int j = 0; j < 16; ++j) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_off + 32 * j, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int v = 0; v < 32; ++v) r[v] = __float_as_uint(__uint_as_float(r[v]) * factor);
                    tmem_st32(tmem + lane_off + 32 * j, r);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(bars + 8 * (kOReady0 + e));
            ++n_flagged;
            MLA_TRACE_ADD(8, MLA_TRACE_NOW() - tc0);
        }
        prev = it;
        prev_inv_l = inv_l;
        have_prev = true;
    }
    if (have_prev) {
        // last item: every PV is done when the MMA thread's final commit lands
        if (!MLA_TIMED(10, wait_warp(bars + 8 * kDrain, 0, w))) goto done;
        tc_fence_after();
        [[maybe_unused]] const long long te0 = MLA_TRACE_NOW();
        write_output(p, prev, prev_inv_l, tmem, lane_off, row);
        MLA_TRACE_ADD(9, MLA_TRACE_NOW() - te0);
    }
done:
    tc_fence_before();
    if (warp == 2 && lane == 0) MLA_TRACE_FLUSH(6, 10, 6);
}

// ---------------------------------------------------------------------------- kernel

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_bf16_kernel(const __grid_constant__ CUtensorMap tm_pool, const Params p)
{
    using namespace dev;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x >> 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kOffBars;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffTmemHolder);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
    const bool misaligned = (sbase & 1023u) != 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(bars + 8 * (kFull0 + s), 1);
            mbar_init(bars + 8 * (kEmpty0 + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars + 8 * (kSFull0 + b), 1);
            mbar_init(bars + 8 * (kSFree0 + b), 4);        // one arrive per softmax warp
            mbar_init(bars + 8 * (kMsgFree0 + b), 1 + 4);  // PV commit + four correction warps
            mbar_init(bars + 8 * (kMsgFull0 + b), 1);      // the MMA thread's arm + the copies' bytes
            mbar_init(bars + 8 * (kOReady0 + b), 128);
            mbar_init(bars + 8 * (kODrain0 + b), 1);
        }
        mbar_init(bars + 8 * kQReady, 128);
        mbar_init(bars + 8 * kDrain, 1);
        int bad = misaligned ? 1 : 0;
        if (misaligned) raise_error(p.dev_error, MLA_DEVERR_SMEM_ALIGN);
        if (p.plan[kHdrMagic] != kPlanMagic || p.plan[kHdrVersion] != kPlanVersion) {
            raise_error(p.dev_error, MLA_DEVERR_BAD_PLAN);
            bad = 1;
        }
        *abort_flag = bad;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers exist before anyone arrives remotely
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtx w{p.timeout_ns, abort_flag, p.dev_error};

    if (!*abort_flag) {
        const int n_clusters = p.plan[kHdrClusters];
        const int items_off = p.plan[kHdrItemsOff];
        const int cl_off = p.plan[kHdrClusterOff];
        const int item_begin = cluster < n_clusters ? p.plan[cl_off + cluster] : 0;
        const int item_end = cluster < n_clusters ? p.plan[cl_off + cluster + 1] : 0;
        if (rank == 0) {
            if (warp == 0)
                score_producer(&tm_pool, p, item_begin, item_end, items_off, sbase, bars, w, lane);
            else if (warp == 1) {
                if (lane == 0) score_mma(p, item_begin, item_end, items_off, sbase, bars, tmem, w);
            } else
                score_softmax(p, item_begin, item_end, items_off, smem, sbase, bars, tmem, w, warp, lane);
        } else {
            if (warp == 0)
                run_producer(&tm_pool, p, item_begin, item_end, items_off, sbase, bars, 8, kValueStages,
                             kValueStageBytes, l2_policy_evict_first(), w, lane);
            else if (warp == 1) {
                if (lane == 0) value_mma(p, item_begin, item_end, items_off, smem, sbase, bars, tmem, w);
            } else
                value_correction(p, item_begin, item_end, items_off, smem, bars, tmem, w, warp, lane,
                                 threadIdx.x - 64);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    cluster_sync();  // no remote access into a CTA that has finished
}

}  // namespace decode
}  // namespace mla
