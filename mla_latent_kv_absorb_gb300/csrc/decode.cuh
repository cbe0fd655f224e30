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
//   rank 0, the score CTA: q_abs lives in TMEM (256 columns, the A operand of "TS" MMAs; each
//     item's rows arrive through the TMA ring as four entries ahead of its pages and the MMA
//     thread copies them in with tcgen05.cp) and q_R in shared memory (16 KB); the scores of
//     four pages at a time go to the other 256
//     TMEM columns, one N=256 MMA per K step.  At N=256 each MMA carries 128 cycles of tensor
//     work, which hides the issuing thread's own overhead (its warp shares an SM sub-partition
//     with softmax warps); at N=64 the single issuing thread, not the tensor pipe, was the limit.
//     Pages stream through a ring of K-chunks (one 64-column box of four pages, 32 KB).  Eight
//     softmax warps in two sets (pages 0-1 and 2-3 of a group) each pull two pages of scores
//     into registers, free the score buffer at once, agree on the group's running max through
//     shared memory, write P (bf16, 16 KB per page) into local shared memory, and ship it to
//     the value CTA with asynchronous bulk copies that complete the peer's barrier by byte
//     count.
//   rank 1, the value CTA: O lives in TMEM (512 columns); per page it runs PV from P and its
//     own copy of the page's 512 latent columns; four warps apply the (rare) rescales, zero
//     the unused slots of a sequence's last page, and write the normalised output.
// Both CTAs stream the same pages with their own TMA ring; the score CTA reads first with an
// evict-last hint and the value CTA second with evict-first, so HBM sees each page once.
//
// Online softmax with lazy rescaling: the running max m used for exp2 only moves when a tile's
// max exceeds it by more than 8 (log2 units); then l and O are scaled by exp2(m_old - m_new).
// P values stay <= 2^8, and the final division by l makes the result exact whatever m is.
//
// Pipelines (all waits bounded; see ptx.cuh):
//   kv_full/kv_empty[S]   TMA rings: 4 K-chunk stages in the score CTA, 2 page stages in the
//                         value CTA
//   s_full/s_free         the four-page score buffer (score CTA)
//   q_ready               q_R of an item written to shared memory (score CTA softmax warps)
//   stg_ready[4]          a staged P message is complete (four softmax warps of one set)
//   stg_freed             counter, not a barrier: messages whose staging slot may be reused
//                         (published by the tracker thread, which alone waits on copied)
//   msg_full[4]           P + per-row statistics landed in the value CTA (bulk copies; armed
//                         by the value CTA's acknowledgement thread)
//   copied[4]             (score CTA) message m has landed in the value CTA (acknowledgement
//                         thread): its staging slot may be reused before PV has consumed it
//   msg_free[4]           PV using that P finished (value CTA's MMA commit, multicast to rank 0)
//                         and the value CTA's four correction warps have read the statistics:
//                         the value CTA's buffer may take a new message.  Four message buffers
//                         keep the DSMEM copy and PV round trip off the critical path.
//   A parity wait is valid only while the awaited phase is the current one or the last
//   completed one, so every barrier has waiters that follow all of its phases in order.
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

constexpr int kThreads = 352;                     // producer, MMA, 8 softmax / 4 correction, shipper
constexpr int kShipperWarp = 10;
constexpr int kAckWarp = 6;                       // value CTA: message acknowledgements
constexpr int kChunkStages = 4;
constexpr int kValueStages = 2;
constexpr int kMaxStages = 4;
constexpr int kStagingSlots = 4;                  // score CTA: P messages staged ahead of the peer
constexpr int kMsgSlots = 4;                      // value CTA: P messages it can hold
constexpr int kBoxBytes = 64 * 128;               // 64 tokens x 64 bf16 columns
constexpr int kBoxesPerRow = 9;                   // c_KV: 8 boxes, k_R: 1 box
constexpr int kGroupPages = 4;                    // pages per score MMA (N = 256)
constexpr int kChunkBytes = kGroupPages * kBoxBytes;  // one box column of a four-page group
constexpr int kQueryEntries = 4;                  // ring entries carrying an item's q_abs (two 16 KB boxes each)
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
// score CTA: q_R (K-major, 128-byte swizzle), the K-chunk ring, the staging ring of P messages
// and their statistics blocks
constexpr int kOffQR = 0;
constexpr int kOffChunks = kOffQR + 128 * 128;
constexpr int kOffScoreStaging = kOffChunks + kChunkStages * kChunkBytes;
constexpr int kOffStatsStaging = kOffScoreStaging + kStagingSlots * kPBytes;
// score CTA: the two softmax sets exchange row maxima and partial sums here (double-buffered)
constexpr int kOffXchg = kOffStatsStaging + kStagingSlots * kStatsBytes;
// value CTA: stages, then the P buffers (1024-aligned, the MMA reads them) and their statistics
constexpr int kOffP = kValueStages * kValueStageBytes;
constexpr int kOffStats = kOffP + kMsgSlots * kPBytes;
constexpr int kScoreEnd = kOffXchg + 4 * 2 * 128 * 4;
constexpr int kValueEnd0 = kOffStats + kMsgSlots * kStatsBytes;
// value CTA: one 32 x 32 fp32 transpose tile per correction warp for the output write-out
// (rows padded to 144 bytes, so that both the row-wise writes and the column-wise reads of
// 16-byte vectors fall in distinct bank groups)
constexpr int kOutTileRowBytes = 144;
constexpr int kOutTileBytes = 32 * kOutTileRowBytes;
constexpr int kOffOutTile = (kValueEnd0 + 15) / 16 * 16;
constexpr int kValueEnd = kOffOutTile + 4 * kOutTileBytes;
constexpr int kOffBars = ((kScoreEnd > kValueEnd ? kScoreEnd : kValueEnd) + 7) / 8 * 8;

enum Bar : int {
    kFull0 = 0,
    kEmpty0 = kFull0 + kMaxStages,
    kSFull0 = kEmpty0 + kMaxStages,
    kSFree0 = kSFull0 + 2,
    kQReady = kSFree0 + 2,
    kMsgFree0 = kQReady + 1,
    kMsgFull0 = kMsgFree0 + kMsgSlots,
    kCopied0 = kMsgFull0 + kMsgSlots,
    kOReady0 = kCopied0 + kMsgSlots,
    kODrain0 = kOReady0 + 2,
    kDrain = kODrain0 + 2,
    kStgReady0 = kDrain + 1,
    kAbsFull0 = kStgReady0 + kStagingSlots,  // absorb prologue: operands of K-chunk 0 / 1 landed
    kAbsDone = kAbsFull0 + 2,                 // absorb prologue: the job's MMAs finished
    kAbsEpi = kAbsDone + 1,                   // absorb prologue: the job's rows left TMEM
    kNumBars = kAbsEpi + 1
};

constexpr int kOffTmemHolder = kOffBars + 8 * kNumBars;
constexpr int kOffAbort = kOffTmemHolder + 4;
constexpr int kOffStgFreed = kOffAbort + 4;  // score CTA: messages whose staging slot may be reused
constexpr int kSmemBytes = ((kOffStgFreed + 4 + 127) / 128) * 128;
static_assert(kOffP % 1024 == 0, "P buffers are MMA operands (1024-byte aligned)");
static_assert(kChunkStages <= kMaxStages && kValueStages <= kMaxStages, "barrier slots per ring");
static_assert(kOffBars % 8 == 0, "barriers need 8-byte alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffOutTile % 16 == 0 && kOutTileRowBytes % 16 == 0, "the output tile is read and written in 16-byte vectors");
static_assert(kStatsWarpBytes % 16 == 0 && kPWarpBytes % 16 == 0, "bulk copies move multiples of 16 bytes");

// TMEM columns
constexpr uint32_t kQCol = 0;      // score CTA: q_abs, 256 columns (512 bf16 per lane)
constexpr uint32_t kSCol = 256;    // score CTA: the 256-column score buffer (four pages)
constexpr uint32_t kTmemCols = 512;

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8
constexpr uint32_t kSoftmaxBarrier = 1;    // named barrier of the eight softmax warps

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
// Event timeline of cluster 0 (global timer, ns): trace[kEvBase + kind * kEvSlots + index].
constexpr int kEvBase = 4096, kEvSlots = 512;
#define MLA_EV(kind, idx)                                                                              \
    do {                                                                                               \
        if (p.trace && (blockIdx.x >> 1) == 0 && (idx) < kEvSlots)                                    \
            p.trace[kEvBase + (kind) * kEvSlots + (idx)] = (long long)dev::globaltimer_ns();           \
    } while (0)
#define MLA_TRACE_FLUSH(first, last, total_slot)                                                    \
    do {                                                                                            \
        tr_[(total_slot)] = clock64() - tstart_;                                                    \
        if (p.trace)                                                                                \
            for (int s_ = (first); s_ <= (last); ++s_) p.trace[blockIdx.x * kTraceSlots + s_] = tr_[s_]; \
    } while (0)
#else
#define MLA_TIMED(slot, expr) (expr)
#define MLA_EV(kind, idx) do { } while (0)
#define MLA_TRACE_DECL do { } while (0)
#define MLA_TRACE_ADD(slot, v) do { } while (0)
#define MLA_TRACE_NOW() 0LL
#define MLA_TRACE_FLUSH(first, last, total_slot) do { } while (0)
#endif

struct Params {
    const int32_t* plan;
    const __nv_bfloat16* q_abs;  // [B][128][512]: the absorbed queries (written by the prologue when fused)
    __nv_bfloat16* q_abs_out;    // the same buffer, written by the absorb prologue; null when q_abs is an input
    uint32_t* absorb_sync;       // [2] absorb jobs finished, score CTAs past the wait; null when not fused
    int32_t absorb_jobs;         // 128 heads x tiles of 128 sequences (absorb prologue)
    int32_t batch;
    const __nv_bfloat16* q_r;    // [B][128][64]
    const int32_t* block_table;  // [sequences][max_pages]; an item reads row item.table_row
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
    int seq, page_begin, page_end, seq_len, slot, table_row;
};

__device__ __forceinline__ Item load_item(const int32_t* plan, int items_off, int i)
{
    const int4 a = *reinterpret_cast<const int4*>(plan + items_off + kItemWords * i);
    const int4 b = *reinterpret_cast<const int4*>(plan + items_off + kItemWords * i + 4);
    return Item{a.x, a.y, a.z, a.w, b.x, b.y};
}

// ---------------------------------------------------------------------------- absorb prologue

// With the absorb fused into this kernel (page 1 section 4, path B: q_abs = q_c W_UK per head),
// every CTA of the grid first computes q_abs for one head and one tile of 128 sequences (job j
// = 128 t + h, CTA c takes jobs c, c + grid, ...): q_c[tile, h, :] (128 x 128) times W_UK[h]
// (128 x 512) on tcgen05 into the CTA's TMEM, bf16 rows to global memory.  Its shared memory
// and TMEM are free until the roles below start.  A job is published by a release increment
// of absorb_sync[0]; each score CTA waits for all of them before it loads its first query.
constexpr int kAbsA = 0;                     // q_c: two K-chunks of [128 rows x 64] (16 KB each)
constexpr int kAbsAChunk = 128 * 64 * 2;
constexpr int kAbsW = 2 * kAbsAChunk;        // W_UK[h]: two K-chunks of eight [64 K x 64 N] boxes
constexpr int kAbsWChunk = 8 * 64 * 64 * 2;
constexpr uint32_t kAbsBarrier = 2;          // named barrier of the four epilogue warps
static_assert(kAbsW + 2 * kAbsWChunk <= kOffBars, "the absorb operands fit below the barriers");

__device__ __forceinline__ void absorb_jobs(const CUtensorMap* tm_qc, const CUtensorMap* tm_wuk, const Params& p,
                                            uint32_t sbase, uint32_t bars, uint32_t tmem, const dev::WaitCtx& w,
                                            int warp, int lane)
{
    using namespace dev;
    int n = 0;  // jobs this CTA has done
    for (int j = blockIdx.x; j < p.absorb_jobs; j += gridDim.x, ++n) {
        const int h = j % 128, t = j / 128;
        if (warp == 0) {
            if (lane == 0) {
                // the previous job's MMAs have read the tiles before they are overwritten
                if (n > 0 && !wait_phase(bars + 8 * kAbsDone, n - 1, w)) break;
                const uint64_t pol = l2_policy_evict_first();  // each head's weights are read once
#pragma unroll 1
                for (int kc = 0; kc < 2; ++kc) {
                    const uint32_t full = bars + 8 * (kAbsFull0 + kc);
                    mbar_arrive_expect_tx(full, kAbsAChunk + kAbsWChunk);
                    tma_load_2d(sbase + kAbsA + kc * kAbsAChunk, tm_qc, full, h * 128 + 64 * kc, 128 * t, pol);
                    for (int nb = 0; nb < 8; ++nb)
                        tma_load_2d(sbase + kAbsW + kc * kAbsWChunk + nb * 8192, tm_wuk, full, 64 * nb,
                                    h * 128 + 64 * kc, pol);
                }
            }
        } else if (warp == 1) {
            if (lane == 0) {
                constexpr uint32_t idesc = idesc_bf16(128, 256, false, true);
                // the previous job's rows have left TMEM before these MMAs overwrite it
                bool ok = n == 0 || wait_phase(bars + 8 * kAbsEpi, n - 1, w);
#pragma unroll 1
                for (int kc = 0; kc < 2 && ok; ++kc) {
                    ok = wait_phase(bars + 8 * (kAbsFull0 + kc), n, w);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int half = 0; half < 2; ++half)
                            mma_ss(tmem + 256 * half, smem_desc(sbase + kAbsA + kc * kAbsAChunk + k * 32, 16, 1024),
                                   smem_desc(sbase + kAbsW + kc * kAbsWChunk + half * (kAbsWChunk / 2) + k * 2048, 8192,
                                             1024),
                                   idesc, (kc | k) != 0 ? 1u : 0u);
                }
                mma_commit(bars + 8 * kAbsDone);  // also on an early exit: arrives when issued MMAs finish
            }
        } else if (warp >= 2 && warp < 6) {
            // warp & 3 selects the TMEM lane quarter: row m of the tile, 512 columns
            const int q = warp & 3, m = 128 * t + 32 * q + lane;
            if (__all_sync(0xffffffffu, wait_phase(bars + 8 * kAbsDone, n, w) && !*w.abort)) {
                tc_fence_after();
                uint4* dst = reinterpret_cast<uint4*>(p.q_abs_out + ((int64_t)m * 128 + h) * 512);
#pragma unroll 1
                for (int c = 0; c < 16; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 32 * c, r);
                    tmem_wait_ld();
                    if (m < p.batch) {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[4 * c + v] = make_uint4(
                                pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
                    }
                }
            }
            tc_fence_before();
            __threadfence();  // the rows are visible GPU-wide before the job is published
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8 * kAbsEpi);
            named_barrier_or(kAbsBarrier, 128, false);
            if (warp == 2 && lane == 0) {
                fence_proxy_async_all();  // score CTAs read these rows with TMA
                red_release_gpu_add_u32(p.absorb_sync, 1u);
            }
        }
    }
}

// Score CTA producer, fused absorb: wait (bounded) until every absorb job of the grid is
// published, then count this CTA out; the last score CTA to pass zeroes both words for the next
// launch (no job can still be running then).  Returns false if the wait ran out.
__device__ __forceinline__ bool absorb_wait(const Params& p, const dev::WaitCtx& w)
{
    using namespace dev;
    bool ok = ld_acquire_gpu_u32(p.absorb_sync) >= (uint32_t)p.absorb_jobs;
    if (!ok) {
        const uint64_t t0 = globaltimer_ns();
        while (!ok && !*w.abort) {
            ok = ld_acquire_gpu_u32(p.absorb_sync) >= (uint32_t)p.absorb_jobs;
            if (!ok && globaltimer_ns() - t0 > w.timeout_ns) {
                *w.abort = 1;
                raise_error(w.dev_error, MLA_DEVERR_TIMEOUT);
                break;
            }
        }
    }
    fence_proxy_async_all();  // the TMA loads of q_abs come after the rows the other CTAs wrote
    if (atomicAdd(p.absorb_sync + 1, 1u) == gridDim.x / 2 - 1) {
        atomicExch(p.absorb_sync, 0u);
        atomicExch(p.absorb_sync + 1, 0u);
    }
    return ok;
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
        const int32_t* bt = p.block_table + (int64_t)it.table_row * p.max_pages;
        for (int pg0 = it.page_begin; pg0 < it.page_end && ok; pg0 += 32) {
            const int n = min(32, it.page_end - pg0);
            int page = 0;
            if (lane < n) {
                page = pg0 + lane < p.max_pages ? __ldg(bt + pg0 + lane) : -1;  // past the row: bad page
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
                        MLA_EV(13, g);
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

// Streams this cluster's pages as K-chunks: chunk j of a four-page group holds 64-column box j
// (boxes 0-7: c_KV, box 8: k_R) of the group's pages in rows 0-63, 64-127, 128-191, 192-255.
__device__ __forceinline__ void score_producer(const CUtensorMap* tm, const CUtensorMap* tm_q, const Params& p,
                                               int item_begin, int item_end, int items_off, uint32_t sbase,
                                               uint32_t bars, const dev::WaitCtx& w, int lane)
{
    using namespace dev;
    MLA_TRACE_DECL;
    const uint64_t policy = l2_policy_evict_last();  // the value CTA reads these pages next
    if (lane == 0) {
        tma_prefetch_desc(tm);
        tma_prefetch_desc(tm_q);
    }
    int s = 0, phase = 0, c = 0;
    bool ok = true;
    if (p.absorb_sync && lane == 0) ok = absorb_wait(p, w);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    for (int i = item_begin; i < item_end && ok; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        const int32_t* bt = p.block_table + (int64_t)it.table_row * p.max_pages;
        if (lane == 0) {
            // the item's q_abs rows (128 heads x 512 dims) as four ring entries of two 64-dim
            // boxes each, ahead of its pages
            if (i == item_begin && !p.absorb_sync) griddep_wait();  // q_abs comes from the kernel launched before
            for (int j = 0; j < kQueryEntries && ok; ++j, ++c) {
                if (c >= kChunkStages) ok = MLA_TIMED(1, wait_phase(bars + 8 * (kEmpty0 + s), phase - 1, w));
                if (!ok) break;
                const uint32_t full = bars + 8 * (kFull0 + s);
                const uint32_t dst = sbase + kOffChunks + s * kChunkBytes;
                mbar_arrive_expect_tx(full, kChunkBytes);
                tma_load_2d(dst, tm_q, full, 128 * j, 128 * it.seq, policy);
                tma_load_2d(dst + kChunkBytes / 2, tm_q, full, 128 * j + 64, 128 * it.seq, policy);
                if (++s == kChunkStages) {
                    s = 0;
                    ++phase;
                }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        for (int pg0 = it.page_begin; pg0 < it.page_end && ok; pg0 += 32) {
            const int n = min(32, it.page_end - pg0);  // a multiple of 4 unless it ends the item
            int page = 0;
            if (lane < n) {
                page = pg0 + lane < p.max_pages ? __ldg(bt + pg0 + lane) : -1;  // past the row: bad page
                if (page < 0 || page >= p.num_pool_pages) raise_error(p.dev_error, MLA_DEVERR_BAD_PAGE);
            }
            for (int j = 0; j < n && ok; j += kGroupPages) {
                const int npg = min(kGroupPages, n - j);
                int pages[kGroupPages];
#pragma unroll
                for (int q = 0; q < kGroupPages; ++q) pages[q] = __shfl_sync(0xffffffffu, page, min(j + q, 31));
                if (lane == 0) {
#pragma unroll 1
                    for (int box = 0; box < kBoxesPerRow && ok; ++box, ++c) {
                        if (c >= kChunkStages)
                            ok = MLA_TIMED(1, wait_phase(bars + 8 * (kEmpty0 + s), phase - 1, w));
                        if (!ok) break;
                        const uint32_t full = bars + 8 * (kFull0 + s);
                        const uint32_t dst = sbase + kOffChunks + s * kChunkBytes;
                        mbar_arrive_expect_tx(full, npg * kBoxBytes);
                        // an out-of-range page id reads as zeros (TMA fills outside the tensor)
                        for (int q = 0; q < npg; ++q) tma_load_3d(dst + q * kBoxBytes, tm, full, 64 * box, 0, pages[q], policy);
                        MLA_EV(0, c);
                        if (++s == kChunkStages) {
                            s = 0;
                            ++phase;
                        }
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

// QK of a four-page group: S[128 heads x N tokens] (N = 64 per page, 256 for a full group)
// accumulated over the nine K-chunks: chunks 0-7 take q_abs from TMEM ("TS"), chunk 8 takes
// q_R from shared memory.  Descriptors are built once and advanced by constants (16-byte
// units in the low bits) and the ring position is a wrapping counter, so the one issuing
// thread spends few instructions per MMA.
__device__ __forceinline__ void score_mma(const Params& p, int item_begin, int item_end, int items_off, uint32_t sbase,
                                          uint32_t bars, uint32_t tmem, const dev::WaitCtx& w)
{
    using namespace dev;
    const uint64_t chunk_desc0 = smem_desc(sbase + kOffChunks, 16, 1024);
    const uint64_t qr_desc = smem_desc(sbase + kOffQR, 16, 1024);
    const uint32_t full0 = bars + 8 * kFull0, empty0 = bars + 8 * kEmpty0;
    const uint32_t d = tmem + kSCol;
    MLA_TRACE_DECL;
    int s = 0, phase = 0, G = 0, n_item = 0;
    for (int i = item_begin; i < item_end; ++i, ++n_item) {
        const Item it = load_item(p.plan, items_off, i);
        // q_abs into TMEM columns 0-255 (dims 64 k .. 64 k + 63 -> columns 32 k .. 32 k + 31), once
        // the previous item's QK, which reads those columns, has finished
        if (n_item > 0 && !MLA_TIMED(5, wait_phase(bars + 8 * kSFull0, G - 1, w))) goto out;
#pragma unroll 1
        for (int j = 0; j < kQueryEntries; ++j) {
            if (!MLA_TIMED(3, wait_phase(full0 + 8 * s, phase, w))) goto out;
            tc_fence_after();
            const uint64_t src = smem_desc(sbase + kOffChunks + s * kChunkBytes, 16, 1024);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4)
                    tmem_cp_128x256b(tmem + kQCol + 64 * j + 32 * h + 8 * k4,
                                     src + (uint64_t)(h * ((kChunkBytes / 2) >> 4) + 2 * k4));
            mma_commit(empty0 + 8 * s);
            if (++s == kChunkStages) {
                s = 0;
                ++phase;
            }
        }
        bool qr_ready = false;
        for (int pg = it.page_begin; pg < it.page_end; pg += kGroupPages, ++G) {
            const int npg = min(kGroupPages, it.page_end - pg);
            const uint32_t idesc = idesc_bf16(128, 64 * npg, false, false);
            if (G >= 1 && !MLA_TIMED(4, wait_phase(bars + 8 * kSFree0, G - 1, w))) goto out;
            MLA_EV(3, G);
#pragma unroll 1
            for (int box = 0; box < kBoxesPerRow; ++box) {  // rolled: a small loop stays in the instruction cache
                if (!MLA_TIMED(3, wait_phase(full0 + 8 * s, phase, w))) goto out;
                MLA_EV(1, 9 * G + box);
                tc_fence_after();
                const uint64_t b0 = chunk_desc0 + (uint64_t)(s * (kChunkBytes >> 4));
                if (box < 8) {
                    const uint32_t a0 = tmem + kQCol + 32 * box;
                    mma_ts(d, a0, b0, idesc, box != 0 ? 1u : 0u);
                    mma_ts(d, a0 + 8, b0 + 2, idesc, 1u);
                    mma_ts(d, a0 + 16, b0 + 4, idesc, 1u);
                    mma_ts(d, a0 + 24, b0 + 6, idesc, 1u);
                } else {
                    if (!qr_ready) {  // q_R of this item is in shared memory
                        if (!MLA_TIMED(5, wait_phase(bars + 8 * kQReady, n_item, w))) goto out;
                        tc_fence_after();
                        qr_ready = true;
                    }
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
            mma_commit(bars + 8 * kSFull0);
            MLA_EV(2, G);
        }
    }
out:
    mma_commit(bars + 8 * kDrain);
    drain_phase(bars + 8 * kDrain, 0, w.timeout_ns);
    MLA_TRACE_ADD(12, G);
    MLA_TRACE_FLUSH(2, 5, 2);
    MLA_TRACE_FLUSH(12, 12, 2);
}

// q_R of row `row` into row `row` of the K-major, 128-byte-swizzled q_R tile in shared memory
// (softmax set 0; q_abs reaches TMEM through the TMA ring and tcgen05.cp).
__device__ __forceinline__ void load_query_rope(const Params& p, int seq, int row, uint8_t* qr_smem)
{
    using namespace dev;
    const uint4* qr = reinterpret_cast<const uint4*>(p.q_r + ((int64_t)seq * 128 + row) * 64);
    uint8_t* dst = qr_smem + (row >> 3) * 1024 + (row & 7) * 128;
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = __ldg(qr + k);
#pragma unroll
    for (int k = 0; k < 8; ++k) *reinterpret_cast<uint4*>(dst + ((k ^ (row & 7)) << 4)) = v[k];
    fence_proxy_async_cta();  // read by the MMA (async proxy)
}

// Slots past the sequence end read as -infinity (the raw score there may be anything, NaN
// included): then the page maximum skips them and their p is 2^-inf = 0.  Only a sequence's
// last page has such slots.
__device__ __forceinline__ void page_mask(uint32_t (&sr)[64], int valid)
{
    if (valid < 64) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
            if (j >= valid) sr[j] = __float_as_uint(-INFINITY);
    }
}

// Softmax of one page held in registers (masked by page_mask): p = 2^(s * scale * log2(e) - m)
// (one FMA and one MUFU.EX2 per score), and writes P as bf16 straight into this thread's row of
// the swizzled staging tile (16-byte chunk c of the row goes to chunk c ^ (row & 7)).  Returns
// the row sum of p.
__device__ __forceinline__ float page_softmax(const uint32_t (&sr)[64], float scale_log2, float m_used,
                                              uint8_t* stage_row, int row)
{
    using namespace dev;
    float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint32_t pk[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = 8 * c + 2 * q;
            const float p0 = ex2_approx(fmaf(__uint_as_float(sr[j]), scale_log2, -m_used));
            const float p1 = ex2_approx(fmaf(__uint_as_float(sr[j + 1]), scale_log2, -m_used));
            pk[q] = pack_bf16x2(p0, p1);
            l8[(2 * q) & 7] += p0;
            l8[(2 * q + 1) & 7] += p1;
        }
        *reinterpret_cast<uint4*>(stage_row + ((c ^ (row & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    return ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
}

// Row max of a page's raw scores (masked by page_mask), 8-way tree.
__device__ __forceinline__ float page_max(const uint32_t (&sr)[64])
{
    float m8[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) m8[a] = __uint_as_float(sr[a]);
#pragma unroll
    for (int j = 8; j < 64; ++j) m8[j & 7] = fmaxf(m8[j & 7], __uint_as_float(sr[j]));
    return fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
}

// Finish this warp's part of staged message `slot`: its statistics block (per-row O rescale
// factor, 1/l on the item's last page, flags), then mark the warp's share ready for the shipper.
__device__ __forceinline__ void stage_message(uint8_t* smem, uint32_t bars, int slot, int q4, int lane, float factor,
                                              float inv_l, bool last, bool tail)
{
    using namespace dev;
    float* stats = reinterpret_cast<float*>(smem + kOffStatsStaging + slot * kStatsBytes + q4 * kStatsWarpBytes);
    stats[lane] = factor;
    if (last) stats[32 + lane] = inv_l;
    const bool any_rescale = __any_sync(0xffffffffu, factor != 1.f);
    if (lane == 0) reinterpret_cast<uint32_t*>(stats)[64] = (any_rescale ? 1u : 0u) | (tail ? 2u : 0u);
    fence_proxy_async_cta();  // the staged P and statistics are read by the shipper's bulk copies
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (kStgReady0 + slot));
}

// Staging tracker (one thread): follows every phase of copied, in message order, and publishes
// how many messages have landed in the value CTA, which frees their staging slots for the
// softmax warps.
__device__ __forceinline__ void score_tracker(const Params& p, int item_begin, int item_end, int items_off,
                                              uint8_t* smem, uint32_t bars, const dev::WaitCtx& w)
{
    using namespace dev;
    uint32_t* freed = reinterpret_cast<uint32_t*>(smem + kOffStgFreed);
    int k = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        for (int t = it.page_begin; t < it.page_end; ++t, ++k) {
            if (!wait_phase<true>(bars + 8 * (kCopied0 + k % kMsgSlots), k / kMsgSlots, w)) return;
            MLA_EV(9, k);
            st_release_u32(freed, (uint32_t)(k + 1));  // messages 0 .. k copied
        }
    }
}

// Shipper (one thread): sends the staged messages in order to the value CTA, two bulk copies
// each (P, statistics) that complete the peer's msg_full barrier by byte count, once the value
// CTA has finished with the message that last used the same buffer.  It alone waits on
// msg_free and follows all of its phases.
__device__ __forceinline__ void score_shipper(const Params& p, int item_begin, int item_end, int items_off,
                                              uint8_t* smem, uint32_t sbase, uint32_t bars, const dev::WaitCtx& w)
{
    using namespace dev;
    const uint32_t r_p = map_to_cta(sbase + kOffP, 1);
    const uint32_t r_stats = map_to_cta(sbase + kOffStats, 1);
    const uint32_t r_msg_full = map_to_cta(bars + 8 * kMsgFull0, 1);
    MLA_TRACE_DECL;
    int m = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        for (int t = it.page_begin; t < it.page_end; ++t, ++m) {
            const int slot = m % kStagingSlots, buf = m % kMsgSlots;
            if (!MLA_TIMED(14, wait_phase(bars + 8 * (kStgReady0 + slot), m / kStagingSlots, w))) goto out;
            if (m >= kMsgSlots &&  // the value CTA is done with the message that last used buffer buf
                !MLA_TIMED(15, wait_phase<true>(bars + 8 * (kMsgFree0 + buf), m / kMsgSlots - 1, w)))
                goto out;
            const uint32_t bar = r_msg_full + 8 * buf;
            bulk_copy_to_cta(r_p + buf * kPBytes, sbase + kOffScoreStaging + slot * kPBytes, kPBytes, bar);
            bulk_copy_to_cta(r_stats + buf * kStatsBytes, sbase + kOffStatsStaging + slot * kStatsBytes,
                             kStatsBytes, bar);
            MLA_EV(8, m);
        }
    }
    // the value CTA's last commits and arrivals land in this CTA: wait for them before it ends
    for (int k = (m > kMsgSlots ? m - kMsgSlots : 0); k < m; ++k)
        if (!wait_phase<true>(bars + 8 * (kMsgFree0 + k % kMsgSlots), k / kMsgSlots, w)) break;
out:
    MLA_TRACE_FLUSH(14, 15, 0);
}

// Wait (bounded) until at least `target` staged messages have been consumed; warp-uniform.
__device__ __forceinline__ bool wait_freed(const uint32_t* freed, uint32_t target, const dev::WaitCtx& w)
{
    using namespace dev;
    bool ok = ld_acquire_u32(freed) >= target;
    if (!ok && !*w.abort) {
        const uint64_t t0 = globaltimer_ns();
        while (true) {
            if (ld_acquire_u32(freed) >= target) { ok = true; break; }
            if (*w.abort) break;
            if (globaltimer_ns() - t0 > w.timeout_ns) {
                *w.abort = 1;
                raise_error(w.dev_error, MLA_DEVERR_TIMEOUT);
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void score_softmax(const Params& p, int item_begin, int item_end, int items_off,
                                              uint8_t* smem, uint32_t sbase, uint32_t bars, uint32_t tmem,
                                              const dev::WaitCtx& w, int warp, int lane)
{
    using namespace dev;
    const int q4 = warp & 3, row = 32 * q4 + lane;
    const int set = (warp - 2) >> 2;               // 0: pages 0-1 of a group, 1: pages 2-3
    const bool leader = (warp == 2 && lane == 0);  // writes the wait-cycle trace, if enabled
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const uint32_t p_row_off = (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
    const uint32_t* freed = reinterpret_cast<const uint32_t*>(smem + kOffStgFreed);
    float* xchg = reinterpret_cast<float*>(smem + kOffXchg);  // [slot 2][kind 2: max, l][set 2][128]
    MLA_TRACE_DECL;
    int g = 0, G = 0;  // pages (messages) and four-page groups
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        [[maybe_unused]] const long long tq0 = MLA_TRACE_NOW();
        if (set == 0) load_query_rope(p, it.seq, row, smem + kOffQR);
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * kQReady);
        MLA_TRACE_ADD(9, MLA_TRACE_NOW() - tq0);
        float m_used = -INFINITY, l_mine = 0.f, l_total = 0.f;
        for (int pg = it.page_begin; pg < it.page_end; pg += kGroupPages, ++G) {
            const int npg = min(kGroupPages, it.page_end - pg);
            const int n_mine = max(0, min(2, npg - 2 * set));
            const bool last_group = (pg + kGroupPages >= it.page_end);
            float* xs = xchg + (G & 1) * 2 * 2 * 128;
            // Both sets must reach every named barrier below the same number of times: a failed
            // (timed-out) wait only clears `ok`, and each barrier ORs the abort state so that the
            // two sets leave together.
            bool ok = MLA_TIMED(7, wait_warp(bars + 8 * kSFull0, G, w));
            if (lane == 0 && (warp == 2 || warp == 6)) MLA_EV(warp == 2 ? 4 : 15, G);
            [[maybe_unused]] const long long tc0 = MLA_TRACE_NOW();
            uint32_t sr[2][64];
            const int t0 = pg + 2 * set;
            const int valid0 = min(64, it.seq_len - 64 * t0), valid1 = min(64, it.seq_len - 64 * (t0 + 1));
            float mx = -INFINITY;
            if (ok) {
                tc_fence_after();
                if (n_mine > 0) {
                    const uint32_t scol = tmem + lane_off + kSCol + 128 * set;
                    tmem_ld32(scol, *reinterpret_cast<uint32_t(*)[32]>(&sr[0][0]));
                    tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[0][32]));
                    if (n_mine > 1) {
                        tmem_ld32(scol + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[1][0]));
                        tmem_ld32(scol + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[1][32]));
                    }
                    tmem_wait_ld();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars + 8 * kSFree0);  // the next group's QK may start
                if (lane == 0 && warp == 2) MLA_EV(5, G);
                MLA_TRACE_ADD(14, MLA_TRACE_NOW() - tc0);
                if (n_mine > 0) {
                    page_mask(sr[0], valid0);
                    mx = page_max(sr[0]);
                }
                if (n_mine > 1) {
                    page_mask(sr[1], valid1);
                    mx = fmaxf(mx, page_max(sr[1]));
                }
            }
            MLA_TRACE_ADD(11, MLA_TRACE_NOW() - tc0);

            // group max, agreed between the two sets, drives the lazy rescale
            xs[set * 128 + row] = mx * p.scale_log2;
            if (MLA_TIMED(13, named_barrier_or(kSoftmaxBarrier, 256, !ok || *w.abort))) return;
            if (lane == 0 && warp == 2) MLA_EV(6, G);
            const float gm = fmaxf(xs[row], xs[128 + row]);
            float factor = 1.f;
            if (gm > m_used + kRescaleThreshold) {
                if (pg != it.page_begin) factor = ex2_approx(m_used - gm);
                m_used = gm;
            }
            l_mine *= factor;

            // P of my pages goes into staging slot (message % 4), free once the value CTA has
            // consumed the message four before; every page but the item's last is handed to the
            // shipper at once, the last waits for 1/l below
            // (one loop body for both pages, the code small in the instruction cache: the second
            // page moves into the first one's registers)
            bool hold_last = false;
#pragma unroll 1
            for (int j = 0; j < 2; ++j) {
                if (j >= n_mine || !ok) break;
                if (j == 1) {
#pragma unroll
                    for (int k = 0; k < 64; ++k) sr[0][k] = sr[1][k];
                }
                const int gg = g + 2 * set + j;
                const int slot = gg % kStagingSlots;
                if (gg >= kStagingSlots)
                    ok = MLA_TIMED(8, wait_freed(freed, (uint32_t)(gg - kStagingSlots + 1), w));
                if (!ok) break;
                [[maybe_unused]] const long long tw0 = MLA_TRACE_NOW();
                l_mine += page_softmax(sr[0], p.scale_log2, m_used, smem + kOffScoreStaging + slot * kPBytes + p_row_off,
                                       row);
                const float f_page = (set == 0 && j == 0) ? factor : 1.f;  // O rescale precedes page 0
                if (t0 + j == it.page_end - 1)
                    hold_last = true;
                else
                    stage_message(smem, bars, slot, q4, lane, f_page, 0.f, false, (j ? valid1 : valid0) < 64);
                MLA_TRACE_ADD(10, MLA_TRACE_NOW() - tw0);
            }
            if (last_group) {  // 1/l for the item's last page needs both sets' sums
                xs[256 + set * 128 + row] = l_mine;
                if (MLA_TIMED(13, named_barrier_or(kSoftmaxBarrier, 256, !ok || *w.abort))) return;
                l_total = xs[256 + row] + xs[256 + 128 + row];
                if (hold_last) {
                    const int j = n_mine - 1;
                    const int slot = (g + 2 * set + j) % kStagingSlots;
                    const float f_page = (set == 0 && j == 0) ? factor : 1.f;
                    stage_message(smem, bars, slot, q4, lane, f_page, 1.f / l_total, true, (j ? valid1 : valid0) < 64);
                }
            }
            if (lane == 0 && (warp == 2 || warp == 6)) MLA_EV(warp == 2 ? 7 : 14, G);
            g += npg;
        }
        if (set == 0) {
            const float lse_val = (m_used + log2f(l_total)) * 0.69314718055994531f;
            if (it.slot < 0)
                p.lse[(int64_t)it.seq * 128 + row] = lse_val;
            else
                p.ws_lse[(int64_t)it.slot * 128 + row] = lse_val;
        }
    }
    if (leader) MLA_TRACE_FLUSH(6, 11, 6);
    if (leader) MLA_TRACE_FLUSH(13, 13, 6);
}

// ---------------------------------------------------------------------------- value CTA

__device__ __forceinline__ uint32_t msg_flags(const uint8_t* smem, int buf)
{
    const volatile uint32_t* f = reinterpret_cast<const volatile uint32_t*>(smem + kOffStats + buf * kStatsBytes);
    const int w = kStatsWarpBytes / 4;
    return f[64] | f[w + 64] | f[2 * w + 64] | f[3 * w + 64];
}

// Message acknowledgement (one thread of the value CTA): arms msg_full for each message in
// order (expected bytes; the copies may land before or after) and, as soon as the message has
// landed, tells the score CTA that its staging slot is free (copied).  Keeping this off the MMA
// thread lets the score CTA reuse staging slots without waiting for PV.
__device__ __forceinline__ void value_ack(const Params& p, int item_begin, int item_end, int items_off,
                                          uint32_t bars, const dev::WaitCtx& w)
{
    using namespace dev;
    const uint32_t r_copied = map_to_cta(bars + 8 * kCopied0, 0);
    int g = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int buf = g % kMsgSlots;
            mbar_arrive_expect_tx(bars + 8 * (kMsgFull0 + buf), kMsgBytes);
            if (!wait_phase<true>(bars + 8 * (kMsgFull0 + buf), g / kMsgSlots, w)) return;
            mbar_arrive_remote(r_copied + 8 * buf);
        }
    }
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
            const int s = g % kValueStages, buf = g % kMsgSlots;
            if (!MLA_TIMED(3, wait_phase(bars + 8 * (kFull0 + s), g / kValueStages, w))) goto out;
            MLA_EV(12, g);
            if (!MLA_TIMED(4, wait_phase<true>(bars + 8 * (kMsgFull0 + buf), g / kMsgSlots, w))) goto out;
            MLA_EV(10, g);
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
            MLA_EV(11, g);
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
// item's split partial (fp32).  Lane `lane` of correction warp q4 owns TMEM lane (head)
// 32 q4 + lane.  Each 32-column slice goes through the warp's tile in shared memory: written
// one head row per lane, read back so that consecutive lanes cover consecutive columns of one
// head, and every store instruction writes whole 128-byte lines (four heads at a time in fp32,
// eight in bf16) instead of 16 bytes in each of 32 lines.
template <class KernelParams>  // this kernel's Params, or the FP8 kernel's (same output fields)
__device__ __forceinline__ void write_output(const KernelParams& p, const Item& it, float inv_l, uint32_t tmem,
                                             uint32_t lane_off, uint8_t* tile, int q4, int lane)
{
    using namespace dev;
    float* mine = reinterpret_cast<float*>(tile + lane * kOutTileRowBytes);
#pragma unroll 1
    for (int j = 0; j < 16; ++j) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + 32 * j, r);
        tmem_wait_ld();
#pragma unroll
        for (int v = 0; v < 8; ++v)
            reinterpret_cast<float4*>(mine)[v] =
                make_float4(__uint_as_float(r[4 * v + 0]) * inv_l, __uint_as_float(r[4 * v + 1]) * inv_l,
                            __uint_as_float(r[4 * v + 2]) * inv_l, __uint_as_float(r[4 * v + 3]) * inv_l);
        __syncwarp();
        if (it.slot < 0) {
            // bf16: four lanes per head row (8 columns each), eight rows per instruction
            const int c8 = lane & 3;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int rr = 8 * k + (lane >> 2);
                const float4* src = reinterpret_cast<const float4*>(tile + rr * kOutTileRowBytes) + 2 * c8;
                const float4 a = src[0], b = src[1];
                uint4 o;
                o.x = pack_bf16x2(a.x, a.y);
                o.y = pack_bf16x2(a.z, a.w);
                o.z = pack_bf16x2(b.x, b.y);
                o.w = pack_bf16x2(b.z, b.w);
                *reinterpret_cast<uint4*>(p.o_lat + ((int64_t)it.seq * 128 + 32 * q4 + rr) * 512 + 32 * j + 8 * c8) = o;
            }
        } else {
            // fp32: eight lanes per head row (4 columns each), four rows per instruction
            const int c4 = lane & 7;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int rr = 4 * k + (lane >> 3);
                const float4 a = reinterpret_cast<const float4*>(tile + rr * kOutTileRowBytes)[c4];
                *reinterpret_cast<float4*>(p.ws_o + ((int64_t)it.slot * 128 + 32 * q4 + rr) * 512 + 32 * j + 4 * c4) = a;
            }
        }
        __syncwarp();  // the tile is rewritten by the next slice
    }
}

__device__ __forceinline__ void value_correction(const Params& p, int item_begin, int item_end, int items_off,
                                                 uint8_t* smem, uint32_t bars, uint32_t tmem, const dev::WaitCtx& w,
                                                 int warp, int lane, int tid128)
{
    using namespace dev;
    const int q4 = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    uint8_t* out_tile = smem + kOffOutTile + q4 * kOutTileBytes;
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
            const int buf = g % kMsgSlots;
            if (!MLA_TIMED(7, wait_warp<true>(bars + 8 * (kMsgFull0 + buf), g / kMsgSlots, w))) goto done;
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
                write_output(p, prev, prev_inv_l, tmem, lane_off, out_tile, q4, lane);
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
        write_output(p, prev, prev_inv_l, tmem, lane_off, out_tile, q4, lane);
        MLA_TRACE_ADD(9, MLA_TRACE_NOW() - te0);
    }
done:
    tc_fence_before();
    if (warp == 2 && lane == 0) MLA_TRACE_FLUSH(6, 10, 6);
}

// ---------------------------------------------------------------------------- kernel

// 11 warps: three SM sub-partitions hold three of them, and a sub-partition's 16K registers then
// allow at most 3 x 32 x 168.
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(168)
decode_bf16_kernel(const __grid_constant__ CUtensorMap tm_pool, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_qc, const __grid_constant__ CUtensorMap tm_wuk, const Params p)
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
            mbar_init(bars + 8 * (kSFree0 + b), 8);        // one arrive per softmax warp
            mbar_init(bars + 8 * (kOReady0 + b), 128);
            mbar_init(bars + 8 * (kODrain0 + b), 1);
        }
        for (int b = 0; b < kMsgSlots; ++b) {
            mbar_init(bars + 8 * (kMsgFree0 + b), 1 + 4);  // PV commit + four correction warps
            mbar_init(bars + 8 * (kMsgFull0 + b), 1);      // the MMA thread's arm + the copies' bytes
            mbar_init(bars + 8 * (kCopied0 + b), 1);       // the value MMA thread saw the message land
        }
        mbar_init(bars + 8 * kQReady, 8);                  // one arrive per softmax warp
        for (int s = 0; s < kStagingSlots; ++s) mbar_init(bars + 8 * (kStgReady0 + s), 4);  // one set's warps
        *reinterpret_cast<volatile uint32_t*>(smem + kOffStgFreed) = 0;
        mbar_init(bars + 8 * kDrain, 1);
        mbar_init(bars + 8 * (kAbsFull0 + 0), 1);
        mbar_init(bars + 8 * (kAbsFull0 + 1), 1);
        mbar_init(bars + 8 * kAbsDone, 1);
        mbar_init(bars + 8 * kAbsEpi, 4);  // one arrive per epilogue warp
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

    if (!*abort_flag && p.absorb_sync) {
        absorb_jobs(&tm_qc, &tm_wuk, p, sbase, bars, tmem, w, warp, lane);
        tc_fence_before();
        __syncthreads();  // the prologue's tiles and TMEM columns are free again
        tc_fence_after();
    }
    if (!*abort_flag) {
        const int n_clusters = p.plan[kHdrClusters];
        const int items_off = p.plan[kHdrItemsOff];
        const int cl_off = p.plan[kHdrClusterOff];
        const int item_begin = cluster < n_clusters ? p.plan[cl_off + cluster] : 0;
        const int item_end = cluster < n_clusters ? p.plan[cl_off + cluster + 1] : 0;
        if (rank == 0) {
            if (warp == 0)
                score_producer(&tm_pool, &tm_q, p, item_begin, item_end, items_off, sbase, bars, w, lane);
            else if (warp == 1) {
                if (lane == 0) score_mma(p, item_begin, item_end, items_off, sbase, bars, tmem, w);
            } else if (warp == kShipperWarp) {
                if (lane == 0) score_shipper(p, item_begin, item_end, items_off, smem, sbase, bars, w);
                else if (lane == 1) score_tracker(p, item_begin, item_end, items_off, smem, bars, w);
            } else if (warp >= 2 && warp < 10)
                score_softmax(p, item_begin, item_end, items_off, smem, sbase, bars, tmem, w, warp, lane);
        } else {
            if (warp == 0)
                run_producer(&tm_pool, p, item_begin, item_end, items_off, sbase, bars, 8, kValueStages,
                             kValueStageBytes, l2_policy_evict_first(), w, lane);
            else if (warp == 1) {
                if (lane == 0) value_mma(p, item_begin, item_end, items_off, smem, sbase, bars, tmem, w);
            } else if (warp == kAckWarp) {
                if (lane == 0) value_ack(p, item_begin, item_end, items_off, bars, w);
            } else if (warp >= 2 && warp < 6)
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
