// decode_fp8.cuh -- the paged MLA decode of decode.cuh for a latent cache stored as FP8 e4m3
// with one fp32 scale per token (the RoPE key k_R stays bf16), on the e4m3 tensor cores.
//
// What it computes: as decode.cuh, with each cached latent row c_t = float(c8_t) * sigma_t
// (page 1, "撕開 DeepSeek MLA 源碼", section 5, on FP8 caches).  Nothing converts the cache:
// the e4m3 rows go from HBM through TMA straight into the operand tiles of kind::f8f6f4 MMAs.
//
// Scores.  s[h,t] = scale * (q_abs[h] . c_t + q_R[h] . k_R[t])
//                 = scale * sigma_t * 2^-e_h * (q~[h] . c8_t + q_R[h] 2^e_h . k_R[t] / sigma_t)
// where q~[h] = q_abs[h] * 2^e_h, the power of two 2^e_h putting row h's largest magnitude in
// [128, 256).  q~ is held as a pair of e4m3 matrices q_hi = e4m3(q~), q_lo = e4m3(q~ - q_hi).
// A bf16 value has eight significant bits; rounding it to four leaves a residual that is a
// multiple of its last bit and at most eight of them, which four bits hold, so q_hi + q_lo = q~
// exactly wherever |q~| >= 1/4 (below, within 2^-10); QK runs one e4m3 MMA for each, which at
// twice the bf16 rate costs the tensor time of one bf16 MMA.  A converter warp divides each
// page's k_R rows by sigma_t in shared memory (bf16x2 fused multiply-adds by a two-part 1/sigma,
// one rounding), so that the RoPE MMA (bf16, q_R 2^e_h) accumulates into the same fp32 scores.
// That rounding, 2^-9 relative per element, is the path's main score noise (a power-of-two
// sigma_t makes it exact; a second bf16 part would need 32 KB of shared memory or 256 TMEM
// columns that the layout below does not have).  The softmax then scales column t
// by sigma_t and row h by 2^-e_h.
//
// Output.  o[h] = sum_t p[h,t] sigma_t c8_t / l[h].  The PV operand is P~ = p * sigma_t * g,
// with g a power of two per item chosen from the item's largest sigma so that P~ <= 448, split
// the same way into e4m3 hi + lo and packed into one 128-byte row per head (bytes 0-63: hi of
// the page's 64 tokens, bytes 64-127: lo).  The score CTA ships p as bf16 (with sigma_t g per
// token); four warps of the value CTA form P~ in place before PV.  PV runs e4m3 MMAs on the raw c8 page (B operand
// MN-major) and the last page's 1/(g l) normalises.  The lazy-rescale threshold is 4 (log2
// units), so p <= 16 and the typical P~ stays above 1/4, where the pair is exact to 2^-8; below
// that its absolute error is at most 2^-10, against a running maximum of at least 14.
//
// Bytes per cached token: 512 (e4m3) + 4 (scale) + 128 (k_R) = 644, against 1,152 in bf16.
//
// Layout of the pair (sm_103a), as decode.cuh:
//   rank 0, the score CTA: q_hi and q_lo in TMEM (128 columns each, four e4m3 per 32-bit
//     column), the scores of four pages in the other 256 columns.  Per four-page group the four
//     128-column boxes of c8 (8 KB per page, 32 KB per K-chunk) stream through a three-slot
//     ring, and the k_R boxes (8 KB per page) through a buffer of their own.  An item's bf16
//     q_abs rows go through the same ring ahead of its pages (four entries of two 64-dim boxes);
//     the MMA thread copies them into the score columns (tcgen05.cp) and the softmax warps turn
//     them into the e4m3 pair, so the query costs coalesced TMA traffic and no register file.  Eight softmax warps, the shipper and tracker as in
//     the bf16 kernel; warp 11 turns k_R into k_R / sigma and writes the per-token factors the
//     softmax needs (sigma * scale * log2(e), sigma * g).
//   rank 1, the value CTA: O in TMEM (512 columns), four 32 KB c8 page stages, PV from P~;
//     warps 7-10 form P~ from the shipped p.
//
// Pipelines: those of decode.cuh, plus
//   kr_landed             the group's k_R boxes have landed in the k_R buffer (TMA bytes;
//                         waited by warp 11, which loads them)
//   kr_full / kr_empty    k_R / sigma is in place (warp 11) / the MMA has read it (commit)
//   sig_ready             counter: groups whose token factors are written (warp 11)
//   p_ready[4]            the value CTA's P~ of a message is written (its four converter warps)
//   q_raw                 the item's bf16 query is in the score columns (the MMA thread's commit
//                         after its copies; waited by the softmax warps)
#pragma once
#include "decode.cuh"

namespace mla {
namespace decode_fp8 {

using decode::Item;
using decode::kTraceSlots;
using decode::load_item;
using decode::wait_freed;
using decode::write_output;
using decode::kOutTileBytes;
#ifdef MLA_DECODE_TRACE
using decode::kEvBase;
using decode::kEvSlots;
#endif

constexpr int kThreads = 384;                     // 12 warps, roles in the kernel below
constexpr int kShipperWarp = 10;
constexpr int kKrWarp = 11;                       // score CTA: k_R / sigma, token factors
constexpr int kAckWarp = 6;                       // value CTA: message acknowledgements
constexpr int kPConvWarp0 = 7;                    // value CTA: warps 7-10 turn P into P~ (e4m3 pair)
constexpr int kChunkStages = 3;                   // score CTA: c8 K-chunk ring
constexpr int kQueryEntries = 4;                  // ring entries carrying an item's q_abs (two 16 KB boxes each)
constexpr int kValueStages = 4;
constexpr int kMaxStages = 4;
constexpr int kStagingSlots = 4;
constexpr int kMsgSlots = 4;
constexpr int kBoxBytes = 64 * 128;               // 64 tokens x 128 bytes (128 e4m3 or 64 bf16)
constexpr int kC8Boxes = 4;                       // a c8 row: four 128-column boxes
constexpr int kChunksPerGroup = kC8Boxes;         // c8 K-chunks per group (k_R has its own buffer)
constexpr int kGroupPages = 4;                    // pages per score MMA (N = 256)
constexpr int kChunkBytes = kGroupPages * kBoxBytes;    // 32 KB
constexpr int kValueStageBytes = kC8Boxes * kBoxBytes;  // 32 KB: one page of c8
constexpr int kPBytes = 128 * 128;                // P~: 128 heads x (64 hi + 64 lo) e4m3
// Per message statistics, one block per softmax warp: factor[32], inv_l[32], a 16-byte flags
// slot (as decode.cuh), then sig_p of 16 of the page's tokens (warp k: tokens 16k..16k+15).
constexpr int kStatsWarpBytes = 128 + 128 + 16 + 64;
constexpr int kSigPWord = 68;                     // float index of sig_p in a warp's block
constexpr int kStatsBytes = 4 * kStatsWarpBytes;
constexpr int kPWarpBytes = kPBytes / 4;
constexpr int kMsgBytes = kPBytes + kStatsBytes;
constexpr int kSigSlots = 4;                      // token factors of four groups
constexpr int kSigGroupBytes = 2 * 256 * 4 + 16;  // sig_s[256], sig_p[256], g
// score CTA
constexpr int kOffQR = 0;
constexpr int kOffChunks = kOffQR + 128 * 128;
constexpr int kOffKr = kOffChunks + kChunkStages * kChunkBytes;   // k_R of one group (32 KB)
constexpr int kOffScoreStaging = kOffKr + kChunkBytes;
constexpr int kOffStatsStaging = kOffScoreStaging + kStagingSlots * kPBytes;
constexpr int kOffXchg = kOffStatsStaging + kStagingSlots * kStatsBytes;
constexpr int kOffSig = kOffXchg + 4 * 2 * 128 * 4;
constexpr int kScoreEnd = kOffSig + kSigSlots * kSigGroupBytes;
// value CTA
constexpr int kOffP = kValueStages * kValueStageBytes;
constexpr int kOffStats = kOffP + kMsgSlots * kPBytes;
// one 32 x 32 fp32 transpose tile per correction warp for the output write-out (as decode.cuh)
constexpr int kOffOutTile = (kOffStats + kMsgSlots * kStatsBytes + 15) / 16 * 16;
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
    kKrLanded = kStgReady0 + kStagingSlots,
    kKrFull = kKrLanded + 1,
    kKrEmpty = kKrFull + 1,
    kPReady0 = kKrEmpty + 1,
    kQRaw = kPReady0 + kMsgSlots,
    kNumBars = kQRaw + 1
};

constexpr int kOffTmemHolder = kOffBars + 8 * kNumBars;
constexpr int kOffAbort = kOffTmemHolder + 4;
constexpr int kOffStgFreed = kOffAbort + 4;     // score CTA: messages whose staging slot may be reused
constexpr int kOffSigReady = kOffStgFreed + 4;  // score CTA: groups whose token factors are written
constexpr int kSmemBytes = ((kOffSigReady + 4 + 127) / 128) * 128;
static_assert(kOffChunks % 1024 == 0 && kOffKr % 1024 == 0 && kOffP % 1024 == 0 && kOffScoreStaging % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");
static_assert(kOffSig % 16 == 0 && kSigGroupBytes % 16 == 0, "token factors are read as float4");
static_assert(kChunkStages <= kMaxStages && kValueStages <= kMaxStages, "barrier slots per ring");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kStatsWarpBytes % 16 == 0 && kPWarpBytes % 16 == 0, "bulk copies move multiples of 16 bytes");

// TMEM columns
constexpr uint32_t kQHiCol = 0;    // score CTA: q_hi, 128 columns (512 e4m3 per lane)
constexpr uint32_t kQLoCol = 128;  // score CTA: q_lo
constexpr uint32_t kSCol = 256;    // score CTA: the 256-column score buffer (four pages)
constexpr uint32_t kTmemCols = 512;

constexpr float kRescaleThreshold = 4.0f;  // log2 units: p stays <= 16
constexpr float kPTildeTop = 28.0f;        // 448 / 16: P~ bound divided by the largest p
constexpr uint32_t kSoftmaxBarrier = 1;    // named barrier of the eight softmax warps

struct Params {
    const int32_t* plan;
    const __nv_bfloat16* q_abs;  // [B][128][512]
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
    const float* kv_scale;       // [pages][64] per-token scale of the e4m3 latent rows
    long long* trace;            // instrumented builds only, else null
};

// ---------------------------------------------------------------------------- e4m3 helpers

// kind::f8f6f4 with e4m3 A and B (format 0) and fp32 D: the bit layout of idesc_f16.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool a_mn_major, bool b_mn_major)
{
    return dev::idesc_f16(M, N, a_mn_major, b_mn_major);
}

// D[tmem] (+)= A * B with e4m3 operands: A from tensor memory (four e4m3 along K per 32-bit
// column) or from a shared-memory descriptor, B from a shared-memory descriptor.
__device__ __forceinline__ void mma_ts_e4m3(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_ss_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
        : "memory");
}

// Four values -> their e4m3 pair, little-endian bytes x0..x3: hi = e4m3(x) (through f16, which
// holds x to 2^-11), lo = e4m3(x - hi) (the f16 difference is exact).  |x| <= 448.
__device__ __forceinline__ void split_e4m3x4(float x0, float x1, float x2, float x3, uint32_t& hi, uint32_t& lo)
{
    asm("{\n\t.reg .b32 h01, h23, b01, b23, r01, r23;\n\t.reg .b16 e01, e23, l01, l23;\n\t"
        "cvt.rn.f16x2.f32 h01, %3, %2;\n\t"
        "cvt.rn.f16x2.f32 h23, %5, %4;\n\t"
        "cvt.rn.satfinite.e4m3x2.f16x2 e01, h01;\n\t"
        "cvt.rn.satfinite.e4m3x2.f16x2 e23, h23;\n\t"
        "cvt.rn.f16x2.e4m3x2 b01, e01;\n\t"
        "cvt.rn.f16x2.e4m3x2 b23, e23;\n\t"
        "sub.rn.f16x2 r01, h01, b01;\n\t"
        "sub.rn.f16x2 r23, h23, b23;\n\t"
        "cvt.rn.satfinite.e4m3x2.f16x2 l01, r01;\n\t"
        "cvt.rn.satfinite.e4m3x2.f16x2 l23, r23;\n\t"
        "mov.b32 %0, {e01, e23};\n\t"
        "mov.b32 %1, {l01, l23};\n\t}"
        : "=r"(hi), "=r"(lo)
        : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// 2^e as a float, e clamped to [-64, 64].
__device__ __forceinline__ float exp2i(int e)
{
    e = max(-64, min(64, e));
    return __int_as_float((127 + e) << 23);
}

// ---------------------------------------------------------------------------- TMA producers

// Value CTA: each page's 512 c8 columns as four 128-byte-wide boxes into a four-stage ring.
__device__ __forceinline__ void value_producer(const CUtensorMap* tm_c8, const Params& p, int item_begin,
                                               int item_end, int items_off, uint32_t sbase, uint32_t bars,
                                               const dev::WaitCtx& w, int lane)
{
    using namespace dev;
    const uint64_t policy = l2_policy_evict_first();  // the score CTA has read these pages already
    if (lane == 0) tma_prefetch_desc(tm_c8);
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
                    const int s = g % kValueStages;
                    if (g >= kValueStages) ok = wait_phase_ool(bars + 8 * (kEmpty0 + s), g / kValueStages - 1, w);
                    if (ok) {
                        const uint32_t full = bars + 8 * (kFull0 + s);
                        const uint32_t dst = sbase + s * kValueStageBytes;
                        mbar_arrive_expect_tx(full, kValueStageBytes);
                        // an out-of-range page id reads as zeros (TMA fills outside the tensor)
                        for (int x = 0; x < kC8Boxes; ++x)
                            tma_load_3d(dst + x * kBoxBytes, tm_c8, full, 128 * x, 0, pj, policy);
                        MLA_EV(16, g);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                ++g;
            }
        }
    }
    if (lane == 0 && *w.abort) {  // loads still in flight must land before the CTA exits
        for (int k = (g > kValueStages ? g - kValueStages : 0); k < g; ++k)
            drain_phase(bars + 8 * (kFull0 + k % kValueStages), k / kValueStages, w.timeout_ns);
    }
}

// Score CTA: chunk j of a four-page group holds c8 box j (128 columns) of the group's pages in
// rows 0-63, 64-127, 128-191, 192-255, through a three-slot ring; the k_R box has a buffer of
// its own that warp 11 fills (see kr_convert).
__device__ __forceinline__ void score_producer(const CUtensorMap* tm_c8, const CUtensorMap* tm_q, const Params& p,
                                               int item_begin, int item_end, int items_off, uint32_t sbase,
                                               uint32_t bars, const dev::WaitCtx& w, int lane)
{
    using namespace dev;
    const uint64_t policy = l2_policy_evict_last();  // the value CTA reads these pages next
    if (lane == 0) {
        tma_prefetch_desc(tm_c8);
        tma_prefetch_desc(tm_q);
    }
    int s = 0, phase = 0, c = 0;
    bool ok = true;
    for (int i = item_begin; i < item_end && ok; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        const int32_t* bt = p.block_table + (int64_t)it.table_row * p.max_pages;
        if (lane == 0) {
            // the item's q_abs rows (128 heads x 512 dims) as four ring entries of two 64-dim
            // boxes each, ahead of its pages; the softmax warps read and release them
            if (i == item_begin) griddep_wait();  // q_abs comes from the kernel launched before
            for (int j = 0; j < kQueryEntries && ok; ++j, ++c) {
                if (c >= kChunkStages) ok = wait_phase_ool(bars + 8 * (kEmpty0 + s), phase - 1, w);
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
                    for (int box = 0; box < kChunksPerGroup && ok; ++box, ++c) {
                        if (c >= kChunkStages) ok = wait_phase_ool(bars + 8 * (kEmpty0 + s), phase - 1, w);
                        if (!ok) break;
                        const uint32_t dst = sbase + kOffChunks + s * kChunkBytes;
                        const uint32_t full = bars + 8 * (kFull0 + s);
                        mbar_arrive_expect_tx(full, npg * kBoxBytes);
                        for (int q = 0; q < npg; ++q)
                            tma_load_3d(dst + q * kBoxBytes, tm_c8, full, 128 * box, 0, pages[q], policy);
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
}

// ---------------------------------------------------------------------------- score CTA

// Warp 11.  Per item, g = 2^floor(log2(28 / max sigma)) over the item's tokens (so that P~ =
// p sigma g <= 16 * 28 = 448).  Per four-page group: once the MMA has read the previous group's
// k_R (kr_empty), load this group's k_R boxes into the k_R buffer (TMA, kr_landed); meanwhile
// write the token factors for the softmax (sig_s = sigma * scale * log2(e) and sig_p = sigma *
// g, both 0 past the sequence end, and g) into factor slot G % 4; then divide every k_R row by
// its token's sigma in place and arrive on kr_full for the MMA.  Factor slot G % 4 is free when
// it is written: the MMA had read k_R of group G - 1, so it had started group G - 1, which it
// does after s_free of group G - 2; every softmax warp had finished group G - 3 then, and slot
// G % 4 last held group G - 4.  Owning the k_R loads keeps them off the c8 ring: the load for
// group G + 1 starts as soon as the MMA has taken group G's k_R.
__device__ __forceinline__ void kr_convert(const CUtensorMap* tm_kr, const Params& p, int item_begin, int item_end,
                                           int items_off, uint8_t* smem, uint32_t sbase, uint32_t bars,
                                           const dev::WaitCtx& w, int lane)
{
    using namespace dev;
    uint32_t* sig_ready = reinterpret_cast<uint32_t*>(smem + kOffSigReady);
    const uint64_t policy = l2_policy_evict_first();  // nobody else reads k_R
    if (lane == 0) tma_prefetch_desc(tm_kr);
    int G = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        const int32_t* bt = p.block_table + (int64_t)it.table_row * p.max_pages;
        // largest scale over the item's tokens: lane k takes pages k, k + 32, ...; a page's
        // sixteen scale loads are in flight together, and the next page id is loaded before them,
        // so each page costs one memory round trip
        const auto page_at = [&](int pg) {
            return (pg < it.page_end && pg < p.max_pages) ? __ldg(bt + pg) : -1;
        };
        float smax = 0.f;
        int page = page_at(it.page_begin + lane);
        for (int pg = it.page_begin + lane; pg < it.page_end; pg += 32) {
            const int next = page_at(pg + 32);
            if (page >= 0 && page < p.num_pool_pages) {  // a bad id is reported by the producers
                const int valid = min(64, it.seq_len - 64 * pg);
                const float4* sc = reinterpret_cast<const float4*>(p.kv_scale + (int64_t)page * 64);
                float4 x[16];
#pragma unroll
                for (int v = 0; v < 16; ++v) x[v] = __ldg(sc + v);
#pragma unroll
                for (int v = 0; v < 16; ++v) {
                    if (4 * v + 0 < valid) smax = fmaxf(smax, x[v].x);
                    if (4 * v + 1 < valid) smax = fmaxf(smax, x[v].y);
                    if (4 * v + 2 < valid) smax = fmaxf(smax, x[v].z);
                    if (4 * v + 3 < valid) smax = fmaxf(smax, x[v].w);
                }
            }
            page = next;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        float g = 1.f;
        if (smax > 0.f) {
            int ex;
            frexpf(kPTildeTop / smax, &ex);  // 28 / smax in [2^(ex-1), 2^ex)
            g = exp2i(ex - 1);
        }
        for (int pg = it.page_begin; pg < it.page_end; pg += kGroupPages, ++G) {
            const int npg = min(kGroupPages, it.page_end - pg);
            float* sig = reinterpret_cast<float*>(smem + kOffSig + (G % kSigSlots) * kSigGroupBytes);
            // Token t = lane + 32 k of the group (row t of the k_R buffer) sits in page k / 2 at
            // slot lane + 32 (k & 1).  All page ids, then all eight scales, are loaded before any
            // is used, so the group costs two memory round trips.
            int page_mine = 0;
            if (lane < npg) {
                page_mine = pg + lane < p.max_pages ? __ldg(bt + pg + lane) : -1;
                if (page_mine < 0 || page_mine >= p.num_pool_pages) page_mine = -1;  // reported by the producers
            }
            int pages[kGroupPages];
#pragma unroll
            for (int q = 0; q < kGroupPages; ++q) pages[q] = __shfl_sync(0xffffffffu, page_mine, q);
            // the MMA has read the previous group's k_R: load this group's (a bad page id, -1 here,
            // reads zeros: TMA fills outside the tensor)
            if (G >= 1 && !wait_warp_ool(bars + 8 * kKrEmpty, G - 1, w)) return;
            if (lane == 0) {
                const uint32_t landed = bars + 8 * kKrLanded;
                mbar_arrive_expect_tx(landed, npg * kBoxBytes);
                for (int q = 0; q < npg; ++q)
                    tma_load_3d(sbase + kOffKr + q * kBoxBytes, tm_kr, landed, 0, 0, pages[q], policy);
            }
            float sigma[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                sigma[k] = __ldg(p.kv_scale + (int64_t)max(pages[k >> 1], 0) * 64 + lane + 32 * (k & 1));
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int t = lane + 32 * k, q = k >> 1;
                const bool in_seq = q < npg && 64 * (pg + q) + (t & 63) < it.seq_len;
                const bool valid = in_seq && pages[q] >= 0;
                // a zero scale (a zero latent row) enters the score side as 2^-64, so that k_R /
                // sigma stays finite and sigma (q . c8 + q_R . k_R / sigma) is still q_R . k_R;
                // a slot past the sequence end gets NaN, which the softmax's maximum skips
                // (fmaxf returns the other operand), so the maximum needs no mask
                sig[t] = valid ? fmaxf(sigma[k], 5.421011e-20f) * p.scale_log2 : (in_seq ? 0.f : __int_as_float(0x7fc00000));
                sig[256 + t] = valid ? sigma[k] * g : 0.f;
            }
            if (lane == 0) sig[512] = g;
            if (lane == 0) MLA_EV(18, G);
            if (!wait_warp_ool(bars + 8 * kKrLanded, G, w)) {
                if (lane == 0) drain_phase(bars + 8 * kKrLanded, G, w.timeout_ns);  // the load in flight
                return;
            }
            if (lane == 0) MLA_EV(19, G);
            uint8_t* rows = smem + kOffKr;
            const float inv_scale = 1.f / p.scale_log2;
#pragma unroll 1
            for (int t = lane; t < 64 * npg; t += 32) {
                // 1 / sigma_t (sigma >= 2^-64); a slot past the sequence end gets 0 (its score is masked)
                const float ss = sig[t];
                const float inv = ss > 0.f ? 1.f / (ss * inv_scale) : 0.f;
                // 1/sigma as a bf16 pair inv_hi + inv_lo; k * inv_hi + (k * inv_lo) in one fused
                // bf16x2 multiply-add rounds once (the inner product is 2^-8 smaller, so its own
                // rounding is below 2^-16 of the result)
                const float inv_hi_f = __bfloat162float(__float2bfloat16_rn(inv));
                const uint32_t inv_hi = pack_bf16x2(inv_hi_f, inv_hi_f);
                const uint32_t inv_lo = pack_bf16x2(inv - inv_hi_f, inv - inv_hi_f);
                uint8_t* row = rows + t * 128;  // 16-byte chunks in any order: the divide is per element
                uint4 v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = *reinterpret_cast<const uint4*>(row + (((j + lane) & 7) << 4));
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    v[j].x = fma_bf16x2(v[j].x, inv_hi, mul_bf16x2(v[j].x, inv_lo));
                    v[j].y = fma_bf16x2(v[j].y, inv_hi, mul_bf16x2(v[j].y, inv_lo));
                    v[j].z = fma_bf16x2(v[j].z, inv_hi, mul_bf16x2(v[j].z, inv_lo));
                    v[j].w = fma_bf16x2(v[j].w, inv_hi, mul_bf16x2(v[j].w, inv_lo));
                    *reinterpret_cast<uint4*>(row + (((j + lane) & 7) << 4)) = v[j];
                }
            }
            fence_proxy_async_cta();  // the k_R rows are read by the MMA (async proxy)
            __syncwarp();
            if (lane == 0) {
                st_release_u32(sig_ready, (uint32_t)(G + 1));
                mbar_arrive(bars + 8 * kKrFull);
                MLA_EV(13, G);
            }
        }
    }
}

// QK of a four-page group: S[128 heads x N tokens] accumulated over k_R and the four c8
// K-chunks: k_R / sigma (its own buffer) against q_R 2^e (shared memory), four bf16 MMAs of K =
// 16; then each c8 chunk against q_hi and q_lo (TMEM, "TS"), eight e4m3 MMAs of K = 32.
__device__ __forceinline__ void score_mma(const Params& p, int item_begin, int item_end, int items_off, uint32_t sbase,
                                          uint32_t bars, uint32_t tmem, const dev::WaitCtx& w)
{
    using namespace dev;
    const uint64_t chunk_desc0 = smem_desc(sbase + kOffChunks, 16, 1024);
    const uint64_t kr_desc = smem_desc(sbase + kOffKr, 16, 1024);
    const uint64_t qr_desc = smem_desc(sbase + kOffQR, 16, 1024);
    const uint32_t full0 = bars + 8 * kFull0, empty0 = bars + 8 * kEmpty0;
    const uint32_t d = tmem + kSCol;
    int s = 0, phase = 0, G = 0, n_item = 0;
    for (int i = item_begin; i < item_end; ++i, ++n_item) {
        const Item it = load_item(p.plan, items_off, i);
        // The item's bf16 query rows into the score columns (free once the softmax has read the
        // previous item's last scores): dims 64 k .. 64 k + 63 -> columns 32 k .. 32 k + 31 of lane
        // h for head h; the softmax warps turn them into the e4m3 pair (q_ready).
        if (n_item > 0 && !wait_phase_ool(bars + 8 * kSFree0, G - 1, w)) goto out;
#pragma unroll 1
        for (int j = 0; j < kQueryEntries; ++j) {
            if (!wait_phase_ool(full0 + 8 * s, phase, w)) goto out;
            tc_fence_after();
            const uint64_t src = smem_desc(sbase + kOffChunks + s * kChunkBytes, 16, 1024);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4)
                    tmem_cp_128x256b(d + 64 * j + 32 * h + 8 * k4,
                                     src + (uint64_t)(h * ((kChunkBytes / 2) >> 4) + 2 * k4));
            mma_commit(empty0 + 8 * s);
            if (++s == kChunkStages) {
                s = 0;
                ++phase;
            }
        }
        mma_commit(bars + 8 * kQRaw);
        if (!wait_phase_ool(bars + 8 * kQReady, n_item, w)) goto out;
        tc_fence_after();
        for (int pg = it.page_begin; pg < it.page_end; pg += kGroupPages, ++G) {
            const int npg = min(kGroupPages, it.page_end - pg);
            const uint32_t idesc8 = idesc_e4m3(128, 64 * npg, false, false);
            const uint32_t idesc16 = idesc_bf16(128, 64 * npg, false, false);
            if (G >= 1 && !wait_phase_ool(bars + 8 * kSFree0, G - 1, w)) goto out;
            MLA_EV(3, G);
            if (!wait_phase_ool(bars + 8 * kKrFull, G, w)) goto out;
            MLA_EV(1, 5 * G);
            tc_fence_after();
            mma_ss(d, qr_desc, kr_desc, idesc16, 0u);
            mma_ss(d, qr_desc + 2, kr_desc + 2, idesc16, 1u);
            mma_ss(d, qr_desc + 4, kr_desc + 4, idesc16, 1u);
            mma_ss(d, qr_desc + 6, kr_desc + 6, idesc16, 1u);
            mma_commit(bars + 8 * kKrEmpty);
#pragma unroll 1
            for (int box = 0; box < kChunksPerGroup; ++box) {
                if (!wait_phase_ool(full0 + 8 * s, phase, w)) goto out;
                MLA_EV(1, 5 * G + 1 + box);
                tc_fence_after();
                const uint64_t b0 = chunk_desc0 + (uint64_t)(s * (kChunkBytes >> 4));
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    const uint32_t a0 = tmem + (part ? kQLoCol : kQHiCol) + 32 * box;
                    mma_ts_e4m3(d, a0, b0, idesc8, 1u);
                    mma_ts_e4m3(d, a0 + 8, b0 + 2, idesc8, 1u);
                    mma_ts_e4m3(d, a0 + 16, b0 + 4, idesc8, 1u);
                    mma_ts_e4m3(d, a0 + 24, b0 + 6, idesc8, 1u);
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
}

// The query of row `row`: the MMA thread has copied the item's bf16 q_abs rows into the score
// columns (column k of lane h: dims 2k, 2k + 1 of head h; commit on q_raw).  Set k reads its
// dims 256k..256k+255 (columns 128k..128k+127) twice: once for the largest magnitude, which the
// sets agree on through `mx_xchg` (one word per row and set) and which sets e (bf16 magnitudes
// order as their 15-bit patterns), and once to convert them, times 2^e, into the e4m3 pair in
// TMEM columns 64k.. of q_hi and of q_lo.  Set 0 writes q_R 2^e (exact) to row `row` of the
// K-major, 128-byte-swizzled q_R tile.  *r_h = 2^-e.  Both sets reach the barrier, so a failed
// wait makes both return false.
__device__ __noinline__ bool load_query(const Params& p, int seq, int row, int set, int n_item, uint32_t bars,
                                        uint32_t taddr, uint8_t* qr_smem, uint32_t* mx_xchg, const dev::WaitCtx& w,
                                        float* r_h)
{
    using namespace dev;
    const uint32_t raw = taddr + kSCol + 128 * set;
    uint4 qrv[8];  // set 0: q_R of the row, loaded while the query copies land
    if (set == 0) {
        const uint4* qr = reinterpret_cast<const uint4*>(p.q_r + ((int64_t)seq * 128 + row) * 64);
#pragma unroll
        for (int v = 0; v < 8; ++v) qrv[v] = __ldg(qr + v);
    }
    const bool ok = wait_warp_ool(bars + 8 * kQRaw, n_item, w);
    uint32_t mx = 0;
    if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            tmem_ld32(raw + 32 * j, r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) mx = max(mx, max(r[k] & 0x7FFFu, (r[k] >> 16) & 0x7FFFu));
        }
    }
    mx_xchg[set * 128 + row] = mx;
    if (named_barrier_or(kSoftmaxBarrier, 256, !ok || *w.abort)) return false;
    mx = max(mx_xchg[row], mx_xchg[128 + row]);
    // max |q| in [2^E, 2^(E+1)) with E = exponent field - 127; 2^(7-E) maps it into [128, 256)
    const int e = (mx == 0) ? 0 : max(-64, min(64, 7 - ((int)(mx >> 7) - 127)));
    const float sc = exp2i(e);
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {  // 64 dims -> 16 TMEM columns of q_hi and of q_lo
        uint32_t r[32], hi[16], lo[16];
        tmem_ld32(raw + 32 * j, r);
        tmem_wait_ld();
#pragma unroll
        for (int v = 0; v < 16; ++v)
            split_e4m3x4(bf16_lo(r[2 * v]) * sc, bf16_hi(r[2 * v]) * sc, bf16_lo(r[2 * v + 1]) * sc,
                         bf16_hi(r[2 * v + 1]) * sc, hi[v], lo[v]);
        tmem_st16(taddr + kQHiCol + 64 * set + 16 * j, hi);
        tmem_st16(taddr + kQLoCol + 64 * set + 16 * j, lo);
    }
    if (set == 0) {
        uint8_t* dst = qr_smem + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            uint4 x = qrv[v];
            x.x = pack_bf16x2(bf16_lo(x.x) * sc, bf16_hi(x.x) * sc);
            x.y = pack_bf16x2(bf16_lo(x.y) * sc, bf16_hi(x.y) * sc);
            x.z = pack_bf16x2(bf16_lo(x.z) * sc, bf16_hi(x.z) * sc);
            x.w = pack_bf16x2(bf16_lo(x.w) * sc, bf16_hi(x.w) * sc);
            *reinterpret_cast<uint4*>(dst + ((v ^ (row & 7)) << 4)) = x;
        }
        fence_proxy_async_cta();  // read by the MMA (async proxy)
    }
    tmem_wait_st();
    *r_h = exp2i(-e);
    return true;
}

// Scales one page of raw scores in registers in place, y[t] = S[t] * sig_s[t] (sig_s = sigma_t *
// scale * log2(e): log2 units before the row factor), and returns their row max over the slots
// before the sequence end: past it sig_s is NaN, so y is NaN whatever the raw score, and fmaxf
// skips it.
__device__ __forceinline__ float page_scale_max(uint32_t (&sr)[64], const float* sig_s)
{
    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int v = 0; v < 16; ++v) {
        const float4 f = *reinterpret_cast<const float4*>(sig_s + 4 * v);
        const int j = 4 * v;
        const float y0 = __uint_as_float(sr[j + 0]) * f.x, y1 = __uint_as_float(sr[j + 1]) * f.y;
        const float y2 = __uint_as_float(sr[j + 2]) * f.z, y3 = __uint_as_float(sr[j + 3]) * f.w;
        sr[j + 0] = __float_as_uint(y0);
        sr[j + 1] = __float_as_uint(y1);
        sr[j + 2] = __float_as_uint(y2);
        sr[j + 3] = __float_as_uint(y3);
        m4[0] = fmaxf(m4[0], y0);
        m4[1] = fmaxf(m4[1], y1);
        m4[2] = fmaxf(m4[2], y2);
        m4[3] = fmaxf(m4[3], y3);
    }
    return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}

// Softmax of one page scaled by page_scale_max: p = 2^(y[t] 2^-e - m) (0 past the sequence end),
// written as bf16 into this thread's row of the swizzled staging tile (16-byte chunk c of the row
// goes to chunk c ^ (row & 7)), the layout of the bf16 kernel.  The value CTA scales it by
// sigma_t g and splits it into the e4m3 pair.  Returns the row sum of p.
__device__ __forceinline__ float page_softmax(const uint32_t (&sr)[64], float r_h, float m_used, uint8_t* stage_row,
                                              int row)
{
    using namespace dev;
    float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint32_t pk[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = 8 * c + 2 * q;
            // past the sequence end y is NaN: fmaxf(NaN, -inf) = -inf and 2^-inf = 0
            const float p0 = ex2_approx(fmaxf(fmaf(__uint_as_float(sr[j]), r_h, -m_used), -INFINITY));
            const float p1 = ex2_approx(fmaxf(fmaf(__uint_as_float(sr[j + 1]), r_h, -m_used), -INFINITY));
            pk[q] = pack_bf16x2(p0, p1);
            l4[(2 * q) & 3] += p0;
            l4[(2 * q + 1) & 3] += p1;
        }
        *reinterpret_cast<uint4*>(stage_row + ((c ^ (row & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    return (l4[0] + l4[1]) + (l4[2] + l4[3]);
}

// Finish this warp's part of staged message `slot`: its statistics block (per-row O rescale
// factor, 1/(g l) on the item's last page, flags, sig_p of tokens 16 q4..16 q4 + 15 of the
// page), then mark the warp's share ready.
__device__ __forceinline__ void stage_message(uint8_t* smem, uint32_t bars, int slot, int q4, int lane, float factor,
                                              float inv_l, bool last, bool tail, const float* sig_p_page)
{
    using namespace dev;
    float* stats = reinterpret_cast<float*>(smem + kOffStatsStaging + slot * kStatsBytes + q4 * kStatsWarpBytes);
    stats[lane] = factor;
    if (last) stats[32 + lane] = inv_l;
    if (lane < 16) stats[kSigPWord + lane] = sig_p_page[16 * q4 + lane];
    const bool any_rescale = __any_sync(0xffffffffu, factor != 1.f);
    if (lane == 0) reinterpret_cast<uint32_t*>(stats)[64] = (any_rescale ? 1u : 0u) | (tail ? 2u : 0u);
    fence_proxy_async_cta();  // the staged P~ and statistics are read by the shipper's bulk copies
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (kStgReady0 + slot));
}

// Staging tracker (one thread): follows every phase of copied and publishes how many messages
// have landed in the value CTA (their staging slots are free).  It shares warp 10 with the
// shipper, so both poll with the inline wait: spinning inside an out-of-line call, one of the two
// lanes could hold the warp while the other starved.
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
            st_release_u32(freed, (uint32_t)(k + 1));
        }
    }
}

// Shipper (one thread): sends the staged messages in order, two bulk copies each (P~,
// statistics) completing the peer's msg_full by byte count, once the value CTA is done with the
// message that last used the same buffer.
__device__ __forceinline__ void score_shipper(const Params& p, int item_begin, int item_end, int items_off,
                                              uint8_t* smem, uint32_t sbase, uint32_t bars, const dev::WaitCtx& w)
{
    using namespace dev;
    const uint32_t r_p = map_to_cta(sbase + kOffP, 1);
    const uint32_t r_stats = map_to_cta(sbase + kOffStats, 1);
    const uint32_t r_msg_full = map_to_cta(bars + 8 * kMsgFull0, 1);
    int m = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        for (int t = it.page_begin; t < it.page_end; ++t, ++m) {
            const int slot = m % kStagingSlots, buf = m % kMsgSlots;
            if (!wait_phase(bars + 8 * (kStgReady0 + slot), m / kStagingSlots, w)) return;
            if (m >= kMsgSlots && !wait_phase<true>(bars + 8 * (kMsgFree0 + buf), m / kMsgSlots - 1, w)) return;
            const uint32_t bar = r_msg_full + 8 * buf;
            bulk_copy_to_cta(r_p + buf * kPBytes, sbase + kOffScoreStaging + slot * kPBytes, kPBytes, bar);
            bulk_copy_to_cta(r_stats + buf * kStatsBytes, sbase + kOffStatsStaging + slot * kStatsBytes, kStatsBytes,
                             bar);
            MLA_EV(8, m);
        }
    }
    // the value CTA's last commits and arrivals land in this CTA: wait for them before it ends
    for (int k = (m > kMsgSlots ? m - kMsgSlots : 0); k < m; ++k)
        if (!wait_phase<true>(bars + 8 * (kMsgFree0 + k % kMsgSlots), k / kMsgSlots, w)) break;
}

__device__ __forceinline__ void score_softmax(const Params& p, int item_begin, int item_end, int items_off,
                                              uint8_t* smem, uint32_t bars, uint32_t tmem, const dev::WaitCtx& w,
                                              int warp, int lane)
{
    using namespace dev;
    const int q4 = warp & 3, row = 32 * q4 + lane;
    const int set = (warp - 2) >> 2;  // 0: pages 0-1 of a group, 1: pages 2-3
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const uint32_t p_row_off = (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
    const uint32_t* freed = reinterpret_cast<const uint32_t*>(smem + kOffStgFreed);
    const uint32_t* sig_ready = reinterpret_cast<const uint32_t*>(smem + kOffSigReady);
    float* xchg = reinterpret_cast<float*>(smem + kOffXchg);  // [slot 2][kind 2: max, l][set 2][128]
    int g = 0, G = 0;  // pages (messages) and four-page groups
    for (int i = item_begin, n_item = 0; i < item_end; ++i, ++n_item) {
        const Item it = load_item(p.plan, items_off, i);
        // The exchange slot of the query maxima: the group-max slot that the next group does not
        // use.  Group G - 1 (the previous item's last group, which also ran the l barrier) read it
        // before every softmax thread passed that barrier; group G + 1 writes it only after the
        // first barrier of group G, behind every thread's read here.  (Every item has a page.)
        float r_h;
        if (!load_query(p, it.seq, row, set, n_item, bars, tmem + lane_off, smem + kOffQR,
                        reinterpret_cast<uint32_t*>(xchg + ((G + 1) & 1) * 2 * 2 * 128), w, &r_h))
            return;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * kQReady);
        float m_used = -INFINITY, l_mine = 0.f, l_total = 0.f, g_item = 1.f;
        for (int pg = it.page_begin; pg < it.page_end; pg += kGroupPages, ++G) {
            const int npg = min(kGroupPages, it.page_end - pg);
            const int n_mine = max(0, min(2, npg - 2 * set));
            const bool last_group = (pg + kGroupPages >= it.page_end);
            float* xs = xchg + (G & 1) * 2 * 2 * 128;
            const float* sig = reinterpret_cast<const float*>(smem + kOffSig + (G % kSigSlots) * kSigGroupBytes);
            // Both sets reach every named barrier below the same number of times: a failed wait
            // only clears `ok`, and each barrier ORs the abort state so the sets leave together.
            bool ok = wait_warp_ool(bars + 8 * kSFull0, G, w);
            if (lane == 0 && warp == 2) MLA_EV(4, G);
            // One page of scores in registers at a time (a second one would spill into local
            // memory, which the shared-memory carve-out leaves little L1 for): the second page is
            // read first, for its max only, then the first page, which stays; the second is read
            // again after the first page's P, and the score buffer is freed after that read.
            // (One loop body reads both pages: the code stays small in the instruction cache.)
            uint32_t sr[64];
            const uint32_t scol = tmem + lane_off + kSCol + 128 * set;
            const int t0 = pg + 2 * set;
            const int valid0 = min(64, it.seq_len - 64 * t0), valid1 = min(64, it.seq_len - 64 * (t0 + 1));
            float mx = -INFINITY;
            if (ok) ok = wait_freed(sig_ready, (uint32_t)(G + 1), w);  // this group's token factors
            if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int j = n_mine - 1; j >= 0; --j) {
                    tmem_ld32(scol + 64 * j, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                    tmem_ld32(scol + 64 * j + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                    tmem_wait_ld();
                    mx = fmaxf(mx, page_scale_max(sr, sig + 64 * (2 * set + j)));
                }
                if (n_mine < 2) {  // nothing left to read: the next group's QK may start
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars + 8 * kSFree0);
                }
                g_item = sig[512];
                if (lane == 0 && warp == 2) MLA_EV(5, G);
            }

            // group max (log2 units), agreed between the two sets, drives the lazy rescale
            xs[set * 128 + row] = mx * r_h;
            if (named_barrier_or(kSoftmaxBarrier, 256, !ok || *w.abort)) return;
            if (lane == 0 && warp == 2) MLA_EV(6, G);
            const float gm = fmaxf(xs[row], xs[128 + row]);
            float factor = 1.f;
            if (gm > m_used + kRescaleThreshold) {
                if (pg != it.page_begin) factor = ex2_approx(m_used - gm);
                m_used = gm;
            }
            l_mine *= factor;

            // P~ of my pages into staging slot (message % 4), free once the value CTA received
            // the message four before; the item's last page waits for 1/(g l) below
            bool hold_last = false;
#pragma unroll 1
            for (int j = 0; j < 2; ++j) {
                if (j >= n_mine || !ok) break;
                if (j == 1) {  // the second page again, then the score buffer is free
                    tmem_ld32(scol + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                    tmem_ld32(scol + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                    tmem_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars + 8 * kSFree0);
                    page_scale_max(sr, sig + 64 * (2 * set + 1));  // scaled again (its max is known)
                }
                const int gg = g + 2 * set + j;
                const int slot = gg % kStagingSlots;
                if (gg >= kStagingSlots) ok = wait_freed(freed, (uint32_t)(gg - kStagingSlots + 1), w);
                if (!ok) break;
                l_mine += page_softmax(sr, r_h, m_used, smem + kOffScoreStaging + slot * kPBytes + p_row_off, row);
                const float f_page = (set == 0 && j == 0) ? factor : 1.f;  // O rescale precedes page 0
                if (t0 + j == it.page_end - 1)
                    hold_last = true;
                else
                    stage_message(smem, bars, slot, q4, lane, f_page, 0.f, false, (j ? valid1 : valid0) < 64,
                                  sig + 256 + 64 * (2 * set + j));
            }
            if (last_group) {  // 1/(g l) for the item's last page needs both sets' sums
                xs[256 + set * 128 + row] = l_mine;
                if (named_barrier_or(kSoftmaxBarrier, 256, !ok || *w.abort)) return;
                l_total = xs[256 + row] + xs[256 + 128 + row];
                if (hold_last) {
                    const int j = n_mine - 1;
                    const int slot = (g + 2 * set + j) % kStagingSlots;
                    const float f_page = (set == 0 && j == 0) ? factor : 1.f;
                    stage_message(smem, bars, slot, q4, lane, f_page, 1.f / (g_item * l_total), true,
                                  (j ? valid1 : valid0) < 64, sig + 256 + 64 * (2 * set + j));
                }
            }
            if (lane == 0 && warp == 2) MLA_EV(7, G);
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
}

// ---------------------------------------------------------------------------- value CTA

__device__ __forceinline__ uint32_t msg_flags(const uint8_t* smem, int buf)
{
    const volatile uint32_t* f = reinterpret_cast<const volatile uint32_t*>(smem + kOffStats + buf * kStatsBytes);
    const int w = kStatsWarpBytes / 4;
    return f[64] | f[w + 64] | f[2 * w + 64] | f[3 * w + 64];
}

// Message acknowledgement (one thread): arms msg_full for each message in order and, once it
// has landed, tells the score CTA its staging slot is free (copied).
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
            if (!wait_phase_ool<true>(bars + 8 * (kMsgFull0 + buf), g / kMsgSlots, w)) return;
            mbar_arrive_remote(r_copied + 8 * buf);
        }
    }
}

// PV of a page: O[128 x 512] += P~_hi [128 x 64] c8 + P~_lo [128 x 64] c8, as two N = 256
// halves of four e4m3 MMAs (K = 32): A = the P~ rows (K-major, hi in bytes 0-63, lo in 64-127),
// B = the page's c8 stage (tokens along K, 128-column boxes along N: MN-major).
__device__ __forceinline__ void value_mma(const Params& p, int item_begin, int item_end, int items_off,
                                          const uint8_t* smem, uint32_t sbase, uint32_t bars, uint32_t tmem,
                                          const dev::WaitCtx& w)
{
    using namespace dev;
    constexpr uint32_t idesc = idesc_e4m3(128, 256, false, true);
    const uint64_t p_desc0 = smem_desc(sbase + kOffP, 16, 1024);
    const uint64_t v_desc0 = smem_desc(sbase, kBoxBytes, 1024);
    int g = 0, n_flagged = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int s = g % kValueStages, buf = g % kMsgSlots;
            if (!wait_phase_ool(bars + 8 * (kFull0 + s), g / kValueStages, w)) goto out;
            MLA_EV(15, g);
            if (!wait_phase_ool<true>(bars + 8 * (kMsgFull0 + buf), g / kMsgSlots, w)) goto out;
            if (!wait_phase_ool(bars + 8 * (kPReady0 + buf), g / kMsgSlots, w)) goto out;  // P~ written
            MLA_EV(10, g);
            // The correction warps go first on flagged tiles and on the first tile of every item
            // after the first; both sides apply the same rule, so o_ready phases stay paired.
            if (msg_flags(smem, buf) != 0 || (t == it.page_begin && i != item_begin)) {
                const int e = n_flagged & 1;
                mma_commit(bars + 8 * (kODrain0 + e));  // arrives once every earlier PV is done
                if (!wait_phase_ool(bars + 8 * (kOReady0 + e), n_flagged >> 1, w)) goto out;
                ++n_flagged;
            }
            tc_fence_after();
            {
                const uint64_t a0 = p_desc0 + (uint64_t)(buf * (kPBytes >> 4));
                const uint64_t b0 = v_desc0 + (uint64_t)(s * (kValueStageBytes >> 4));
                const uint32_t acc0 = (t == it.page_begin) ? 0u : 1u;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint64_t bh = b0 + (uint64_t)(half * ((2 * kBoxBytes) >> 4));
                    const uint32_t d = tmem + 256 * half;
                    mma_ss_e4m3(d, a0, bh, idesc, acc0);                        // hi, tokens 0-31
                    mma_ss_e4m3(d, a0 + 2, bh + (4096 >> 4), idesc, 1u);        // hi, tokens 32-63
                    mma_ss_e4m3(d, a0 + 4, bh, idesc, 1u);                      // lo, tokens 0-31
                    mma_ss_e4m3(d, a0 + 6, bh + (4096 >> 4), idesc, 1u);        // lo, tokens 32-63
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
}

// P -> P~ (four warps, thread = head row, in place in the message buffer): row h's 64 bf16 p
// times sig_p[t] = sigma_t g (0 past the sequence end) from the message's statistics, split into
// the e4m3 pair: 16-byte chunks 0-3 of the row take hi of tokens 0-63, chunks 4-7 lo (chunk c
// at c ^ (h & 7), the 128-byte swizzle the MMA reads).  The whole row is read before any of it
// is written.  p <= 16 and sig_p <= 28 keep P~ <= 448.
__device__ __forceinline__ void value_pconvert(const Params& p, int item_begin, int item_end, int items_off,
                                            uint8_t* smem, uint32_t bars, const dev::WaitCtx& w, int row, int lane)
{
    using namespace dev;
    int g = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int buf = g % kMsgSlots;
            if (!wait_warp_ool<true>(bars + 8 * (kMsgFull0 + buf), g / kMsgSlots, w)) return;
            if (lane == 0 && row == 0) MLA_EV(12, g);
            const uint8_t* stats = smem + kOffStats + buf * kStatsBytes;
            uint8_t* prow = smem + kOffP + buf * kPBytes + (row >> 3) * 1024 + (row & 7) * 128;
            uint4 x[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) x[c] = *reinterpret_cast<const uint4*>(prow + ((c ^ (row & 7)) << 4));
#pragma unroll
            for (int k = 0; k < 4; ++k) {  // tokens 16k..16k+15: chunks 2k, 2k+1 of p
                const float* sp = reinterpret_cast<const float*>(stats + k * kStatsWarpBytes) + kSigPWord;
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 v = x[2 * k + h];
                    const float4 f0 = *reinterpret_cast<const float4*>(sp + 8 * h);
                    const float4 f1 = *reinterpret_cast<const float4*>(sp + 8 * h + 4);
                    split_e4m3x4(bf16_lo(v.x) * f0.x, bf16_hi(v.x) * f0.y, bf16_lo(v.y) * f0.z, bf16_hi(v.y) * f0.w,
                                 hi[2 * h], lo[2 * h]);
                    split_e4m3x4(bf16_lo(v.z) * f1.x, bf16_hi(v.z) * f1.y, bf16_lo(v.w) * f1.z, bf16_hi(v.w) * f1.w,
                                 hi[2 * h + 1], lo[2 * h + 1]);
                }
                *reinterpret_cast<uint4*>(prow + ((k ^ (row & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(prow + (((k + 4) ^ (row & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_cta();  // read by the MMA (async proxy)
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8 * (kPReady0 + buf));
            if (lane == 0 && row == 0) MLA_EV(14, g);
        }
    }
}

// The normalised output of an item, O / (g l), leaves through decode.cuh's write_output (its
// inv_l here carries the item's token-factor normaliser g as well).

__device__ __forceinline__ void value_correction(const Params& p, int item_begin, int item_end, int items_off,
                                                 uint8_t* smem, uint32_t bars, uint32_t tmem, const dev::WaitCtx& w,
                                                 int warp, int lane, int tid128)
{
    using namespace dev;
    const int q4 = warp & 3;
    uint8_t* out_tile = smem + kOffOutTile + q4 * kOutTileBytes;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const uint32_t r_msg_free = dev::map_to_cta(dev::smem_u32(smem) + kOffBars + 8 * kMsgFree0, 0);
    int g = 0, n_flagged = 0;
    Item prev{};
    float prev_inv_l = 0.f;
    bool have_prev = false;  // an item whose output is still in TMEM
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        float inv_l = 0.f;
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int buf = g % kMsgSlots;
            if (!wait_warp_ool<true>(bars + 8 * (kMsgFull0 + buf), g / kMsgSlots, w)) goto done;
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
            const int e = n_flagged & 1;
            if (!wait_warp_ool(bars + 8 * (kODrain0 + e), n_flagged >> 1, w)) goto done;
            tc_fence_after();
            if (boundary) {  // the previous item's output leaves TMEM before this PV overwrites it
                write_output(p, prev, prev_inv_l, tmem, lane_off, out_tile, q4, lane);
                have_prev = false;
            }
            if (flags & 2u) {
                // slots past the sequence end may hold anything (NaN codes): zero them so that
                // P~ = 0 times them stays 0 in the PV contraction
                const int valid = min(64, it.seq_len - 64 * t);
                const int s = g % kValueStages;
                if (!wait_warp_ool(bars + 8 * (kFull0 + s), g / kValueStages, w)) goto done;
                uint8_t* stage = smem + s * kValueStageBytes;
                const int chunks = (64 - valid) * 32;  // rows x (4 boxes x 8 chunks of 16 B)
                for (int c = tid128; c < chunks; c += 128) {
                    const int r = valid + (c >> 5), box = (c >> 3) & 3, ch = c & 7;
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
        }
        prev = it;
        prev_inv_l = inv_l;
        have_prev = true;
    }
    if (have_prev) {
        // last item: every PV is done when the MMA thread's final commit lands
        if (!wait_warp_ool(bars + 8 * kDrain, 0, w)) goto done;
        tc_fence_after();
        write_output(p, prev, prev_inv_l, tmem, lane_off, out_tile, q4, lane);
    }
done:
    tc_fence_before();
}

// ---------------------------------------------------------------------------- kernel

// Code size matters here: twelve warps run different roles, and when their hot loops do not fit
// in the instruction caches every role slows down (instruction-fetch stalls led the profile of
// a 163 KB build).  So the per-chunk and per-row loops stay rolled, barrier polling runs out of
// line, and the query load (once per item) is a separate function.
// 12 warps: each SM sub-partition holds three, and its 16K registers allow 3 x 32 x 168.
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(168)
decode_fp8_kernel(const __grid_constant__ CUtensorMap tm_c8, const __grid_constant__ CUtensorMap tm_kr,
                  const __grid_constant__ CUtensorMap tm_q, const Params p)
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
            mbar_init(bars + 8 * (kPReady0 + b), 4);       // the four P converter warps
            mbar_init(bars + 8 * (kMsgFree0 + b), 1 + 4);  // PV commit + four correction warps
            mbar_init(bars + 8 * (kMsgFull0 + b), 1);      // the acknowledgement thread's arm + the bytes
            mbar_init(bars + 8 * (kCopied0 + b), 1);       // the message landed in the value CTA
        }
        mbar_init(bars + 8 * kQReady, 8);                  // one arrive per softmax warp
        mbar_init(bars + 8 * kQRaw, 1);                    // the MMA thread's commit after the query copies
        for (int s = 0; s < kStagingSlots; ++s) mbar_init(bars + 8 * (kStgReady0 + s), 4);  // one set's warps
        mbar_init(bars + 8 * kKrLanded, 1);
        mbar_init(bars + 8 * kKrFull, 1);   // warp 11: the group's k_R / sigma is in place
        mbar_init(bars + 8 * kKrEmpty, 1);  // the MMA's commit after the k_R MMAs
        *reinterpret_cast<volatile uint32_t*>(smem + kOffStgFreed) = 0;
        *reinterpret_cast<volatile uint32_t*>(smem + kOffSigReady) = 0;
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
                score_producer(&tm_c8, &tm_q, p, item_begin, item_end, items_off, sbase, bars, w, lane);
            else if (warp == 1) {
                if (lane == 0) score_mma(p, item_begin, item_end, items_off, sbase, bars, tmem, w);
            } else if (warp >= 2 && warp < 10)
                score_softmax(p, item_begin, item_end, items_off, smem, bars, tmem, w, warp, lane);
            else if (warp == kShipperWarp) {
                if (lane == 0) score_shipper(p, item_begin, item_end, items_off, smem, sbase, bars, w);
                else if (lane == 1) score_tracker(p, item_begin, item_end, items_off, smem, bars, w);
            } else if (warp == kKrWarp)
                kr_convert(&tm_kr, p, item_begin, item_end, items_off, smem, sbase, bars, w, lane);
        } else {
            if (warp == 0)
                value_producer(&tm_c8, p, item_begin, item_end, items_off, sbase, bars, w, lane);
            else if (warp == 1) {
                if (lane == 0) value_mma(p, item_begin, item_end, items_off, smem, sbase, bars, tmem, w);
            } else if (warp >= 2 && warp < 6)
                value_correction(p, item_begin, item_end, items_off, smem, bars, tmem, w, warp, lane,
                                 threadIdx.x - 64);
            else if (warp == kAckWarp) {
                if (lane == 0) value_ack(p, item_begin, item_end, items_off, bars, w);
            } else if (warp >= kPConvWarp0 && warp < kPConvWarp0 + 4)
                value_pconvert(p, item_begin, item_end, items_off, smem, bars, w, 32 * (warp - kPConvWarp0) + lane,
                               lane);
            // warp 11 of the value CTA has no role
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

}  // namespace decode_fp8
}  // namespace mla
