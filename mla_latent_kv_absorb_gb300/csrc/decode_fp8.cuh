// decode_fp8.cuh -- the paged MLA decode of decode.cuh for a latent cache stored as FP8 e4m3
// with one fp32 scale per token (the RoPE key k_R stays bf16).
//
// What it computes: as decode.cuh, with each cached latent row c_t = float(c8_t) * sigma_t
// (page 1, "撕開 DeepSeek MLA 源碼", section 5, on FP8 caches).  Converter warps in both CTAs
// of a pair turn the e4m3 rows of each page into f16(f16(c8) * f16(sigma)) in shared memory,
// laid out exactly as the TMA's 128-byte-swizzled boxes (one hardware e4m3x2 -> f16x2
// conversion, exact, and one packed f16 multiply per two values).  The latent part of QK and
// PV then run as f16 MMAs (q_abs is converted to f16 when it is loaded into tensor memory, P
// is packed as f16), the RoPE part of QK stays bf16 (q_R and the cached k_R); both accumulate
// in fp32.  Against the exact dequantised value the f16 product is off by at most about 2^-10
// relative, as long as it is an f16 normal number (|value| >= 2^-14).
//
// Bytes per cached token: 512 (e4m3) + 4 (scale) + 128 (k_R) = 644, against 1,152 in bf16.
//
// Layout of the pair (sm_103a):
//   rank 0, the score CTA: q_abs in TMEM (256 columns), scores of two pages at a time in one
//     of two 128-column TMEM buffers (N=128 MMAs).  The producer loads each two-page group as
//     eight raw e4m3 K-chunks (one 64-column box of two pages, 8 KB, into a four-slot raw
//     ring) and one k_R chunk straight into the 16-bit K-chunk ring (six 16 KB slots); four
//     converter warps fill the ring from the raw ring, each owning whole chunks (warp k takes
//     boxes k and k + 4 of every group), so four chunks convert at once.  Eight softmax warps
//     (one page each per group) and a shipper warp as in the bf16 kernel.
//   rank 1, the value CTA: the producer loads each page's 32 KB of e4m3 into a two-slot raw
//     ring; eight converter warps write the f16 page (64 KB) into one of two PV stages; PV,
//     corrections and output as in the bf16 kernel.
// Fifteen warps per CTA, so every thread is capped at 128 registers (four warps share an SM
// sub-partition's 16K registers); one page of scores per softmax thread fits in that.
//
// Pipelines (all waits bounded, see ptx.cuh): those of the bf16 kernel, plus
//   raw_full[4]/raw_empty[4]   the raw e4m3 rings (TMA bytes / the converter warp that owns the
//                              chunk in the score CTA, all eight converter warps in the value CTA)
//   kv_full[S]                 16-bit ring slot filled: the owning converter warp, or (k_R chunk
//                              of the score CTA) the producer's arrival plus the TMA bytes; in
//                              the value CTA the eight converter warps
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "plan.h"
#include "ptx.cuh"

namespace mla {
namespace decode_fp8 {

constexpr int kThreads = 480;                     // 15 warps, roles below
constexpr int kShipperWarp = 10;
constexpr int kScoreConvertWarp0 = 11;            // score CTA: warps 11-14 convert
constexpr int kScoreConvertWarps = 4;
constexpr int kValueConvertWarp0 = 6;             // value CTA: warps 6-13 convert
constexpr int kValueConvertWarps = 8;
constexpr int kChunkStages = 6;                   // score CTA: bf16 K-chunk ring
constexpr int kValueStages = 2;                   // value CTA: bf16 page stages
constexpr int kMaxStages = 6;
constexpr int kRawSlots = 4;                      // score CTA: raw e4m3 K-chunks
constexpr int kValueRawSlots = 2;                 // value CTA: raw e4m3 pages
constexpr int kStagingSlots = 4;                  // score CTA: P messages staged ahead of the peer
constexpr int kBoxBytes = 64 * 128;               // 64 tokens x 64 bf16 columns
constexpr int kRawBoxBytes = 64 * 64;             // 64 tokens x 64 e4m3 columns
constexpr int kBoxesPerRow = 9;                   // c_KV: 8 boxes, k_R: 1 box
constexpr int kGroupPages = 2;                    // pages per score MMA (N = 128)
constexpr int kChunkBytes = kGroupPages * kBoxBytes;        // 16 KB
constexpr int kRawChunkBytes = kGroupPages * kRawBoxBytes;  // 8 KB
constexpr int kValueStageBytes = 8 * kBoxBytes;   // 65,536: c_KV only, bf16
constexpr int kValueRawBytes = 8 * kRawBoxBytes;  // 32,768: c_KV only, e4m3
constexpr int kPBytes = 128 * 128;                // P: 128 heads x 64 tokens bf16
// Per message statistics, one 272-byte block per softmax warp (32 heads): factor[32] (rescale
// of those O rows), inv_l[32] (1/l, last tile of an item), then a 16-byte flags slot (bit 0:
// one of the rows rescales, bit 1: the page has slots past the sequence end).
constexpr int kStatsWarpBytes = 128 + 128 + 16;
constexpr int kStatsBytes = 4 * kStatsWarpBytes;
constexpr int kPWarpBytes = kPBytes / 4;
constexpr int kMsgBytes = kPBytes + kStatsBytes;
// score CTA: q_R, the bf16 K-chunk ring, the raw ring, the staging ring of P messages and
// their statistics, the softmax sets' exchange area
constexpr int kOffQR = 0;
constexpr int kOffChunks = kOffQR + 128 * 128;
constexpr int kOffRaw = kOffChunks + kChunkStages * kChunkBytes;
constexpr int kOffScoreStaging = kOffRaw + kRawSlots * kRawChunkBytes;
constexpr int kOffStatsStaging = kOffScoreStaging + kStagingSlots * kPBytes;
constexpr int kOffXchg = kOffStatsStaging + kStagingSlots * kStatsBytes;
constexpr int kScoreEnd = kOffXchg + 4 * 2 * 128 * 4;
// value CTA: bf16 stages, raw pages, two P buffers (1024-aligned, the MMA reads them), stats
constexpr int kOffValueRaw = kValueStages * kValueStageBytes;
constexpr int kOffP = kOffValueRaw + kValueRawSlots * kValueRawBytes;
constexpr int kOffStats = kOffP + 2 * kPBytes;
constexpr int kValueEnd = kOffStats + 2 * kStatsBytes;
constexpr int kOffBars = ((kScoreEnd > kValueEnd ? kScoreEnd : kValueEnd) + 7) / 8 * 8;

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
    kStgReady0 = kDrain + 1,
    kRawFull0 = kStgReady0 + kStagingSlots,
    kRawEmpty0 = kRawFull0 + kRawSlots,
    kNumBars = kRawEmpty0 + kRawSlots
};

constexpr int kOffTmemHolder = kOffBars + 8 * kNumBars;
constexpr int kOffAbort = kOffTmemHolder + 4;
constexpr int kOffStgFreed = kOffAbort + 4;  // score CTA: messages whose staging slot may be reused
constexpr int kSmemBytes = ((kOffStgFreed + 4 + 127) / 128) * 128;
static_assert(kChunkStages <= kMaxStages && kValueStages <= kMaxStages, "barrier slots per ring");
static_assert(kValueRawSlots <= kRawSlots, "raw barrier slots");
static_assert(kRawSlots == kScoreConvertWarps, "score converter warp k owns raw slot k");
static_assert(kOffChunks % 1024 == 0 && kOffP % 1024 == 0 && kOffValueRaw % 1024 == 0 && kOffRaw % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kStatsWarpBytes % 16 == 0 && kPWarpBytes % 16 == 0, "bulk copies move multiples of 16 bytes");

// TMEM columns
constexpr uint32_t kQCol = 0;      // score CTA: q_abs, 256 columns (512 bf16 per lane)
constexpr uint32_t kSCol = 256;    // score CTA: two 128-column score buffers (two pages each)
constexpr uint32_t kTmemCols = 512;

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8
constexpr uint32_t kSoftmaxBarrier = 1;    // named barrier of the eight softmax warps



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
    const float* kv_scale;       // [pages][64] per-token scale of the e4m3 latent rows
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

// ---------------------------------------------------------------------------- e4m3 -> bf16

// Four e4m3 codes (little-endian in `w`) -> two f16x2 words of code * scale: the hardware
// conversion to f16 is exact, the packed multiply rounds once.
__device__ __forceinline__ uint2 convert4(uint32_t w, uint32_t sig2)
{
    uint32_t a, b;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t"
        "mul.rn.f16x2 %0, %0, %3;\n\t"
        "mul.rn.f16x2 %1, %1, %3;\n\t}"
        : "=r"(a), "=r"(b)
        : "r"(w), "r"(sig2));
    return make_uint2(a, b);
}

// One 64-column row: 64 e4m3 bytes at `src` -> 64 f16 (128 bytes) at row `r` of a 128-byte
// swizzled tile (16-byte chunk c of the row lands at chunk c ^ (r & 7)).  `sig2` holds the
// token's scale in both f16 halves.
__device__ __forceinline__ void convert_row64(const uint8_t* src, uint8_t* dst_row, int r, uint32_t sig2)
{
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * h);
        const uint2 a0 = convert4(v.x, sig2), a1 = convert4(v.y, sig2);
        const uint2 b0 = convert4(v.z, sig2), b1 = convert4(v.w, sig2);
        *reinterpret_cast<uint4*>(dst_row + (((2 * h) ^ (r & 7)) << 4)) = make_uint4(a0.x, a0.y, a1.x, a1.y);
        *reinterpret_cast<uint4*>(dst_row + (((2 * h + 1) ^ (r & 7)) << 4)) = make_uint4(b0.x, b0.y, b1.x, b1.y);
    }
}

// A scale in both halves of an f16x2 word.
__device__ __forceinline__ uint32_t splat_f16(float x) { return dev::pack_f16x2(x, x); }

// Scale of token `tok` of physical page `page` (0 for an out-of-range page, whose TMA boxes
// read as zeros).
__device__ __forceinline__ float token_scale(const Params& p, int page, int tok)
{
    return (page >= 0 && page < p.num_pool_pages) ? __ldg(p.kv_scale + (int64_t)page * 64 + tok) : 0.f;
}

// ---------------------------------------------------------------------------- value CTA loads

// Streams the e4m3 latent columns of this cluster's pages (eight 64-column boxes, 32 KB per
// page) into the two-slot raw ring.
__device__ __forceinline__ void value_producer(const CUtensorMap* tm, const Params& p, int item_begin, int item_end,
                                               int items_off, uint32_t sbase, uint32_t bars, const dev::WaitCtx& w,
                                               int lane)
{
    using namespace dev;
    const uint64_t policy = l2_policy_evict_first();  // the score CTA brought these pages into L2
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
                    const int s = g % kValueRawSlots;
                    if (g >= kValueRawSlots) ok = wait_phase(bars + 8 * (kRawEmpty0 + s), g / kValueRawSlots - 1, w);
                    if (ok) {
                        const uint32_t full = bars + 8 * (kRawFull0 + s);
                        const uint32_t dst = sbase + kOffValueRaw + s * kValueRawBytes;
                        mbar_arrive_expect_tx(full, kValueRawBytes);
                        for (int x = 0; x < 8; ++x) tma_load_3d(dst + x * kRawBoxBytes, tm, full, 64 * x, 0, pj, policy);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                ++g;
            }
        }
    }
    if (lane == 0 && *w.abort) {  // loads still in flight must land before the CTA exits
        for (int k = (g > kValueRawSlots ? g - kValueRawSlots : 0); k < g; ++k)
            drain_phase(bars + 8 * (kRawFull0 + k % kValueRawSlots), k / kValueRawSlots, w.timeout_ns);
    }
}

// Eight warps: raw e4m3 page -> f16 PV stage (eight 64-column boxes, 128-byte swizzle).
// Thread t converts a quarter row: row t / 4, boxes 2 (t % 4) and 2 (t % 4) + 1.
__device__ __forceinline__ void value_convert(const Params& p, int item_begin, int item_end, int items_off,
                                              uint8_t* smem, uint32_t bars, const dev::WaitCtx& w, int cw, int lane)
{
    using namespace dev;
    const int t = 32 * cw + lane, r = t >> 2, quarter = t & 3;
    int g = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        const int32_t* bt = p.block_table + (int64_t)it.seq * p.max_pages;
        for (int pg = it.page_begin; pg < it.page_end; ++pg, ++g) {
            const uint32_t sig2 = splat_f16(token_scale(p, __ldg(bt + pg), r));
            const int rs = g % kValueRawSlots, s = g % kValueStages;
            if (!wait_warp(bars + 8 * (kRawFull0 + rs), g / kValueRawSlots, w)) return;
            if (g >= kValueStages && !wait_warp(bars + 8 * (kEmpty0 + s), g / kValueStages - 1, w)) return;
            const uint8_t* raw = smem + kOffValueRaw + rs * kValueRawBytes;
            uint8_t* stage = smem + s * kValueStageBytes;
#pragma unroll
            for (int b = 2 * quarter; b < 2 * quarter + 2; ++b)
                convert_row64(raw + b * kRawBoxBytes + r * 64, stage + b * kBoxBytes + r * 128, r, sig2);
            fence_proxy_async_cta();  // read by the MMA (async proxy)
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bars + 8 * (kFull0 + s));
                mbar_arrive(bars + 8 * (kRawEmpty0 + rs));
            }
        }
    }
}

// ---------------------------------------------------------------------------- score CTA

// Per two-page group: eight raw e4m3 K-chunks (box j of the group's pages, 4 KB each) into
// the raw ring, then the k_R chunk (bf16, 8 KB per page) straight into the K-chunk ring.
__device__ __forceinline__ void score_producer(const CUtensorMap* tm_c8, const CUtensorMap* tm_kr, const Params& p,
                                               int item_begin, int item_end, int items_off, uint32_t sbase,
                                               uint32_t bars, const dev::WaitCtx& w, int lane)
{
    using namespace dev;
    const uint64_t policy = l2_policy_evict_normal();  // the value CTA reads these pages next
    if (lane == 0) {
        tma_prefetch_desc(tm_c8);
        tma_prefetch_desc(tm_kr);
    }
    int c = 0, rc = 0;  // bf16 ring chunks (nine per group), raw chunks (eight per group)
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
                int pages[kGroupPages];
#pragma unroll
                for (int q = 0; q < kGroupPages; ++q) pages[q] = __shfl_sync(0xffffffffu, page, min(j + q, 31));
                if (lane == 0) {
                    for (int box = 0; box < 8 && ok; ++box, ++rc, ++c) {
                        const int rs = rc % kRawSlots;
                        if (rc >= kRawSlots) ok = wait_phase(bars + 8 * (kRawEmpty0 + rs), rc / kRawSlots - 1, w);
                        if (!ok) break;
                        const uint32_t full = bars + 8 * (kRawFull0 + rs);
                        const uint32_t dst = sbase + kOffRaw + rs * kRawChunkBytes;
                        mbar_arrive_expect_tx(full, npg * kRawBoxBytes);
                        for (int q = 0; q < npg; ++q) tma_load_3d(dst + q * kRawBoxBytes, tm_c8, full, 64 * box, 0, pages[q], policy);
                    }
                    if (ok) {  // the k_R chunk
                        const int s = c % kChunkStages;
                        if (c >= kChunkStages) ok = wait_phase(bars + 8 * (kEmpty0 + s), c / kChunkStages - 1, w);
                        if (ok) {
                            const uint32_t full = bars + 8 * (kFull0 + s);
                            const uint32_t dst = sbase + kOffChunks + s * kChunkBytes;
                            mbar_arrive_expect_tx(full, npg * kBoxBytes);
                            for (int q = 0; q < npg; ++q) tma_load_3d(dst + q * kBoxBytes, tm_kr, full, 0, 0, pages[q], policy);
                        }
                        ++c;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
        }
    }
    if (lane == 0 && *w.abort) {  // loads still in flight must land before the CTA exits
        for (int k = (rc > kRawSlots ? rc - kRawSlots : 0); k < rc; ++k)
            drain_phase(bars + 8 * (kRawFull0 + k % kRawSlots), k / kRawSlots, w.timeout_ns);
        // k_R chunks: the last kChunkStages ring positions may hold loads in flight
        for (int k = (c > kChunkStages ? c - kChunkStages : 0); k < c; ++k)
            if (k % kBoxesPerRow == kBoxesPerRow - 1)
                drain_phase(bars + 8 * (kFull0 + k % kChunkStages), k / kChunkStages, w.timeout_ns);
    }
}

// Four warps: raw e4m3 K-chunk -> f16 K-chunk (two pages x 64 rows x 64 columns, 128-byte
// swizzle).  Warp k owns boxes k and k + 4 of every group (hence raw slot k); lane l converts
// rows l, l + 32 (page 0) and l + 64, l + 96 (page 1) of its chunks.
__device__ __forceinline__ void score_convert(const Params& p, int item_begin, int item_end, int items_off,
                                              uint8_t* smem, uint32_t bars, const dev::WaitCtx& w, int cw, int lane)
{
    using namespace dev;
    int G = 0;  // two-page groups
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        const int32_t* bt = p.block_table + (int64_t)it.seq * p.max_pages;
        for (int pg = it.page_begin; pg < it.page_end; pg += kGroupPages, ++G) {
            const int npg = min(kGroupPages, it.page_end - pg);
            uint32_t sig2[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int rho = lane + 32 * k;
                sig2[k] = (rho < 64 * npg) ? splat_f16(token_scale(p, __ldg(bt + pg + (rho >> 6)), rho & 63)) : 0u;
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int box = cw + 4 * half;
                const int rc = 8 * G + box, c = 9 * G + box;
                const int rs = cw, s = c % kChunkStages;
                if (!wait_warp(bars + 8 * (kRawFull0 + rs), rc / kRawSlots, w)) return;
                if (c >= kChunkStages && !wait_warp(bars + 8 * (kEmpty0 + s), c / kChunkStages - 1, w)) return;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int rho = lane + 32 * k;
                    if (rho < 64 * npg)
                        convert_row64(smem + kOffRaw + rs * kRawChunkBytes + rho * 64,
                                      smem + kOffChunks + s * kChunkBytes + rho * 128, rho, sig2[k]);
                }
                fence_proxy_async_cta();  // read by the MMA (async proxy)
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bars + 8 * (kFull0 + s));
                    mbar_arrive(bars + 8 * (kRawEmpty0 + rs));
                }
            }
        }
    }
}

// QK of a two-page group: S[128 heads x N tokens] (N = 64 per page, 128 for a full group) in
// score buffer G % 2, accumulated over the nine K-chunks: chunks 0-7 take q_abs from TMEM ("TS"), chunk 8 takes
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
    int s = 0, phase = 0, G = 0, n_item = 0;
    for (int i = item_begin; i < item_end; ++i, ++n_item) {
        const Item it = load_item(p.plan, items_off, i);
        if (!wait_phase(bars + 8 * kQReady, n_item, w)) goto out;
        tc_fence_after();
        for (int pg = it.page_begin; pg < it.page_end; pg += kGroupPages, ++G) {
            const int npg = min(kGroupPages, it.page_end - pg);
            const uint32_t idesc_c = idesc_f16(128, 64 * npg, false, false);   // f16 q_abs x f16 latent
            const uint32_t idesc_r = idesc_bf16(128, 64 * npg, false, false);  // bf16 q_R x bf16 k_R
            const int buf = G & 1;
            const uint32_t d = tmem + kSCol + 128 * buf;
            if (G >= 2 && !wait_phase(bars + 8 * (kSFree0 + buf), (G >> 1) - 1, w)) goto out;
#pragma unroll
            for (int box = 0; box < kBoxesPerRow; ++box) {
                if (!wait_phase(full0 + 8 * s, phase, w)) goto out;
                tc_fence_after();
                const uint64_t b0 = chunk_desc0 + (uint64_t)(s * (kChunkBytes >> 4));
                if (box < 8) {
                    const uint32_t a0 = tmem + kQCol + 32 * box;
                    mma_ts(d, a0, b0, idesc_c, box != 0 ? 1u : 0u);
                    mma_ts(d, a0 + 8, b0 + 2, idesc_c, 1u);
                    mma_ts(d, a0 + 16, b0 + 4, idesc_c, 1u);
                    mma_ts(d, a0 + 24, b0 + 6, idesc_c, 1u);
                } else {
                    mma_ss(d, qr_desc, b0, idesc_r, 1u);
                    mma_ss(d, qr_desc + 2, b0 + 2, idesc_r, 1u);
                    mma_ss(d, qr_desc + 4, b0 + 4, idesc_r, 1u);
                    mma_ss(d, qr_desc + 6, b0 + 6, idesc_r, 1u);
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
}

// The query of row `row` (q_abs as f16 in TMEM, the A operand of the f16 MMAs; q_R stays
// bf16): softmax set 0 writes q_abs dims 0..255 to TMEM columns 0..127 of lane
// `row` and q_R to row `row` of the K-major, 128-byte-swizzled q_R tile in shared memory; set 1
// writes q_abs dims 256..511 to columns 128..255.
// Two bf16 (one word) -> two f16, rounded to nearest even.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    return dev::pack_f16x2(dev::bf16_lo(w), dev::bf16_hi(w));
}

__device__ __forceinline__ void load_query(const Params& p, int seq, int row, int set, uint32_t taddr,
                                           uint8_t* qr_smem)
{
    using namespace dev;
    const uint4* qa = reinterpret_cast<const uint4*>(p.q_abs + ((int64_t)seq * 128 + row) * 512) + 32 * set;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const uint4 x = __ldg(qa + 8 * c + v);
            r[4 * v + 0] = bf16x2_to_f16x2(x.x);
            r[4 * v + 1] = bf16x2_to_f16x2(x.y);
            r[4 * v + 2] = bf16x2_to_f16x2(x.z);
            r[4 * v + 3] = bf16x2_to_f16x2(x.w);
        }
        tmem_st32(taddr + kQCol + 128 * set + 32 * c, r);
    }
    if (set == 0) {
        const uint4* qr = reinterpret_cast<const uint4*>(p.q_r + ((int64_t)seq * 128 + row) * 64);
        uint8_t* dst = qr_smem + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
        for (int v = 0; v < 8; ++v) *reinterpret_cast<uint4*>(dst + ((v ^ (row & 7)) << 4)) = __ldg(qr + v);
        fence_proxy_async_cta();  // read by the MMA (async proxy)
    }
    tmem_wait_st();
}

// Softmax of one page held in registers: masks slots past the sequence end, p = 2^(s * scale *
// log2(e) - m) (one FMA and one MUFU.EX2 per score), and writes P as f16 straight into this
// thread's row of the swizzled staging tile (16-byte chunk c of the row goes to chunk c ^ (row
// & 7)).  Returns the row sum of p.
__device__ __forceinline__ float page_softmax(uint32_t (&sr)[64], int valid, float scale_log2, float m_used,
                                              uint8_t* stage_row, int row)
{
    using namespace dev;
    if (valid < 64) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
            if (j >= valid) sr[j] = __float_as_uint(-INFINITY);
    }
    float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint32_t pk[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = 8 * c + 2 * q;
            const float p0 = ex2_approx(fmaf(__uint_as_float(sr[j]), scale_log2, -m_used));
            const float p1 = ex2_approx(fmaf(__uint_as_float(sr[j + 1]), scale_log2, -m_used));
            pk[q] = pack_f16x2(p0, p1);
            l8[(2 * q) & 7] += p0;
            l8[(2 * q + 1) & 7] += p1;
        }
        *reinterpret_cast<uint4*>(stage_row + ((c ^ (row & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    return ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
}

// Row max of a page's raw scores (slots past the sequence end excluded), 8-way tree.
__device__ __forceinline__ float page_max(const uint32_t (&sr)[64], int valid)
{
    float m8[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) m8[a] = (a < valid) ? __uint_as_float(sr[a]) : -INFINITY;
#pragma unroll
    for (int j = 8; j < 64; ++j) m8[j & 7] = fmaxf(m8[j & 7], (j < valid) ? __uint_as_float(sr[j]) : -INFINITY);
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

// Shipper (one thread): sends the staged messages in order to the value CTA, two bulk copies
// each (P, statistics) that complete the peer's msg_full barrier by byte count.  It alone waits
// on msg_free, follows all of its phases, and publishes how many messages the value CTA has
// consumed, which frees their staging slots for the softmax warps.
__device__ __forceinline__ void score_shipper(const Params& p, int item_begin, int item_end, int items_off,
                                              uint8_t* smem, uint32_t sbase, uint32_t bars, const dev::WaitCtx& w)
{
    using namespace dev;
    const uint32_t r_p = map_to_cta(sbase + kOffP, 1);
    const uint32_t r_stats = map_to_cta(sbase + kOffStats, 1);
    const uint32_t r_msg_full = map_to_cta(bars + 8 * kMsgFull0, 1);
    uint32_t* freed = reinterpret_cast<uint32_t*>(smem + kOffStgFreed);
    int m = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        for (int t = it.page_begin; t < it.page_end; ++t, ++m) {
            const int slot = m % kStagingSlots, buf = m & 1;
            if (!wait_phase(bars + 8 * (kStgReady0 + slot), m / kStagingSlots, w)) goto out;
            if (m >= 2) {
                if (!wait_phase<true>(bars + 8 * (kMsgFree0 + buf), (m >> 1) - 1, w)) goto out;
                st_release_u32(freed, (uint32_t)(m - 1));  // messages 0 .. m-2 consumed
            }
            const uint32_t bar = r_msg_full + 8 * buf;
            bulk_copy_to_cta(r_p + buf * kPBytes, sbase + kOffScoreStaging + slot * kPBytes, kPBytes, bar);
            bulk_copy_to_cta(r_stats + buf * kStatsBytes, sbase + kOffStatsStaging + slot * kStatsBytes,
                             kStatsBytes, bar);
        }
    }
    // the value CTA's last commits and arrivals land in this CTA: wait for them before it ends
    for (int k = (m > 2 ? m - 2 : 0); k < m; ++k)
        if (!wait_phase<true>(bars + 8 * (kMsgFree0 + (k & 1)), k >> 1, w)) break;
out:
    return;
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
    const int set = (warp - 2) >> 2;               // page 0 or page 1 of each two-page group
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const uint32_t p_row_off = (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
    const uint32_t* freed = reinterpret_cast<const uint32_t*>(smem + kOffStgFreed);
    float* xchg = reinterpret_cast<float*>(smem + kOffXchg);  // [slot 2][kind 2: max, l][set 2][128]
    int g = 0, G = 0;  // pages (messages) and two-page groups
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        load_query(p, it.seq, row, set, tmem + lane_off, smem + kOffQR);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * kQReady);
        float m_used = -INFINITY, l_mine = 0.f, l_total = 0.f;
        for (int pg = it.page_begin; pg < it.page_end; pg += kGroupPages, ++G) {
            const int npg = min(kGroupPages, it.page_end - pg);
            const bool mine = set < npg;
            const bool last_group = (pg + kGroupPages >= it.page_end);
            const int buf = G & 1;
            float* xs = xchg + buf * 2 * 2 * 128;
            // Both sets must reach every named barrier below the same number of times: a failed
            // (timed-out) wait only clears `ok`, and each barrier ORs the abort state so that the
            // two sets leave together.
            bool ok = wait_warp(bars + 8 * (kSFull0 + buf), G >> 1, w);
            uint32_t sr[64];
            const int t = pg + set;
            const int valid = min(64, it.seq_len - 64 * t);
            float mx = -INFINITY;
            if (ok) {
                tc_fence_after();
                if (mine) {
                    const uint32_t scol = tmem + lane_off + kSCol + 128 * buf + 64 * set;
                    tmem_ld32(scol, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                    tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                    tmem_wait_ld();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars + 8 * (kSFree0 + buf));  // QK of group G + 2 may start
                if (mine) mx = page_max(sr, valid);
            }

            // group max, agreed between the two sets, drives the lazy rescale
            xs[set * 128 + row] = mx * p.scale_log2;
            if (named_barrier_or(kSoftmaxBarrier, 256, !ok || *w.abort)) return;
            const float gm = fmaxf(xs[row], xs[128 + row]);
            float factor = 1.f;
            if (gm > m_used + kRescaleThreshold) {
                if (pg != it.page_begin) factor = ex2_approx(m_used - gm);
                m_used = gm;
            }
            l_mine *= factor;

            // P of my page goes into staging slot (message % 4), free once the value CTA has
            // consumed the message four before; every page but the item's last is handed to the
            // shipper at once, the last waits for 1/l below
            const int gg = g + set;
            const int slot = gg % kStagingSlots;
            const float f_page = set == 0 ? factor : 1.f;  // the O rescale precedes the group's first page
            const bool hold_last = mine && t == it.page_end - 1;
            if (mine && ok) {
                if (gg >= kStagingSlots)
                    ok = wait_freed(freed, (uint32_t)(gg - kStagingSlots + 1), w);
                if (ok) {
                    l_mine += page_softmax(sr, valid, p.scale_log2, m_used,
                                           smem + kOffScoreStaging + slot * kPBytes + p_row_off, row);
                    if (!hold_last) stage_message(smem, bars, slot, q4, lane, f_page, 0.f, false, valid < 64);
                }
            }
            if (last_group) {  // 1/l for the item's last page needs both sets' sums
                xs[256 + set * 128 + row] = l_mine;
                if (named_barrier_or(kSoftmaxBarrier, 256, !ok || *w.abort)) return;
                l_total = xs[256 + row] + xs[256 + 128 + row];
                if (hold_last) stage_message(smem, bars, slot, q4, lane, f_page, 1.f / l_total, true, valid < 64);
            }
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

__device__ __forceinline__ void value_mma(const Params& p, int item_begin, int item_end, int items_off,
                                          const uint8_t* smem, uint32_t sbase, uint32_t bars, uint32_t tmem,
                                          const dev::WaitCtx& w)
{
    using namespace dev;
    constexpr uint32_t idesc = idesc_f16(128, 256, false, true);  // f16 P x f16 latent page
    const uint64_t p_desc0 = smem_desc(sbase + kOffP, 16, 1024);
    const uint64_t v_desc0 = smem_desc(sbase, kBoxBytes, 1024);
    int g = 0, n_flagged = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int s = g % kValueStages, buf = g & 1;
            if (!wait_phase(bars + 8 * (kFull0 + s), g / kValueStages, w)) goto out;
            // expect this message's bytes (the copies may land before or after this)
            mbar_arrive_expect_tx(bars + 8 * (kMsgFull0 + buf), kMsgBytes);
            if (!wait_phase<true>(bars + 8 * (kMsgFull0 + buf), g >> 1, w)) goto out;
            // The correction warps go first on flagged tiles (rescale O, zero a tail) and on the
            // first tile of every item after the first (their epilogue still reads O, which this
            // PV overwrites).  Both sides apply the same rule, so o_ready phases stay paired.
            if (msg_flags(smem, buf) != 0 || (t == it.page_begin && i != item_begin)) {
                const int e = n_flagged & 1;
                mma_commit(bars + 8 * (kODrain0 + e));  // arrives once every earlier PV is done
                if (!wait_phase(bars + 8 * (kOReady0 + e), n_flagged >> 1, w)) goto out;
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
    int g = 0, n_flagged = 0;
    Item prev{};
    float prev_inv_l = 0.f;
    bool have_prev = false;  // an item whose output is still in TMEM
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        float inv_l = 0.f;
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int buf = g & 1;
            if (!wait_warp<true>(bars + 8 * (kMsgFull0 + buf), g >> 1, w)) goto done;
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
            if (!wait_warp(bars + 8 * (kODrain0 + e), n_flagged >> 1, w)) goto done;
            tc_fence_after();
            if (boundary) {  // the previous item's output leaves TMEM before this PV overwrites it
                write_output(p, prev, prev_inv_l, tmem, lane_off, row);
                have_prev = false;
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
        }
        prev = it;
        prev_inv_l = inv_l;
        have_prev = true;
    }
    if (have_prev) {
        // last item: every PV is done when the MMA thread's final commit lands
        if (!wait_warp(bars + 8 * kDrain, 0, w)) goto done;
        tc_fence_after();
        write_output(p, prev, prev_inv_l, tmem, lane_off, row);
    }
done:
    tc_fence_before();
}

// ---------------------------------------------------------------------------- kernel

// 15 warps: three SM sub-partitions hold four of them, and a sub-partition's 16K registers then
// allow at most 4 x 32 x 128.
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(128)
decode_fp8_kernel(const __grid_constant__ CUtensorMap tm_c8, const __grid_constant__ CUtensorMap tm_kr, const Params p)
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
        // score CTA: one converter warp (or the k_R load) per ring slot fill; value CTA: eight
        const uint32_t fillers = rank == 0 ? 1u : (uint32_t)kValueConvertWarps;
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(bars + 8 * (kFull0 + s), fillers);
            mbar_init(bars + 8 * (kEmpty0 + s), 1);
        }
        for (int s = 0; s < kRawSlots; ++s) {
            mbar_init(bars + 8 * (kRawFull0 + s), 1);  // producer's arm + TMA bytes
            mbar_init(bars + 8 * (kRawEmpty0 + s), fillers);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars + 8 * (kSFull0 + b), 1);
            mbar_init(bars + 8 * (kSFree0 + b), 8);        // one arrive per softmax warp
            mbar_init(bars + 8 * (kMsgFree0 + b), 1 + 4);  // PV commit + four correction warps
            mbar_init(bars + 8 * (kMsgFull0 + b), 1);      // the MMA thread's arm + the copies' bytes
            mbar_init(bars + 8 * (kOReady0 + b), 128);
            mbar_init(bars + 8 * (kODrain0 + b), 1);
        }
        mbar_init(bars + 8 * kQReady, 8);                  // one arrive per softmax warp
        for (int s = 0; s < kStagingSlots; ++s) mbar_init(bars + 8 * (kStgReady0 + s), 4);  // one set's warps
        *reinterpret_cast<volatile uint32_t*>(smem + kOffStgFreed) = 0;
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
                score_producer(&tm_c8, &tm_kr, p, item_begin, item_end, items_off, sbase, bars, w, lane);
            else if (warp == 1) {
                if (lane == 0) score_mma(p, item_begin, item_end, items_off, sbase, bars, tmem, w);
            } else if (warp >= 2 && warp < 10)
                score_softmax(p, item_begin, item_end, items_off, smem, sbase, bars, tmem, w, warp, lane);
            else if (warp == kShipperWarp) {
                if (lane == 0) score_shipper(p, item_begin, item_end, items_off, smem, sbase, bars, w);
            } else if (warp >= kScoreConvertWarp0 && warp < kScoreConvertWarp0 + kScoreConvertWarps)
                score_convert(p, item_begin, item_end, items_off, smem, bars, w, warp - kScoreConvertWarp0, lane);
        } else {
            if (warp == 0)
                value_producer(&tm_c8, p, item_begin, item_end, items_off, sbase, bars, w, lane);
            else if (warp == 1) {
                if (lane == 0) value_mma(p, item_begin, item_end, items_off, smem, sbase, bars, tmem, w);
            } else if (warp >= 2 && warp < 6)
                value_correction(p, item_begin, item_end, items_off, smem, bars, tmem, w, warp, lane,
                                 threadIdx.x - 64);
            else if (warp >= kValueConvertWarp0 && warp < kValueConvertWarp0 + kValueConvertWarps)
                value_convert(p, item_begin, item_end, items_off, smem, bars, w, warp - kValueConvertWarp0, lane);
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
