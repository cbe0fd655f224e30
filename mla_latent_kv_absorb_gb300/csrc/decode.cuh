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
//   rank 0, the score CTA: q = [q_abs | q_R] lives in TMEM (288 columns, the A operand of a
//     "TS" MMA), scores go to two 64-column TMEM buffers; four warps run the softmax and write
//     P (bf16, 16 KB per page) straight into the value CTA's shared memory (DSMEM).
//   rank 1, the value CTA: O lives in TMEM (512 columns); per page it runs PV from P and its
//     own copy of the page's 512 latent columns; four warps apply the (rare) rescales and
//     write the normalised output.
// Both CTAs stream the same pages with their own TMA ring (the second read of a page is an L2
// hit), so HBM sees each page once.
//
// Online softmax with lazy rescaling: the running max m used for exp2 only moves when a tile's
// max exceeds it by more than 8 (log2 units); then l and O are scaled by exp2(m_old - m_new).
// P values stay <= 2^8, and the final division by l makes the result exact whatever m is.
//
// Pipelines (all waits bounded; see ptx.cuh):
//   kv_full/kv_empty[3]   TMA ring of pages (per CTA)
//   s_full/s_free[2]      score buffers (score CTA)
//   q_ready               query loaded into TMEM for an item (score CTA)
//   msg_full[2]           P + per-row factors landed in the value CTA (arrived remotely)
//   msg_free[2]           PV using that P finished (value CTA's MMA commit, multicast to rank 0)
//   o_ready[2]            value CTA's correction warps done with a tile (rescale, tail zeroing)
//   pv_done               every PV (value CTA)
#pragma once
#include "plan.h"
#include "ptx.cuh"

namespace mla {
namespace decode {

constexpr int kThreads = 192;
constexpr int kStages = 3;
constexpr int kBoxBytes = 64 * 128;               // 64 tokens x 64 bf16 columns
constexpr int kScoreStageBytes = 9 * kBoxBytes;   // 73,728: c_KV (8 boxes) + k_R (1 box)
constexpr int kValueStageBytes = 8 * kBoxBytes;   // 65,536: c_KV only
constexpr int kPBytes = 128 * 128;                // P: 128 heads x 64 tokens bf16
constexpr int kOffP = kStages * kValueStageBytes; // value CTA: two P buffers
constexpr int kOffFactor = kOffP + 2 * kPBytes;   // float [2][128]
constexpr int kOffInvL = kOffFactor + 2 * 512;    // float [2][128]
constexpr int kOffBars = kOffInvL + 2 * 512;

enum Bar : int {
    kFull0 = 0,
    kEmpty0 = 3,
    kSFull0 = 6,
    kSFree0 = 8,
    kQReady = 10,
    kMsgFree0 = 11,
    kMsgFull0 = 13,
    kOReady0 = 15,
    kPvDone = 17,
    kDrain = 18,
    kNumBars = 19
};

constexpr int kOffTmemHolder = kOffBars + 8 * kNumBars;
constexpr int kOffAbort = kOffTmemHolder + 4;
constexpr int kSmemBytes = ((kOffAbort + 4 + 127) / 128) * 128;
static_assert(kStages * kScoreStageBytes <= kOffFactor, "score stages overlap the message area");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM columns
constexpr uint32_t kQCol = 0;      // score CTA: query, 288 columns (576 bf16 per lane)
constexpr uint32_t kSCol = 320;    // score CTA: two 64-column score buffers
constexpr uint32_t kTmemCols = 512;

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8

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

// Streams the pages of this cluster's items into the ring; `boxes` 64-column boxes per page
// (9 for the score CTA: latent + RoPE key, 8 for the value CTA: latent only).
__device__ __forceinline__ void run_producer(const CUtensorMap* tm, const Params& p, int item_begin, int item_end,
                                             int items_off, uint32_t sbase, uint32_t bars, int boxes,
                                             int stage_bytes, const dev::WaitCtx& w, int lane)
{
    using namespace dev;
    const uint64_t policy = l2_policy_evict_first();
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
                    const int s = g % kStages;
                    if (g >= kStages) ok = wait_phase(bars + 8 * (kEmpty0 + s), g / kStages - 1, w);
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
        for (int k = (g > kStages ? g - kStages : 0); k < g; ++k)
            drain_phase(bars + 8 * (kFull0 + k % kStages), k / kStages, w.timeout_ns);
    }
}

// ---------------------------------------------------------------------------- score CTA

__device__ __forceinline__ void score_mma(const Params& p, int item_begin, int item_end, int items_off, uint32_t sbase,
                                          uint32_t bars, uint32_t tmem, const dev::WaitCtx& w)
{
    using namespace dev;
    constexpr uint32_t idesc = idesc_bf16(128, 64, false, false);
    int g = 0, n_item = 0;
    for (int i = item_begin; i < item_end; ++i, ++n_item) {
        const Item it = load_item(p.plan, items_off, i);
        if (!wait_phase(bars + 8 * kQReady, n_item, w)) goto out;
        tc_fence_after();
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int s = g % kStages, buf = g & 1;
            if (!wait_phase(bars + 8 * (kFull0 + s), g / kStages, w)) goto out;
            if (g >= 2 && !wait_phase(bars + 8 * (kSFree0 + buf), (g >> 1) - 1, w)) goto out;
            tc_fence_after();
            const uint32_t d = tmem + kSCol + 64 * buf;
            const uint32_t stage = sbase + s * kScoreStageBytes;
#pragma unroll
            for (int k = 0; k < 36; ++k) {
                // K step k covers row dims 16k..16k+15: box k/4, 32-byte column step k%4
                const uint64_t b_desc = smem_desc(stage + (k >> 2) * kBoxBytes + (k & 3) * 32, 16, 1024);
                mma_ts(d, tmem + kQCol + 8 * k, b_desc, idesc, k > 0 ? 1u : 0u);
            }
            mma_commit(bars + 8 * (kEmpty0 + s));
            mma_commit(bars + 8 * (kSFull0 + buf));
        }
    }
out:
    mma_commit(bars + 8 * kDrain);
    drain_phase(bars + 8 * kDrain, 0, w.timeout_ns);
}

__device__ __forceinline__ void score_softmax(const Params& p, int item_begin, int item_end, int items_off,
                                              uint32_t sbase, uint32_t bars, uint32_t tmem, const dev::WaitCtx& w,
                                              int warp, int lane)
{
    using namespace dev;
    const int q4 = warp & 3, row = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    // addresses in the value CTA (rank 1)
    const uint32_t r_p = map_to_cta(sbase + kOffP, 1);
    const uint32_t r_factor = map_to_cta(sbase + kOffFactor, 1);
    const uint32_t r_invl = map_to_cta(sbase + kOffInvL, 1);
    const uint32_t r_msg_full = map_to_cta(bars + 8 * kMsgFull0, 1);
    const uint32_t p_row_off = (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
    int g = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        // query row -> TMEM lane `row`, columns 0..287 (two bf16 per column, K order)
        {
            const uint4* qa = reinterpret_cast<const uint4*>(p.q_abs + ((int64_t)it.seq * 128 + row) * 512);
            const uint4* qr = reinterpret_cast<const uint4*>(p.q_r + ((int64_t)it.seq * 128 + row) * 64);
#pragma unroll 1
            for (int c = 0; c < 9; ++c) {
                uint32_t r[32];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const uint4 x = (c < 8) ? __ldg(qa + 8 * c + v) : __ldg(qr + v);
                    r[4 * v + 0] = x.x;
                    r[4 * v + 1] = x.y;
                    r[4 * v + 2] = x.z;
                    r[4 * v + 3] = x.w;
                }
                tmem_st32(tmem + lane_off + kQCol + 32 * c, r);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bars + 8 * kQReady);
        }
        float m_used = -INFINITY, l = 0.f;
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int buf = g & 1;
            if (!wait_warp(bars + 8 * (kSFull0 + buf), g >> 1, w)) return;
            tc_fence_after();
            uint32_t sr[64];
            tmem_ld32(tmem + lane_off + kSCol + 64 * buf, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
            tmem_ld32(tmem + lane_off + kSCol + 64 * buf + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bars + 8 * (kSFree0 + buf));

            const int valid = min(64, it.seq_len - 64 * t);
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float x = (j < valid) ? __uint_as_float(sr[j]) * p.scale_log2 : -INFINITY;
                sr[j] = __float_as_uint(x);
                mx = fmaxf(mx, x);
            }
            float factor = 1.f;
            if (mx > m_used + kRescaleThreshold) {
                if (t != it.page_begin) {
                    factor = exp2f(m_used - mx);
                    l *= factor;
                }
                m_used = mx;
            }
            uint32_t pk[32];
            float psum = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float p0 = exp2f(__uint_as_float(sr[2 * j]) - m_used);
                const float p1 = exp2f(__uint_as_float(sr[2 * j + 1]) - m_used);
                pk[j] = pack_bf16x2(p0, p1);
                psum += bf16_lo(pk[j]) + bf16_hi(pk[j]);
            }
            l += psum;

            if (g >= 2 && !wait_warp<true>(bars + 8 * (kMsgFree0 + buf), (g >> 1) - 1, w)) return;
            const uint32_t dst = r_p + buf * kPBytes + p_row_off;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_cluster_v4(dst + ((uint32_t)(c ^ (row & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                              pk[4 * c + 3]);
            st_cluster_f32(r_factor + buf * 512 + 4 * row, factor);
            if (t == it.page_end - 1) st_cluster_f32(r_invl + buf * 512 + 4 * row, 1.f / l);
            fence_proxy_async_cluster();
            mbar_arrive_remote(r_msg_full + 8 * buf);
        }
        const float lse_val = (m_used + log2f(l)) * 0.69314718055994531f;
        if (it.slot < 0)
            p.lse[(int64_t)it.seq * 128 + row] = lse_val;
        else
            p.ws_lse[(int64_t)it.slot * 128 + row] = lse_val;
    }
    // the value CTA's last commits arrive here: wait for them before this CTA can finish
    for (int k = (g > 2 ? g - 2 : 0); k < g; ++k)
        if (!wait_warp<true>(bars + 8 * (kMsgFree0 + (k & 1)), k >> 1, w)) return;
}

// ---------------------------------------------------------------------------- value CTA

__device__ __forceinline__ void value_mma(const Params& p, int item_begin, int item_end, int items_off, uint32_t sbase,
                                          uint32_t bars, uint32_t tmem, const dev::WaitCtx& w)
{
    using namespace dev;
    constexpr uint32_t idesc = idesc_bf16(128, 256, false, true);
    int g = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int s = g % kStages, buf = g & 1;
            if (!wait_phase(bars + 8 * (kFull0 + s), g / kStages, w)) goto out;
            if (!wait_phase<true>(bars + 8 * (kMsgFull0 + buf), g >> 1, w)) goto out;
            if (!wait_phase(bars + 8 * (kOReady0 + buf), g >> 1, w)) goto out;
            tc_fence_after();
            const uint32_t stage = sbase + s * kValueStageBytes;
            const uint32_t pbuf = sbase + kOffP + buf * kPBytes;
            const bool first = (t == it.page_begin);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    // A = P [128 heads x 16 tokens] K-major; B = page [16 tokens x 256 dims] MN-major
                    const uint64_t a_desc = smem_desc(pbuf + k * 32, 16, 1024);
                    const uint64_t b_desc = smem_desc(stage + half * 4 * kBoxBytes + k * 2048, kBoxBytes, 1024);
                    mma_ss(tmem + 256 * half, a_desc, b_desc, idesc, (!first || k > 0) ? 1u : 0u);
                }
            }
            mma_commit(bars + 8 * (kEmpty0 + s));
            mma_commit(bars + 8 * kPvDone);
            mma_commit_multicast(bars + 8 * (kMsgFree0 + buf), 0x1);
        }
    }
out:
    mma_commit(bars + 8 * kDrain);
    drain_phase(bars + 8 * kDrain, 0, w.timeout_ns);
}

__device__ __forceinline__ bool wait_pv(uint32_t bars, int upto, int& seen, const dev::WaitCtx& w)
{
    while (seen < upto) {
        if (!dev::wait_warp(bars + 8 * kPvDone, seen, w)) return false;
        ++seen;
    }
    return true;
}

__device__ __forceinline__ void value_correction(const Params& p, int item_begin, int item_end, int items_off,
                                                 uint8_t* smem, uint32_t sbase, uint32_t bars, uint32_t tmem,
                                                 const dev::WaitCtx& w, int warp, int lane, int tid128)
{
    using namespace dev;
    const int q4 = warp & 3, row = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float* factors = reinterpret_cast<const float*>(smem + kOffFactor);
    const float* invls = reinterpret_cast<const float*>(smem + kOffInvL);
    int g = 0, pv_seen = 0;
    for (int i = item_begin; i < item_end; ++i) {
        const Item it = load_item(p.plan, items_off, i);
        float inv_l = 0.f;
        for (int t = it.page_begin; t < it.page_end; ++t, ++g) {
            const int buf = g & 1;
            if (!wait_warp<true>(bars + 8 * (kMsgFull0 + buf), g >> 1, w)) return;
            const float factor = factors[buf * 128 + row];
            if (t == it.page_end - 1) inv_l = invls[buf * 128 + row];
            const int valid = min(64, it.seq_len - 64 * t);
            if (valid < 64) {
                // slots past the sequence end may hold anything (NaN): zero them so that
                // p = 0 times them stays 0 in the PV contraction
                const int s = g % kStages;
                if (!wait_warp(bars + 8 * (kFull0 + s), g / kStages, w)) return;
                uint8_t* stage = smem + s * kValueStageBytes;
                const int chunks = (64 - valid) * 64;  // rows x (8 boxes x 8 chunks of 16 B)
                for (int c = tid128; c < chunks; c += 128) {
                    const int r = valid + (c >> 6), box = (c >> 3) & 7, ch = c & 7;
                    *reinterpret_cast<uint4*>(stage + box * kBoxBytes + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_cta();
            }
            const bool need = (t != it.page_begin) && (factor != 1.f);
            if (__any_sync(0xffffffffu, need)) {
                if (!wait_pv(bars, g, pv_seen, w)) return;
                tc_fence_after();
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
            mbar_arrive(bars + 8 * (kOReady0 + buf));
        }
        // epilogue: O / l
        if (!wait_pv(bars, g, pv_seen, w)) return;
        tc_fence_after();
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
        tc_fence_before();
    }
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
        mbar_init(bars + 8 * kFull0 + 0, 1);
        mbar_init(bars + 8 * kFull0 + 8, 1);
        mbar_init(bars + 8 * kFull0 + 16, 1);
        for (int s = 0; s < kStages; ++s) mbar_init(bars + 8 * (kEmpty0 + s), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars + 8 * (kSFull0 + b), 1);
            mbar_init(bars + 8 * (kSFree0 + b), 128);
            mbar_init(bars + 8 * (kMsgFree0 + b), 1);
            mbar_init(bars + 8 * (kMsgFull0 + b), 128);
            mbar_init(bars + 8 * (kOReady0 + b), 128);
        }
        mbar_init(bars + 8 * kQReady, 128);
        mbar_init(bars + 8 * kPvDone, 1);
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
                run_producer(&tm_pool, p, item_begin, item_end, items_off, sbase, bars, 9, kScoreStageBytes, w, lane);
            else if (warp == 1) {
                if (lane == 0) score_mma(p, item_begin, item_end, items_off, sbase, bars, tmem, w);
            } else
                score_softmax(p, item_begin, item_end, items_off, sbase, bars, tmem, w, warp, lane);
        } else {
            if (warp == 0)
                run_producer(&tm_pool, p, item_begin, item_end, items_off, sbase, bars, 8, kValueStageBytes, w, lane);
            else if (warp == 1) {
                if (lane == 0) value_mma(p, item_begin, item_end, items_off, sbase, bars, tmem, w);
            } else
                value_correction(p, item_begin, item_end, items_off, smem, sbase, bars, tmem, w, warp, lane,
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
