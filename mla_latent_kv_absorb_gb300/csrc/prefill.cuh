// prefill.cuh -- causal attention of a chunk of new tokens over their sequence in the
// decompressed form (page 1 section 4, path A: per-head keys k_h = W_UK[h] c and values
// v_h = W_UV[h] c; section 6: chunks of at least the prefill threshold of 256 new tokens take
// this form, shorter ones the absorbed decode).
//
// The chunk's T new tokens are positions S - T .. S - 1 of a sequence of S tokens whose cache
// rows are already written; query i (position S - T + i) attends to keys 0 .. S - T + i:
//   s_ij = (q_c[i,h] . k[h,j] + q_R[i,h] . k_R[j]) * softmax_scale,
//   out[i,h] = sum_j softmax_j(s_ij) v[h,j].
// The keys and values were decompressed before this kernel into k [128][S][128] and
// v [128][S][128] (head-major); k_R comes from the gathered cache rows [S][576] (columns
// 512..575).
//
// One CTA = two tiles of 128 queries (A and B) of one head, sharing every 64-key tile, so 40 KB
// of keys and values feed twice the MMA work (the per-SM TMA ingress, not the tensor core, set
// the pace with one query tile).  Keys (k and k_R, 24 KB a tile) and values (16 KB) have rings
// of their own, three stages each: a key stage is refilled as soon as its QK products are
// done, long before the tile's PV.  Warp 0 streams the queries and keys, warp 2 the values,
// warp 1 issues the MMAs (PV of tile n, then QK of tile n + 2), warps 3-6 run the online
// softmax of query tile A and warps 7-10 that of B, one query row per thread (its TMEM lane).
// TMEM per query tile: two 64-column score buffers and a 128-column output (512 columns in
// all).  P goes back into the first 32 columns of its score buffer (bf16 pairs), where the PV
// MMA reads it as a tensor-memory operand: no shared memory for P, and no wait on the previous
// PV before it is written (the buffer's last reader, PV of tile n - 2, finished before the
// scores of tile n were complete).
//   QK:  S[128 x 64]  = Q [128 x 192] (q_c | q_R, three 64-column K-major chunks in shared memory)
//                       x K tile [64 x 192] (k | k_R, three K-major chunks)
//   PV:  O[128 x 128] += P [128 x 64] (bf16 in TMEM)
//                       x V tile [64 keys x 128] (MN-major: keys are K, dims are N)
// The running max moves only when a tile's max exceeds it by more than 8 (log2 units); the
// output is then rescaled in TMEM before the tile's PV.  Every wait is bounded.
#pragma once
#include "ptx.cuh"
#ifdef MLA_PREFILL_TRACE
#include <cstdio>
#endif

namespace mla {
namespace prefill {

#ifdef MLA_PREFILL_TRACE
// instrumented builds only: event times (ns from the CTA's start) of CTA (0, 0), printed at its end
constexpr int kTraceTiles = 24;
#define PF_TRACE(arr, n, k) \
    do { if (trace_cta && (n) < kTraceTiles) (arr)[(n) * 4 + (k)] = globaltimer_ns() - trace_t0; } while (0)
#else
#define PF_TRACE(arr, n, k) \
    do { } while (0)
#endif

constexpr int kQ = 128;        // queries per query tile (MMA M)
constexpr int kQT = 2;         // query tiles per CTA
constexpr int kKV = 64;        // keys per key/value tile
constexpr int kThreads = 32 * (3 + 4 * kQT);  // warps 0, 2 TMA, warp 1 MMA + TMEM, 4 softmax warps per query tile
constexpr int kSoftmaxWarp0 = 3;
constexpr int kQChunk = kQ * 64 * 2;                       // [128 rows][64] bf16, 16 KB
constexpr int kQBytes = 3 * kQChunk;                       // one query tile: q_c 0-63, q_c 64-127, q_R
constexpr int kKVBox = kKV * 64 * 2;                       // [64 rows][64] bf16, 8 KB
constexpr int kKStage = 3 * kKVBox;                        // k 0-63, k 64-127, k_R
constexpr int kVStage = 2 * kKVBox;                        // v 0-63, v 64-127
constexpr int kStages = 3;
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQT * kQBytes;               // 96 KB
constexpr int kOffV = kOffK + kStages * kKStage;           // 168 KB
constexpr int kOffBar = kOffV + kStages * kVStage;         // 216 KB
constexpr int kSmemBytes = kOffBar + 256;
constexpr uint32_t kTmemCols = 512;                        // per query tile t: S at 256 t + {0, 64}, O at 256 t + 128
constexpr float kRescaleLog2 = 8.f;

struct Params {
    int seq_len;          // S
    int chunk_len;        // T
    float scale_log2;     // softmax_scale * log2(e)
    __nv_bfloat16* out;   // [T][128][128]
    uint32_t* dev_error;
    uint64_t timeout_ns;
};

// barrier slots (8 bytes each) from kOffBar
enum : int {
    kBarQ = 0,
    kBarKFull = 1,      // [stage]
    kBarKEmpty = 4,     // [stage]
    kBarVFull = 7,      // [stage]
    kBarVEmpty = 10,    // [stage]
    kBarSFull = 13,     // [tile][buffer]
    kBarPReady = 17,    // [tile][buffer], 128 arrivals
    kBarPvDone = 21,    // [tile]
    kBarDone = 23,      // every MMA of the CTA has finished
    kBarCount = 24,
};
// Phase bookkeeping.  A barrier waited by parity must never run two phases ahead of its waiter:
//   S full [t][b]   completes for tiles b, b + 2, ...; QK of tile n + 2 is issued only after the
//                   MMA thread has seen P of tile n ready, so the softmax is never two behind.
//   P ready [t][b]  arrives for tiles b, b + 2, ...; the softmax makes P of tile n + 2 only from
//                   the scores of tile n + 2, which follow the PV of tile n.
//   PV done [t]     completes for every tile; the softmax waits it (for tile n - 1) only while
//                   at tile n, after the scores of tile n, whose commit covers the PV of tile
//                   n - 2, so exactly one phase can be pending.  The final read of O waits on
//                   kBarDone instead.

__global__ void __launch_bounds__(kThreads, 1)
prefill_attn_kernel(const __grid_constant__ CUtensorMap tm_qc, const __grid_constant__ CUtensorMap tm_qr,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_kr,
                    const __grid_constant__ CUtensorMap tm_v, const Params p)
{
    using namespace dev;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = blockIdx.x * kQ * kQT, h = blockIdx.y;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kOffBar;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kBarCount);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const auto bar = [&](int id, int k) { return bars + 8 * (id + k); };

    if (sbase & 1023u) {
        if (threadIdx.x == 0) raise_error(p.dev_error, MLA_DEVERR_SMEM_ALIGN);
        return;
    }
    // key/value tiles this CTA needs: up to the position of its last valid query
    const int first_pos = p.seq_len - p.chunk_len;
    const int last_q = min(i0 + kQ * kQT, p.chunk_len) - 1;
    const int n_tiles = (first_pos + last_q) / kKV + 1;

    if (threadIdx.x == 0) {
        mbar_init(bar(kBarQ, 0), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarKFull, s), 1);
            mbar_init(bar(kBarKEmpty, s), 1);
            mbar_init(bar(kBarVFull, s), 1);
            mbar_init(bar(kBarVEmpty, s), 1);
        }
        for (int t = 0; t < kQT; ++t) {
            mbar_init(bar(kBarSFull, 2 * t), 1);
            mbar_init(bar(kBarSFull, 2 * t + 1), 1);
            mbar_init(bar(kBarPReady, 2 * t), 128);
            mbar_init(bar(kBarPReady, 2 * t + 1), 128);
            mbar_init(bar(kBarPvDone, t), 1);
        }
        mbar_init(bar(kBarDone, 0), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtx w{p.timeout_ns, abort_flag, p.dev_error};
#ifdef MLA_PREFILL_TRACE
    const bool trace_cta = blockIdx.x == 0 && blockIdx.y == 0;
    const uint64_t trace_t0 = globaltimer_ns();
    uint64_t tr[kTraceTiles * 4] = {};
#endif

    if (warp == 0 || warp == 2) {
        if (lane == 0) {
            // warp 0: the queries, then the key tiles; warp 2: the value tiles
            const uint64_t pol = l2_policy_evict_last();  // the head's other query tiles re-read them
            const bool keys = warp == 0;
            if (keys) {
                mbar_arrive_expect_tx(bar(kBarQ, 0), kQT * kQBytes);
                for (int t = 0; t < kQT; ++t) {
                    const uint32_t q = sbase + kOffQ + t * kQBytes;
                    tma_load_3d(q, &tm_qc, bar(kBarQ, 0), 0, h, i0 + kQ * t, pol);
                    tma_load_3d(q + kQChunk, &tm_qc, bar(kBarQ, 0), 64, h, i0 + kQ * t, pol);
                    tma_load_3d(q + 2 * kQChunk, &tm_qr, bar(kBarQ, 0), 0, h, i0 + kQ * t, pol);
                }
            }
            const int full_id = keys ? kBarKFull : kBarVFull, empty_id = keys ? kBarKEmpty : kBarVEmpty;
            int issued = 0;
            for (int n = 0; n < n_tiles; ++n) {
                const int s = n % kStages;
                if (n >= kStages && !wait_phase(bar(empty_id, s), (n / kStages - 1) & 1, w)) break;
                const uint32_t full = bar(full_id, s);
                const int j0 = n * kKV;
                if (keys) {
                    const uint32_t st = sbase + kOffK + s * kKStage;
                    mbar_arrive_expect_tx(full, kKStage);
                    tma_load_3d(st, &tm_k, full, 0, j0, h, pol);
                    tma_load_3d(st + kKVBox, &tm_k, full, 64, j0, h, pol);
                    tma_load_2d(st + 2 * kKVBox, &tm_kr, full, 512, j0, pol);
                } else {
                    const uint32_t st = sbase + kOffV + s * kVStage;
                    mbar_arrive_expect_tx(full, kVStage);
                    tma_load_3d(st, &tm_v, full, 0, j0, h, pol);
                    tma_load_3d(st + kKVBox, &tm_v, full, 64, j0, h, pol);
                }
                ++issued;
            }
            // loads in flight land before the CTA can exit
            if (keys) drain_phase(bar(kBarQ, 0), 0, w.timeout_ns);
            for (int n = (issued > kStages ? issued - kStages : 0); n < issued; ++n)
                drain_phase(bar(full_id, n % kStages), (n / kStages) & 1, w.timeout_ns);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, kKV, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, 128, false, true);
            // both query tiles' scores for key tile n; the key stage is released when they finish
            const auto issue_qk = [&](int n) -> bool {
                const int s = n & 1, ks = n % kStages;
                if (!wait_phase(bar(kBarKFull, ks), (n / kStages) & 1, w)) return false;
                tc_fence_after();
                const uint32_t st = sbase + kOffK + ks * kKStage;
#pragma unroll 1
                for (int t = 0; t < kQT; ++t) {
#pragma unroll 1
                    for (int c = 0; c < 3; ++c) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t a = smem_desc(sbase + kOffQ + t * kQBytes + c * kQChunk + 32 * k, 16, 1024);
                            const uint64_t b = smem_desc(st + c * kKVBox + 32 * k, 16, 1024);
                            mma_ss(tmem + 256 * t + s * kKV, a, b, idesc_qk, (c | k) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(bar(kBarSFull, 2 * t + s));
                }
                mma_commit(bar(kBarKEmpty, ks));
                return true;
            };
            bool ok = wait_phase(bar(kBarQ, 0), 0, w) && (tc_fence_after(), issue_qk(0)) &&
                      (n_tiles < 2 || issue_qk(1));
            for (int n = 0; ok && n < n_tiles; ++n) {
                // PV of tile n for both query tiles, then the scores of tile n + 2 into the freed
                // score buffers
                const int vs = n % kStages;
                if (!(ok = wait_phase(bar(kBarVFull, vs), (n / kStages) & 1, w))) break;
                PF_TRACE(tr, n, 0);
                const uint32_t vt = sbase + kOffV + vs * kVStage;
#pragma unroll 1
                for (int t = 0; t < kQT && ok; ++t) {
                    if (!(ok = wait_phase(bar(kBarPReady, 2 * t + (n & 1)), (n >> 1) & 1, w))) break;
                    PF_TRACE(tr, n, 1 + t);
                    tc_fence_after();
                    const uint32_t pt = tmem + 256 * t + (n & 1) * kKV;  // P in its score buffer
#pragma unroll
                    for (int k = 0; k < kKV / 16; ++k) {
                        const uint64_t b = smem_desc(vt + 2048 * k, 8192, 1024);
                        mma_ts(tmem + 256 * t + 128, pt + 8 * k, b, idesc_pv, (n | k) != 0 ? 1u : 0u);
                    }
                    mma_commit(bar(kBarPvDone, t));
                }
                if (!ok) break;
                mma_commit(bar(kBarVEmpty, vs));
                if (n + 2 < n_tiles && !(ok = issue_qk(n + 2))) break;
                PF_TRACE(tr, n, 3);
            }
            mma_commit(bar(kBarDone, 0));  // arrives when every MMA issued here has finished
#ifdef MLA_PREFILL_TRACE
            if (trace_cta)
                for (int n = 0; n < kTraceTiles && n < n_tiles; ++n)
                    printf("mma %2d v %7llu pA %7llu pB %7llu qk+2 %7llu\n", n, (unsigned long long)tr[4 * n],
                           (unsigned long long)tr[4 * n + 1], (unsigned long long)tr[4 * n + 2],
                           (unsigned long long)tr[4 * n + 3]);
#endif
        }
    } else {
        // softmax of query tile t: warp (3..10) & 3 selects the TMEM lane quarter, one row per thread
        const int t = (warp - kSoftmaxWarp0) >> 2;
        const int q4 = warp & 3, row = 32 * q4 + lane, i = i0 + kQ * t + row;
        const int qpos = min(first_pos + i, p.seq_len - 1);
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const uint32_t t_s = tmem + lane_base + 256 * t, t_o = t_s + 128;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int n = 0; n < n_tiles; ++n) {
            const int s = n & 1;
            if (!(ok = wait_warp(bar(kBarSFull, 2 * t + s), (n >> 1) & 1, w))) break;
            PF_TRACE(tr, n, 0);
            tc_fence_after();
            uint32_t r[2][32];
            tmem_ld32(t_s + s * kKV, r[0]);
            tmem_ld32(t_s + s * kKV + 32, r[1]);
            tmem_wait_ld();
            const int j0 = n * kKV;
            float x[64];
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float v = __uint_as_float(r[c >> 5][c & 31]) * p.scale_log2;
                x[c] = j0 + c <= qpos ? v : -INFINITY;
                mt = fmaxf(mt, x[c]);
            }
            // the running max: set by the first tile, moved later only by more than the threshold
            const bool grow = n > 0 && mt > m + kRescaleLog2;
            const float f = grow ? ex2_approx(m - mt) : 1.f;
            if (n == 0 || grow) m = mt;
            float sum = 0.f;
            uint32_t pk[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float a = ex2_approx(x[2 * k] - m), b = ex2_approx(x[2 * k + 1] - m);
                sum += a + b;
                pk[k] = pack_bf16x2(a, b);
            }
            l = l * f + sum;
            if (__any_sync(0xffffffffu, grow)) {
                // rescale O once the previous tile's PV has finished with it; every lane of the
                // warp takes part (factor 1 where the max stayed)
                if (!(ok = wait_warp(bar(kBarPvDone, t), (n - 1) & 1, w))) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_o + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
                    tmem_st32(t_o + 32 * c, o);
                }
            }
            PF_TRACE(tr, n, 1);
            tmem_st32(t_s + s * kKV, pk);  // P over the scores it was made from
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(kBarPReady, 2 * t + s));
            PF_TRACE(tr, n, 2);
        }
#ifdef MLA_PREFILL_TRACE
        if (trace_cta && lane == 0 && (warp == kSoftmaxWarp0 || warp == kSoftmaxWarp0 + 4))
            for (int n = 0; n < kTraceTiles && n < n_tiles; ++n)
                printf("smx t%d %2d s %7llu computed %7llu arrived %7llu\n", t, n, (unsigned long long)tr[4 * n],
                       (unsigned long long)tr[4 * n + 1], (unsigned long long)tr[4 * n + 2]);
#endif
        if (ok && wait_warp(bar(kBarDone, 0), 0, w)) {
            tc_fence_after();
            const float inv = 1.f / l;
            __nv_bfloat16* dst = p.out + ((int64_t)i * 128 + h) * 128;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(t_o + 32 * c, o);
                tmem_wait_ld();
                if (i < p.chunk_len) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        d4[v] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv),
                                           pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv),
                                           pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv),
                                           pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) drain_phase(bar(kBarDone, 0), 0, w.timeout_ns);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace prefill
}  // namespace mla
