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
// One CTA = two tiles of 128 queries (A and B) of one head, sharing every 128-key tile, so the
// key and value bytes feed twice the MMA work (the per-SM TMA ingress, not the tensor core, set
// the pace with one query tile).  The tensor core's cost is per instruction up to N = 256, so
// the key tile is 128 wide: each QK instruction is M = 128 queries x N = 128 keys.  TMEM per
// query tile: one 128-column score buffer and a 128-column output (512 columns in all); the
// softmax writes P (bf16 pairs) back over the first 64 columns of its scores, where the PV MMA
// reads it as a tensor-memory operand.  With one score buffer per query tile the two tiles
// alternate: the MMA order per key tile n is PV_A(n), QK_A(n+1), PV_B(n), QK_B(n+1), so while
// one tile's softmax runs the tensor core works on the other tile's products.
//   QK:  S[128 x 128] = Q [128 x 192] (q_c | q_R, three 64-column K-major chunks in shared memory)
//                       x K tile [128 x 192] (k | k_R, three K-major chunks)
//   PV:  O[128 x 128] += P [128 x 128] (bf16 in TMEM)
//                       x V tile [128 keys x 128] (MN-major: keys are K, dims are N)
// Warp 0 streams the queries and keys (two stages), warp 2 the values (one stage: a value tile
// is needed only after the next key tile's QK products), warp 1 issues the MMAs, warps 3-6 and
// 7-10 run the online softmax of tiles A and B, one query row per thread (its TMEM lane).
// Every warp has exactly one role.  (Measured alternatives: 96-key tiles with two value stages,
// 6.7 ms on the bench chunk, and one ring of two 48 KB slots shared by keys and values, 6.4 ms,
// both slower than this layout's 5.8 ms: the wider QK instruction matters more than hiding the
// value load.)  The
// running max moves only when a tile's max exceeds it by more than 8 (log2 units); the output
// is then rescaled in TMEM before the tile's PV.  Every wait is bounded.
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
constexpr int kKV = 128;       // keys per key/value tile (QK MMA N)
constexpr int kThreads = 32 * (3 + 4 * kQT);  // warps 0, 2 TMA, warp 1 MMA + TMEM, 4 softmax warps per query tile
constexpr int kSoftmaxWarp0 = 3;
constexpr int kQChunk = kQ * 64 * 2;                       // [128 rows][64] bf16, 16 KB
constexpr int kQBytes = 3 * kQChunk;                       // one query tile: q_c 0-63, q_c 64-127, q_R
constexpr int kKVBox = kKV * 64 * 2;                       // [128 rows][64] bf16, 16 KB
constexpr int kKStage = 3 * kKVBox;                        // k 0-63, k 64-127, k_R
constexpr int kVStage = 2 * kKVBox;                        // v 0-63, v 64-127
constexpr int kKStages = 2;
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQT * kQBytes;               // 96 KB
constexpr int kOffV = kOffK + kKStages * kKStage;          // 192 KB
constexpr int kOffBar = kOffV + kVStage;                   // 224 KB
constexpr int kSmemBytes = kOffBar + 256;
constexpr uint32_t kTmemCols = 512;                        // per query tile t: S at 256 t, O at 256 t + 128
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
    kBarKEmpty = 3,     // [stage]
    kBarVFull = 5,
    kBarVEmpty = 6,
    kBarSFull = 7,      // [tile]
    kBarPReady = 9,     // [tile], 128 arrivals
    kBarDone = 11,      // every MMA of the CTA has finished
    kBarCount = 12,
};
// Phase bookkeeping.  A barrier waited by parity must never run two phases ahead of its waiter:
//   S full [t]   completes once per key tile; QK_t(n + 1) is issued only after the MMA thread has
//                seen P_t(n) ready, i.e. after the softmax finished tile n.
//   P ready [t]  arrives once per key tile; P_t(n + 1) needs S_t(n + 1), issued after PV_t(n),
//                i.e. after the MMA thread waited for P_t(n).
//   K, V rings   each stage is refilled only after its consumer's commit, waited in order.
// The rescale of O at tile n needs PV_t(n - 1) finished: S_t(n) complete implies it (QK_t(n) was
// issued after PV_t(n - 1) and a commit covers every earlier MMA of the thread).  The final read
// of O waits on kBarDone.

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
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(bar(kBarKFull, s), 1);
            mbar_init(bar(kBarKEmpty, s), 1);
        }
        mbar_init(bar(kBarVFull, 0), 1);
        mbar_init(bar(kBarVEmpty, 0), 1);
        for (int t = 0; t < kQT; ++t) {
            mbar_init(bar(kBarSFull, t), 1);
            mbar_init(bar(kBarPReady, t), 128);
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
            const int stages = keys ? kKStages : 1;
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
                const int s = n % stages;
                if (n >= stages && !wait_phase(bar(empty_id, s), (n / stages - 1) & 1, w)) break;
                const uint32_t full = bar(full_id, s);
                const int j0 = n * kKV;
                if (keys) {
                    const uint32_t st = sbase + kOffK + s * kKStage;
                    mbar_arrive_expect_tx(full, kKStage);
                    tma_load_3d(st, &tm_k, full, 0, j0, h, pol);
                    tma_load_3d(st + kKVBox, &tm_k, full, 64, j0, h, pol);
                    tma_load_2d(st + 2 * kKVBox, &tm_kr, full, 512, j0, pol);
                } else {
                    const uint32_t st = sbase + kOffV;
                    mbar_arrive_expect_tx(full, kVStage);
                    tma_load_3d(st, &tm_v, full, 0, j0, h, pol);
                    tma_load_3d(st + kKVBox, &tm_v, full, 64, j0, h, pol);
                }
                ++issued;
            }
            // loads in flight land before the CTA can exit
            if (keys) drain_phase(bar(kBarQ, 0), 0, w.timeout_ns);
            for (int n = (issued > stages ? issued - stages : 0); n < issued; ++n)
                drain_phase(bar(full_id, n % stages), (n / stages) & 1, w.timeout_ns);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, kKV, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, 128, false, true);
            // the scores of query tile t for key tile n (its key stage has landed)
            const auto issue_qk = [&](int t, int n) {
                const uint32_t st = sbase + kOffK + (n % kKStages) * kKStage;
#pragma unroll 1
                for (int c = 0; c < 3; ++c) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t a = smem_desc(sbase + kOffQ + t * kQBytes + c * kQChunk + 32 * k, 16, 1024);
                        const uint64_t b = smem_desc(st + c * kKVBox + 32 * k, 16, 1024);
                        mma_ss(tmem + 256 * t, a, b, idesc_qk, (c | k) != 0 ? 1u : 0u);
                    }
                }
                mma_commit(bar(kBarSFull, t));
            };
            // PV of query tile t for key tile n: P from its score buffer, V from the value stage
            const auto issue_pv = [&](int t, int n) {
                const uint32_t pt = tmem + 256 * t;
#pragma unroll
                for (int k = 0; k < kKV / 16; ++k) {
                    const uint64_t b = smem_desc(sbase + kOffV + 2048 * k, kKVBox, 1024);
                    mma_ts(tmem + 256 * t + 128, pt + 8 * k, b, idesc_pv, (n | k) != 0 ? 1u : 0u);
                }
            };
            bool ok = wait_phase(bar(kBarQ, 0), 0, w) && wait_phase(bar(kBarKFull, 0), 0, w);
            if (ok) {
                tc_fence_after();
                for (int t = 0; t < kQT; ++t) issue_qk(t, 0);
                mma_commit(bar(kBarKEmpty, 0));
            }
            for (int n = 0; ok && n < n_tiles; ++n) {
                const bool more = n + 1 < n_tiles;
                if (!(ok = wait_phase(bar(kBarVFull, 0), n & 1, w))) break;
                if (more && !(ok = wait_phase(bar(kBarKFull, (n + 1) % kKStages), ((n + 1) / kKStages) & 1, w)))
                    break;
                PF_TRACE(tr, n, 0);
#pragma unroll 1
                for (int t = 0; t < kQT; ++t) {
                    if (!(ok = wait_phase(bar(kBarPReady, t), n & 1, w))) break;
                    PF_TRACE(tr, n, 1 + t);
                    tc_fence_after();
                    issue_pv(t, n);
                    if (t == kQT - 1) mma_commit(bar(kBarVEmpty, 0));
                    if (more) issue_qk(t, n + 1);  // into the score buffer PV_t(n) has just read
                }
                if (!ok) break;
                if (more) mma_commit(bar(kBarKEmpty, (n + 1) % kKStages));
                PF_TRACE(tr, n, 3);
            }
            mma_commit(bar(kBarDone, 0));  // arrives when every MMA issued here has finished
#ifdef MLA_PREFILL_TRACE
            if (trace_cta)
                for (int n = 0; n < kTraceTiles && n < n_tiles; ++n)
                    printf("mma %2d kv %7llu pA %7llu pB %7llu end %7llu\n", n, (unsigned long long)tr[4 * n],
                           (unsigned long long)tr[4 * n + 1], (unsigned long long)tr[4 * n + 2],
                           (unsigned long long)tr[4 * n + 3]);
#endif
        }
    } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4 * kQT) {
        // softmax of query tile t: warp (3..10) & 3 selects the TMEM lane quarter, one row per thread
        const int t = (warp - kSoftmaxWarp0) >> 2;
        const int q4 = warp & 3, row = 32 * q4 + lane, i = i0 + kQ * t + row;
        const int qpos = min(first_pos + i, p.seq_len - 1);
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const uint32_t t_s = tmem + lane_base + 256 * t, t_o = t_s + 128;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int n = 0; n < n_tiles; ++n) {
            if (!(ok = wait_warp(bar(kBarSFull, t), n & 1, w))) break;
            PF_TRACE(tr, n, 0);
            tc_fence_after();
            const int j0 = n * kKV;
            // pass 1: the tile's row max (keys past the query's position masked)
            float mt = -INFINITY;
#pragma unroll 1
            for (int c = 0; c < kKV / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(t_s + 32 * c, r);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    if (j0 + 32 * c + k <= qpos) mt = fmaxf(mt, __uint_as_float(r[k]) * p.scale_log2);
            }
            // the running max: set by the first tile, moved later only by more than the threshold
            const bool grow = n > 0 && mt > m + kRescaleLog2;
            const float f = grow ? ex2_approx(m - mt) : 1.f;
            if (n == 0 || grow) m = mt;
            if (__any_sync(0xffffffffu, grow)) {
                // rescale O (the previous tile's PV has finished: see the phase notes); every lane
                // of the warp takes part, factor 1 where the max stayed
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
            // pass 2: P = 2^(s - m) in bf16 pairs over the first 64 columns of the scores (the P
            // of chunk c lands on columns already read)
            float sum = 0.f;
#pragma unroll 1
            for (int c = 0; c < kKV / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(t_s + 32 * c, r);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int j = j0 + 32 * c + 2 * k;
                    const float a = j <= qpos ? ex2_approx(__uint_as_float(r[2 * k]) * p.scale_log2 - m) : 0.f;
                    const float b = j + 1 <= qpos ? ex2_approx(__uint_as_float(r[2 * k + 1]) * p.scale_log2 - m) : 0.f;
                    sum += a + b;
                    pk[k] = pack_bf16x2(a, b);
                }
                tmem_st16(t_s + 16 * c, pk);
            }
            l = l * f + sum;
            tmem_wait_st();
            PF_TRACE(tr, n, 1);
            tc_fence_before();
            mbar_arrive(bar(kBarPReady, t));
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
