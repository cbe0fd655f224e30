// prefill.cuh -- causal attention of a chunk of new tokens over their sequence in the
// decompressed form (page 1 section 4, path A: per-head keys k_h = W_UK[h] c and values
// v_h = W_UV[h] c; section 6: chunks of at least the prefill threshold of 256 new tokens take
// this form, shorter ones the absorbed decode).
//
// The chunk's T new tokens are positions S - T .. S - 1 of a sequence of S tokens whose cache
// rows are already written; query i (position S - T + i) attends to keys 0 .. S - T + i:
//   s_ij = (q_c[i,h] . k[j,h] + q_R[i,h] . k_R[j]) * softmax_scale,
//   out[i,h] = sum_j softmax_j(s_ij) v[j,h].
// The keys and values were decompressed before this kernel into k [S][128][128] and
// v [S][128][128]; k_R comes from the gathered cache rows [S][576] (columns 512..575).
//
// One CTA = 128 queries of one head (the MMA's M).  Warp 0 streams key/value tiles of 64 keys
// (two stages), warp 1 issues the MMAs, warps 2-5 run the online softmax, one query row per
// thread (its TMEM lane).  TMEM: two 64-column score buffers and the 128-column output.
//   QK:  S[128 x 64]  = Q [128 x 192] (q_c | q_R, three 64-column K-major chunks)
//                       x K tile [64 x 192] (k | k_R, three K-major chunks)
//   PV:  O[128 x 128] += P [128 x 64] (bf16, K-major, written by the softmax warps)
//                       x V tile [64 keys x 128] (MN-major: keys are K, dims are N)
// The running max moves only when a tile's max exceeds it by more than 8 (log2 units); the
// output is then rescaled in TMEM before the tile's PV.  Every wait is bounded.
#pragma once
#include "ptx.cuh"

namespace mla {
namespace prefill {

constexpr int kQ = 128;        // queries per CTA
constexpr int kKV = 64;        // keys per tile
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 softmax
constexpr int kQChunk = kQ * 64 * 2;                       // [128 rows][64] bf16, 16 KB
constexpr int kKVBox = kKV * 64 * 2;                       // [64 rows][64] bf16, 8 KB
constexpr int kStageBytes = 5 * kKVBox;                    // k 0-63, k 64-127, k_R, v 0-63, v 64-127
constexpr int kStages = 2;
constexpr int kPBytes = kQ * kKV * 2;                      // [128 queries][64 keys] bf16
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + 3 * kQChunk;                // 48 KB
constexpr int kOffP = kOffKV + kStages * kStageBytes;      // 128 KB
constexpr int kOffBar = kOffP + 2 * kPBytes;               // 160 KB
constexpr int kSmemBytes = kOffBar + 256;
constexpr uint32_t kTmemCols = 256;                        // S0 0-63, S1 64-127, O 128-255
constexpr float kRescaleLog2 = 8.f;

struct Params {
    int seq_len;          // S
    int chunk_len;        // T
    float scale_log2;     // softmax_scale * log2(e)
    __nv_bfloat16* out;   // [T][128][128]
    uint32_t* dev_error;
    uint64_t timeout_ns;
};

// barrier offsets (8 bytes each) from kOffBar
enum : int {
    kBarQ = 0,
    kBarKvFull = 1,    // 2
    kBarKvEmpty = 3,   // 2
    kBarSFull = 5,     // 2
    kBarPReady = 7,    // 2
    kBarPvDone = 9,    // 2
    kBarDone = 11,
    kBarCount = 12,
};

__global__ void __launch_bounds__(kThreads, 1)
prefill_attn_kernel(const __grid_constant__ CUtensorMap tm_qc, const __grid_constant__ CUtensorMap tm_qr,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_kr,
                    const __grid_constant__ CUtensorMap tm_v, const Params p)
{
    using namespace dev;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = blockIdx.x * kQ, h = blockIdx.y;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kOffBar;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kBarCount);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const auto bar = [&](int id, int k) { return bars + 8 * (id + k); };

    if (sbase & 1023u) {
        if (threadIdx.x == 0) raise_error(p.dev_error, MLA_DEVERR_SMEM_ALIGN);
        return;
    }
    // keys this query tile needs: up to the position of its last valid query
    const int first_pos = p.seq_len - p.chunk_len;
    const int last_q = min(i0 + kQ, p.chunk_len) - 1;
    const int n_tiles = (first_pos + last_q) / kKV + 1;

    if (threadIdx.x == 0) {
        mbar_init(bar(kBarQ, 0), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(kBarKvFull, s), 1);
            mbar_init(bar(kBarKvEmpty, s), 1);
            mbar_init(bar(kBarSFull, s), 1);
            mbar_init(bar(kBarPReady, s), 128);
            mbar_init(bar(kBarPvDone, s), 1);
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

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();  // every query tile of the head re-reads them
            mbar_arrive_expect_tx(bar(kBarQ, 0), 3 * kQChunk);
            tma_load_3d(sbase + kOffQ, &tm_qc, bar(kBarQ, 0), 0, h, i0, pol);
            tma_load_3d(sbase + kOffQ + kQChunk, &tm_qc, bar(kBarQ, 0), 64, h, i0, pol);
            tma_load_3d(sbase + kOffQ + 2 * kQChunk, &tm_qr, bar(kBarQ, 0), 0, h, i0, pol);
            int issued = 0;
            for (int n = 0; n < n_tiles; ++n) {
                const int s = n & 1;
                if (n >= 2 && !wait_phase(bar(kBarKvEmpty, s), ((n - 2) >> 1) & 1, w)) break;
                const uint32_t st = sbase + kOffKV + s * kStageBytes, full = bar(kBarKvFull, s);
                const int j0 = n * kKV;
                mbar_arrive_expect_tx(full, kStageBytes);
                tma_load_3d(st, &tm_k, full, 0, h, j0, pol);
                tma_load_3d(st + kKVBox, &tm_k, full, 64, h, j0, pol);
                tma_load_2d(st + 2 * kKVBox, &tm_kr, full, 512, j0, pol);
                tma_load_3d(st + 3 * kKVBox, &tm_v, full, 0, h, j0, pol);
                tma_load_3d(st + 4 * kKVBox, &tm_v, full, 64, h, j0, pol);
                ++issued;
            }
            // loads in flight land before the CTA can exit
            drain_phase(bar(kBarQ, 0), 0, w.timeout_ns);
            for (int n = (issued > 2 ? issued - 2 : 0); n < issued; ++n)
                drain_phase(bar(kBarKvFull, n & 1), (n >> 1) & 1, w.timeout_ns);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, kKV, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, 128, false, true);
            const auto issue_qk = [&](int n) -> bool {
                const int s = n & 1;
                if (!wait_phase(bar(kBarKvFull, s), (n >> 1) & 1, w)) return false;
                tc_fence_after();
                const uint32_t st = sbase + kOffKV + s * kStageBytes;
#pragma unroll 1
                for (int c = 0; c < 3; ++c) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t a = smem_desc(sbase + kOffQ + c * kQChunk + 32 * k, 16, 1024);
                        const uint64_t b = smem_desc(st + c * kKVBox + 32 * k, 16, 1024);
                        mma_ss(tmem + s * kKV, a, b, idesc_qk, (c | k) != 0 ? 1u : 0u);
                    }
                }
                mma_commit(bar(kBarSFull, s));
                return true;
            };
            bool ok = wait_phase(bar(kBarQ, 0), 0, w) && (tc_fence_after(), issue_qk(0));
            for (int n = 0; ok && n < n_tiles; ++n) {
                if (n + 1 < n_tiles && !issue_qk(n + 1)) break;
                const int s = n & 1;
                if (!wait_phase(bar(kBarPReady, s), (n >> 1) & 1, w)) break;
                tc_fence_after();
                const uint32_t pt = sbase + kOffP + s * kPBytes, st = sbase + kOffKV + s * kStageBytes;
#pragma unroll
                for (int k = 0; k < kKV / 16; ++k) {
                    const uint64_t a = smem_desc(pt + 32 * k, 16, 1024);
                    const uint64_t b = smem_desc(st + 3 * kKVBox + 2048 * k, 8192, 1024);
                    mma_ss(tmem + 128, a, b, idesc_pv, (n | k) != 0 ? 1u : 0u);
                }
                mma_commit(bar(kBarPvDone, s));
                mma_commit(bar(kBarKvEmpty, s));
            }
            mma_commit(bar(kBarDone, 0));  // arrives when every MMA issued here has finished
        }
    } else {
        // softmax: warp (2..5) & 3 selects the TMEM lane quarter, one query row per thread
        const int q4 = warp & 3, row = 32 * q4 + lane, i = i0 + row;
        const int qpos = min(first_pos + i, p.seq_len - 1);
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int n = 0; n < n_tiles; ++n) {
            const int s = n & 1;
            if (!(ok = wait_warp(bar(kBarSFull, s), (n >> 1) & 1, w))) break;
            tc_fence_after();
            uint32_t r[2][32];
            tmem_ld32(tmem + lane_base + s * kKV, r[0]);
            tmem_ld32(tmem + lane_base + s * kKV + 32, r[1]);
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
            const bool first = n == 0;
            const bool grow = !first && mt > m + kRescaleLog2;
            if (__any_sync(0xffffffffu, grow)) {
                // rescale O (every lane of the warp takes part in the TMEM access; factor 1 where
                // the row's max did not move) once the previous tile's PV has finished
                if (!(ok = wait_warp(bar(kBarPvDone, (n - 1) & 1), ((n - 1) >> 1) & 1, w))) break;
                tc_fence_after();
                const float f = grow ? ex2_approx(m - mt) : 1.f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_base + 128 + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
                    tmem_st32(tmem + lane_base + 128 + 32 * c, o);
                }
                tmem_wait_st();
                if (grow) {
                    l *= f;
                    m = mt;
                }
            }
            if (first) m = mt;
            // P = 2^(s - m) into this tile's P buffer, once the PV two tiles back has read it
            if (n >= 2 && !(ok = wait_warp(bar(kBarPvDone, s), ((n - 2) >> 1) & 1, w))) break;
            uint8_t* prow = smem + kOffP + s * kPBytes + row * 128;
            float sum = 0.f;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                uint32_t pk[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a = ex2_approx(x[8 * c8 + 2 * k] - m), b = ex2_approx(x[8 * c8 + 2 * k + 1] - m);
                    sum += a + b;
                    pk[k] = pack_bf16x2(a, b);
                }
                *reinterpret_cast<uint4*>(prow + ((c8 ^ (row & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            l += sum;
            fence_proxy_async_cta();  // the P tile is read by the tensor core (async proxy)
            tc_fence_before();
            mbar_arrive(bar(kBarPReady, s));
        }
        if (ok && wait_warp(bar(kBarPvDone, (n_tiles - 1) & 1), ((n_tiles - 1) >> 1) & 1, w)) {
            tc_fence_after();
            const float inv = 1.f / l;
            __nv_bfloat16* dst = p.out + ((int64_t)i * 128 + h) * 128;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + 128 + 32 * c, o);
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
