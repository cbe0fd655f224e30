// head_gemm.cuh -- per-head GEMMs of the decode step on tcgen05 tensor cores:
//
//   absorb   (page 1 section 4, path B):  q_abs[b,h,c] = sum_d q_c[b,h,d] * W_UK[h,d,c]
//   out-proj (value side of absorption):  out[b,h,d]   = sum_c o_lat[b,h,c] * W_UV[h,d,c]
//
//   decompression (page 1 section 4, path A): k[h,s,d] = sum_c c_KV[s,c] * W_UK[h,d,c] and
//            v[h,s,d] = sum_c c_KV[s,c] * W_UV[h,d,c], the out-proj shape with one activation
//            row per token shared by all heads, written head-major.
//
// One CTA computes a 128 (batch rows) x N_TILE tile of one head.  The batch rows are the MMA's
// M dimension, so small batches leave rows empty (TMA fills rows past the batch with zeros,
// which costs no HBM traffic) and the kernel is a stream over the head's weight slice: both
// GEMMs read 16 MiB of weights per step whatever the batch.
//
// Roles: warp 0 issues TMA loads into a ring of K-chunk stages (64 K elements = one 128-byte
// swizzle row per operand row), warp 1 allocates TMEM and one lane issues the MMAs, warps 2-5
// read the fp32 accumulator out of TMEM and store bf16 rows.
//
// Operand layouts in shared memory (128-byte swizzle, 8-row atoms of 1024 bytes):
//   A (activations)   [128 rows x 64 K] K-major, one TMA box.
//   W, absorb         W_UK[h] rows are K (d) and columns N (c): MN-major B.  N_TILE/64 boxes
//                     of [64 K rows x 64 N] 8 KB each; LBO = 8 KB (next 64 N), SBO = 1 KB.
//   W, out-proj       W_UV[h] rows are N (d) and columns K (c): K-major B, one box of
//                     [N_TILE rows x 64 K]; SBO = 1 KB.
#pragma once
#include "ptx.cuh"

namespace mla {
namespace gemm {

template <int K_TOTAL, int N_TILE, bool W_MN_MAJOR, int STAGES>
struct Cfg {
    static constexpr int kKC = 64;
    static constexpr int kNK = K_TOTAL / kKC;
    static constexpr int kABytes = 128 * kKC * 2;
    static constexpr int kWBytes = N_TILE * kKC * 2;
    static constexpr int kStageBytes = kABytes + kWBytes;
    static constexpr int kData = STAGES * kStageBytes;
    static constexpr int kBarOff = kData;
    static constexpr int kSmemBytes = kData + 256;
    static constexpr uint32_t kTmemCols = N_TILE < 32 ? 32 : N_TILE;
    static_assert(K_TOTAL % kKC == 0, "K must be a multiple of 64");
    static_assert(N_TILE % 64 == 0 && N_TILE <= 256, "N tile must be 64..256 in steps of 64");
    static_assert((N_TILE & (N_TILE - 1)) == 0, "N tile must be a power of two (TMEM allocation)");
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
};

struct Args {
    __nv_bfloat16* out;
    int a_x_per_head;        // K_TOTAL when each head has its own activation row, 0 when shared
    int batch;
    int64_t out_row_stride;  // elements between consecutive batch rows of `out`
    int64_t out_head_stride; // elements between the outputs of consecutive heads
    int n_total;             // N of one head (512 absorb, 128 out-proj)
    uint32_t* dev_error;
    uint64_t timeout_ns;
};

template <int K_TOTAL, int N_TILE, bool W_MN_MAJOR, int STAGES>
__global__ void __launch_bounds__(192, 1)
head_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w, const Args args)
{
    using C = Cfg<K_TOTAL, N_TILE, W_MN_MAJOR, STAGES>;
    using namespace dev;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int n0 = blockIdx.x * N_TILE, h = blockIdx.y, m0 = blockIdx.z * 128;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + C::kBarOff;          // STAGES barriers
    const uint32_t bar_empty = bar_full + 8 * STAGES;      // STAGES barriers
    const uint32_t bar_done = bar_empty + 8 * STAGES;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kBarOff + 8 * (2 * STAGES + 1));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    if (sbase & 1023u) {  // uniform over the CTA: nothing has been started yet
        if (threadIdx.x == 0) raise_error(args.dev_error, MLA_DEVERR_SMEM_ALIGN);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtx w{args.timeout_ns, abort_flag, args.dev_error};

    griddep_launch_dependents();  // the next kernel of the step may be scheduled
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_a);
            tma_prefetch_desc(&tm_w);
            const uint64_t pol_w = l2_policy_evict_first();  // weights: read once per step
            const uint64_t pol_a = l2_policy_evict_last();   // activations: re-read by other N tiles
            const auto load_w = [&](int kc, int s) {
                const uint32_t w_dst = sbase + s * C::kStageBytes + C::kABytes;
                if (W_MN_MAJOR) {
#pragma unroll
                    for (int i = 0; i < N_TILE / 64; ++i)
                        tma_load_2d(w_dst + i * 8192, &tm_w, bar_full + 8 * s, n0 + 64 * i, h * K_TOTAL + kc * C::kKC,
                                    pol_w);
                } else {
                    tma_load_2d(w_dst, &tm_w, bar_full + 8 * s, kc * C::kKC, h * args.n_total + n0, pol_w);
                }
            };
            // The weights do not depend on the kernel before this one: the first stages' weights
            // are in flight before the wait for its output (the activations).
            const int early = C::kNK < STAGES ? C::kNK : STAGES;
            for (int kc = 0; kc < early; ++kc) {
                mbar_arrive_expect_tx(bar_full + 8 * kc, C::kStageBytes);
                load_w(kc, kc);
            }
            griddep_wait();
            int issued = 0;
            for (int kc = 0; kc < C::kNK; ++kc) {
                const int s = kc % STAGES;
                if (kc >= early) {
                    if (!wait_phase(bar_empty + 8 * s, kc / STAGES - 1, w)) break;
                    mbar_arrive_expect_tx(bar_full + 8 * s, C::kStageBytes);
                    load_w(kc, s);
                }
                tma_load_2d(sbase + s * C::kStageBytes, &tm_a, bar_full + 8 * s, h * args.a_x_per_head + kc * C::kKC,
                            m0, pol_a);
                ++issued;
            }
            if (*abort_flag) {  // let loads already in flight land before the CTA can exit
                for (int kc = (issued > STAGES ? issued - STAGES : 0); kc < issued; ++kc)
                    drain_phase(bar_full + 8 * (kc % STAGES), kc / STAGES, w.timeout_ns);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, N_TILE, false, W_MN_MAJOR);
            for (int kc = 0; kc < C::kNK; ++kc) {
                const int s = kc % STAGES;
                if (!wait_phase(bar_full + 8 * s, kc / STAGES, w)) break;
                tc_fence_after();
                const uint32_t a_base = sbase + s * C::kStageBytes, w_base = a_base + C::kABytes;
#pragma unroll
                for (int k = 0; k < C::kKC / 16; ++k) {
                    const uint64_t a_desc = smem_desc(a_base + k * 32, 16, 1024);
                    const uint64_t b_desc = W_MN_MAJOR ? smem_desc(w_base + k * 2048, 8192, 1024)
                                                       : smem_desc(w_base + k * 32, 16, 1024);
                    mma_ss(tmem, a_desc, b_desc, idesc, (kc | k) != 0 ? 1u : 0u);
                }
                mma_commit(bar_empty + 8 * s);
            }
            mma_commit(bar_done);  // also covers an early exit: arrives when issued MMAs finish
        }
    } else {
        // epilogue: warp (2..5) & 3 selects the TMEM lane quarter it may read
        const int q = warp & 3, row = 32 * q + lane, m = m0 + row;
        if (__all_sync(0xffffffffu, wait_phase(bar_done, 0, w) && !*abort_flag)) {
            tc_fence_after();
            __nv_bfloat16* dst = args.out + (int64_t)m * args.out_row_stride + (int64_t)h * args.out_head_stride + n0;
#pragma unroll 1
            for (int j = 0; j < N_TILE / 32; ++j) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 32 * j, r);
                tmem_wait_ld();
                if (m < args.batch) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * j);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 o;
                        o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                        o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                        o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                        o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                        d4[v] = o;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // all MMAs this CTA issued have finished before their TMEM goes away
        if (lane == 0) drain_phase(bar_done, 0, w.timeout_ns);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace gemm
}  // namespace mla
