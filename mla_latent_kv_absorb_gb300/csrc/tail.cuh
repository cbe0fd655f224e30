// tail.cuh -- the end of the decode step in one kernel: the KV-split reduction ("stage 2" on the
// Kimi K3 decode time-share page, "Inside the blocks") fused with the W_UV projection (the value
// side of absorption, page 1 section 1).  For head h and every sequence b of a 128-row tile:
//
//   o_lat[b,h,:] = sum_j exp(lse_j - lse) o_j      lse = log sum_j exp(lse_j)     (split sequences)
//   o_lat[b,h,:] = as the decode kernel wrote it                                  (single-item ones)
//   out[b,h,d]   = sum_c o_lat[b,h,c] W_UV[h,d,c]
//
// One CTA per (head, 128-row tile).  W_UV[h] (128 KB, K-major) streams through a ring of six
// 16 KB K-chunks, the first six issued before the wait for the decode kernel's output
// (programmatic dependent launch); all sixteen warps then merge the rows of the tile (one row
// each per pass, the first four partial rows in flight while the log-sum-exp is formed) straight
// into the bf16 A operand in shared memory (128-byte swizzle, the layout a TMA box would give) and
// write the merged o_lat and lse; warp 1 issues the 32 MMAs (M = 128 rows, N = 128, K = 512) once
// the rows are in, warp 0 refills the W ring, and warps 2-5 read the fp32 result out of TMEM and
// store bf16 rows.  The merge arithmetic per
// element is that of the separate merge kernel (same order, same functions), so the fused
// result equals the unfused one bit for bit.
#pragma once
#include "plan.h"
#include "ptx.cuh"

namespace mla {
namespace tail {

constexpr int kThreads = 512;            // all 16 warps merge; then warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kMergeWarps = kThreads / 32;
constexpr int kKC = 64;                  // K elements per chunk: one 128-byte swizzle row
constexpr int kNK = 512 / kKC;
constexpr int kChunkBytes = 128 * kKC * 2;  // 16 KB: 128 rows x 64 K, for A and for W
constexpr int kWStages = 6;              // W_UV K-chunks in flight: six of eight load before the merge
constexpr int kOffA = 0;
constexpr int kOffW = kNK * kChunkBytes;
constexpr int kOffBars = kOffW + kWStages * kChunkBytes;
enum Bar : int { kFull0 = 0, kEmpty0 = kWStages, kAReady = 2 * kWStages, kDone, kNumBars };
constexpr int kOffComb = kOffBars + 8 * kNumBars;  // int2[128]: (first partial, parts) per tile row
constexpr int kOffTmemHolder = kOffComb + 128 * 8;
constexpr int kOffAbort = kOffTmemHolder + 4;
constexpr int kSmemBytes = kOffAbort + 12;
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kMergeBarrier = 1;  // named barrier of the merge warps
static_assert(kOffW % 1024 == 0 && kChunkBytes % 1024 == 0, "MMA operands are 1024-byte aligned");
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Args {
    const int32_t* plan;
    const float* ws_o;     // [partials][128][512]
    const float* ws_lse;   // [partials][128]
    __nv_bfloat16* o_lat;  // [B][128][512]: read for single-item sequences, written for merged ones
    float* lse;            // [B][128]: written for merged sequences
    __nv_bfloat16* out;    // [B][128][128]
    int batch;
    uint32_t* dev_error;
    uint64_t timeout_ns;
};

// Lane `lane` owns dims 16 lane .. 16 lane + 15 of a row: K-chunk lane / 4, 16-byte units
// 2 (lane % 4) and 2 (lane % 4) + 1 of that chunk's 128-byte row, stored swizzled.
__device__ __forceinline__ void put_a_row(uint8_t* smem, int r, int lane, uint4 lo, uint4 hi)
{
    uint8_t* row = smem + kOffA + (lane >> 2) * kChunkBytes + (r >> 3) * 1024 + (r & 7) * 128;
    const int u = 2 * (lane & 3);
    *reinterpret_cast<uint4*>(row + ((u ^ (r & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(row + (((u + 1) ^ (r & 7)) << 4)) = hi;
}

// Merge the n partials of (sequence b, head h) starting at partial `first` into this lane's 16
// dims; returns lse.  Same arithmetic as the separate merge kernel, element by element (the same
// max and sum trees, the same weights, each element summed in partial order); only the order of
// the loads differs: the first four partial rows are requested before the log-sum-exp.
__device__ __forceinline__ float merge_row(const Args& a, int first, int n, int h, int lane, float (&acc)[16])
{
    const float4* rows = reinterpret_cast<const float4*>(a.ws_o + ((int64_t)first * 128 + h) * 512) + 4 * lane;
    constexpr int64_t kPartStride = 128 * 512 / 4;  // float4s between partial j and j + 1
    const int n0 = min(4, n);
    float4 x[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v)
            x[u][v] = u < n0 ? rows[u * kPartStride + v] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float l0 = lane < n ? a.ws_lse[(int64_t)(first + lane) * 128 + h] : -INFINITY;
    float mx = l0;
    for (int j = lane + 32; j < n; j += 32) mx = fmaxf(mx, a.ws_lse[(int64_t)(first + j) * 128 + h]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = lane < n ? expf(l0 - mx) : 0.f;
    for (int j = lane + 32; j < n; j += 32) sum += expf(a.ws_lse[(int64_t)(first + j) * 128 + h] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float L = mx + logf(sum);
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    for (int j0 = 0; j0 < n; j0 += 32) {
        const int cnt = min(32, n - j0);
        const float wj = lane < cnt ? expf((j0 == 0 ? l0 : a.ws_lse[(int64_t)(first + j0 + lane) * 128 + h]) - L) : 0.f;
        int j = 0;
        for (; j + 4 <= cnt; j += 4) {
            if (j0 + j != 0) {  // the first four rows are already in x
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v) x[u][v] = rows[(j0 + j + u) * kPartStride + v];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float wgt = __shfl_sync(0xffffffffu, wj, j + u);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    acc[4 * v + 0] += wgt * x[u][v].x;
                    acc[4 * v + 1] += wgt * x[u][v].y;
                    acc[4 * v + 2] += wgt * x[u][v].z;
                    acc[4 * v + 3] += wgt * x[u][v].w;
                }
            }
        }
        for (; j < cnt; ++j) {
            const float wgt = __shfl_sync(0xffffffffu, wj, j);
            if (j0 + j < n0) {  // still in x (n < 4)
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float4 y = j == 0 ? x[0][v] : (j == 1 ? x[1][v] : x[2][v]);
                    acc[4 * v + 0] += wgt * y.x;
                    acc[4 * v + 1] += wgt * y.y;
                    acc[4 * v + 2] += wgt * y.z;
                    acc[4 * v + 3] += wgt * y.w;
                }
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float4 y = rows[(j0 + j) * kPartStride + v];
                    acc[4 * v + 0] += wgt * y.x;
                    acc[4 * v + 1] += wgt * y.y;
                    acc[4 * v + 2] += wgt * y.z;
                    acc[4 * v + 3] += wgt * y.w;
                }
            }
        }
    }
    return L;
}

// 16 warps at 128 registers fill the SM's register file (one CTA per SM: shared memory).
__global__ void __maxnreg__(128)
merge_out_proj_kernel(const __grid_constant__ CUtensorMap tm_w, const Args args)
{
    using namespace dev;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int h = blockIdx.x, m0 = blockIdx.y * 128;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kOffBars;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffTmemHolder);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);

    if (sbase & 1023u) {  // uniform over the CTA: nothing has been started yet
        if (threadIdx.x == 0) raise_error(args.dev_error, MLA_DEVERR_SMEM_ALIGN);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(bars + 8 * (kFull0 + s), 1);
            mbar_init(bars + 8 * (kEmpty0 + s), 1);
        }
        mbar_init(bars + 8 * kAReady, kMergeWarps);
        mbar_init(bars + 8 * kDone, 1);
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
    const WaitCtx w{args.timeout_ns, abort_flag, args.dev_error};

    griddep_launch_dependents();
    const uint64_t pol = l2_policy_evict_first();  // W_UV is read once per step
    if (warp == 0 && lane == 0) {
        // W_UV does not depend on the kernel before this one: the first stages stream in at once
        tma_prefetch_desc(&tm_w);
        for (int kc = 0; kc < kWStages; ++kc) {
            mbar_arrive_expect_tx(bars + 8 * (kFull0 + kc), kChunkBytes);
            tma_load_2d(sbase + kOffW + kc * kChunkBytes, &tm_w, bars + 8 * (kFull0 + kc), kc * kKC, h * 128, pol);
        }
    }

    // ---- all warps: the A operand (bf16 rows of o_lat for head h)
    int2* comb = reinterpret_cast<int2*>(smem + kOffComb);
    griddep_wait();  // partials, o_lat and the plan come from the decode kernel
    for (int r = threadIdx.x; r < 128; r += kThreads) comb[r] = make_int2(-1, 0);
    named_barrier_or(kMergeBarrier, kThreads, false);
    const int n_comb = args.plan[kHdrCombine];
    const int32_t* entries = args.plan + args.plan[kHdrCombineOff];
    for (int e = threadIdx.x; e < n_comb; e += kThreads) {
        const int4 c = *reinterpret_cast<const int4*>(entries + kCombineWords * e);
        if (c.x >= m0 && c.x < m0 + 128) comb[c.x - m0] = make_int2(c.y, c.z);
    }
    named_barrier_or(kMergeBarrier, kThreads, false);
    for (int r = warp; r < 128 && m0 + r < args.batch; r += kMergeWarps) {
        const int b = m0 + r;
        const int2 c = comb[r];
        uint4* ol = reinterpret_cast<uint4*>(args.o_lat + ((int64_t)b * 128 + h) * 512 + 16 * lane);
        if (c.x < 0) {  // a single item wrote this row already
            put_a_row(smem, r, lane, ol[0], ol[1]);
        } else {
            float acc[16];
            const float L = merge_row(args, c.x, c.y, h, lane, acc);
            const uint4 lo = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                        pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
            const uint4 hi = make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                                        pack_bf16x2(acc[12], acc[13]), pack_bf16x2(acc[14], acc[15]));
            put_a_row(smem, r, lane, lo, hi);
            ol[0] = lo;
            ol[1] = hi;
            if (lane == 0) args.lse[(int64_t)b * 128 + h] = L;
        }
    }
    fence_proxy_async_cta();  // the rows are read by the MMA (async proxy)
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * kAReady);

    if (warp == 0) {
        if (lane == 0) {  // the rest of W_UV as the MMAs free the stages
            int issued = kWStages;
            for (int kc = kWStages; kc < kNK; ++kc, ++issued) {
                const int s = kc % kWStages;
                if (!wait_phase(bars + 8 * (kEmpty0 + s), kc / kWStages - 1, w)) break;
                mbar_arrive_expect_tx(bars + 8 * (kFull0 + s), kChunkBytes);
                tma_load_2d(sbase + kOffW + s * kChunkBytes, &tm_w, bars + 8 * (kFull0 + s), kc * kKC, h * 128, pol);
            }
            if (*abort_flag) {  // loads in flight land before the CTA can exit
                for (int kc = issued - kWStages; kc < issued; ++kc)
                    drain_phase(bars + 8 * (kFull0 + kc % kWStages), kc / kWStages, w.timeout_ns);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
            if (wait_phase(bars + 8 * kAReady, 0, w)) {
                tc_fence_after();
                for (int kc = 0; kc < kNK; ++kc) {
                    const int s = kc % kWStages;
                    if (!wait_phase(bars + 8 * (kFull0 + s), kc / kWStages, w)) break;
                    tc_fence_after();
                    const uint32_t a_base = sbase + kOffA + kc * kChunkBytes, w_base = sbase + kOffW + s * kChunkBytes;
#pragma unroll
                    for (int k = 0; k < kKC / 16; ++k)
                        mma_ss(tmem, smem_desc(a_base + k * 32, 16, 1024), smem_desc(w_base + k * 32, 16, 1024), idesc,
                               (kc | k) != 0 ? 1u : 0u);
                    mma_commit(bars + 8 * (kEmpty0 + s));
                }
            }
            mma_commit(bars + 8 * kDone);  // also covers an early exit: arrives when issued MMAs finish
        }
    } else if (warp < 6) {
        // ---- epilogue, warps 2-5: warp & 3 selects the TMEM lane quarter it may read
        const int q = warp & 3, row = 32 * q + lane, m = m0 + row;
        if (__all_sync(0xffffffffu, wait_phase(bars + 8 * kDone, 0, w) && !*abort_flag)) {
            tc_fence_after();
            __nv_bfloat16* dst = args.out + ((int64_t)m * 128 + h) * 128;
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 32 * j, v);
                tmem_wait_ld();
                if (m < args.batch) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * j);
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        d4[t] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * t + 0]), __uint_as_float(v[8 * t + 1])),
                                           pack_bf16x2(__uint_as_float(v[8 * t + 2]), __uint_as_float(v[8 * t + 3])),
                                           pack_bf16x2(__uint_as_float(v[8 * t + 4]), __uint_as_float(v[8 * t + 5])),
                                           pack_bf16x2(__uint_as_float(v[8 * t + 6]), __uint_as_float(v[8 * t + 7])));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // every MMA this CTA issued has finished before its TMEM goes away
        if (lane == 0) drain_phase(bars + 8 * kDone, 0, w.timeout_ns);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace tail
}  // namespace mla
