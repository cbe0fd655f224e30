// combine.cuh -- the KV-split reduction ("stage 2" on the Kimi K3 decode time-share page,
// "Inside the blocks"): merge the partial results of a sequence's work items.
//
// Partial j of head h carries a normalised latent output o_j (512 fp32) and lse_j (natural
// log).  The merge is the log-sum-exp identity:
//   lse = log sum_j exp(lse_j),   o_lat = sum_j exp(lse_j - lse) * o_j.
// One warp per (sequence, head): lane j holds partial j's log-sum-exp and merge weight (32
// partials per pass), the lanes split the 512 dims 16 each, and the partial rows are read as
// 2 KB of coalesced float4 loads.  Latency, not bandwidth, sets the time of this small kernel,
// so the work list entry is read before the wait for the decode kernel, and after it the
// log-sum-exps and the first eight partial rows are all requested at once (one round trip for
// up to eight partials).  Bytes: n_parts * 2 KB per (sequence, head), from L2 in the step.
#pragma once
#include "plan.h"
#include "ptx.cuh"

namespace mla {
namespace combine {

constexpr int kHeadsPerCta = 4;

constexpr int kRowsInFlight = 8;  // partial rows requested together

__global__ void __launch_bounds__(32 * kHeadsPerCta)
combine_kernel(const int32_t* __restrict__ plan, const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
               __nv_bfloat16* __restrict__ o_lat, float* __restrict__ lse)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    dev::griddep_launch_dependents();  // the projection may start streaming its weights
    // the plan was copied before the step's first kernel: it may be read before the wait
    const int32_t* entry = plan + __ldg(plan + kHdrCombineOff) + kCombineWords * blockIdx.x;
    const int seq = __ldg(entry), first = __ldg(entry + 1), n = __ldg(entry + 2);
    const int h = blockIdx.y * kHeadsPerCta + warp;
    const float4* rows = reinterpret_cast<const float4*>(ws_o + ((int64_t)first * 128 + h) * 512) + lane;
    constexpr int64_t kPartStride = 128 * 512 / 4;  // float4s between partial j and j + 1
    dev::griddep_wait();  // the partials come from the decode kernel

    // the first pass's log-sum-exps and rows, all in flight together
    float lse_j = lane < n ? ws_lse[(int64_t)(first + lane) * 128 + h] : -INFINITY;
    float4 x[kRowsInFlight][4];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v)
            x[u][v] = u < n ? rows[u * kPartStride + 32 * v] : make_float4(0.f, 0.f, 0.f, 0.f);

    // L = log sum_j exp(lse_j) over all n partials (lanes beyond 32 loop)
    float mx = lse_j;
    for (int j = lane + 32; j < n; j += 32) mx = fmaxf(mx, ws_lse[(int64_t)(first + j) * 128 + h]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = lane < n ? expf(lse_j - mx) : 0.f;
    for (int j = lane + 32; j < n; j += 32) sum += expf(ws_lse[(int64_t)(first + j) * 128 + h] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float L = mx + logf(sum);

    float4 acc[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    float wj = lane < n ? expf(lse_j - L) : 0.f;  // weights of partials 0..31
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
        const float wgt = __shfl_sync(0xffffffffu, wj, u);  // 0 past n
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            acc[v].x += wgt * x[u][v].x;
            acc[v].y += wgt * x[u][v].y;
            acc[v].z += wgt * x[u][v].z;
            acc[v].w += wgt * x[u][v].w;
        }
    }
    // partials past the first eight, eight at a time
    for (int j0 = kRowsInFlight; j0 < n; j0 += kRowsInFlight) {
        if ((j0 & 31) == 0)
            wj = j0 + lane < n ? expf(ws_lse[(int64_t)(first + j0 + lane) * 128 + h] - L) : 0.f;
#pragma unroll
        for (int u = 0; u < kRowsInFlight; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v)
                x[u][v] = j0 + u < n ? rows[(j0 + u) * kPartStride + 32 * v] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kRowsInFlight; ++u) {
            const float wgt = __shfl_sync(0xffffffffu, wj, (j0 + u) & 31);
            if (j0 + u < n) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    acc[v].x += wgt * x[u][v].x;
                    acc[v].y += wgt * x[u][v].y;
                    acc[v].z += wgt * x[u][v].z;
                    acc[v].w += wgt * x[u][v].w;
                }
            }
        }
    }
    uint2* dst = reinterpret_cast<uint2*>(o_lat + ((int64_t)seq * 128 + h) * 512) + lane;
#pragma unroll
    for (int v = 0; v < 4; ++v)
        dst[32 * v] = make_uint2(dev::pack_bf16x2(acc[v].x, acc[v].y), dev::pack_bf16x2(acc[v].z, acc[v].w));
    if (lane == 0) lse[(int64_t)seq * 128 + h] = L;
}

}  // namespace combine
}  // namespace mla
