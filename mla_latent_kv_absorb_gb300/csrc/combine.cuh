// combine.cuh -- the KV-split reduction ("stage 2" on the Kimi K3 decode time-share page,
// "Inside the blocks"): merge the partial results of a sequence's work items.
//
// Partial j of head h carries a normalised latent output o_j (512 fp32) and lse_j (natural
// log).  The merge is the log-sum-exp identity:
//   lse = log sum_j exp(lse_j),   o_lat = sum_j exp(lse_j - lse) * o_j.
// One warp per (sequence, head): lane j holds partial j's log-sum-exp and merge weight (32
// partials per pass), the lanes split the 512 dims 16 each, and the partial rows are read as
// 2 KB of coalesced float4 loads, four partials at a time so the loads overlap.  HBM/L2 bound:
// n_parts * 2 KB per (sequence, head).
#pragma once
#include "plan.h"
#include "ptx.cuh"

namespace mla {
namespace combine {

constexpr int kHeadsPerCta = 4;

__global__ void __launch_bounds__(32 * kHeadsPerCta)
combine_kernel(const int32_t* __restrict__ plan, const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
               __nv_bfloat16* __restrict__ o_lat, float* __restrict__ lse)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    dev::griddep_launch_dependents();  // the projection may start streaming its weights
    dev::griddep_wait();               // the partials come from the decode kernel
    const int32_t* entry = plan + plan[kHdrCombineOff] + kCombineWords * blockIdx.x;
    const int seq = entry[0], first = entry[1], n = entry[2];
    const int h = blockIdx.y * kHeadsPerCta + warp;

    float mx = -INFINITY;
    for (int j = lane; j < n; j += 32) mx = fmaxf(mx, ws_lse[(int64_t)(first + j) * 128 + h]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int j = lane; j < n; j += 32) sum += expf(ws_lse[(int64_t)(first + j) * 128 + h] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float L = mx + logf(sum);

    float4 acc[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* rows = reinterpret_cast<const float4*>(ws_o + ((int64_t)first * 128 + h) * 512) + lane;
    constexpr int64_t kPartStride = 128 * 512 / 4;  // float4s between partial j and j + 1
    for (int j0 = 0; j0 < n; j0 += 32) {
        const int cnt = min(32, n - j0);
        const float wj = lane < cnt ? expf(ws_lse[(int64_t)(first + j0 + lane) * 128 + h] - L) : 0.f;
        int j = 0;
        for (; j + 4 <= cnt; j += 4) {
            float4 x[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) x[u][v] = rows[(j0 + j + u) * kPartStride + 32 * v];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float wgt = __shfl_sync(0xffffffffu, wj, j + u);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    acc[v].x += wgt * x[u][v].x;
                    acc[v].y += wgt * x[u][v].y;
                    acc[v].z += wgt * x[u][v].z;
                    acc[v].w += wgt * x[u][v].w;
                }
            }
        }
        for (; j < cnt; ++j) {
            const float wgt = __shfl_sync(0xffffffffu, wj, j);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float4 x = rows[(j0 + j) * kPartStride + 32 * v];
                acc[v].x += wgt * x.x;
                acc[v].y += wgt * x.y;
                acc[v].z += wgt * x.z;
                acc[v].w += wgt * x.w;
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
