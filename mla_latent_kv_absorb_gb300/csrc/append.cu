// append.cu -- mla_append_kv: write new tokens' rows into the paged latent cache (declared in
// include/mla.h).
//
// Each token stores its 512-d latent c_KV and its 64-d rotated RoPE key k_R once ("撕開
// DeepSeek MLA 源碼", section 1); pages hold 64 tokens (section 3).  For the FP8 cache the
// latent is quantised on the way in: one fp32 scale per token, sigma = max|c| / 448, and the
// e4m3 code nearest c / sigma.  For the NVFP4 cache (the page's "NVFP4 quantized gather" names
// the format; the two-level scaling below is this library's reading): sigma = max|c| / 2688 per
// token, one e4m3 scale per 16 latent values, S_b = nearest e4m3 to ((max|c| over the block) /
// sigma) / 6, and the e2m1 code nearest c / (sigma S_b).
//
// One warp per token.  A token is 1152 bytes of bf16 input and at most 1152 bytes of output,
// so the kernel is a few coalesced 16-byte loads and stores per lane; at decode batch sizes it
// is launch-bound and no staging in shared memory or TMA would pay.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "../../include/mla.h"
#include "nvtx_range.h"

namespace mla {
void set_last_error_text(const char* text);
}

namespace mla::append {

constexpr int kWarps = 8;  // tokens per CTA

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// e4m3 codes of (lo, hi): round to nearest, ties to even, magnitudes past 448 give 448 with
// their sign (the hardware conversion).  lo lands in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// e2m1 codes of (lo, hi): round to nearest, ties to even, magnitudes past 6 give 6 with their sign
// (the hardware conversion); lo lands in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// Value of an e4m3 code (exact: through f16).
__device__ __forceinline__ float e4m3_value(uint32_t code)
{
    uint32_t h2;
    const uint16_t c = (uint16_t)(code & 0xFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Slot of token i, or -1 when the token is skipped (negative slot, or out of the pool: then
// the error bit is set).
__device__ __forceinline__ int64_t token_slot(const int32_t* slots, int64_t i, int64_t num_slots, uint32_t* dev_error,
                                              int lane)
{
    const int32_t slot = __ldg(slots + i);
    if (slot < 0) return -1;
    if (slot >= num_slots) {
        if (lane == 0) atomicOr(dev_error, MLA_DEVERR_BAD_SLOT);
        return -1;
    }
    return slot;
}

// bf16 cache: row = c_KV (64 x 16 B) then k_R (8 x 16 B), 72 x 16 B per slot.
__global__ void __launch_bounds__(kWarps * 32) append_bf16_kernel(const uint4* __restrict__ c_kv,
                                                                   const uint4* __restrict__ k_r,
                                                                   const int32_t* __restrict__ slots, int n,
                                                                   int64_t num_slots, uint4* __restrict__ pool,
                                                                   uint32_t* dev_error)
{
    const int lane = threadIdx.x & 31;
    const int64_t i = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (i >= n) return;
    const int64_t slot = token_slot(slots, i, num_slots, dev_error, lane);
    if (slot < 0) return;
    const uint4* src = c_kv + i * 64;
    uint4* dst = pool + slot * 72;
    const uint4 a = __ldg(src + lane), b = __ldg(src + 32 + lane);
    dst[lane] = a;
    dst[32 + lane] = b;
    if (lane < 8) dst[64 + lane] = __ldg(k_r + i * 8 + lane);
}

// FP8 cache: lane l quantises latent elements [16 l, 16 l + 16) and stores their 16 codes.
__global__ void __launch_bounds__(kWarps * 32) append_fp8_kernel(const uint4* __restrict__ c_kv,
                                                                  const uint4* __restrict__ k_r,
                                                                  const int32_t* __restrict__ slots, int n,
                                                                  int64_t num_slots, uint4* __restrict__ c8,
                                                                  float* __restrict__ scale, uint4* __restrict__ kr,
                                                                  uint32_t* dev_error)
{
    const int lane = threadIdx.x & 31;
    const int64_t i = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (i >= n) return;
    const int64_t slot = token_slot(slots, i, num_slots, dev_error, lane);
    if (slot < 0) return;
    const uint4* src = c_kv + i * 64 + 2 * lane;
    const uint4 a = __ldg(src), b = __ldg(src + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float v[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        v[2 * k] = bf16_lo(w[k]);
        v[2 * k + 1] = bf16_hi(w[k]);
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sigma = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint32_t codes[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float q0 = __fdiv_rn(v[4 * k], sigma), q1 = __fdiv_rn(v[4 * k + 1], sigma);
        const float q2 = __fdiv_rn(v[4 * k + 2], sigma), q3 = __fdiv_rn(v[4 * k + 3], sigma);
        codes[k] = e4m3x2(q0, q1) | (e4m3x2(q2, q3) << 16);
    }
    c8[slot * 32 + lane] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
    if (lane < 8) kr[slot * 8 + lane] = __ldg(k_r + i * 8 + lane);
    if (lane == 0) scale[slot] = sigma;
}

// NVFP4 cache: 288-byte rows, the 512 latent codes (two per byte, value 2j in the low nibble of
// byte j) then 32 e4m3 block scales.  Lane l owns block l, latent values [16 l, 16 l + 16): its
// 8 code bytes and its scale byte.  All arithmetic in fp32 with IEEE division, in the order of the
// format's definition; a block whose scale rounds to zero stores zeros of its values' signs.
__global__ void __launch_bounds__(kWarps * 32) append_nvfp4_kernel(const uint4* __restrict__ c_kv,
                                                                    const uint4* __restrict__ k_r,
                                                                    const int32_t* __restrict__ slots, int n,
                                                                    int64_t num_slots, uint8_t* __restrict__ rows,
                                                                    float* __restrict__ scale, uint4* __restrict__ kr,
                                                                    uint32_t* dev_error)
{
    constexpr int kRowBytes = 512 / 2 + 512 / 16;
    const int lane = threadIdx.x & 31;
    const int64_t i = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (i >= n) return;
    const int64_t slot = token_slot(slots, i, num_slots, dev_error, lane);
    if (slot < 0) return;
    const uint4* src = c_kv + i * 64 + 2 * lane;
    const uint4 a = __ldg(src), b = __ldg(src + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float v[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        v[2 * k] = bf16_lo(w[k]);
        v[2 * k + 1] = bf16_hi(w[k]);
    }
    float bmax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) bmax = fmaxf(bmax, fabsf(v[k]));
    float amax = bmax;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sigma = amax > 0.f ? __fdiv_rn(amax, 2688.f) : 1.f;
    const uint32_t s8 = e4m3x2(__fdiv_rn(__fdiv_rn(bmax, sigma), 6.f), 0.f) & 0xFFu;
    const float den = __fmul_rn(sigma, e4m3_value(s8));
    uint32_t code[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t byte;
        if (den == 0.f)
            byte = (signbit(v[2 * k]) ? 0x8u : 0u) | (signbit(v[2 * k + 1]) ? 0x80u : 0u);
        else
            byte = e2m1x2(__fdiv_rn(v[2 * k], den), __fdiv_rn(v[2 * k + 1], den));
        code[k >> 2] |= byte << (8 * (k & 3));
    }
    uint8_t* row = rows + slot * kRowBytes;
    *reinterpret_cast<uint2*>(row + 8 * lane) = make_uint2(code[0], code[1]);
    row[256 + lane] = (uint8_t)s8;
    if (lane < 8) kr[slot * 8 + lane] = __ldg(k_r + i * 8 + lane);
    if (lane == 0) scale[slot] = sigma;
}

}  // namespace mla::append

namespace {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" MLA_API mla_status mla_append_kv(int32_t num_tokens, const void* c_kv, const void* k_r,
                                            const int32_t* slots, mla_kv_dtype kv_dtype, int32_t num_pool_pages,
                                            void* kv_pool, float* kv_scale, void* kr_pool, uint32_t* dev_error,
                                            void* stream)
{
    const mla::NvtxRange nvtx_range("mla_append_kv");
    using namespace mla::append;
    if (num_tokens < 0 || num_pool_pages <= 0) return MLA_ERR_INVALID_ARG;
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3 && kv_dtype != MLA_KV_NVFP4)
        return MLA_ERR_INVALID_ARG;
    if (num_tokens == 0) return MLA_OK;
    if (!c_kv || !k_r || !slots || !kv_pool || !dev_error) return MLA_ERR_INVALID_ARG;
    const bool fp8 = kv_dtype != MLA_KV_BF16;  // both quantised caches keep a scale and k_R apart
    if (fp8 && (!kv_scale || !kr_pool)) return MLA_ERR_INVALID_ARG;
    if (!aligned(c_kv, 16) || !aligned(k_r, 16) || !aligned(kv_pool, 16) || !aligned(slots, 4) ||
        !aligned(dev_error, 4) || (fp8 && (!aligned(kr_pool, 16) || !aligned(kv_scale, 4))))
        return MLA_ERR_ALIGNMENT;
    const int64_t num_slots = (int64_t)num_pool_pages * MLA_PAGE_SIZE;
    const dim3 grid((unsigned)(((int64_t)num_tokens + kWarps - 1) / kWarps)), block(kWarps * 32);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint4* src_c = static_cast<const uint4*>(c_kv);
    const uint4* src_r = static_cast<const uint4*>(k_r);
    if (kv_dtype == MLA_KV_NVFP4)
        append_nvfp4_kernel<<<grid, block, 0, s>>>(src_c, src_r, slots, num_tokens, num_slots,
                                                   static_cast<uint8_t*>(kv_pool), kv_scale,
                                                   static_cast<uint4*>(kr_pool), dev_error);
    else if (fp8)
        append_fp8_kernel<<<grid, block, 0, s>>>(src_c, src_r, slots, num_tokens, num_slots,
                                                 static_cast<uint4*>(kv_pool), kv_scale, static_cast<uint4*>(kr_pool),
                                                 dev_error);
    else
        append_bf16_kernel<<<grid, block, 0, s>>>(src_c, src_r, slots, num_tokens, num_slots,
                                                  static_cast<uint4*>(kv_pool), dev_error);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char msg[200];
        snprintf(msg, sizeof msg, "append kernel launch: %s (%s)", cudaGetErrorString(e), cudaGetErrorName(e));
        mla::set_last_error_text(msg);
        return MLA_ERR_CUDA;
    }
    return MLA_OK;
}
