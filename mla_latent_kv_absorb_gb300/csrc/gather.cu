// gather.cu -- mla_gather_kv: the rows of each sequence, in logical order, out of the paged latent
// cache into one contiguous bf16 array (declared in include/mla.h).
//
// Page 1 names an "NVFP4 quantized gather" in its table of contents, and its section 5 describes
// the kernel that reads packed fp4 pages with 16-byte vector loads: a paged cache in, a contiguous
// dequantised one out, for the consumers that want whole rows (prefill over a cached prefix, the
// decompressed form).  bf16 cache: the rows are copied.  FP8 cache: each latent value is the e4m3
// code times the token's fp32 scale, one fp32 rounding, then bf16.  NVFP4 cache: the e2m1 code
// times its block's e4m3 scale (exact) times the token's scale, one fp32 rounding, then bf16.
//
// One warp per token, lane l owning latent values [16 l, 16 l + 16) (one NVFP4 block): 8 or 16
// bytes of codes in, 32 bytes of bf16 out, k_R copied by lanes 0-7.  A streaming copy: no shared
// memory or TMA would pay.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "../../include/mla.h"
#include "nvtx_range.h"

namespace mla {
void set_last_error_text(const char* text);
}

namespace mla::gather {

constexpr int kWarps = 8;  // tokens per CTA

__device__ __forceinline__ float f16_lo(uint32_t h2) { return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))); }
__device__ __forceinline__ float f16_hi(uint32_t h2) { return __half2float(__ushort_as_half((unsigned short)(h2 >> 16))); }

// Two e4m3 codes (low byte first) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two)
{
    uint32_t r;
    const uint16_t c = (uint16_t)(two & 0xFFFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
    return r;
}

// Two e2m1 codes (one byte, value 0 in the low nibble) -> f16x2, exact.
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
    return r;
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

struct Args {
    int kv_dtype;
    const uint8_t* pool;          // bf16 rows [pages][64][576], e4m3 [pages][64][512] or NVFP4 [pages][64][288]
    const float* scale;           // [pages][64]
    const uint4* kr;              // bf16 [pages][64][64]
    int64_t num_pool_pages;
    const int32_t* block_table;   // [B][max_pages]
    int max_pages;
    const int32_t* seq_lens;      // [B], or NULL: one sequence of one_len tokens (cu_seqlens unused)
    const int32_t* cu_seqlens;    // [B + 1]
    int32_t one_len;
    uint4* out;                   // bf16 [total][576]
    uint32_t* dev_error;
};

// grid (ceil(max_pages * 64 / kWarps), B): warp w of CTA x takes token x * kWarps + w of sequence y.
__global__ void __launch_bounds__(kWarps * 32) gather_kv_kernel(const Args a)
{
    const int lane = threadIdx.x & 31, b = blockIdx.y;
    const int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= (a.seq_lens ? __ldg(a.seq_lens + b) : a.one_len)) return;
    const int64_t pg = t / 64;
    const int32_t page = pg < a.max_pages ? __ldg(a.block_table + (int64_t)b * a.max_pages + pg) : -1;
    if (page < 0 || page >= a.num_pool_pages) {
        if (lane == 0) atomicOr(a.dev_error, MLA_DEVERR_BAD_PAGE);
        return;
    }
    const int64_t tok = (int64_t)page * 64 + t % 64;
    uint4* dst = a.out + ((a.seq_lens ? (int64_t)__ldg(a.cu_seqlens + b) : 0) + t) * 72;  // 72 x 16 bytes per row
    if (a.kv_dtype == MLA_KV_BF16) {
        const uint4* src = reinterpret_cast<const uint4*>(a.pool) + tok * 72;
        dst[lane] = __ldg(src + lane);
        dst[32 + lane] = __ldg(src + 32 + lane);
        if (lane < 8) dst[64 + lane] = __ldg(src + 64 + lane);
        return;
    }
    const float sigma = __ldg(a.scale + tok);
    float v[16];
    if (a.kv_dtype == MLA_KV_FP8_E4M3) {
        const uint4 c = __ldg(reinterpret_cast<const uint4*>(a.pool) + tok * 32 + lane);
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = e4m3x2_f16x2(w[k]), hi = e4m3x2_f16x2(w[k] >> 16);
            v[4 * k + 0] = __fmul_rn(f16_lo(lo), sigma);
            v[4 * k + 1] = __fmul_rn(f16_hi(lo), sigma);
            v[4 * k + 2] = __fmul_rn(f16_lo(hi), sigma);
            v[4 * k + 3] = __fmul_rn(f16_hi(hi), sigma);
        }
    } else {
        const uint8_t* row = a.pool + tok * 288;
        const uint2 c = __ldg(reinterpret_cast<const uint2*>(row) + lane);
        const float s_b = f16_lo(e4m3x2_f16x2(__ldg(row + 256 + lane)));
        const uint32_t w[2] = {c.x, c.y};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t h2 = e2m1x2_f16x2((w[k >> 2] >> (8 * (k & 3))) & 0xFFu);
            v[2 * k + 0] = __fmul_rn(f16_lo(h2) * s_b, sigma);  // the first product is exact
            v[2 * k + 1] = __fmul_rn(f16_hi(h2) * s_b, sigma);
        }
    }
    dst[2 * lane] = make_uint4(bf16x2_rn(v[0], v[1]), bf16x2_rn(v[2], v[3]), bf16x2_rn(v[4], v[5]),
                               bf16x2_rn(v[6], v[7]));
    dst[2 * lane + 1] = make_uint4(bf16x2_rn(v[8], v[9]), bf16x2_rn(v[10], v[11]), bf16x2_rn(v[12], v[13]),
                                   bf16x2_rn(v[14], v[15]));
    if (lane < 8) dst[64 + lane] = __ldg(a.kr + tok * 8 + lane);
}

}  // namespace mla::gather

namespace {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// grid over the tokens of max_pages pages of `batch` sequences
mla_status launch(const mla::gather::Args& a, int32_t max_pages, int32_t batch, void* stream)
{
    using namespace mla::gather;
    const int64_t tokens = (int64_t)max_pages * 64;
    const dim3 grid((unsigned)((tokens + kWarps - 1) / kWarps), (unsigned)batch), block(kWarps * 32);
    gather_kv_kernel<<<grid, block, 0, static_cast<cudaStream_t>(stream)>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char msg[200];
        snprintf(msg, sizeof msg, "gather kernel launch: %s (%s)", cudaGetErrorString(e), cudaGetErrorName(e));
        mla::set_last_error_text(msg);
        return MLA_ERR_CUDA;
    }
    return MLA_OK;
}

}  // namespace

extern "C" MLA_API mla_status mla_gather_kv(mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale,
                                            const void* kr_pool, int32_t num_pool_pages, const int32_t* block_table,
                                            int32_t max_pages_per_seq, const int32_t* seq_lens,
                                            const int32_t* cu_seqlens, int32_t batch, void* out, uint32_t* dev_error,
                                            void* stream)
{
    const mla::NvtxRange nvtx_range("mla_gather_kv");
    using namespace mla::gather;
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3 && kv_dtype != MLA_KV_NVFP4) return MLA_ERR_INVALID_ARG;
    if (batch <= 0 || num_pool_pages <= 0 || max_pages_per_seq <= 0) return MLA_ERR_INVALID_ARG;
    if (!kv_pool || !block_table || !seq_lens || !cu_seqlens || !out || !dev_error) return MLA_ERR_INVALID_ARG;
    const bool quant = kv_dtype != MLA_KV_BF16;
    if (quant && (!kv_scale || !kr_pool)) return MLA_ERR_INVALID_ARG;
    if (!aligned(kv_pool, 16) || !aligned(out, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
        !aligned(cu_seqlens, 4) || !aligned(dev_error, 4) || (quant && (!aligned(kr_pool, 16) || !aligned(kv_scale, 4))))
        return MLA_ERR_ALIGNMENT;
    if (batch > 65535) return MLA_ERR_UNSUPPORTED;  // the grid's y dimension
    Args a;
    a.kv_dtype = (int)kv_dtype;
    a.pool = static_cast<const uint8_t*>(kv_pool);
    a.scale = kv_scale;
    a.kr = static_cast<const uint4*>(kr_pool);
    a.num_pool_pages = num_pool_pages;
    a.block_table = block_table;
    a.max_pages = max_pages_per_seq;
    a.seq_lens = seq_lens;
    a.cu_seqlens = cu_seqlens;
    a.one_len = 0;
    a.out = static_cast<uint4*>(out);
    a.dev_error = dev_error;
    return launch(a, max_pages_per_seq, batch, stream);
}

namespace mla {
// One sequence of seq_len tokens (its block-table row given), rows to out [seq_len][576]; the
// caller has checked the arguments as mla_gather_kv does.
mla_status gather_one_sequence(mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale, const void* kr_pool,
                               int32_t num_pool_pages, const int32_t* block_table_row, int32_t max_pages,
                               int32_t seq_len, void* out, uint32_t* dev_error, void* stream)
{
    using namespace mla::gather;
    Args a;
    a.kv_dtype = (int)kv_dtype;
    a.pool = static_cast<const uint8_t*>(kv_pool);
    a.scale = kv_scale;
    a.kr = static_cast<const uint4*>(kr_pool);
    a.num_pool_pages = num_pool_pages;
    a.block_table = block_table_row;
    a.max_pages = max_pages;
    a.seq_lens = nullptr;
    a.cu_seqlens = nullptr;
    a.one_len = seq_len;
    a.out = static_cast<uint4*>(out);
    a.dev_error = dev_error;
    return launch(a, (seq_len + 63) / 64, 1, stream);
}
}  // namespace mla
