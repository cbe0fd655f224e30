// api.cu -- the C ABI of libmla_gb300.so (declared in include/mla.h): host-side argument
// checks, TMA tensor-map encoding and kernel launches.  No allocation, no global mutable state
// (the driver entry point for tensor-map encoding is looked up once, thread-safely).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <utility>

#include "../../include/mla.h"
#include "combine.cuh"
#include "decode.cuh"
#include "decode_fp8.cuh"
#include "head_gemm.cuh"
#include "nvtx_range.h"
#include "plan.h"
#include "prefill.cuh"
#include "tail.cuh"

namespace {

using mla::gemm::Cfg;

// absorb: K = 128 (d_hc), N tile 256 of 512 (d_c), W_UK is MN-major for the MMA; 256 CTAs of
// 96 KB (two per SM) run as one wave
constexpr int kAbsorbN = 256;
constexpr int kAbsorbStages = 2;
using AbsorbCfg = Cfg<128, kAbsorbN, true, kAbsorbStages>;
// out-proj: K = 512 (d_c), the whole head's N = 128 (d_hc) per CTA, W_UV is K-major for the MMA;
// six of the eight K-chunks in flight, 128 CTAs of 192 KB (one wave)
constexpr int kOutN = 128;
constexpr int kOutStages = 6;
using OutCfg = Cfg<512, kOutN, false, kOutStages>;

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

#ifdef MLA_DECODE_TRACE
long long* g_trace = nullptr;  // wait-cycle accounting buffer, instrumented builds only
#endif

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// Tiled tensor map.  dims/strides innermost first; strides in bytes for dims 1.. (rank - 1
// entries).
bool make_map(CUtensorMap* m, CUtensorMapDataType type, CUtensorMapSwizzle swizzle, const void* base, int rank,
              const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return enc(m, type, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 tensor map with 128-byte swizzle.
bool make_map_bf16(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box)
{
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B, base, rank, dims, strides, box);
}

// Text of the last CUDA failure seen by this host thread (thread-local: no shared state).
thread_local char t_last_error[256] = "no error";

mla_status record_cuda(cudaError_t e, const char* where)
{
    if (e == cudaSuccess) return MLA_OK;
    snprintf(t_last_error, sizeof t_last_error, "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
    return MLA_ERR_CUDA;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename K>
bool set_smem(K kernel, int bytes)
{
    return record_cuda(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                       "cudaFuncSetAttribute(max dynamic shared memory)") == MLA_OK;
}

mla_status launch_status()
{
    return record_cuda(cudaGetLastError(), "kernel launch");
}

// Launch with programmatic stream serialisation: the kernel may be scheduled before the kernel
// ahead of it in the stream has finished (once that one allows it) and waits for that kernel's
// output itself (griddepcontrol.wait), so its prologue and its independent loads overlap the
// other's tail.  Every kernel of the step that reads the previous one's output does that wait.
template <typename... KArgs, typename... Args>
mla_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return record_cuda(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...), "cudaLaunchKernelEx");
}

// Shared by absorb and out-proj: activations [batch][128][K] (K-major rows of 128*K), weights
// [128][128][512].
// shared_act_row > 0: one activation row of that many elements per batch row, shared by all
// heads (the first K_TOTAL elements are the operand).
// head_major: out is [128 heads][batch][n_total] instead of [batch][128 heads][n_total].
template <int K_TOTAL, int N_TILE, bool W_MN, int STAGES>
mla_status launch_head_gemm(const void* act, const void* weight, void* out, int32_t batch, int n_total,
                            cuuint32_t w_box_rows, bool pdl, void* stream, int shared_act_row = 0,
                            bool head_major = false)
{
    using C = Cfg<K_TOTAL, N_TILE, W_MN, STAGES>;
    CUtensorMap tm_a, tm_w;
    const cuuint64_t a_row = shared_act_row > 0 ? (cuuint64_t)shared_act_row : (cuuint64_t)128 * K_TOTAL;
    const cuuint64_t a_dims[2] = {a_row, (cuuint64_t)batch};
    const cuuint64_t a_str[1] = {a_row * 2};
    const cuuint32_t a_box[2] = {64, 128};
    const cuuint64_t w_dims[2] = {512, 128 * 128};
    const cuuint64_t w_str[1] = {512 * 2};
    const cuuint32_t w_box[2] = {64, w_box_rows};
    if (!make_map_bf16(&tm_a, act, 2, a_dims, a_str, a_box) || !make_map_bf16(&tm_w, weight, 2, w_dims, w_str, w_box))
        return MLA_ERR_CUDA;
    auto kernel = mla::gemm::head_gemm_kernel<K_TOTAL, N_TILE, W_MN, STAGES>;
    if (!set_smem(kernel, C::kSmemBytes)) return MLA_ERR_CUDA;
    mla::gemm::Args args;
    args.out = static_cast<__nv_bfloat16*>(out);
    args.a_x_per_head = shared_act_row > 0 ? 0 : K_TOTAL;
    args.batch = batch;
    args.out_row_stride = head_major ? (int64_t)n_total : (int64_t)128 * n_total;
    args.out_head_stride = head_major ? (int64_t)batch * n_total : (int64_t)n_total;
    args.n_total = n_total;
    args.dev_error = nullptr;
    args.timeout_ns = kDefaultTimeoutNs;
    const dim3 grid(n_total / N_TILE, 128, (batch + 127) / 128);
    if (pdl) return launch_pdl(kernel, grid, dim3(192), C::kSmemBytes, static_cast<cudaStream_t>(stream), tm_a, tm_w, args);
    kernel<<<grid, 192, C::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(tm_a, tm_w, args);
    return launch_status();
}

bool plan_header_ok(const mla_plan_info* info)
{
    return info && info->batch > 0 && info->num_clusters > 0 && info->num_items > 0 && info->num_partials >= 0 &&
           info->num_combine >= 0 && info->plan_bytes > 0 && info->workspace_bytes >= 0 && info->wait_timeout_ns > 0;
}

__global__ void wait_timeout_kernel(uint32_t* dev_error, uint64_t timeout_ns)
{
    using namespace mla::dev;
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);  // nothing will ever arrive
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtx w{timeout_ns, &abort_flag, dev_error};
        wait_phase(smem_u32(&bar), 0, w);
    }
    __syncthreads();
}

}  // namespace

#ifdef MLA_DECODE_TRACE
extern "C" __attribute__((visibility("default"))) void mla_debug_set_trace(long long* trace) { g_trace = trace; }
extern "C" __attribute__((visibility("default"))) int mla_debug_timeout_sites(unsigned long long* host, int n, int clear)
{
    if (n > 1024) n = 1024;
    if (cudaMemcpyFromSymbol(host, mla::dev::g_timeout_site, sizeof(unsigned long long) * n) != cudaSuccess) return -1;
    if (clear) {
        static unsigned long long zeros[1024];
        cudaMemcpyToSymbol(mla::dev::g_timeout_site, zeros, sizeof zeros);
    }
    return 0;
}
#endif

// The e4m3 cache: c8 [pages][64][512] bytes (boxes of 128 columns x 64 tokens, 128-byte
// swizzle: the e4m3 MMAs read them as they land), kr_pool [pages][64][64] bf16 (64x64 boxes,
// 128-byte swizzle), one fp32 scale per token (read with plain loads).
mla_status launch_decode_fp8(const mla_plan_info* info, const void* plan_dev, const void* q_abs, const void* q_r,
                             const void* kv_pool, const float* kv_scale, const void* kr_pool, int32_t num_pool_pages,
                             const int32_t* block_table, int32_t max_pages_per_seq, float softmax_scale,
                             void* workspace, void* o_lat, float* lse, uint32_t* dev_error, void* stream)
{
    if (!aligned16(kr_pool) || (reinterpret_cast<uintptr_t>(kv_scale) & 3u)) return MLA_ERR_ALIGNMENT;
    CUtensorMap tm_c8, tm_kr, tm_q;
    const cuuint64_t c_dims[3] = {512, 64, (cuuint64_t)num_pool_pages};
    const cuuint64_t c_strides[2] = {512, 64 * 512};
    const cuuint32_t c_box[3] = {128, 64, 1};
    const cuuint64_t r_dims[3] = {64, 64, (cuuint64_t)num_pool_pages};
    const cuuint64_t r_strides[2] = {64 * 2, 64 * 64 * 2};
    const cuuint32_t r_box[3] = {64, 64, 1};
    if (!make_map(&tm_c8, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_128B, kv_pool, 3, c_dims, c_strides,
                  c_box) ||
        !make_map_bf16(&tm_kr, kr_pool, 3, r_dims, r_strides, r_box))
        return MLA_ERR_CUDA;
    // q_abs as [batch * 128 rows][512], boxes of 128 rows (one query row's heads) x 64 dims
    const cuuint64_t q_dims[2] = {512, (cuuint64_t)info->batch * 128};
    const cuuint64_t q_str[1] = {512 * 2};
    const cuuint32_t q_box[2] = {64, 128};
    if (!make_map_bf16(&tm_q, q_abs, 2, q_dims, q_str, q_box)) return MLA_ERR_CUDA;

    mla::decode_fp8::Params p;
    p.plan = static_cast<const int32_t*>(plan_dev);
    p.q_abs = static_cast<const __nv_bfloat16*>(q_abs);
    p.q_r = static_cast<const __nv_bfloat16*>(q_r);
    p.block_table = block_table;
    p.max_pages = max_pages_per_seq;
    p.num_pool_pages = num_pool_pages;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.o_lat = static_cast<__nv_bfloat16*>(o_lat);
    p.lse = lse;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_lse = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                    (size_t)info->num_partials * mla::kPartialOBytes)
                         : nullptr;
    p.dev_error = dev_error;
    p.timeout_ns = (uint64_t)info->wait_timeout_ns;
    p.kv_scale = kv_scale;
#ifdef MLA_DECODE_TRACE
    p.trace = g_trace;
#else
    p.trace = nullptr;
#endif

    if (!set_smem(mla::decode_fp8::decode_fp8_kernel, mla::decode_fp8::kSmemBytes)) return MLA_ERR_CUDA;
    return launch_pdl(mla::decode_fp8::decode_fp8_kernel, dim3(2 * info->num_clusters), dim3(mla::decode_fp8::kThreads),
                      mla::decode_fp8::kSmemBytes, static_cast<cudaStream_t>(stream), tm_c8, tm_kr, tm_q, p);
}

// Host checks shared by the decode entry points (nothing is launched when one fails).
mla_status check_decode_args(const mla_plan_info* info, const void* plan_dev, const void* q_abs, const void* q_r,
                             mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale, const void* kr_pool,
                             int32_t num_pool_pages, const int32_t* block_table, int32_t max_pages_per_seq,
                             float softmax_scale, const void* workspace, size_t workspace_bytes, const void* o_lat,
                             const float* lse, const uint32_t* dev_error)
{
    if (!plan_header_ok(info) || !plan_dev || !q_abs || !q_r || !kv_pool || !block_table || !o_lat || !lse ||
        !dev_error)
        return MLA_ERR_INVALID_ARG;
    if (num_pool_pages <= 0 || max_pages_per_seq <= 0 || !(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
        return MLA_ERR_INVALID_ARG;
    if (kv_dtype == MLA_KV_NVFP4) return MLA_ERR_UNSUPPORTED;  // written by mla_append_kv; no decode kernel reads it
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
    if (kv_dtype == MLA_KV_FP8_E4M3 && (!kv_scale || !kr_pool)) return MLA_ERR_INVALID_ARG;
    if (!aligned16(plan_dev) || !aligned16(q_abs) || !aligned16(q_r) || !aligned16(kv_pool) || !aligned16(o_lat) ||
        !aligned16(lse) || (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(dev_error) & 3u))
        return MLA_ERR_ALIGNMENT;
    if (info->workspace_bytes > 0) {
        if (!workspace || workspace_bytes < (size_t)info->workspace_bytes) return MLA_ERR_WORKSPACE;
        if (!aligned16(workspace)) return MLA_ERR_ALIGNMENT;
    }
    return MLA_OK;
}

// The bf16 decode kernel.  With q_c, w_uk and absorb_sync given, the absorb runs as the kernel's
// prologue (q_abs is then an output) and the kernel is an ordinary launch; otherwise q_abs is an
// input written by the kernel before it, and the launch is programmatic (it may start early).
mla_status launch_decode_bf16(const mla_plan_info* info, const void* plan_dev, const void* q_abs, const void* q_r,
                              const void* kv_pool, int32_t num_pool_pages, const int32_t* block_table,
                              int32_t max_pages_per_seq, float softmax_scale, void* workspace, void* o_lat, float* lse,
                              uint32_t* dev_error, void* stream, const void* q_c, const void* w_uk,
                              uint32_t* absorb_sync)
{
    const bool fused = absorb_sync != nullptr;
    CUtensorMap tm_pool, tm_q, tm_qc, tm_wuk;
    const cuuint64_t dims[3] = {576, 64, (cuuint64_t)num_pool_pages};
    const cuuint64_t strides[2] = {576 * 2, 64 * 576 * 2};
    const cuuint32_t box[3] = {64, 64, 1};
    // q_abs as [batch * 128 rows][512], boxes of 128 rows (one sequence's heads) x 64 dims
    const cuuint64_t q_dims[2] = {512, (cuuint64_t)info->batch * 128};
    const cuuint64_t q_str[1] = {512 * 2};
    const cuuint32_t q_box[2] = {64, 128};
    if (!make_map_bf16(&tm_pool, kv_pool, 3, dims, strides, box) || !make_map_bf16(&tm_q, q_abs, 2, q_dims, q_str, q_box))
        return MLA_ERR_CUDA;
    tm_qc = tm_q;
    tm_wuk = tm_q;
    if (fused) {
        // the absorb prologue's operands: q_c rows [batch][128 x 128] in 128-row x 64 boxes, and
        // W_UK [128 x 128 rows][512] in 64 x 64 boxes (MN-major B)
        const cuuint64_t c_dims[2] = {128 * 128, (cuuint64_t)info->batch};
        const cuuint64_t c_str[1] = {128 * 128 * 2};
        const cuuint32_t c_box[2] = {64, 128};
        const cuuint64_t w_dims[2] = {512, 128 * 128};
        const cuuint64_t w_str[1] = {512 * 2};
        const cuuint32_t w_box[2] = {64, 64};
        if (!make_map_bf16(&tm_qc, q_c, 2, c_dims, c_str, c_box) || !make_map_bf16(&tm_wuk, w_uk, 2, w_dims, w_str, w_box))
            return MLA_ERR_CUDA;
    }

    mla::decode::Params p;
    p.plan = static_cast<const int32_t*>(plan_dev);
    p.q_abs = static_cast<const __nv_bfloat16*>(q_abs);
    p.q_abs_out = fused ? static_cast<__nv_bfloat16*>(const_cast<void*>(q_abs)) : nullptr;
    p.absorb_sync = absorb_sync;
    p.absorb_jobs = fused ? 128 * ((info->batch + 127) / 128) : 0;
    p.batch = info->batch;
    p.q_r = static_cast<const __nv_bfloat16*>(q_r);
    p.block_table = block_table;
    p.max_pages = max_pages_per_seq;
    p.num_pool_pages = num_pool_pages;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.o_lat = static_cast<__nv_bfloat16*>(o_lat);
    p.lse = lse;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_lse = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                    (size_t)info->num_partials * mla::kPartialOBytes)
                         : nullptr;
    p.dev_error = dev_error;
    p.timeout_ns = (uint64_t)info->wait_timeout_ns;
#ifdef MLA_DECODE_TRACE
    p.trace = g_trace;
#else
    p.trace = nullptr;
#endif

    if (!set_smem(mla::decode::decode_bf16_kernel, mla::decode::kSmemBytes)) return MLA_ERR_CUDA;
    if (!fused)
        return launch_pdl(mla::decode::decode_bf16_kernel, dim3(2 * info->num_clusters), dim3(mla::decode::kThreads),
                          mla::decode::kSmemBytes, static_cast<cudaStream_t>(stream), tm_pool, tm_q, tm_qc, tm_wuk, p);
    // enough CTA pairs that no CTA takes more than one absorb job while one fits per SM, and
    // never fewer than the plan's (pairs past the plan's only run absorb jobs)
    int dev = 0, sms = 0;
    if (record_cuda(cudaGetDevice(&dev), "cudaGetDevice") != MLA_OK ||
        record_cuda(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute") != MLA_OK)
        return MLA_ERR_CUDA;
    const int clusters = std::max(info->num_clusters, std::min(sms / 2, (p.absorb_jobs + 1) / 2));
    mla::decode::decode_bf16_kernel<<<dim3(2 * clusters), dim3(mla::decode::kThreads), mla::decode::kSmemBytes,
                                      static_cast<cudaStream_t>(stream)>>>(tm_pool, tm_q, tm_qc, tm_wuk, p);
    return launch_status();
}

extern "C" mla_status mla_absorb_q(const void* q_c, const void* w_uk, void* q_abs, int32_t batch, void* stream)
{
    const mla::NvtxRange nvtx_range("mla_absorb_q");
    if (!q_c || !w_uk || !q_abs || batch <= 0) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_c) || !aligned16(w_uk) || !aligned16(q_abs)) return MLA_ERR_ALIGNMENT;
    // the step's first kernel: an ordinary launch (it allows the decode kernel to start early)
    return launch_head_gemm<128, kAbsorbN, true, kAbsorbStages>(q_c, w_uk, q_abs, batch, 512, 64, false, stream);
}

extern "C" mla_status mla_out_proj(const void* o_lat, const void* w_uv, void* out, int32_t batch, void* stream)
{
    const mla::NvtxRange nvtx_range("mla_out_proj");
    if (!o_lat || !w_uv || !out || batch <= 0) return MLA_ERR_INVALID_ARG;
    if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(out)) return MLA_ERR_ALIGNMENT;
    // streams W_UV while the merge (or the decode) before it finishes
    return launch_head_gemm<512, kOutN, false, kOutStages>(o_lat, w_uv, out, batch, 128, kOutN, true, stream);
}

extern "C" mla_status mla_decode_paged(const mla_plan_info* info, const void* plan_dev, const void* q_abs,
                                       const void* q_r, mla_kv_dtype kv_dtype, const void* kv_pool,
                                       const float* kv_scale, const void* kr_pool, int32_t num_pool_pages,
                                       const int32_t* block_table, int32_t max_pages_per_seq, float softmax_scale,
                                       void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                                       uint32_t* dev_error, void* stream)
{
    const mla::NvtxRange nvtx_range("mla_decode_paged");
    const mla_status st = check_decode_args(info, plan_dev, q_abs, q_r, kv_dtype, kv_pool, kv_scale, kr_pool,
                                            num_pool_pages, block_table, max_pages_per_seq, softmax_scale, workspace,
                                            workspace_bytes, o_lat, lse, dev_error);
    if (st != MLA_OK) return st;
    if (kv_dtype == MLA_KV_FP8_E4M3)
        return launch_decode_fp8(info, plan_dev, q_abs, q_r, kv_pool, kv_scale, kr_pool, num_pool_pages, block_table,
                                 max_pages_per_seq, softmax_scale, workspace, o_lat, lse, dev_error, stream);

    return launch_decode_bf16(info, plan_dev, q_abs, q_r, kv_pool, num_pool_pages, block_table, max_pages_per_seq,
                              softmax_scale, workspace, o_lat, lse, dev_error, stream, nullptr, nullptr, nullptr);
}


extern "C" mla_status mla_absorb_decode_paged(const mla_plan_info* info, const void* plan_dev, const void* q_c,
                                              const void* w_uk, void* q_abs, uint32_t* absorb_sync, const void* q_r,
                                              mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale,
                                              const void* kr_pool, int32_t num_pool_pages, const int32_t* block_table,
                                              int32_t max_pages_per_seq, float softmax_scale, void* workspace,
                                              size_t workspace_bytes, void* o_lat, float* lse, uint32_t* dev_error,
                                              void* stream)
{
    const mla::NvtxRange nvtx_range("mla_absorb_decode_paged");
    if (!q_c || !w_uk || !q_abs || !absorb_sync || !info) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_c) || !aligned16(w_uk) || (reinterpret_cast<uintptr_t>(absorb_sync) & 7u)) return MLA_ERR_ALIGNMENT;
    if (kv_dtype == MLA_KV_FP8_E4M3) {
        // the e4m3 decode kernel has no absorb prologue: the absorb runs as its own kernel first
        mla_status st = mla_absorb_q(q_c, w_uk, q_abs, info->batch, stream);
        if (st != MLA_OK) return st;
        return mla_decode_paged(info, plan_dev, q_abs, q_r, kv_dtype, kv_pool, kv_scale, kr_pool, num_pool_pages,
                                block_table, max_pages_per_seq, softmax_scale, workspace, workspace_bytes, o_lat, lse,
                                dev_error, stream);
    }
    const mla_status st = check_decode_args(info, plan_dev, q_abs, q_r, kv_dtype, kv_pool, kv_scale, kr_pool,
                                            num_pool_pages, block_table, max_pages_per_seq, softmax_scale, workspace,
                                            workspace_bytes, o_lat, lse, dev_error);
    if (st != MLA_OK) return st;
    return launch_decode_bf16(info, plan_dev, q_abs, q_r, kv_pool, num_pool_pages, block_table, max_pages_per_seq,
                              softmax_scale, workspace, o_lat, lse, dev_error, stream, q_c, w_uk, absorb_sync);
}

extern "C" mla_status mla_combine_splits(const mla_plan_info* info, const void* plan_dev, const void* workspace,
                                         size_t workspace_bytes, void* o_lat, float* lse, void* stream)
{
    const mla::NvtxRange nvtx_range("mla_combine_splits");
    if (!plan_header_ok(info) || !plan_dev || !o_lat || !lse) return MLA_ERR_INVALID_ARG;
    if (info->num_combine == 0) return MLA_OK;
    if (!workspace || workspace_bytes < (size_t)info->workspace_bytes) return MLA_ERR_WORKSPACE;
    if (!aligned16(plan_dev) || !aligned16(workspace) || !aligned16(o_lat) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return MLA_ERR_ALIGNMENT;
    const float* ws_o = static_cast<const float*>(workspace);
    const float* ws_lse = reinterpret_cast<const float*>(static_cast<const char*>(workspace) +
                                                         (size_t)info->num_partials * mla::kPartialOBytes);
    const dim3 grid(info->num_combine, 128 / mla::combine::kHeadsPerCta);
    return launch_pdl(mla::combine::combine_kernel, grid, dim3(32 * mla::combine::kHeadsPerCta), 0,
                      static_cast<cudaStream_t>(stream), static_cast<const int32_t*>(plan_dev), ws_o, ws_lse,
                      static_cast<__nv_bfloat16*>(o_lat), lse);
}

extern "C" mla_status mla_merge_out_proj(const mla_plan_info* info, const void* plan_dev, const void* workspace,
                                         size_t workspace_bytes, void* o_lat, float* lse, const void* w_uv, void* out,
                                         uint32_t* dev_error, void* stream)
{
    const mla::NvtxRange nvtx_range("mla_merge_out_proj");
    if (!plan_header_ok(info) || !plan_dev || !o_lat || !lse || !w_uv || !out) return MLA_ERR_INVALID_ARG;
    if (info->num_combine > 0 && (!workspace || workspace_bytes < (size_t)info->workspace_bytes))
        return MLA_ERR_WORKSPACE;
    if (!aligned16(plan_dev) || !aligned16(o_lat) || !aligned16(w_uv) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (workspace && !aligned16(workspace)) ||
        (reinterpret_cast<uintptr_t>(dev_error) & 3u))
        return MLA_ERR_ALIGNMENT;
    CUtensorMap tm_w;
    const cuuint64_t w_dims[2] = {512, 128 * 128};
    const cuuint64_t w_str[1] = {512 * 2};
    const cuuint32_t w_box[2] = {mla::tail::kKC, 128};
    if (!make_map_bf16(&tm_w, w_uv, 2, w_dims, w_str, w_box)) return MLA_ERR_CUDA;
    mla::tail::Args a;
    a.plan = static_cast<const int32_t*>(plan_dev);
    a.ws_o = static_cast<const float*>(workspace);
    a.ws_lse = workspace ? reinterpret_cast<const float*>(static_cast<const char*>(workspace) +
                                                          (size_t)info->num_partials * mla::kPartialOBytes)
                         : nullptr;
    a.o_lat = static_cast<__nv_bfloat16*>(o_lat);
    a.lse = lse;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.batch = info->batch;
    a.dev_error = dev_error;
    a.timeout_ns = (uint64_t)info->wait_timeout_ns;
    if (!set_smem(mla::tail::merge_out_proj_kernel, mla::tail::kSmemBytes)) return MLA_ERR_CUDA;
    return launch_pdl(mla::tail::merge_out_proj_kernel, dim3(128, (info->batch + 127) / 128), dim3(mla::tail::kThreads),
                      mla::tail::kSmemBytes, static_cast<cudaStream_t>(stream), tm_w, a);
}

namespace mla {
// gather.cu: one sequence's cache rows into contiguous bf16 rows [seq_len][576]
mla_status gather_one_sequence(mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale, const void* kr_pool,
                               int32_t num_pool_pages, const int32_t* block_table_row, int32_t max_pages,
                               int32_t seq_len, void* out, uint32_t* dev_error, void* stream);
}  // namespace mla

namespace {

// Workspace of the decompressed prefill: gathered rows [S][576], k [128][S][128], v [128][S][128]
// (bf16, head-major), each section 1024-byte aligned.
struct PrefillLayout {
    size_t rows, k, v, total;
};

PrefillLayout prefill_layout(int64_t seq_len)
{
    const auto up = [](size_t x) { return (x + 1023) & ~(size_t)1023; };
    const size_t rows = up((size_t)seq_len * 576 * 2), kv = up((size_t)seq_len * 128 * 128 * 2);
    return PrefillLayout{0, rows, rows + kv, rows + 2 * kv};
}

}  // namespace

extern "C" size_t mla_prefill_workspace_bytes(int32_t seq_len)
{
    return seq_len > 0 ? prefill_layout(seq_len).total : 0;
}

extern "C" mla_status mla_prefill_decompressed(mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale,
                                               const void* kr_pool, int32_t num_pool_pages,
                                               const int32_t* block_table_row, int32_t max_pages, int32_t seq_len,
                                               int32_t chunk_len, const void* q_c, const void* q_r, const void* w_uk,
                                               const void* w_uv, float softmax_scale, void* workspace,
                                               size_t workspace_bytes, void* out, uint32_t* dev_error, void* stream)
{
    const mla::NvtxRange nvtx_range("mla_prefill_decompressed");
    if (!kv_pool || !block_table_row || !q_c || !q_r || !w_uk || !w_uv || !workspace || !out || !dev_error)
        return MLA_ERR_INVALID_ARG;
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3 && kv_dtype != MLA_KV_NVFP4) return MLA_ERR_INVALID_ARG;
    if (kv_dtype != MLA_KV_BF16 && (!kv_scale || !kr_pool)) return MLA_ERR_INVALID_ARG;
    if (seq_len < 1 || chunk_len < 1 || chunk_len > seq_len || num_pool_pages < 1 || max_pages < 1 ||
        (seq_len + 63) / 64 > max_pages || !(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(kv_pool) || !aligned16(q_c) || !aligned16(q_r) || !aligned16(w_uk) || !aligned16(w_uv) ||
        !aligned16(workspace) || !aligned16(out) || (reinterpret_cast<uintptr_t>(block_table_row) & 3u) ||
        (reinterpret_cast<uintptr_t>(dev_error) & 3u) ||
        (kv_dtype != MLA_KV_BF16 && (!aligned16(kr_pool) || (reinterpret_cast<uintptr_t>(kv_scale) & 3u))))
        return MLA_ERR_ALIGNMENT;
    if ((int64_t)seq_len > (int64_t)65535 * 128) return MLA_ERR_UNSUPPORTED;  // grid z of the decompression
    const PrefillLayout lay = prefill_layout(seq_len);
    if (workspace_bytes < lay.total) return MLA_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    void *rows = ws + lay.rows, *k = ws + lay.k, *v = ws + lay.v;

    // 1. the sequence's cache rows, dequantised to bf16
    mla_status st = mla::gather_one_sequence(kv_dtype, kv_pool, kv_scale, kr_pool, num_pool_pages, block_table_row,
                                             max_pages, seq_len, rows, dev_error, stream);
    if (st != MLA_OK) return st;
    // 2. per-head keys and values (the out-proj GEMM shape, activations shared by the heads)
    if ((st = launch_head_gemm<512, kOutN, false, kOutStages>(rows, w_uk, k, seq_len, 128, kOutN, false, stream, 576,
                                                              true)) != MLA_OK ||
        (st = launch_head_gemm<512, kOutN, false, kOutStages>(rows, w_uv, v, seq_len, 128, kOutN, false, stream, 576,
                                                              true)) != MLA_OK)
        return st;
    // 3. causal attention of the chunk's queries
    CUtensorMap tm_qc, tm_qr, tm_k, tm_kr, tm_v;
    const cuuint64_t qc_dims[3] = {128, 128, (cuuint64_t)chunk_len};
    const cuuint64_t qc_str[2] = {128 * 2, 128 * 128 * 2};
    const cuuint64_t qr_dims[3] = {64, 128, (cuuint64_t)chunk_len};
    const cuuint64_t qr_str[2] = {64 * 2, 128 * 64 * 2};
    const cuuint32_t q_box[3] = {64, 1, 128};
    // k and v head-major [128 heads][S][128]: boxes of 64 dims x one key tile of one head
    constexpr cuuint32_t kKeys = mla::prefill::kKV;
    const cuuint64_t k_dims[3] = {128, (cuuint64_t)seq_len, 128};
    const cuuint64_t k_str[2] = {128 * 2, (cuuint64_t)seq_len * 128 * 2};
    const cuuint32_t k_box[3] = {64, kKeys, 1};
    const cuuint64_t r_dims[2] = {576, (cuuint64_t)seq_len};
    const cuuint64_t r_str[1] = {576 * 2};
    const cuuint32_t r_box[2] = {64, kKeys};
    if (!make_map_bf16(&tm_qc, q_c, 3, qc_dims, qc_str, q_box) || !make_map_bf16(&tm_qr, q_r, 3, qr_dims, qr_str, q_box) ||
        !make_map_bf16(&tm_k, k, 3, k_dims, k_str, k_box) || !make_map_bf16(&tm_kr, rows, 2, r_dims, r_str, r_box) ||
        !make_map_bf16(&tm_v, v, 3, k_dims, k_str, k_box))
        return MLA_ERR_CUDA;
    mla::prefill::Params p;
    p.seq_len = seq_len;
    p.chunk_len = chunk_len;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.dev_error = dev_error;
    p.timeout_ns = kDefaultTimeoutNs;
    if (!set_smem(mla::prefill::prefill_attn_kernel, mla::prefill::kSmemBytes)) return MLA_ERR_CUDA;
    constexpr int kQueriesPerCta = mla::prefill::kQ * mla::prefill::kQT;
    const dim3 grid((unsigned)((chunk_len + kQueriesPerCta - 1) / kQueriesPerCta), 128);
    mla::prefill::prefill_attn_kernel<<<grid, mla::prefill::kThreads, mla::prefill::kSmemBytes,
                                        static_cast<cudaStream_t>(stream)>>>(tm_qc, tm_qr, tm_k, tm_kr, tm_v, p);
    return launch_status();
}

extern "C" const char* mla_last_error_string(void) { return t_last_error; }

namespace mla {
// For the library's other translation units: replace this thread's last-error text.
void set_last_error_text(const char* text) { snprintf(t_last_error, sizeof t_last_error, "%s", text); }
}  // namespace mla

extern "C" mla_status mla_read_device_error(const uint32_t* dev_error, uint32_t* host_bits, void* stream)
{
    if (!dev_error) return MLA_ERR_INVALID_ARG;
    uint32_t bits = 0;
    if (cudaMemcpyAsync(&bits, dev_error, sizeof bits, cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream)) !=
            cudaSuccess ||
        cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (host_bits) *host_bits = bits;
    return bits ? MLA_ERR_DEVICE_FAULT : MLA_OK;
}

extern "C" mla_status mla_debug_wait_timeout(uint32_t* dev_error, int64_t timeout_ns, void* stream)
{
    if (!dev_error || timeout_ns < 1000000 || timeout_ns > 10000000000LL) return MLA_ERR_INVALID_ARG;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_error, (uint64_t)timeout_ns);
    return launch_status();
}

namespace {

// Host checks of the step-from-host entry points, then the plan for seq_lens into
// bufs->plan_host (nothing is copied or launched here).
mla_status step_prepare(const int32_t* seq_lens, int32_t batch, int32_t num_sms, const mla_plan_options* opts,
                        const void* q_c_host, const void* q_r_host, int32_t max_pages_per_seq,
                        const mla_step_buffers* bufs, const void* out_host, mla_plan_info* info)
{
    if (!seq_lens || batch <= 0 || !q_c_host || !q_r_host || !bufs || !out_host || !bufs->plan_host ||
        !bufs->plan || !bufs->block_table || max_pages_per_seq <= 0)
        return MLA_ERR_INVALID_ARG;
    for (int32_t b = 0; b < batch; ++b)  // every page of every sequence has a block-table entry
        if (seq_lens[b] > 0 && (seq_lens[b] + 63) / 64 > max_pages_per_seq) return MLA_ERR_INVALID_ARG;
    const mla_status st = mla_plan_splits(seq_lens, batch, num_sms, opts, bufs->plan_host, bufs->plan_capacity, info);
    if (st != MLA_OK) return st;
    if (info->workspace_bytes > 0 && (!bufs->workspace || bufs->workspace_bytes < (size_t)info->workspace_bytes))
        return MLA_ERR_WORKSPACE;
    return MLA_OK;
}

// The step's stream work after planning: the plan copy (when copy_plan), the block table and
// query copies, absorb, decode, merge, projection, and the output copy back.
mla_status step_enqueue(const mla_plan_info& info, bool copy_plan, const void* q_c_host, const void* q_r_host,
                        const int32_t* block_table_host, int32_t max_pages_per_seq, const void* w_uk, const void* w_uv,
                        mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale, const void* kr_pool,
                        int32_t num_pool_pages, float softmax_scale, const mla_step_buffers* bufs, void* out_host,
                        cudaStream_t s)
{
    const int32_t batch = info.batch;  // query rows
    const int32_t table_rows = info.batch / std::max(1, info.queries_per_seq);
    const size_t q_c_bytes = (size_t)batch * 128 * 128 * 2, q_r_bytes = (size_t)batch * 128 * 64 * 2;
    if (copy_plan && record_cuda(cudaMemcpyAsync(bufs->plan, bufs->plan_host, (size_t)info.plan_bytes,
                                                 cudaMemcpyHostToDevice, s),
                                 "cudaMemcpyAsync(plan)") != MLA_OK)
        return MLA_ERR_CUDA;
    if (block_table_host &&
        record_cuda(cudaMemcpyAsync(bufs->block_table, block_table_host,
                                    (size_t)table_rows * (size_t)max_pages_per_seq * sizeof(int32_t),
                                    cudaMemcpyHostToDevice, s),
                    "cudaMemcpyAsync(block table)") != MLA_OK)
        return MLA_ERR_CUDA;
    if (record_cuda(cudaMemcpyAsync(bufs->q_c, q_c_host, q_c_bytes, cudaMemcpyHostToDevice, s),
                    "cudaMemcpyAsync(q_c)") != MLA_OK ||
        record_cuda(cudaMemcpyAsync(bufs->q_r, q_r_host, q_r_bytes, cudaMemcpyHostToDevice, s),
                    "cudaMemcpyAsync(q_r)") != MLA_OK)
        return MLA_ERR_CUDA;
    mla_status st;
    if ((st = mla_absorb_q(bufs->q_c, w_uk, bufs->q_abs, batch, s)) != MLA_OK) return st;
    if ((st = mla_decode_paged(&info, bufs->plan, bufs->q_abs, bufs->q_r, kv_dtype, kv_pool, kv_scale, kr_pool,
                               num_pool_pages, bufs->block_table, max_pages_per_seq, softmax_scale, bufs->workspace,
                               bufs->workspace_bytes, bufs->o_lat, bufs->lse, bufs->dev_error, s)) != MLA_OK)
        return st;
    if ((st = mla_combine_splits(&info, bufs->plan, bufs->workspace, bufs->workspace_bytes, bufs->o_lat, bufs->lse,
                                 s)) != MLA_OK)
        return st;
    if ((st = mla_out_proj(bufs->o_lat, w_uv, bufs->out, batch, s)) != MLA_OK) return st;
    return record_cuda(cudaMemcpyAsync(out_host, bufs->out, (size_t)batch * 128 * 128 * 2, cudaMemcpyDeviceToHost, s),
                       "cudaMemcpyAsync(out)");
}

// True when p is host memory the CUDA runtime has page-locked (cudaHostAlloc / cudaHostRegister).
bool pinned_host(const void* p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();  // the failed query leaves its error behind: clear it
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

// Loads the step's kernels (and sets their shared-memory limits) outside any stream capture, so
// that module loading never happens while a graph is being captured.
mla_status step_load_kernels(mla_kv_dtype kv_dtype)
{
    using AbsK = decltype(&mla::gemm::head_gemm_kernel<128, kAbsorbN, true, kAbsorbStages>);
    const AbsK absorb = mla::gemm::head_gemm_kernel<128, kAbsorbN, true, kAbsorbStages>;
    const AbsK outp = mla::gemm::head_gemm_kernel<512, kOutN, false, kOutStages>;
    if (!set_smem(absorb, AbsorbCfg::kSmemBytes) || !set_smem(outp, OutCfg::kSmemBytes)) return MLA_ERR_CUDA;
    const bool dec_ok = kv_dtype == MLA_KV_FP8_E4M3
                            ? set_smem(mla::decode_fp8::decode_fp8_kernel, mla::decode_fp8::kSmemBytes)
                            : set_smem(mla::decode::decode_bf16_kernel, mla::decode::kSmemBytes);
    if (!dec_ok) return MLA_ERR_CUDA;
    cudaFuncAttributes fa;
    return record_cuda(cudaFuncGetAttributes(&fa, mla::combine::combine_kernel), "cudaFuncGetAttributes(combine)");
}

}  // namespace

// The whole step from host memory: plan on the host, one asynchronous copy per input, the step's
// kernels (absorb, decode, merge, projection), the output copy back, one stream synchronisation.
extern "C" mla_status mla_decode_step_host(const int32_t* seq_lens, int32_t batch, int32_t num_sms,
                                           const mla_plan_options* opts, const void* q_c_host, const void* q_r_host,
                                           const int32_t* block_table_host, int32_t max_pages_per_seq,
                                           const void* w_uk, const void* w_uv, mla_kv_dtype kv_dtype,
                                           const void* kv_pool, const float* kv_scale, const void* kr_pool,
                                           int32_t num_pool_pages, float softmax_scale, const mla_step_buffers* bufs,
                                           void* out_host, mla_plan_info* info_out, void* stream)
{
    const mla::NvtxRange nvtx_range("mla_decode_step_host");
    mla_plan_info info{};
    mla_status st = step_prepare(seq_lens, batch, num_sms, opts, q_c_host, q_r_host, max_pages_per_seq, bufs,
                                 out_host, &info);
    if (st != MLA_OK && st != MLA_ERR_WORKSPACE) return st;
    if (info_out) *info_out = info;
    if (st != MLA_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = step_enqueue(info, true, q_c_host, q_r_host, block_table_host, max_pages_per_seq, w_uk, w_uv, kv_dtype,
                           kv_pool, kv_scale, kr_pool, num_pool_pages, softmax_scale, bufs, out_host, s)) != MLA_OK)
        return st;
    return record_cuda(cudaStreamSynchronize(s), "cudaStreamSynchronize");
}

// A captured step for fixed sequence lengths: the per-step copies and kernels as one executable
// CUDA graph (the plan was copied to the device once, when the graph was made).
struct mla_step_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int device = -1;
};

extern "C" mla_status mla_step_graph_create(const int32_t* seq_lens, int32_t batch, int32_t num_sms,
                                            const mla_plan_options* opts, const void* q_c_host, const void* q_r_host,
                                            const int32_t* block_table_host, int32_t max_pages_per_seq,
                                            const void* w_uk, const void* w_uv, mla_kv_dtype kv_dtype,
                                            const void* kv_pool, const float* kv_scale, const void* kr_pool,
                                            int32_t num_pool_pages, float softmax_scale,
                                            const mla_step_buffers* bufs, void* out_host, mla_plan_info* info_out,
                                            void* stream, mla_step_graph** graph_out)
{
    const mla::NvtxRange nvtx_range("mla_step_graph_create");
    if (!graph_out) return MLA_ERR_INVALID_ARG;
    *graph_out = nullptr;
    mla_plan_info info{};
    mla_status st = step_prepare(seq_lens, batch, num_sms, opts, q_c_host, q_r_host, max_pages_per_seq, bufs,
                                 out_host, &info);
    if (st != MLA_OK && st != MLA_ERR_WORKSPACE) return st;
    if (info_out) *info_out = info;
    if (st != MLA_OK) return st;
    // the graph's copies are DMA from page-locked host memory
    if (!pinned_host(q_c_host) || !pinned_host(q_r_host) || !pinned_host(out_host) ||
        (block_table_host && !pinned_host(block_table_host)))
        return MLA_ERR_INVALID_ARG;
    if ((st = step_load_kernels(kv_dtype)) != MLA_OK) return st;
    int dev = 0;
    if (record_cuda(cudaGetDevice(&dev), "cudaGetDevice") != MLA_OK) return MLA_ERR_CUDA;
    // the plan goes to the device once, outside the graph
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (record_cuda(cudaMemcpyAsync(bufs->plan, bufs->plan_host, (size_t)info.plan_bytes, cudaMemcpyHostToDevice, s),
                    "cudaMemcpyAsync(plan)") != MLA_OK ||
        record_cuda(cudaStreamSynchronize(s), "cudaStreamSynchronize") != MLA_OK)
        return MLA_ERR_CUDA;
    // capture on a stream of our own (the caller's may be the legacy default stream, which
    // cannot be captured)
    cudaStream_t cs = nullptr;
    if (record_cuda(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking), "cudaStreamCreateWithFlags") != MLA_OK)
        return MLA_ERR_CUDA;
    cudaGraph_t graph = nullptr;
    st = record_cuda(cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal), "cudaStreamBeginCapture");
    if (st == MLA_OK) {
        st = step_enqueue(info, false, q_c_host, q_r_host, block_table_host, max_pages_per_seq, w_uk, w_uv, kv_dtype,
                          kv_pool, kv_scale, kr_pool, num_pool_pages, softmax_scale, bufs, out_host, cs);
        const mla_status end = record_cuda(cudaStreamEndCapture(cs, &graph), "cudaStreamEndCapture");
        if (st == MLA_OK) st = end;
    }
    cudaStreamDestroy(cs);
    cudaGraphExec_t exec = nullptr;
    if (st == MLA_OK)
        st = record_cuda(cudaGraphInstantiate(&exec, graph, 0), "cudaGraphInstantiate");
    if (st != MLA_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
    }
    mla_step_graph* g = new mla_step_graph;
    g->graph = graph;
    g->exec = exec;
    g->device = dev;
    *graph_out = g;
    return MLA_OK;
}

extern "C" mla_status mla_step_graph_run(mla_step_graph* graph, int32_t wait, void* stream)
{
    const mla::NvtxRange nvtx_range("mla_step_graph_run");
    if (!graph || !graph->exec) return MLA_ERR_INVALID_ARG;
    int dev = -1;
    if (record_cuda(cudaGetDevice(&dev), "cudaGetDevice") != MLA_OK) return MLA_ERR_CUDA;
    if (dev != graph->device) return MLA_ERR_INVALID_ARG;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (record_cuda(cudaGraphLaunch(graph->exec, s), "cudaGraphLaunch") != MLA_OK) return MLA_ERR_CUDA;
    if (!wait) return MLA_OK;
    return record_cuda(cudaStreamSynchronize(s), "cudaStreamSynchronize");
}

extern "C" mla_status mla_step_graph_destroy(mla_step_graph* graph)
{
    if (!graph) return MLA_OK;
    mla_status st = MLA_OK;
    if (graph->exec && cudaGraphExecDestroy(graph->exec) != cudaSuccess) st = MLA_ERR_CUDA;
    if (graph->graph && cudaGraphDestroy(graph->graph) != cudaSuccess) st = MLA_ERR_CUDA;
    delete graph;
    return st;
}
