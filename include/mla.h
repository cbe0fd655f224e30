/*
 * mla.h -- C ABI of libmla_gb300.so: Multi-Head Latent Attention decode over a paged latent
 * KV cache with matrix absorption, for NVIDIA GB300 (sm_103a).
 *
 * The operations follow "撕開 DeepSeek MLA 源碼：C++ 與 TensorRT-LLM 算子設計優化全景"
 * (jh158.com/news/60867, "P1" below) and the split-KV decode of the Kimi K3 decode
 * time-share page (jinnpan.com/sources/kimi-k3-kda-time-share.html, "P3" below).
 *
 * Fixed geometry (P1 section 1 and the mla_config.h block of section 3): 128 heads, content
 * head dim d_hc = 128, latent dim d_c = 512, decoupled RoPE dim d_R = 64, so one cache row is
 * 576 elements; pages hold 64 tokens (P1 section 3, page_size 64).
 *
 * Conventions shared by every entry point
 *   - Pointers marked "device" are CUDA device pointers; "host" pointers are ordinary memory.
 *   - bf16 tensors are passed as void* and are contiguous, row-major, in the shapes stated.
 *   - The caller allocates and owns every buffer, workspaces included.  The library allocates
 *     no device memory for data; the one exception to "no allocation" is
 *     mla_step_graph_create, whose handle holds a host object and a CUDA graph until
 *     mla_step_graph_destroy.  Its only global mutable state is the fixed device array behind
 *     mla_decode_paged_static_ws (and that call's per-device address cache); every other call
 *     is safe from several host threads.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only enqueue work and
 *     return; results are ready when the stream reaches them.  The exceptions, which wait for
 *     the stream: mla_decode_step_host, mla_step_graph_create and mla_step_graph_run with
 *     `wait` set (and mla_read_device_error).
 *   - Arguments, shapes, alignment and workspace sizes are checked on the host before any
 *     launch; a failed check returns an error and enqueues nothing.  A failed launch returns
 *     MLA_ERR_CUDA.  Problems only the GPU can see (a block-table entry outside the pool, a
 *     wait that timed out) set bits in the caller's device word `dev_error`; the kernel then
 *     ends early and never traps.  Read it with mla_read_device_error().
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_NUM_HEADS 128
#define MLA_HEAD_DIM 128   /* d_hc */
#define MLA_LATENT_DIM 512 /* d_c  */
#define MLA_ROPE_DIM 64    /* d_R  */
#define MLA_ROW_DIM 576    /* d_c + d_R */
#define MLA_PAGE_SIZE 64

typedef enum mla_status {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, bad enum, inconsistent plan */
    MLA_ERR_ALIGNMENT = 2,    /* a pointer is not 16-byte aligned (TMA and vector loads need it) */
    MLA_ERR_UNSUPPORTED = 3,  /* a size the kernels do not handle (e.g. plan too large) */
    MLA_ERR_WORKSPACE = 4,    /* a caller buffer is smaller than required */
    MLA_ERR_CUDA = 5,         /* a CUDA runtime/driver call or a launch failed */
    MLA_ERR_DEVICE_FAULT = 6  /* mla_read_device_error found a non-zero device error word */
} mla_status;

typedef enum mla_kv_dtype {
    MLA_KV_BF16 = 0,     /* one bf16 pool [pages][64][576]: c_KV (512) then k_R (64) per row */
    MLA_KV_FP8_E4M3 = 1, /* c_KV as e4m3 codes [pages][64][512], fp32 scale [pages][64], k_R bf16 [pages][64][64] */
    MLA_KV_NVFP4 = 2     /* c_KV as NVFP4 rows [pages][64][288] (256 bytes of e2m1 codes, two per byte with
                            value 2j in the low nibble of byte j, then 32 e4m3 scales, one per 16 values),
                            fp32 scale [pages][64], k_R bf16 [pages][64][64].  Written by mla_append_kv,
                            read by mla_gather_kv; the decode calls return MLA_ERR_UNSUPPORTED for it */
} mla_kv_dtype;

/* Bits of the device error word. */
#define MLA_DEVERR_BAD_PAGE 1u    /* a block-table entry outside [0, num_pool_pages): read as zeros */
#define MLA_DEVERR_TIMEOUT 2u     /* a bounded wait ran out; the kernel stopped early */
#define MLA_DEVERR_SMEM_ALIGN 4u  /* shared memory was not 1024-byte aligned; nothing computed */
#define MLA_DEVERR_BAD_PLAN 8u    /* the device plan image failed its header check */
#define MLA_DEVERR_BAD_SLOT 16u   /* mla_append_kv: a slot at or past num_pool_pages * 64; that token skipped */

MLA_API const char* mla_status_string(mla_status status);

/* Text of the last CUDA runtime failure (MLA_ERR_CUDA) seen by the calling host thread. */
MLA_API const char* mla_last_error_string(void);

/* ---------------------------------------------------------------- a1: split planning (host only)
 *
 * P3 ("Inside the blocks") splits the decode KV scan over many workgroups and merges the
 * pieces in a separate KV-split reduction.  Here each sequence's pages are cut into
 * contiguous work items so that every CTA pair (two SMs) streams about the same number of
 * pages; sequences cut into several items get a log-sum-exp merge (mla_combine_splits).
 */
typedef struct mla_plan_options {
    int32_t min_pages_per_split; /* 0 = default 8: no item boundary closer than this to a sequence edge */
    int32_t max_clusters;        /* 0 = num_sms / 2; otherwise at most this many CTA pairs */
    int64_t wait_timeout_ns;     /* 0 = default 2e9: bound on every device-side wait */
    int32_t item_cost_pages;     /* balance pages plus this many pages' worth of cost for each item
                                    of a CTA pair after its first (a second item reloads the query
                                    and writes an output); 0 = the default charge of 7 pages,
                                    < 0 = no charge: equal page runs */
    int32_t queries_per_seq;     /* query tokens per sequence, q (0 or 1 = ordinary decode; at most
                                    MLA_MAX_QUERIES_PER_SEQ).  With q > 1 (several new tokens per
                                    sequence decoded at once: speculative drafts, a short chunk)
                                    the plan covers batch * q query rows, row b * q + t being token
                                    t of sequence b, which sees the first S_b - q + 1 + t cached
                                    tokens (causal among the new tokens, which the cache already
                                    holds; S_b >= q).  Every per-row tensor of the calls below
                                    (q_c, q_R, q_abs, o_lat, lse, out) then has batch * q rows of
                                    128 heads; the block table keeps one row per sequence.  Each
                                    query row scans its pages on its own (no shared scan). */
} mla_plan_options;
#define MLA_MAX_QUERIES_PER_SEQ 4096

typedef struct mla_plan_info {
    int32_t batch;           /* query rows: sequences x queries_per_seq */
    int32_t num_clusters;    /* CTA pairs the decode launch uses (grid = 2 * num_clusters CTAs) */
    int32_t num_items;       /* work items (sequence, page range) */
    int32_t num_partials;    /* items that write a split partial into the workspace */
    int32_t num_combine;     /* sequences with more than one item */
    int32_t max_splits;      /* most items any one sequence has */
    int32_t total_pages;     /* sum over query rows of ceil(visible length / 64) */
    int32_t queries_per_seq; /* q of the plan (1 for ordinary decode) */
    int64_t plan_bytes;      /* bytes of the plan image written to plan_host */
    int64_t workspace_bytes; /* bytes mla_decode_paged needs in `workspace` */
    int64_t wait_timeout_ns;
} mla_plan_info;

/* Upper bound on the plan image size for `batch` query rows (sequences x queries_per_seq) on
 * `num_sms` SMs. */
MLA_API size_t mla_plan_bytes_max(int32_t batch, int32_t num_sms);

/* Builds the plan image in host memory.
 *   seq_lens   host int32 [batch], each >= max(1, queries_per_seq) (the context length S_b of
 *              sequence b, new tokens included)
 *   num_sms    SMs of the device the decode runs on (>= 2)
 *   opts       may be NULL (defaults)
 *   plan_host  host buffer of plan_capacity bytes (>= mla_plan_bytes_max(batch * q, num_sms)); the caller copies
 *              info->plan_bytes of it to device memory (16-byte aligned) for the calls below.
 * Pure host code: needs no GPU. */
MLA_API mla_status mla_plan_splits(const int32_t* seq_lens, int32_t batch, int32_t num_sms,
                           const mla_plan_options* opts, void* plan_host, size_t plan_capacity,
                           mla_plan_info* info);

/* ---------------------------------------------------------------- a2: absorb W_UK into the query
 *
 * P1 section 4, path B: q_abs[b,h,c] = sum_d q_c[b,h,d] * W_UK[h,d,c].
 *   q_c   device bf16 [batch][128][128]
 *   w_uk  device bf16 [128][128][512]   (heads, d_hc, d_c)
 *   q_abs device bf16 [batch][128][512] (fp32 accumulation, rounded once to bf16)
 * All three 16-byte aligned.  Tensor cores (tcgen05), one 128-row batch tile per CTA. */
MLA_API mla_status mla_absorb_q(const void* q_c, const void* w_uk, void* q_abs, int32_t batch, void* stream);

/* ---------------------------------------------------------------- a3-a8: paged decode
 *
 * For every work item of the plan: gather its pages through the block table, score all 128
 * heads against each cached row, s = (q_abs . c_KV + q_R . k_R) * softmax_scale (P1 section 4),
 * run an online softmax and accumulate P . c_KV in the 512-d latent space.
 *   plan_dev        device copy of the plan image (16-byte aligned); info = its host header
 *   q_abs           device bf16 [batch][128][512]   (from mla_absorb_q)
 *   q_r             device bf16 [batch][128][64]    (already rotated)
 *   kv_dtype        MLA_KV_BF16: kv_pool = bf16 [num_pool_pages][64][576]; kv_scale, kr_pool NULL
 *                   MLA_KV_FP8_E4M3: kv_pool = e4m3 codes [num_pool_pages][64][512],
 *                   kv_scale = fp32 [num_pool_pages][64] (the stored value times the scale is
 *                   the latent), kr_pool = bf16 [num_pool_pages][64][64]; kv_pool and
 *                   kr_pool 16-byte aligned, kv_scale 4-byte aligned; scales finite and >= 0
 *                   (absmax / 448 per token; 0 marks an all-zero latent row).  The codes feed e4m3
 *                   tensor-core MMAs as loaded; q_abs and P enter them as e4m3 pairs (hi +
 *                   lo, about 2^-8 relative), the scales are applied to the scores and to P
 *                   per token, and k_R / scale is formed in bf16 for the RoPE MMA.
 *   block_table     device int32 [batch / q][max_pages_per_seq] (q = info->queries_per_seq: one
 *                   row per sequence, shared by its q query rows); entry p of row b is the physical
 *                   page of tokens 64p..64p+63 of sequence b.  Only the first ceil(S_b/64)
 *                   entries of a row are read, and never an entry at or past
 *                   max_pages_per_seq: a sequence whose pages do not fit in its row (this call
 *                   has no host copy of the lengths to check) reads its missing pages as zeros
 *                   and sets MLA_DEVERR_BAD_PAGE, like an entry outside the pool.
 *   softmax_scale   1/sqrt(d_hc + d_R) for the pages' model
 *   workspace       device buffer of info->workspace_bytes (split partials), 16-byte aligned;
 *                   may be NULL when info->workspace_bytes == 0
 *   o_lat           device bf16 [batch][128][512]: normalised latent output of sequences that
 *                   have a single item (the others are written by mla_combine_splits)
 *   lse             device fp32 [batch][128]: natural-log sum of exp(scores), same rule
 *   dev_error       device uint32 error word (MLA_DEVERR_* bits are OR-ed in), 4-byte aligned
 * Slots past S_b in a sequence's last page may hold anything (NaN included): they are masked. */
MLA_API mla_status mla_decode_paged(const mla_plan_info* info, const void* plan_dev,
                            const void* q_abs, const void* q_r,
                            mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale,
                            const void* kr_pool, int32_t num_pool_pages,
                            const int32_t* block_table, int32_t max_pages_per_seq,
                            float softmax_scale, void* workspace, size_t workspace_bytes,
                            void* o_lat, float* lse, uint32_t* dev_error, void* stream);

/* ---------------------------------------------------------------- a2 + a3-a8 in one kernel
 *
 * The absorb (P1 section 4, path B: q_abs = q_c W_UK per head) as the prologue of the paged
 * decode: every CTA of the decode grid first forms q_abs for one head and one tile of 128
 * sequences on the tensor cores (the grid gets extra CTA pairs, which do only that, when the plan
 * has fewer pairs than 64 per 128-sequence tile), writes the rows to `q_abs` and publishes the
 * job in absorb_sync; the score CTAs wait for all jobs before their first query.  One launch
 * instead of two, and the absorb no longer sits in front of the decode as a kernel of its own.
 *   q_c, w_uk     as mla_absorb_q (batch = info->batch)
 *   q_abs         device bf16 [batch][128][512], written (the same values mla_absorb_q writes)
 *   absorb_sync   device uint32[2], 8-byte aligned, zero before the first call; every call that
 *                 sets no MLA_DEVERR_* bit leaves it zero again.  After a call that did set one,
 *                 zero it before the next call.  Calls that may overlap on the GPU need one each.
 *   the rest      as mla_decode_paged.
 * It is an ordinary launch: it starts after the stream's previous work has finished (a
 * programmatic early start could overlap a previous step's merge, which still reads o_lat).
 * With the e4m3 cache (MLA_KV_FP8_E4M3) the absorb runs as its own kernel (mla_absorb_q) and the
 * decode follows it; absorb_sync is then not touched. */
MLA_API mla_status mla_absorb_decode_paged(const mla_plan_info* info, const void* plan_dev, const void* q_c,
                                           const void* w_uk, void* q_abs, uint32_t* absorb_sync, const void* q_r,
                                           mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale,
                                           const void* kr_pool, int32_t num_pool_pages, const int32_t* block_table,
                                           int32_t max_pages_per_seq, float softmax_scale, void* workspace,
                                           size_t workspace_bytes, void* o_lat, float* lse, uint32_t* dev_error,
                                           void* stream);

/* ---------------------------------------------------------------- a9: merge split partials
 *
 * P3's KV-split reduction: for each sequence with several items,
 *   lse = log sum_j exp(lse_j),  o_lat = sum_j exp(lse_j - lse) o_j,
 * reading the partials mla_decode_paged left in `workspace`.  Writes o_lat (bf16) and lse
 * (fp32) for those sequences only.  A plan with num_combine == 0 enqueues nothing. */
MLA_API mla_status mla_combine_splits(const mla_plan_info* info, const void* plan_dev, const void* workspace,
                              size_t workspace_bytes, void* o_lat, float* lse, void* stream);

/* ---------------------------------------------------------------- a10: W_UV projection
 *
 * out[b,h,d] = sum_c o_lat[b,h,c] * W_UV[h,d,c]   (W_UV laid out like W_UK: heads, d_hc, d_c)
 *   o_lat device bf16 [batch][128][512], w_uv device bf16 [128][128][512],
 *   out   device bf16 [batch][128][128].  Tensor cores (tcgen05), fp32 accumulation. */
MLA_API mla_status mla_out_proj(const void* o_lat, const void* w_uv, void* out, int32_t batch, void* stream);

/* ---------------------------------------------------------------- a9 + a10 in one kernel
 *
 * The step's tail fused (P3 "Inside the blocks": the KV-split reduction; P1 section 1: W_UV
 * applied after the attention): for every sequence, the log-sum-exp merge of its split partials
 * (as mla_combine_splits) and out = W_UV o_lat (as mla_out_proj), in one launch.  Per head, the
 * merged rows go straight into the projection's operand in shared memory; W_UV streams in while
 * the decode kernel before it finishes (programmatic dependent launch).
 *   info, plan_dev, workspace   the plan and the split partials mla_decode_paged wrote
 *                               (workspace may be NULL when info->num_combine == 0)
 *   o_lat, lse                  read for single-item sequences; for split sequences the merged
 *                               o_lat (bf16) and lse (fp32) are written, as mla_combine_splits does
 *   w_uv, out                   as mla_out_proj, with batch = info->batch
 *   dev_error                   device uint32 word for MLA_DEVERR_* bits (a bounded wait that ran
 *                               out), 4-byte aligned, or NULL
 * The merged rows, and so `out`, are bit-identical to mla_combine_splits + mla_out_proj. */
MLA_API mla_status mla_merge_out_proj(const mla_plan_info* info, const void* plan_dev, const void* workspace,
                                      size_t workspace_bytes, void* o_lat, float* lse, const void* w_uv, void* out,
                                      uint32_t* dev_error, void* stream);

/* ---------------------------------------------------------------- cache append (the write side)
 *
 * P1 section 1: each token stores, once, its 512-d latent c_KV and its 64-d RoPE key k_R (576
 * elements); every later decode step reads that row.  P1 section 3 pages the cache in blocks of
 * 64 tokens.  This call writes num_tokens new rows into the pool: token i goes to slot
 * slots[i] = physical page * 64 + row within the page (the caller derives it from its block
 * table: page block_table[b][t / 64], row t % 64 for position t of sequence b).
 *   c_kv   device bf16 [num_tokens][512], k_r device bf16 [num_tokens][64] (already rotated)
 *   slots  device int32 [num_tokens]; a negative slot skips the token (padding); a slot at or
 *          past num_pool_pages * 64 skips it and sets MLA_DEVERR_BAD_SLOT in *dev_error
 *   bf16 cache: kv_pool [pages][64][576] receives c_KV then k_R; kv_scale and kr_pool are
 *          ignored.
 *   FP8 cache (MLA_KV_FP8_E4M3): per token, over the 512 latent values only,
 *          sigma = max_i |c_i| / 448 in fp32 (1 when the row is all zeros), and code_i = the
 *          e4m3 value nearest c_i / sigma (fp32 quotient, ties to the even code); kv_pool
 *          [pages][64][512] receives the codes, kv_scale [pages][64] sigma, kr_pool
 *          [pages][64][64] k_R unchanged.  Rows must be finite.
 * The result is exact: byte for byte what the stated rule gives.  Two tokens with the same slot
 * race (one of them wins).  c_kv, k_r, kv_pool and kr_pool 16-byte aligned, slots, kv_scale
 * and dev_error 4-byte aligned.  num_tokens == 0 enqueues nothing.  One warp per token, plain
 * vector loads and stores (a few hundred bytes per token: launch-bound at decode batch sizes). */
MLA_API mla_status mla_append_kv(int32_t num_tokens, const void* c_kv, const void* k_r, const int32_t* slots,
                                 mla_kv_dtype kv_dtype, int32_t num_pool_pages, void* kv_pool, float* kv_scale,
                                 void* kr_pool, uint32_t* dev_error, void* stream);

/* ---------------------------------------------------------------- gather: paged cache -> contiguous rows
 *
 * P1's "NVFP4 quantized gather" (table of contents; section 5 on reading packed fp4 pages with
 * 16-byte vector loads): every sequence's cache rows, in logical order, out of the paged pool into
 * one contiguous bf16 array, dequantised on the way, for consumers that want whole rows.
 *   kv_dtype, kv_pool, kv_scale, kr_pool, num_pool_pages   the cache, as for mla_decode_paged
 *                     (kv_pool 16-byte aligned), or MLA_KV_NVFP4 as for mla_append_kv
 *   block_table       device int32 [batch / info->queries_per_seq][max_pages_per_seq]
 *   seq_lens          device int32 [batch], each <= max_pages_per_seq * 64
 *   cu_seqlens        device int32 [batch + 1]: row offsets, cu_seqlens[b + 1] = cu_seqlens[b] + seq_lens[b]
 *   out               device bf16 [cu_seqlens[batch]][576], 16-byte aligned: c_KV then k_R per row
 *   dev_error         device uint32 word: MLA_DEVERR_BAD_PAGE for an entry outside the pool
 *                     (that row is not written)
 * bf16 cache: the stored bits.  FP8 cache: each latent value is float(code) * sigma in fp32 (one
 * rounding), then rounded to bf16 (nearest, ties to even).  NVFP4 cache: float(e2m1 code) *
 * float(e4m3 block scale) (exact) * sigma in fp32 (one rounding), then to bf16.  k_R is copied.
 * One warp per token; a streaming copy (at most 1152 bytes written per token). */
MLA_API mla_status mla_gather_kv(mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale,
                                 const void* kr_pool, int32_t num_pool_pages, const int32_t* block_table,
                                 int32_t max_pages_per_seq, const int32_t* seq_lens, const int32_t* cu_seqlens,
                                 int32_t batch, void* out, uint32_t* dev_error, void* stream);

/* ---------------------------------------------------------------- decode + merge, no allocation
 *
 * The pages describe no counterpart of this call: it is a convenience of this library.
 * mla_decode_paged followed by mla_combine_splits, with the split-partial workspace taken from
 * a fixed device array inside the library instead of from the caller.  The call allocates no
 * device memory itself.  It is meant for callers that cannot allocate at the point of the call:
 * code running inside a custom allocator's own callbacks (allocating there would re-enter the
 * allocator), runtimes that reserve all device memory up front and forbid later allocation,
 * and embedders with no caching allocator to take a workspace from.
 *
 * Arguments, layouts and results are those of mla_decode_paged (o_lat and lse end up final for
 * every sequence, as after mla_combine_splits).
 * Limit: the array holds MLA_STATIC_WS_MAX_PARTIALS split partials (MLA_STATIC_WS_BYTES bytes,
 * about 33.6 MB, per device); a plan with more partials is rejected with MLA_ERR_WORKSPACE and
 * the reason in mla_last_error_string().  Plan with fewer clusters, or use mla_decode_paged.
 * Nothing in the array needs to start at zero: each call's decode launch writes every partial
 * that its merge launch reads.
 * Set-up: the first call on each device (with that device current) looks up the array's device
 * address and, through it, loads the library module that holds the array; make that first call
 * before any stream capture.  The address is cached per device for the life of the process, so
 * the cache must not outlive the device's primary context: after cudaDeviceReset (or any
 * teardown of the primary context) do not call this entry point again in that process.
 * Memory: the array costs device memory only on devices where the module is loaded.  Under the
 * CUDA runtime's default lazy module loading that happens on the first call; with
 * CUDA_MODULE_LOADING=EAGER every device that creates a context holds the array from then on.
 * One array per device: calls whose kernels may overlap (different streams, or several host
 * threads on one device) race on it and corrupt each other's results.  Calls in order on one
 * stream are safe. */
#define MLA_STATIC_WS_MAX_PARTIALS 128
#define MLA_STATIC_WS_BYTES ((size_t)MLA_STATIC_WS_MAX_PARTIALS * (128u * 512u * 4u + 128u * 4u))
MLA_API mla_status mla_decode_paged_static_ws(const mla_plan_info* info, const void* plan_dev,
                            const void* q_abs, const void* q_r,
                            mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale,
                            const void* kr_pool, int32_t num_pool_pages,
                            const int32_t* block_table, int32_t max_pages_per_seq,
                            float softmax_scale, void* o_lat, float* lse, uint32_t* dev_error,
                            void* stream);

/* ---- prefill chunk, decompressed form -------------------------------------------------------
 * P1 section 4 gives two forms of the same attention: path A decompresses per-head keys and
 * values (k_h = W_UK[h] c, v_h = W_UV[h] c) and attends with head dim 128 + 64; path B absorbs
 * W_UK into the query (the decode calls above).  Section 3's mla_config.h sets
 * kPrefillThresh = 256 and section 6 measures the switch: chunks of at least 256 new tokens
 * run path A, shorter ones path B (the decode with opts->queries_per_seq = chunk length).
 * This call runs path A for the last chunk_len tokens of one sequence of seq_len tokens whose
 * cache rows (the chunk's included) are already in the pool: query t (position
 * seq_len - chunk_len + t) attends causally to positions 0 .. seq_len - chunk_len + t, and
 *   out[t,h,:] = sum_j softmax_j((q_c[t,h] . k_h[j] + q_R[t,h] . k_R[j]) * softmax_scale) v_h[j].
 * Steps, all on `stream`: the sequence's rows gathered into bf16 (dequantised for FP8 and
 * NVFP4 caches, as mla_gather_kv), k_h and v_h for all heads (tcgen05 GEMMs), then a causal
 * attention kernel (2 x 128 queries x 1 head per CTA sharing 128-key tiles, online softmax).
 *   kv_dtype, kv_pool, kv_scale, kr_pool, num_pool_pages   the cache, as mla_gather_kv
 *   block_table_row  device int32 [max_pages]: the sequence's pages (ceil(seq_len/64) <= max_pages)
 *   q_c, q_r         device bf16 [chunk_len][128][128] / [chunk_len][128][64]
 *   w_uk, w_uv       device bf16 [128][128][512]
 *   workspace        device, >= mla_prefill_workspace_bytes(seq_len), 16-byte aligned: the
 *                    gathered rows [seq_len][576], k and v [128 heads][seq_len][128]
 *   out              device bf16 [chunk_len][128][128]
 * 1 <= chunk_len <= seq_len <= 65535 * 128.  Device-side problems (a page outside the pool, a
 * wait that ran out) set bits in dev_error. */
MLA_API size_t mla_prefill_workspace_bytes(int32_t seq_len);
MLA_API mla_status mla_prefill_decompressed(mla_kv_dtype kv_dtype, const void* kv_pool, const float* kv_scale,
                                            const void* kr_pool, int32_t num_pool_pages,
                                            const int32_t* block_table_row, int32_t max_pages, int32_t seq_len,
                                            int32_t chunk_len, const void* q_c, const void* q_r, const void* w_uk,
                                            const void* w_uv, float softmax_scale, void* workspace,
                                            size_t workspace_bytes, void* out, uint32_t* dev_error, void* stream);

/* ---- the whole step from host memory in one call ------------------------------------------
 * For callers whose queries, block table and lengths live in host memory: plans the step for
 * `seq_lens` on the host (as mla_plan_splits), copies the plan, the block table (when
 * block_table_host is not NULL) and the queries to the device (one cudaMemcpyAsync each, from
 * pinned memory for asynchronous DMA), runs absorb, decode, merge and out-proj on `stream`,
 * copies `out` back to out_host and waits for the stream.  One library call instead of a dozen
 * binding-level operations; it computes exactly what the four calls above compute.
 *   `batch` counts sequences; with opts->queries_per_seq = q > 1 every per-row tensor has
 *   R = batch * q query rows (R = batch otherwise).
 *   bufs              the device buffers, owned by the caller and sized for R rows:
 *                       q_c, q_r, q_abs, o_lat, lse, out (as above), dev_error,
 *                       block_table  int32 [batch][max_pages_per_seq] (written when a host table
 *                                    is given, else read as it stands),
 *                       plan         >= mla_plan_bytes_max(R, num_sms) bytes, 16-byte aligned,
 *                       workspace    workspace_bytes >= the plan's workspace_bytes (else
 *                                    MLA_ERR_WORKSPACE before anything is copied or launched);
 *                     and plan_host: pinned host memory of plan_capacity >= mla_plan_bytes_max(R, num_sms).
 *   q_c_host, q_r_host  host bf16 [R][128][128] / [R][128][64]
 *   out_host          host bf16 [R][128][128], receives out
 *   info_out          may be NULL; receives the plan header
 * A sequence whose ceil(S_b/64) pages exceed max_pages_per_seq is rejected with
 * MLA_ERR_INVALID_ARG before anything is copied or launched.
 * Device-side errors land in bufs->dev_error as for mla_decode_paged (read it afterwards). */
typedef struct mla_step_buffers {
    void* q_c;
    void* q_r;
    void* q_abs;
    int32_t* block_table;
    void* plan;
    void* workspace;
    size_t workspace_bytes;
    void* o_lat;
    float* lse;
    void* out;
    uint32_t* dev_error;
    void* plan_host;
    size_t plan_capacity;
} mla_step_buffers;

MLA_API mla_status mla_decode_step_host(const int32_t* seq_lens, int32_t batch, int32_t num_sms,
                                        const mla_plan_options* opts, const void* q_c_host, const void* q_r_host,
                                        const int32_t* block_table_host, int32_t max_pages_per_seq,
                                        const void* w_uk, const void* w_uv, mla_kv_dtype kv_dtype,
                                        const void* kv_pool, const float* kv_scale, const void* kr_pool,
                                        int32_t num_pool_pages, float softmax_scale, const mla_step_buffers* bufs,
                                        void* out_host, mla_plan_info* info_out, void* stream);

/* ---- the step from host memory as a captured CUDA graph ------------------------------------
 * For a run of steps with unchanged sequence lengths (and the same host and device buffers):
 * mla_step_graph_create does what mla_decode_step_host does up to the launches -- the same
 * arguments, checks and plan -- then copies the plan to the device once (on `stream`, waiting
 * for it) and captures, on a stream of its own, the per-step work as one CUDA graph: the block
 * table (when block_table_host is not NULL) and query copies to the device, absorb, decode,
 * merge, out-proj and the copy of `out` back to out_host.  Each mla_step_graph_run launches that
 * graph on `stream` (any stream of the device the graph was made on) and, when `wait` is
 * non-zero, waits for it; every launch reads the host buffers as they are at that time, so the
 * caller writes the next step's queries (and table) into the same buffers between runs.
 * Lengths or buffers that change need a new graph: the plan, the grid sizes and every pointer
 * are fixed in it.
 *   q_c_host, q_r_host, out_host, block_table_host: page-locked host memory (cudaHostAlloc or
 *     cudaHostRegister), else MLA_ERR_INVALID_ARG before anything is copied or captured.
 *   graph_out: receives the handle (NULL on failure); the handle owns host memory and the
 *     graph, released by mla_step_graph_destroy (NULL is accepted and ignored).
 * Results are bit-identical to mla_decode_step_host with the same inputs.  Launches of one graph
 * on different streams, or of two graphs sharing buffers, may overlap and race on the buffers:
 * order them on one stream.  Device-side errors land in bufs->dev_error. */
typedef struct mla_step_graph mla_step_graph;
MLA_API mla_status mla_step_graph_create(const int32_t* seq_lens, int32_t batch, int32_t num_sms,
                                         const mla_plan_options* opts, const void* q_c_host, const void* q_r_host,
                                         const int32_t* block_table_host, int32_t max_pages_per_seq,
                                         const void* w_uk, const void* w_uv, mla_kv_dtype kv_dtype,
                                         const void* kv_pool, const float* kv_scale, const void* kr_pool,
                                         int32_t num_pool_pages, float softmax_scale, const mla_step_buffers* bufs,
                                         void* out_host, mla_plan_info* info_out, void* stream,
                                         mla_step_graph** graph_out);
MLA_API mla_status mla_step_graph_run(mla_step_graph* graph, int32_t wait, void* stream);
MLA_API mla_status mla_step_graph_destroy(mla_step_graph* graph);

/* ---------------------------------------------------------------- device error word
 *
 * Waits for `stream`, copies the device word to *host_bits (may be NULL) and returns
 * MLA_ERR_DEVICE_FAULT if any bit is set, MLA_OK otherwise.  Does not clear the word. */
MLA_API mla_status mla_read_device_error(const uint32_t* dev_error, uint32_t* host_bits, void* stream);

/* Test hook for the bounded waits: launches one CTA that waits on a barrier nothing will
 * ever complete, giving up after timeout_ns (1 ms .. 10 s).  The kernel must set
 * MLA_DEVERR_TIMEOUT in *dev_error and return; the context stays usable. */
MLA_API mla_status mla_debug_wait_timeout(uint32_t* dev_error, int64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MLA_GB300_H */
