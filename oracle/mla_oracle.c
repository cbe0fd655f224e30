/*
 * mla_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow CPU statement of Multi-Head Latent Attention decode over a paged latent
 * cache. It exists only to check the CUDA library: the tests, the smoke check and the
 * bench's CPU-baseline leg call it; nothing in the library links or calls it, and it
 * shares no source with the CUDA code.
 *
 * What it follows ("撕開 DeepSeek MLA 源碼：C++ 與 TensorRT-LLM 算子設計優化全景",
 * jh158.com/news/60867):
 *   section 1   - one cache row per token: a 512-d latent c_KV followed by a 64-d decoupled
 *                 RoPE key k_R, shared by all 128 heads (576 elements, 1.125 KB in bf16);
 *   section 3   - mla_config.h: 128 heads, d_hc = 128, d_c = 512, d_R = 64; page_size 64;
 *   section 4   - verify_absorption(): the naive path decompresses k_h = W_UK[h] c with
 *                 W_UK laid out (heads, d_hc, d_c); its score is
 *                 (q_c . k_h + q_R . k_R) / sqrt(d_hc + d_R).  The absorbed path forms
 *                 q_abs[h] = sum_d q_c[h,d] W_UK[h,d,:] and scores (q_abs . c + q_R . k_R)
 *                 with the same scale.
 * The value side (v_h = W_UV[h] c, softmax-weighted sum) is the standard attention
 * definition; W_UV is read with the same (heads, d_hc, d_c) layout as W_UK because the page
 * prints only W_UK's.  Decode with split-KV (a "stage 1" KV scan and a "stage 2" KV-split
 * reduction) is named by the Kimi K3 decode time-share page (jinnpan.com/sources/
 * kimi-k3-kda-time-share.html, "Inside the blocks" table); its log-sum-exp merge is the
 * textbook identity for partial softmax sums.
 *
 * Arithmetic: bf16 / e4m3 / fp32 inputs are widened exactly to double and every product
 * and sum is taken in double.  Loops follow the definitions with no blocking or reordering
 * beyond them.  OpenMP only spreads independent (sequence, head) rows over cores.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { NH = 128, DHC = 128, DC = 512, DR = 64, DROW = 576, PG = 64 };
/* NVFP4 row of one token: 256 bytes of packed e2m1 codes, then 32 e4m3 block scales */
enum { NV_CODES = DC / 2, NV_BLOCKS = DC / 16, NV_ROW = NV_CODES + NV_BLOCKS };

/* ------------------------------------------------------------------ element decoding */

/* bf16 is the top half of an IEEE binary32. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 (the "fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, and S.1111.111 is NaN.  Exponent field 0 is subnormal:
 * value = m/8 * 2^-6.  Otherwise value = (1 + m/8) * 2^(e-7). */
double oracle_e4m3_value(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

void oracle_e4m3_decode(const uint8_t* codes, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_value(codes[i]);
}

/* e2m1 (the element type of NVFP4): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit, no
 * infinities or NaN.  Exponent field 0 is subnormal (0 or 0.5); field e > 0 is (1 + m/2) 2^(e-1):
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Codes are the low 4 bits. */
double oracle_e2m1_value(uint8_t code)
{
    const int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ the paged cache */

typedef struct {
    int kv_fp8;               /* 0: bf16 rows [N][64][576]; 1: e4m3 c_KV + fp32 scale + bf16 k_R;
                                 2: NVFP4 c_KV (e2m1 codes, e4m3 scale per 16 values, fp32 scale per
                                 token) + bf16 k_R */
    int num_pages;
    const uint16_t* pool;     /* bf16 [N][64][576] */
    const uint8_t* c8;        /* e4m3 [N][64][512]; NVFP4: rows [N][64][288], 256 bytes of packed e2m1
                                 codes (value 2j in the low nibble of byte j, 2j + 1 in the high
                                 nibble) then 32 e4m3 scales, one per 16 latent values */
    const float* scale;       /* fp32 [N][64] */
    const uint16_t* kr;       /* bf16 [N][64][64] */
} cache_view;

/* Token t of a sequence lives in slot t % 64 of physical page block_table_row[t / 64].
 * Writes its 512 latent values and 64 RoPE-key values.  Returns -1 for an out-of-range page. */
static int gather_row(const cache_view* cv, const int32_t* bt_row, int64_t t, double* ckv, double* kr)
{
    int64_t page = bt_row[t / PG], slot = t % PG;
    if (page < 0 || page >= cv->num_pages) return -1;
    int64_t tok = page * PG + slot;
    if (!cv->kv_fp8) {
        const uint16_t* row = cv->pool + tok * DROW;
        for (int i = 0; i < DC; ++i) ckv[i] = bf16_value(row[i]);
        for (int i = 0; i < DR; ++i) kr[i] = bf16_value(row[DC + i]);
    } else if (cv->kv_fp8 == 1) {
        /* dequantised latent: the stored code times the token's scale */
        const uint8_t* row = cv->c8 + tok * DC;
        double sigma = (double)cv->scale[tok];
        for (int i = 0; i < DC; ++i) ckv[i] = oracle_e4m3_value(row[i]) * sigma;
        const uint16_t* r = cv->kr + tok * DR;
        for (int i = 0; i < DR; ++i) kr[i] = bf16_value(r[i]);
    } else {
        /* NVFP4: e2m1 code times its block's e4m3 scale times the token's fp32 scale (exact in double) */
        const uint8_t* row = cv->c8 + tok * NV_ROW;
        const uint8_t* bs = row + NV_CODES;
        double sigma = (double)cv->scale[tok];
        for (int i = 0; i < DC; ++i) {
            const uint8_t code = (i & 1) ? (uint8_t)(row[i / 2] >> 4) : (uint8_t)(row[i / 2] & 0x0F);
            ckv[i] = oracle_e2m1_value(code) * oracle_e4m3_value(bs[i / 16]) * sigma;
        }
        const uint16_t* r = cv->kr + tok * DR;
        for (int i = 0; i < DR; ++i) kr[i] = bf16_value(r[i]);
    }
    return 0;
}

static cache_view make_view(int kv_fp8, int num_pages, const uint16_t* pool, const uint8_t* c8,
                            const float* scale, const uint16_t* kr)
{
    cache_view cv;
    cv.kv_fp8 = kv_fp8;
    cv.num_pages = num_pages;
    cv.pool = pool;
    cv.c8 = c8;
    cv.scale = scale;
    cv.kr = kr;
    return cv;
}

/* ------------------------------------------------------------------ naive (decompressed) path */

/*
 * The definition.  For each sequence b and each listed head h:
 *   k_t = W_UK[h] c_t,  v_t = W_UV[h] c_t                       (each 128-d)
 *   s_t = (q_c[b,h] . k_t + q_R[b,h] . k_R,t) * softmax_scale     for t < S_b
 *   p_t = exp(s_t - max s) / sum_u exp(s_u - max s)
 *   out[b,h] = sum_t p_t v_t
 * out is [B][n_heads][128].  If probs is not NULL it receives p as [B][n_heads][max_pages*64]
 * (zero past S_b).  Returns 0, or -1 if a block-table entry is out of range.
 */
int oracle_decode_naive(int B, const int32_t* seq_lens, const int32_t* block_table, int max_pages,
                        int kv_fp8, int num_pages, const uint16_t* pool, const uint8_t* c8,
                        const float* scale, const uint16_t* kr,
                        const uint16_t* q_c, const uint16_t* q_r,
                        const uint16_t* w_uk, const uint16_t* w_uv,
                        double softmax_scale, int n_heads, const int32_t* heads,
                        double* out, double* probs)
{
    cache_view cv = make_view(kv_fp8, num_pages, pool, c8, scale, kr);
    int bad = 0;
    const int64_t tasks = (int64_t)B * n_heads;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t task = 0; task < tasks; ++task) {
        const int b = (int)(task / n_heads), hi = (int)(task % n_heads), h = heads[hi];
        const int64_t S = seq_lens[b];
        const int32_t* bt = block_table + (int64_t)b * max_pages;
        double* Wk = (double*)malloc(sizeof(double) * DHC * DC);
        double* Wv = (double*)malloc(sizeof(double) * DHC * DC);
        double* s = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
        double qc[DHC], qr[DR], ckv[DC], kvr[DR], k[DHC], v[DHC], acc[DHC];
        for (int i = 0; i < DHC * DC; ++i) {
            Wk[i] = bf16_value(w_uk[(int64_t)h * DHC * DC + i]);
            Wv[i] = bf16_value(w_uv[(int64_t)h * DHC * DC + i]);
        }
        for (int d = 0; d < DHC; ++d) qc[d] = bf16_value(q_c[((int64_t)b * NH + h) * DHC + d]);
        for (int r = 0; r < DR; ++r) qr[r] = bf16_value(q_r[((int64_t)b * NH + h) * DR + r]);

        /* scores */
        double mx = -INFINITY;
        for (int64_t t = 0; t < S; ++t) {
            if (gather_row(&cv, bt, t, ckv, kvr)) { bad = 1; s[t] = -INFINITY; continue; }
            for (int d = 0; d < DHC; ++d) {
                double a = 0.0;
                for (int c = 0; c < DC; ++c) a += Wk[d * DC + c] * ckv[c];
                k[d] = a;
            }
            double dot = 0.0;
            for (int d = 0; d < DHC; ++d) dot += qc[d] * k[d];
            for (int r = 0; r < DR; ++r) dot += qr[r] * kvr[r];
            s[t] = dot * softmax_scale;
            if (s[t] > mx) mx = s[t];
        }
        /* softmax denominator */
        double den = 0.0;
        for (int64_t t = 0; t < S; ++t) den += exp(s[t] - mx);
        /* weighted sum of decompressed values */
        for (int d = 0; d < DHC; ++d) acc[d] = 0.0;
        for (int64_t t = 0; t < S; ++t) {
            double p = exp(s[t] - mx) / den;
            if (probs) probs[((int64_t)b * n_heads + hi) * (int64_t)max_pages * PG + t] = p;
            if (gather_row(&cv, bt, t, ckv, kvr)) continue;
            for (int d = 0; d < DHC; ++d) {
                double a = 0.0;
                for (int c = 0; c < DC; ++c) a += Wv[d * DC + c] * ckv[c];
                v[d] = a;
            }
            for (int d = 0; d < DHC; ++d) acc[d] += p * v[d];
        }
        if (probs)
            for (int64_t t = S; t < (int64_t)max_pages * PG; ++t)
                probs[((int64_t)b * n_heads + hi) * (int64_t)max_pages * PG + t] = 0.0;
        for (int d = 0; d < DHC; ++d) out[((int64_t)b * n_heads + hi) * DHC + d] = acc[d];
        free(Wk);
        free(Wv);
        free(s);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ absorbed path, step by step */

/* q_abs[b,h,c] = sum_d q_c[b,h,d] W_UK[h,d,c]   (page 1 section 4, einsum 'qhd,hdc->qhc') */
void oracle_absorb_q(int B, const uint16_t* q_c, const uint16_t* w_uk, double* q_abs)
{
    const int64_t tasks = (int64_t)B * NH;
#pragma omp parallel for schedule(static)
    for (int64_t task = 0; task < tasks; ++task) {
        const int b = (int)(task / NH), h = (int)(task % NH);
        double acc[DC];
        for (int c = 0; c < DC; ++c) acc[c] = 0.0;
        for (int d = 0; d < DHC; ++d) {
            double q = bf16_value(q_c[((int64_t)b * NH + h) * DHC + d]);
            for (int c = 0; c < DC; ++c) acc[c] += q * bf16_value(w_uk[((int64_t)h * DHC + d) * DC + c]);
        }
        for (int c = 0; c < DC; ++c) q_abs[((int64_t)b * NH + h) * DC + c] = acc[c];
    }
}

/*
 * Attention in the latent space over the pages [page_begin[b], page_end[b]) of sequence b
 * (tokens below S_b only):
 *   s_t   = (q_lat[b,h] . c_t + q_R[b,h] . k_R,t) * softmax_scale
 *   lse   = log sum_t exp(s_t)                                  (natural log)
 *   o_lat = sum_t exp(s_t - lse) c_t                            (512-d)
 * q_lat is [B][128][512] in double, so a caller can pass either the oracle's own q_abs or
 * bf16-rounded values.  o_lat is [B][n_heads][512], lse [B][n_heads].  A range holding no
 * token gives lse = -inf and o_lat = 0.  Returns -1 if a block-table entry is out of range.
 */
int oracle_latent_attention(int B, const double* q_lat, const uint16_t* q_r,
                            const int32_t* seq_lens, const int32_t* block_table, int max_pages,
                            const int32_t* page_begin, const int32_t* page_end,
                            int kv_fp8, int num_pages, const uint16_t* pool, const uint8_t* c8,
                            const float* scale, const uint16_t* kr,
                            double softmax_scale, int n_heads, const int32_t* heads,
                            double* o_lat, double* lse)
{
    cache_view cv = make_view(kv_fp8, num_pages, pool, c8, scale, kr);
    int bad = 0;
    const int64_t tasks = (int64_t)B * n_heads;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t task = 0; task < tasks; ++task) {
        const int b = (int)(task / n_heads), hi = (int)(task % n_heads), h = heads[hi];
        const int32_t* bt = block_table + (int64_t)b * max_pages;
        int64_t t0 = (int64_t)page_begin[b] * PG, t1 = (int64_t)page_end[b] * PG;
        if (t1 > seq_lens[b]) t1 = seq_lens[b];
        const int64_t n = t1 > t0 ? t1 - t0 : 0;
        double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        const double* q = q_lat + ((int64_t)b * NH + h) * DC;
        double qr[DR], ckv[DC], kvr[DR], acc[DC];
        for (int r = 0; r < DR; ++r) qr[r] = bf16_value(q_r[((int64_t)b * NH + h) * DR + r]);

        double mx = -INFINITY;
        for (int64_t i = 0; i < n; ++i) {
            if (gather_row(&cv, bt, t0 + i, ckv, kvr)) { bad = 1; s[i] = -INFINITY; continue; }
            double dot = 0.0;
            for (int c = 0; c < DC; ++c) dot += q[c] * ckv[c];
            for (int r = 0; r < DR; ++r) dot += qr[r] * kvr[r];
            s[i] = dot * softmax_scale;
            if (s[i] > mx) mx = s[i];
        }
        double den = 0.0;
        for (int64_t i = 0; i < n; ++i) den += exp(s[i] - mx);
        const double l = n > 0 ? mx + log(den) : -INFINITY;
        for (int c = 0; c < DC; ++c) acc[c] = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            if (gather_row(&cv, bt, t0 + i, ckv, kvr)) continue;
            double p = exp(s[i] - l);
            for (int c = 0; c < DC; ++c) acc[c] += p * ckv[c];
        }
        for (int c = 0; c < DC; ++c) o_lat[((int64_t)b * n_heads + hi) * DC + c] = acc[c];
        lse[(int64_t)b * n_heads + hi] = l;
        free(s);
    }
    return bad ? -1 : 0;
}

/* out[b,h,d] = sum_c o_lat[b,h,c] W_UV[h,d,c]   (o_lat in double, [B][128][512]) */
void oracle_out_proj(int B, const double* o_lat, const uint16_t* w_uv, double* out)
{
    const int64_t tasks = (int64_t)B * NH;
#pragma omp parallel for schedule(static)
    for (int64_t task = 0; task < tasks; ++task) {
        const int b = (int)(task / NH), h = (int)(task % NH);
        const double* o = o_lat + ((int64_t)b * NH + h) * DC;
        for (int d = 0; d < DHC; ++d) {
            double a = 0.0;
            for (int c = 0; c < DC; ++c) a += o[c] * bf16_value(w_uv[((int64_t)h * DHC + d) * DC + c]);
            out[((int64_t)b * NH + h) * DHC + d] = a;
        }
    }
}

/*
 * Log-sum-exp merge of n partial results of the same rows ("stage 2" split reduction).
 * Part j of row r has lse[j][r] and a normalised output o[j][r][0..DC).  Then
 *   lse_out[r] = log sum_j exp(lse[j][r]),   o_out[r] = sum_j exp(lse[j][r] - lse_out[r]) o[j][r].
 * Parts with lse = -inf (no tokens) carry no weight.
 */
void oracle_lse_combine(int rows, int n, const double* lse, const double* o, double* lse_out, double* o_out)
{
    for (int r = 0; r < rows; ++r) {
        double mx = -INFINITY;
        for (int j = 0; j < n; ++j)
            if (lse[(int64_t)j * rows + r] > mx) mx = lse[(int64_t)j * rows + r];
        double sum = 0.0;
        for (int j = 0; j < n; ++j) sum += (mx == -INFINITY) ? 0.0 : exp(lse[(int64_t)j * rows + r] - mx);
        const double L = (sum > 0.0) ? mx + log(sum) : -INFINITY;
        lse_out[r] = L;
        for (int c = 0; c < DC; ++c) o_out[(int64_t)r * DC + c] = 0.0;
        for (int j = 0; j < n; ++j) {
            const double lj = lse[(int64_t)j * rows + r];
            if (lj == -INFINITY) continue;
            const double w = exp(lj - L);
            for (int c = 0; c < DC; ++c) o_out[(int64_t)r * DC + c] += w * o[((int64_t)j * rows + r) * DC + c];
        }
    }
}

/* ------------------------------------------------------------------ cache append (write side) */

/*
 * The e4m3 code nearest a finite float, ties to the code with the even mantissa field, and a
 * magnitude at or past 448 (the largest finite code) gives 448.  The sign is kept, zero
 * results included.  Straight from the format's definition (oracle_e4m3_value above): the
 * non-negative finite codes 0x00..0x7E have increasing values, so take the last one not above
 * |x| and the one after it and keep the nearer.
 */
uint8_t oracle_e4m3_encode(float x)
{
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    int lo = 0;
    while (lo + 1 <= 0x7E && oracle_e4m3_value((uint8_t)(lo + 1)) <= a) ++lo;
    const double below = oracle_e4m3_value((uint8_t)lo);
    if (below == a) return sign | (uint8_t)lo;
    const int hi = lo + 1;
    const double d_lo = a - below, d_hi = oracle_e4m3_value((uint8_t)hi) - a;
    int c;
    if (d_lo < d_hi)
        c = lo;
    else if (d_hi < d_lo)
        c = hi;
    else
        c = (lo & 1) ? hi : lo; /* a tie: the even mantissa field */
    return sign | (uint8_t)c;
}

void oracle_e4m3_encode_many(const float* x, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

/*
 * One token's latent for the FP8 cache: sigma = (largest |c_i|) / 448 in fp32, or 1 when the
 * row is all zeros; code_i = the e4m3 code nearest c_i / sigma, the quotient taken in fp32.
 * c is the token's 512 bf16 latent values.  Returns sigma.
 */
float oracle_quantize_token(const uint16_t* c, uint8_t* codes)
{
    float amax = 0.0f;
    for (int i = 0; i < DC; ++i) {
        const float v = fabsf((float)bf16_value(c[i]));
        if (v > amax) amax = v;
    }
    const float sigma = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int i = 0; i < DC; ++i) codes[i] = oracle_e4m3_encode((float)bf16_value(c[i]) / sigma);
    return sigma;
}

/*
 * The e2m1 code nearest a finite value, ties to the code with the even mantissa field (m = 0),
 * magnitudes at or past 6 (the largest) give 6; the sign is kept, zero results included.  The
 * non-negative codes 0..7 have increasing values: take the last one not above |x| and the next.
 */
uint8_t oracle_e2m1_encode(float x)
{
    const uint8_t sign = signbit(x) ? 0x8 : 0x0;
    const double a = fabs((double)x);
    if (a >= 6.0) return sign | 0x7;
    int k = 0;  /* the largest magnitude code not above a */
    while (k + 1 <= 7 && oracle_e2m1_value((uint8_t)(k + 1)) <= a) ++k;
    const double v_below = oracle_e2m1_value((uint8_t)k);
    if (v_below == a) return sign | (uint8_t)k;
    const double gap_below = a - v_below, gap_above = oracle_e2m1_value((uint8_t)(k + 1)) - a;
    int code = k;
    if (gap_above < gap_below || (gap_above == gap_below && (k & 1)))
        code = k + 1; /* nearer above, or a tie whose even mantissa field (m = 0) is above */
    return sign | (uint8_t)code;
}

void oracle_e2m1_encode_many(const float* x, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_encode(x[i]);
}

/*
 * One token's latent for the NVFP4 cache (two-level scaling: an fp32 scale per token and an e4m3
 * scale per 16 consecutive latent values, e2m1 codes).  All in fp32, in this order:
 *   sigma  = (largest |c_i| of the token) / 2688   (2688 = 6 * 448), or 1 for an all-zero row;
 *   t_b    = ((largest |c_i| of block b) / sigma) / 6,   S_b = the e4m3 code nearest t_b;
 *   code_i = the e2m1 code nearest c_i / (sigma * S_b), or a zero of c_i's sign when S_b is 0.
 * c is the token's 512 bf16 latent values; row receives the 288-byte NVFP4 row: 256 bytes of
 * codes (value 2j in the low nibble of byte j), then the 32 block scales.  Returns sigma.
 */
float oracle_quantize_token_nvfp4(const uint16_t* c, uint8_t* row)
{
    uint8_t* codes = row;
    uint8_t* bscale = row + NV_CODES;
    float amax = 0.0f;
    for (int i = 0; i < DC; ++i) {
        const float v = fabsf((float)bf16_value(c[i]));
        if (v > amax) amax = v;
    }
    const float sigma = amax > 0.0f ? amax / 2688.0f : 1.0f;
    for (int b = 0; b < DC / 16; ++b) {
        float bmax = 0.0f;
        for (int i = 16 * b; i < 16 * b + 16; ++i) {
            const float v = fabsf((float)bf16_value(c[i]));
            if (v > bmax) bmax = v;
        }
        const uint8_t s8 = oracle_e4m3_encode((bmax / sigma) / 6.0f);
        bscale[b] = s8;
        const float den = sigma * (float)oracle_e4m3_value(s8);
        for (int i = 16 * b; i < 16 * b + 16; ++i) {
            const float x = (float)bf16_value(c[i]);
            uint8_t q;
            if (den == 0.0f)
                q = signbit(x) ? 0x8 : 0x0;
            else
                q = oracle_e2m1_encode(x / den);
            if (i & 1)
                codes[i / 2] = (uint8_t)((codes[i / 2] & 0x0F) | (q << 4));
            else
                codes[i / 2] = q;
        }
    }
    return sigma;
}

/* The bf16 nearest a float, ties to even (NaN stays a quiet NaN): keep the top 16 bits after
 * adding half of the dropped part's range, plus one when the kept part is odd. */
static uint16_t bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

/*
 * Gather (page 1, the "NVFP4 quantized gather" of the table of contents and section 5): the
 * rows of each sequence, in logical order, out of the paged cache into one contiguous bf16
 * array out[cu_seqlens[b] + t][576] (c_KV then k_R).  bf16 cache: the stored bits.  FP8 cache:
 * each latent value is float(e4m3 code) * sigma in fp32 (one rounding), then rounded to bf16.
 * NVFP4 cache: float(e2m1 code) * float(e4m3 block scale) (exact) * sigma in fp32 (one rounding),
 * then to bf16.  k_R is copied.  Returns -1 if a block-table entry is out of range (that row
 * is left untouched), else 0.
 */
int oracle_gather_kv(int B, const int32_t* seq_lens, const int32_t* block_table, int max_pages,
                     const int32_t* cu_seqlens, int kv_fp8, int num_pages, const uint16_t* pool,
                     const uint8_t* c8, const float* scale, const uint16_t* kr, uint16_t* out)
{
    int status = 0;
    for (int b = 0; b < B; ++b) {
        for (int64_t t = 0; t < seq_lens[b]; ++t) {
            const int64_t page = block_table[(int64_t)b * max_pages + t / PG];
            if (page < 0 || page >= num_pages) {
                status = -1;
                continue;
            }
            const int64_t tok = page * PG + (t % PG);
            uint16_t* dst = out + ((int64_t)cu_seqlens[b] + t) * DROW;
            if (kv_fp8 == 0) {
                memcpy(dst, pool + tok * DROW, DROW * sizeof(uint16_t));
                continue;
            }
            const float sigma = scale[tok];
            if (kv_fp8 == 1) {
                const uint8_t* row = c8 + tok * DC;
                for (int i = 0; i < DC; ++i) dst[i] = bf16_rne((float)oracle_e4m3_value(row[i]) * sigma);
            } else {
                const uint8_t* row = c8 + tok * NV_ROW;
                for (int i = 0; i < DC; ++i) {
                    const uint8_t byte = row[i >> 1];
                    const uint8_t e2 = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
                    const float v = (float)oracle_e2m1_value(e2) * (float)oracle_e4m3_value(row[NV_CODES + i / 16]);
                    dst[i] = bf16_rne(v * sigma);
                }
            }
            memcpy(dst + DC, kr + tok * DR, DR * sizeof(uint16_t));
        }
    }
    return status;
}

/*
 * Write n tokens into the paged cache (page 1 section 1: one row of c_KV and k_R per token;
 * section 3: 64-token pages).  Token i goes to slot slots[i] = page * 64 + row; a negative slot
 * skips the token, and so does a slot at or past num_pages * 64 (then the call returns -1).
 * bf16 cache: pool row = the token's c_KV then k_R.  FP8 cache (kv_fp8 = 1): c8 row = the
 * codes of oracle_quantize_token, scale = its sigma, kr row = k_R.  NVFP4 cache (kv_fp8 = 2): c8
 * row = the 288-byte row of oracle_quantize_token_nvfp4, scale = its sigma, kr row = k_R.
 */
int oracle_append_kv(int n, const uint16_t* c_kv, const uint16_t* k_r, const int32_t* slots, int kv_fp8,
                     int num_pages, uint16_t* pool, uint8_t* c8, float* scale, uint16_t* kr)
{
    int status = 0;
    for (int i = 0; i < n; ++i) {
        const int64_t slot = slots[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_pages * PG) {
            status = -1;
            continue;
        }
        const uint16_t* c = c_kv + (int64_t)i * DC;
        const uint16_t* r = k_r + (int64_t)i * DR;
        if (!kv_fp8) {
            uint16_t* row = pool + slot * DROW;
            for (int j = 0; j < DC; ++j) row[j] = c[j];
            for (int j = 0; j < DR; ++j) row[DC + j] = r[j];
        } else if (kv_fp8 == 1) {
            scale[slot] = oracle_quantize_token(c, c8 + slot * DC);
            for (int j = 0; j < DR; ++j) kr[slot * DR + j] = r[j];
        } else {
            scale[slot] = oracle_quantize_token_nvfp4(c, c8 + slot * NV_ROW);
            memcpy(kr + slot * DR, r, DR * sizeof(uint16_t)); /* k_R unchanged */
        }
    }
    return status;
}

/*
 * Several new tokens of a sequence decoded in one step.  Page 1 section 6 (with the
 * kPrefillThresh = 256 of section 3's mla_config.h) runs chunks of fewer than 256 new tokens
 * through the absorbed decode path; speculative drafts are the same shape.  Reading taken:
 * the cache already holds the q new tokens of sequence b (S_b counts them), new token t
 * (0 <= t < q) is the token at position S_b - q + t, and it attends causally to positions
 * 0 .. S_b - q + t of its sequence.  Each new token is then an ordinary decode query over a
 * prefix of the sequence.  Query row b*q + t of the per-row tensors is token t of sequence b.
 * Fills row_len[b*q + t] = S_b - q + 1 + t (tokens visible to that query) and
 * row_table[b*q + t] = b (the block-table row holding its pages).  Returns -1 (nothing
 * written) if q < 1 or some S_b < q, else 0.
 */
int oracle_query_rows(int B, int q, const int32_t* seq_lens, int32_t* row_len, int32_t* row_table)
{
    if (q < 1) return -1;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < q) return -1;
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < q; ++t) {
            const int64_t row = (int64_t)b * q + t;
            row_len[row] = seq_lens[b] - q + 1 + t;
            row_table[row] = b;
        }
    return 0;
}
