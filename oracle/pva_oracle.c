/*
 * Plain CPU oracle for the paged variable-length attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this code.  The product path
 * (the CUDA library and its Python binding) never calls it, and this file
 * shares no code, header, table or helper with that path.
 *
 * What it computes follows the pages literally, slowly and in order:
 *
 *   - "The attention backend and a reference implementation" (mini-sglang
 *     from Scratch, ch. 5), section "Variable-length, paged attention with
 *     prefixes": write this step's K/V into the pool first, then for each
 *     request gather its whole KV through its page-table row, build the
 *     [n, kv_len] bottom-right causal mask (query r sits at absolute position
 *     kv_len - n + r and sees keys j <= kv_len - n + r), and apply
 *     softmax(scale * Q K^T) V with grouped-query heads (enable_gqa).
 *   - "Variable-length batching and one mixed forward pass", section
 *     "Layout and metadata": query_start_loc / seq_lens / slot_mapping /
 *     block tables; prefill, chunked prefill and decode are the same
 *     computation with different (cached, new) lengths.
 *
 * Readings taken where the pages leave a step open (each restated in the
 * design notes of the repository):
 *   - page table entries are page ids; the pool slot of position j of
 *     request i is page_table[i][j / page_size] * page_size + j % page_size
 *     (with page_size 1 this is exactly the token-slot table of ch. 5);
 *   - q head h uses kv head h / (Hq / Hkv) (the grouping of enable_gqa);
 *   - LSE is the natural-log log-sum-exp of the scaled, masked scores;
 *   - a slot_mapping entry of -1 means "no write" (padding token);
 *   - arithmetic is fp32 (the precision the pages run their reference
 *     backend in), sums taken in index order.
 *
 * Storage types: bf16 values are passed as their raw 16-bit patterns
 * (uint16_t); bf16 -> fp32 is exact (the pattern becomes the high half).
 *
 * FP8 KV pool (a pool element type the pages name only as a KV-cache dtype
 * choice, "Attention backends: ...", the kv_cache_dtype of the backend
 * interface): one byte per element in the E4M3 format of the OCP 8-bit
 * floating-point specification, with one fp32 scale per kv head for K and
 * one for V.  Readings: a stored element is e4m3(x / scale[g]) (fp32 division,
 * round to nearest even, values beyond the largest finite 448 saturate); the
 * attention reads e4m3 * scale[g] (fp32 product) and is otherwise unchanged.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static float bf16_bits_to_float(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * E4M3: sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  Exponent field 0
 * holds the subnormals m * 2^-9; fields 1..15 the normals 2^(e-7) * (1 + m/8),
 * except S.1111.111, the only NaN.  There are no infinities; the largest finite
 * value is 2^8 * 1.75 = 448.
 */
float oracle_e4m3_decode(uint8_t b) {
    const int e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (float)((b & 0x80) ? -v : v);
}

/*
 * Nearest E4M3 value of x, ties to the even mantissa; |x| above 448 (also
 * infinities) gives +-448; NaN gives the NaN code with x's sign.  The rounding
 * is done in double on the magnitude divided by the quantum of its binade (an
 * exact power-of-two division), so rint() sees the exact quotient.
 */
uint8_t oracle_e4m3_encode(float x) {
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    const double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    double quantum;
    if (a < ldexp(1.0, -6)) {
        quantum = ldexp(1.0, -9);  /* subnormal spacing */
    } else {
        int e2;
        frexp(a, &e2);  /* a = f * 2^e2, f in [0.5, 1): a in [2^(e2-1), 2^e2) */
        quantum = ldexp(1.0, e2 - 1 - 3);
    }
    const double v = rint(a / quantum) * quantum; /* default rounding mode: to nearest, ties to even */
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6)) return (uint8_t)(sign | (int)(v / ldexp(1.0, -9)));
    int e2;
    frexp(v, &e2);
    const int e = e2 - 1;                                   /* v in [2^e, 2^(e+1)) */
    const int m = (int)((v / ldexp(1.0, e) - 1.0) * 8.0);  /* exact: v has 3 fraction bits */
    return (uint8_t)(sign | ((e + 7) << 3) | m);
}

void oracle_e4m3_encode_array(int64_t n, const float *x, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(int64_t n, const uint8_t *b, float *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(b[i]);
}

/* Number of OpenMP threads the attention loop will use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Pool slot of absolute position j of request i.
 * Follows: page-level block tables ("Variable-length batching ...",
 * section "Implementation": slot_mapping_for(table, pos, block_size)) and
 * the ch. 5 page table read with page_size 1.
 */
static int64_t slot_of(const int32_t *page_table, int64_t ld, int page_size, int i, int64_t j) {
    int64_t page = page_table[(int64_t)i * ld + j / page_size];
    return page * page_size + j % page_size;
}

/*
 * slot_mapping for this step's new tokens: request i's n_i new tokens are its
 * last n_i positions kv_len_i - n_i .. kv_len_i - 1 ("The attention backend
 * and a reference implementation", the worked example: out_loc is
 * page_table[i, cached:len]).
 * Returns 0, or -(i+1) if request i has n_i > kv_len_i or n_i < 0.
 */
int oracle_slot_mapping(int B, const int32_t *cu_seqlens_q, const int32_t *cache_seqlens,
                        const int32_t *page_table, int64_t ld, int page_size, int64_t *slots_out) {
    for (int i = 0; i < B; ++i) {
        int n = cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        int L = cache_seqlens[i];
        if (n < 0 || n > L) return -(i + 1);
        for (int r = 0; r < n; ++r)
            slots_out[cu_seqlens_q[i] + r] = slot_of(page_table, ld, page_size, i, (int64_t)(L - n + r));
    }
    return 0;
}

/*
 * store_kvcache: pool[slot[t]][h][:] = new[t][h][:] for K and V, as raw bits.
 * ("The attention backend ...", TorchAttnBackend.forward: store_kv before
 * any read; "Attention backends: ...", step 2: do_kv_cache_update is a
 * scatter by slot.)  slot -1 = skip.  Returns 0, or -(t+1) for the first
 * token whose slot is out of range (nothing is written for that token).
 */
int oracle_store_kvcache(int64_t T, int Hkv, int D, const uint16_t *k, const uint16_t *v,
                         const int64_t *slots, int64_t num_slots, uint16_t *k_pool, uint16_t *v_pool) {
    int rc = 0;
    const int64_t row = (int64_t)Hkv * D;
    for (int64_t t = 0; t < T; ++t) {
        int64_t s = slots[t];
        if (s == -1) continue;
        if (s < 0 || s >= num_slots) {
            if (rc == 0) rc = (int)-(t + 1);
            continue;
        }
        memcpy(k_pool + s * row, k + t * row, (size_t)row * sizeof(uint16_t));
        memcpy(v_pool + s * row, v + t * row, (size_t)row * sizeof(uint16_t));
    }
    return rc;
}

/*
 * store_kvcache into an FP8 pool: pool[slot[t]][h][d] = e4m3(float(new[t][h][d])
 * / scale[h]) for K and V.  Same slot rules and return value as above.
 */
int oracle_store_kvcache_fp8(int64_t T, int Hkv, int D, const uint16_t *k, const uint16_t *v,
                             const int64_t *slots, int64_t num_slots, const float *k_scale,
                             const float *v_scale, uint8_t *k_pool, uint8_t *v_pool) {
    int rc = 0;
    const int64_t row = (int64_t)Hkv * D;
    for (int64_t t = 0; t < T; ++t) {
        int64_t s = slots[t];
        if (s == -1) continue;
        if (s < 0 || s >= num_slots) {
            if (rc == 0) rc = (int)-(t + 1);
            continue;
        }
        for (int h = 0; h < Hkv; ++h)
            for (int d = 0; d < D; ++d) {
                const int64_t src = t * row + (int64_t)h * D + d, dst = s * row + (int64_t)h * D + d;
                const float kx = bf16_bits_to_float(k[src]) / k_scale[h];
                const float vx = bf16_bits_to_float(v[src]) / v_scale[h];
                k_pool[dst] = oracle_e4m3_encode(kx);
                v_pool[dst] = oracle_e4m3_encode(vx);
            }
    }
    return rc;
}

/*
 * The bottom-right causal mask of one request: M[r][j] = (j <= L - n + r),
 * for r < n and j < L ("The attention backend and a reference
 * implementation", the mask figure and "query r sits at absolute position
 * kv_len - n + r").
 */
void oracle_causal_mask(int n, int L, uint8_t *mask_out) {
    for (int r = 0; r < n; ++r)
        for (int j = 0; j < L; ++j)
            mask_out[(int64_t)r * L + j] = (uint8_t)(j <= L - n + r);
}

/*
 * Attention over the paged pool, one request and one q head at a time.
 *
 *   for each request i with n = cu[i+1]-cu[i] > 0 and L = cache_seqlens[i]:
 *     K_i[j], V_i[j] = pool[slot_of(i, j)]        j < L   (the page-table gather)
 *     M = bottom-right causal mask [n, L]
 *     for each q head h (kv head g = h / (Hq/Hkv)) and row r:
 *       S[j] = scale * sum_d q[cu_i + r][h][d] * K_i[j][g][d]   (masked -> -inf)
 *       m = max_j S[j];  p_j = exp(S[j] - m);  l = sum_j p_j
 *       out[cu_i + r][h][:] = sum_j p_j V_i[j][g][:] / l
 *       lse[cu_i + r][h]    = m + log(l)
 *
 * row_select (optional, [T*Hq] bytes): when given, only rows (t, h) with a
 * nonzero byte are computed; others are left untouched.  This lets a test
 * check sampled rows of a batch too large to compute whole.
 *
 * Returns 0, or -(i+1) when request i violates n <= L or reads a page id
 * outside [0, num_pages).
 */
/* One pool element as fp32: a bf16 pattern, or an E4M3 byte times its head's scale. */
static float pool_value(const void *pool, int fp8, int64_t idx, float scale) {
    if (fp8) return oracle_e4m3_decode(((const uint8_t *)pool)[idx]) * scale;
    return bf16_bits_to_float(((const uint16_t *)pool)[idx]);
}

static int attention_core(int B, const int32_t *cu_seqlens_q, const int32_t *cache_seqlens,
                          const int32_t *page_table, int64_t ld, int page_size, int64_t num_pages,
                          int Hq, int Hkv, int D, float scale, const uint16_t *q,
                          const void *k_pool, const void *v_pool, int fp8, const float *k_scale,
                          const float *v_scale, const uint8_t *row_select, float *out, float *lse) {
    const int group = Hq / Hkv;
    const int64_t kv_row = (int64_t)Hkv * D;

    /* Validate first, so that the parallel loop below never reads out of range. */
    for (int i = 0; i < B; ++i) {
        int n = cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        int L = cache_seqlens[i];
        if (n < 0 || n > L) return -(i + 1);
        int64_t pages = n > 0 ? (L + page_size - 1) / page_size : 0;
        for (int64_t p = 0; p < pages; ++p) {
            int32_t id = page_table[(int64_t)i * ld + p];
            if (id < 0 || id >= num_pages) return -(i + 1);
        }
    }

    int rc = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t work = 0; work < (int64_t)B * Hq; ++work) {
        const int i = (int)(work / Hq);
        const int h = (int)(work % Hq);
        const int n = cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        const int L = cache_seqlens[i];
        if (n == 0) continue;
        const int q0 = cu_seqlens_q[i];
        const int g = h / group;

        if (row_select) {
            int any = 0;
            for (int r = 0; r < n && !any; ++r) any = row_select[(int64_t)(q0 + r) * Hq + h] != 0;
            if (!any) continue;
        }

        /* gather this kv head's keys and values through the page table */
        float *Ki = (float *)malloc(sizeof(float) * (size_t)L * D);
        float *Vi = (float *)malloc(sizeof(float) * (size_t)L * D);
        uint8_t *M = (uint8_t *)malloc((size_t)n * L);
        float *S = (float *)malloc(sizeof(float) * (size_t)L);
        float *qf = (float *)malloc(sizeof(float) * (size_t)D);
        if (!Ki || !Vi || !M || !S || !qf) {
            free(Ki); free(Vi); free(M); free(S); free(qf);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            rc = -1000000;
            continue;
        }
        const float ks = fp8 ? k_scale[g] : 1.0f, vs = fp8 ? v_scale[g] : 1.0f;
        for (int64_t j = 0; j < L; ++j) {
            const int64_t row0 = slot_of(page_table, ld, page_size, i, j) * kv_row + (int64_t)g * D;
            for (int d = 0; d < D; ++d) {
                Ki[j * D + d] = pool_value(k_pool, fp8, row0 + d, ks);
                Vi[j * D + d] = pool_value(v_pool, fp8, row0 + d, vs);
            }
        }
        oracle_causal_mask(n, L, M);

        for (int r = 0; r < n; ++r) {
            const int64_t t = q0 + r;
            if (row_select && !row_select[t * Hq + h]) continue;
            const uint16_t *qr = q + (t * Hq + h) * D;
            for (int d = 0; d < D; ++d) qf[d] = bf16_bits_to_float(qr[d]);

            float m = -INFINITY;
            for (int64_t j = 0; j < L; ++j) {
                if (!M[(int64_t)r * L + j]) {
                    S[j] = -INFINITY;
                    continue;
                }
                float acc = 0.0f;
                for (int d = 0; d < D; ++d) acc += qf[d] * Ki[j * D + d];
                S[j] = scale * acc;
                if (S[j] > m) m = S[j];
            }
            float l = 0.0f;
            float *o = out + (t * Hq + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0f;
            for (int64_t j = 0; j < L; ++j) {
                if (!M[(int64_t)r * L + j]) continue;
                float p = expf(S[j] - m);
                l += p;
                for (int d = 0; d < D; ++d) o[d] += p * Vi[j * D + d];
            }
            for (int d = 0; d < D; ++d) o[d] /= l;
            if (lse) lse[t * Hq + h] = m + logf(l);
        }
        free(Ki); free(Vi); free(M); free(S); free(qf);
    }
    return rc;
}

int oracle_attention(int B, const int32_t *cu_seqlens_q, const int32_t *cache_seqlens,
                     const int32_t *page_table, int64_t ld, int page_size, int64_t num_pages,
                     int Hq, int Hkv, int D, float scale,
                     const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                     const uint8_t *row_select, float *out, float *lse) {
    return attention_core(B, cu_seqlens_q, cache_seqlens, page_table, ld, page_size, num_pages, Hq, Hkv, D,
                          scale, q, k_pool, v_pool, 0, NULL, NULL, row_select, out, lse);
}

/* The same attention over an FP8 pool (elements read as e4m3 * scale of their kv head). */
int oracle_attention_fp8(int B, const int32_t *cu_seqlens_q, const int32_t *cache_seqlens,
                         const int32_t *page_table, int64_t ld, int page_size, int64_t num_pages,
                         int Hq, int Hkv, int D, float scale,
                         const uint16_t *q, const uint8_t *k_pool, const uint8_t *v_pool,
                         const float *k_scale, const float *v_scale,
                         const uint8_t *row_select, float *out, float *lse) {
    return attention_core(B, cu_seqlens_q, cache_seqlens, page_table, ld, page_size, num_pages, Hq, Hkv, D,
                          scale, q, k_pool, v_pool, 1, k_scale, v_scale, row_select, out, lse);
}
