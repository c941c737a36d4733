/*
 * pkv_oracle.c -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.
 *
 * A plain, slow, fp64 CPU oracle for attention over a paged (block-sparse
 * row) KV cache.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this library; the product path never calls it and
 * shares no code with it.
 *
 * What it computes (FlashInfer pages):
 *  - Page-table gather: token t of request b lives in physical page
 *    kv_indices[kv_indptr[b] + t / page_size], slot t % page_size
 *    ("FlashInfer" guide, section 2 "Page-Level Attention"; fdeinterviews
 *    summary, paragraph "One format for every KV layout").  The number of
 *    tokens is (pages - 1) * page_size + kv_last_page_len[b].
 *  - Attention per query row and query head over the gathered K, V:
 *    s_t = sm_scale * <q, k_t>; with soft-capping, s_t <- cap * tanh(s_t / cap)
 *    (the logits transform of the fdeinterviews paragraph "Customizable
 *    attention"); lse = ln sum_t exp(s_t); o = sum_t exp(s_t - lse) v_t.
 *  - Causal prefill ("The Interface", causal=True): row i of a request with
 *    qo_len rows and kv_len keys may see keys t <= i + kv_len - qo_len
 *    (the mask aligned to the end of the KV sequence).
 *  - Custom mask (the mask a variant supplies, fdeinterviews "Customizable
 *    attention"; token trees of speculative decoding, greptalks "Radix Tree /
 *    Token Tree"): request b's boolean matrix [qo_len, kv_len], row-major,
 *    packed one bit per entry (least significant bit first in each byte),
 *    the requests back to back from bit 0; row i sees key t only if its bit
 *    is 1, in addition to the causal rule.
 *  - merge_state (guide section 3, "Cascade Attention" and "FlashDecoding"):
 *    states (o_i, lse_i) over disjoint key sets combine as
 *    lse = ln sum_i exp(lse_i), o = sum_i exp(lse_i - lse) o_i.
 * Query head h reads kv head h / (num_qo_heads / num_kv_heads) (contiguous
 * head groups, the GQA head-group packing of the greptalks summary).
 * An empty key set gives o = 0 and lse = -inf.
 *
 * Storage: q and kv_data are 16-bit (fp16 or bf16), decoded exactly to
 * double here from the IEEE-754 binary16 and bfloat16 definitions.
 * Layouts: q [total_q, Hq, d]; kv_data [num_pages, 2, Hkv, page_size, d]
 * with K at index 0 and V at index 1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };
enum { ORACLE_OK = 0, ORACLE_BAD_ARG = -1, ORACLE_BAD_INDEX = -2, ORACLE_NO_MEM = -3 };

/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);              /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);  /* (1 + m/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE-754 binary32. */
static double decode_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double decode(uint16_t x, int dtype) {
    return dtype == ORACLE_BF16 ? decode_bf16(x) : decode_f16(x);
}

void pkv_oracle_decode16(const uint16_t* in, double* out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = decode(in[i], dtype);
}

typedef struct {
    int batch, num_qo_heads, num_kv_heads, head_dim, page_size, dtype;
    const uint16_t* kv_data;
    int64_t num_pages;
    const int32_t* kv_indptr;
    const int32_t* kv_indices;
    const int32_t* kv_last_page_len;
} paged_kv;

static int64_t kv_len_of(const paged_kv* c, int b) {
    int64_t n = (int64_t)c->kv_indptr[b + 1] - c->kv_indptr[b];
    if (n <= 0) return 0;
    return (n - 1) * c->page_size + c->kv_last_page_len[b];
}

/* Address of the 16-bit row of token t (kv_sel 0 = K, 1 = V) for kv head kvh. */
static const uint16_t* token_row(const paged_kv* c, int b, int64_t t, int kv_sel, int kvh) {
    int64_t page = c->kv_indices[c->kv_indptr[b] + t / c->page_size];
    int64_t slot = t % c->page_size;
    int64_t row = ((page * 2 + kv_sel) * c->num_kv_heads + kvh) * c->page_size + slot;
    return c->kv_data + row * c->head_dim;
}

static int check_table(const paged_kv* c) {
    if (c->batch < 0 || c->num_kv_heads <= 0 || c->num_qo_heads <= 0 || c->head_dim <= 0 ||
        c->page_size <= 0 || c->num_qo_heads % c->num_kv_heads)
        return ORACLE_BAD_ARG;
    if (c->kv_indptr[0] != 0) return ORACLE_BAD_INDEX;
    for (int b = 0; b < c->batch; ++b) {
        int32_t n = c->kv_indptr[b + 1] - c->kv_indptr[b];
        if (n < 0) return ORACLE_BAD_INDEX;
        int32_t last = c->kv_last_page_len[b];
        if (n > 0 && (last < 1 || last > c->page_size)) return ORACLE_BAD_INDEX;
        for (int32_t j = c->kv_indptr[b]; j < c->kv_indptr[b + 1]; ++j)
            if (c->kv_indices[j] < 0 || c->kv_indices[j] >= c->num_pages) return ORACLE_BAD_INDEX;
    }
    return ORACLE_OK;
}

/* Tokens of request b, gathered through the page table: out[kv_len][head_dim]. */
int pkv_oracle_gather(int batch, int num_kv_heads, int head_dim, int page_size, int dtype,
                      const uint16_t* kv_data, int64_t num_pages, const int32_t* kv_indptr,
                      const int32_t* kv_indices, const int32_t* kv_last_page_len, int b,
                      int kv_sel, int kvh, double* out, int64_t out_rows) {
    paged_kv c = {batch, num_kv_heads, num_kv_heads, head_dim, page_size, dtype, kv_data,
                  num_pages, kv_indptr, kv_indices, kv_last_page_len};
    int st = check_table(&c);
    if (st) return st;
    if (b < 0 || b >= batch || kv_sel < 0 || kv_sel > 1 || kvh < 0 || kvh >= num_kv_heads)
        return ORACLE_BAD_ARG;
    int64_t n = kv_len_of(&c, b);
    if (out_rows < n) return ORACLE_BAD_ARG;
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t* r = token_row(&c, b, t, kv_sel, kvh);
        for (int k = 0; k < head_dim; ++k) out[t * head_dim + k] = decode(r[k], dtype);
    }
    return (int)n;
}

/* Request that owns global query row r (qo_indptr is non-decreasing). */
static int owner_of(const int32_t* qo_indptr, int batch, int64_t r) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (qo_indptr[mid] <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

/*
 * Attention for the query rows listed in `rows` (global row ids into q), or
 * for every row when rows == NULL.  o: [n_out, Hq, d] doubles; lse: [n_out, Hq].
 * logits_cap <= 0 turns soft-capping off.  Returns 0 or a negative error.
 */
int pkv_oracle_attention(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                         int page_size, int dtype, const uint16_t* q, int64_t total_q,
                         const int32_t* qo_indptr, const uint16_t* kv_data, int64_t num_pages,
                         const int32_t* kv_indptr, const int32_t* kv_indices,
                         const int32_t* kv_last_page_len, int causal, double sm_scale,
                         double logits_cap, const uint8_t* mask, const int64_t* rows, int64_t n_rows,
                         double* o, double* lse, int num_threads) {
    paged_kv c = {batch, num_qo_heads, num_kv_heads, head_dim, page_size, dtype, kv_data,
                  num_pages, kv_indptr, kv_indices, kv_last_page_len};
    int st = check_table(&c);
    if (st) return st;
    if (qo_indptr[0] != 0 || qo_indptr[batch] != total_q) return ORACLE_BAD_INDEX;
    for (int b = 0; b < batch; ++b)
        if (qo_indptr[b + 1] < qo_indptr[b]) return ORACLE_BAD_INDEX;
    int64_t n_out = rows ? n_rows : total_q;
    for (int64_t i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= total_q) return ORACLE_BAD_ARG;
    int64_t max_kv = 0;
    for (int b = 0; b < batch; ++b) {
        int64_t n = kv_len_of(&c, b);
        if (n > max_kv) max_kv = n;
    }
    const int group = num_qo_heads / num_kv_heads;
    const int64_t jobs = n_out * num_qo_heads;
    /* first bit of each request's mask block */
    int64_t* mask_off = NULL;
    if (mask) {
        mask_off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(batch + 1));
        if (!mask_off) return ORACLE_NO_MEM;
        mask_off[0] = 0;
        for (int b = 0; b < batch; ++b)
            mask_off[b + 1] = mask_off[b] + ((int64_t)qo_indptr[b + 1] - qo_indptr[b]) * kv_len_of(&c, b);
    }
    int failed = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel num_threads(num_threads)
#endif
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1));
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        double* acc = (double*)malloc(sizeof(double) * (size_t)head_dim);
        if (!s || !qv || !acc) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (int64_t job = 0; job < jobs; ++job) {
                int64_t out_row = job / num_qo_heads;
                int h = (int)(job % num_qo_heads);
                int64_t r = rows ? rows[out_row] : out_row;
                int b = owner_of(qo_indptr, batch, r);
                int64_t i = r - qo_indptr[b];
                int64_t qo_len = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
                int64_t kv_len = kv_len_of(&c, b);
                int64_t visible = causal ? i + kv_len - qo_len + 1 : kv_len;
                if (visible > kv_len) visible = kv_len;
                if (visible < 0) visible = 0;
                int kvh = h / group;
                const uint16_t* qr = q + (r * num_qo_heads + h) * head_dim;
                for (int k = 0; k < head_dim; ++k) qv[k] = decode(qr[k], dtype);
                double* orow = o + (out_row * num_qo_heads + h) * head_dim;
                double* lrow = lse + out_row * num_qo_heads + h;
                int64_t n_seen = 0;
                double mx = -INFINITY;
                for (int64_t t = 0; t < visible; ++t) {
                    if (mask) {
                        int64_t bit = mask_off[b] + i * kv_len + t;
                        if (!((mask[bit >> 3] >> (bit & 7)) & 1)) {
                            s[t] = -INFINITY;
                            continue;
                        }
                    }
                    ++n_seen;
                    const uint16_t* kr = token_row(&c, b, t, 0, kvh);
                    double dot = 0.0;
                    for (int k = 0; k < head_dim; ++k) dot += qv[k] * decode(kr[k], dtype);
                    double logit = sm_scale * dot;
                    if (logits_cap > 0.0) logit = logits_cap * tanh(logit / logits_cap);
                    s[t] = logit;
                    if (logit > mx) mx = logit;
                }
                if (n_seen == 0) {
                    for (int k = 0; k < head_dim; ++k) orow[k] = 0.0;
                    *lrow = -INFINITY;
                    continue;
                }
                double sum = 0.0;
                for (int64_t t = 0; t < visible; ++t)
                    if (s[t] != -INFINITY) sum += exp(s[t] - mx);
                double l = mx + log(sum);
                for (int k = 0; k < head_dim; ++k) acc[k] = 0.0;
                for (int64_t t = 0; t < visible; ++t) {
                    if (s[t] == -INFINITY) continue;
                    double w = exp(s[t] - l);
                    const uint16_t* vr = token_row(&c, b, t, 1, kvh);
                    for (int k = 0; k < head_dim; ++k) acc[k] += w * decode(vr[k], dtype);
                }
                for (int k = 0; k < head_dim; ++k) orow[k] = acc[k];
                *lrow = l;
            }
        }
        free(s);
        free(qv);
        free(acc);
    }
    free(mask_off);
    return failed ? ORACLE_NO_MEM : ORACLE_OK;
}

/*
 * merge_state over num_states attention states of n rows each.
 * o: [num_states][n][d]; lse: [num_states][n]; outputs o_out [n][d], lse_out [n].
 */
void pkv_oracle_merge_states(int64_t num_states, int64_t n, int64_t d, const double* o,
                             const double* lse, double* o_out, double* lse_out) {
    for (int64_t r = 0; r < n; ++r) {
        double m = -INFINITY;
        for (int64_t k = 0; k < num_states; ++k)
            if (lse[k * n + r] > m) m = lse[k * n + r];
        double* out = o_out + r * d;
        if (m == -INFINITY) {
            for (int64_t j = 0; j < d; ++j) out[j] = 0.0;
            lse_out[r] = -INFINITY;
            continue;
        }
        double total = 0.0;
        for (int64_t k = 0; k < num_states; ++k) total += exp(lse[k * n + r] - m);
        double l = m + log(total);
        for (int64_t j = 0; j < d; ++j) out[j] = 0.0;
        for (int64_t k = 0; k < num_states; ++k) {
            double w = exp(lse[k * n + r] - l);
            if (w == 0.0) continue;
            const double* in = o + (k * n + r) * d;
            for (int64_t j = 0; j < d; ++j) out[j] += w * in[j];
        }
        lse_out[r] = l;
    }
}

int pkv_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
