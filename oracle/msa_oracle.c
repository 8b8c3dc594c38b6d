/*
 * FP64 CPU oracle for MSA block-sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that tests, the smoke check and the bench's
 * CPU-baseline leg have an independent, slow, obviously correct statement of
 * what the CUDA library must compute.  It shares no code, header, table or
 * helper with the CUDA sources.
 *
 * Sources (the four pages the method is described on):
 *   [P2] vLLM PR 60684 "MSA prefill takes the E4M3 query natively":
 *        section Performance (benchmark shapes: top-16 of 128-token pages,
 *        position of a chunk's tokens at the tail of the sequence), section
 *        Details / "Scales" (q scale folds into the softmax scale, K and V
 *        scales per tensor), section Validation (acceptance rule).
 *   [P4] vLLM docs, vllm.models.minimax_m3.nvidia.sparse_attention_msa,
 *        MiniMaxM3SparseMSAImpl.forward: build_k2q_csr(prefill_topk, cu_q,
 *        cu_k, 128, total_rows=total_kv_blocks, qhead_per_kv) followed by
 *        sparse_atten_func(..., causal=True, softmax_scale, page_table=
 *        block_table, seqused_k=seq_lens).
 *
 * Everything is computed in double.  Readings of points the pages leave open
 * (each one is listed with its reason in the design notes of the repository):
 *   R1  top-k values are logical page ids of the token's own request and are
 *       mapped to physical pages through block_table[b, p];
 *   R2  the selection is per KV head and shared by its G = Hq / Hkv query
 *       heads; query head hq belongs to KV head hq / G;
 *   R4  a page listed twice counts once (set semantics);
 *   R5  a page after the token's own page contributes no key (causal mask);
 *   R6  an id >= the request's page count, or < -1, is ignored, as is a
 *       logical page whose block_table entry is outside [0, num_pages);
 *   R9  score = (q . k) * softmax_scale with q = dec(Q) * q_scale,
 *       k = dec(K) * k_scale, v = dec(V) * v_scale;
 *   R11 lse is the natural log of the sum of exp(score) over attended keys;
 *   R16 keys at or past seq_len are masked;
 *   R24 a BF16 query ([P2] Details: the BF16-Q x FP8-K/V mode stages K/V up
 *       to BF16; Overview: a BF16 query already carries q_scale) enters as
 *       q = bf16(Q) * q_scale, everything else unchanged.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_D 128
#define ORACLE_PAGE 128
#define ORACLE_TOPK 16

/* OCP 8-bit floating point, E4M3 ("FN": no infinities).  Bit 7 sign, bits
 * 6..3 exponent with bias 7, bits 2..0 mantissa.  Exponent 0 holds the
 * subnormals m * 2^-9; exponent 15 with mantissa 7 is NaN; every other code
 * is (1 + m/8) * 2^(e-7), so the largest finite magnitude is 1.75 * 2^8 = 448.
 */
double oracle_e4m3_decode(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest E4M3 value to x, ties to the even code (round to nearest even on
 * the format's grid), magnitudes past the largest finite value 448 saturated
 * to 448.  On [2^k, 2^(k+1)) the grid step is 2^(k-3) for k >= -6; below
 * 2^-6 it is the subnormal step 2^-9.  x must not be NaN. */
uint8_t oracle_e4m3_encode(double x) {
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    double q;
    if (a < ldexp(1.0, -6)) {
        q = ldexp(1.0, -9);
    } else {
        int k;
        frexp(a, &k);               /* a = f * 2^k with f in [0.5, 1) */
        q = ldexp(1.0, (k - 1) - 3);
    }
    const double n = a / q;         /* exact: q is a power of two */
    const double f = floor(n);
    const double r = n - f;
    const double m = (r > 0.5 || (r == 0.5 && fmod(f, 2.0) == 1.0)) ? f + 1.0 : f;
    const double v = m * q;         /* on the grid, <= 448 */
    if (v < ldexp(1.0, -6))         /* subnormal: m * 2^-9, m = 0..7 */
        return sign | (uint8_t)(v / ldexp(1.0, -9));
    int k;
    frexp(v, &k);
    const int e = (k - 1) + 7;      /* v in [2^(e-7), 2^(e-6)) */
    const int mant = (int)(ldexp(v, -(k - 1)) * 8.0) - 8;
    return sign | (uint8_t)((e << 3) | mant);
}

/* OCP 4-bit floating point, E2M1: bit 3 sign, bits 2..1 exponent with bias
 * 1, bit 0 mantissa.  Exponent 0 is the subnormal 0.5 * m; every other code
 * is (1 + m/2) * 2^(e-1).  The magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1_decode(uint8_t code) {
    const int sign = (code >> 3) & 1;
    const int e = (code >> 1) & 0x3;
    const int m = code & 0x1;
    const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/*
 * NVFP4 page pool -> the E4M3 pool an E4M3-query kernel reads ([P2] vLLM
 * PR 60684, Details: with an E4M3 query each NVFP4 code times its block
 * scale is dequantised to E4M3; the K and V global scales stay outside, on
 * the scores and in the combine).  kv4 holds, per (page, KV head), a K slot
 * then a V slot; a slot is 128 tokens x 64 bytes of codes (element 2i in the
 * low nibble of byte i) followed by 128 tokens x 8 E4M3 scales (scale b for
 * elements 16b .. 16b+15).  kv8 is [page][KV head][128][256], K then V.
 */
void oracle_nvfp4_to_e4m3(const uint8_t *kv4, int64_t page_heads, uint8_t *kv8) {
    const int64_t slot = ORACLE_PAGE * (ORACLE_D / 2) + ORACLE_PAGE * (ORACLE_D / 16);
#pragma omp parallel for schedule(static)
    for (int64_t ph = 0; ph < page_heads; ++ph) {
        for (int s = 0; s < 2; ++s) {
            const uint8_t *codes = kv4 + (ph * 2 + s) * slot;
            const uint8_t *scales = codes + ORACLE_PAGE * (ORACLE_D / 2);
            for (int t = 0; t < ORACLE_PAGE; ++t) {
                for (int e = 0; e < ORACLE_D; ++e) {
                    const uint8_t byte = codes[t * (ORACLE_D / 2) + e / 2];
                    const uint8_t nib = (e & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
                    const double v = oracle_e2m1_decode(nib) *
                                     oracle_e4m3_decode(scales[t * (ORACLE_D / 16) + e / 16]);
                    kv8[(ph * ORACLE_PAGE + t) * (2 * ORACLE_D) + s * ORACLE_D + e] =
                        oracle_e4m3_encode(v);
                }
            }
        }
    }
}

/* bfloat16: bit 15 sign, bits 14..7 exponent with bias 127, bits 6..0
 * mantissa.  Exponent 0 holds the subnormals m * 2^-133; exponent 255 is
 * infinity (mantissa 0) or NaN; every other code is (1 + m/128) * 2^(e-127).
 */
double oracle_bf16_decode(uint16_t code) {
    const int sign = (code >> 15) & 1;
    const int e = (code >> 7) & 0xFF;
    const int m = code & 0x7F;
    double v;
    if (e == 0xFF) return m ? NAN : (sign ? -INFINITY : INFINITY);
    if (e == 0)
        v = ldexp((double)m, -133);
    else
        v = ldexp(1.0 + (double)m / 128.0, e - 127);
    return sign ? -v : v;
}

static double g_dec[256];
static int g_dec_ready = 0;

static void init_table(void) {
    if (g_dec_ready) return;
    for (int c = 0; c < 256; ++c) g_dec[c] = oracle_e4m3_decode((uint8_t)c);
    g_dec_ready = 1;
}

/* request that owns global query token t: cu_q[b] <= t < cu_q[b+1] */
static int request_of(const int32_t *cu_q, int B, int64_t t) {
    for (int b = 0; b < B; ++b)
        if (t >= cu_q[b] && t < cu_q[b + 1]) return b;
    return -1;
}

static int cmp_int(const void *a, const void *b) {
    int x = *(const int *)a, y = *(const int *)b;
    return (x > y) - (x < y);
}

/*
 * Distinct valid logical pages selected by (token t, KV head h), ascending.
 * Returns how many were written to pages[0..15].
 */
static int selected_pages(const int32_t *topk, int Hkv, int64_t t, int h,
                          int P, const int32_t *bt_row, int64_t num_pages,
                          int pages[ORACLE_TOPK]) {
    int n = 0;
    for (int j = 0; j < ORACLE_TOPK; ++j) {
        int p = topk[(t * Hkv + h) * ORACLE_TOPK + j];
        if (p < 0 || p >= P) continue;                       /* R6, padding */
        int32_t phys = bt_row[p];
        if (phys < 0 || (int64_t)phys >= num_pages) continue; /* R6 */
        int dup = 0;
        for (int i = 0; i < n; ++i) dup |= (pages[i] == p);
        if (dup) continue;                                    /* R4 */
        pages[n++] = p;
    }
    qsort(pages, n, sizeof(int), cmp_int);
    return n;
}

/*
 * Attention for the listed query tokens (all tokens when tokens == NULL).
 *   q      [T][Hq][128]          E4M3 codes (q16 == NULL), or
 *   q16    [T][Hq][128]          bfloat16 codes (q == NULL; R24)
 *   kv     [num_pages][Hkv][128][256] E4M3 codes, K = bytes 0..127, V = 128..255
 *   topk   [T][Hkv][16]          logical page ids, -1 = padding
 *   block_table [B][bt_stride]
 *   out    [n][Hq][128], lse [n][Hq], nkeys [n][Hkv] (nullable)
 * Returns 0, or -1 when a listed token belongs to no request.
 */
static int attention_rows(const uint8_t *q, const uint16_t *q16,
                          const uint8_t *kv, int64_t num_pages,
                          const int32_t *topk, const int32_t *block_table,
                          int bt_stride, const int32_t *cu_q, const int32_t *cu_k,
                          int B, int Hq, int Hkv, double q_scale, double k_scale,
                          double v_scale, double softmax_scale,
                          const int64_t *tokens, int64_t n_tokens, double *out,
                          double *lse, int32_t *nkeys, int nthreads) {
    init_table();
    const int G = Hq / Hkv;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t w = 0; w < n_tokens * Hkv; ++w) {
        const int64_t n = w / Hkv;
        const int h = (int)(w % Hkv);
        const int64_t t = tokens ? tokens[n] : n;
        const int b = request_of(cu_q, B, t);
        if (b < 0) { bad = 1; continue; }
        const int64_t qlen = cu_q[b + 1] - cu_q[b];
        const int64_t seq = cu_k[b + 1] - cu_k[b];
        const int64_t pos = seq - qlen + (t - cu_q[b]);
        const int P = (int)((seq + ORACLE_PAGE - 1) / ORACLE_PAGE);
        const int32_t *bt_row = block_table + (int64_t)b * bt_stride;
        int pages[ORACLE_TOPK];
        const int np = selected_pages(topk, Hkv, t, h, P, bt_row, num_pages,
                                      pages);

        /* the attended key set: every key of a selected page that is not
         * after the query (causal) and not past the sequence end */
        int64_t keys[ORACLE_TOPK * ORACLE_PAGE];
        int nk = 0;
        for (int i = 0; i < np; ++i)
            for (int kk = 0; kk < ORACLE_PAGE; ++kk) {
                int64_t k = (int64_t)pages[i] * ORACLE_PAGE + kk;
                if (k <= pos && k < seq) keys[nk++] = k;
            }
        if (nkeys) nkeys[n * Hkv + h] = nk;

        double s[ORACLE_TOPK * ORACLE_PAGE];
        for (int g = 0; g < G; ++g) {
            const int hq = h * G + g;
            double *o = out + (n * Hq + hq) * ORACLE_D;
            double qv[ORACLE_D];
            for (int d = 0; d < ORACLE_D; ++d) {
                const int64_t at = (t * Hq + hq) * ORACLE_D + d;
                qv[d] = (q16 ? oracle_bf16_decode(q16[at]) : g_dec[q[at]]) * q_scale;
            }
            if (nk == 0) {
                for (int d = 0; d < ORACLE_D; ++d) o[d] = 0.0;
                lse[n * Hq + hq] = -INFINITY;
                continue;
            }
            double m = -INFINITY;
            for (int i = 0; i < nk; ++i) {
                const int64_t k = keys[i];
                const int64_t phys = bt_row[k / ORACLE_PAGE];
                const uint8_t *row =
                    kv + ((phys * Hkv + h) * ORACLE_PAGE + k % ORACLE_PAGE) *
                             (2 * ORACLE_D);
                double dot = 0.0;
                for (int d = 0; d < ORACLE_D; ++d)
                    dot += qv[d] * (g_dec[row[d]] * k_scale);
                s[i] = dot * softmax_scale;
                if (s[i] > m) m = s[i];
            }
            double sum = 0.0;
            for (int d = 0; d < ORACLE_D; ++d) o[d] = 0.0;
            for (int i = 0; i < nk; ++i) {
                const int64_t k = keys[i];
                const int64_t phys = bt_row[k / ORACLE_PAGE];
                const uint8_t *row =
                    kv + ((phys * Hkv + h) * ORACLE_PAGE + k % ORACLE_PAGE) *
                             (2 * ORACLE_D);
                const double e = exp(s[i] - m);
                sum += e;
                for (int d = 0; d < ORACLE_D; ++d)
                    o[d] += e * (g_dec[row[ORACLE_D + d]] * v_scale);
            }
            for (int d = 0; d < ORACLE_D; ++d) o[d] /= sum;
            lse[n * Hq + hq] = m + log(sum);
        }
    }
    return bad ? -1 : 0;
}

/* E4M3 query over E4M3 K/V ([P2] Overview). */
int oracle_attention(const uint8_t *q, const uint8_t *kv, int64_t num_pages,
                     const int32_t *topk, const int32_t *block_table,
                     int bt_stride, const int32_t *cu_q, const int32_t *cu_k,
                     int B, int Hq, int Hkv, double q_scale, double k_scale,
                     double v_scale, double softmax_scale,
                     const int64_t *tokens, int64_t n_tokens, double *out,
                     double *lse, int32_t *nkeys, int nthreads) {
    return attention_rows(q, NULL, kv, num_pages, topk, block_table, bt_stride,
                          cu_q, cu_k, B, Hq, Hkv, q_scale, k_scale, v_scale,
                          softmax_scale, tokens, n_tokens, out, lse, nkeys,
                          nthreads);
}

/* BF16 query over E4M3 K/V ([P2] Details: the BF16-Q x FP8-K/V mode; R24). */
int oracle_attention_bf16q(const uint16_t *q16, const uint8_t *kv,
                           int64_t num_pages, const int32_t *topk,
                           const int32_t *block_table, int bt_stride,
                           const int32_t *cu_q, const int32_t *cu_k, int B,
                           int Hq, int Hkv, double q_scale, double k_scale,
                           double v_scale, double softmax_scale,
                           const int64_t *tokens, int64_t n_tokens,
                           double *out, double *lse, int32_t *nkeys,
                           int nthreads) {
    return attention_rows(NULL, q16, kv, num_pages, topk, block_table,
                          bt_stride, cu_q, cu_k, B, Hq, Hkv, q_scale, k_scale,
                          v_scale, softmax_scale, tokens, n_tokens, out, lse,
                          nkeys, nthreads);
}

/*
 * Page-to-query CSR, by plain loops (build_k2q_csr of [P4]).
 * Row index: h * total_rows + off_b + p, off_b = sum of the page counts of
 * requests before b (total_rows = total_kv_blocks).  A row lists the query
 * tokens that selected the page, in ascending token order, each with the
 * slot j at which the page first appears in the token's list.  An entry is
 * kept when it is valid (R6), not a repeat (R4) and not after the token's own
 * page (R5).  slot_mask[t][h] has bit j set for every kept entry.
 *
 * Returns the number of entries, -1 when the requests need more rows than
 * total_rows, -2 when cap is too small.
 */
int64_t oracle_k2q_csr(const int32_t *topk, const int32_t *block_table,
                       int bt_stride, int64_t num_pages, const int32_t *cu_q,
                       const int32_t *cu_k, int B, int Hkv, int64_t total_rows,
                       int32_t *row_ptr, int32_t *q_idx, uint8_t *slot,
                       int64_t cap, uint16_t *slot_mask) {
    int64_t *off = (int64_t *)calloc((size_t)B + 1, sizeof(int64_t));
    for (int b = 0; b < B; ++b) {
        int64_t seq = cu_k[b + 1] - cu_k[b];
        off[b + 1] = off[b] + (seq + ORACLE_PAGE - 1) / ORACLE_PAGE;
    }
    if (off[B] > total_rows) { free(off); return -1; }
    const int64_t rows = (int64_t)Hkv * total_rows;
    int64_t *count = (int64_t *)calloc((size_t)rows + 1, sizeof(int64_t));
    const int64_t T = cu_q[B];

    for (int pass = 0; pass < 2; ++pass) {
        int64_t *cursor = NULL;
        if (pass == 1) {
            row_ptr[0] = 0;
            for (int64_t r = 0; r < rows; ++r)
                row_ptr[r + 1] = (int32_t)(row_ptr[r] + count[r]);
            if (row_ptr[rows] > cap) { free(count); free(off); return -2; }
            cursor = (int64_t *)calloc((size_t)rows + 1, sizeof(int64_t));
        }
        for (int b = 0; b < B; ++b) {
            const int64_t qlen = cu_q[b + 1] - cu_q[b];
            const int64_t seq = cu_k[b + 1] - cu_k[b];
            const int P = (int)((seq + ORACLE_PAGE - 1) / ORACLE_PAGE);
            const int32_t *bt_row = block_table + (int64_t)b * bt_stride;
            for (int64_t t = cu_q[b]; t < cu_q[b + 1]; ++t) {
                const int64_t pos = seq - qlen + (t - cu_q[b]);
                const int64_t own = pos / ORACLE_PAGE;
                for (int h = 0; h < Hkv; ++h) {
                    uint16_t mask = 0;
                    for (int j = 0; j < ORACLE_TOPK; ++j) {
                        int p = topk[(t * Hkv + h) * ORACLE_TOPK + j];
                        if (p < 0 || p >= P) continue;
                        int32_t phys = bt_row[p];
                        if (phys < 0 || (int64_t)phys >= num_pages) continue;
                        if (p > own) continue;
                        int dup = 0;
                        for (int i = 0; i < j; ++i)
                            dup |= (topk[(t * Hkv + h) * ORACLE_TOPK + i] == p);
                        if (dup) continue;
                        const int64_t r = (int64_t)h * total_rows + off[b] + p;
                        mask |= (uint16_t)(1u << j);
                        if (pass == 0) {
                            count[r] += 1;
                        } else {
                            const int64_t at = row_ptr[r] + cursor[r]++;
                            q_idx[at] = (int32_t)t;
                            slot[at] = (uint8_t)j;
                        }
                    }
                    if (pass == 1 && slot_mask) slot_mask[t * Hkv + h] = mask;
                }
            }
        }
        if (cursor) free(cursor);
    }
    (void)T;
    const int64_t nnz = row_ptr[rows];
    free(count);
    free(off);
    return nnz;
}

/*
 * Merge of split partials by log-sum-exp: for each row, with M the largest
 * finite lse_j, L = M + log(sum_j exp(lse_j - M)) and
 * out = sum_j exp(lse_j - L) * O_j.  Slots whose lse is -inf are empty; a
 * row with no filled slot gives out = 0 and lse = -inf.
 *   part_o [rows][S][D], part_lse [rows][S], out [rows][D], lse [rows]
 */
void oracle_combine(const double *part_o, const double *part_lse,
                    int64_t rows, int S, int D, double *out, double *lse) {
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int j = 0; j < S; ++j) {
            double l = part_lse[r * S + j];
            if (l > M) M = l;
        }
        double *o = out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (M == -INFINITY) { lse[r] = -INFINITY; continue; }
        double sum = 0.0;
        for (int j = 0; j < S; ++j) {
            double l = part_lse[r * S + j];
            if (l == -INFINITY) continue;
            sum += exp(l - M);
        }
        const double L = M + log(sum);
        for (int j = 0; j < S; ++j) {
            double l = part_lse[r * S + j];
            if (l == -INFINITY) continue;
            const double w = exp(l - L);
            for (int d = 0; d < D; ++d) o[d] += w * part_o[(r * S + j) * D + d];
        }
        lse[r] = L;
    }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
