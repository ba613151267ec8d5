/*
 * CPU oracle for sparse flash attention (top-K index form and block-sparse
 * BSR form).  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark call it; the product path never does.
 * It shares no code, header or constant with the CUDA library.
 *
 * Arithmetic is IEEE double throughout.  Inputs are the same fp16 / bf16
 * buffers the GPU reads, widened exactly to double; outputs are double.
 * The steps follow the pages' definitions in their order, one query row at a
 * time, with a plain two-pass softmax (no online rescaling, no blocking):
 *
 *   Top-K form -- "SparseFlashAttention 算子 API 描述":
 *     §2 算子定义 / 稀疏机制: each (b, n2, s1) owns topK int32 positions in
 *         [0, S2), shared by the N1/N2 query heads of that KV head.
 *     §2 具体子步骤: sparse gather of K and V rows, GQA expansion (query head
 *         n1 reads KV head n1 / (N1/N2), as the golden's unsqueeze/expand/
 *         reshape does), scaled dot product (scores = (q . k_sel) * scale),
 *         optional causal mask, softmax over the topK slots, weighted sum.
 *     §2 因果掩码 and §3 规则与约束: with is_causal, slot i of query row s1
 *         is masked when idx > s1 + (S2 - S1) (bottom-right aligned
 *         diagonal; idx equal to the diagonal stays visible).
 *     §3 规则与约束 and §5 (nan_to_num): a row whose slots are all masked
 *         outputs 0.
 *     §2 布局说明: BSND and BNSD layouts for every tensor, sparseIndices
 *         included.
 *     §3 语义约束: value may be the prefix view key[..., :Dv]; `ldv` is the
 *         element distance between consecutive value rows (Dv for a separate
 *         contiguous value tensor, Dk for the prefix view).
 *   Block-sparse form -- "flashinfer.sparse", BlockSparseAttentionWrapper:
 *     the class description (scipy bsr_matrix convention, any block R x C)
 *     and plan(): indptr has MB + 1 = ceil(M / R) + 1 entries, indices hold
 *     block columns < NB = N / C; query row i may attend key column j iff
 *     block (i / R, j / C) is stored.  num_qo_heads is a multiple of
 *     num_kv_heads (grouped-query attention, qo head h reads kv head
 *     h / (Hq / Hkv)).
 *     plan() `mask` (nnz, R, C): element (r, c) of the k-th stored block (in
 *     indices order) says whether query row (i / R) * R + r may attend key
 *     column indices[k] * C + c; `packed_mask` is that tensor flattened and
 *     bit-packed.  Bit order within a byte is not given on the page: read as
 *     most significant bit first (element e is bit 7 - e % 8 of byte e / 8).
 *     plan() `causal`: applied only when no mask is given; read as the same
 *     bottom-right rule the prefill page pins with its tril example (key
 *     column j visible to query row i iff j <= i + (N - M)).
 *   LSE -- run() / run_return_lse(): "log-sum-exp of attention logits".
 *     Read as the natural logarithm of sum_j exp(scaled logit j) over the
 *     unmasked positions; -inf for a fully masked row.
 *   Soft cap -- plan() `logits_soft_cap` of both block-sparse wrappers: when
 *     cap > 0 a logit x becomes cap * tanh(x / cap).  The page does not say
 *     whether x includes sm_scale; read as the scaled logit sm_scale * q.k
 *     (the softmax input), so the LSE is over the capped logits.
 *   FP8 -- BlockSparseAttentionWrapper plan() `q_data_type` / `kv_data_type`
 *     and run() `scale_q` [num_qo_heads], `scale_k`, `scale_v`
 *     [num_kv_heads] ("per-head quantisation scales, for FP8"; 1.0 when not
 *     given); the formats are the two the operator page's precision table
 *     names, E4M3 and E5M2.  Read as dequantisation: the value an element
 *     stands for is its decoded code times its head's scale, and attention
 *     runs on those values (q of qo head h times scale_q[h], k and v of kv
 *     head g times scale_k[g] and scale_v[g]).
 *
 * Return codes: 0 ok, -1 bad argument, -2 an index outside [0, S2) (the
 * operator spec makes in-range indices a precondition).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_INDEX (-2)

/* IEEE binary16 -> double, exact. */
static double oracle_f16(uint16_t h) {
    int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(m + 1024), e - 25);
    return sign ? -v : v;
}

/* bfloat16 -> double, exact (bf16 is the top half of a binary32). */
static double oracle_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double oracle_load(const uint16_t* p, int64_t i, int dtype) {
    return dtype == 1 ? oracle_bf16(p[i]) : oracle_f16(p[i]);
}

/* The 8-bit floating-point formats, decoded exactly:
 *   E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities, the
 *         all-ones exponent with mantissa 7 is NaN (largest finite 448);
 *         exponent 0 is subnormal, m/8 * 2^-6.
 *   E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits with IEEE rules
 *         (exponent 31: infinity for mantissa 0, else NaN; largest finite
 *         57344); exponent 0 is subnormal, m/4 * 2^-14. */
static double oracle_e4m3(uint8_t c) {
    const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);               /* (m / 8) 2^-6 */
    else v = ldexp((double)(8 + m), e - 10);            /* (1 + m / 8) 2^(e - 7) */
    return sign ? -v : v;
}

static double oracle_e5m2(uint8_t c) {
    const int sign = c >> 7, e = (c >> 2) & 31, m = c & 3;
    double v;
    if (e == 31) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -16);         /* (m / 4) 2^-14 */
    else v = ldexp((double)(4 + m), e - 17);            /* (1 + m / 4) 2^(e - 15) */
    return sign ? -v : v;
}

/* Element i of a tensor of element type `dtype`: 0 f16, 1 bf16, 2 E4M3,
 * 3 E5M2. */
static double oracle_elem(const void* p, int64_t i, int dtype) {
    switch (dtype) {
        case 0: return oracle_f16(((const uint16_t*)p)[i]);
        case 1: return oracle_bf16(((const uint16_t*)p)[i]);
        case 2: return oracle_e4m3(((const uint8_t*)p)[i]);
        default: return oracle_e5m2(((const uint8_t*)p)[i]);
    }
}

/* Decoded values of `n` codes of `dtype` (the pins read the decoders through
 * this). */
void oracle_decode(const void* codes, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_elem(codes, i, dtype);
}

typedef struct {
    int B, S1, S2, N1, N2, Dk, Dv, topK, layout, causal, dtype;
    int64_t ldv;
    double scale;
} oracle_sfa_shape;

/* Element offsets of one head-row in each tensor (§2 布局说明). */
static int64_t off_q(const oracle_sfa_shape* s, int b, int n1, int s1) {
    return s->layout == 0 ? (((int64_t)b * s->S1 + s1) * s->N1 + n1) * s->Dk
                          : (((int64_t)b * s->N1 + n1) * s->S1 + s1) * s->Dk;
}
static int64_t row_kv(const oracle_sfa_shape* s, int b, int n2, int s2) {
    return s->layout == 0 ? ((int64_t)b * s->S2 + s2) * s->N2 + n2
                          : ((int64_t)b * s->N2 + n2) * s->S2 + s2;
}
static int64_t off_idx(const oracle_sfa_shape* s, int b, int n2, int s1) {
    return s->layout == 0 ? (((int64_t)b * s->S1 + s1) * s->N2 + n2) * s->topK
                          : (((int64_t)b * s->N2 + n2) * s->S1 + s1) * s->topK;
}
static int64_t row_out(const oracle_sfa_shape* s, int b, int n1, int s1) {
    return s->layout == 0 ? ((int64_t)b * s->S1 + s1) * s->N1 + n1
                          : ((int64_t)b * s->N1 + n1) * s->S1 + s1;
}

/*
 * One output row (b, n1, s1) of the top-K form, written to y_row[0..Dv) and
 * *lse_row.  `scores` and `weights` are caller scratch of topK doubles.
 */
static int oracle_sfa_row(const oracle_sfa_shape* s, const uint16_t* q, const uint16_t* k,
                          const uint16_t* v, const int32_t* idx, int b, int n1, int s1,
                          double* scores, double* weights, double* y_row, double* lse_row) {
    const int G = s->N1 / s->N2;
    const int n2 = n1 / G;                       /* GQA expansion */
    const int32_t* si = idx + off_idx(s, b, n2, s1);
    const int64_t qo = off_q(s, b, n1, s1);
    const int diag = s1 + (s->S2 - s->S1);       /* bottom-right diagonal */
    int any_visible = 0;

    /* Sparse gather + scaled dot product + causal mask. */
    for (int i = 0; i < s->topK; ++i) {
        int32_t id = si[i];
        if (id < 0 || id >= s->S2) return ORACLE_BAD_INDEX;
        const int64_t ko = row_kv(s, b, n2, id) * s->Dk;
        double dot = 0.0;
        for (int d = 0; d < s->Dk; ++d)
            dot += oracle_load(q, qo + d, s->dtype) * oracle_load(k, ko + d, s->dtype);
        scores[i] = dot * s->scale;
        if (s->causal && id > diag) scores[i] = -INFINITY;
        else any_visible = 1;
    }

    /* Softmax over the topK slots.  All slots masked: softmax is 0/0 = NaN in
     * every slot, which nan_to_num turns into 0, so the row's output is 0. */
    if (!any_visible) {
        for (int e = 0; e < s->Dv; ++e) y_row[e] = 0.0;
        if (lse_row) *lse_row = -INFINITY;
        return ORACLE_OK;
    }
    double mx = -INFINITY;
    for (int i = 0; i < s->topK; ++i) if (scores[i] > mx) mx = scores[i];
    double sum = 0.0;
    for (int i = 0; i < s->topK; ++i) {
        weights[i] = exp(scores[i] - mx);        /* exp(-inf) = 0 for masked */
        sum += weights[i];
    }
    for (int i = 0; i < s->topK; ++i) weights[i] /= sum;
    if (lse_row) *lse_row = mx + log(sum);

    /* Weighted sum of the gathered value rows. */
    for (int e = 0; e < s->Dv; ++e) y_row[e] = 0.0;
    for (int i = 0; i < s->topK; ++i) {
        const int64_t vo = row_kv(s, b, n2, si[i]) * s->ldv;
        for (int e = 0; e < s->Dv; ++e)
            y_row[e] += weights[i] * oracle_load(v, vo + e, s->dtype);
    }
    return ORACLE_OK;
}

static int oracle_sfa_check(const oracle_sfa_shape* s) {
    if (s->B < 1 || s->S1 < 1 || s->S2 < 1 || s->N1 < 1 || s->N2 < 1 || s->Dk < 1 ||
        s->Dv < 1 || s->topK < 1)
        return ORACLE_BAD_ARG;
    if (s->N1 % s->N2 != 0 || s->Dv > s->Dk || s->ldv < s->Dv) return ORACLE_BAD_ARG;
    if (s->layout != 0 && s->layout != 1) return ORACLE_BAD_ARG;
    if (s->dtype != 0 && s->dtype != 1) return ORACLE_BAD_ARG;
    if (s->causal && s->S1 > s->S2) return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

/*
 * Full top-K sparse attention.  y has the output's shape in `layout`
 * ([B,S1,N1,Dv] for BSND, [B,N1,S1,Dv] for BNSD); lse (nullable) is
 * [B,S1,N1] or [B,N1,S1].
 */
int oracle_sfa(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t ldv,
               const int32_t* idx, int B, int S1, int S2, int N1, int N2, int Dk, int Dv,
               int topK, double scale, int layout, int causal, int dtype, double* y,
               double* lse) {
    oracle_sfa_shape s = {B, S1, S2, N1, N2, Dk, Dv, topK, layout, causal, dtype, ldv, scale};
    int rc = oracle_sfa_check(&s);
    if (rc) return rc;
    const int64_t rows = (int64_t)B * N1 * S1;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)topK);
        double* weights = (double*)malloc(sizeof(double) * (size_t)topK);
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            int b = (int)(r / ((int64_t)N1 * S1));
            int n1 = (int)((r / S1) % N1);
            int s1 = (int)(r % S1);
            int64_t o = row_out(&s, b, n1, s1);
            int e = (scores && weights)
                        ? oracle_sfa_row(&s, q, k, v, idx, b, n1, s1, scores, weights,
                                         y + o * Dv, lse ? lse + o : NULL)
                        : ORACLE_BAD_ARG;
            if (e) {
#pragma omp atomic write
                err = e;
            }
        }
        free(scores);
        free(weights);
    }
    return err;
}

/*
 * Selected rows only: rows[3*r .. 3*r+2] = (b, n1, s1).  y_rows is
 * nrows x Dv, lse_rows (nullable) nrows.
 */
int oracle_sfa_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t ldv,
                    const int32_t* idx, int B, int S1, int S2, int N1, int N2, int Dk, int Dv,
                    int topK, double scale, int layout, int causal, int dtype,
                    const int64_t* rows, int64_t nrows, double* y_rows, double* lse_rows) {
    oracle_sfa_shape s = {B, S1, S2, N1, N2, Dk, Dv, topK, layout, causal, dtype, ldv, scale};
    int rc = oracle_sfa_check(&s);
    if (rc) return rc;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)topK);
        double* weights = (double*)malloc(sizeof(double) * (size_t)topK);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            int b = (int)rows[3 * r], n1 = (int)rows[3 * r + 1], s1 = (int)rows[3 * r + 2];
            int e;
            if (b < 0 || b >= B || n1 < 0 || n1 >= N1 || s1 < 0 || s1 >= S1 || !scores || !weights)
                e = ORACLE_BAD_ARG;
            else
                e = oracle_sfa_row(&s, q, k, v, idx, b, n1, s1, scores, weights,
                                   y_rows + r * Dv, lse_rows ? lse_rows + r : NULL);
            if (e) {
#pragma omp atomic write
                err = e;
            }
        }
        free(scores);
        free(weights);
    }
    return err;
}

/* ---------------------------------------------------------------------- */
/* Block-sparse (BSR) form.  q: (M, Hq, d), k/v: (N, Hkv, d), NHD; y: (M, Hq, d);
 * lse: (M, Hq). */

typedef struct {
    int M, N, R, C, Hq, Hkv, d;
    int q_dtype, kv_dtype;        /* element types of q and of k / v (oracle_elem codes) */
    double scale;
    const uint8_t* packed_mask;   /* NULL: every stored block is full */
    int causal;                   /* used only without a mask */
    double softcap;               /* > 0: logits become softcap * tanh(logit / softcap) */
    const double* scale_q;        /* [Hq] or NULL (1.0): dequantisation scale of q */
    const double* scale_k;        /* [Hkv] or NULL */
    const double* scale_v;        /* [Hkv] or NULL */
} oracle_bsr_shape;

/* plan()'s logits_soft_cap ("flashinfer.sparse", both wrappers): a logit x
 * (the scaled score sm_scale * q.k) becomes cap * tanh(x / cap) when cap > 0. */
static double oracle_soft_cap(double x, double cap) { return cap > 0.0 ? cap * tanh(x / cap) : x; }

static int oracle_bsr_check(const oracle_bsr_shape* s, const int32_t* indptr,
                            const int32_t* indices) {
    if (s->M < 1 || s->N < 1 || s->R < 1 || s->C < 1 || s->Hq < 1 || s->Hkv < 1 || s->d < 1)
        return ORACLE_BAD_ARG;
    if (s->N % s->C != 0 || s->Hq % s->Hkv != 0) return ORACLE_BAD_ARG;
    if (s->q_dtype < 0 || s->q_dtype > 3 || s->kv_dtype < 0 || s->kv_dtype > 3)
        return ORACLE_BAD_ARG;
    const int MB = (s->M + s->R - 1) / s->R, NB = s->N / s->C;
    if (indptr[0] != 0) return ORACLE_BAD_ARG;
    for (int i = 0; i < MB; ++i) {
        if (indptr[i + 1] < indptr[i]) return ORACLE_BAD_ARG;
        for (int j = indptr[i]; j < indptr[i + 1]; ++j)
            if (indices[j] < 0 || indices[j] >= NB) return ORACLE_BAD_INDEX;
    }
    return ORACLE_OK;
}

/* One output row (query row i, qo head h).  `allowed` is caller scratch of N
 * bytes, `scores` of N doubles. */
static void oracle_bsr_row(const oracle_bsr_shape* s, const void* q, const void* k,
                           const void* v, const int32_t* indptr, const int32_t* indices,
                           int i, int h, unsigned char* allowed, double* scores, double* y_row,
                           double* lse_row) {
    const int kvh = h / (s->Hq / s->Hkv);
    const int br = i / s->R;
    /* The dense mask row: column j allowed iff its block (br, j / C) is stored
     * and, with a mask, its element (i % R, j % C) of that block is set. */
    memset(allowed, 0, (size_t)s->N);
    for (int jj = indptr[br]; jj < indptr[br + 1]; ++jj)
        for (int c = 0; c < s->C; ++c) {
            unsigned char ok = 1;
            if (s->packed_mask) {
                const int64_t e = ((int64_t)jj * s->R + (i - br * s->R)) * s->C + c;
                ok = (unsigned char)((s->packed_mask[e >> 3] >> (7 - (e & 7))) & 1);
            }
            allowed[(int64_t)indices[jj] * s->C + c] = ok;
        }
    if (!s->packed_mask && s->causal)
        for (int j = 0; j < s->N; ++j)
            if ((int64_t)j > (int64_t)i + (s->N - s->M)) allowed[j] = 0;

    /* dequantisation scales of this row's qo head and kv head */
    const double sq = s->scale_q ? s->scale_q[h] : 1.0;
    const double sk = s->scale_k ? s->scale_k[kvh] : 1.0;
    const double sv = s->scale_v ? s->scale_v[kvh] : 1.0;
    const int64_t qo = ((int64_t)i * s->Hq + h) * s->d;
    double mx = -INFINITY;
    for (int j = 0; j < s->N; ++j) {
        if (!allowed[j]) continue;
        const int64_t ko = ((int64_t)j * s->Hkv + kvh) * s->d;
        double dot = 0.0;
        for (int e = 0; e < s->d; ++e)
            dot += (sq * oracle_elem(q, qo + e, s->q_dtype)) *
                   (sk * oracle_elem(k, ko + e, s->kv_dtype));
        scores[j] = oracle_soft_cap(dot * s->scale, s->softcap);
        if (scores[j] > mx) mx = scores[j];
    }
    for (int e = 0; e < s->d; ++e) y_row[e] = 0.0;
    if (mx == -INFINITY) {               /* no stored block in this row: output 0 */
        if (lse_row) *lse_row = -INFINITY;
        return;
    }
    double sum = 0.0;
    for (int j = 0; j < s->N; ++j) {
        if (!allowed[j]) continue;
        scores[j] = exp(scores[j] - mx);
        sum += scores[j];
    }
    for (int j = 0; j < s->N; ++j) {
        if (!allowed[j]) continue;
        const double w = scores[j] / sum;
        const int64_t vo = ((int64_t)j * s->Hkv + kvh) * s->d;
        for (int e = 0; e < s->d; ++e) y_row[e] += w * (sv * oracle_elem(v, vo + e, s->kv_dtype));
    }
    if (lse_row) *lse_row = mx + log(sum);
}

int oracle_bsr_cap(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* indptr,
                   const int32_t* indices, const uint8_t* packed_mask, int causal, int M, int N,
                   int R, int C, int Hq, int Hkv, int d, double scale, double softcap, int dtype,
                   double* y, double* lse) {
    oracle_bsr_shape s = {M, N, R, C, Hq, Hkv, d, dtype, dtype, scale, packed_mask, causal,
                          softcap, NULL, NULL, NULL};
    int rc = oracle_bsr_check(&s, indptr, indices);
    if (rc) return rc;
    const int64_t rows = (int64_t)M * Hq;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        unsigned char* allowed = (unsigned char*)malloc((size_t)N);
        double* scores = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            if (!allowed || !scores) {
#pragma omp atomic write
                err = ORACLE_BAD_ARG;
                continue;
            }
            int i = (int)(r / Hq), h = (int)(r % Hq);
            oracle_bsr_row(&s, q, k, v, indptr, indices, i, h, allowed, scores, y + r * d,
                           lse ? lse + r : NULL);
        }
        free(allowed);
        free(scores);
    }
    return err;
}

int oracle_bsr_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* indptr,
                  const int32_t* indices, const uint8_t* packed_mask, int causal, int M, int N,
                  int R, int C, int Hq, int Hkv, int d, double scale, int dtype, double* y,
                  double* lse) {
    return oracle_bsr_cap(q, k, v, indptr, indices, packed_mask, causal, M, N, R, C, Hq, Hkv, d,
                          scale, 0.0, dtype, y, lse);
}

int oracle_bsr(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* indptr,
               const int32_t* indices, int M, int N, int R, int C, int Hq, int Hkv, int d,
               double scale, int dtype, double* y, double* lse) {
    return oracle_bsr_ex(q, k, v, indptr, indices, NULL, 0, M, N, R, C, Hq, Hkv, d, scale, dtype,
                         y, lse);
}

/* Selected rows only: rows[2*r], rows[2*r+1] = (query row i, qo head h). */
int oracle_bsr_rows_cap(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const int32_t* indptr, const int32_t* indices, const uint8_t* packed_mask,
                        int causal, int M, int N, int R, int C, int Hq, int Hkv, int d,
                        double scale, double softcap, int dtype, const int64_t* rows,
                        int64_t nrows, double* y_rows, double* lse_rows) {
    oracle_bsr_shape s = {M, N, R, C, Hq, Hkv, d, dtype, dtype, scale, packed_mask, causal,
                          softcap, NULL, NULL, NULL};
    int rc = oracle_bsr_check(&s, indptr, indices);
    if (rc) return rc;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        unsigned char* allowed = (unsigned char*)malloc((size_t)N);
        double* scores = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            int i = (int)rows[2 * r], h = (int)rows[2 * r + 1];
            if (!allowed || !scores || i < 0 || i >= M || h < 0 || h >= Hq) {
#pragma omp atomic write
                err = ORACLE_BAD_ARG;
                continue;
            }
            oracle_bsr_row(&s, q, k, v, indptr, indices, i, h, allowed, scores, y_rows + r * d,
                           lse_rows ? lse_rows + r : NULL);
        }
        free(allowed);
        free(scores);
    }
    return err;
}

int oracle_bsr_rows_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* indptr, const int32_t* indices, const uint8_t* packed_mask,
                       int causal, int M, int N, int R, int C, int Hq, int Hkv, int d, double scale,
                       int dtype, const int64_t* rows, int64_t nrows, double* y_rows,
                       double* lse_rows) {
    return oracle_bsr_rows_cap(q, k, v, indptr, indices, packed_mask, causal, M, N, R, C, Hq, Hkv,
                               d, scale, 0.0, dtype, rows, nrows, y_rows, lse_rows);
}

int oracle_bsr_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const int32_t* indptr, const int32_t* indices, int M, int N, int R, int C,
                    int Hq, int Hkv, int d, double scale, int dtype, const int64_t* rows,
                    int64_t nrows, double* y_rows, double* lse_rows) {
    return oracle_bsr_rows_ex(q, k, v, indptr, indices, NULL, 0, M, N, R, C, Hq, Hkv, d, scale,
                              dtype, rows, nrows, y_rows, lse_rows);
}

/* Block-sparse attention with element types of their own for q and k / v
 * (any of f16, bf16, E4M3, E5M2) and run()'s per-head dequantisation scales
 * (each NULL = 1.0).  rows = NULL: every (i, h) row in order, y (M, Hq, d);
 * else rows[2r], rows[2r+1] = (query row i, qo head h), y (nrows, d). */
int oracle_bsr_scaled(const void* q, const void* k, const void* v, const int32_t* indptr,
                      const int32_t* indices, const uint8_t* packed_mask, int causal, int M, int N,
                      int R, int C, int Hq, int Hkv, int d, double scale, double softcap,
                      int q_dtype, int kv_dtype, const double* scale_q, const double* scale_k,
                      const double* scale_v, const int64_t* rows, int64_t nrows, double* y,
                      double* lse) {
    oracle_bsr_shape s = {M, N, R, C, Hq, Hkv, d, q_dtype, kv_dtype, scale, packed_mask, causal,
                          softcap, scale_q, scale_k, scale_v};
    int rc = oracle_bsr_check(&s, indptr, indices);
    if (rc) return rc;
    const int64_t n = rows ? nrows : (int64_t)M * Hq;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        unsigned char* allowed = (unsigned char*)malloc((size_t)N);
        double* scores = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n; ++r) {
            const int i = rows ? (int)rows[2 * r] : (int)(r / Hq);
            const int h = rows ? (int)rows[2 * r + 1] : (int)(r % Hq);
            if (!allowed || !scores || i < 0 || i >= M || h < 0 || h >= Hq) {
#pragma omp atomic write
                err = ORACLE_BAD_ARG;
                continue;
            }
            oracle_bsr_row(&s, q, k, v, indptr, indices, i, h, allowed, scores, y + r * d,
                           lse ? lse + r : NULL);
        }
        free(allowed);
        free(scores);
    }
    return err;
}

/* ---------------------------------------------------------------------- */
/* Variable block-sparse form -- "flashinfer.sparse",
 * VariableBlockSparseAttentionWrapper: per kv head g, the query rows are cut
 * into MB blocks of sizes row_sz[g][0..MB) and the key columns into NB blocks
 * of sizes col_sz[g][0..NB); query row i of qo head h (kv head
 * g = h / (Hq / Hkv)) may attend key column j iff
 * mask_map[g][row block of i][column block of j].  plan() `causal`: read as
 * the bottom-right rule (j visible to i iff j <= i + (N - M)), applied on top
 * of the block mask.  Layouts as run(): q (Hq, M, d), k / v (Hkv, N, d)
 * (HND); y (Hq, M, d) and lse (Hq, M) follow q's layout (the page's return
 * description prints [M, num_qo_heads, head_dim]; read as q's own layout).
 * mask_map bytes are 0 / nonzero.  Every g's row sizes sum to M and column
 * sizes to N (else -1). */
typedef struct {
    const uint16_t *q, *k, *v;
    const uint8_t* mask_map;
    const int32_t *row_sz, *col_sz;
    int MB, NB, M, N, Hq, Hkv, d, causal, dtype;
    double scale;
    double softcap;               /* > 0: soft-capped logits, as oracle_soft_cap */
} varbsr_problem;

/* Row r = h * M + i of the variable block-sparse output (y_row: d values).
 * colblk, scores, allowed: N-element scratch. */
static void varbsr_row(const varbsr_problem* s, int64_t r, int* colblk, double* scores,
                       unsigned char* allowed, double* y_row, double* lse_row) {
    const int G = s->Hq / s->Hkv;
    const int h = (int)(r / s->M), i = (int)(r % s->M), g = h / G;
    const int MB = s->MB, NB = s->NB, N = s->N, M = s->M, d = s->d;
    const int32_t *row_sz = s->row_sz, *col_sz = s->col_sz;
    /* row block of i, column block of every j, for kv head g */
    int rb = 0, acc = 0;
    while (acc + row_sz[(int64_t)g * MB + rb] <= i) acc += row_sz[(int64_t)g * MB + rb++];
    for (int cb = 0, j = 0; cb < NB; ++cb)
        for (int c = 0; c < col_sz[(int64_t)g * NB + cb]; ++c) colblk[j++] = cb;
    double mx = -INFINITY;
    for (int j = 0; j < N; ++j) {
        allowed[j] = s->mask_map[((int64_t)g * MB + rb) * NB + colblk[j]] != 0;
        if (s->causal && (int64_t)j > (int64_t)i + (N - M)) allowed[j] = 0;
        if (!allowed[j]) continue;
        double dot = 0.0;
        for (int e = 0; e < d; ++e)
            dot += oracle_load(s->q, ((int64_t)h * M + i) * d + e, s->dtype) *
                   oracle_load(s->k, ((int64_t)g * N + j) * d + e, s->dtype);
        scores[j] = oracle_soft_cap(dot * s->scale, s->softcap);
        if (scores[j] > mx) mx = scores[j];
    }
    for (int e = 0; e < d; ++e) y_row[e] = 0.0;
    if (mx == -INFINITY) {
        if (lse_row) *lse_row = -INFINITY;
        return;
    }
    double sum = 0.0;
    for (int j = 0; j < N; ++j)
        if (allowed[j]) {
            scores[j] = exp(scores[j] - mx);
            sum += scores[j];
        }
    for (int j = 0; j < N; ++j) {
        if (!allowed[j]) continue;
        const double w = scores[j] / sum;
        for (int e = 0; e < d; ++e) y_row[e] += w * oracle_load(s->v, ((int64_t)g * N + j) * d + e, s->dtype);
    }
    if (lse_row) *lse_row = mx + log(sum);
}

static int varbsr_setup(varbsr_problem* s) {
    const int MB = s->MB, NB = s->NB;
    if (MB < 1 || NB < 1 || s->M < 1 || s->N < 1 || s->Hq < 1 || s->Hkv < 1 || s->d < 1 ||
        s->Hq % s->Hkv != 0)
        return ORACLE_BAD_ARG;
    if (s->dtype != 0 && s->dtype != 1) return ORACLE_BAD_ARG;
    for (int g = 0; g < s->Hkv; ++g) {
        int64_t sr = 0, sc = 0;
        for (int b = 0; b < MB; ++b) {
            if (s->row_sz[(int64_t)g * MB + b] < 0) return ORACLE_BAD_ARG;
            sr += s->row_sz[(int64_t)g * MB + b];
        }
        for (int b = 0; b < NB; ++b) {
            if (s->col_sz[(int64_t)g * NB + b] < 0) return ORACLE_BAD_ARG;
            sc += s->col_sz[(int64_t)g * NB + b];
        }
        if (sr != s->M || sc != s->N) return ORACLE_BAD_ARG;
    }
    return ORACLE_OK;
}

/* Rows rows[0..n) (each h * M + i) of the output: y (n, d), lse (n);
 * softcap > 0 soft-caps the logits. */
int oracle_varbsr_rows_cap(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const uint8_t* mask_map, const int32_t* row_sz, const int32_t* col_sz,
                           int MB, int NB, int M, int N, int Hq, int Hkv, int d, int causal,
                           double scale, double softcap, int dtype, const int64_t* rows, int64_t n,
                           double* y, double* lse) {
    varbsr_problem s = {q, k, v, mask_map, row_sz, col_sz, MB, NB, M, N, Hq, Hkv, d, causal, dtype,
                        scale, softcap};
    int err = varbsr_setup(&s);
    if (err != ORACLE_OK) return err;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= (int64_t)Hq * M) return ORACLE_BAD_ARG;
#pragma omp parallel
    {
        int* colblk = (int*)malloc(sizeof(int) * (size_t)N);
        double* scores = (double*)malloc(sizeof(double) * (size_t)N);
        unsigned char* allowed = (unsigned char*)malloc((size_t)N);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < n; ++t) {
            if (!colblk || !scores || !allowed) {
#pragma omp atomic write
                err = ORACLE_BAD_ARG;
                continue;
            }
            varbsr_row(&s, rows[t], colblk, scores, allowed, y + t * d, lse ? lse + t : NULL);
        }
        free(colblk);
        free(scores);
        free(allowed);
    }
    return err;
}

/* The whole output: y (Hq, M, d), lse (Hq, M); softcap > 0 soft-caps the logits. */
int oracle_varbsr_cap(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      const uint8_t* mask_map, const int32_t* row_sz, const int32_t* col_sz, int MB,
                      int NB, int M, int N, int Hq, int Hkv, int d, int causal, double scale,
                      double softcap, int dtype, double* y, double* lse) {
    varbsr_problem s = {q, k, v, mask_map, row_sz, col_sz, MB, NB, M, N, Hq, Hkv, d, causal, dtype,
                        scale, softcap};
    int err = varbsr_setup(&s);
    if (err != ORACLE_OK) return err;
#pragma omp parallel
    {
        int* colblk = (int*)malloc(sizeof(int) * (size_t)N);
        double* scores = (double*)malloc(sizeof(double) * (size_t)N);
        unsigned char* allowed = (unsigned char*)malloc((size_t)N);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < (int64_t)Hq * M; ++r) {
            if (!colblk || !scores || !allowed) {
#pragma omp atomic write
                err = ORACLE_BAD_ARG;
                continue;
            }
            varbsr_row(&s, r, colblk, scores, allowed, y + r * d, lse ? lse + r : NULL);
        }
        free(colblk);
        free(scores);
        free(allowed);
    }
    return err;
}

int oracle_varbsr(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                  const uint8_t* mask_map, const int32_t* row_sz, const int32_t* col_sz, int MB,
                  int NB, int M, int N, int Hq, int Hkv, int d, int causal, double scale,
                  int dtype, double* y, double* lse) {
    return oracle_varbsr_cap(q, k, v, mask_map, row_sz, col_sz, MB, NB, M, N, Hq, Hkv, d, causal,
                             scale, 0.0, dtype, y, lse);
}

int oracle_varbsr_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const uint8_t* mask_map, const int32_t* row_sz, const int32_t* col_sz,
                       int MB, int NB, int M, int N, int Hq, int Hkv, int d, int causal,
                       double scale, int dtype, const int64_t* rows, int64_t n, double* y,
                       double* lse) {
    return oracle_varbsr_rows_cap(q, k, v, mask_map, row_sz, col_sz, MB, NB, M, N, Hq, Hkv, d,
                                  causal, scale, 0.0, dtype, rows, n, y, lse);
}
