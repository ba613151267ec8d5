/*
 * Seeded synthetic inputs for sparse flash attention workloads.
 *
 * This file generates random numbers and index lists only; it contains none of
 * the attention arithmetic.  Every value is a pure function of (seed, stream,
 * counter), so the same call gives the same bytes on any machine and any
 * thread count.  Both the CPU oracle and the CUDA path consume the buffers it
 * fills (the Python wrapper rounds the float32 normals to fp16/bf16 once, and
 * those rounded buffers go to both sides).
 *
 * Generator: the splitmix64 output function (Steele, Lea & Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014; constants as in
 * Vigna's public-domain splitmix64.c) applied to a Weyl sequence, used here as
 * a counter-based hash.  Normals: Box-Muller (Box & Muller 1958) on 53-bit
 * uniforms.  Bounded integers: Lemire's multiply-shift on 64-bit draws.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYN_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t syn_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of one independent stream: hash of (seed, stream id). */
static inline uint64_t syn_key(uint64_t seed, uint64_t stream) {
    return syn_mix(syn_mix(seed + SYN_GOLDEN) ^ (stream * 0xD1B54A32D192ED03ULL));
}

/* The counter-th 64-bit draw of a stream. */
static inline uint64_t syn_draw(uint64_t key, uint64_t counter) {
    return syn_mix(key + SYN_GOLDEN * (counter + 1));
}

/* Uniform on (0, 1]: 53 random bits, never 0 so that log() is finite. */
static inline double syn_unit(uint64_t r) {
    return ((double)(r >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}

/* Uniform integer in [0, n) for 0 < n < 2^32 (multiply-shift). */
static inline uint32_t syn_below(uint64_t r, uint32_t n) {
    return (uint32_t)(((r >> 32) * (uint64_t)n) >> 32);
}

/* n float32 samples of N(0,1).  Element 2j and 2j+1 are the cosine and sine
 * halves of Box-Muller pair j, which uses draws 2j and 2j+1 of the stream. */
void syn_normal_f32(uint64_t seed, uint64_t stream, int64_t n, float* out) {
    const uint64_t key = syn_key(seed, stream);
    const int64_t npairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < npairs; ++j) {
        double u1 = syn_unit(syn_draw(key, 2 * (uint64_t)j));
        double u2 = syn_unit(syn_draw(key, 2 * (uint64_t)j + 1));
        double rad = sqrt(-2.0 * log(u1));
        double ang = 6.283185307179586476925 * u2;
        out[2 * j] = (float)(rad * cos(ang));
        if (2 * j + 1 < n) out[2 * j + 1] = (float)(rad * sin(ang));
    }
}

static int syn_cmp_i32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Draw `count` distinct values from [lo, lo + range) into out (random order),
 * by a partial Fisher-Yates shuffle of scratch[0..range).  Draws are taken from
 * stream `key` starting at counter `*ctr`, which advances. */
static void syn_distinct(uint64_t key, uint64_t* ctr, int32_t lo, int32_t range,
                         int32_t count, int32_t* scratch, int32_t* out) {
    for (int32_t i = 0; i < range; ++i) scratch[i] = lo + i;
    for (int32_t i = 0; i < count; ++i) {
        uint32_t j = (uint32_t)i + syn_below(syn_draw(key, (*ctr)++), (uint32_t)(range - i));
        int32_t t = scratch[i]; scratch[i] = scratch[j]; scratch[j] = t;
        out[i] = scratch[i];
    }
}

/* Shuffle out[0..n) in place (Fisher-Yates). */
static void syn_shuffle(uint64_t key, uint64_t* ctr, int32_t* a, int32_t n) {
    for (int32_t i = n - 1; i > 0; --i) {
        uint32_t j = syn_below(syn_draw(key, (*ctr)++), (uint32_t)(i + 1));
        int32_t t = a[i]; a[i] = a[j]; a[j] = t;
    }
}

/*
 * rows x topk index lists, each `topk` distinct values drawn uniformly from
 * [0, range) in random order (sorted ascending if `sorted` != 0).  Row r uses
 * its own stream (seed, r), so rows are independent of the row count.
 */
int syn_index_uniform(uint64_t seed, int64_t rows, int32_t range, int32_t topk,
                      int sorted, int32_t* out) {
    if (topk < 0 || range <= 0 || topk > range) return -1;
    int err = 0;
#pragma omp parallel
    {
        int32_t* scratch = (int32_t*)malloc(sizeof(int32_t) * (size_t)range);
        if (!scratch) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(static)
            for (int64_t r = 0; r < rows; ++r) {
                uint64_t key = syn_key(seed, (uint64_t)r), ctr = 0;
                int32_t* row = out + r * (int64_t)topk;
                syn_distinct(key, &ctr, 0, range, topk, scratch, row);
                if (sorted) qsort(row, (size_t)topk, sizeof(int32_t), syn_cmp_i32);
            }
            free(scratch);
        }
    }
    return err;
}

/*
 * Index lists with a causal structure, for a [B, S1, N2, topK] (BSND order)
 * index tensor over a key length S2 >= S1.  Row (b, s1, n2) has diagonal
 * d = s1 + S2 - S1: positions [0, d] are visible, (d, S2) lie above the
 * bottom-right diagonal.
 *   - rows with b == 0 and s1 < full_masked_rows: all topK drawn WITH
 *     replacement from (d, S2) (so the whole row is masked; duplicates occur);
 *   - other rows: n_above = min(round(masked_frac * topK), |(d, S2)|) distinct
 *     positions from (d, S2) and topK - n_above distinct from [0, d], then the
 *     row is shuffled.
 * Returns -1 if some row cannot be filled.
 */
int syn_index_causal_mix(uint64_t seed, int32_t B, int32_t S1, int32_t N2, int32_t S2,
                         int32_t topk, double masked_frac, int32_t full_masked_rows,
                         int32_t* out) {
    if (S1 > S2 || topk <= 0) return -1;
    int32_t n_above_nominal = (int32_t)floor(masked_frac * (double)topk + 0.5);
    int err = 0;
    const int64_t rows = (int64_t)B * S1 * N2;
#pragma omp parallel
    {
        int32_t* scratch = (int32_t*)malloc(sizeof(int32_t) * (size_t)S2);
        if (!scratch) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(static)
            for (int64_t r = 0; r < rows; ++r) {
                int32_t b = (int32_t)(r / ((int64_t)S1 * N2));
                int32_t s1 = (int32_t)((r / N2) % S1);
                int32_t d = s1 + (S2 - S1);
                int32_t above = S2 - 1 - d;
                uint64_t key = syn_key(seed, (uint64_t)r), ctr = 0;
                int32_t* row = out + r * (int64_t)topk;
                if (b == 0 && s1 < full_masked_rows) {
                    if (above <= 0) {
#pragma omp atomic write
                        err = -1;
                        continue;
                    }
                    for (int32_t i = 0; i < topk; ++i)
                        row[i] = d + 1 + (int32_t)syn_below(syn_draw(key, ctr++), (uint32_t)above);
                    continue;
                }
                int32_t n_above = n_above_nominal < above ? n_above_nominal : above;
                int32_t n_vis = topk - n_above;
                if (n_vis > d + 1) {
#pragma omp atomic write
                    err = -1;
                    continue;
                }
                if (n_above > 0) syn_distinct(key, &ctr, d + 1, above, n_above, scratch, row);
                syn_distinct(key, &ctr, 0, d + 1, n_vis, scratch, row + n_above);
                syn_shuffle(key, &ctr, row, topk);
            }
            free(scratch);
        }
    }
    return err;
}

/*
 * Block-sparse row structure over MB x NB blocks: block (i, i) is always
 * present (when i < NB); every other block independently with probability p.
 * Writes indptr[MB + 1] and, if indices != NULL, the column indices in CSR
 * order with columns ascending.  Returns nnz.
 */
int64_t syn_bsr_pattern(uint64_t seed, int32_t MB, int32_t NB, double p,
                        int32_t* indptr, int32_t* indices) {
    const uint64_t key = syn_key(seed, 0);
    const uint64_t thresh = (p >= 1.0) ? UINT64_MAX : (uint64_t)(p * 18446744073709551616.0);
    int64_t nnz = 0;
    indptr[0] = 0;
    for (int32_t i = 0; i < MB; ++i) {
        for (int32_t j = 0; j < NB; ++j) {
            int on = (i == j) || (syn_draw(key, (uint64_t)i * (uint64_t)NB + (uint64_t)j) < thresh);
            if (on) {
                if (indices) indices[nnz] = j;
                ++nnz;
            }
        }
        indptr[i + 1] = (int32_t)nnz;
    }
    return nnz;
}
