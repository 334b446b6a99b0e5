/*
 * per_oracle.c -- the plain serial CPU oracle.  TEST INFRASTRUCTURE ONLY:
 * only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline arm load
 * it; the CUDA library never does.  See per_oracle.h for the sources and the
 * meaning of every function.
 *
 * Everything here is written for a reader checking it against the pages by
 * eye: serial loops, no blocking, no reordering.  Compile with
 * -O2 -ffp-contract=off (no fused multiply-add; IEEE round-to-nearest).
 */
#include "per_oracle.h"

#include <math.h>
#include <stddef.h>
#include <stdlib.h>

/* ------------------------------------------------------------------------ */
/* Philox [PHILOX]: a 10-round product of multiply-hi/lo bijections keyed by a
 * Weyl sequence.  Constants are the ones the paper publishes for the 4x32
 * and 4x64 variants. */

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)x0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

static void mulhilo64(uint64_t a, uint64_t b, uint64_t* hi, uint64_t* lo) {
    /* schoolbook 64x64 -> 128 with 32-bit limbs (portable, no __int128) */
    uint64_t a_lo = a & 0xffffffffu, a_hi = a >> 32;
    uint64_t b_lo = b & 0xffffffffu, b_hi = b >> 32;
    uint64_t ll = a_lo * b_lo, lh = a_lo * b_hi, hl = a_hi * b_lo, hh = a_hi * b_hi;
    uint64_t mid = (ll >> 32) + (lh & 0xffffffffu) + (hl & 0xffffffffu);
    *lo = (mid << 32) | (ll & 0xffffffffu);
    *hi = hh + (lh >> 32) + (hl >> 32) + (mid >> 32);
}

void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
    uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t hi0, lo0, hi1, lo1;
        mulhilo64(0xD2E7470EE14C6C93ull, x0, &hi0, &lo0);
        mulhilo64(0xCA5A826395121157ull, x2, &hi1, &lo1);
        uint64_t y0 = hi1 ^ x1 ^ k0;
        uint64_t y1 = lo1;
        uint64_t y2 = hi0 ^ x3 ^ k1;
        uint64_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += 0x9E3779B97F4A7C15ull;
        k1 += 0xBB67AE8584CAA73Bull;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

uint32_t oracle_philox_word(uint64_t seed, uint64_t offset, uint64_t k) {
    uint64_t c = offset + k;
    uint32_t ctr[4] = {(uint32_t)c, (uint32_t)(c >> 32), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return out[0];
}

float oracle_u01_open_closed(uint64_t seed, uint64_t offset, uint64_t k) {
    uint32_t x = oracle_philox_word(seed, offset, k);
    return (float)((double)((x >> 8) + 1u) / 16777216.0); /* exact: 24-bit integer / 2^24 */
}

float oracle_u01_closed_open(uint64_t seed, uint64_t offset, uint64_t k) {
    uint32_t x = oracle_philox_word(seed, offset, k);
    return (float)((double)(x >> 8) / 16777216.0);
}

/* ------------------------------------------------------------------------ */
/* Scan path: priority^alpha, the CDF, thresholds and searchsorted. */

void oracle_pow_alpha64(const float* p, int64_t n, double alpha, double* pa) {
    for (int64_t i = 0; i < n; ++i) pa[i] = pow((double)p[i], alpha);
}

void oracle_cdf64(const float* p, int64_t n, double alpha, double* C) {
    /* [PR615] "one thread serially prefix-summing B floats": the serial result
     * the parallel scan is measured against, here in fp64. */
    double run = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        run = run + pow((double)p[i], alpha);
        C[i] = run;
    }
}

void oracle_thresholds(int64_t B, uint64_t seed, uint64_t offset, const float* u01,
                       float T, float* u_out) {
    const float fB = (float)B;
    for (int64_t k = 0; k < B; ++k) {
        float U = u01 ? u01[k] : oracle_u01_open_closed(seed, offset, (uint64_t)k);
        float a = (float)k + U;     /* fl32(k + U) */
        float b = a / fB;           /* fl32(. / B) */
        float u = b * T;            /* fl32(. * T) */
        u_out[k] = u;
    }
}

/* i.i.d. thresholds (foxhunt "CUDA Kernels": each sampling thread draws its
 * own threshold in [0, total)): u_k = fl32(U_k * T), U_k from the same Philox
 * stream as the stratified thresholds (or u01). */
void oracle_thresholds_iid(int64_t B, uint64_t seed, uint64_t offset, const float* u01,
                           float T, float* u_out) {
    for (int64_t k = 0; k < B; ++k) {
        float U = u01 ? u01[k] : oracle_u01_open_closed(seed, offset, (uint64_t)k);
        u_out[k] = U * T;           /* fl32(U * T) */
    }
}

int64_t oracle_lower_bound_f32(const float* c, int64_t n, float u) {
    int64_t lo = 0, hi = n; /* first i in [lo,hi) with c[i] >= u */
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (c[mid] < u) lo = mid + 1; else hi = mid;
    }
    return lo < n ? lo : n - 1;
}

int64_t oracle_lower_bound_f64(const double* c, int64_t n, double u) {
    int64_t lo = 0, hi = n;
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (c[mid] < u) lo = mid + 1; else hi = mid;
    }
    return lo < n ? lo : n - 1;
}

void oracle_sample_cdf_f32(const float* c, int64_t n, int64_t B, uint64_t seed,
                           uint64_t offset, const float* u01, int32_t* idx, float* u_out) {
    float T = c[n - 1];
    float* u = (float*)malloc((size_t)B * sizeof(float));
    oracle_thresholds(B, seed, offset, u01, T, u);
    for (int64_t k = 0; k < B; ++k) {
        idx[k] = (int32_t)oracle_lower_bound_f32(c, n, u[k]);
        if (u_out) u_out[k] = u[k];
    }
    free(u);
}

void oracle_sample_cdf_f64(const double* C, int64_t n, int64_t B, uint64_t seed,
                           uint64_t offset, const float* u01, int32_t* idx, float* u_out) {
    float T = (float)C[n - 1];
    float* u = (float*)malloc((size_t)B * sizeof(float));
    oracle_thresholds(B, seed, offset, u01, T, u);
    for (int64_t k = 0; k < B; ++k) {
        idx[k] = (int32_t)oracle_lower_bound_f64(C, n, (double)u[k]);
        if (u_out) u_out[k] = u[k];
    }
    free(u);
}

/* ------------------------------------------------------------------------ */

void oracle_apply_updates(float* prio, const int32_t* idx, const float* p, int64_t n) {
    for (int64_t k = 0; k < n; ++k) prio[idx[k]] = p[k];
}

/* ------------------------------------------------------------------------ */
/* Sum segment tree [SEGTREE]: index 0 unused, root 1, children 2j and 2j+1,
 * leaf for item i at cap_pow2 + i, capacity rounded up to a power of two. */

void oracle_tree_leaves(const float* p, int64_t n, double alpha, int64_t cap_pow2, float* leaves) {
    for (int64_t i = 0; i < cap_pow2; ++i)
        leaves[i] = i < n ? (float)pow((double)p[i], alpha) : 0.0f;
}

void oracle_tree_build(const float* leaves, int64_t cap_pow2, float* tree) {
    tree[0] = 0.0f;
    for (int64_t i = 0; i < cap_pow2; ++i) tree[cap_pow2 + i] = leaves[i];
    for (int64_t j = cap_pow2 - 1; j >= 1; --j) tree[j] = tree[2 * j] + tree[2 * j + 1];
}

int64_t oracle_tree_descend(const float* tree, int64_t cap_pow2, float u) {
    int64_t j = 1;
    while (j < cap_pow2) {
        float L = tree[2 * j];
        float R = tree[2 * j + 1];
        if (u > L && R > 0.0f) {
            u = u - L;
            j = 2 * j + 1;
        } else {
            j = 2 * j;
        }
    }
    return j - cap_pow2;
}

void oracle_sample_tree(const float* tree, int64_t cap_pow2, int64_t B, uint64_t seed,
                        uint64_t offset, const float* u01, int iid, int32_t* idx, float* u_out) {
    float T = tree[1];
    float* u = (float*)malloc((size_t)B * sizeof(float));
    if (iid) oracle_thresholds_iid(B, seed, offset, u01, T, u);
    else oracle_thresholds(B, seed, offset, u01, T, u);
    for (int64_t k = 0; k < B; ++k) {
        idx[k] = (int32_t)oracle_tree_descend(tree, cap_pow2, u[k]);
        if (u_out) u_out[k] = u[k];
    }
    free(u);
}

/* ------------------------------------------------------------------------ */

void oracle_is_weights(const float* p, int64_t n_valid, double alpha, const int32_t* idx,
                       int64_t B, double beta, double* w) {
    double total = 0.0;
    for (int64_t i = 0; i < n_valid; ++i) total += pow((double)p[i], alpha);
    double wmax = 0.0;
    for (int64_t k = 0; k < B; ++k) {
        double P = pow((double)p[idx[k]], alpha) / total;
        w[k] = pow((double)n_valid * P, -beta);
        if (w[k] > wmax) wmax = w[k];
    }
    for (int64_t k = 0; k < B; ++k) w[k] = w[k] / wmax;
}

/* ------------------------------------------------------------------------ */
/* Row-batched systematic resampling [PF]. */

static float row_threshold(int64_t j, float U, int64_t P) {
    float a = (float)j + U;   /* fl32(j + U) */
    return a / (float)P;      /* fl32(. / P) */
}

void oracle_resample_row(const float* lw, int64_t P, float U, double* C, int32_t* idx,
                         float* u_out) {
    double m = -INFINITY;
    for (int64_t i = 0; i < P; ++i) if ((double)lw[i] > m) m = (double)lw[i];
    double s = 0.0;
    for (int64_t i = 0; i < P; ++i) s += exp((double)lw[i] - m);
    double* c = C ? C : (double*)malloc((size_t)P * sizeof(double));
    double run = 0.0;
    for (int64_t i = 0; i < P; ++i) {
        run += exp((double)lw[i] - m) / s;
        c[i] = run;
    }
    for (int64_t j = 0; j < P; ++j) {
        float u = row_threshold(j, U, P);
        idx[j] = (int32_t)oracle_lower_bound_f64(c, P, (double)u);
        if (u_out) u_out[j] = u;
    }
    if (!C) free(c);
}

void oracle_resample_row_on_cdf(const float* c, int64_t P, float U, int32_t* idx) {
    for (int64_t j = 0; j < P; ++j) idx[j] = (int32_t)oracle_lower_bound_f32(c, P, row_threshold(j, U, P));
}

void oracle_resample(const float* lw, int64_t rows, int64_t P, uint64_t seed, uint64_t offset,
                     const float* u_rows, int32_t* idx) {
    for (int64_t b = 0; b < rows; ++b) {
        float U = u_rows ? u_rows[b] : oracle_u01_closed_open(seed, offset, (uint64_t)b);
        oracle_resample_row(lw + b * P, P, U, NULL, idx + b * P, NULL);
    }
}

/* The rest of the particle-filter resample step (POPCORNBENCH particle
 * filter, reference forward: the resampled particles are gathered along the
 * particle axis and the log-weights of the new set are all -log P):
 * out_state[b][j][:] = state[b][idx[b][j]][:], out_logw[b][j] = fl32(-log P). */
void oracle_resample_gather(const float* state, int64_t rows, int64_t P, int64_t D, const int32_t* idx,
                            float* out_state, float* out_logw) {
    const float reset = (float)(-log((double)P));
    for (int64_t b = 0; b < rows; ++b) {
        for (int64_t j = 0; j < P; ++j) {
            const int64_t i = idx[b * P + j];
            for (int64_t d = 0; d < D; ++d) out_state[(b * P + j) * D + d] = state[(b * P + i) * D + d];
            if (out_logw) out_logw[b * P + j] = reset;
        }
    }
}

/* ---- rank-based PER ------------------------------------------------------
 * Named on the segment-tree page ("Non-Goals": rank-based PER is a separate
 * code path) without a definition; the reading used here is the standard one:
 * rank 1 is the highest stored priority (ties: lower index first), item i's
 * priority is 1 / rank(i), and the proportional machinery (p^alpha, CDF,
 * stratified thresholds, IS weights) runs over ranks. */

static const float* g_rank_p; /* comparator context (the oracle is single-threaded) */

static int rank_cmp(const void* a, const void* b) {
    const int32_t i = *(const int32_t*)a, j = *(const int32_t*)b;
    const float pi = g_rank_p[i] + 0.0f, pj = g_rank_p[j] + 0.0f; /* -0 ranks as +0 */
    if (pi > pj) return -1;
    if (pi < pj) return 1;
    return (i > j) - (i < j);
}

/* order[r] = the item of rank r + 1. */
void oracle_rank_order(const float* p, int64_t n, int32_t* order) {
    for (int64_t i = 0; i < n; ++i) order[i] = (int32_t)i;
    g_rank_p = p;
    qsort(order, (size_t)n, sizeof(int32_t), rank_cmp);
}

/* q[r] = fl32(1 / (r + 1)): the priority of rank r + 1. */
void oracle_rank_priorities(int64_t n, float* q) {
    for (int64_t r = 0; r < n; ++r) q[r] = 1.0f / (float)(r + 1);
}
