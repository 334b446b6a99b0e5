/*
 * per_oracle.h -- plain, serial CPU oracle for proportional prioritized
 * experience replay sampling (cdf_scan).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this library: only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline arm may.  It shares no code with the CUDA library (no common
 * headers, helpers, tables or constants); the only thing both sides see is
 * the seeded synthetic input generator in workloads/.
 *
 * Arithmetic: fp64 wherever the method does not itself fix the precision;
 * fp32 exactly where the definition is an fp32 expression (the sampling
 * thresholds and the fp32 pairwise sum tree).  Built with -ffp-contract=off
 * so that no multiply-add is fused.
 *
 * Sources (page title, section):
 *   [PR615]  PufferLib PR #615 "trainer: parallel build_cdf scan + tiled
 *            mingru backward", section 1 "Parallel build_cdf".
 *   [SEGTREE] foxhunt design doc "GPU Segment Tree for PER Sampling",
 *            sections "Tree Layout", "Operations", "Integration".
 *   [PF]     POPCORNBENCH trace Kimi-K2.6 / l2_p48 (fused particle filter),
 *            the reference forward's resampling steps (logsumexp, exp,
 *            cumsum, u=(arange+rand)/P, searchsorted, clamp).
 *   [PHILOX] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 *            as 1, 2, 3", SC'11 (the Philox-4x32 and 4x64 bijections).
 *
 * Parity pins: every function below is pinned by a CPU test in
 * tests/test_oracle.py against something other than itself (closed forms,
 * exact integer arithmetic, brute-force enumeration, and the independent
 * Philox implementations of cuRAND's host generator (4x32) and numpy (4x64)).
 */
#ifndef PER_ORACLE_H
#define PER_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- counter-based RNG [PHILOX] -------------------------------------- */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]);
/* First Philox4x32-10 word for key=seed, counter=(offset+k as 64 bits, 0, 0). */
uint32_t oracle_philox_word(uint64_t seed, uint64_t offset, uint64_t k);
/* U in (0,1]: ((x>>8)+1) * 2^-24.  Used for PER thresholds. */
float oracle_u01_open_closed(uint64_t seed, uint64_t offset, uint64_t k);
/* U in [0,1): (x>>8) * 2^-24.  Used for row resampling (torch.rand range). */
float oracle_u01_closed_open(uint64_t seed, uint64_t offset, uint64_t k);

/* ---- PER scan path ----------------------------------------------------- */
/* pa_i = pow(p_i, alpha) in fp64 (C pow: pow(0,0)=1). */
void oracle_pow_alpha64(const float* p, int64_t n, double alpha, double* pa);
/* C_i = sum_{j<=i} pow(p_j, alpha), serial left-to-right fp64 [PR615]. */
void oracle_cdf64(const float* p, int64_t n, double alpha, double* C);
/* Stratified thresholds u_k = fl32(fl32(fl32(k + U_k) / B) * T), U_k in
 * (0,1] from Philox (or u01[k] when u01 != NULL).  fp32 throughout. */
void oracle_thresholds(int64_t B, uint64_t seed, uint64_t offset, const float* u01,
                       float T, float* u_out);
/* i.i.d. thresholds u_k = fl32(U_k * T), U_k as above (foxhunt "CUDA
 * Kernels": one threshold per sampling thread, uniform over the total). */
void oracle_thresholds_iid(int64_t B, uint64_t seed, uint64_t offset, const float* u01,
                           float T, float* u_out);
/* searchsorted(right=False) == lower_bound; returns n-1 when every c[i] < u
 * (the clamp of [PF]). */
int64_t oracle_lower_bound_f32(const float* c, int64_t n, float u);
int64_t oracle_lower_bound_f64(const double* c, int64_t n, double u);
/* Sample B stratified indices by searching an fp32 CDF (T = c[n-1]). */
void oracle_sample_cdf_f32(const float* c, int64_t n, int64_t B, uint64_t seed,
                           uint64_t offset, const float* u01, int32_t* idx, float* u_out);
/* Sample B stratified indices by searching the fp64 CDF C (T = fl32(C[n-1])). */
void oracle_sample_cdf_f64(const double* C, int64_t n, int64_t B, uint64_t seed,
                           uint64_t offset, const float* u01, int32_t* idx, float* u_out);

/* ---- priority updates ---------------------------------------------------- */
/* Apply updates in batch order: prio[idx[k]] = p[k]; a later duplicate wins. */
void oracle_apply_updates(float* prio, const int32_t* idx, const float* p, int64_t n);

/* ---- sum segment tree [SEGTREE] ---------------------------------------- */
/* fl32(pow(p, alpha)) leaves for i<n, zero padding up to cap_pow2. */
void oracle_tree_leaves(const float* p, int64_t n, double alpha, int64_t cap_pow2, float* leaves);
/* tree[0..2*cap_pow2): tree[cap_pow2+i] = leaves[i]; tree[j] = fl32(tree[2j] +
 * tree[2j+1]) for j = cap_pow2-1 .. 1; tree[0] = 0 (unused). */
void oracle_tree_build(const float* leaves, int64_t cap_pow2, float* tree);
/* Root-to-leaf descent: at node j with children L=tree[2j], R=tree[2j+1]:
 * if (u > L and R > 0) { u = fl32(u - L); j = 2j+1 } else j = 2j.
 * Returns the leaf index j - cap_pow2. */
int64_t oracle_tree_descend(const float* tree, int64_t cap_pow2, float u);
/* B samples with T = tree[1]: stratified thresholds, or with iid != 0 the
 * i.i.d. thresholds of oracle_thresholds_iid. */
void oracle_sample_tree(const float* tree, int64_t cap_pow2, int64_t B, uint64_t seed,
                        uint64_t offset, const float* u01, int iid, int32_t* idx, float* u_out);

/* ---- importance-sampling weights --------------------------------------- */
/* P_i = pa_i / sum_{j<n_valid} pa_j (fp64); w_k = (n_valid * P_{idx_k})^-beta,
 * then divided by max_k w_k. */
void oracle_is_weights(const float* p, int64_t n_valid, double alpha, const int32_t* idx,
                       int64_t B, double beta, double* w);

/* ---- row-batched systematic resampling [PF] ---------------------------- */
/* One row of P log-weights: m = max, s = sum exp(lw - m), w = exp(lw - m)/s,
 * C = cumsum(w) (fp64), u_j = fl32(fl32(j + U)/P), idx_j = lower_bound(C, u_j)
 * clamped to P-1.  C may be NULL. */
void oracle_resample_row(const float* lw, int64_t P, float U, double* C, int32_t* idx,
                         float* u_out);
/* Same thresholds, searched on a given fp32 row CDF c (P values). */
void oracle_resample_row_on_cdf(const float* c, int64_t P, float U, int32_t* idx);
/* rows x P, U_b = u_rows[b] or Philox (offset + b) in [0,1). */
void oracle_resample(const float* lw, int64_t rows, int64_t P, uint64_t seed, uint64_t offset,
                     const float* u_rows, int32_t* idx);
/* Rank-based PER (reading: rank 1 = highest priority, ties by lower index;
 * priority of rank r is 1/r; then the proportional path over ranks).
 * order[r] = item of rank r + 1; q[r] = fl32(1 / (r + 1)). */
void oracle_rank_order(const float* p, int64_t n, int32_t* order);
void oracle_rank_priorities(int64_t n, float* q);

/* Gather of the resampled particles and reset of the log-weights (the rest
 * of the particle filter's resample step): state and out_state are
 * float32[rows][P][D], idx int32[rows][P]; out_logw (may be NULL)
 * float32[rows][P] = fl32(-log P). */
void oracle_resample_gather(const float* state, int64_t rows, int64_t P, int64_t D, const int32_t* idx,
                            float* out_state, float* out_logw);

#ifdef __cplusplus
}
#endif
#endif
