/*
 * per.h -- C ABI of the GB300 (sm_103a) proportional prioritized-experience-
 * replay sampling library.
 *
 * What it computes (sources by page title and section):
 *   - PufferLib PR #615 "trainer: parallel build_cdf scan + tiled mingru
 *     backward", section 1 "Parallel build_cdf": the prioritized-replay CDF
 *     is an inclusive prefix sum of the B priorities, rebuilt once per
 *     minibatch update, and must stay allocation- and sync-free.
 *   - foxhunt "GPU Segment Tree for PER Sampling": sections "Tree Layout"
 *     (flat array, root 1, children 2j/2j+1, leaf of item i at
 *     capacity_pow2+i, capacity rounded up to a power of two), "Operations"
 *     (batched update = write leaves then recompute parent sums; sample =
 *     root-to-leaf descent going left when the threshold is <= the left sum),
 *     "Integration" (priority^alpha folded into the update; insert_batch;
 *     update_priorities; total_priority = tree[1]), "Non-Goals" (alpha, beta
 *     and the IS weights themselves are unchanged PER).
 *   - POPCORNBENCH Kimi-K2.6 / l2_p48 particle-filter trace: the reference
 *     forward's resampling -- logsumexp normalisation, exp, cumsum over the
 *     particle axis, systematic thresholds u_j = (j + U_b)/P with one U_b per
 *     row, searchsorted(right=False), clamp to P-1.
 *
 * Conventions (every call):
 *   - Device pointers ("d_") are CUDA global-memory addresses on the device
 *     that was current when the context was created; the caller owns them and
 *     they must stay valid until the stream work that uses them completes.
 *     Host pointers are marked "h_".
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call except per_create (which allocates the context's
 *     device memory), per_total_host, per_check, per_destroy and
 *     per_build_cdf_noalloc (whose own note below governs it) is asynchronous
 *     and stream-ordered: it allocates nothing, never synchronises the host,
 *     and may be captured in a CUDA graph.
 *   - Argument errors return PER_ERR_ARG (or PER_ERR_STATE / PER_ERR_EMPTY)
 *     before anything is launched.  A failed launch returns PER_ERR_CUDA.
 *     Errors found on the device (a bounded wait that ran out, a value out of
 *     range, a negative or NaN priority) are recorded in the context's status
 *     word; per_check() reads and clears it.
 *   - Indices are int32; capacity <= 2^30.  One context must not be used by
 *     two streams at the same time (calls on one context are not
 *     thread-safe).
 *   - Randomness is explicit: a (seed, offset) pair selects Philox4x32-10
 *     counters offset+k under key seed (Salmon et al., SC'11), or the caller
 *     passes the uniforms in.  Results are bit-reproducible run to run.
 */
#ifndef PER_GB300_H
#define PER_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct per_ctx per_ctx;

typedef enum {
    PER_OK = 0,
    PER_ERR_ARG = 1,      /* bad argument (null, size, alignment, mode) */
    PER_ERR_CUDA = 2,     /* a CUDA runtime call or launch failed */
    PER_ERR_OOM = 3,      /* per_create could not allocate device memory */
    PER_ERR_TIMEOUT = 4,  /* a bounded device-side wait ran out */
    PER_ERR_EMPTY = 5,    /* nothing to sample: size 0 or total priority 0 */
    PER_ERR_STATE = 6,    /* structure not enabled in this context */
    PER_ERR_RANGE = 7,    /* a sum exceeded the exact-carry range */
    PER_ERR_VALUE = 8     /* a negative or NaN priority was seen */
} per_status;

/* Structures kept by a context (flags of per_create) and sampling modes. */
#define PER_SCAN 1u /* raw priorities + CDF built by per_build_cdf (PR #615) */
#define PER_TREE 2u /* sum segment tree of priority^alpha (foxhunt) */
#define PER_IID 4u  /* sampling-mode flag, with PER_TREE: i.i.d. thresholds (foxhunt "CUDA Kernels") */
#define PER_RANK 8u /* rank-based PER: priority 1/rank (foxhunt "Non-Goals"); a context flag on its own */

/* Human-readable name of a status code (static storage; never NULL). */
const char* per_status_str(per_status s);

/*
 * per_create -- allocate a context for `capacity` items (1 <= capacity <=
 * 2^30) with exponent `alpha` >= 0 (pa_i = p_i^alpha; foxhunt "Integration":
 * priority^alpha is applied inside the update, not kept as a separate
 * buffer).  `flags` is PER_SCAN, PER_TREE or both, or PER_RANK alone (then
 * capacity <= 2^24; see per_rank_build).  All device memory the
 * context will ever use is allocated here (raw priorities, the CDF, the tree
 * of 2*capacity_pow2 floats, scan descriptors, update scratch) and
 * zero-filled on `stream`, which is synchronised before returning.  The size
 * (number of valid items) starts at 0.  On error *out is NULL.
 */
per_status per_create(per_ctx** out, int64_t capacity, float alpha, uint32_t flags, void* stream);

/* per_destroy -- synchronise the device and free everything the context
 * owns.  NULL is accepted. */
per_status per_destroy(per_ctx* ctx);

/* per_set_size -- number of valid items n (0 <= n <= capacity): the CDF
 * covers [0, n) and IS weights use N = n.  Host-side only; nothing launched.
 * Items >= n keep whatever priority they hold (in the tree they contribute
 * their leaf value, 0 until written). */
per_status per_set_size(per_ctx* ctx, int64_t n);
int64_t per_size(const per_ctx* ctx);
int64_t per_capacity_pow2(const per_ctx* ctx);

/*
 * per_set_priorities -- bulk load: raw priorities d_prio[0..n) (float32, n <=
 * capacity, 16-byte aligned) become items 0..n-1, the size becomes n, and
 * when PER_TREE is set the tree leaves become p^alpha (zero beyond n) and all
 * internal sums are rebuilt in the fixed pairwise order of foxhunt "Tree
 * Layout".  Items >= n are reset to priority 0.
 */
per_status per_set_priorities(per_ctx* ctx, const float* d_prio, int64_t n, void* stream);

/*
 * per_update -- batched priority update (foxhunt "Operations" / Update and
 * "Integration" / update_priorities_gpu, insert_batch): for k in [0, n),
 * item d_idx[k] gets raw priority d_prio[k] (>= 0).  When an index occurs
 * more than once the LAST occurrence in batch order wins.  Updates the raw
 * priorities (read by the next per_build_cdf) and, with PER_TREE, writes leaf
 * p^alpha and recomputes every affected internal sum as tree[j] =
 * tree[2j] + tree[2j+1] -- bit-identical to rebuilding the whole tree.
 * Indices must lie in [0, capacity); the size is not changed (insert_batch
 * is per_update followed by per_set_size).  n may be 0.
 */
per_status per_update(per_ctx* ctx, const int32_t* d_idx, const float* d_prio, int32_t n,
                      void* stream);

/*
 * per_build_cdf -- PR #615 "Parallel build_cdf": cdf[i] = sum_{j<=i} p_j^alpha
 * over the n valid items, as one single-pass decoupled-lookback scan with
 * p^alpha fused into the load.  The result is monotone non-decreasing and
 * bit-reproducible (tile carries are summed exactly in 128-bit fixed point
 * with 60 fractional bits; each tile's sum of p^alpha must stay below 2^44,
 * else PER_ERR_RANGE is recorded, and a unit sum -- a tile's, or a 512-item
 * slice's in the streaming scan of large inputs -- is truncated to a
 * multiple of 2^-60 in the carries, so a unit whose sum is below 2^-60 adds
 * nothing to the items after it and its own values are clamped to the
 * carry before it).  Requires PER_SCAN and n >= 1.  The CDF is read through
 * per_cdf_ptr(); cdf[n-1] is the total.
 */
per_status per_build_cdf(per_ctx* ctx, void* stream);

/*
 * per_build_cdf_noalloc -- the build_cdf scan for callers that cannot
 * allocate device memory.  (The method's sources have no counterpart: it is
 * an interface addition of this library.)  Some callers cannot call
 * cudaMalloc -- code running inside another framework's operator or callback
 * where the host application owns all device memory through its own pool, or
 * a latency-critical loop where cudaMalloc's implicit device synchronisation
 * is not acceptable.  This call needs no context: it reads d_prio[0..n)
 * (float32, >= 0, 16-byte aligned), writes d_cdf[0..n) (16-byte aligned) =
 * the inclusive prefix sum of d_prio^alpha, with the same kernels and the
 * same bit-exact result as per_build_cdf, and allocates nothing.
 *
 * Its scratch (tile sums and tile records for the lookbacks and a few
 * counters) is a fixed ~260 KiB array compiled into the library, held by
 * every GPU that loads the library
 * until the process exits; hence n <= 16,777,216 (2^24), larger n returns
 * PER_ERR_ARG without launching.  The first call on each device performs a
 * one-time set-up with that device current (resolves the array's address,
 * clears it with two small kernels on `stream` and synchronises `stream`);
 * make that first call before any stream capture.  All calls on a device
 * share the array: calls whose work overlaps on the GPU (different streams
 * with no ordering between them) race and give wrong results -- serialise
 * them.  Device-side errors (negative/NaN priority, range, a bounded wait
 * that ran out: 1 = timeout, 2 = range, 4 = value) are OR-ed into *d_status;
 * d_status is the call's only error channel, so with d_status == NULL they
 * go unreported.  The array needs no re-arming after an error.
 */
per_status per_build_cdf_noalloc(const float* d_prio, int64_t n, float alpha, float* d_cdf, int* d_status,
                                 void* stream);

/*
 * per_rank_build -- rank-based PER (PER_RANK contexts).  foxhunt's segment-
 * tree page ("Non-Goals") lists rank-based PER as a separate code path and
 * does not define it; this library reads it as the usual rank-based variant:
 * the n valid items are ordered by descending raw priority, ties broken by
 * the lower index first (-0 and +0 are equal; priorities must be >= 0 and
 * not NaN, else PER_ERR_VALUE is recorded and the order is unspecified), the
 * item of rank r (1-based) gets priority q_r = fl32(1 / r), and everything
 * downstream is proportional PER over ranks: pa_r = q_r^alpha, the CDF
 * cdf[r-1] = sum_{s<=r} pa_s (built with the per_build_cdf scan, exact
 * carries, so bit-reproducible), stratified thresholds, IS weights.
 * The sort is a stable LSD radix sort (four 8-bit passes); it leaves
 * order[r-1] = the item of rank r (per_rank_order_ptr).  The rank CDF depends
 * only on n and alpha, so it is rebuilt only when the size changed since the
 * previous per_rank_build.  Call it after priorities change and before
 * sampling: per_sample / per_is_weights / per_total with mode PER_RANK return
 * PER_ERR_STATE when the size changed since the last per_rank_build (a
 * per_update without a new per_rank_build samples from the previous order).
 * Requires PER_RANK and size >= 1 (PER_ERR_EMPTY).
 * Above 262,144 items the last radix pass stores the inverse permutation
 * (rank of each item, used by per_is_weights) with L2 eviction priority
 * evict_last, and the call's last launch returns those lines to the normal
 * priority: once the call's work is done, L2 holds nothing at a raised
 * priority.
 */
per_status per_rank_build(per_ctx* ctx, void* stream);

/*
 * per_sample -- draw B stratified samples (1 <= B <= 2^24):
 *   u_k = fl32(fl32(fl32(k + U_k) / B) * T),  U_k in (0, 1],
 * or, with mode PER_TREE | PER_IID, B independent samples (foxhunt "CUDA
 * Kernels": one threshold per sampling thread, uniform over the total):
 *   u_k = fl32(U_k * T),
 * U_k = ((x >> 8) + 1) * 2^-24 with x the first word of Philox4x32-10 at
 * counter (offset + k, 0, 0) under key seed, or U_k = d_u01[k] when d_u01 is
 * not NULL (values in (0,1]).
 *   mode PER_SCAN: T = cdf[n-1]; idx_k = first i with cdf[i] >= u_k
 *     (searchsorted(right=False)), clamped to n-1.  Needs per_build_cdf first.
 *   mode PER_TREE: T = tree[1]; root-to-leaf descent (foxhunt "Operations" /
 *     Sample): at node j with children L, R: if u > L and R > 0 then
 *     { u = u - L; go right } else go left.
 *   mode PER_RANK: as PER_SCAN on the rank CDF (T = rank cdf[n-1]), giving a
 *     rank r_k; idx_k = order[r_k], the item of that rank.
 * d_out_idx receives int32[B].  Total 0 records PER_ERR_EMPTY.
 */
per_status per_sample(per_ctx* ctx, int32_t B, uint64_t seed, uint64_t offset, int mode,
                      const float* d_u01, int32_t* d_out_idx, void* stream);
/* (PER_IID with PER_SCAN is PER_ERR_ARG: the scan path's staged windows rely
 * on sorted thresholds.) */

/*
 * per_is_weights -- importance-sampling weights for sampled items d_idx[0..B):
 *   w_k = (N * P(idx_k))^-beta / max_k (N * P(idx_k))^-beta,
 * P(i) = pa_i / total, N = size -- computed as (pa_min / pa_{idx_k})^beta
 * with pa_min the smallest pa in the batch (the max-normalised form; N and the
 * total cancel).  pa comes from the tree leaves with PER_TREE, from
 * q_{rank(i)}^alpha in a PER_RANK context (item indices must be < size and
 * sorted by per_rank_build; others record PER_ERR_VALUE), else p^alpha of
 * the raw priorities.  d_out_w receives float32[B]; the largest weight is
 * exactly 1.  beta >= 0.  A batch containing a zero-priority item yields
 * non-finite weights.
 */
per_status per_is_weights(per_ctx* ctx, const int32_t* d_idx, int32_t B, float beta,
                          float* d_out_w, void* stream);

/*
 * per_sample_weighted -- per_sample followed by per_is_weights on the drawn
 * indices, in one call: the same arguments, checks and results as the two
 * calls, bit for bit.  On the scan path, when the CDF's coarse index fits a
 * CTA's shared memory (size <= 262,144 items), both run in one cooperative
 * launch (sampling, then the batch minimum across CTAs through one grid
 * barrier, then the weights); otherwise the two launches run in order.
 */
per_status per_sample_weighted(per_ctx* ctx, int32_t B, uint64_t seed, uint64_t offset, int mode,
                               const float* d_u01, float beta, int32_t* d_out_idx, float* d_out_w,
                               void* stream);

/*
 * per_step -- one minibatch step of proportional PER (PufferLib PR #615: the
 * prefix sum is rebuilt once per minibatch update; foxhunt "Integration":
 * update, then sample with IS weights): per_update(d_upd_idx, d_upd_prio,
 * n_upd) when n_upd > 0, then per_build_cdf (per_rank_build in a PER_RANK
 * context, mode PER_RANK), then per_sample_weighted(B,
 * seed, offset, mode, d_u01, beta, d_out_idx, d_out_w) -- the same
 * arguments, checks and results as those calls, bit for bit.  For scan-only
 * contexts (PER_SCAN without PER_TREE, mode PER_SCAN) of size <= 262,144
 * and B <= 1024 per 2048 items, the three run in one cooperative launch with
 * grid barriers between them; otherwise as the separate calls, in order.
 * n_upd >= 0; the update buffers may be NULL when n_upd == 0.  Errors as the
 * separate calls (PER_ERR_ARG before any launch).
 */
per_status per_step(per_ctx* ctx, const int32_t* d_upd_idx, const float* d_upd_prio, int32_t n_upd, int32_t B,
                    uint64_t seed, uint64_t offset, int mode, const float* d_u01, float beta, int32_t* d_out_idx,
                    float* d_out_w, void* stream);

/*
 * per_gather -- copy the sampled transitions out of a replay buffer laid out
 * as one fixed-size row per item (PufferLib PR #615 samples a minibatch of
 * transitions by index from its prioritized buffers):
 *   d_out[k][:] = d_rows[d_idx[k]][:]   for k in [0, B),
 * rows of row_bytes bytes (16 <= row_bytes <= 2^20, a multiple of 16; d_rows
 * and d_out 16-byte aligned; d_rows holds `capacity` rows).  An index outside
 * [0, capacity) records PER_ERR_VALUE and leaves its output row unwritten.
 * d_out must not overlap d_rows.
 */
per_status per_gather(per_ctx* ctx, const void* d_rows, int64_t row_bytes, const int32_t* d_idx, int32_t B,
                      void* d_out, void* stream);

/*
 * per_step_gather -- per_step followed by per_gather(d_rows, row_bytes,
 * d_out_idx, B, d_out_rows): one whole PER step that also returns the sampled
 * transitions, with the same results as the two calls.  On per_step's fused
 * path the copy runs inside the same launch (each CTA copies the rows of the
 * samples it drew); otherwise the gather is a separate launch.  When nothing
 * can be sampled (PER_ERR_EMPTY recorded) the output rows are unspecified.
 * d_rows must not be NULL.  Errors as per_step and per_gather.
 */
per_status per_step_gather(per_ctx* ctx, const int32_t* d_upd_idx, const float* d_upd_prio, int32_t n_upd, int32_t B,
                           uint64_t seed, uint64_t offset, int mode, const float* d_u01, float beta,
                           int32_t* d_out_idx, float* d_out_w, const void* d_rows, int64_t row_bytes,
                           void* d_out_rows, void* stream);

/* per_total -- total priority (foxhunt "Integration" / total_priority):
 * mode PER_TREE reads tree[1], PER_SCAN reads cdf[n-1] (after per_build_cdf),
 * PER_RANK the rank CDF's last value sum_r q_r^alpha (after per_rank_build).
 * per_total writes one float to device memory; per_total_host synchronises
 * `stream` and returns it in *h_out. */
per_status per_total(per_ctx* ctx, int mode, float* d_out, void* stream);
per_status per_total_host(per_ctx* ctx, int mode, float* h_out, void* stream);

/* Device pointers owned by the context (read-only views, valid until
 * per_destroy): raw priorities float[capacity], CDF float[capacity] (first
 * size entries meaningful), tree float[2*capacity_pow2] (NULL without
 * PER_TREE). */
const float* per_priorities_ptr(const per_ctx* ctx);
const float* per_cdf_ptr(const per_ctx* ctx);
const float* per_tree_ptr(const per_ctx* ctx);
/* PER_RANK contexts (NULL otherwise): order int32[capacity] (first size
 * entries: the item of rank 1, 2, ...) and the rank CDF float[capacity]. */
const int32_t* per_rank_order_ptr(const per_ctx* ctx);
const float* per_rank_cdf_ptr(const per_ctx* ctx);

/*
 * per_check -- synchronise `stream`, read and clear the device status word.
 * Returns PER_OK, or the first recorded error among PER_ERR_TIMEOUT,
 * PER_ERR_RANGE, PER_ERR_VALUE, PER_ERR_EMPTY.
 */
per_status per_check(per_ctx* ctx, void* stream);

/*
 * per_debug_drop_tile -- fault injection for tests of the failure path (no
 * counterpart on the pages; the failure-detection plan of this library):
 * the NEXT scan on this context -- per_build_cdf, or the scan inside
 * per_step / per_rank_build -- loses one message, as if it had been dropped:
 * in the one-wave scan (inputs that fit one wave of CTAs) tile `tile` does
 * not publish its carry word; in the streaming scan of larger inputs tile
 * `tile` does not publish its record (neither its sum nor its inclusive
 * prefix).  Every wait for it then runs out after the bounded-wait limit
 * (about 2 s): the kernels record PER_ERR_TIMEOUT (read by per_check), stop
 * waiting, finish, and leave the context usable for the next call, whose
 * result is correct again.  That call's CDF (and samples) are unspecified.
 * Tiles of the one-wave scan are 2048 items (n <= 2^19) or 4096 items, of
 * the streaming scan 16384 items; a tile the call does not have changes
 * nothing.  tile = -1 cancels.  Host-side only; the injection
 * applies to one call and is then cleared.  Never needed outside tests.
 */
per_status per_debug_drop_tile(per_ctx* ctx, int64_t tile);

/*
 * per_resample -- row-batched systematic resampling (POPCORNBENCH particle
 * filter, reference forward): d_logw is float32[rows][P] row-major (16-byte
 * aligned, 4 <= P <= 2^23, P % 4 == 0, rows >= 1).  Per row b:
 *   w_i = exp(lw_i - m) / s  (m = row max, s = sum_i exp(lw_i - m)),
 *   c = cumsum(w),  u_j = fl32(fl32(j + U_b) / P),  U_b in [0, 1)
 *   idx_j = first i with c_i >= u_j (searchsorted, right=False), clamped P-1
 * U_b = (x >> 8) * 2^-24 from Philox (offset + b) under key seed, or
 * d_u_rows[b] when not NULL.  d_out_idx (16-byte aligned) receives
 * int32[rows][P].  If d_out_cdf (16-byte aligned) is not NULL it receives the
 * float32[rows][P] CDF that was searched.  Needs no context and no scratch.
 * A row whose log-weights are all -inf or contain NaN gives unspecified
 * indices in [0, P).  A row is scanned by up to 8 CTAs (one cluster).
 * PER_ERR_ARG: null or misaligned pointers, rows < 1, P < 4, P % 4 != 0,
 * P > 2^23, or so many rows that the grid would exceed 2^31 - 1 CTAs.
 */
per_status per_resample(const float* d_logw, int32_t rows, int32_t P, uint64_t seed,
                        uint64_t offset, const float* d_u_rows, int32_t* d_out_idx,
                        float* d_out_cdf, void* stream);

/*
 * per_resample_step -- the particle filter's whole resample step
 * (POPCORNBENCH particle filter, reference forward): per_resample of d_logw
 * as above (indices to d_out_idx), then the resampled particles' states
 * gathered along the particle axis,
 *   d_out_state[b][j][:] = d_state[b][idx_j][:]   (float32[rows][P][D]),
 * and, when d_out_logw is not NULL, every log-weight of the new set reset to
 * fl32(-log P) (float32[rows][P]; d_out_logw may be d_logw itself).  One
 * launch.  d_out_state must not overlap d_state.  All pointers 16-byte
 * aligned; 1 <= D <= 4096 (D % 4 == 0 copies 16 bytes at a time).  Errors as
 * per_resample.
 */
per_status per_resample_step(const float* d_logw, const float* d_state, int32_t rows, int32_t P, int32_t D,
                             uint64_t seed, uint64_t offset, const float* d_u_rows, int32_t* d_out_idx,
                             float* d_out_state, float* d_out_logw, void* stream);

/* Number of this library's kernel launches issued by the calling process so
 * far (host-side counter; used to report launches per benchmark step). */
uint64_t per_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* PER_GB300_H */
