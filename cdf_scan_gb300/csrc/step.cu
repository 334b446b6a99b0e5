// step.cu -- one PER minibatch step in one cooperative launch (scan mode):
// apply a batch of priority updates (the last occurrence of an index wins),
// rebuild the CDF of p^alpha over the buffer, and draw B stratified samples
// with their importance-sampling weights.  The CTA that scans a tile first
// applies the updates that fall in it (every CTA reads the whole batch and
// elects the last writer of each of its items in shared memory), so the
// update needs no grid barrier; the scan (scan_core.cuh) and the sampler
// with its weights (sample_core.cuh) are the ones of per_build_cdf and
// per_sample_weighted, with grid barriers where those calls had kernel
// boundaries.  The results are those of per_update + per_build_cdf +
// per_sample_weighted, bit for bit.  (PufferLib
// PR #615: the prefix sum is rebuilt once per minibatch update and CUDA-graph
// capture is the launch-overhead fix; foxhunt "GPU Segment Tree for PER
// Sampling" section "Integration": update, then sample, with the IS weights
// of the batch.)
#include "gather_core.cuh"
#include "sample_core.cuh"
#include "scan_core.cuh"

namespace {

constexpr int kStepThreads = 256;               // the one-wave scan's tile: 256 x 8 items
constexpr int kStepTile = kStepThreads * 8;

struct StepParams {
    ScanParams scan;
    // sampling and weights
    int B;
    uint64_t seed, offset;
    float alpha, beta;
    bool alpha_one;
    int32_t* __restrict__ out;
    float* __restrict__ out_w;
    // updates
    const int32_t* __restrict__ upd_idx;
    const float* __restrict__ upd_p;
    int n_upd;
    int64_t capacity;
    float* prio;                 // the buffer the updates write (== scan.p)
    unsigned long long* ticket;  // grid-barrier word
    unsigned* step_min;          // call counter, then the batch-minimum word of even and odd calls
    // optional copy of the sampled transitions: out_rows[k] = rows[out[k]]
    const uint4* rows;           // [capacity][row_chunks] x 16 bytes, or nullptr
    int row_chunks;
    uint4* out_rows;             // [B][row_chunks] x 16 bytes
};

// CTA c owns items [c * TILE, (c + 1) * TILE) (the grid is exactly the
// tiles; capacity <= tiles * TILE when there are updates):
//   0. one bulk copy brings the tile's priorities into shared memory while
//      the update batch is read;
//   1. the last batch position of each of the CTA's items is elected in
//      shared memory (atomicMax), and the winners' priorities are written
//      to the buffer and to the shared copy -- no other CTA touches these
//      items, so no grid barrier;
//   2. the tile is scanned from the shared copy (wave_scan_tile); its CDF
//      values stay in shared memory, and warp 0's lookback, which reads every
//      tile's sum word, also gives the previous tile's last CDF value, this
//      tile's and T;
//   3. with T = cdf[n-1] = fl32 of the exact total and the previous tile's
//      last value (neither waits for another tile's scan), the CTA takes
//      exactly the strata k whose
//      threshold u_k falls in (previous last, own last] -- their lower_bound
//      lies in this tile -- searches them in shared memory and computes
//      p^alpha of the hits;
//   4. the batch minimum of p^alpha goes through one atomicMin word and one
//      grid barrier, then the weights.
// With `rows`, step 3 also copies each hit's transition row to out_rows[k]
// (one warp per round's hits, gather_core.cuh) before the barrier.
// Thresholds are Philox draws (U in (0, 1]), so u_k lies within a rounding
// margin of stratum k's interval (k T/B, (k+1) T/B]; the CTA evaluates the
// strata whose interval meets its range widened by that margin.
__global__ void __launch_bounds__(kStepThreads) per_step_kernel(StepParams S) {
    constexpr int THREADS = kStepThreads, TILE = kStepTile;
    __shared__ __align__(16) float s_p[TILE];    // the tile's priorities (after the updates)
    __shared__ __align__(16) float s_cdf[TILE];  // the tile's CDF values
    __shared__ int s_win[TILE];                  // last batch position updating each item
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ unsigned s_parity;
    __shared__ float s_red[THREADS / 32];
    __shared__ float s_bound[3];  // previous tile's last value, own last value, T
    __shared__ int s_krange[2];   // strata [k_lo, k_hi) this CTA evaluates
    __shared__ float s_min;
    __shared__ int s_gk[THREADS / 32][32];  // a warp's hits for the row copy
    __shared__ int s_gi[THREADS / 32][32];

    const int c = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    const int n = static_cast<int>(S.scan.n);
    const int lo = c * TILE;
    const int valid = min(TILE, n - lo);  // >= 1
    const int bulk = valid & ~3;
    int* status = S.scan.status;

    // ---- 0. the tile's priorities ------------------------------------------
    if (threadIdx.x == 0) {
        s_parity = ld_relaxed_u32(S.step_min) & 1u;
        mbar_init(&s_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect_tx(&s_bar, static_cast<unsigned>(bulk) * 4u);
        if (bulk) bulk_copy_g2s(s_p, S.scan.p + lo, static_cast<unsigned>(bulk) * 4u, &s_bar);
    }
    if (S.n_upd > 0)
        for (int j = threadIdx.x; j < TILE; j += THREADS) s_win[j] = -1;
    __syncthreads();

    // ---- 1. the updates of this tile ----------------------------------------
    bool bad = false;
    if (S.n_upd > 0) {
        constexpr int kU = 32;  // batch positions per thread per round, loads issued first
        for (int k0 = 0; k0 < S.n_upd; k0 += THREADS * kU) {
            int32_t iv[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int k = k0 + u * THREADS + threadIdx.x;
                iv[u] = k < S.n_upd ? __ldg(S.upd_idx + k) : 0;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int k = k0 + u * THREADS + threadIdx.x;
                if (k >= S.n_upd) continue;
                const int32_t i = iv[u];
                if (i < 0 || i >= S.capacity) {
                    bad = true;  // every CTA sees it; any one of them flags it
                    continue;
                }
                if (i >= lo && i < lo + TILE) atomicMax(&s_win[i - lo], k);
            }
        }
    }
    if (!mbar_wait_bounded(&s_bar, 0)) atomicOr(status, ST_TIMEOUT);
    for (int j = bulk + threadIdx.x; j < valid; j += THREADS) s_p[j] = S.scan.p[lo + j];  // 0-3 tail items
    __syncthreads();
    if (S.n_upd > 0) {
        for (int j = threadIdx.x; j < TILE; j += THREADS) {
            const int k = s_win[j];
            if (k >= 0) {
                const float v = __ldg(S.upd_p + k);
                if (!(v >= 0.f)) bad = true;
                S.prio[lo + j] = v;
                if (j < valid) s_p[j] = v;
            }
        }
        __syncthreads();
    }
    if (bad) atomicOr(status, ST_VALUE);

    // ---- 2. the scan of this tile ---------------------------------------------
    // s_bound = the previous tile's last CDF value, this tile's, and T, from
    // warp 0's lookback alone (no other tile's local scan is waited for)
    const unsigned epoch = wave_scan_tile<THREADS>(S.scan, c, s_p, s_cdf, s_bound);
    __syncthreads();  // s_cdf complete
    if (threadIdx.x == 0) {
        if (c == 0) s_bound[0] = -__int_as_float(0x7f800000);
        const float own = s_bound[1], T = s_bound[2];
        // strata whose interval (k T/B, (k+1) T/B], widened by the rounding
        // margin of the threshold, meets (prev, own].  k = x B / T in fp32:
        // fl32(B / T) and the product each err by at most 2^-24 relative, so
        // for x <= T the computed k is within B * 2^-23 <= 2 of the exact one
        // (B <= 2^24), covered by 3 more strata of margin; the strata are
        // then decided one by one (mine), so a wider range costs only time.
        const int B = S.B;
        const int margin = 2 + (B >> 20) + 3;
        const float scale = __fdiv_rn(static_cast<float>(B), T);
        s_krange[0] = c == 0 ? 0 : max(0, __float2int_rd(__fmul_rn(s_bound[0], scale)) - margin);
        s_krange[1] = c == G - 1 ? B : min(B, __float2int_ru(__fmul_rn(own, scale)) + margin + 1);
    }
    __syncthreads();
    const float prev = s_bound[0], own = s_bound[1], T = s_bound[2];
    const int B = S.B;
    // once T is known every tile has read the epoch and published its word
    // (T needed all of them), so the epoch and the call counter may move on
    auto finish = [&]() {
        if (c == 0 && threadIdx.x == 0) {
            advance_scan_epoch(S.scan, epoch);
            S.step_min[1 + (s_parity ^ 1u)] = 0x7f800000u;  // +inf for the next call
            S.step_min[0] = S.step_min[0] + 1u;
        }
    };
    if (!(T > 0.f)) {  // nothing to sample: every CTA sees the same T
        if (c == 0 && threadIdx.x == 0) atomicOr(status, ST_EMPTY);
        const int per = (B + G - 1) / G;
        for (int k = c * per + threadIdx.x; k < min(B, (c + 1) * per); k += THREADS) S.out[k] = 0;
        finish();
        return;
    }

    // ---- 3. the strata of this tile -------------------------------------------
    const float fB = static_cast<float>(B);
    const int k_lo = s_krange[0], k_hi = s_krange[1];
    auto mine = [&](float u) { return (c == 0 || u > prev) && (c == G - 1 || u <= own); };
    float m = __int_as_float(0x7f800000);  // +inf
    int k_first = -1;                      // this thread's hit in the first round (weights from registers)
    float pa_first = 0.f;
    const int warp = threadIdx.x >> 5;
    for (int k0 = k_lo; k0 < k_hi; k0 += THREADS) {  // uniform bound: whole warps run every round
        const int k = k0 + threadIdx.x;
        bool hit = false;
        int idx = 0;
        if (k < k_hi) {
            const float u =
                stratified_threshold(k, u01_open_closed(S.seed, S.offset + static_cast<uint64_t>(k)), fB, T);
            if (mine(u)) {
                hit = true;
                idx = min(lo + smem_lower_bound(s_cdf, 0, valid, u), n - 1);
                S.out[k] = idx;
                const float pa = pow_accurate(s_p[idx - lo], S.alpha, S.alpha_one);
                m = fminf(m, pa);
                if (k0 == k_lo) {
                    k_first = k;
                    pa_first = pa;
                } else {
                    S.out_w[k] = pa;  // staged until the minimum is known
                }
            }
        }
        if (S.rows) gather_hits_warp(S.rows, S.capacity, S.row_chunks, S.out_rows, hit, k, idx, s_gk[warp], s_gi[warp]);
    }

    // ---- 4. the batch minimum, then the weights --------------------------------
    m = block_min<THREADS>(m, s_red) + 0.f;  // a -0 minimum becomes +0
    unsigned* min_word = S.step_min + 1 + s_parity;
    if (threadIdx.x == 0) atomicMin(min_word, __float_as_uint(m));
    grid_barrier(S.ticket, status, ST_TIMEOUT);
    if (threadIdx.x == 0) s_min = __uint_as_float(ld_relaxed_u32(min_word));
    __syncthreads();
    finish();
    const float pa_min = s_min;
    if (k_first >= 0) S.out_w[k_first] = powf(__fdiv_rn(pa_min, pa_first), S.beta);
    for (int k0 = k_lo + THREADS; k0 < k_hi; k0 += THREADS) {
        const int k = k0 + threadIdx.x;
        if (k >= k_hi) continue;
        const float u = stratified_threshold(k, u01_open_closed(S.seed, S.offset + static_cast<uint64_t>(k)), fB, T);
        if (mine(u)) S.out_w[k] = powf(__fdiv_rn(pa_min, __ldcg(S.out_w + k)), S.beta);
    }
}

}  // namespace

// The fused step for scan-only contexts whose CDF fits one wave of
// 2048-item tiles, with Philox thresholds; PER_ERR_STATE (nothing launched)
// when it does not apply.
per_status launch_step(per_ctx* ctx, const int32_t* upd_idx, const float* upd_p, int n_upd, int B, uint64_t seed,
                       uint64_t offset, const float* u01, float beta, int32_t* out, float* out_w, const void* rows,
                       int64_t row_bytes, void* out_rows, cudaStream_t s) {
    constexpr int TILE = kStepTile;
    const int64_t n = ctx->size;
    if (ctx->flags != PER_SCAN || u01 || !ctx->step_min || n < 1 || n > (int64_t(1) << 19)) return PER_ERR_STATE;
    const int64_t tiles = (n + TILE - 1) / TILE;
    if (tiles > ctx->scan_desc_tiles) return PER_ERR_STATE;
    // every index an update may name lies in some CTA's tile
    if (n_upd > 0 && ctx->capacity > tiles * TILE) return PER_ERR_STATE;
    static DeviceCache cache;
    const int per_sm = device_cached(cache, []() {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, per_step_kernel, kStepThreads, 0) != cudaSuccess)
            return 0;
        return b < 1 ? 1 : b;
    });
    if (per_sm == 0) return PER_ERR_CUDA;
    if (tiles > static_cast<int64_t>(per_sm) * ctx->num_sms) return PER_ERR_STATE;
    StepParams S = {};
    S.scan.p = ctx->prio;
    S.scan.cdf = ctx->cdf;
    S.scan.n = n;
    S.scan.alpha = ctx->alpha;
    S.scan.alpha_one = ctx->alpha == 1.0f;
    S.scan.pow_mode = ctx->alpha == 1.0f ? 1 : (ctx->alpha == 0.0f ? 2 : 0);
    S.scan.pow_lim = pow_limit(ctx->alpha);
    S.scan.cdf_v8 = (reinterpret_cast<uintptr_t>(ctx->cdf) & 31u) == 0;
    S.scan.desc = ctx->scan_desc;
    S.scan.desc_tiles = ctx->scan_desc_tiles;
    S.scan.ctrs = ctx->ctrs;
    S.scan.status = ctx->status;
    S.scan.num_tiles = static_cast<unsigned>(tiles);
    S.scan.coarse = ctx->coarse;
    S.scan.drop_tile = ctx->drop_tile;  // a fault injected for one call only
    ctx->drop_tile = -1;
    S.B = B;
    S.seed = seed;
    S.offset = offset;
    S.alpha = ctx->alpha;
    S.beta = beta;
    S.alpha_one = ctx->alpha == 1.0f;
    S.out = out;
    S.out_w = out_w;
    S.upd_idx = upd_idx;
    S.upd_p = upd_p;
    S.n_upd = n_upd;
    S.capacity = ctx->capacity;
    S.prio = ctx->prio;
    S.ticket = ctx->tickets + TK_STEP;
    S.step_min = ctx->step_min;
    S.rows = static_cast<const uint4*>(rows);
    S.row_chunks = static_cast<int>(row_bytes / 16);
    S.out_rows = static_cast<uint4*>(out_rows);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles));
    cfg.blockDim = dim3(kStepThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, per_step_kernel, S);
    per_note_launch();
    return cuda_status(e);
}
