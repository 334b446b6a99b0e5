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
#include "sample_core.cuh"
#include "scan_core.cuh"

namespace {

constexpr int kStepThreads = 256;  // the one-wave scan's tile: 256 x 8 items

struct StepParams {
    ScanParams scan;
    SampleParams sample;
    const int32_t* __restrict__ upd_idx;
    const float* __restrict__ upd_p;
    int n_upd;
    int64_t capacity;
    float* prio;
    unsigned long long* ticket;  // grid-barrier word of every phase
    unsigned* step_min;          // call counter, then the batch-minimum word of even and odd calls
    int* status;
    int per_cta;  // samples per CTA
};

// CTA c owns scan tile c (the grid is exactly the tiles) and samples
// [c * per_cta, (c + 1) * per_cta).
template <int SPT>
__global__ void __launch_bounds__(kStepThreads) per_step_kernel(StepParams S) {
    extern __shared__ __align__(128) float s_dyn[];  // the sampler's coarse index and window
    constexpr int THREADS = kStepThreads;

    // ---- 1. priority updates of this CTA's tile ----------------------------
    // The CTA owns items [c * TILE, (c + 1) * TILE) (the launcher guarantees
    // capacity <= gridDim.x * TILE): it reads the whole batch, keeps in
    // shared memory the last batch position of each of its items, writes
    // the winners' priorities, and scans them below -- no other CTA reads
    // or writes these items, so no grid barrier is needed.
    if (S.n_upd > 0) {
        constexpr int TILE = THREADS * 8;
        __shared__ int s_win[TILE];
        const int64_t lo = static_cast<int64_t>(blockIdx.x) * TILE;
        for (int j = threadIdx.x; j < TILE; j += THREADS) s_win[j] = -1;
        __syncthreads();
        bool bad = false;
        constexpr int kU = 8;  // batch positions per thread per round, loads issued first
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
        __syncthreads();
        for (int j = threadIdx.x; j < TILE; j += THREADS) {
            const int k = s_win[j];
            if (k >= 0) {
                const float v = __ldg(S.upd_p + k);
                if (!(v >= 0.f)) bad = true;
                S.prio[lo + j] = v;
            }
        }
        if (bad) atomicOr(S.status, ST_VALUE);
        __syncthreads();  // this CTA's new priorities before its scan reads them
    }

    // ---- 2. build_cdf: tile blockIdx.x ------------------------------------
    // (this call's parity picks the batch-minimum word: step_min[0] counts
    // the calls, every CTA reads it before the grid barrier below, CTA 0
    // advances it after the weights' barrier and resets the next call's word)
    __shared__ unsigned s_parity;
    if (threadIdx.x == 0) s_parity = ld_relaxed_u32(S.step_min) & 1u;
    const unsigned scan_epoch = wave_scan_tile<THREADS>(S.scan, blockIdx.x);
    grid_barrier(S.ticket, S.status, ST_TIMEOUT);  // CDF and coarse index complete
    if (threadIdx.x == 0) {
        if (blockIdx.x == 0) {
            advance_scan_epoch(S.scan, scan_epoch);
            S.step_min[1 + (s_parity ^ 1u)] = 0x7f800000u;  // +inf for the next call
        }
        // the sampler's bulk copies (async proxy) read what this launch wrote
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncthreads();

    // ---- 3. samples and IS weights ----------------------------------------
    SampleParams sp = S.sample;
    sp.min_word = S.step_min + 1 + s_parity;
    const int k0 = static_cast<int>(blockIdx.x) * S.per_cta;
    const int kend = min(sp.B, k0 + S.per_cta);
    coarse_sample<THREADS, SPT, true>(sp, k0 < kend ? k0 : kend, kend, s_dyn);
    if (blockIdx.x == 0 && threadIdx.x == 0) S.step_min[0] = S.step_min[0] + 1u;  // every CTA has read it
}

template <int SPT>
per_status launch_step_cfg(const StepParams& S, unsigned grid, cudaStream_t s) {
    const int smem = (kCoarseCap + kWindowCap) * static_cast<int>(sizeof(float));
    static int per_sm = 0;
    if (per_sm == 0) {
        if (cudaFuncSetAttribute(per_step_kernel<SPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, per_step_kernel<SPT>, kStepThreads, smem) !=
                cudaSuccess)
            return PER_ERR_CUDA;
        if (per_sm < 1) per_sm = 1;
    }
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return PER_ERR_CUDA;
    if (static_cast<int64_t>(grid) > static_cast<int64_t>(per_sm) * sms) return PER_ERR_STATE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, per_step_kernel<SPT>, S);
    per_note_launch();
    return cuda_status(e);
}

}  // namespace

// The fused step for scan-only contexts whose CDF fits one wave of
// 2048-item tiles and whose coarse index fits the sampler's staging buffer;
// PER_ERR_STATE (nothing launched) when it does not apply.
per_status launch_step(per_ctx* ctx, const int32_t* upd_idx, const float* upd_p, int n_upd, int B, uint64_t seed,
                       uint64_t offset, const float* u01, float beta, int32_t* out, float* out_w, cudaStream_t s) {
    constexpr int TILE = kStepThreads * 8;
    const int64_t n = ctx->size;
    if (ctx->flags != PER_SCAN || !ctx->coarse || n < 1 || n > (int64_t(1) << 19)) return PER_ERR_STATE;
    if ((n + kCoarseStride - 1) / kCoarseStride > kCoarseCap) return PER_ERR_STATE;
    const int64_t tiles = (n + TILE - 1) / TILE;
    // every index an update may name lies in some CTA's tile
    if (n_upd > 0 && ctx->capacity > tiles * TILE) return PER_ERR_STATE;
    if (tiles > ctx->scan_desc_tiles || tiles > ctx->slot_n) return PER_ERR_STATE;
    const int64_t per_cta = (B + tiles - 1) / tiles;
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
    S.sample.cdf = ctx->cdf;
    S.sample.coarse = ctx->coarse;
    S.sample.n = static_cast<int>(n);
    S.sample.B = B;
    S.sample.seed = seed;
    S.sample.offset = offset;
    S.sample.u01 = u01;
    S.sample.out = out;
    S.sample.status = ctx->status;
    S.sample.prio = ctx->prio;
    S.sample.alpha = ctx->alpha;
    S.sample.alpha_one = ctx->alpha == 1.0f;
    S.sample.beta = beta;
    S.sample.out_w = out_w;
    S.sample.slots = ctx->slots;
    S.sample.ticket = ctx->tickets + TK_STEP;
    S.upd_idx = upd_idx;
    S.upd_p = upd_p;
    S.n_upd = n_upd;
    S.capacity = ctx->capacity;
    S.prio = ctx->prio;
    S.ticket = ctx->tickets + TK_STEP;
    S.step_min = ctx->step_min;
    S.status = ctx->status;
    S.per_cta = static_cast<int>(per_cta);
    const unsigned grid = static_cast<unsigned>(tiles);
    if (per_cta <= kStepThreads) return launch_step_cfg<1>(S, grid, s);
    if (per_cta <= 2 * kStepThreads) return launch_step_cfg<2>(S, grid, s);
    if (per_cta <= 4 * kStepThreads) return launch_step_cfg<4>(S, grid, s);
    return PER_ERR_STATE;
}
