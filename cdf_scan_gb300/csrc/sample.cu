// sample.cu -- stratified inverse-CDF sampling on the scan path.
//
// idx_k = first i with cdf[i] >= u_k (searchsorted, right=False; clamp to
// n-1), with u_k = fl32(fl32(fl32(k + U_k)/B) * T) and T = cdf[n-1]
// (POPCORNBENCH particle-filter trace: searchsorted + clamp semantics;
// foxhunt "GPU Segment Tree for PER Sampling" section "Problem": the O(n)
// path is prefix sum + searchsorted).
//
// Stratified thresholds are sorted in k, so the samples of one CTA map to one
// contiguous window [i_lo, i_hi] of the CDF.  The CTA finds the two window
// ends with a warp-wide 32-ary search (one gather of 32 probes per round,
// ~log32(n) rounds), stages the window in shared memory with one bulk copy
// (cp.async.bulk completing on an mbarrier), and every thread finishes its
// searches in shared memory.  Windows larger than the staging buffer (very
// skewed priorities) fall back to a global binary search inside the window.
#include "sample_core.cuh"

namespace {

// Window buffer of the large-n sampler (24 KB): with the samples per CTA
// sized to fill ~2/3 of it, up to 8 CTAs of 256 threads share an SM, enough
// to hide the searches' dependent shared-memory loads and to keep windows in
// flight (1M samples over 16M: 23.0 us against 27.1 with 48 KB windows).
constexpr int kScanWindowCap = 6144;

// lower_bound over cdf[0..n) by one warp (all lanes get the answer).
__device__ int warp_lower_bound(const float* __restrict__ c, int n, float u, int lane) {
    int lo = 0, hi = n;  // answer in [lo, hi]; hi == n: nothing >= u found yet
    while (hi - lo > 32) {
        const int step = (hi - lo + 31) / 32;
        int pos = lo + (lane + 1) * step - 1;
        if (pos > hi - 1) pos = hi - 1;
        const float v = __ldg(c + pos);
        const unsigned ge = __ballot_sync(PER_FULL_MASK, v >= u);
        if (ge == 0u) {
            lo = hi;
        } else {
            const int f = __ffs(ge) - 1;
            const int pf = __shfl_sync(PER_FULL_MASK, pos, f);
            const int pprev = __shfl_sync(PER_FULL_MASK, pos, f > 0 ? f - 1 : 0);
            hi = pf;
            lo = f > 0 ? pprev + 1 : lo;
        }
    }
    const int pos = lo + lane;
    const bool ge = pos < hi && __ldg(c + pos) >= u;
    const unsigned m = __ballot_sync(PER_FULL_MASK, ge);
    const int ans = m ? lo + __ffs(m) - 1 : hi;
    return ans < n ? ans : n - 1;
}

// The window ends of every CTA of sample_scan_kernel, one warp per end:
// bounds[2j] = lower_bound of CTA j's first threshold, bounds[2j + 1] of its
// last (the thresholds and the searches the sampler would make itself, so
// they are the same values).  The ends of all CTAs are searched at once,
// instead of one CTA after another in front of each window copy.
__global__ void __launch_bounds__(256) sample_bounds_kernel(SampleParams P, int* __restrict__ bounds, int per_cta,
                                                             int ctas) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the sampler may be scheduled
    const int lane = threadIdx.x & 31;
    const int w = static_cast<int>((blockIdx.x * 256u + threadIdx.x) >> 5);
    if (w >= 2 * ctas) return;
    const float T = __ldg(P.cdf + P.n - 1);
    if (!(T > 0.f)) return;  // the sampler reports the empty buffer
    const int j = w >> 1;
    const int k0 = j * per_cta;
    const int k = (w & 1) ? min(P.B, k0 + per_cta) - 1 : k0;
    const float u = stratified_threshold(k, draw_u(P, k), static_cast<float>(P.B), T);
    const int b = warp_lower_bound(P.cdf, P.n, u, lane);
    if (lane == 0) bounds[w] = b;
}

// One CTA per THREADS x SPT consecutive strata: the thresholds, then (after
// the bounds launch, of which this launch is a programmatic dependent) the
// window [lower_bound(first), lower_bound(last)] staged by one bulk copy and
// searched in shared memory.
template <int THREADS, int SPT>
__global__ void __launch_bounds__(THREADS) sample_scan_kernel(SampleParams P, const int* __restrict__ bounds) {
    extern __shared__ __align__(128) float s_win[];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ int s_lo, s_hi;

    const int k0 = blockIdx.x * THREADS * SPT;
    const int kend = min(P.B, k0 + THREADS * SPT);  // exclusive
    const float T = __ldg(P.cdf + P.n - 1);
    if (!(T > 0.f)) {
        if (threadIdx.x == 0) atomicOr(P.status, ST_EMPTY);
        for (int s = 0; s < SPT; ++s) {
            const int k = k0 + threadIdx.x + s * THREADS;
            if (k < kend) P.out[k] = 0;
        }
        return;
    }
    const float fB = static_cast<float>(P.B);

    float u[SPT];
#pragma unroll
    for (int s = 0; s < SPT; ++s) {
        const int k = k0 + threadIdx.x + s * THREADS;
        u[s] = k < kend ? stratified_threshold(k, draw_u(P, k), fB, T) : 0.f;
    }
    // the window ends: from the bounds launch
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) {
        s_lo = __ldcg(bounds + 2 * blockIdx.x);
        s_hi = __ldcg(bounds + 2 * blockIdx.x + 1);
    }
    __syncthreads();
    const int ilo = s_lo, ihi = s_hi;
    const int a0 = ilo & ~3;
    const int a1 = (ihi + 4) & ~3;  // exclusive; the CDF allocation is padded
    int res[SPT];
    if (a1 - a0 <= kScanWindowCap) {
        if (threadIdx.x == 0) {
            mbar_init(&s_bar, 1);
            const unsigned bytes = static_cast<unsigned>(a1 - a0) * 4u;
            mbar_arrive_expect_tx(&s_bar, bytes);
            bulk_copy_g2s(s_win, P.cdf + a0, bytes, &s_bar);
        }
        __syncthreads();
        if (!mbar_wait_bounded(&s_bar, 0)) atomicOr(P.status, ST_TIMEOUT);
#pragma unroll
        for (int s = 0; s < SPT; ++s) {
            int lo = ilo - a0, hi = ihi - a0;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (s_win[mid] < u[s]) lo = mid + 1;
                else hi = mid;
            }
            res[s] = a0 + lo;
        }
    } else {
#pragma unroll
        for (int s = 0; s < SPT; ++s) {
            int lo = ilo, hi = ihi;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (__ldg(P.cdf + mid) < u[s]) lo = mid + 1;
                else hi = mid;
            }
            res[s] = lo;
        }
    }
#pragma unroll
    for (int s = 0; s < SPT; ++s) {
        const int k = k0 + threadIdx.x + s * THREADS;
        if (k < kend) P.out[k] = sample_item(P, res[s]);
    }
}

// ---- with the coarse index (coarse_sample) -------------------------------------
template <int THREADS, int SPT, bool WEIGHTS>
__global__ void __launch_bounds__(THREADS) sample_coarse_kernel(SampleParams P) {
    extern __shared__ __align__(128) float s_dyn[];  // kCoarseCap coarse entries, then the window
    const int k0 = blockIdx.x * THREADS * SPT;
    coarse_sample<THREADS, SPT, WEIGHTS>(P, k0, min(P.B, k0 + THREADS * SPT), s_dyn);
}

template <int THREADS, int SPT, bool WEIGHTS>
per_status launch_coarse_cfg(const SampleParams& P, cudaStream_t s) {
    const int per_cta = THREADS * SPT;
    const unsigned grid = static_cast<unsigned>((P.B + per_cta - 1) / per_cta);
    const int smem = (kCoarseCap + kWindowCap) * static_cast<int>(sizeof(float));
    static DeviceCache cache;
    const int per_sm = device_cached(cache, [&]() {
        int b = 0;
        if (cudaFuncSetAttribute(sample_coarse_kernel<THREADS, SPT, WEIGHTS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, sample_coarse_kernel<THREADS, SPT, WEIGHTS>, THREADS,
                                                          smem) != cudaSuccess)
            return 0;
        return b < 1 ? 1 : b;
    });
    if (per_sm == 0) return PER_ERR_CUDA;
    if (!WEIGHTS) {
        sample_coarse_kernel<THREADS, SPT, WEIGHTS><<<grid, THREADS, smem, s>>>(P);
        per_note_launch();
        return cuda_status(cudaGetLastError());
    }
    // the grid barrier needs every CTA resident at once: cooperative launch
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return PER_ERR_CUDA;
    if (static_cast<int64_t>(grid) > static_cast<int64_t>(per_sm) * sms) return PER_ERR_STATE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, sample_coarse_kernel<THREADS, SPT, WEIGHTS>, P);
    per_note_launch();
    return cuda_status(e);
}

template <int THREADS, int SPT>
per_status launch_cfg(const SampleParams& P, int* bounds, int64_t bounds_n, cudaStream_t s) {
    const int per_cta = THREADS * SPT;
    const unsigned grid = static_cast<unsigned>((P.B + per_cta - 1) / per_cta);
    // opt in to the window buffer's dynamic shared memory once per
    // instantiation and device (needed above the default 48 KB limit)
    static DeviceCache cache;
    if (!device_cached(cache, []() {
            return cudaFuncSetAttribute(sample_scan_kernel<THREADS, SPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kScanWindowCap * sizeof(float))) == cudaSuccess
                       ? 1
                       : 0;
        }))
        return PER_ERR_CUDA;
    if (!bounds || static_cast<int64_t>(grid) > bounds_n) return PER_ERR_STATE;
    sample_bounds_kernel<<<(2 * grid + 7) / 8, 256, 0, s>>>(P, bounds, per_cta, static_cast<int>(grid));
    per_note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = kScanWindowCap * sizeof(float);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, sample_scan_kernel<THREADS, SPT>, P, static_cast<const int*>(bounds));
    per_note_launch();
    return cuda_status(e);
}

}  // namespace

// Samples per CTA: aim the expected window (n/B items per sample, uniform
// case) at ~2/3 of the staging buffer, and keep at least ~2 CTAs per SM busy
// when B is small.
namespace {

// Samples per CTA of the coarse-index path: few (128) so that small batches
// spread over several CTAs, each with a short chain of copies and searches
// (1024 samples over 8192 items: 2.8 us against 5.6 with one CTA of 1024),
// more while the grid would exceed 4 CTAs per SM (every CTA stages the
// coarse index), and fewer while the expected window (n/B items per sample)
// would exceed ~2/3 of the staging buffer.
int coarse_per_cta(int B, double ratio, int num_sms) {
    int per_cta = 128;
    while (per_cta < 1024 && (B + per_cta - 1) / per_cta > 4 * num_sms) per_cta <<= 1;
    while (per_cta > 32 && ratio * per_cta > (2.0 * kWindowCap) / 3.0) per_cta >>= 1;
    return per_cta;
}

// The coarse-index path with or without fused weights; PER_ERR_STATE when it
// does not apply.
template <bool WEIGHTS>
per_status launch_coarse(const SampleParams& P, int per_cta, cudaStream_t s) {
    switch (per_cta) {
        case 1024: return launch_coarse_cfg<256, 4, WEIGHTS>(P, s);
        case 512: return launch_coarse_cfg<256, 2, WEIGHTS>(P, s);
        case 256: return launch_coarse_cfg<256, 1, WEIGHTS>(P, s);
        case 128: return launch_coarse_cfg<128, 1, WEIGHTS>(P, s);
        case 64: return launch_coarse_cfg<64, 1, WEIGHTS>(P, s);
        default: return launch_coarse_cfg<32, 1, WEIGHTS>(P, s);
    }
}

SampleParams sample_params(per_ctx* ctx, int B, uint64_t seed, uint64_t offset, const float* u01, int32_t* out) {
    SampleParams P = {};
    const bool rank = (ctx->flags & PER_RANK) != 0;  // draw ranks from the rank CDF, write their items
    P.cdf = rank ? ctx->rank_cdf : ctx->cdf;
    P.order = rank ? ctx->rank_order : nullptr;
    P.n = static_cast<int>(ctx->size);
    P.B = B;
    P.seed = seed;
    P.offset = offset;
    P.u01 = u01;
    P.out = out;
    P.status = ctx->status;
    P.coarse = rank ? ctx->rank_coarse : ctx->coarse;
    return P;
}

bool coarse_fits(const per_ctx* ctx) {
    const float* coarse = (ctx->flags & PER_RANK) ? ctx->rank_coarse : ctx->coarse;
    return coarse && (ctx->size + kCoarseStride - 1) / kCoarseStride <= kCoarseCap;
}

}  // namespace

// Samples per CTA: aim the expected window (n/B items per sample, uniform
// case) at ~2/3 of the staging buffer, and keep at least ~2 CTAs per SM busy
// when B is small.
per_status launch_sample_scan(per_ctx* ctx, int B, uint64_t seed, uint64_t offset, const float* u01,
                              int32_t* out, cudaStream_t s) {
    SampleParams P = sample_params(ctx, B, seed, offset, u01, out);
    const double ratio = static_cast<double>(P.n) / static_cast<double>(B);
    if (coarse_fits(ctx)) return launch_coarse<false>(P, coarse_per_cta(B, ratio, ctx->num_sms), s);
    int per_cta = 1024;
    while (per_cta > 32 && ratio * per_cta > (2.0 * kScanWindowCap) / 3.0) per_cta >>= 1;
    while (per_cta > 32 && (B + per_cta - 1) / per_cta < 2 * ctx->num_sms) per_cta >>= 1;
    switch (per_cta) {
        case 1024: return launch_cfg<256, 4>(P, ctx->sample_bounds, ctx->sample_bounds_n, s);
        case 512: return launch_cfg<256, 2>(P, ctx->sample_bounds, ctx->sample_bounds_n, s);
        case 256: return launch_cfg<256, 1>(P, ctx->sample_bounds, ctx->sample_bounds_n, s);
        case 128: return launch_cfg<128, 1>(P, ctx->sample_bounds, ctx->sample_bounds_n, s);
        case 64: return launch_cfg<64, 1>(P, ctx->sample_bounds, ctx->sample_bounds_n, s);
        default: return launch_cfg<32, 1>(P, ctx->sample_bounds, ctx->sample_bounds_n, s);
    }
}

// Sampling with the IS weights fused into the same launch (scan path with the
// coarse index); PER_ERR_STATE when the fused path does not apply.
per_status launch_sample_scan_weighted(per_ctx* ctx, int B, uint64_t seed, uint64_t offset, const float* u01,
                                       float beta, int32_t* out, float* out_w, cudaStream_t s) {
    if (!coarse_fits(ctx)) return PER_ERR_STATE;
    SampleParams P = sample_params(ctx, B, seed, offset, u01, out);
    P.prio = (ctx->flags & PER_RANK) ? ctx->rank_q : ctx->prio;  // weights of the drawn ranks
    P.alpha = ctx->alpha;
    P.alpha_one = ctx->alpha == 1.0f;
    P.beta = beta;
    P.out_w = out_w;
    P.slots = ctx->slots;
    P.ticket = ctx->tickets + TK_SAMPLE;
    const double ratio = static_cast<double>(P.n) / static_cast<double>(B);
    const int per_cta = coarse_per_cta(B, ratio, ctx->num_sms);
    if ((B + per_cta - 1) / per_cta > ctx->slot_n) return PER_ERR_STATE;
    return launch_coarse<true>(P, per_cta, s);
}
