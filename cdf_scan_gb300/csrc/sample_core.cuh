// sample_core.cuh -- stratified inverse-CDF sampling with the coarse CDF
// index, shared by the sampling kernels (sample.cu) and the fused PER step
// (step.cu).  idx_k = first i with cdf[i] >= u_k (searchsorted, right=False;
// clamp to n-1), u_k = fl32(fl32(fl32(k + U_k)/B) * T), T = cdf[n-1]
// (POPCORNBENCH particle-filter trace: searchsorted + clamp semantics;
// foxhunt "GPU Segment Tree for PER Sampling" section "Problem": the O(n)
// path is prefix sum + searchsorted).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kWindowCap = 12288;  // floats staged per CTA (48 KB)

struct SampleParams {
    const float* __restrict__ cdf;
    const float* __restrict__ coarse;  // coarse[j] = cdf[min(64j + 63, n - 1)], or nullptr
    int n;
    int B;
    uint64_t seed, offset;
    const float* __restrict__ u01;
    int32_t* __restrict__ out;
    int* status;
    // fused importance-sampling weights (per_sample_weighted)
    const float* __restrict__ prio;
    float alpha;
    bool alpha_one;
    float beta;
    float* __restrict__ out_w;
    float* slots;                // [gridDim.x] per-CTA minima
    unsigned long long* ticket;  // grid-barrier ticket
    unsigned* min_word;          // or one word every CTA atomicMin's (float bits; +inf on entry)
    // rank-based PER: the CDF is over ranks and out[k] = order[rank] (nullptr: out[k] = the index drawn)
    const int32_t* __restrict__ order;
};

__device__ __forceinline__ int32_t sample_item(const SampleParams& P, int r) { return P.order ? __ldg(P.order + r) : r; }

__device__ __forceinline__ float draw_u(const SampleParams& P, int k) {
    return P.u01 ? P.u01[k] : u01_open_closed(P.seed, P.offset + static_cast<uint64_t>(k));
}

// ---- with the coarse index -------------------------------------------------
//
// build_cdf leaves coarse[j] = cdf[min(64j + 63, n - 1)].  When the whole
// index fits a CTA's shared memory, one bulk copy stages it; the first block
// j with coarse[j] >= u holds lower_bound(cdf, u) (coarse is a subsequence of
// the non-decreasing CDF), so the CTA's window is found without a single
// dependent global load, then staged with a second bulk copy and searched
// per thread in shared memory.

constexpr int kCoarseCap = 4096;  // coarse entries staged per CTA (16 KB)

// Minimum over the CTA of one value per thread (result on every thread).
template <int THREADS>
__device__ __forceinline__ float block_min(float m, float* s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fminf(m, __shfl_xor_sync(PER_FULL_MASK, m, o));
    __syncthreads();  // s_red may still be read from a previous use
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    float b = s_red[0];
    for (int w = 1; w < THREADS / 32; ++w) b = fminf(b, s_red[w]);
    return b;
}

__device__ __forceinline__ int smem_lower_bound(const float* a, int lo, int hi, float u) {
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < u) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Samples k0 .. kend-1 (kend - k0 <= THREADS * SPT; an empty range only
// takes part in the weights' grid barrier) with the coarse index staged in
// s_dyn (kCoarseCap floats, then the kWindowCap-float window).  The CDF and
// the priorities are read through L2 (.cg), so a launch that wrote them
// before a grid barrier reads them back coherently.
template <int THREADS, int SPT, bool WEIGHTS>
__device__ __forceinline__ void coarse_sample(const SampleParams& P, int k0, int kend, float* s_dyn) {
    float* s_coarse = s_dyn;
    float* s_win = s_dyn + kCoarseCap;
    __shared__ __align__(8) uint64_t s_bar[2];
    __shared__ int s_lo, s_hi;

    const bool any = k0 < kend;
    const int nc = (P.n + kCoarseStride - 1) / kCoarseStride;
    if (threadIdx.x == 0) {
        mbar_init(&s_bar[0], 1);
        mbar_init(&s_bar[1], 1);
        if (any) {
            // whole 16-byte groups; the coarse allocation is padded past nc
            const unsigned bytes = (static_cast<unsigned>(nc) * 4u + 15u) & ~15u;
            mbar_arrive_expect_tx(&s_bar[0], bytes);
            bulk_copy_g2s(s_coarse, P.coarse, bytes, &s_bar[0]);
        }
    }
    const float T = __ldcg(P.cdf + P.n - 1);
    if (!(T > 0.f)) {
        if (threadIdx.x == 0) {
            atomicOr(P.status, ST_EMPTY);
            if (any && !mbar_wait_bounded(&s_bar[0], 0)) atomicOr(P.status, ST_TIMEOUT);  // no copy in flight
        }
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
    __syncthreads();  // barrier initialisation visible to every thread
    int res[SPT];
#pragma unroll
    for (int s = 0; s < SPT; ++s) res[s] = 0;
    if (any) {
        if (!mbar_wait_bounded(&s_bar[0], 0)) atomicOr(P.status, ST_TIMEOUT);
        if (threadIdx.x == 0) {
            const float uf = stratified_threshold(k0, draw_u(P, k0), fB, T);
            s_lo = smem_lower_bound(s_coarse, 0, nc, uf);
        }
        if (threadIdx.x == (THREADS > 32 ? 32 : 0)) {
            const float ul = stratified_threshold(kend - 1, draw_u(P, kend - 1), fB, T);
            s_hi = smem_lower_bound(s_coarse, 0, nc, ul);
        }
        __syncthreads();
        const int jl = min(s_lo, nc - 1), jh = min(s_hi, nc - 1);
        const int a0 = jl * kCoarseStride;
        const int a1 = min(jh * kCoarseStride + kCoarseStride, P.n);  // exclusive
        const int a1r = (a1 + 3) & ~3;                                 // the CDF allocation is padded
        if (a1r - a0 <= kWindowCap) {
            if (threadIdx.x == 0) {
                const unsigned bytes = static_cast<unsigned>(a1r - a0) * 4u;
                mbar_arrive_expect_tx(&s_bar[1], bytes);
                bulk_copy_g2s(s_win, P.cdf + a0, bytes, &s_bar[1]);
            }
            if (!mbar_wait_bounded(&s_bar[1], 0)) atomicOr(P.status, ST_TIMEOUT);
#pragma unroll
            for (int s = 0; s < SPT; ++s) res[s] = min(a0 + smem_lower_bound(s_win, 0, a1 - a0, u[s]), P.n - 1);
        } else {
            // a very skewed window: each thread finds its own 64-item block, then
            // searches it in global memory
#pragma unroll
            for (int s = 0; s < SPT; ++s) {
                const int j = min(smem_lower_bound(s_coarse, jl, jh + 1, u[s]), nc - 1);
                int lo = j * kCoarseStride, hi = min(lo + kCoarseStride, P.n);
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (__ldcg(P.cdf + mid) < u[s]) lo = mid + 1;
                    else hi = mid;
                }
                res[s] = min(lo, P.n - 1);
            }
        }
#pragma unroll
        for (int s = 0; s < SPT; ++s) {
            const int k = k0 + threadIdx.x + s * THREADS;
            if (k < kend) P.out[k] = sample_item(P, res[s]);
        }
    }
    if (WEIGHTS) {
        // the IS weights of the batch, exactly as per_is_weights computes
        // them: pa = powf(p, alpha) of every sample, the batch minimum
        // across CTAs (slots + one grid barrier), w = (pa_min / pa)^beta
        __shared__ float s_red[THREADS / 32];
        float pa[SPT];
        float m = __int_as_float(0x7f800000);  // +inf
#pragma unroll
        for (int s = 0; s < SPT; ++s) {
            const int k = k0 + threadIdx.x + s * THREADS;
            pa[s] = k < kend ? pow_accurate(__ldcg(P.prio + res[s]), P.alpha, P.alpha_one) : m;
            m = fminf(m, pa[s]);
        }
        // minima as non-negative floats (a -0 becomes +0), whose order is
        // the order of their bits
        m = block_min<THREADS>(m, s_red) + 0.f;
        float pa_min;
        if (P.min_word) {
            __shared__ float s_min;
            if (threadIdx.x == 0) atomicMin(P.min_word, __float_as_uint(m));
            grid_barrier(P.ticket, P.status, ST_TIMEOUT);
            if (threadIdx.x == 0) s_min = __uint_as_float(ld_relaxed_u32(P.min_word));
            __syncthreads();
            pa_min = s_min;
        } else {
            if (threadIdx.x == 0) P.slots[blockIdx.x] = m;
            grid_barrier(P.ticket, P.status, ST_TIMEOUT);
            float g = __int_as_float(0x7f800000);
            for (int j = threadIdx.x; j < static_cast<int>(gridDim.x); j += THREADS)
                g = fminf(g, __ldcg(P.slots + j));
            pa_min = block_min<THREADS>(g, s_red);
        }
#pragma unroll
        for (int s = 0; s < SPT; ++s) {
            const int k = k0 + threadIdx.x + s * THREADS;
            if (k < kend) P.out_w[k] = powf(__fdiv_rn(pa_min, pa[s]), P.beta);
        }
    }
}

}  // namespace
