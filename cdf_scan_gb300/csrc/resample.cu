// resample.cu -- row-batched systematic resampling (POPCORNBENCH particle
// filter, reference forward: logsumexp-normalised weights, exp, cumsum along
// the particle axis, u_j = (j + U_b)/P with one U_b per row, searchsorted
// (right=False), clamp to P-1).
//
// One CTA per row, two passes over the row (the second mostly from L2):
//   A. online max / sum of exp(lw - max) (fp32, fixed combine order);
//   B. exp(lw - m) quantised to 40-bit fixed point and scanned with exact
//      64-bit integer sums (monotone and order-independent), c_i =
//      fl32(fl32(E_i) * fl32(2^-40 / s)); then, instead of one binary search
//      per output, every particle i computes n(c) = #{j : u_j <= c} for its
//      own c_i and its predecessor's c_{i-1} in closed form (a guess from
//      c*P - U corrected by at most a couple of exact threshold evaluations)
//      and writes i into outputs [n(c_{i-1}), n(c_i)) -- exactly the outputs
//      whose lower_bound lands on i.  The last particle's run extends to P,
//      which is the clamp.
#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kThreads = 1024;
constexpr int kChunk = kThreads * 4;
constexpr float kFix = 1099511627776.0f;  // 2^40

struct ResampleParams {
    const float* __restrict__ logw;
    int P;
    uint64_t seed, offset;
    const float* __restrict__ u_rows;
    int32_t* __restrict__ out;
    float* __restrict__ out_cdf;
};

__device__ __forceinline__ void lse_combine(float& m, float& s, float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) {
        m = m2;
        s = s2;
        return;
    }
    if (m2 > m) {
        s = s * expf(m - m2) + s2;
        m = m2;
    } else {
        s = s + s2 * expf(m2 - m);
    }
}

__device__ __forceinline__ void lse_add(float& m, float& s, float x) {
    if (x == -INFINITY) return;
    if (x > m) {
        s = (m == -INFINITY) ? 1.f : s * expf(m - x) + 1.f;
        m = x;
    } else {
        s += expf(x - m);
    }
}

// Threshold u_j = fl32(fl32(j + U) / P).
__device__ __forceinline__ float row_threshold(int j, float U, float fP) {
    return __fdiv_rn(__fadd_rn(__int2float_rn(j), U), fP);
}

// #{ j in [0, P) : u_j <= c }.
__device__ __forceinline__ int count_le(float c, float U, int P, float fP) {
    const float g = __fsub_rn(__fmul_rn(c, fP), U);
    int j;
    if (!(g >= 0.f)) j = -1;
    else if (g >= fP) j = P - 1;
    else j = static_cast<int>(g);
    while (j + 1 < P && row_threshold(j + 1, U, fP) <= c) ++j;
    while (j >= 0 && row_threshold(j, U, fP) > c) --j;
    return j + 1;
}

__global__ void __launch_bounds__(kThreads) resample_kernel(ResampleParams R) {
    __shared__ float s_m[kThreads / 32], s_s[kThreads / 32];
    __shared__ unsigned long long s_tot[kThreads / 32];
    __shared__ float s_stats[2];
    const int b = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int P = R.P;
    const float* row = R.logw + static_cast<size_t>(b) * P;
    int32_t* orow = R.out + static_cast<size_t>(b) * P;

    // ---- A: max and sum of exp(lw - max) -----------------------------------
    float m = -INFINITY, s = 0.f;
    for (int i0 = threadIdx.x * 4; i0 < P; i0 += kChunk) {
        const float4 q = ld_f4(row + i0);
        lse_add(m, s, q.x);
        lse_add(m, s, q.y);
        lse_add(m, s, q.z);
        lse_add(m, s, q.w);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(PER_FULL_MASK, m, o);
        const float s2 = __shfl_xor_sync(PER_FULL_MASK, s, o);
        lse_combine(m, s, m2, s2);
    }
    if (lane == 0) {
        s_m[warp] = m;
        s_s[warp] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float bm = s_m[0], bs = s_s[0];
        for (int w = 1; w < kThreads / 32; ++w) lse_combine(bm, bs, s_m[w], s_s[w]);
        s_stats[0] = bm;
        s_stats[1] = bs;
    }
    __syncthreads();
    const float rmax = s_stats[0];
    const float scale = __fdiv_rn(1.0f / kFix, s_stats[1]);
    const float fP = static_cast<float>(P);
    const float U = R.u_rows ? R.u_rows[b] : u01_closed_open(R.seed, R.offset + static_cast<uint64_t>(b));

    // ---- B: exact fixed-point scan, then scatter each particle's run --------
    unsigned long long carry = 0ull;
    for (int c0 = 0; c0 < P; c0 += kChunk) {
        const int i0 = c0 + threadIdx.x * 4;
        const bool in = i0 < P;
        float4 q = in ? ld_f4(row + i0) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        const float xs[4] = {q.x, q.y, q.z, q.w};
        unsigned long long f[4], r[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float w = xs[e] == -INFINITY ? 0.f : expf(xs[e] - rmax);
            f[e] = __float2ull_rz(__fmul_rn(w, kFix));
        }
        r[0] = f[0];
        r[1] = r[0] + f[1];
        r[2] = r[1] + f[2];
        r[3] = r[2] + f[3];
        unsigned long long x = r[3];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned long long y = __shfl_up_sync(PER_FULL_MASK, x, d);
            if (lane >= d) x += y;
        }
        if (lane == 31) s_tot[warp] = x;
        __syncthreads();
        const unsigned long long t = s_tot[lane];
        unsigned long long wi = t;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned long long y = __shfl_up_sync(PER_FULL_MASK, wi, d);
            if (lane >= d) wi += y;
        }
        const unsigned long long warp_off = __shfl_sync(PER_FULL_MASK, wi - t, warp);
        const unsigned long long chunk_total = __shfl_sync(PER_FULL_MASK, wi, 31);
        const unsigned long long base = carry + warp_off + (x - r[3]);
        __syncthreads();  // s_tot reused by the next chunk
        carry += chunk_total;
        if (!in) continue;

        float cv[4];
        int nprev = i0 == 0 ? 0 : count_le(__fmul_rn(__ull2float_rn(base), scale), U, P, fP);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const unsigned long long E = base + r[e];
            cv[e] = __fmul_rn(__ull2float_rn(E), scale);
            const int i = i0 + e;
            const int ncur = (i == P - 1) ? P : count_le(cv[e], U, P, fP);
            for (int j = nprev; j < ncur; ++j) orow[j] = i;
            nprev = ncur > nprev ? ncur : nprev;
        }
        if (R.out_cdf) st_f4(R.out_cdf + static_cast<size_t>(b) * P + i0, make_float4(cv[0], cv[1], cv[2], cv[3]));
    }
}

}  // namespace

per_status launch_resample(const float* logw, int rows, int P, uint64_t seed, uint64_t offset,
                           const float* u_rows, int32_t* out, float* out_cdf, cudaStream_t s) {
    ResampleParams R;
    R.logw = logw;
    R.P = P;
    R.seed = seed;
    R.offset = offset;
    R.u_rows = u_rows;
    R.out = out;
    R.out_cdf = out_cdf;
    resample_kernel<<<static_cast<unsigned>(rows), kThreads, 0, s>>>(R);
    per_note_launch();
    return cuda_status(cudaGetLastError());
}
