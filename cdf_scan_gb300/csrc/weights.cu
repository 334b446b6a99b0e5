// weights.cu -- importance-sampling weights for a sampled batch.
//
// w_k = (N * P(idx_k))^-beta / max_k (N * P(idx_k))^-beta with P(i) = pa_i /
// total (the PER correction the foxhunt design doc lists as unchanged under
// "Non-Goals").  N and the total cancel, so the kernels compute the
// equivalent max-normalised form w_k = (pa_min / pa_{idx_k})^beta, pa_min the
// smallest pa in the batch: the weight of the batch minimum is exactly 1.
//
// Two launches over many SMs (the powers dominate, so the work is spread):
//   1. gather pa for every sample (tree leaves, or p^alpha of the raw
//      priorities) into the output buffer; warp-shuffle + block minimum, then
//      an order-independent atomicMin on the float's bit pattern (valid for
//      non-negative floats);
//   2. w_k = (pa_min / pa_k)^beta in place; the last CTA resets the minimum
//      word for the next call.
#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kThreads = 256;

struct IswParams {
    const int32_t* __restrict__ idx;
    int B;
    const float* __restrict__ leaves;  // tree leaves (pa) or nullptr
    const float* __restrict__ prio;    // raw priorities when leaves == nullptr
    float alpha;
    bool alpha_one;
    float beta;
    int64_t capacity;
    float* out;
    unsigned* ctrs;
    int* status;
};

__global__ void __launch_bounds__(kThreads) gather_min_kernel(IswParams P) {
    __shared__ float s_min[kThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float m = __int_as_float(0x7f800000);  // +inf
    bool bad = false;
    for (int k = blockIdx.x * kThreads + threadIdx.x; k < P.B; k += gridDim.x * kThreads) {
        const int32_t i = P.idx[k];
        float pa;
        if (i < 0 || i >= P.capacity) {
            bad = true;
            pa = __int_as_float(0x7fc00000);  // NaN
        } else if (P.leaves) {
            pa = __ldg(P.leaves + i);
        } else {
            pa = pow_accurate(__ldg(P.prio + i), P.alpha, P.alpha_one);
        }
        P.out[k] = pa;
        m = fminf(m, pa);
    }
    if (bad) atomicOr(P.status, ST_VALUE);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fminf(m, __shfl_xor_sync(PER_FULL_MASK, m, o));
    if (lane == 0) s_min[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float bm = s_min[0];
        for (int w = 1; w < kThreads / 32; ++w) bm = fminf(bm, s_min[w]);
        atomicMin(P.ctrs + CTR_ISW_MIN, __float_as_uint(bm));
    }
}

__global__ void __launch_bounds__(kThreads) weights_kernel(IswParams P) {
    const float pa_min = __uint_as_float(ld_relaxed_u32(P.ctrs + CTR_ISW_MIN));
    for (int k = blockIdx.x * kThreads + threadIdx.x; k < P.B; k += gridDim.x * kThreads)
        P.out[k] = powf(__fdiv_rn(pa_min, P.out[k]), P.beta);
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned done = atomicAdd(P.ctrs + CTR_ISW_DONE, 1u);
        if (done == gridDim.x - 1u) {
            P.ctrs[CTR_ISW_DONE] = 0u;
            P.ctrs[CTR_ISW_MIN] = 0xffffffffu;  // above every non-negative float
        }
    }
}

}  // namespace

per_status launch_is_weights(per_ctx* ctx, const int32_t* idx, int B, float beta, float* out, cudaStream_t s) {
    IswParams P;
    P.idx = idx;
    P.B = B;
    const bool tree = (ctx->flags & PER_TREE) != 0;
    P.leaves = tree ? ctx->tree + ctx->cap_pow2 : nullptr;
    P.prio = ctx->prio;
    P.alpha = ctx->alpha;
    P.alpha_one = ctx->alpha == 1.0f;
    P.beta = beta;
    P.capacity = ctx->capacity;
    P.out = out;
    P.ctrs = ctx->ctrs;
    P.status = ctx->status;
    int ctas = (B + kThreads - 1) / kThreads;
    const int max_ctas = 8 * ctx->num_sms;
    if (ctas > max_ctas) ctas = max_ctas;
    gather_min_kernel<<<ctas, kThreads, 0, s>>>(P);
    weights_kernel<<<ctas, kThreads, 0, s>>>(P);
    per_note_launch(2);
    return cuda_status(cudaGetLastError());
}
