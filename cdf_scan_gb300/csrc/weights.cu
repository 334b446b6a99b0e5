// weights.cu -- importance-sampling weights for a sampled batch.
//
// w_k = (N * P(idx_k))^-beta / max_k (N * P(idx_k))^-beta with P(i) = pa_i /
// total (the PER correction the foxhunt design doc lists as unchanged under
// "Non-Goals").  N and the total cancel, so the kernels compute the
// equivalent max-normalised form w_k = (pa_min / pa_{idx_k})^beta, pa_min the
// smallest pa in the batch: the weight of the batch minimum is exactly 1.
//
// One cooperative launch over many SMs (the powers dominate, so the work is
// spread):
//   1. every sample's pa (tree leaf, or p^alpha of the raw priority) goes to
//      the output buffer, and each CTA leaves its minimum in a slot;
//   2. after one grid barrier every CTA reads all the slots (an
//      order-independent minimum) and writes w_k = (pa_min / pa_k)^beta in
//      place.  Nothing needs resetting between calls.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kThreads = 256;

struct IswParams {
    const int32_t* __restrict__ idx;
    int B;
    const float* __restrict__ leaves;  // tree leaves (pa) or nullptr
    const float* __restrict__ prio;    // raw priorities when leaves == nullptr
    const int32_t* __restrict__ rank_of;  // rank-based PER: pa = q[rank_of[i]]^alpha (prio = q), else nullptr
    float alpha;
    bool alpha_one;
    float beta;
    int64_t capacity;
    float* out;
    float* slots;                 // [gridDim.x] per-CTA minima
    unsigned long long* ticket;   // grid-barrier ticket
    int* status;
};

// Minimum over the CTA of one value per thread (result on every thread).
__device__ __forceinline__ float block_min(float m, float* s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fminf(m, __shfl_xor_sync(PER_FULL_MASK, m, o));
    __syncthreads();  // s_red may still be read from a previous use
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    float b = s_red[0];
    for (int w = 1; w < kThreads / 32; ++w) b = fminf(b, s_red[w]);
    return b;
}

__global__ void __launch_bounds__(kThreads) is_weights_kernel(IswParams P) {
    __shared__ float s_red[kThreads / 32];
    const int stride = gridDim.x * kThreads;
    float m = __int_as_float(0x7f800000);  // +inf
    bool bad = false;
    for (int k = blockIdx.x * kThreads + threadIdx.x; k < P.B; k += stride) {
        const int32_t i = P.idx[k];
        float pa;
        if (i < 0 || i >= P.capacity) {
            bad = true;
            pa = __int_as_float(0x7fc00000);  // NaN
        } else if (P.leaves) {
            pa = __ldg(P.leaves + i);
        } else {
            pa = pow_accurate(__ldg(P.prio + (P.rank_of ? __ldg(P.rank_of + i) : i)), P.alpha, P.alpha_one);
        }
        P.out[k] = pa;
        m = fminf(m, pa);
    }
    if (bad) atomicOr(P.status, ST_VALUE);
    m = block_min(m, s_red) + 0.f;  // a -0 minimum becomes +0, as in the fused sampler
    if (threadIdx.x == 0) P.slots[blockIdx.x] = m;
    grid_barrier(P.ticket, P.status, ST_TIMEOUT);
    float g = __int_as_float(0x7f800000);
    for (int j = threadIdx.x; j < static_cast<int>(gridDim.x); j += kThreads) g = fminf(g, __ldcg(P.slots + j));
    const float pa_min = block_min(g, s_red);
    for (int k = blockIdx.x * kThreads + threadIdx.x; k < P.B; k += stride)
        P.out[k] = powf(__fdiv_rn(pa_min, P.out[k]), P.beta);
}

}  // namespace

per_status launch_is_weights(per_ctx* ctx, const int32_t* idx, int B, float beta, float* out, cudaStream_t s) {
    static DeviceCache cache;
    const int per_sm = device_cached(cache, []() {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, is_weights_kernel, kThreads, 0) != cudaSuccess) return 0;
        return b < 1 ? 1 : b;
    });
    if (per_sm == 0) return PER_ERR_CUDA;
    IswParams P;
    P.idx = idx;
    P.B = B;
    const bool tree = (ctx->flags & PER_TREE) != 0;
    P.leaves = tree ? ctx->tree + ctx->cap_pow2 : nullptr;
    const bool rank = (ctx->flags & PER_RANK) != 0;
    P.prio = rank ? ctx->rank_q : ctx->prio;
    P.rank_of = rank ? ctx->rank_of : nullptr;
    P.alpha = ctx->alpha;
    P.alpha_one = ctx->alpha == 1.0f;
    P.beta = beta;
    P.capacity = rank ? ctx->rank_sorted_n : ctx->capacity;  // only the sorted items have a rank
    P.out = out;
    P.slots = ctx->slots;
    P.ticket = ctx->tickets + TK_ISW;
    P.status = ctx->status;
    int ctas = (B + kThreads - 1) / kThreads;
    const int max_ctas = std::min(per_sm * ctx->num_sms, ctx->slot_n);
    if (ctas > max_ctas) ctas = max_ctas;
    // cooperative: the grid barrier needs every CTA resident at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, is_weights_kernel, P);
    per_note_launch();
    return cuda_status(e);
}
