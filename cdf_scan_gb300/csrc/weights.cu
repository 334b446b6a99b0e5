// weights.cu -- importance-sampling weights for a sampled batch.
//
// w_k = (N * P(idx_k))^-beta / max_k (N * P(idx_k))^-beta with P(i) = pa_i /
// total (the PER correction the foxhunt design doc lists as unchanged under
// "Non-Goals").  N and the total cancel, so the kernel computes the
// equivalent max-normalised form w_k = (pa_min / pa_{idx_k})^beta, pa_min the
// smallest pa in the batch: the weight of the batch minimum is exactly 1.
//
// One persistent cooperative launch: pass 1 gathers pa for the batch (tree
// leaves, or p^alpha of the raw priorities) into the output buffer and
// reduces the minimum (warp shuffles, then an order-independent atomicMin on
// the float's bit pattern, valid for non-negative floats); a grid barrier with
// a bounded wait; pass 2 turns pa into weights in place.  The last CTA to
// leave resets the minimum for the next call.
#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kThreads = 512;

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

__device__ __forceinline__ void grid_barrier(unsigned* ctrs, int* status) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned gen = ld_relaxed_u32(ctrs + CTR_ISW_BAR_GEN);
        __threadfence();
        const unsigned arrived = atomicAdd(ctrs + CTR_ISW_BAR_COUNT, 1u);
        if (arrived == gridDim.x - 1u) {
            atomicExch(ctrs + CTR_ISW_BAR_COUNT, 0u);
            __threadfence();
            atomicAdd(ctrs + CTR_ISW_BAR_GEN, 1u);
        } else {
            unsigned spins = 0;
            while (ld_acquire_u32(ctrs + CTR_ISW_BAR_GEN) == gen) {
                if (++spins > kSpinLimit) {
                    atomicOr(status, ST_TIMEOUT);
                    break;
                }
                __nanosleep(spins < 64 ? 32 : 256);
            }
        }
        __threadfence();
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads) is_weights_kernel(IswParams P) {
    __shared__ float s_min[kThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
            pa = pow_alpha(__ldg(P.prio + i), P.alpha, P.alpha_one);
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
    grid_barrier(P.ctrs, P.status);
    const float pa_min = __uint_as_float(ld_relaxed_u32(P.ctrs + CTR_ISW_MIN));
    for (int k = blockIdx.x * kThreads + threadIdx.x; k < P.B; k += stride) {
        const float ratio = __fdiv_rn(pa_min, P.out[k]);
        P.out[k] = powf(ratio, P.beta);
    }
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

per_status is_weights_configure(int device, int* max_ctas) {
    int num_sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return PER_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, is_weights_kernel, kThreads, 0) != cudaSuccess)
        return PER_ERR_CUDA;
    *max_ctas = num_sms * (per_sm > 0 ? per_sm : 1);
    return PER_OK;
}

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
    static int max_ctas = 0;
    if (max_ctas == 0 && is_weights_configure(ctx->device, &max_ctas) != PER_OK) return PER_ERR_CUDA;
    // ~4 items per thread, never more CTAs than can be resident at once
    int ctas = (B + 4 * kThreads - 1) / (4 * kThreads);
    if (ctas > max_ctas) ctas = max_ctas;
    if (ctas < 1) ctas = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, is_weights_kernel, P);
    per_note_launch();
    return cuda_status(e);
}
