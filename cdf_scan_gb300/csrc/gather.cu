// gather.cu -- per_gather: out[k] = rows[idx[k]] for B sampled indices, rows
// of `chunks` x 16 bytes (the transitions of a replay buffer, one row per
// item).  The copy of per_step_gather's fused path, as its own launch.
#include <algorithm>

#include "gather_core.cuh"
#include "internal.h"

namespace {

constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(const uint4* __restrict__ rows, int64_t n_rows,
                                                                     int chunks, const int32_t* __restrict__ idx,
                                                                     int B, uint4* __restrict__ out, int* status) {
    __shared__ int s_k[kGatherThreads / 32][32];
    __shared__ int s_i[kGatherThreads / 32][32];
    const int warp = threadIdx.x >> 5;
    bool bad = false;
    // grid-stride over rounds of one index per thread; the loop bound is
    // uniform, so whole warps take part in every call
    for (int k0 = blockIdx.x * kGatherThreads; k0 < B; k0 += gridDim.x * kGatherThreads) {
        const int k = k0 + threadIdx.x;
        const bool hit = k < B;
        const int i = hit ? __ldg(idx + k) : 0;
        if (hit && (i < 0 || i >= n_rows)) bad = true;
        gather_hits_warp(rows, n_rows, chunks, out, hit, k, i, s_k[warp], s_i[warp]);
    }
    if (bad) atomicOr(status, ST_VALUE);
}

}  // namespace

per_status launch_gather(per_ctx* ctx, const void* rows, int64_t row_bytes, const int32_t* idx, int B, void* out,
                         cudaStream_t s) {
    const int chunks = static_cast<int>(row_bytes / 16);
    const int64_t want = (static_cast<int64_t>(B) + kGatherThreads - 1) / kGatherThreads;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(want, 16LL * ctx->num_sms));
    gather_rows_kernel<<<grid, kGatherThreads, 0, s>>>(static_cast<const uint4*>(rows), ctx->capacity, chunks, idx, B,
                                                       static_cast<uint4*>(out), ctx->status);
    per_note_launch();
    return cuda_status(cudaGetLastError());
}
