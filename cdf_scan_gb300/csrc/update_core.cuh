// update_core.cuh -- the scan-mode priority update (p[idx_k] = new_k, the
// last occurrence of an index in batch order wins), shared by the update
// kernel (tree.cu) and the fused PER step (step.cu).  Two grid-wide phases
// with a grid barrier between them:
//   elect: every batch position k raises winner[idx_k] to (epoch << 32 | k)
//          with a 64-bit atomicMax, so the largest position of each index
//          survives;
//   apply: each position that won writes its priority.
// The epoch is read by every CTA before the barrier and advanced once after
// it, so winner slots never need clearing.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace {

// Positions k = first, first + stride, ... of the batch.  Invalid indices
// set `bad` (ST_VALUE) and take no part.
__device__ __forceinline__ void update_elect(const int32_t* __restrict__ idx, int n, int64_t capacity,
                                             unsigned long long* winner, unsigned epoch, int first, int stride,
                                             bool& bad) {
    for (int k = first; k < n; k += stride) {
        const int32_t i = idx[k];
        if (i < 0 || i >= capacity) {
            bad = true;
            continue;
        }
        atomicMax(winner + i, (static_cast<unsigned long long>(epoch) << 32) | static_cast<unsigned>(k));
    }
}

// After the grid barrier: winners write their priorities (negative or NaN
// ones set `bad`).
__device__ __forceinline__ void update_apply(const int32_t* __restrict__ idx, const float* __restrict__ p, int n,
                                             int64_t capacity, const unsigned long long* winner,
                                             float* __restrict__ prio, unsigned epoch, int first, int stride,
                                             bool& bad) {
    for (int k = first; k < n; k += stride) {
        const int32_t i = idx[k];
        if (i < 0 || i >= capacity) continue;
        if (__ldcg(winner + i) == ((static_cast<unsigned long long>(epoch) << 32) | static_cast<unsigned>(k))) {
            const float v = p[k];
            if (!(v >= 0.f)) bad = true;
            prio[i] = v;
        }
    }
}

}  // namespace
