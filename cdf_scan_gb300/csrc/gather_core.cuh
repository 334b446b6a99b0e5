// gather_core.cuh -- copying the sampled transitions out of a replay buffer:
// out_row[k] = rows[idx_k] for fixed-size rows of `chunks` x 16 bytes
// (PufferLib PR #615 samples a minibatch of transitions by index from its
// prioritized buffers; the copy is the last step of a PER step).
#pragma once

#include "common.cuh"

namespace {

// One warp copies the rows of up to 32 hits: lane l holds hit (k, idx) when
// `hit` is set.  The hits are compacted into s_k / s_i (32 entries, this
// warp's own), then the warp's lanes take the hits' 16-byte chunks in order
// (consecutive lanes, consecutive chunks of one row: coalesced on both
// sides), four chunks in flight per lane.  Every lane of the warp calls it.
// Rows whose index is outside [0, n_rows) are skipped (the caller flags them).
__device__ __forceinline__ void gather_hits_warp(const uint4* __restrict__ rows, int64_t n_rows, int chunks,
                                                 uint4* __restrict__ out, bool hit, int k, int idx, int* s_k,
                                                 int* s_i) {
    const int lane = threadIdx.x & 31;
    const unsigned m = __ballot_sync(PER_FULL_MASK, hit);
    if (m == 0u) return;
    if (hit) {
        const int pos = __popc(m & ((1u << lane) - 1u));
        s_k[pos] = k;
        s_i[pos] = idx;
    }
    __syncwarp();
    const int total = __popc(m) * chunks;
    constexpr int kInFlight = 4;
    for (int t0 = 0; t0 < total; t0 += 32 * kInFlight) {
        uint4 v[kInFlight];
        int h[kInFlight], ch[kInFlight];
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) {
            const int t = t0 + u * 32 + lane;
            h[u] = -1;
            if (t < total) {
                const int hh = t / chunks;
                ch[u] = t - hh * chunks;
                const int i = s_i[hh];
                if (i >= 0 && i < n_rows) {
                    h[u] = hh;
                    v[u] = __ldg(rows + static_cast<int64_t>(i) * chunks + ch[u]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kInFlight; ++u)
            if (h[u] >= 0) out[static_cast<int64_t>(s_k[h[u]]) * chunks + ch[u]] = v[u];
    }
    __syncwarp();  // s_k / s_i may be refilled by the next call
}

}  // namespace
