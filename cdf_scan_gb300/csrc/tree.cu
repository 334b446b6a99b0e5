// tree.cu -- the sum segment tree (foxhunt "GPU Segment Tree for PER
// Sampling"): layout from section "Tree Layout" (tree[0] unused, root 1,
// children 2j and 2j+1, leaf of item i at cap_pow2 + i), batched update and
// root-to-leaf sampling from section "Operations", priority^alpha folded into
// the update and insert/update/total from section "Integration".
//
// The design doc's update launches one thread per index that writes its leaf
// and walks to the root; threads sharing an ancestor race and duplicate
// indices land in arbitrary order.  Here every update is deterministic and
// equal, bit for bit, to rebuilding the whole tree in the fixed pairwise order
// tree[j] = tree[2j] + tree[2j+1]:
//
//  * small batches (n <= 1024, depth <= 20): one CTA sorts (index, position)
//    keys, keeps the last occurrence of each index, writes those leaves, builds
//    the sorted list of dirty nodes of every level, fetches the unchanged
//    sibling of every dirty node in one parallel round of loads, then
//    recomputes the dirty nodes level by level in shared memory;
//  * large batches: the last writer of each index is elected with a 64-bit
//    atomicMax on (epoch << 32 | position), the winners write their leaves,
//    and the tree is rebuilt bottom-up by a few level-group launches.
//
// Sampling stages the top levels of the tree in shared memory with one bulk
// copy and finishes the descent from L2.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace {

// ============================================================== sampling ====

constexpr int kTopLevels = 12;  // nodes [0, 2^13) = 32 KB staged per CTA

struct TreeSampleParams {
    const float* __restrict__ tree;
    int log2cap;
    int staged_levels;  // children of node j are staged iff j < 2^staged_levels
    int B;
    uint64_t seed, offset;
    const float* __restrict__ u01;
    int32_t* __restrict__ out;
    int* status;
};

template <int THREADS>
__global__ void __launch_bounds__(THREADS) sample_tree_kernel(TreeSampleParams P) {
    extern __shared__ __align__(128) float s_top[];
    __shared__ __align__(8) uint64_t s_bar;
    // at least 16 bytes (the bulk-copy granule; the tree allocation is padded)
    const unsigned top_bytes = max(16u, (2u << P.staged_levels) * 4u);
    if (threadIdx.x == 0) {
        mbar_init(&s_bar, 1);
        mbar_arrive_expect_tx(&s_bar, top_bytes);
        bulk_copy_g2s(s_top, P.tree, top_bytes, &s_bar);
    }
    const int k = blockIdx.x * THREADS + threadIdx.x;
    const float T = __ldg(P.tree + 1);
    float u = 0.f;
    if (k < P.B) {
        const float U = P.u01 ? P.u01[k] : u01_open_closed(P.seed, P.offset + static_cast<uint64_t>(k));
        u = stratified_threshold(k, U, static_cast<float>(P.B), T);
    }
    __syncthreads();  // barrier initialised before anyone waits on it
    if (!mbar_wait_bounded(&s_bar, 0)) atomicOr(P.status, ST_TIMEOUT);
    if (k >= P.B) return;
    if (!(T > 0.f)) {
        if (threadIdx.x == 0) atomicOr(P.status, ST_EMPTY);
        P.out[k] = 0;
        return;
    }
    const unsigned staged = 1u << P.staged_levels;
    unsigned j = 1;
    for (int d = 0; d < P.log2cap; ++d) {
        float L, R;
        if (j < staged) {
            L = s_top[2 * j];
            R = s_top[2 * j + 1];
        } else {
            const float2 lr = __ldg(reinterpret_cast<const float2*>(P.tree + 2 * static_cast<size_t>(j)));
            L = lr.x;
            R = lr.y;
        }
        if (u > L && R > 0.f) {
            u = __fsub_rn(u, L);
            j = 2 * j + 1;
        } else {
            j = 2 * j;
        }
    }
    P.out[k] = static_cast<int32_t>(j - (1u << P.log2cap));
}

// ================================================== pairwise rebuild ========

// One launch recomputes `levels` levels above level `bottom` (nodes
// [2^bottom, 2^(bottom+1))).  Each CTA owns 2^levels consecutive bottom nodes.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) rebuild_levels_kernel(float* __restrict__ tree, int bottom, int levels) {
    extern __shared__ float s_nodes[];
    const int width = 1 << levels;  // bottom nodes per CTA
    const size_t first = (static_cast<size_t>(1) << bottom) + static_cast<size_t>(blockIdx.x) * width;
    for (int i = threadIdx.x; i < width; i += THREADS) s_nodes[i] = tree[first + i];
    __syncthreads();
    size_t level_first = first;
    int w = width;
    for (int l = 0; l < levels; ++l) {
        const int half = w >> 1;
        level_first >>= 1;
        for (int i = threadIdx.x; i < half; i += THREADS) {
            const float v = __fadd_rn(s_nodes[2 * i], s_nodes[2 * i + 1]);
            tree[level_first + i] = v;
            s_nodes[i + width] = v;  // staging copy in the upper half
        }
        __syncthreads();
        for (int i = threadIdx.x; i < half; i += THREADS) s_nodes[i] = s_nodes[i + width];
        __syncthreads();
        w = half;
    }
}

per_status rebuild_tree(per_ctx* ctx, cudaStream_t s) {
    constexpr int kGroup = 12;
    int bottom = ctx->log2_cap;
    while (bottom > 0) {
        const int levels = bottom < kGroup ? bottom : kGroup;
        const unsigned ctas = 1u << (bottom - levels);
        const size_t smem = 2 * (static_cast<size_t>(1) << levels) * sizeof(float);
        rebuild_levels_kernel<256><<<ctas, 256, smem, s>>>(ctx->tree, bottom, levels);
        per_note_launch();
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return PER_ERR_CUDA;
        bottom -= levels;
    }
    return PER_OK;
}

// Leaves from raw priorities: leaf i = p_i^alpha for i < n, 0 otherwise.
__global__ void leaves_from_prio_kernel(float* __restrict__ tree, const float* __restrict__ prio, int64_t n,
                                        int64_t cap_pow2, float alpha, bool alpha_one, int* status) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= cap_pow2) return;
    float v = 0.f;
    if (i < n) {
        const float p = prio[i];
        if (!(p >= 0.f)) atomicOr(status, ST_VALUE);
        v = pow_alpha(p, alpha, alpha_one);
    }
    tree[cap_pow2 + i] = v;
}

// ====================================================== large-batch update ===

__global__ void elect_last_writer_kernel(const int32_t* __restrict__ idx, int n, int64_t capacity,
                                         unsigned long long* winner, const unsigned* ctrs, int* status) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n) return;
    const int32_t i = idx[k];
    if (i < 0 || i >= capacity) {
        atomicOr(status, ST_VALUE);
        return;
    }
    const unsigned epoch = ld_relaxed_u32(ctrs + CTR_UPD_EPOCH);
    atomicMax(winner + i, (static_cast<unsigned long long>(epoch) << 32) | static_cast<unsigned>(k));
}

__global__ void apply_winners_kernel(const int32_t* __restrict__ idx, const float* __restrict__ p, int n,
                                     int64_t capacity, const unsigned long long* __restrict__ winner,
                                     float* __restrict__ prio, float* __restrict__ tree, int64_t cap_pow2,
                                     float alpha, bool alpha_one, unsigned* ctrs, int* status) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned epoch = ld_relaxed_u32(ctrs + CTR_UPD_EPOCH);
    if (k < n) {
        const int32_t i = idx[k];
        if (i >= 0 && i < capacity &&
            winner[i] == ((static_cast<unsigned long long>(epoch) << 32) | static_cast<unsigned>(k))) {
            const float v = p[k];
            if (!(v >= 0.f)) atomicOr(status, ST_VALUE);
            prio[i] = v;
            if (tree) tree[cap_pow2 + i] = pow_alpha(v, alpha, alpha_one);
        }
    }
    // the last CTA advances the epoch for the next update
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned done = atomicAdd(ctrs + CTR_UPD_DONE, 1u);
        if (done == gridDim.x - 1u) {
            ctrs[CTR_UPD_DONE] = 0u;
            ctrs[CTR_UPD_EPOCH] = epoch + 1u;  // 2^32 updates before a wrap
        }
    }
}

// ====================================================== small-batch update ===

constexpr int kSmallN = 1024;       // one key per thread
constexpr int kSmallMaxDepth = 20;  // cap_pow2 <= 2^20
// Entries over all levels: sum_d min(2^d, 1024) for d = 0..20.
constexpr int kListCap = 1023 + 1024 * 11;

struct SmallSmem {
    unsigned long long key[kSmallN];
    int node[kListCap];
    float val[kListCap];
    float sib[kListCap];
    unsigned short cstart[kListCap];
    int level_off[kSmallMaxDepth + 2];
    int level_cnt[kSmallMaxDepth + 2];
    int warp_cnt[32];
};

// Block-wide exclusive count of `flag` over the 1024 threads; returns the
// thread's offset and writes the total to *total (all threads).
__device__ __forceinline__ int block_excl_count(bool flag, int* warp_cnt, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned m = __ballot_sync(PER_FULL_MASK, flag);
    if (lane == 0) warp_cnt[warp] = __popc(m);
    __syncthreads();
    const int c = warp_cnt[lane];
    int incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(PER_FULL_MASK, incl, d);
        if (lane >= d) incl += y;
    }
    const int warp_excl = __shfl_sync(PER_FULL_MASK, incl - c, warp);
    *total = __shfl_sync(PER_FULL_MASK, incl, 31);
    __syncthreads();  // warp_cnt may be reused
    return warp_excl + __popc(m & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(kSmallN) small_update_kernel(const int32_t* __restrict__ idx,
                                                               const float* __restrict__ p, int n,
                                                               int64_t capacity, float* __restrict__ prio,
                                                               float* __restrict__ tree, int log2cap,
                                                               float alpha, bool alpha_one, int* status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SmallSmem& S = *reinterpret_cast<SmallSmem*>(smem_raw);
    const int tid = threadIdx.x;
    const unsigned cap_pow2 = 1u << log2cap;

    // ---- keys: (index << 32) | position; invalid / absent -> all ones -----
    unsigned long long key = ~0ull;
    if (tid < n) {
        const int32_t i = idx[tid];
        if (i >= 0 && i < capacity) key = (static_cast<unsigned long long>(i) << 32) | static_cast<unsigned>(tid);
        else atomicOr(status, ST_VALUE);
    }
    // ---- bitonic sort, ascending (shuffles below stride 32, smem above) ----
    for (int size = 2; size <= kSmallN; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const bool up = (tid & size) == 0;
            unsigned long long other;
            if (stride >= 32) {
                S.key[tid] = key;
                __syncthreads();
                other = S.key[tid ^ stride];
                __syncthreads();
            } else {
                other = __shfl_xor_sync(PER_FULL_MASK, key, stride);
            }
            const bool lower = (tid & stride) == 0;
            const bool take_min = (lower == up);
            key = take_min ? (other < key ? other : key) : (other > key ? other : key);
        }
    }
    S.key[tid] = key;
    __syncthreads();

    // ---- last occurrence of each index wins; write its leaf ----------------
    const bool valid = key != ~0ull;
    const unsigned my_index = static_cast<unsigned>(key >> 32);
    bool winner = false;
    if (valid) {
        const unsigned long long next = tid + 1 < kSmallN ? S.key[tid + 1] : ~0ull;
        winner = next == ~0ull || static_cast<unsigned>(next >> 32) != my_index;
    }
    int total;
    const int e = block_excl_count(winner, S.warp_cnt, &total);
    if (tid == 0) {
        S.level_off[log2cap] = 0;
        S.level_cnt[log2cap] = total;
    }
    if (winner) {
        const float v = p[static_cast<unsigned>(key)];
        if (!(v >= 0.f)) atomicOr(status, ST_VALUE);
        const float leaf = pow_alpha(v, alpha, alpha_one);
        prio[my_index] = v;
        tree[cap_pow2 + my_index] = leaf;
        S.node[e] = static_cast<int>(cap_pow2 + my_index);
        S.val[e] = leaf;
    }
    __syncthreads();

    // ---- dirty-node lists, one level at a time (sorted, unique) ------------
    for (int d = log2cap; d > 0; --d) {
        const int off = S.level_off[d], cnt = S.level_cnt[d];
        const int next_off = off + cnt;
        bool first = false;
        int parent = 0;
        if (tid < cnt) {
            parent = S.node[off + tid] >> 1;
            first = tid == 0 || (S.node[off + tid - 1] >> 1) != parent;
        }
        int pcount;
        const int pe = block_excl_count(first, S.warp_cnt, &pcount);
        if (first) {
            S.node[next_off + pe] = parent;
            S.cstart[next_off + pe] = static_cast<unsigned short>(off + tid);
        }
        if (tid == 0) {
            S.level_off[d - 1] = next_off;
            S.level_cnt[d - 1] = pcount;
        }
        __syncthreads();
    }

    // ---- one parallel round: fetch every clean sibling of a dirty node -----
    const int entries = S.level_off[0] + S.level_cnt[0];
    for (int d = log2cap; d > 0; --d) {
        const int off = S.level_off[d], cnt = S.level_cnt[d];
        for (int t = tid; t < cnt; t += kSmallN) {
            const int j = S.node[off + t];
            const bool left = (j & 1) == 0;
            const bool sib_dirty = left ? (t + 1 < cnt && S.node[off + t + 1] == j + 1)
                                        : (t > 0 && S.node[off + t - 1] == j - 1);
            S.sib[off + t] = sib_dirty ? 0.f : __ldg(tree + (j ^ 1));
        }
    }
    (void)entries;
    __syncthreads();

    // ---- recompute dirty nodes bottom-up in the fixed left + right order ---
    for (int d = log2cap - 1; d >= 0; --d) {
        const int off = S.level_off[d], cnt = S.level_cnt[d];
        const int coff = S.level_off[d + 1], ccnt = S.level_cnt[d + 1];
        for (int t = tid; t < cnt; t += kSmallN) {
            const int j = S.node[off + t];
            const int c0 = S.cstart[off + t];
            float left, right;
            if (S.node[c0] == 2 * j) {
                left = S.val[c0];
                right = (c0 + 1 < coff + ccnt && S.node[c0 + 1] == 2 * j + 1) ? S.val[c0 + 1] : S.sib[c0];
            } else {
                left = S.sib[c0];
                right = S.val[c0];
            }
            const float v = __fadd_rn(left, right);
            S.val[off + t] = v;
            tree[j] = v;
        }
        __syncthreads();
    }
}

}  // namespace

// ======================================================== host launchers ====

per_status launch_sample_tree(per_ctx* ctx, int B, uint64_t seed, uint64_t offset, const float* u01,
                              int32_t* out, cudaStream_t s) {
    TreeSampleParams P;
    P.tree = ctx->tree;
    P.log2cap = ctx->log2_cap;
    P.staged_levels = ctx->log2_cap < kTopLevels ? ctx->log2_cap : kTopLevels;
    P.B = B;
    P.seed = seed;
    P.offset = offset;
    P.u01 = u01;
    P.out = out;
    P.status = ctx->status;
    const size_t smem = std::max<size_t>(16, (static_cast<size_t>(2) << P.staged_levels) * sizeof(float));
    const int threads = B >= 64 * ctx->num_sms ? 256 : 128;
    const unsigned grid = static_cast<unsigned>((B + threads - 1) / threads);
    if (threads == 256) sample_tree_kernel<256><<<grid, 256, smem, s>>>(P);
    else sample_tree_kernel<128><<<grid, 128, smem, s>>>(P);
    per_note_launch();
    return cuda_status(cudaGetLastError());
}

per_status launch_tree_from_prio(per_ctx* ctx, cudaStream_t s) {
    const int64_t cap = ctx->cap_pow2;
    leaves_from_prio_kernel<<<static_cast<unsigned>((cap + 255) / 256), 256, 0, s>>>(
        ctx->tree, ctx->prio, ctx->size, cap, ctx->alpha, ctx->alpha == 1.0f, ctx->status);
    per_note_launch();
    if (cudaGetLastError() != cudaSuccess) return PER_ERR_CUDA;
    return rebuild_tree(ctx, s);
}

per_status launch_update(per_ctx* ctx, const int32_t* idx, const float* p, int n, cudaStream_t s) {
    const bool has_tree = (ctx->flags & PER_TREE) != 0;
    if (has_tree && n <= kSmallN && ctx->log2_cap <= kSmallMaxDepth) {
        static bool attr_set = false;  // per process; the attribute is per function
        const size_t smem = sizeof(SmallSmem);
        if (!attr_set) {
            if (cudaFuncSetAttribute(small_update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)) != cudaSuccess)
                return PER_ERR_CUDA;
            attr_set = true;
        }
        small_update_kernel<<<1, kSmallN, smem, s>>>(idx, p, n, ctx->capacity, ctx->prio, ctx->tree,
                                                     ctx->log2_cap, ctx->alpha, ctx->alpha == 1.0f, ctx->status);
        per_note_launch();
        return cuda_status(cudaGetLastError());
    }
    const unsigned grid = static_cast<unsigned>((n + 255) / 256);
    elect_last_writer_kernel<<<grid, 256, 0, s>>>(idx, n, ctx->capacity, ctx->winner, ctx->ctrs, ctx->status);
    apply_winners_kernel<<<grid, 256, 0, s>>>(idx, p, n, ctx->capacity, ctx->winner, ctx->prio,
                                              has_tree ? ctx->tree : nullptr, ctx->cap_pow2, ctx->alpha,
                                              ctx->alpha == 1.0f, ctx->ctrs, ctx->status);
    per_note_launch(2);
    if (cudaGetLastError() != cudaSuccess) return PER_ERR_CUDA;
    return has_tree ? rebuild_tree(ctx, s) : PER_OK;
}
