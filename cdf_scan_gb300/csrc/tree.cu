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
//  * small batches (n <= 4096): one thread-block cluster of up to 16 CTAs,
//    CTA r owning the r-th subtree below the top levels, so every duplicate
//    of an index meets in one CTA: a shared-memory hash table keeps the last
//    occurrence of each index, the winners write their leaves, and the dirty
//    64-wide subtrees are recomputed six levels per pass by one warp each;
//    after one cluster barrier CTA 0 recomputes the few top levels;
//  * large batches: the last writer of each index is elected with a 64-bit
//    atomicMax on (epoch << 32 | position), the winners write their leaves,
//    and the tree is rebuilt bottom-up by a few level-group launches.
//
// Sampling stages the top levels of the tree in shared memory with one bulk
// copy and finishes the descent from L2.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "update_core.cuh"

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
    bool iid;  // thresholds U_k * T (foxhunt "CUDA Kernels") instead of stratified
    int32_t* __restrict__ out;
    int* status;
};

// One step of the descent (foxhunt "Operations" / Sample, with the guard of
// the zero-sum right child): from node j with child sums L and R.
__device__ __forceinline__ void descend_step(float& u, unsigned& j, float L, float R) {
    if (u > L && R > 0.f) {
        u = __fsub_rn(u, L);
        j = 2 * j + 1;
    } else {
        j = 2 * j;
    }
}

// The N sums of one contiguous level run (N = 4, 8, 16: float4 loads; the
// run starts at a multiple of N floats, so they are aligned).
template <int N>
__device__ __forceinline__ void load_run(const float* p, float (&r)[N]) {
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p) + q);
        r[4 * q] = v.x;
        r[4 * q + 1] = v.y;
        r[4 * q + 2] = v.z;
        r[4 * q + 3] = v.w;
    }
}

// One descent step inside a loaded run: the node at position r of the level
// above has its children at 2r and 2r + 1 of this run (selects, no indexed
// register access).
template <int N>
__device__ __forceinline__ void descend_run(float& u, unsigned& r, const float (&run)[N]) {
    float L = run[0], R = run[1];
#pragma unroll
    for (int q = 1; q < N / 2; ++q) {
        L = r == static_cast<unsigned>(q) ? run[2 * q] : L;
        R = r == static_cast<unsigned>(q) ? run[2 * q + 1] : R;
    }
    descend_step(u, r, L, R);
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS) sample_tree_kernel(TreeSampleParams P) {
    extern __shared__ __align__(128) float s_top[];
    __shared__ __align__(8) uint64_t s_bar;
    // at least 16 bytes (the bulk-copy granule; the tree allocation is padded)
    const unsigned top_bytes = max(16u, (2u << P.staged_levels) * 4u);
    // launched as a programmatic dependent of the previous launch (typically
    // the previous update): nothing is read from global memory before it ends
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
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
        u = P.iid ? __fmul_rn(U, T) : stratified_threshold(k, U, static_cast<float>(P.B), T);
    }
    __syncthreads();  // barrier initialised before anyone waits on it
    if (!mbar_wait_bounded(&s_bar, 0)) atomicOr(P.status, ST_TIMEOUT);
    if (k >= P.B) return;
    if (!(T > 0.f)) {
        if (threadIdx.x == 0) atomicOr(P.status, ST_EMPTY);
        P.out[k] = 0;
        return;
    }
    unsigned j = 1;
    int d = 0;
    for (; d < P.staged_levels && d < P.log2cap; ++d)  // the staged levels, from shared memory
        descend_step(u, j, s_top[2 * j], s_top[2 * j + 1]);
    // the rest in groups of up to 4 levels: the nodes e levels below j are
    // the contiguous run [j * 2^e, (j + 1) * 2^e), so the 2 + 4 + 8 + 16
    // sums any 4 decisions can need come in one round of independent loads
    while (d < P.log2cap) {
        const int g = min(4, P.log2cap - d);
        const float* t = P.tree;
        float r1[2], r2[4], r3[8], r4[16];
        const float2 a = __ldg(reinterpret_cast<const float2*>(t + (static_cast<size_t>(j) << 1)));
        r1[0] = a.x;
        r1[1] = a.y;
        if (g >= 2) load_run<4>(t + (static_cast<size_t>(j) << 2), r2);
        if (g >= 3) load_run<8>(t + (static_cast<size_t>(j) << 3), r3);
        if (g >= 4) load_run<16>(t + (static_cast<size_t>(j) << 4), r4);
        unsigned r = 0;  // position below j at the current level
        descend_run<2>(u, r, r1);
        if (g >= 2) descend_run<4>(u, r, r2);
        if (g >= 3) descend_run<8>(u, r, r3);
        if (g >= 4) descend_run<16>(u, r, r4);
        j = (j << g) + r;
        d += g;
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
        v = pow_accurate(p, alpha, alpha_one);
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
            if (tree) tree[cap_pow2 + i] = pow_accurate(v, alpha, alpha_one);
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

// Scan-only contexts: the last occurrence of every index wins, in one
// cooperative launch (update_core.cuh: elect, grid barrier, apply); CTA 0
// advances the winner epoch after the barrier.
__global__ void __launch_bounds__(256) update_scan_kernel(const int32_t* __restrict__ idx,
                                                          const float* __restrict__ p, int n, int64_t capacity,
                                                          unsigned long long* winner, float* __restrict__ prio,
                                                          unsigned* ctrs, unsigned long long* ticket, int* status) {
    const unsigned epoch = ld_relaxed_u32(ctrs + CTR_UPD_EPOCH);
    const int first = blockIdx.x * blockDim.x + threadIdx.x, stride = gridDim.x * blockDim.x;
    bool bad = false;
    update_elect(idx, n, capacity, winner, epoch, first, stride, bad);
    grid_barrier(ticket, status, ST_TIMEOUT);
    if (blockIdx.x == 0 && threadIdx.x == 0) ctrs[CTR_UPD_EPOCH] = epoch + 1u;  // 2^32 updates before a wrap
    update_apply(idx, p, n, capacity, winner, prio, epoch, first, stride, bad);
    if (bad) atomicOr(status, ST_VALUE);
}

// ====================================================== small-batch update ===
//
// One CTA.  (1) Each index is inserted into a shared-memory hash table
// (index -> largest batch position, via atomicCAS / atomicMax), so the last
// occurrence of every index wins; the winners write raw priority and leaf.
// (2) The dirty part of the tree is recomputed in passes of six levels: for
// every updated leaf, the 64-wide subtree (64 nodes of the pass's bottom
// level) containing it is recomputed by one warp -- each lane adds one pair,
// then five shuffle levels -- and all its 63 nodes are written.  Clean nodes
// of a dirty subtree are rewritten with the value they already hold (every
// stored node equals the sum of its stored children), so the result is the
// full pairwise rebuild, bit for bit, and concurrent writers of one node
// always write the same value.  A per-pass hash set skips subtrees already
// claimed by another index.

constexpr int kSmallN = 4096;            // indices per batch on this path
constexpr int kSmallThreads = 1024;
constexpr int kHashSlots = 2 * kSmallN;  // power of two
constexpr unsigned kEmpty = 0xffffffffu;

struct SmallSmem {
    unsigned key[kHashSlots];    // index -> slot
    int pos[kHashSlots];         // largest batch position of the slot's index
    unsigned claim[kHashSlots];  // subtrees claimed in the current pass
    int slot_of[kSmallN];        // slot of batch entry k (-1: invalid index)
    unsigned leaf[kSmallN];      // distinct updated leaves
    unsigned job[kSmallN];       // distinct subtrees of the current pass
    int n_leaf, n_job;
};

__device__ __forceinline__ unsigned hash_u32(unsigned x) {
    x ^= x >> 16;
    x *= 0x7feb352dU;
    x ^= x >> 15;
    x *= 0x846ca68bU;
    x ^= x >> 16;
    return x;
}

// Insert `key` into a table of kHashSlots slots (at most kSmallN keys, so a
// free slot always exists); returns its slot and whether this call created it.
__device__ __forceinline__ int hash_insert(unsigned* keys, unsigned key, bool& inserted) {
    unsigned h = hash_u32(key) & (kHashSlots - 1);
    for (int probe = 0; probe < kHashSlots; ++probe) {
        const unsigned prev = atomicCAS(&keys[h], kEmpty, key);
        if (prev == kEmpty || prev == key) {
            inserted = prev == kEmpty;
            return static_cast<int>(h);
        }
        h = (h + 1) & (kHashSlots - 1);
    }
    inserted = false;
    return -1;
}

// One warp recomputes up to kJobBatch subtrees at once.  Subtree j has bottom
// nodes [first_j, first_j + width) (width a power of two, 2..64) and is
// recomputed through log2(width) levels: lane l adds bottom pair l, then
// shuffles combine neighbours, always left + right.  The batch is processed
// level by level, so the kJobBatch shuffle chains are independent and their
// latencies overlap.
constexpr int kJobBatch = 8;

__device__ __forceinline__ void recompute_subtrees(float* tree, const unsigned* first, int count, int width,
                                                   int lane) {
    const int levels = 31 - __clz(width);
    const bool active = 2 * lane < width;
    float v[kJobBatch];
    unsigned node[kJobBatch];
#pragma unroll
    for (int j = 0; j < kJobBatch; ++j) {
        float2 ab = make_float2(0.f, 0.f);
        const unsigned f = j < count ? first[j] : 0u;
        if (j < count && active)  // plain loads: written earlier by this CTA or cluster
            ab = *reinterpret_cast<const float2*>(tree + f + 2 * lane);
        v[j] = __fadd_rn(ab.x, ab.y);
        node[j] = (f >> 1) + lane;
    }
#pragma unroll
    for (int j = 0; j < kJobBatch; ++j)
        if (j < count && active) tree[node[j]] = v[j];
    for (int l = 1; l < levels; ++l) {
        const unsigned delta = 1u << (l - 1);
        const bool writer = active && (lane & ((1 << l) - 1)) == 0;
        float right[kJobBatch];
#pragma unroll
        for (int j = 0; j < kJobBatch; ++j) right[j] = __shfl_down_sync(PER_FULL_MASK, v[j], delta);
#pragma unroll
        for (int j = 0; j < kJobBatch; ++j) {
            node[j] >>= 1;
            if (writer) {
                v[j] = __fadd_rn(v[j], right[j]);
                if (j < count) tree[node[j]] = v[j];
            }
        }
    }
}

// The same for subtrees of width 32 * M (M = 4 or 8: seven or eight levels):
// lane l folds bottom nodes [l*M, (l+1)*M) through log2(M) levels in
// registers, writing each level, then five shuffle levels fold the 32 lane
// values -- the same sums, always left + right, as the pairwise rebuild.
template <int M, int JB>
__device__ __forceinline__ void recompute_wide(float* tree, const unsigned* first, int count, int lane) {
    static_assert(M == 4 || M == 8, "four or eight bottom nodes per lane");
    constexpr int LM = M == 4 ? 2 : 3;
    // every job's loads first: the stores below may alias them as far as the
    // compiler knows, so loads issued after a store would wait one by one
    float x[JB][M];
#pragma unroll
    for (int j = 0; j < JB; ++j) {
#pragma unroll
        for (int q = 0; q < M / 4; ++q) {
            float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < count)  // plain loads: written earlier by this CTA
                t = *reinterpret_cast<const float4*>(tree + first[j] + M * lane + 4 * q);
            x[j][4 * q] = t.x;
            x[j][4 * q + 1] = t.y;
            x[j][4 * q + 2] = t.z;
            x[j][4 * q + 3] = t.w;
        }
    }
    float v[JB];
    unsigned node[JB];
#pragma unroll
    for (int j = 0; j < JB; ++j) {
        unsigned at = first[j] + M * lane;  // node of x[j][0]
#pragma unroll
        for (int l = 0, m = M / 2; l < LM; ++l, m /= 2) {
            at >>= 1;
#pragma unroll
            for (int q = 0; q < m; ++q) {
                x[j][q] = __fadd_rn(x[j][2 * q], x[j][2 * q + 1]);
                if (j < count) tree[at + q] = x[j][q];
            }
        }
        v[j] = x[j][0];
        node[j] = at;
    }
#pragma unroll
    for (int l = 1; l <= 5; ++l) {
        const unsigned delta = 1u << (l - 1);
        const bool writer = (lane & ((1 << l) - 1)) == 0;
        float right[JB];
#pragma unroll
        for (int j = 0; j < JB; ++j) right[j] = __shfl_down_sync(PER_FULL_MASK, v[j], delta);
#pragma unroll
        for (int j = 0; j < JB; ++j) {
            node[j] >>= 1;
            if (writer) {
                v[j] = __fadd_rn(v[j], right[j]);
                if (j < count) tree[node[j]] = v[j];
            }
        }
    }
}

// Append `value` to list[*count] for every lane with `take`, one shared
// atomic per warp.
__device__ __forceinline__ void warp_append(bool take, unsigned value, unsigned* list, int* count, int lane) {
    const unsigned m = __ballot_sync(PER_FULL_MASK, take);
    if (!m) return;
    int base = 0;
    const int leader = __ffs(m) - 1;
    if (lane == leader) base = atomicAdd(count, __popc(m));
    base = __shfl_sync(PER_FULL_MASK, base, leader);
    if (take) list[base + __popc(m & ((1u << lane) - 1u))] = value;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ unsigned cluster_ctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Launched as one cluster of C CTAs (C a power of two, 1..16, C <= cap/64).
// CTA r owns the leaves under node C + r, i.e. items [r*cap/C, (r+1)*cap/C):
// every duplicate of an index lands in the same CTA, so the last-writer rule
// and the subtree recompute are CTA-local and the C subtrees are disjoint.
// After one cluster barrier CTA 0 recomputes the top log2(C) levels.
__global__ void __launch_bounds__(kSmallThreads) small_update_kernel(const int32_t* __restrict__ idx,
                                                                     const float* __restrict__ p, int n,
                                                                     int64_t capacity, float* __restrict__ prio,
                                                                     float* tree, int log2cap, float alpha,
                                                                     bool alpha_one, int* status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SmallSmem& S = *reinterpret_cast<SmallSmem*>(smem_raw);
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    constexpr int kWarpsPerCta = kSmallThreads / 32;
    const unsigned cap_pow2 = 1u << log2cap;
    const unsigned C = gridDim.x;               // cluster size == grid size
    const unsigned rank = cluster_ctarank();
    const int top = 31 - __clz(C);              // level of the CTA subtree roots
    const unsigned span = cap_pow2 >> top;      // leaves per CTA
    const unsigned lo = rank * span;

    for (int i = tid; i < kHashSlots; i += kSmallThreads) {
        S.key[i] = kEmpty;
        S.pos[i] = -1;
        S.claim[i] = kEmpty;
    }
    if (tid == 0) S.n_leaf = 0;
    // launched as a programmatic dependent of the previous launch (typically
    // the sampler): nothing is read from global memory before it ends
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();

    // ---- (1) the last occurrence of each index wins ---------------------------
    for (int k = tid; k < n; k += kSmallThreads) {
        const int32_t i = idx[k];
        int slot = -1;
        if (i >= 0 && i < capacity) {
            if (static_cast<unsigned>(i) - lo < span) {
                bool ins;
                slot = hash_insert(S.key, static_cast<unsigned>(i), ins);
                atomicMax(&S.pos[slot], k);
            }
        } else if (rank == 0) {
            atomicOr(status, ST_VALUE);
        }
        S.slot_of[k] = slot;
    }
    __syncthreads();
    for (int k0 = 0; k0 < n; k0 += kSmallThreads) {  // warp-uniform trip count
        const int k = k0 + tid;
        bool win = false;
        unsigned i = 0;
        if (k < n) {
            const int slot = S.slot_of[k];
            if (slot >= 0 && S.pos[slot] == k) {
                win = true;
                i = S.key[slot];
                const float v = p[k];
                if (!(v >= 0.f)) atomicOr(status, ST_VALUE);
                prio[i] = v;
                tree[cap_pow2 + i] = pow_accurate(v, alpha, alpha_one);
            }
        }
        warp_append(win, i, S.leaf, &S.n_leaf, lane);
    }
    __syncthreads();
    const int n_leaf = S.n_leaf;

    // ---- (2) recompute this CTA's dirty subtrees, up to eight levels per pass --
    for (int bottom = log2cap; bottom > top;) {
        const int levels = bottom - top < 8 ? bottom - top : 8;
        const int width = 1 << levels;
        const int shift = (log2cap - bottom) + levels;  // leaf >> shift = subtree number
        if (tid == 0) S.n_job = 0;
        __syncthreads();
        for (int w0 = 0; w0 < n_leaf; w0 += kSmallThreads) {  // warp-uniform trip count
            const int w = w0 + tid;
            const bool has = w < n_leaf;
            const unsigned sub = has ? S.leaf[w] >> shift : 0xffffffffu;
            // one claim per distinct subtree of the warp, then one per table
            const unsigned same = __match_any_sync(PER_FULL_MASK, sub);
            bool ins = false;
            if (has && lane == __ffs(same) - 1) hash_insert(S.claim, sub, ins);
            warp_append(ins, sub, S.job, &S.n_job, lane);
        }
        __syncthreads();
        const int n_job = S.n_job;
        const int jb = width <= 64 ? kJobBatch : kJobBatch / 2;  // subtrees per warp at once
        for (int j0 = warp * jb; j0 < n_job; j0 += kWarpsPerCta * jb) {
            unsigned first[kJobBatch];
            const int count = n_job - j0 < jb ? n_job - j0 : jb;
#pragma unroll
            for (int j = 0; j < kJobBatch; ++j)
                first[j] = j < count ? (1u << bottom) + S.job[j0 + j] * static_cast<unsigned>(width) : 0u;
            if (width <= 64)
                recompute_subtrees(tree, first, count, width, lane);
            else if (width == 128)
                recompute_wide<4, kJobBatch / 2>(tree, first, count, lane);
            else
                recompute_wide<8, kJobBatch / 2>(tree, first, count, lane);
        }
        for (int i = tid; i < kHashSlots; i += kSmallThreads) S.claim[i] = kEmpty;
        __syncthreads();  // this pass's nodes written (visible to the CTA) and claims cleared
        bottom -= levels;
    }

    // ---- (3) the top levels, from the C subtree roots ---------------------------
    if (C > 1) {
        cluster_sync_all();  // every CTA's subtree root is written (release/acquire)
        if (rank == 0 && warp == 0) {
            const unsigned first = C;  // nodes [C, 2C) are the subtree roots
            recompute_subtrees(tree, &first, 1, static_cast<int>(C), lane);
        }
    }
}

}  // namespace

// ======================================================== host launchers ====

per_status launch_sample_tree(per_ctx* ctx, int B, uint64_t seed, uint64_t offset, const float* u01, bool iid,
                              int32_t* out, cudaStream_t s) {
    TreeSampleParams P;
    P.tree = ctx->tree;
    P.log2cap = ctx->log2_cap;
    P.staged_levels = ctx->log2_cap < kTopLevels ? ctx->log2_cap : kTopLevels;
    P.B = B;
    P.seed = seed;
    P.offset = offset;
    P.u01 = u01;
    P.iid = iid;
    P.out = out;
    P.status = ctx->status;
    const size_t smem = std::max<size_t>(16, (static_cast<size_t>(2) << P.staged_levels) * sizeof(float));
    const int threads = B >= 64 * ctx->num_sms ? 256 : 128;
    const unsigned grid = static_cast<unsigned>((B + threads - 1) / threads);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see the kernel's first lines
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = threads == 256 ? cudaLaunchKernelEx(&cfg, sample_tree_kernel<256>, P)
                                         : cudaLaunchKernelEx(&cfg, sample_tree_kernel<128>, P);
    per_note_launch();
    return cuda_status(e);
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
    if (has_tree && n <= kSmallN) {
        const size_t smem = sizeof(SmallSmem);
        static DeviceCache cache;  // largest schedulable cluster size, per device
        const int max_cluster = device_cached(cache, [&]() {
            if (cudaFuncSetAttribute(small_update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)) != cudaSuccess)
                return 0;
            const bool nonportable = cudaFuncSetAttribute(small_update_kernel,
                                                          cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                                     cudaSuccess;
            cudaGetLastError();
            int best = 1;
            for (int c = nonportable ? 16 : 8; c > 1; c >>= 1) {
                cudaLaunchConfig_t q = {};
                q.gridDim = dim3(c);
                q.blockDim = dim3(kSmallThreads);
                q.dynamicSmemBytes = smem;
                cudaLaunchAttribute qa[1];
                qa[0].id = cudaLaunchAttributeClusterDimension;
                qa[0].val.clusterDim.x = c;
                qa[0].val.clusterDim.y = 1;
                qa[0].val.clusterDim.z = 1;
                q.attrs = qa;
                q.numAttrs = 1;
                int nc = 0;
                if (cudaOccupancyMaxActiveClusters(&nc, small_update_kernel, &q) == cudaSuccess && nc > 0) {
                    best = c;
                    break;
                }
                cudaGetLastError();
            }
            return best;
        });
        if (max_cluster == 0) return PER_ERR_CUDA;
        int C = max_cluster;
        while (C > 1 && (ctx->cap_pow2 >> 6) < C) C >>= 1;  // at least 64 leaves per CTA
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(C));
        cfg.blockDim = dim3(kSmallThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(C);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see the kernel's first lines
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, small_update_kernel, idx, p, n, ctx->capacity, ctx->prio,
                                                 ctx->tree, ctx->log2_cap, ctx->alpha, ctx->alpha == 1.0f,
                                                 ctx->status);
        per_note_launch();
        return cuda_status(e);
    }
    if (!has_tree) {
        static DeviceCache cache;
        const int per_sm = device_cached(cache, []() {
            int b = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, update_scan_kernel, 256, 0) != cudaSuccess) return 0;
            return b < 1 ? 1 : b;
        });
        if (per_sm == 0) return PER_ERR_CUDA;
        int ctas = (n + 255) / 256;
        if (ctas > per_sm * ctx->num_sms) ctas = per_sm * ctx->num_sms;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ctas));
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, update_scan_kernel, idx, p, n, ctx->capacity, ctx->winner,
                                                 ctx->prio, ctx->ctrs, ctx->tickets + TK_UPD, ctx->status);
        per_note_launch();
        return cuda_status(e);
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
