// rank.cu -- rank-based PER.  The segment-tree page (foxhunt, "Non-Goals")
// names rank-based PER as another code path without defining it; the reading
// used here is the usual one: rank 1 is the highest stored priority (ties:
// lower index first), the item of rank r gets priority 1 / r, and the
// proportional machinery -- q^alpha, the CDF, stratified thresholds, IS
// weights -- runs over ranks.
//
// launch_rank_build sorts the priorities with a stable LSD radix sort: four
// passes of 8-bit digits over a 32-bit key whose ascending order is
// descending priority.  It leaves order[r] = the item of rank r + 1 and
// rank_of[order[r]] = r, and -- when the size changed -- fills the rank
// priorities q[r] = fl32(1 / (r + 1)) and builds their CDF with the scan
// kernels.  Sampling draws ranks from that CDF with the scan-path sampler and
// writes order[rank].
//
// One radix pass is three launches:
//   hist    -- per-tile digit counts, stored digit-major: counts[d][tile];
//   scan    -- one CTA per digit: exclusive scan of counts[d][*] across the
//              tiles, and the digit's total;
//   scatter -- every CTA scans the 256 totals (the digits' first positions),
//              ranks its tile's keys stably and writes them out.
// Inside a tile, warp w owns the contiguous keys [w * 512, (w + 1) * 512) and
// ranks them in 16 rounds of 32 with __match_any_sync peer groups and
// warp-private digit counters; the warps then take digit offsets in warp
// order.  Key order inside a tile is therefore kept, and across tiles the
// scan keeps tile order: the sort is stable.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kSortThreads = 256;
constexpr int kSortItems = kRankTile / kSortThreads;  // 16 keys per thread
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kWarpKeys = kRankTile / kSortWarps;     // 512 keys per warp
constexpr int kScanThreads = 1024;
constexpr int kRankMaxTiles = static_cast<int>(kRankMaxN / kRankTile);
static_assert(kSortThreads == kRadixDigits, "one thread per digit");
static_assert(kWarpKeys == 32 * kSortItems, "a warp ranks 32 keys per round");
static_assert(kRankMaxTiles <= 4 * kScanThreads, "the digit scan takes at most 4 tiles per thread");

// Ascending keys = descending priorities: non-negative floats order like
// their bit patterns, and -0 and +0 share one key.
__device__ __forceinline__ unsigned rank_key(float p) { return ~__float_as_uint(p + 0.f); }

struct SortParams {
    const float* prio;         // pass 0 reads keys from the priorities, values = item indices
    const unsigned* keys_in;   // later passes
    const int32_t* vals_in;
    unsigned* keys_out;        // nullptr in the last pass
    int32_t* vals_out;
    int32_t* rank_of;          // last pass only: rank_of[item] = its position
    unsigned* counts;          // [kRadixDigits][tiles]
    unsigned* totals;          // [kRadixDigits]
    int* status;
    int n;
    int tiles;
    int shift;
    bool first;
};

__device__ __forceinline__ unsigned key_at(const SortParams& S, int i) {
    return S.first ? rank_key(__ldg(S.prio + i)) : __ldg(S.keys_in + i);
}

__device__ __forceinline__ int32_t val_at(const SortParams& S, int i) { return S.first ? i : __ldg(S.vals_in + i); }

__global__ void __launch_bounds__(kSortThreads) radix_hist_kernel(SortParams S) {
    __shared__ unsigned h[kRadixDigits];
    h[threadIdx.x] = 0u;
    __syncthreads();
    const int base = blockIdx.x * kRankTile;
    bool bad = false;
#pragma unroll 4
    for (int e = 0; e < kSortItems; ++e) {
        const int i = base + e * kSortThreads + threadIdx.x;
        if (i < S.n) {
            if (S.first) bad |= !(__ldg(S.prio + i) >= 0.f);  // negative or NaN
            atomicAdd(&h[(key_at(S, i) >> S.shift) & 255u], 1u);
        }
    }
    if (bad) atomicOr(S.status, ST_VALUE);
    __syncthreads();
    S.counts[threadIdx.x * S.tiles + blockIdx.x] = h[threadIdx.x];
}

// CTA d: counts[d][t] becomes the number of keys with digit d in tiles < t,
// and totals[d] the number in all tiles.  Thread j takes tiles 4j .. 4j+3.
__global__ void __launch_bounds__(kScanThreads) radix_digit_scan_kernel(unsigned* counts, unsigned* totals,
                                                                        int tiles) {
    __shared__ unsigned s_w[kScanThreads / 32];
    unsigned* row = counts + static_cast<int64_t>(blockIdx.x) * tiles;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t0 = threadIdx.x * 4;
    unsigned v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = t0 + e < tiles ? row[t0 + e] : 0u;
    const unsigned mine = v[0] + v[1] + v[2] + v[3];
    unsigned x = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned y = __shfl_up_sync(PER_FULL_MASK, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    if (warp == 0) {
        unsigned w = s_w[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned y = __shfl_up_sync(PER_FULL_MASK, w, d);
            if (lane >= d) w += y;
        }
        s_w[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    unsigned run = (warp > 0 ? s_w[warp - 1] : 0u) + (x - mine);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if (t0 + e < tiles) row[t0 + e] = run;
        run += v[e];
    }
    if (threadIdx.x == 0) totals[blockIdx.x] = s_w[31];
}

__global__ void __launch_bounds__(kSortThreads) radix_scatter_kernel(SortParams S) {
    __shared__ unsigned s_cnt[kSortWarps][kRadixDigits];  // per-warp digit counts, then the warps' offsets
    __shared__ unsigned s_base[kRadixDigits];             // this tile's first position per digit
    __shared__ unsigned s_w[kSortWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kSortWarps * kRadixDigits; i += kSortThreads) (&s_cnt[0][0])[i] = 0u;
    {  // exclusive scan of the digit totals (thread = digit), plus this tile's offset
        const unsigned t = S.totals[threadIdx.x];
        unsigned x = t;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned y = __shfl_up_sync(PER_FULL_MASK, x, d);
            if (lane >= d) x += y;
        }
        if (lane == 31) s_w[warp] = x;
        __syncthreads();
        unsigned before = 0u;
        for (int w = 0; w < warp; ++w) before += s_w[w];
        s_base[threadIdx.x] = before + (x - t) + S.counts[threadIdx.x * S.tiles + blockIdx.x];
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    const int base = blockIdx.x * kRankTile + warp * kWarpKeys;
    unsigned key[kSortItems];
    unsigned pos[kSortItems];  // position among the warp's keys of the same digit
#pragma unroll
    for (int r = 0; r < kSortItems; ++r) {
        const int i = base + r * 32 + lane;
        const bool ok = i < S.n;
        key[r] = ok ? key_at(S, i) : 0u;
        const unsigned d = ok ? (key[r] >> S.shift) & 255u : 256u;  // 256: past the end, no counter
        const unsigned peers = __match_any_sync(PER_FULL_MASK, d);
        const int leader = __ffs(peers) - 1;
        unsigned old = 0u;
        if (ok && lane == leader) {
            old = s_cnt[warp][d];
            s_cnt[warp][d] = old + __popc(peers);
        }
        old = __shfl_sync(PER_FULL_MASK, old, leader);
        pos[r] = old + __popc(peers & lt);
    }
    __syncthreads();
    {  // per digit (thread = digit): the warps' offsets inside the tile, in warp order
        const int d = threadIdx.x;
        unsigned run = 0u;
#pragma unroll
        for (int w = 0; w < kSortWarps; ++w) {
            const unsigned c = s_cnt[w][d];
            s_cnt[w][d] = run;
            run += c;
        }
    }
    __syncthreads();
    bool bad = false;
#pragma unroll
    for (int r = 0; r < kSortItems; ++r) {
        const int i = base + r * 32 + lane;
        if (i >= S.n) continue;
        const unsigned d = (key[r] >> S.shift) & 255u;
        const unsigned dst = s_base[d] + s_cnt[warp][d] + pos[r];
        if (dst >= static_cast<unsigned>(S.n)) {  // only if the counts were inconsistent
            bad = true;
            continue;
        }
        const int32_t v = val_at(S, i);
        if (S.keys_out) S.keys_out[dst] = key[r];
        S.vals_out[dst] = v;
        if (S.rank_of) S.rank_of[v] = static_cast<int32_t>(dst);
    }
    if (bad) atomicOr(S.status, ST_RANGE);
}

// q[r] = fl32(1 / (r + 1)), correctly rounded (r + 1 <= 2^24 is exact in fp32).
__global__ void rank_priorities_kernel(float* q, int n) {
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < n; r += gridDim.x * blockDim.x)
        q[r] = __fdiv_rn(1.0f, __int2float_rn(r + 1));
}

}  // namespace

per_status launch_rank_build(per_ctx* ctx, cudaStream_t s) {
    const int n = static_cast<int>(ctx->size);
    if (n < 1 || n > kRankMaxN) return PER_ERR_STATE;
    const int tiles = (n + kRankTile - 1) / kRankTile;
    SortParams S = {};
    S.prio = ctx->prio;
    S.counts = ctx->rank_counts;
    S.totals = ctx->rank_totals;
    S.status = ctx->status;
    S.n = n;
    S.tiles = tiles;
    // pass 0: priorities -> (keys1, vals1); 1 -> (keys0, order); 2 -> (keys1, vals1); 3 -> order
    for (int pass = 0; pass < 4; ++pass) {
        S.first = pass == 0;
        S.shift = 8 * pass;
        const bool odd = (pass & 1) != 0;
        S.keys_in = odd ? ctx->rank_keys1 : ctx->rank_keys0;
        S.vals_in = odd ? ctx->rank_vals1 : ctx->rank_order;
        S.keys_out = pass == 3 ? nullptr : (odd ? ctx->rank_keys0 : ctx->rank_keys1);
        S.vals_out = odd ? ctx->rank_order : ctx->rank_vals1;
        S.rank_of = pass == 3 ? ctx->rank_of : nullptr;
        radix_hist_kernel<<<static_cast<unsigned>(tiles), kSortThreads, 0, s>>>(S);
        radix_digit_scan_kernel<<<kRadixDigits, kScanThreads, 0, s>>>(ctx->rank_counts, ctx->rank_totals, tiles);
        radix_scatter_kernel<<<static_cast<unsigned>(tiles), kSortThreads, 0, s>>>(S);
    }
    per_note_launch(12);
    if (cudaGetLastError() != cudaSuccess) return PER_ERR_CUDA;
    ctx->rank_sorted_n = n;
    if (ctx->rank_q_n != n) {  // q and its CDF depend on n (and the context's alpha) only
        const unsigned grid = static_cast<unsigned>(std::min(1024, (n + 255) / 256));
        rank_priorities_kernel<<<grid, 256, 0, s>>>(ctx->rank_q, n);
        per_note_launch();
        if (cudaGetLastError() != cudaSuccess) return PER_ERR_CUDA;
        const per_status st = launch_build_cdf_of(ctx, ctx->rank_q, n, ctx->rank_cdf, ctx->rank_coarse, s);
        if (st != PER_OK) return st;
        ctx->rank_q_n = n;
    }
    return PER_OK;
}
