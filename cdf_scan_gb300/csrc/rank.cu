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
// Every pass works tile by tile (256 threads, ITEMS keys each):
//   rank   -- warp w owns the tile's keys [w * 32 * ITEMS, (w + 1) * 32 *
//             ITEMS) and ranks them round by round: the lanes holding the
//             same digit (found with one ballot per digit bit, or five
//             ballots on a representative lane -- see warp_rank) take
//             consecutive positions after the warp's running count of it;
//   place  -- the warps take digit offsets in warp order, the digits take
//             tile offsets in digit order, and each key goes to its slot of a
//             tile-local sorted copy in shared memory;
//   write  -- consecutive threads copy consecutive slots out, so the keys of
//             one digit land in consecutive global positions (coalesced).
// Key order inside a tile is kept, and the cross-tile offsets keep tile
// order: the sort is stable.  The cross-tile offsets come from
//   large sizes -- three launches per pass: per-tile digit histograms
//             (digit-major), one CTA per digit scanning its row across the
//             tiles, then the tile pass above (one kernel per kind of pass:
//             first, middle, last), and after the last pass one launch that
//             returns rank_of's L2 lines to the normal eviction priority;
//   small sizes -- one cooperative launch for all four passes: each CTA
//             publishes its tile's digit counts (16 bits each, digit-major),
//             and after a grid barrier sums the counts of all tiles itself:
//             thread d reads digit d's row with at most 16 independent
//             16-byte loads, so the sum costs one round trip to L2.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kBigItems = kRankTile / kSortThreads;  // 16 keys per thread, 4096 per tile
constexpr int kSmallItems = 8;                       // 2048 keys per tile
constexpr int kSmallMaxTiles = 128;                  // cooperative path: n <= 262,144
constexpr int kScanThreads = 1024;
constexpr int kBigMaxTiles = static_cast<int>(kRankMaxN / kRankTile);
static_assert(kSortThreads == kRadixDigits, "one thread per digit");
static_assert(kBigMaxTiles <= 4 * kScanThreads, "the digit scan takes at most 4 tiles per thread");

// Ascending keys = descending priorities: non-negative floats order like
// their bit patterns, and -0 and +0 share one key.
__device__ __forceinline__ unsigned rank_key(float p) { return ~__float_as_uint(p + 0.f); }

// The last tile pass of large sizes writes rank_of in random order, 4 bytes
// at a time (the one-launch sort's at most 1 MiB stays in L2 anyway).  Stored
// with L2 eviction priority evict_last, a line stays in L2 until its 32
// entries have arrived instead of going back to DRAM part-written, over and
// over (16M: 598 -> 540 us for the sort; that pass wrote 370 MB to DRAM for
// 128 MB of order and rank_of).  restore_l2_priority_kernel then returns the
// lines to the normal priority, so that they do not hold L2 after the sort.
__device__ __forceinline__ void store_evict_last(int32_t* a, int32_t v) {
    unsigned long long pol;  // a pure value: the compiler may create it once per thread
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(a), "r"(v), "l"(pol) : "memory");
}

struct SortParams {
    const float* prio;
    unsigned* keys0;
    unsigned* keys1;
    int32_t* vals1;
    int32_t* order;
    int32_t* rank_of;
    unsigned* counts;  // large sizes: [kRadixDigits][tiles]; small: 16-bit, [kRadixDigits][row], row = tiles
                       // rounded up to 8
    unsigned* totals;  // [kRadixDigits] (large sizes)
    int* status;
    unsigned long long* ticket;
    int n;
    int tiles;
    int pass;  // large sizes: the pass of this launch
};

// Buffers of pass p: 0 reads the priorities and writes (keys1, vals1);
// 1 -> (keys0, order); 2 -> (keys1, vals1); 3 -> order and rank_of.
struct PassIO {
    const unsigned* keys_in;
    const int32_t* vals_in;
    unsigned* keys_out;  // nullptr in the last pass
    int32_t* vals_out;
    int shift;
    bool first, last;
};

// What a kernel knows of its pass at compile time: the first (priorities
// in, indices as values), a middle one, the last (order and rank_of out), or
// nothing (the one-launch sort, whose pass is a loop variable).
enum PassKind { kFirstPass, kMiddlePass, kLastPass, kAnyPass };

template <int K>
__device__ __forceinline__ bool first_pass(const PassIO& io) {
    return K == kAnyPass ? io.first : K == kFirstPass;
}
template <int K>
__device__ __forceinline__ bool last_pass(const PassIO& io) {
    return K == kAnyPass ? io.last : K == kLastPass;
}

__device__ __forceinline__ PassIO pass_io(const SortParams& S, int pass) {
    PassIO io;
    const bool odd = (pass & 1) != 0;
    io.first = pass == 0;
    io.last = pass == 3;
    io.shift = 8 * pass;
    io.keys_in = odd ? S.keys1 : S.keys0;
    io.vals_in = odd ? S.vals1 : S.order;
    io.keys_out = io.last ? nullptr : (odd ? S.keys0 : S.keys1);
    io.vals_out = odd ? S.order : S.vals1;
    return io;
}

// The tile pass's table of one lane per warp and digit (see warp_rank); the
// one-launch sort has none.
template <int ITEMS>
struct RankRep {};
template <>
struct RankRep<kBigItems> {
    unsigned char rep[kSortWarps][kRadixDigits + 4];
};

template <int ITEMS>
struct SortSmem : RankRep<ITEMS> {
    unsigned keys[kSortThreads * ITEMS];         // the tile, sorted by digit
    int32_t vals[kSortThreads * ITEMS];
    unsigned cnt[kSortWarps][kRadixDigits];      // per-warp digit counts, then local offsets
    int off[kRadixDigits];                       // global position - local slot, per digit
    unsigned w[kSortWarps];
};

// The lanes of the warp whose digit equals this lane's (valid lanes), or the
// invalid lanes (invalid lanes, which pass d = 0): one ballot per digit bit.
// Eight ballots cost far less than one __match_any_sync.  (The tile pass of
// large sizes takes its groups with five ballots instead: see warp_rank.)
__device__ __forceinline__ unsigned digit_peers(unsigned d, bool valid) {
    const unsigned v = __ballot_sync(PER_FULL_MASK, valid);
    unsigned peers = valid ? v : ~v;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const bool bit = ((d >> b) & 1u) != 0u;
        const unsigned m = __ballot_sync(PER_FULL_MASK, bit);
        peers &= bit ? m : ~m;
    }
    return peers;
}

// Exclusive scan of one value per thread over the CTA (thread order); *total
// receives the sum.  Reuses s_w: callers separate two uses by a barrier.
__device__ __forceinline__ unsigned block_excl_scan(unsigned v, unsigned* s_w, unsigned* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned y = __shfl_up_sync(PER_FULL_MASK, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    unsigned before = 0u, all = 0u;
#pragma unroll
    for (int w = 0; w < kSortWarps; ++w) {
        const unsigned c = s_w[w];
        if (w < warp) before += c;
        all += c;
    }
    *total = all;
    __syncthreads();
    return before + (x - v);
}

// Rank step: the warp's keys of this tile and, per key, its position among
// the warp's keys of the same digit; sm.cnt[warp][d] ends as the warp's count
// of digit d (sm.cnt zeroed by the caller).  Positions are below 32 * ITEMS
// and two share a register (round r in bits 16 * (r & 1) of pos[r / 2]):
// with one per register the tile pass spilled at 3 CTAs per SM.
//
// The tile pass (K != kAnyPass) finds each round's digit groups in two
// steps: every lane writes its lane number to its digit's byte of
// sm.rep[warp] and reads the byte back -- one lane of the group, the same for
// the whole group, whichever store landed -- and the groups are then the
// lanes with equal representatives, a 5-bit value: five ballots instead of
// eight.  The group's lanes read its running count together, and the
// representative adds the group's size.  16M sort: 553 -> 514 us.  The
// one-launch sort keeps the eight ballots and a leader's read (with the
// representative lane it measured 47.5 against 45.4 us at 262,144).
template <int ITEMS, int K>
__device__ __forceinline__ void warp_rank(const SortParams& S, const PassIO& io, int tile_base,
                                          unsigned (&key)[ITEMS], unsigned (&pos)[ITEMS / 2], SortSmem<ITEMS>& sm,
                                          bool& bad) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt = (1u << lane) - 1u;
    const int base = tile_base + warp * 32 * ITEMS;
    // all loads first, so that they are in flight together (the ballots below
    // would otherwise keep each round's load waiting for the previous round)
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {
        const int i = base + r * 32 + lane;
        key[r] = 0u;
        if (i < S.n) {
            if (first_pass<K>(io)) {
                // through L2 only (ld.global.cg): the 16M sort measured 599 us
                // this way and 641 us with the read-only path (ld.global.nc)
                const float p = __ldcg(S.prio + i);
                bad |= !(p >= 0.f);  // negative or NaN
                key[r] = rank_key(p);
            } else {
                key[r] = __ldcg(io.keys_in + i);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {
        const bool ok = base + r * 32 + lane < S.n;
        const unsigned d = ok ? (key[r] >> io.shift) & 255u : 0u;
        if constexpr (K == kAnyPass) {
            const unsigned peers = digit_peers(d, ok);
            const int leader = __ffs(peers) - 1;
            unsigned old = 0u;
            if (ok && lane == leader) {
                old = sm.cnt[warp][d];
                sm.cnt[warp][d] = old + __popc(peers);
            }
            old = __shfl_sync(PER_FULL_MASK, old, leader);
            const unsigned pr = old + __popc(peers & lt);  // < 32 * ITEMS
            pos[r >> 1] = (r & 1) ? (pos[r >> 1] | (pr << 16)) : pr;
        } else {
            unsigned char* slot = &sm.rep[warp][ok ? d : kRadixDigits];  // invalid lanes: a group of their own
            *slot = static_cast<unsigned char>(lane);
            __syncwarp();
            const int rep = *slot;
            unsigned peers = PER_FULL_MASK;
#pragma unroll
            for (int b = 0; b < 5; ++b) {
                const bool bit = ((rep >> b) & 1) != 0;
                const unsigned m = __ballot_sync(PER_FULL_MASK, bit);
                peers &= bit ? m : ~m;
            }
            const unsigned old = sm.cnt[warp][d];  // the group's lanes read one word
            __syncwarp();
            if (ok && lane == rep) sm.cnt[warp][d] = old + __popc(peers);
            const unsigned pr = old + __popc(peers & lt);  // < 32 * ITEMS
            pos[r >> 1] = (r & 1) ? (pos[r >> 1] | (pr << 16)) : pr;
        }
        __syncwarp();
    }
}

// Thread = digit d: turn the warps' counts of d into offsets in warp order;
// returns the tile's count of d.
template <int ITEMS>
__device__ __forceinline__ unsigned warp_offsets(SortSmem<ITEMS>& sm) {
    const int d = threadIdx.x;
    unsigned run = 0u;
#pragma unroll
    for (int w = 0; w < kSortWarps; ++w) {
        const unsigned c = sm.cnt[w][d];
        sm.cnt[w][d] = run;
        run += c;
    }
    return run;
}

// Place and write steps.  On entry sm.cnt[w][d] is the local slot of warp
// w's first key of digit d and sm.off[d] = global position - local slot.
template <int ITEMS, int K>
__device__ __forceinline__ void place_and_write(const SortParams& S, const PassIO& io, int tile_base,
                                                const unsigned (&key)[ITEMS], const unsigned (&pos)[ITEMS / 2],
                                                SortSmem<ITEMS>& sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int base = tile_base + warp * 32 * ITEMS;
    int32_t val[ITEMS];
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {  // loads first, all in flight together
        const int i = base + r * 32 + lane;
        val[r] = first_pass<K>(io) ? i : (i < S.n ? __ldcg(io.vals_in + i) : 0);
    }
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {
        const int i = base + r * 32 + lane;
        if (i >= S.n) continue;
        const unsigned d = (key[r] >> io.shift) & 255u;
        const unsigned slot = sm.cnt[warp][d] + ((pos[r >> 1] >> (16 * (r & 1))) & 0xffffu);
        if (slot >= static_cast<unsigned>(kSortThreads * ITEMS)) continue;  // only if the counts were inconsistent
        sm.keys[slot] = key[r];
        sm.vals[slot] = val[r];
    }
    __syncthreads();
    const int valid = min(kSortThreads * ITEMS, S.n - tile_base);
    bool bad = false;
    for (int j = threadIdx.x; j < valid; j += kSortThreads) {
        const unsigned k = sm.keys[j];
        const int32_t v = sm.vals[j];
        const unsigned dst = static_cast<unsigned>(sm.off[(k >> io.shift) & 255u] + j);
        if (dst >= static_cast<unsigned>(S.n) || static_cast<unsigned>(v) >= static_cast<unsigned>(S.n)) {
            // only if the counts were inconsistent
            bad = true;
            continue;
        }
        if (!last_pass<K>(io)) io.keys_out[dst] = k;
        io.vals_out[dst] = v;
        if constexpr (K == kLastPass) {
            store_evict_last(S.rank_of + v, static_cast<int32_t>(dst));  // restored after the pass
        } else {
            if (last_pass<K>(io)) S.rank_of[v] = static_cast<int32_t>(dst);  // the one-launch sort: 1 MiB at most
        }
    }
    if (bad) atomicOr(S.status, ST_RANGE);
}

// ---- large sizes: three launches per pass ----------------------------------

// Per-tile digit counts, stored digit-major: counts[d][tile], from per-warp
// sub-histograms of shared-memory atomics (plain atomics measured faster here
// than adding once per peer group found with ballots or __match_any_sync).
template <bool FIRST>
__global__ void __launch_bounds__(kSortThreads) radix_hist_kernel(SortParams S) {
    __shared__ unsigned h[kSortWarps][kRadixDigits];
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kSortWarps * kRadixDigits; i += kSortThreads) (&h[0][0])[i] = 0u;
    __syncthreads();
    // launched as a programmatic dependent of the previous pass's tile pass
    // (passes 1-3): its keys are complete only once that launch is done.
    // The digit scan may be scheduled only after this wait: the next tile
    // pass, scheduled once every digit-scan CTA has started, loads the keys
    // written by the previous tile pass before its own wait, and that launch
    // is two launches back -- a wait covers the launch directly before only.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const PassIO io = pass_io(S, S.pass);
    const int tile_base = blockIdx.x * kRankTile;
    bool bad = false;
    unsigned k[kBigItems];
    bool ok[kBigItems];
#pragma unroll
    for (int e = 0; e < kBigItems / 4; ++e) {  // all loads first, in flight together
        const int i0 = tile_base + (e * kSortThreads + threadIdx.x) * 4;
        if (i0 + 3 < S.n) {
            if (FIRST) {
                const float4 p = __ldg(reinterpret_cast<const float4*>(S.prio + i0));
                bad |= !(p.x >= 0.f) || !(p.y >= 0.f) || !(p.z >= 0.f) || !(p.w >= 0.f);
                k[4 * e] = rank_key(p.x); k[4 * e + 1] = rank_key(p.y);
                k[4 * e + 2] = rank_key(p.z); k[4 * e + 3] = rank_key(p.w);
            } else {
                const uint4 q = __ldcg(reinterpret_cast<const uint4*>(io.keys_in + i0));
                k[4 * e] = q.x; k[4 * e + 1] = q.y; k[4 * e + 2] = q.z; k[4 * e + 3] = q.w;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) ok[4 * e + c] = true;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = i0 + c;
                ok[4 * e + c] = i < S.n;
                k[4 * e + c] = 0u;
                if (i < S.n) {
                    if (FIRST) {
                        const float p = __ldg(S.prio + i);
                        bad |= !(p >= 0.f);
                        k[4 * e + c] = rank_key(p);
                    } else {
                        k[4 * e + c] = __ldcg(io.keys_in + i);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int c = 0; c < kBigItems; ++c)
        if (ok[c]) atomicAdd(&h[warp][(k[c] >> io.shift) & 255u], 1u);
    if (bad) atomicOr(S.status, ST_VALUE);
    __syncthreads();
    unsigned sum = 0u;
#pragma unroll
    for (int w = 0; w < kSortWarps; ++w) sum += h[w][threadIdx.x];
    S.counts[threadIdx.x * S.tiles + blockIdx.x] = sum;
}

// CTA d: counts[d][t] becomes the number of keys with digit d in tiles < t,
// and totals[d] the number in all tiles.  Thread j takes tiles 4j .. 4j+3.
__global__ void __launch_bounds__(kScanThreads) radix_digit_scan_kernel(unsigned* counts, unsigned* totals,
                                                                        int tiles) {
    __shared__ unsigned s_w[kScanThreads / 32];
    // the tile pass may start now: it loads and ranks its keys before it
    // waits for these offsets (those keys are complete: every histogram CTA
    // passed its wait for the previous tile pass before this launch began)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the histogram launch's counts
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

// The tile pass of large sizes: rank, place against the offsets of the
// histogram and digit-scan launches, write.
template <int K>
__global__ void __launch_bounds__(kSortThreads, 3) radix_scatter_kernel(SortParams S) {
    __shared__ SortSmem<kBigItems> sm;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the next histogram may be scheduled
    const PassIO io = pass_io(S, S.pass);
    const int d = threadIdx.x;
    for (int i = threadIdx.x; i < kSortWarps * kRadixDigits; i += kSortThreads) (&sm.cnt[0][0])[i] = 0u;
    __syncthreads();
    const int tile_base = blockIdx.x * kRankTile;
    unsigned key[kBigItems], pos[kBigItems / 2];
    bool bad = false;  // reported by the histogram launch
    warp_rank<kBigItems, K>(S, io, tile_base, key, pos, sm, bad);
    __syncthreads();
    const unsigned cnt_d = warp_offsets(sm);
    unsigned tile_total = 0u, all = 0u;
    const unsigned start_d = block_excl_scan(cnt_d, sm.w, &tile_total);
    // the digit-scan launch's offsets: launched as its programmatic
    // dependent, this CTA waits here for that launch to finish
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const unsigned digit_start = block_excl_scan(S.totals[d], sm.w, &all);
    const unsigned gbase = digit_start + S.counts[d * S.tiles + blockIdx.x];
#pragma unroll
    for (int w = 0; w < kSortWarps; ++w) sm.cnt[w][d] += start_d;
    sm.off[d] = static_cast<int>(gbase) - static_cast<int>(start_d);
    __syncthreads();
    place_and_write<kBigItems, K>(S, io, tile_base, key, pos, sm);
}

// ---- small sizes: all four passes in one cooperative launch ----------------
//
// One CTA per 2048-key tile, all resident.  Per pass: rank the tile, publish
// its digit counts (tile-major), grid barrier, sum every tile's counts (the
// keys before this tile per digit, and the digit totals), place and write,
// grid barrier.  Keys, values and counts written in the launch are read
// through L2 (ld.global.cg).
__global__ void __launch_bounds__(kSortThreads) radix_sort_small_kernel(SortParams S) {
    __shared__ SortSmem<kSmallItems> sm;
    const int d = threadIdx.x;
    const int tile_base = blockIdx.x * kSortThreads * kSmallItems;
    bool bad = false;
    for (int pass = 0; pass < 4; ++pass) {
        const PassIO io = pass_io(S, pass);
        for (int i = threadIdx.x; i < kSortWarps * kRadixDigits; i += kSortThreads) (&sm.cnt[0][0])[i] = 0u;
        __syncthreads();
        unsigned key[kSmallItems], pos[kSmallItems / 2];
        warp_rank<kSmallItems, kAnyPass>(S, io, tile_base, key, pos, sm, bad);
        __syncthreads();
        const unsigned cnt_d = warp_offsets(sm);
        unsigned tile_total = 0u, all = 0u;
        const unsigned start_d = block_excl_scan(cnt_d, sm.w, &tile_total);
        const int row = (S.tiles + 7) & ~7;
        unsigned short* c16 = reinterpret_cast<unsigned short*>(S.counts);
        c16[d * row + static_cast<int>(blockIdx.x)] = static_cast<unsigned short>(cnt_d);  // <= 2048
        if (!grid_barrier(S.ticket, S.status, ST_TIMEOUT)) return;
        const uint4* rp = reinterpret_cast<const uint4*>(c16 + d * row);
        uint4 q[kSmallMaxTiles / 8];
#pragma unroll
        for (int u = 0; u < kSmallMaxTiles / 8; ++u) q[u] = 8 * u < S.tiles ? __ldcg(rp + u) : make_uint4(0u, 0u, 0u, 0u);
        unsigned before = 0u, total = 0u;
#pragma unroll
        for (int u = 0; u < kSmallMaxTiles / 8; ++u) {
            const unsigned w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const int t = 8 * u + h;
                const unsigned v = (w[h >> 1] >> (16 * (h & 1))) & 0xffffu;
                if (t < S.tiles) total += v;
                if (t < static_cast<int>(blockIdx.x)) before += v;
            }
        }
        const unsigned digit_start = block_excl_scan(total, sm.w, &all);
#pragma unroll
        for (int w = 0; w < kSortWarps; ++w) sm.cnt[w][d] += start_d;
        sm.off[d] = static_cast<int>(digit_start + before) - static_cast<int>(start_d);
        __syncthreads();
        place_and_write<kSmallItems, kAnyPass>(S, io, tile_base, key, pos, sm);
        if (pass < 3 && !grid_barrier(S.ticket, S.status, ST_TIMEOUT)) return;
    }
    if (bad) atomicOr(S.status, ST_VALUE);
}

// Normal L2 eviction priority again for the 128-byte lines of a[0, n) (a
// 128-byte aligned; the last line lies in the same allocation).  Launched as a
// programmatic dependent of the last tile pass.
__global__ void __launch_bounds__(256) restore_l2_priority_kernel(const int32_t* a, int n) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t lines = (static_cast<int64_t>(n) * 4 + 127) / 128;
    for (int64_t l = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; l < lines;
         l += static_cast<int64_t>(gridDim.x) * blockDim.x)
        asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(a + l * 32) : "memory");
}

// q[r] = fl32(1 / (r + 1)), correctly rounded (r + 1 <= 2^24 is exact in fp32).
__global__ void rank_priorities_kernel(float* q, int n) {
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < n; r += gridDim.x * blockDim.x)
        q[r] = __fdiv_rn(1.0f, __int2float_rn(r + 1));
}

}  // namespace

static_assert(kSortThreads * kSmallItems == kRankSmallTile, "count buffer sized for the small tiles");

per_status launch_rank_build(per_ctx* ctx, cudaStream_t s) {
    const int n = static_cast<int>(ctx->size);
    if (n < 1 || n > kRankMaxN) return PER_ERR_STATE;
    SortParams S = {};
    S.prio = ctx->prio;
    S.keys0 = ctx->rank_keys0;
    S.keys1 = ctx->rank_keys1;
    S.vals1 = ctx->rank_vals1;
    S.order = ctx->rank_order;
    S.rank_of = ctx->rank_of;
    S.counts = ctx->rank_counts;
    S.totals = ctx->rank_totals;
    S.status = ctx->status;
    S.ticket = ctx->tickets + TK_RANK;
    S.n = n;
    static DeviceCache cache;  // resident CTAs per SM of the cooperative kernel
    const int per_sm = device_cached(cache, []() {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, radix_sort_small_kernel, kSortThreads, 0) != cudaSuccess)
            return 0;
        return b < 1 ? 1 : b;
    });
    if (per_sm == 0) return PER_ERR_CUDA;
    const int small_tiles = (n + kRankSmallTile - 1) / kRankSmallTile;
    if (small_tiles <= kSmallMaxTiles && small_tiles <= per_sm * ctx->num_sms) {
        S.tiles = small_tiles;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(small_tiles));
        cfg.blockDim = dim3(kSortThreads);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, radix_sort_small_kernel, S);
        per_note_launch();
        if (e != cudaSuccess) return PER_ERR_CUDA;
    } else {
        S.tiles = (n + kRankTile - 1) / kRankTile;
        // Each launch is a programmatic dependent of the one before it (but
        // the first, which follows whatever the stream ran before): it is
        // scheduled while that launch finishes and waits for it
        // (griddepcontrol.wait) before its first dependent read.  The tile
        // pass reads the keys of the tile pass before it early; the histogram
        // launch between them lets its dependents start only after its wait.
        auto launch = [&](auto kernel, unsigned grid, unsigned block, bool dependent, auto... args) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(grid);
            cfg.blockDim = dim3(block);
            cfg.stream = s;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = dependent ? 1 : 0;
            return cudaLaunchKernelEx(&cfg, kernel, args...);
        };
        int launched = 0;
        cudaError_t e = cudaSuccess;
        for (int pass = 0; pass < 4 && e == cudaSuccess; ++pass) {
            S.pass = pass;
            const unsigned tiles = static_cast<unsigned>(S.tiles);
            if ((e = launch(pass == 0 ? radix_hist_kernel<true> : radix_hist_kernel<false>, tiles, kSortThreads,
                            pass > 0, S)) != cudaSuccess)
                break;
            ++launched;
            if ((e = launch(radix_digit_scan_kernel, static_cast<unsigned>(kRadixDigits), kScanThreads, true,
                            ctx->rank_counts, ctx->rank_totals, S.tiles)) != cudaSuccess)
                break;
            ++launched;
            auto scatter = pass == 0 ? radix_scatter_kernel<kFirstPass>
                                     : pass == 3 ? radix_scatter_kernel<kLastPass> : radix_scatter_kernel<kMiddlePass>;
            if ((e = launch(scatter, tiles, kSortThreads, true, S)) != cudaSuccess) break;
            ++launched;
        }
        if (e == cudaSuccess) {
            e = launch(restore_l2_priority_kernel, static_cast<unsigned>(ctx->num_sms * 4), 256u, true,
                       static_cast<const int32_t*>(ctx->rank_of), n);
            ++launched;
        }
        per_note_launch(launched);
        if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return PER_ERR_CUDA;
    }
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
