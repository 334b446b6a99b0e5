// internal.h -- context layout and launcher declarations shared by the
// library's translation units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/per.h"

// Device status word bits (recorded by kernels, read by per_check).
enum : int {
    ST_TIMEOUT = 1,  // a bounded wait ran out
    ST_RANGE = 2,    // exact-carry range exceeded
    ST_VALUE = 4,    // negative / NaN priority, or an index out of range
    ST_EMPTY = 8,    // total priority 0 when sampling
};

// Slots of the per-context device counter array.
enum : int {
    CTR_SCAN_TICKET = 0,  // next tile id of the running scan
    CTR_SCAN_DONE = 1,    // tiles finished in the running scan
    CTR_SCAN_EPOCH = 2,   // tags scan descriptors of the current call (>= 1)
    CTR_UPD_EPOCH = 3,    // tags winner slots of the current update (>= 1)
    CTR_UPD_DONE = 4,     // CTAs finished in the running update-apply
    CTR_ISW_MIN = 5,      // running min of pa (float bits) for IS weights
    CTR_ISW_DONE = 8,
    NUM_CTRS = 16
};

struct per_ctx {
    int device;
    int num_sms;
    int64_t capacity;
    int64_t alloc_n;      // capacity rounded up (vector loads may touch the pad)
    int64_t cap_pow2;
    int log2_cap;
    int64_t size;
    float alpha;
    uint32_t flags;

    float* prio;                      // raw priorities [alloc_n]
    float* cdf;                       // CDF [alloc_n] (PER_SCAN)
    float* tree;                      // [2*cap_pow2] (PER_TREE)
    unsigned long long* scan_desc;    // 4 words per scan tile
    int64_t scan_desc_tiles;
    unsigned long long* winner;       // [capacity] epoch-tagged last writer
    unsigned* ctrs;                   // [NUM_CTRS]
    int* status;                      // device status word
    float* coarse;                    // [coarse_n] every 64th CDF value (PER_SCAN)
    int* sample_bounds;               // [2 * sample_bounds_n] window ends of the sampler's CTAs (PER_SCAN, PER_RANK)
    int64_t sample_bounds_n;
    int64_t coarse_n;
    unsigned long long* tickets;      // [NUM_TICKETS] grid-barrier tickets
    float* slots;                     // [slot_n] per-CTA partial results
    int slot_n;
    unsigned* step_min;               // [3] per_step: call counter, then the batch minimum of p^alpha
                                      // (float bits) of even and odd calls
    unsigned long long* scan_rec;     // [scan_rec_tiles * kRecStride] tile records of the streaming scan
    int64_t scan_rec_tiles;
    int64_t drop_tile;                // per_debug_drop_tile: the tile or CTA whose message the next scan withholds (-1)

    // rank-based PER (PER_RANK): the radix sort's buffers, the order it
    // leaves, and the rank priorities with their CDF (which depend on the
    // size only, so they are rebuilt only when the size changes)
    unsigned* rank_keys0;             // [capacity] sort keys (ping)
    unsigned* rank_keys1;             // [capacity] sort keys (pong)
    int32_t* rank_vals1;              // [capacity] item indices (pong)
    int32_t* rank_order;              // [capacity] order[r] = the item of rank r + 1
    int32_t* rank_of;                 // [capacity] rank_of[order[r]] = r
    unsigned* rank_counts;            // [rank_count_words(capacity)] per-tile digit counts
    unsigned* rank_totals;            // [kRadixDigits] digit totals of the running pass
    float* rank_q;                    // [alloc_n] q[r] = 1 / (r + 1)
    float* rank_cdf;                  // [alloc_n] inclusive prefix sum of q^alpha
    float* rank_coarse;               // [coarse_n] every 64th rank-CDF value
    int64_t rank_q_n;                 // size the rank priorities and CDF were built for (0: none)
    int64_t rank_sorted_n;            // size of the last per_rank_build (0: none)
};

// Grid-barrier ticket words (per_ctx::tickets).
enum : int { TK_ISW = 0, TK_UPD = 1, TK_SAMPLE = 2, TK_STEP = 4, TK_RANK = 5, NUM_TICKETS = 8 };

// Items per entry of the coarse CDF index: coarse[j] = cdf[min(64j+63, n-1)].
constexpr int kCoarseStride = 64;

// Streaming scan (inputs larger than one wave): at most kScanMaxGrid CTAs,
// 16384-item tiles, and per tile one record of kRecWords 64-bit words (an
// exact 128-bit sum as four tagged 32-bit pieces) alone in a 128-byte line
// (kRecStride words), for up to scan_rec_tiles(n) tiles.
constexpr int kScanMaxGrid = 1024;
constexpr int kStreamTile = 16384;
constexpr int kRecWords = 4;
constexpr int kRecStride = 16;
inline int64_t scan_rec_tiles(int64_t n) { return (n + kStreamTile - 1) / kStreamTile + 1; }

// 64-bit words of scan state for up to `tiles` tiles: one tagged aggregate
// word per tile, each alone in a 128-byte line (kDescStride words apart) so
// that the lookbacks of a whole wave of CTAs polling them spread over L2
// instead of queueing on a few lines.  Only the one-wave kernels use them,
// so at most kMaxWaveTiles tiles.
constexpr int kDescStride = 16;
constexpr int64_t kMaxWaveTiles = 1024;
inline int64_t scan_state_words(int64_t tiles) { return tiles * kDescStride + 1; }

// Rank-based PER: 8-bit radix digits, sort tiles of 4096 keys (2048 in the
// one-launch sort of small sizes), at most 2^24 items.
constexpr int kRadixDigits = 256;
constexpr int kRankTile = 4096;
constexpr int kRankSmallTile = 2048;
constexpr int64_t kRankMaxN = int64_t(1) << 24;
// Words of the per-tile digit counts for `cap` items: 32-bit counts of
// 4096-key tiles, or 16-bit counts of up to 128 2048-key tiles in rows padded
// to 8 tiles (at least 256 x 128 halves).
inline int64_t rank_count_words(int64_t cap) {
    const int64_t tiles = (cap + kRankSmallTile - 1) / kRankSmallTile;
    return kRadixDigits * (tiles > 64 ? tiles : 64);
}

// Launch set-up that is done once per device (a kernel's dynamic shared-memory
// limit is a per-device function attribute, and occupancy is asked of the
// current device): device_cached returns the value `init` computed the first
// time this cache was used on the current device (init runs with that device
// current, under the cache's lock), or 0 when init returned 0 or the device
// ordinal is not below kMaxDevices.
constexpr int kMaxDevices = 64;
struct DeviceCache {
    std::mutex mu;
    std::atomic<int> value[kMaxDevices] = {};
};
template <class Init>
int device_cached(DeviceCache& cache, Init init) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int v = cache.value[dev].load(std::memory_order_acquire);
    if (v != 0) return v;
    std::lock_guard<std::mutex> lock(cache.mu);
    v = cache.value[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        v = init();
        cache.value[dev].store(v, std::memory_order_release);
    }
    return v;
}

// Host-side launch accounting (per_launch_count).
void per_note_launch(int n = 1);

// Launchers (each returns PER_OK or PER_ERR_CUDA after enqueueing).
per_status launch_build_cdf(per_ctx* ctx, cudaStream_t s);
// The same scan over any n priorities p (16-byte aligned, alloc_n-padded)
// into cdf / coarse, with the context's alpha and scan scratch.
per_status launch_build_cdf_of(per_ctx* ctx, const float* p, int64_t n, float* cdf, float* coarse, cudaStream_t s);
// Rank-based PER: sort the stored priorities (order, rank_of) and, when the
// size changed, rebuild the rank priorities and their CDF.
per_status launch_rank_build(per_ctx* ctx, cudaStream_t s);
per_status launch_sample_scan(per_ctx* ctx, int B, uint64_t seed, uint64_t offset, const float* u01,
                              int32_t* out, cudaStream_t s);
per_status launch_sample_tree(per_ctx* ctx, int B, uint64_t seed, uint64_t offset, const float* u01, bool iid,
                              int32_t* out, cudaStream_t s);
per_status launch_is_weights(per_ctx* ctx, const int32_t* idx, int B, float beta, float* out,
                             cudaStream_t s);
// PER_ERR_STATE (nothing launched) when the fused path does not apply.
per_status launch_sample_scan_weighted(per_ctx* ctx, int B, uint64_t seed, uint64_t offset, const float* u01,
                                       float beta, int32_t* out, float* out_w, cudaStream_t s);
// With `rows` (row_bytes a multiple of 16), also out_rows[k] = rows[out[k]].
per_status launch_step(per_ctx* ctx, const int32_t* upd_idx, const float* upd_p, int n_upd, int B, uint64_t seed,
                       uint64_t offset, const float* u01, float beta, int32_t* out, float* out_w, const void* rows,
                       int64_t row_bytes, void* out_rows, cudaStream_t s);
// out[k] = rows[idx[k]] for k in [0, B), rows of row_bytes (a multiple of 16)
// indexed by item in [0, capacity); other indices flag ST_VALUE.
per_status launch_gather(per_ctx* ctx, const void* rows, int64_t row_bytes, const int32_t* idx, int B, void* out,
                         cudaStream_t s);
per_status launch_update(per_ctx* ctx, const int32_t* idx, const float* p, int n, cudaStream_t s);
per_status launch_tree_from_prio(per_ctx* ctx, cudaStream_t s);
per_status launch_resample(const float* logw, int rows, int P, uint64_t seed, uint64_t offset,
                           const float* u_rows, int32_t* out, float* out_cdf, const float* state, int D,
                           float* out_state, float* out_logw, float reset, cudaStream_t s);

inline per_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PER_OK : PER_ERR_CUDA; }
