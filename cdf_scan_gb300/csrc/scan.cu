// scan.cu -- build_cdf: cdf[i] = sum_{j<=i} p_j^alpha, monotone and
// bit-reproducible, with exact carries between tiles.
//
// Method (PufferLib PR #615, section 1 "Parallel build_cdf": an inclusive
// prefix sum of the priorities rebuilt once per minibatch update, monotone,
// deterministic, allocation- and sync-free).  The two-level block scan and
// the serial kernel described there are prior art.  Two kernels here:
//
//  * Inputs that fit one wave of co-resident CTAs: build_cdf_wave_kernel,
//    one tile per CTA scanned in registers, carries by an exact lookback
//    over tagged tile-sum words (scan_core.cuh).
//  * Larger inputs: build_cdf_stream_kernel, one pass over the input by
//    persistent CTAs -- a producer warp streams tiles through a ring of 1-D
//    bulk copies (TMA) on mbarriers, compute warps scan them locally and park
//    the result in tensor memory, and each tile is written out a few tiles
//    later, once its exact carry has been collected from the tagged records
//    of the tiles before it (a decoupled lookback).
//
// Carries are 128-bit fixed-point integers (60 fractional bits), so they do
// not depend on the order in which partial sums arrive; each unit (tile or
// slice) writes clamp(hi + (lo + local), fl32(E), fl32(E')) with E its exact
// carry as fp32 hi + lo and E' the next unit's, so the CDF is non-decreasing.

#include <mutex>

#include "scan_core.cuh"

namespace {

// Issue the bulk copy of tile `t` into stage buffer `buf` (thread 0 only).
// The copy covers the tile's valid items rounded down to whole 16-byte
// groups; the 0-3 items after that are read with plain loads by the
// consumer, so the source is never read past item n-1.
template <int TILE>
__device__ __forceinline__ void load_tile(const ScanParams& P, unsigned t, float* buf, uint64_t* bar) {
    const int64_t base = static_cast<int64_t>(t) * TILE;
    const int64_t valid = P.n - base < TILE ? P.n - base : TILE;
    const unsigned bytes = static_cast<unsigned>(valid & ~int64_t(3)) * 4u;
    mbar_arrive_expect_tx(bar, bytes);
    if (bytes) bulk_copy_g2s(buf, P.p + base, bytes, bar);
}

// ---- the streaming scan: one pass by persistent CTAs ------------------------
//
// For inputs larger than one wave of tiles.  One CTA per SM (co-resident,
// cooperative launch) takes 16384-item tiles (kStreamTile: 32 slices of 512
// items, two per compute warp) in ticket order from a global counter, so an
// SM that gets less memory bandwidth simply takes fewer tiles.  The slice is
// the unit of the exact carries.  Four roles per CTA, all on the CTA's own
// sequence of tiles k = 0, 1, ...:
//   producer warp: draws tile t_k = ticket++ and streams it into stage
//     k mod STAGES of a ring of 1-D bulk copies (TMA) on mbarriers; once the
//     tickets run out it records how many tiles the CTA got;
//   16 compute warps, two slices each: the local phase of tile k -- per
//     slice its p^alpha (the stage goes back to the producer as soon as both
//     have been read), its fp32 sum (a fixed order), then its local
//     inclusive scan, which waits in tensor memory (TMEM, 256 KB per SM,
//     otherwise unused here: room for NX tiles) -- and then the emit phase
//     of tile k - LAG, whose exclusive prefix has been found meanwhile: the
//     local scans back from TMEM, written out once with each slice's carry
//     (hi, lo, fl32(E), fl32(E')) added;
//   publisher warp: the exact 128-bit fixed-point sums of the tile's slices,
//     their exclusive prefixes within the tile, and the tile's total in its
//     record, tagged "aggregate";
//   two lookback warps, taking the CTA's tiles in turn: the tile's exclusive
//     prefix E from the records of the tiles before it -- the nearest one
//     tagged "inclusive" plus the aggregates after it (a decoupled
//     lookback) -- then E + the tile's total into its record, tagged
//     "inclusive", and the 32 slice carries.
// A record is four 64-bit words, 32 payload bits each under a 32-bit tag
// (call epoch << 1 | inclusive), one 32-byte store, alone in a 128-byte line;
// a reader takes it only when all four tags agree.  All sums are exact
// integers, so E does not depend on where a lookback stopped: the CDF is
// bit-reproducible, and the arithmetic of a slice -- its sum, local scan,
// carry and clamped write -- is the same whichever CTA handles it, and the
// same as in the one-pass-per-slice formulation: sum, scan, add the carry.

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// p^alpha of this lane's run of 8 consecutive items starting at tile item i0
// (stage buffer `buf`).  In a ragged tile (valid < TILE) the 0-3 items past
// the bulk copy are read from global memory and items at or past `valid` are
// 0; full tiles skip both steps.
template <int TILE>
__device__ __forceinline__ void run_values(const ScanParams& P, const float* buf, int64_t tile_base, int valid,
                                           int i0, float (&v)[8], bool& bad) {
    const float4 a = *reinterpret_cast<const float4*>(buf + i0);
    const float4 b = *reinterpret_cast<const float4*>(buf + i0 + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    const bool ragged = valid < TILE;
    const int bulk = valid & ~3;
    if (ragged) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (i0 + e >= bulk) v[e] = i0 + e < valid ? P.p[tile_base + i0 + e] : 0.f;
    }
    pow_alpha_n<8>(v, P.alpha, P.pow_lim, P.pow_mode, bad, [&](int e) {
        const int i = i0 + e;
        return i < bulk ? buf[i] : (i < valid ? P.p[tile_base + i] : 0.f);
    });
    if (ragged) {  // p^0 would be 1
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (i0 + e >= valid) v[e] = 0.f;
    }
}

// Local inclusive scan of a slice's two runs a and b (8 consecutive items
// per lane, lanes in order; b continues from a's last value, a from 0).  Per
// run: the lane-serial sums of its 8 items, a shuffle scan of the lane
// totals, the run's base (carry + the lanes before) added to each item, and
// an exact max-scan that removes the dips fp32 reassociation can leave
// between lanes; the run's last value is the carry into the next.  The
// lane-serial sums and the shuffle scans of the two runs interleave, and a
// run whose values already ascend across the lanes (no NaN, every lane's
// first value at or above the previous lane's last one, or the carry for
// lane 0) skips the max-scan, which would leave it unchanged.
__device__ __forceinline__ void scan_pair(float (&a)[8], float (&b)[8], int lane) {
    float ra[8], rb[8];
    ra[0] = a[0];
    rb[0] = b[0];
#pragma unroll
    for (int e = 1; e < 8; ++e) {
        ra[e] = ra[e - 1] + a[e];
        rb[e] = rb[e - 1] + b[e];
    }
    float xa = ra[7], xb = rb[7];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float ya = __shfl_up_sync(PER_FULL_MASK, xa, d);
        const float yb = __shfl_up_sync(PER_FULL_MASK, xb, d);
        if (lane >= d) {
            xa += ya;
            xb += yb;
        }
    }
    float exa = __shfl_up_sync(PER_FULL_MASK, xa, 1);
    float exb = __shfl_up_sync(PER_FULL_MASK, xb, 1);
    if (lane == 0) exa = exb = 0.f;
    float carry = 0.f;
    // run a, then run b from a's last value
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float(&r)[8] = h == 0 ? ra : rb;
        float(&v)[8] = h == 0 ? a : b;
        const float base = carry + (h == 0 ? exa : exb);
        add_each<8>(base, r);
        float prev = __shfl_up_sync(PER_FULL_MASK, r[7], 1);
        if (lane == 0) prev = carry;
        bool ordered = prev <= r[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) ordered = ordered && r[e - 1] <= r[e];
        if (__all_sync(PER_FULL_MASK, ordered)) {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = r[e];
            carry = __shfl_sync(PER_FULL_MASK, r[7], 31);
        } else {
            float mx = r[7];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const float y = __shfl_up_sync(PER_FULL_MASK, mx, d);
                if (lane >= d) mx = fmaxf(mx, y);
            }
            float pm = __shfl_up_sync(PER_FULL_MASK, mx, 1);
            if (lane == 0) pm = carry;
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = fmaxf(r[e], pm);
            carry = __shfl_sync(PER_FULL_MASK, mx, 31);
        }
    }
}

// p^alpha of this lane's items of its warp's slice of a full tile (runs of 8
// at ibase + r*256), modes 0 and 1: one warp-wide range test (mode 0).
template <int ITEMS>
__device__ __forceinline__ void slice_values(const ScanParams& P, const float* buf, int ibase, float (&v)[ITEMS],
                                             bool& bad) {
#pragma unroll
    for (int r = 0; r < ITEMS / 8; ++r) {
        const float4 a = *reinterpret_cast<const float4*>(buf + ibase + r * 256);
        const float4 b = *reinterpret_cast<const float4*>(buf + ibase + r * 256 + 4);
        v[r * 8 + 0] = a.x; v[r * 8 + 1] = a.y; v[r * 8 + 2] = a.z; v[r * 8 + 3] = a.w;
        v[r * 8 + 4] = b.x; v[r * 8 + 5] = b.y; v[r * 8 + 6] = b.z; v[r * 8 + 7] = b.w;
    }
    if (P.pow_mode == 0) {
        pow_alpha_warp<ITEMS>(v, P.alpha, P.pow_lim, bad,
                              [&](int e) { return buf[ibase + (e >> 3) * 256 + (e & 7)]; });
    } else {  // alpha == 1: the values themselves
        bool ok = true;
#pragma unroll
        for (int e = 0; e < ITEMS; ++e) ok = ok && v[e] >= 0.f;
        if (!ok) bad = true;
    }
}

// Writes one run of a slice: hi + (lo + local) with the slice's carry
// cy = (hi, lo, fl32(E), fl32(E')), clamped to [fl32(E), fl32(E')], and its
// coarse-index entries; item n-1 gets fl32(E') itself, the correctly rounded
// exact total.  (The values are monotone along the run, so the clamp changes
// only a run whose first or last value falls outside.)  FAST: full tile,
// 32-byte aligned cdf.
template <bool FAST, int TILE>
__device__ __forceinline__ void emit_run(const ScanParams& P, float (&v)[8], float4 cy, int64_t tile_base, int i0,
                                         int valid, int lane) {
    add_each<8>(cy.y, v);
    add_each<8>(cy.x, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = fminf(fmaxf(v[e], cy.z), cy.w);
    if (tile_base + i0 <= P.n - 1 && P.n - 1 < tile_base + i0 + 8) {  // the last value is fl32(E_total) exactly
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (tile_base + i0 + e == P.n - 1) v[e] = cy.w;
    }
    // coarse[k] = cdf[min(64k + 63, n - 1)].  In a full tile the entries are
    // the items 64k + 63 (n - 1 is one when it ends the tile): the last item
    // of the run of every eighth lane.  A ragged tile checks each item.
    static_assert(kCoarseStride == 64, "coarse lane rule");
    const bool full = FAST || valid == TILE;
    if (FAST || (full && P.cdf_v8)) {
        st_f8(P.cdf + tile_base + i0, v);
    } else if (full || i0 + 7 < valid) {
        st_f4(P.cdf + tile_base + i0, make_float4(v[0], v[1], v[2], v[3]));
        st_f4(P.cdf + tile_base + i0 + 4, make_float4(v[4], v[5], v[6], v[7]));
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (i0 + e < valid) P.cdf[tile_base + i0 + e] = v[e];
    }
    if (P.coarse) {
        if (full) {
            if ((lane & 7) == 7) P.coarse[(tile_base + i0 + 7) / kCoarseStride] = v[7];
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int64_t g = tile_base + i0 + e;
                if (g < P.n && ((g & (kCoarseStride - 1)) == kCoarseStride - 1 || g == P.n - 1))
                    P.coarse[g / kCoarseStride] = v[e];
            }
        }
    }
}

// Inclusive warp scan of 128-bit integers (all lanes take part).
__device__ __forceinline__ u128 warp_scan_u128(u128 v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint64_t lo = static_cast<uint64_t>(v), hi = static_cast<uint64_t>(v >> 64);
        const uint64_t olo = __shfl_up_sync(PER_FULL_MASK, lo, d);
        const uint64_t ohi = __shfl_up_sync(PER_FULL_MASK, hi, d);
        if (lane >= d) v += (static_cast<u128>(ohi) << 64) | olo;
    }
    return v;
}


// Ring stages (3 x 64 KiB), the lag (tiles) between a tile's local phase and
// its emit phase, and the ring of per-tile exchange state and TMEM slots
// (more than LAG) of the streaming kernel.  The lag covers the latency of a
// lookback (the records of the tiles before it appear over a few
// microseconds), two lookback warps its throughput.  Larger tiles mean fewer
// records, lookbacks and per-tile handshakes per item.
constexpr int kStreamStages = 3;
constexpr int kStreamLag = 3;
constexpr int kStreamXring = 4;
constexpr int kStreamSlices = kStreamTile / 512;      // 512-item slices per tile
constexpr int kStreamSpw = 2;                          // slices per compute warp
constexpr int kStreamWarps = kStreamSlices / kStreamSpw;  // compute warps
constexpr int kStreamLookback = 2;               // lookback warps
constexpr int kStreamThreads = (kStreamWarps + 2 + kStreamLookback) * 32;
// Records per lane per poll of a lookback: a window of 160 tiles, which
// reaches back to the CTA's previous tile (about one tile per CTA of the
// grid earlier).
constexpr int kLookbackQ = 5;

// Record tags of the current call: "aggregate" (the tile's own sum) and
// "inclusive" (the exact prefix through the tile).
__device__ __forceinline__ unsigned tag_aggregate(unsigned epoch) { return epoch << 1; }
__device__ __forceinline__ unsigned tag_inclusive(unsigned epoch) { return (epoch << 1) | 1u; }

__device__ __forceinline__ void publish_record(const ScanParams& P, int64_t t, unsigned tag, u128 v) {
    const unsigned long long tg = static_cast<unsigned long long>(tag) << 32;
    const uint64_t lo = static_cast<uint64_t>(v), hi = static_cast<uint64_t>(v >> 64);
    st_relaxed_v4(P.rec + t * kRecStride, tg | (lo & 0xffffffffull), tg | (lo >> 32), tg | (hi & 0xffffffffull),
                  tg | (hi >> 32));
}

// Exclusive prefix of tile t (t >= 1) by decoupled lookback, one warp.  Lane
// l reads the records of tiles hi - 1 - l - 32q (q < kLookbackQ) of a
// window below hi.  The window is resolved once every record above its
// highest "inclusive" one is present: the answer is that inclusive value
// plus the aggregates above it.  A window without an inclusive record but
// complete adds all of its aggregates and moves down.  Polls until then,
// at most kWaitLimitNs (ST_TIMEOUT, *abort set).
__device__ __forceinline__ u128 lookback(const ScanParams& P, int64_t t, unsigned epoch, int lane,
                                         volatile int* abort) {
    const unsigned tg_a = tag_aggregate(epoch), tg_i = tag_inclusive(epoch);
    u128 acc = 0;
    int64_t hi = t;
    uint64_t t0 = 0;
    while (hi > 0 && !__any_sync(PER_FULL_MASK, *abort != 0)) {
        const int64_t lo = hi > 32 * kLookbackQ ? hi - 32 * kLookbackQ : 0;
        for (;;) {
            unsigned long long w[kLookbackQ][kRecWords];
#pragma unroll
            for (int q = 0; q < kLookbackQ; ++q) {
                const int64_t i = hi - 1 - lane - 32 * q;
                if (i >= lo) ld_relaxed_v4(P.rec + i * kRecStride, w[q][0], w[q][1], w[q][2], w[q][3]);
            }
            // per record: 0 missing, 1 aggregate, 2 inclusive; the lane's
            // highest inclusive record (its smallest q)
            int64_t best = -1;
            unsigned present = 0, incl = 0;
#pragma unroll
            for (int q = 0; q < kLookbackQ; ++q) {
                const int64_t i = hi - 1 - lane - 32 * q;
                if (i < lo) continue;
                const unsigned g = static_cast<unsigned>(w[q][0] >> 32);
                bool same = true;
#pragma unroll
                for (int k = 1; k < kRecWords; ++k) same = same && static_cast<unsigned>(w[q][k] >> 32) == g;
                if (same && (g == tg_a || g == tg_i)) {
                    present |= 1u << q;
                    if (g == tg_i) {
                        incl |= 1u << q;
                        if (best < 0) best = i;
                    }
                }
            }
            // the highest inclusive record of the window
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const int64_t ob = __shfl_xor_sync(PER_FULL_MASK, best, o);
                best = ob > best ? ob : best;
            }
            bool missing = false;  // a record above `best` not yet there
#pragma unroll
            for (int q = 0; q < kLookbackQ; ++q) {
                const int64_t i = hi - 1 - lane - 32 * q;
                if (i >= lo && i > best && !((present >> q) & 1u)) missing = true;
            }
            if (!__any_sync(PER_FULL_MASK, missing)) {
                u128 part = 0;
#pragma unroll
                for (int q = 0; q < kLookbackQ; ++q) {
                    const int64_t i = hi - 1 - lane - 32 * q;
                    if (i >= lo && i >= best) {
                        u128 v = 0;
#pragma unroll
                        for (int k = 0; k < kRecWords; ++k)
                            v |= static_cast<u128>(static_cast<unsigned>(w[q][k])) << (32 * k);
                        part += v;
                    }
                }
                acc += warp_sum_u128(part);
                if (best >= 0) return acc;
                hi = lo;
                break;
            }
            // lane 0's clock for the whole warp, so every lane takes the same branch
            const uint64_t now = __shfl_sync(PER_FULL_MASK, global_ns(), 0);
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitNs) {
                if (lane == 0) {
                    atomicOr(P.status, ST_TIMEOUT);
                    *abort = 1;
                }
                __syncwarp();
                return acc;
            }
            __nanosleep(128);
        }
    }
    return acc;
}

// ---- tensor memory (TMEM) as the lag buffer ----------------------------------
// TMEM is 128 lanes x 512 columns of 32 bits per SM; a warp reaches only the
// 32 lanes of its quarter (warp index mod 4).  Compute warp w keeps the 16
// local-scan values of each of its lanes for its slice h (h < 2) of tile k
// in columns (k mod NX) * 128 + (w / 4) * 32 + h * 16 .. + 15 of lanes
// 32 (w mod 4) + lane: 32 slices x 16 columns per tile in 4 lane quarters,
// NX = 4 tiles = all 512 columns.
constexpr unsigned kTmemCols = 512;

__device__ __forceinline__ void tmem_alloc(unsigned* s_addr) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(s_addr)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(unsigned taddr) {  // whole warp, the allocating one
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kTmemCols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 16 consecutive columns of this lane: store (asynchronous: tmem_wait_st
// before the columns are read back).
__device__ __forceinline__ void tmem_store16(unsigned taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
        "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
        "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
        : "memory");
}
// Waits for this thread's earlier TMEM stores.
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 16 consecutive columns of this lane: load, then wait for the load.
__device__ __forceinline__ void tmem_load16(unsigned taddr, float (&v)[16]) {
    unsigned r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
}

// 20 warps: five per SM sub-partition, whose register file (16,384) holds
// five warps of 96 registers.
__global__ void __maxnreg__(96) build_cdf_stream_kernel(ScanParams P) {
    constexpr int STAGES = kStreamStages, LAG = kStreamLag, NX = kStreamXring;
    constexpr int SLICES = kStreamSlices, SPW = kStreamSpw;
    constexpr int WARPS = kStreamWarps;  // compute warps, SPW 512-item slices each
    constexpr int TILE = kStreamTile;    // SLICES slices x 32 lanes x 16 items
    constexpr int PRODUCER = WARPS, PUBLISHER = WARPS + 1, LOOKBACK0 = WARPS + 2;
    constexpr int SLOT = SLICES * 4;     // TMEM columns per tile (16 per slice, 4 lane quarters)
    static_assert(TILE == SLICES * 512 && SLICES == WARPS * SPW && SLICES <= 32 && WARPS % 4 == 0,
                  "16 items per lane, a slice per lane of the publisher");
    static_assert(NX > LAG, "exchange / TMEM slots for the lagged tiles, plus the one in its sum phase");
    static_assert(NX * SLOT == kTmemCols, "TMEM: NX tile slots");
    extern __shared__ __align__(128) float s_buf[];  // STAGES x TILE
    __shared__ __align__(8) uint64_t s_full[STAGES], s_empty[STAGES], s_sums[NX], s_pub[NX], s_carried[NX];
    __shared__ int64_t s_tile[STAGES];          // tile of each stage
    __shared__ int64_t s_xtile[NX];             // tile of each exchange slot (CTA tile k: slot k % NX),
                                                // for the publisher and lookback warps
    __shared__ float s_sum[NX * SLICES];        // slice sums
    __shared__ ulonglong2 s_pre[NX * SLICES];   // their exact exclusive prefixes within the tile
    __shared__ ulonglong2 s_agg[NX];            // the tile's exact total
    __shared__ float4 s_carry[NX * SLICES];     // slice carries (hi, lo, fl32(E), fl32(E'))
    __shared__ unsigned s_tmem;                 // TMEM base address
    __shared__ volatile int s_abort;            // a wait ran out: nobody waits any more
    __shared__ volatile int s_count;            // tiles this CTA got (known once the tickets run out)
    __shared__ unsigned s_epoch;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t T = P.num_tiles;
    if (threadIdx.x == 0) {
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(&s_full[st], 1);
            mbar_init(&s_empty[st], WARPS);
        }
        for (int x = 0; x < NX; ++x) {
            mbar_init(&s_sums[x], WARPS);
            mbar_init(&s_pub[x], 1);
            mbar_init(&s_carried[x], 1);
        }
        s_abort = 0;
        s_count = 0x7fffffff;
        s_epoch = ld_relaxed_u32(P.ctrs + CTR_SCAN_EPOCH);
    }
    if (warp == 0) tmem_alloc(&s_tmem);  // all 512 columns (one CTA per SM)
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const unsigned epoch = s_epoch;
    // Bounded wait for phase `parity` of `bar`, which belongs to the CTA's
    // tile k: false when the CTA got fewer than k + 1 tiles (nothing will
    // arrive) or after an expired wait.
    auto wait_k = [&](uint64_t* bar, unsigned parity, int k) -> bool {
        if (s_abort) return false;
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = global_ns();
        for (;;) {
            if (k >= s_count || s_abort) return false;
            if (mbar_try_wait_for(bar, parity, 1000u)) return true;
            if (global_ns() - t0 > kWaitLimitNs) {
                s_abort = 1;
                atomicOr(P.status, ST_TIMEOUT);
                return false;
            }
        }
    };
    // the same, decided for the whole warp (every lane waits, and the warp
    // proceeds only if all saw the phase complete), so that the warp stays
    // converged for its shuffles and tcgen05 instructions
    auto wait_w = [&](uint64_t* bar, unsigned parity, int k) -> bool {
        return __all_sync(PER_FULL_MASK, wait_k(bar, parity, k));
    };
    auto aborted_w = [&]() -> bool { return __any_sync(PER_FULL_MASK, s_abort != 0); };
    int issued = 0;  // copies issued (producer thread)

    if (warp == PRODUCER) {
        if (lane == 0) {
            for (int k = 0;; ++k) {
                const int st = k % STAGES;
                if (k >= STAGES && !wait_k(&s_empty[st], static_cast<unsigned>(k / STAGES - 1) & 1u, k - STAGES)) break;
                const int64_t t = atomicAdd(P.ctrs + CTR_SCAN_TICKET, 1u);
                if (t >= T || s_abort) {
                    s_count = k;
                    break;
                }
                s_tile[st] = t;
                load_tile<TILE>(P, static_cast<unsigned>(t), s_buf + st * TILE, &s_full[st]);
                issued = k + 1;
            }
        }
    } else if (warp == PUBLISHER) {
        for (int k = 0;; ++k) {
            const int st = k % NX;
            if (!wait_w(&s_sums[st], static_cast<unsigned>(k / NX) & 1u, k)) break;
            bool range_err = false;
            const u128 f = lane < SLICES ? to_fixed(s_sum[st * SLICES + lane], range_err) : 0;
            if (range_err) atomicOr(P.status, ST_RANGE);
            const u128 incl = warp_scan_u128(f, lane);
            if (lane < SLICES) {
                const u128 ex = incl - f;
                s_pre[st * SLICES + lane] = make_ulonglong2(static_cast<unsigned long long>(ex),
                                                           static_cast<unsigned long long>(ex >> 64));
            }
            const uint64_t tlo = __shfl_sync(PER_FULL_MASK, static_cast<uint64_t>(incl), SLICES - 1);
            const uint64_t thi = __shfl_sync(PER_FULL_MASK, static_cast<uint64_t>(incl >> 64), SLICES - 1);
            const u128 agg = (static_cast<u128>(thi) << 64) | tlo;
            const int64_t t = s_xtile[st];
            __syncwarp();
            if (lane == 0) {
                s_agg[st] = make_ulonglong2(tlo, thi);
                // tile 0's aggregate is already its inclusive prefix
                if (t != P.drop_tile) publish_record(P, t, t == 0 ? tag_inclusive(epoch) : tag_aggregate(epoch), agg);
                mbar_arrive(&s_pub[st]);
            }
        }
    } else if (warp >= LOOKBACK0) {
        for (int k = warp - LOOKBACK0;; k += kStreamLookback) {
            const int st = k % NX;
            if (!wait_w(&s_pub[st], static_cast<unsigned>(k / NX) & 1u, k)) break;
            const int64_t t = s_xtile[st];
            const ulonglong2 a = s_agg[st];
            const u128 E = t > 0 ? lookback(P, t, epoch, lane, &s_abort) : 0;
            if (lane == 0 && t > 0 && t != P.drop_tile)
                publish_record(P, t, tag_inclusive(epoch), E + ((static_cast<u128>(a.y) << 64) | a.x));
            // carries of the sixteen slices, lane w for slice w: E_w = E + the
            // slices before w; E_w' = E_w + slice w's sum
            if (lane < SLICES) {
                const ulonglong2 ep = s_pre[st * SLICES + lane];
                const u128 Ew = E + ((static_cast<u128>(ep.y) << 64) | ep.x);
                bool unused = false;
                const u128 En = Ew + to_fixed(s_sum[st * SLICES + lane], unused);
                float hi, lo;
                fixed_to_float2(Ew, hi, lo);
                s_carry[st * SLICES + lane] = make_float4(hi, lo, hi, fixed_to_float(En));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_carried[st]);
        }
    } else {
        // ======================= compute warps ================================
        // this warp's slices: warp + WARPS h (h < SPW); its TMEM columns of
        // slot 0 (lanes of its quarter), 16 per slice
        const unsigned tbase = s_tmem + (static_cast<unsigned>(32 * (warp & 3)) << 16) +
                               static_cast<unsigned>((warp >> 2) * 16 * SPW);
        bool bad = false;
        int k_end = 0x7fffffff;  // the CTA's tile count, once its local phases ran out
        // tile of exchange slot x in lane x (slot k % NX holds CTA tile k until
        // this warp has written it)
        int64_t ring_tile = 0;
        for (int k = 0; k - LAG < k_end && !aborted_w(); ++k) {
            // the previous iteration's TMEM stores are complete (long since):
            // every tile read back below was stored at least one iteration ago
            tmem_wait_st();
            // ---- local phase of tile k: per slice p^alpha, the sum, the local scan to TMEM
            if (k < k_end) {
                const int st = k % STAGES, x = k % NX;
                if (!wait_w(&s_full[st], static_cast<unsigned>(k / STAGES) & 1u, k)) {
                    k_end = aborted_w() ? 0 : k;
                } else {
                    const int64_t t = s_tile[st];
                    const int64_t tile_base = t * TILE;
                    const int valid = static_cast<int>(P.n - tile_base < TILE ? P.n - tile_base : TILE);
                    const float* buf = s_buf + st * TILE;
                    if (warp == 0 && lane == 0) s_xtile[x] = t;
                    if (lane == x) ring_tile = t;
#pragma unroll 1
                    for (int h = 0; h < SPW; ++h) {
                        const int slice = warp + WARPS * h;
                        const int ibase = slice * 512 + lane * 8;  // this lane's first item of run 0
                        float v[16];
                        float sum = 0.f;
                        if (valid == TILE && P.pow_mode != 2) {
                            // full tile: the slice's values at once, one range test;
                            // the sum in two interleaved chains, then their sum
                            slice_values<16>(P, buf, ibase, v, bad);
                            unsigned long long acc = f2_pack(v[0], v[1]);
#pragma unroll
                            for (int e = 2; e < 16; e += 2) acc = f2_add(acc, f2_pack(v[e], v[e + 1]));
                            float a0, a1;
                            f2_unpack(acc, a0, a1);
                            sum = a0 + a1;
                        } else {
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                float(&u)[8] = *reinterpret_cast<float(*)[8]>(v + 8 * r);
                                run_values<TILE>(P, buf, tile_base, valid, ibase + r * 256, u, bad);
#pragma unroll
                                for (int e = 0; e < 8; ++e) sum += u[e];
                            }
                        }
#pragma unroll
                        for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(PER_FULL_MASK, sum, d);
                        if (lane == 0) s_sum[x * SLICES + slice] = sum;
                        if (h == SPW - 1) {
                            // the stage has been read and the warp's slice sums are in
                            __syncwarp();
                            if (lane == 0) {
                                mbar_arrive(&s_empty[st]);
                                mbar_arrive(&s_sums[x]);
                            }
                        }
                        // the slice's local scan while its carry is being found
                        scan_pair(*reinterpret_cast<float(*)[8]>(v), *reinterpret_cast<float(*)[8]>(v + 8), lane);
                        tmem_store16(tbase + static_cast<unsigned>(x * SLOT + h * 16), v);
                    }
                }
            }
            // ---- emit phase of tile k - LAG: the carries added, clamped, written once
            const int ks = k - LAG;
            if (ks >= 0 && ks < k_end) {
                const int x = ks % NX;
                if (!wait_w(&s_carried[x], static_cast<unsigned>(ks / NX) & 1u, ks)) break;
                const int64_t tile_base = __shfl_sync(PER_FULL_MASK, ring_tile, x) * TILE;
                const int valid = static_cast<int>(P.n - tile_base < TILE ? P.n - tile_base : TILE);
#pragma unroll 1
                for (int h = 0; h < SPW; ++h) {
                    const int slice = warp + WARPS * h;
                    const int ibase = slice * 512 + lane * 8;
                    const float4 cy = s_carry[x * SLICES + slice];
                    float u[16];
                    tmem_load16(tbase + static_cast<unsigned>(x * SLOT + h * 16), u);
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        float(&ur)[8] = *reinterpret_cast<float(*)[8]>(u + 8 * r);
                        if (valid == TILE && P.cdf_v8)
                            emit_run<true, TILE>(P, ur, cy, tile_base, ibase + r * 256, TILE, lane);
                        else
                            emit_run<false, TILE>(P, ur, cy, tile_base, ibase + r * 256, valid, lane);
                    }
                }
            }
        }
        tmem_wait_st();
        if (__any_sync(PER_FULL_MASK, bad) && lane == 0) atomicOr(P.status, ST_VALUE);
    }

    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    if (warp == 0) tmem_dealloc(s_tmem);  // every TMEM access above has completed (waited)
    if (warp == PRODUCER && lane == 0) {
        // after an expired wait some copies may not have been consumed: wait
        // (bounded) for the last copy issued into each stage before exiting
        for (int st = 0; st < STAGES && st < issued; ++st) {
            const int uses = (issued - st + STAGES - 1) / STAGES;
            mbar_wait_bounded(&s_full[st], static_cast<unsigned>(uses - 1) & 1u);
        }
    }
    // the last CTA to finish re-arms the ticket and advances the epoch for
    // the next call
    if (threadIdx.x == 0) {
        const unsigned done = atomicAdd(P.ctrs + CTR_SCAN_DONE, 1u);
        if (done == gridDim.x - 1u) {
            P.ctrs[CTR_SCAN_DONE] = 0u;
            P.ctrs[CTR_SCAN_TICKET] = 0u;
            advance_scan_epoch(P, epoch);
        }
    }
}

// Launch of the streaming kernel: one co-resident wave (cooperative) of at
// most one CTA per SM, which take tiles by ticket.  Each CTA allocates all
// 512 TMEM columns of its SM, so a second CTA on the same SM would wait in
// its allocation for the first one to finish: the grid never exceeds the SM
// count (the kernel's shared memory and registers also fit only one).
per_status launch_scan_stream(ScanParams P, int num_sms, cudaStream_t s) {
    constexpr int TILE = kStreamTile;
    const size_t smem = static_cast<size_t>(kStreamStages) * TILE * sizeof(float);
    if (!P.rec) return PER_ERR_STATE;
    static DeviceCache cache;
    const int per_sm = device_cached(cache, [&]() {
        int b = 0;
        if (cudaFuncSetAttribute(build_cdf_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, build_cdf_stream_kernel, kStreamThreads, smem) !=
                cudaSuccess)
            return 0;
        return b;  // 0: the kernel does not fit an SM (a launch error)
    });
    if (per_sm == 0) return PER_ERR_CUDA;
    const int64_t tiles = (P.n + TILE - 1) / TILE;
    if (tiles > 0x7fffffffll || tiles > P.rec_tiles) return PER_ERR_ARG;
    P.num_tiles = static_cast<unsigned>(tiles);
    int64_t grid = num_sms;
    if (grid > tiles) grid = tiles;
    if (grid > kScanMaxGrid) grid = kScanMaxGrid;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kStreamThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, build_cdf_stream_kernel, P);
    per_note_launch();
    return cuda_status(e);
}

// ---- one wave of tiles (wave_scan_tile) ---------------------------------------
template <int THREADS>
__global__ void __launch_bounds__(THREADS) build_cdf_wave_kernel(ScanParams P) {
    const unsigned epoch = wave_scan_tile<THREADS>(P, blockIdx.x, P.p + static_cast<int64_t>(blockIdx.x) * THREADS * 8,
                                                   nullptr);
    // the last CTA to finish advances the epoch for the next call
    if (threadIdx.x == 0) {
        const unsigned done = atomicAdd(P.ctrs + CTR_SCAN_DONE, 1u);
        if (done == gridDim.x - 1u) {
            P.ctrs[CTR_SCAN_DONE] = 0u;
            advance_scan_epoch(P, epoch);
        }
    }
}

// Launches the one-wave kernel when every tile's CTA can be resident at once;
// returns PER_ERR_STATE (nothing launched) otherwise.
template <int THREADS>
per_status launch_scan_wave(ScanParams P, int num_sms, cudaStream_t s) {
    constexpr int TILE = THREADS * 8;
    static DeviceCache cache;
    const int per_sm = device_cached(cache, []() {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, build_cdf_wave_kernel<THREADS>, THREADS, 0) !=
            cudaSuccess)
            return 0;
        return b < 1 ? 1 : b;
    });
    if (per_sm == 0) return PER_ERR_CUDA;
    const int64_t tiles = (P.n + TILE - 1) / TILE;
    if (tiles > static_cast<int64_t>(num_sms) * per_sm || tiles > P.desc_tiles) return PER_ERR_STATE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles));
    cfg.blockDim = dim3(THREADS);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, build_cdf_wave_kernel<THREADS>, P);
    per_note_launch();
    return cuda_status(e);
}

// One wave of 2048-item tiles for small inputs, of 4096-item tiles up to what
// the GPU holds at once, then the streaming kernel.
per_status scan_dispatch(ScanParams P, int num_sms, cudaStream_t s) {
    if (P.n <= int64_t(1) << 19) {
        const per_status st = launch_scan_wave<256>(P, num_sms, s);
        if (st != PER_ERR_STATE) return st;
    }
    {
        const per_status st = launch_scan_wave<512>(P, num_sms, s);
        if (st != PER_ERR_STATE) return st;
    }
    return launch_scan_stream(P, num_sms, s);
}

}  // namespace

per_status launch_build_cdf(per_ctx* ctx, cudaStream_t s) {
    return launch_build_cdf_of(ctx, ctx->prio, ctx->size, ctx->cdf, ctx->coarse, s);
}

per_status launch_build_cdf_of(per_ctx* ctx, const float* p, int64_t n, float* cdf, float* coarse, cudaStream_t s) {
    ScanParams P;
    P.p = p;
    P.cdf = cdf;
    P.n = n;
    P.alpha = ctx->alpha;
    P.alpha_one = ctx->alpha == 1.0f;
    P.pow_mode = ctx->alpha == 1.0f ? 1 : (ctx->alpha == 0.0f ? 2 : 0);
    P.pow_lim = pow_limit(ctx->alpha);
    P.cdf_v8 = (reinterpret_cast<uintptr_t>(cdf) & 31u) == 0;
    P.desc = ctx->scan_desc;
    P.desc_tiles = ctx->scan_desc_tiles;
    P.ctrs = ctx->ctrs;
    P.status = ctx->status;
    P.num_tiles = 0;
    P.coarse = coarse;
    P.rec = ctx->scan_rec;
    P.rec_tiles = ctx->scan_rec_tiles;
    P.drop_tile = ctx->drop_tile;  // a fault injected for one call only
    ctx->drop_tile = -1;
    return scan_dispatch(P, ctx->num_sms, s);
}

// ====================================================================
// Allocation-free variant of build_cdf (per_build_cdf_noalloc).
//
// Some callers cannot call cudaMalloc: code that runs inside another
// framework's operator or callback, where the host application owns every
// byte of device memory through its own pool, or a latency-critical loop in
// which cudaMalloc's implicit device synchronisation is not acceptable.  This
// entry point runs the same scan kernels as per_build_cdf, but keeps their
// lookback words, tile records and counters in the file-scope array below
// instead of in a context, so the caller only passes the priorities and the
// output CDF and nothing is ever allocated.
//
// The array is part of the library image: every GPU that loads the library
// holds it (about 260 KiB) until the process exits.  All calls on a device
// share it and it keeps the previous call's contents: the kernels leave their
// counters and ticket at rest for the next call even after a bounded wait
// ran out, and their tile words and records carry a per-call tag, so nothing
// needs re-arming.  Two calls whose kernels overlap on the GPU --
// different streams without ordering between them -- race on it and give
// wrong results.  Serialise calls per device.
// ====================================================================

namespace {

constexpr int64_t kNoAllocMaxN = int64_t(1) << 24;  // 16,777,216 items
constexpr int64_t kNoAllocMaxTiles = kMaxWaveTiles;  // tiles of a one-wave scan
constexpr int kNoAllocCtrWords = 8;                 // 16 x u32 counters
constexpr int kNoAllocMaxDevices = kMaxDevices;

}  // namespace

constexpr int64_t kNoAllocStateWords = kNoAllocMaxTiles * kDescStride + 1;  // == scan_state_words(kMaxWaveTiles)
// layout (64-bit words): lookback words | counters | status | tile records
// of the streaming kernel (128-byte aligned)
constexpr int64_t kNoAllocRecOff = (kNoAllocStateWords + kNoAllocCtrWords + 8 + 15) & ~int64_t(15);
constexpr int64_t kNoAllocRecTiles = (kNoAllocMaxN + kStreamTile - 1) / kStreamTile + 1;  // == scan_rec_tiles(max n)
constexpr int64_t kNoAllocWords = kNoAllocRecOff + kNoAllocRecTiles * kRecStride;
static __device__ __align__(256) unsigned long long g_noalloc_scratch[kNoAllocWords];

namespace {

std::mutex g_noalloc_mu;
unsigned long long* g_noalloc_ptr[kNoAllocMaxDevices] = {};
int g_noalloc_sms[kNoAllocMaxDevices] = {};

// Zero the descriptors and counters and start the epoch at 1 (a zero tag
// means "never written").
__global__ void noalloc_init_kernel(unsigned long long* scratch) {
    const int words = static_cast<int>(kNoAllocWords);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < words; i += gridDim.x * blockDim.x) scratch[i] = 0ull;
}

__global__ void noalloc_epoch_kernel(unsigned* ctrs) { ctrs[CTR_SCAN_EPOCH] = 1u; }

}  // namespace

extern "C" per_status per_build_cdf_noalloc(const float* d_prio, int64_t n, float alpha, float* d_cdf,
                                            int* d_status, void* stream) {
    if (!d_prio || !d_cdf || n < 1 || n > kNoAllocMaxN || !(alpha >= 0.f) || alpha > 1e30f) return PER_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(d_prio) & 15u) || (reinterpret_cast<uintptr_t>(d_cdf) & 15u)) return PER_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PER_ERR_CUDA;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return PER_ERR_ARG;
    unsigned long long* scratch = nullptr;
    {
        // One-time set-up per device, done by the first call on that device
        // (with it current): resolve the array's device address -- in host
        // code the array's name is only a host-side stand-in -- clear it,
        // and wait for the clearing, so that later calls on any stream find
        // it ready.
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess) return PER_ERR_CUDA;
            int sms = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PER_ERR_CUDA;
            auto* p = static_cast<unsigned long long*>(addr);
            noalloc_init_kernel<<<16, 256, 0, s>>>(p);
            noalloc_epoch_kernel<<<1, 1, 0, s>>>(reinterpret_cast<unsigned*>(p + kNoAllocStateWords));
            per_note_launch(2);
            if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return PER_ERR_CUDA;
            g_noalloc_sms[dev] = sms;
            g_noalloc_ptr[dev] = p;
        }
        scratch = g_noalloc_ptr[dev];
    }
    ScanParams P;
    P.p = d_prio;
    P.cdf = d_cdf;
    P.n = n;
    P.alpha = alpha;
    P.alpha_one = alpha == 1.0f;
    P.pow_mode = alpha == 1.0f ? 1 : (alpha == 0.0f ? 2 : 0);
    P.pow_lim = pow_limit(alpha);
    P.cdf_v8 = (reinterpret_cast<uintptr_t>(d_cdf) & 31u) == 0;
    P.desc = scratch;
    P.desc_tiles = kNoAllocMaxTiles;
    P.ctrs = reinterpret_cast<unsigned*>(scratch + kNoAllocStateWords);
    P.status = d_status ? d_status : reinterpret_cast<int*>(scratch + kNoAllocStateWords + kNoAllocCtrWords);
    P.num_tiles = 0;
    P.coarse = nullptr;
    P.rec = scratch + kNoAllocRecOff;
    P.rec_tiles = kNoAllocRecTiles;
    P.drop_tile = -1;
    // same kernels and tile choice as per_build_cdf: the one-wave kernels use
    // at most kMaxWaveTiles tile words (launch_scan_wave checks), and larger
    // inputs go to the streaming kernel, whose records cover n <= kNoAllocMaxN
    // (launch_scan_stream checks)
    return scan_dispatch(P, g_noalloc_sms[dev], s);
}
