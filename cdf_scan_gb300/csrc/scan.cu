// scan.cu -- build_cdf: cdf[i] = sum_{j<=i} p_j^alpha in one pass over HBM.
//
// Method (PufferLib PR #615, section 1 "Parallel build_cdf": an inclusive
// prefix sum of the priorities rebuilt once per minibatch update, monotone,
// deterministic, allocation- and sync-free).  The two-level block scan and
// the serial kernel described there are prior art; this is a single-pass
// decoupled-lookback scan:
//
//  * Tiles of 256 threads x ITEMS floats, taken in order from an atomic
//    ticket so every tile a CTA waits on is already running.
//  * p^alpha is applied as the tile is loaded with 128-bit vector loads.
//  * Inside a tile: each warp scans its contiguous chunk with a thread-serial
//    pass over 4 values plus warp shuffles, repairs the 1-ulp dips fp32
//    reassociation can leave between lanes with an exact max-scan, and the
//    warp chunks are chained by a left fold (each warp starts at the previous
//    warp's last value), so local values are monotone by construction.
//  * Across tiles the carry is exact: a tile's fp32 sum becomes a 128-bit
//    fixed-point integer (60 fractional bits) and the lookback adds integers,
//    so the carry of tile t is the same value whatever order and depth the
//    lookback takes -- the result is bit-reproducible run to run.
//  * Each tile turns its exact carry E_t into fp32 hi + lo and writes
//    clamp(hi + (lo + local), fl32(E_t), fl32(E_{t+1})): the clamp bounds are
//    monotone in t, so the whole CDF is non-decreasing.
//  * Descriptors are 4 x 64-bit words (32-bit tag | 32-bit limb); a reader
//    accepts a descriptor only when all four tags match the current call's
//    epoch, so stale descriptors never need clearing.  The last CTA to finish
//    resets the ticket counters and advances the epoch.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kFracBits = 60;
typedef unsigned __int128 u128;

struct ScanParams {
    const float* __restrict__ p;
    float* __restrict__ cdf;
    int64_t n;
    float alpha;
    bool alpha_one;
    unsigned long long* desc;
    int64_t desc_tiles;
    unsigned* ctrs;
    int* status;
    unsigned num_tiles;
};

// fp32 (>= 0) -> fixed point with kFracBits fractional bits, truncating below
// 2^-60.  Values >= 2^44, inf and NaN set range_err.
__device__ __forceinline__ u128 to_fixed(float a, bool& range_err) {
    if (!(a < 17592186044416.0f)) {  // 2^44; also catches NaN and +inf
        range_err = true;
        return static_cast<u128>(1) << 104;
    }
    uint32_t bits = __float_as_uint(a);
    uint32_t ex = bits >> 23;
    uint32_t man = bits & 0x7fffffu;
    if (ex == 0 && man == 0) return 0;
    uint32_t m;
    int e;
    if (ex == 0) {
        m = man;
        e = -149;
    } else {
        m = man | 0x800000u;
        e = static_cast<int>(ex) - 150;
    }
    int sh = e + kFracBits;
    if (sh >= 0) return static_cast<u128>(m) << sh;
    if (sh <= -24) return 0;
    return static_cast<u128>(m >> (-sh));
}

// Correctly rounded (monotone) fixed point -> fp64.
__device__ __forceinline__ double fixed_to_double(u128 x) {
    if (x == 0) return 0.0;
    uint64_t hi = static_cast<uint64_t>(x >> 64), lo = static_cast<uint64_t>(x);
    int lz = hi ? __clzll(static_cast<long long>(hi)) : 64 + __clzll(static_cast<long long>(lo));
    u128 y = x << lz;
    uint64_t top = static_cast<uint64_t>(y >> 64);
    if (static_cast<uint64_t>(y) != 0) top |= 1ull;  // sticky bit
    return ldexp(__ull2double_rn(top), 64 - lz - kFracBits);
}

__device__ __forceinline__ u128 warp_sum_u128(u128 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        uint64_t lo = static_cast<uint64_t>(v), hi = static_cast<uint64_t>(v >> 64);
        uint64_t olo = __shfl_xor_sync(PER_FULL_MASK, lo, o);
        uint64_t ohi = __shfl_xor_sync(PER_FULL_MASK, hi, o);
        v += (static_cast<u128>(ohi) << 64) | olo;
    }
    return v;
}

__device__ __forceinline__ void publish(unsigned long long* d, unsigned tag, u128 v) {
    const unsigned long long t = static_cast<unsigned long long>(tag) << 32;
    uint64_t lo = static_cast<uint64_t>(v), hi = static_cast<uint64_t>(v >> 64);
    st_relaxed_v2(d, t | (lo & 0xffffffffull), t | (lo >> 32));
    st_relaxed_v2(d + 2, t | (hi & 0xffffffffull), t | (hi >> 32));
}

// Reads descriptor `d`: 0 = not yet published this call, 1 = aggregate,
// 2 = inclusive prefix.
__device__ __forceinline__ int read_desc(const unsigned long long* d, unsigned tag_agg, u128& v) {
    unsigned long long w0, w1, w2, w3;
    ld_relaxed_v2(d, w0, w1);
    ld_relaxed_v2(d + 2, w2, w3);
    unsigned g0 = static_cast<unsigned>(w0 >> 32), g1 = static_cast<unsigned>(w1 >> 32);
    unsigned g2 = static_cast<unsigned>(w2 >> 32), g3 = static_cast<unsigned>(w3 >> 32);
    if (g0 != g1 || g1 != g2 || g2 != g3 || (g0 != tag_agg && g0 != tag_agg + 1u)) return 0;
    uint64_t lo = (w0 & 0xffffffffull) | ((w1 & 0xffffffffull) << 32);
    uint64_t hi = (w2 & 0xffffffffull) | ((w3 & 0xffffffffull) << 32);
    v = (static_cast<u128>(hi) << 64) | lo;
    return g0 == tag_agg ? 1 : 2;
}

// ---- scan state in global memory ---------------------------------------------
// For every tile t: aggw[t] = (tag << 32) | fp32 bits of the tile sum, tag
// 2*epoch (aggregate published) or 2*epoch+1 (inclusive prefix published in
// inc[t]); inc[t] = 4 tagged words holding the exact 128-bit inclusive prefix.
// For every full group of 32 tiles: gagg[g] = 4 tagged words holding the
// group's exact sum, published by the group's last tile to arrive (counted
// in gcnt[g], which grows by exactly 32 per call, so no reset is needed).
struct ScanState {
    unsigned long long* aggw;
    unsigned long long* inc;
    unsigned long long* gagg;
    unsigned* gcnt;
};

__device__ __forceinline__ ScanState scan_state(const ScanParams& P) {
    ScanState S;
    S.inc = P.desc;
    S.aggw = P.desc + 4 * P.desc_tiles;
    S.gagg = S.aggw + P.desc_tiles;
    S.gcnt = reinterpret_cast<unsigned*>(S.gagg + 4 * (P.desc_tiles / 32 + 1));
    return S;
}

constexpr int kGroupQ = 4;  // group rounds per poll: 128 groups (4096 tiles) of reach

__device__ __forceinline__ void spin_pause(unsigned& spins, bool& timed_out, int lane, int* status) {
    if (++spins > kSpinLimit) {
        timed_out = true;
        if (lane == 0) atomicOr(status, ST_TIMEOUT);
        return;
    }
    if (spins > 8) __nanosleep(spins < 64 ? 64 : 256);
}

// Inclusive prefix of tile `t` from its record (all lanes; waits until valid).
__device__ u128 read_inc(const ScanState& S, int64_t t, unsigned tag_inc, int lane, int* status) {
    unsigned spins = 0;
    bool timed_out = false;
    u128 v = 0;
    for (;;) {
        const int st = read_desc(S.inc + 4 * t, tag_inc - 1u, v);  // tag_agg = tag_inc - 1
        if (__all_sync(PER_FULL_MASK, st == 2)) return v;
        spin_pause(spins, timed_out, lane, status);
        if (timed_out) return 0;
    }
}

// Exclusive prefix (exact) of tile t, computed by one warp.
//   1. own group: tiles 32g .. t-1 (lane l reads tile 32g + l): the nearest
//      one holding an inclusive prefix ends the walk, otherwise all their
//      aggregates are summed;
//   2. earlier groups, kGroupQ x 32 per poll: group k is "inclusive" when its
//      last tile holds an inclusive prefix, else its published group sum is
//      used; the nearest inclusive group ends the walk.
// Integer sums are exact, so any mix of tile and group sums gives the same
// value: the carry is independent of timing.
__device__ u128 lookback(const ScanState& S, int64_t t, unsigned tag_agg, int lane, int* status) {
    const unsigned tag_inc = tag_agg + 1u;
    const int64_t g = t >> 5;
    const int p = static_cast<int>(t & 31);
    unsigned spins = 0;
    bool timed_out = false;
    u128 part = 0;
    if (p > 0) {
        for (;;) {
            unsigned long long w = 0;
            if (lane < p) w = *reinterpret_cast<volatile const unsigned long long*>(S.aggw + (g << 5) + lane);
            const unsigned tag = static_cast<unsigned>(w >> 32);
            const bool inc = lane < p && tag == tag_inc;
            const bool valid = lane >= p || tag == tag_agg || tag == tag_inc;
            const unsigned incm = __ballot_sync(PER_FULL_MASK, inc);
            const int h = incm ? 31 - __clz(incm) : -1;  // nearest inclusive tile
            const unsigned need = (lane > h && lane < p) ? 1u : 0u;
            if (__all_sync(PER_FULL_MASK, valid || !need)) {
                bool err = false;
                const u128 a = (need && lane < p) ? to_fixed(__uint_as_float(static_cast<unsigned>(w)), err)
                                                  : static_cast<u128>(0);
                part = warp_sum_u128(a);
                if (h >= 0) return part + read_inc(S, (g << 5) + h, tag_inc, lane, status);
                break;
            }
            spin_pause(spins, timed_out, lane, status);
            if (timed_out) return 0;
        }
    }
    // previous groups
    int64_t k0 = g - 1;  // lane l, round q examines group k0 - l - 32q
    u128 acc = part;
    while (k0 >= 0) {
        int st[kGroupQ];
        u128 val[kGroupQ];
        int fq = kGroupQ, fl = 0;
        for (;;) {
#pragma unroll
            for (int q = 0; q < kGroupQ; ++q) {
                const int64_t k = k0 - lane - 32 * q;
                val[q] = 0;
                if (k < 0) {
                    st[q] = 2;  // before group 0: inclusive prefix 0
                } else {
                    const unsigned long long w =
                        *reinterpret_cast<volatile const unsigned long long*>(S.aggw + (k << 5) + 31);
                    if (static_cast<unsigned>(w >> 32) == tag_inc) {
                        st[q] = 3;  // inclusive: value read below
                    } else {
                        st[q] = read_desc(S.gagg + 4 * k, tag_agg, val[q]) == 1 ? 1 : 0;
                    }
                }
            }
            unsigned incm[kGroupQ], invm[kGroupQ];
#pragma unroll
            for (int q = 0; q < kGroupQ; ++q) {
                incm[q] = __ballot_sync(PER_FULL_MASK, st[q] >= 2);
                invm[q] = __ballot_sync(PER_FULL_MASK, st[q] == 0);
            }
            fq = kGroupQ;
            fl = 0;
#pragma unroll
            for (int q = kGroupQ - 1; q >= 0; --q)
                if (incm[q]) {
                    fq = q;
                    fl = __ffs(incm[q]) - 1;
                }
            bool ready = true;
#pragma unroll
            for (int q = 0; q < kGroupQ; ++q) {
                if (q < fq && invm[q]) ready = false;
                if (q == fq && (invm[q] & ((1u << fl) - 1u))) ready = false;
            }
            if (ready) break;
            spin_pause(spins, timed_out, lane, status);
            if (timed_out) return acc;
        }
        u128 c = 0;
#pragma unroll
        for (int q = 0; q < kGroupQ; ++q)
            if (q < fq || (q == fq && lane < fl)) c += val[q];
        acc += warp_sum_u128(c);
        if (fq < kGroupQ) {
            const int64_t k = k0 - fl - 32 * fq;
            if (k >= 0) acc += read_inc(S, (k << 5) + 31, tag_inc, lane, status);
            return acc;
        }
        k0 -= 32 * kGroupQ;
    }
    return acc;
}

// After publishing tile t's aggregate: if t completes a full group, the last
// tile of the group to arrive sums the group's 32 aggregates and publishes
// the group sum.  One warp; the counter's acquire-release ordering makes the
// other tiles' aggregates visible.
__device__ void group_arrive(const ScanState& S, int64_t t, unsigned num_tiles, unsigned tag_agg, int lane,
                             int* status) {
    const int64_t g = t >> 5;
    if ((g << 5) + 31 >= num_tiles) return;  // partial last group: never needed
    unsigned old = 0;
    if (lane == 0) {
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(S.gcnt + g) : "memory");
    }
    old = __shfl_sync(PER_FULL_MASK, old, 0);
    if ((old & 31u) != 31u) return;
    unsigned spins = 0;
    bool timed_out = false;
    for (;;) {
        const unsigned long long w = *reinterpret_cast<volatile const unsigned long long*>(S.aggw + (g << 5) + lane);
        const unsigned tag = static_cast<unsigned>(w >> 32);
        if (__all_sync(PER_FULL_MASK, tag == tag_agg || tag == tag_agg + 1u)) {
            bool err = false;
            const u128 sum = warp_sum_u128(to_fixed(__uint_as_float(static_cast<unsigned>(w)), err));
            if (lane == 0) publish(S.gagg + 4 * g, tag_agg, sum);
            return;
        }
        spin_pause(spins, timed_out, lane, status);
        if (timed_out) return;
    }
}

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

// Persistent scan: each CTA keeps STAGES tiles in flight through a ring of
// shared-memory buffers filled by bulk copies, takes tile ids in increasing
// order from the global ticket, and processes them in that order with a lag
// of one: the local scan of tile k+1 runs before tile k's lookback finishes,
// so the lookback latency overlaps useful work.  Tile k's local values wait
// in its stage buffer until its carry is known.
template <int ITEMS, int STAGES>
__global__ void __launch_bounds__(kThreads) build_cdf_kernel(ScanParams P) {
    static_assert(STAGES >= 3, "one buffer scanning, one awaiting its carry, one loading");
    constexpr int TILE = kThreads * ITEMS;
    constexpr int LANE_ITEMS = 8;             // consecutive items per lane per sub-chunk
    constexpr int SUB = ITEMS / LANE_ITEMS;   // sub-chunks per warp
    constexpr int WCHUNK = 32 * ITEMS;        // items per warp
    extern __shared__ __align__(128) float s_buf[];  // STAGES x TILE
    __shared__ __align__(8) uint64_t s_bar[STAGES];
    __shared__ unsigned s_ticket[STAGES];
    __shared__ unsigned s_epoch;
    __shared__ float s_wtot[2][kWarps];  // by iteration parity: reuse is two barriers apart
    __shared__ float s_agg[2];      // tile sums of the scanned and the pending tile
    __shared__ float s_carry[4];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const ScanState S = scan_state(P);
    if (threadIdx.x == 0) {
        s_epoch = ld_relaxed_u32(P.ctrs + CTR_SCAN_EPOCH);
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(&s_bar[st], 1);
            const unsigned t = atomicAdd(P.ctrs + CTR_SCAN_TICKET, 1u);
            s_ticket[st] = t;
            if (t < P.num_tiles) load_tile<TILE>(P, t, s_buf + st * TILE, &s_bar[st]);
        }
    }
    __syncthreads();
    const unsigned epoch = s_epoch;
    const unsigned tag_agg = 2u * epoch;
    int pend_slot = -1;          // stage holding the tile that awaits its carry
    unsigned pend_t = 0;

    for (int it = 0;; ++it) {
        const int st = it % STAGES;
        const unsigned t = s_ticket[st];
        const bool have = t < P.num_tiles;
        if (have) {
            if (!mbar_wait_bounded(&s_bar[st], static_cast<unsigned>(it / STAGES) & 1u))
                atomicOr(P.status, ST_TIMEOUT);
            float* buf = s_buf + st * TILE;
            const int64_t tile_base = static_cast<int64_t>(t) * TILE;
            const int64_t valid = P.n - tile_base < TILE ? P.n - tile_base : TILE;
            const int bulk = static_cast<int>(valid & ~int64_t(3));
            const bool full = valid == TILE;

            // ---- load from shared memory + p^alpha --------------------------
            float v[ITEMS];
            bool bad = false;
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int i0 = warp * WCHUNK + s * 256 + lane * LANE_ITEMS + 4 * h;
                    float4 q = *reinterpret_cast<const float4*>(buf + i0);
                    if (!full) {
                        float e4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = i0 + e;
                            if (i >= bulk) e4[e] = i < valid ? P.p[tile_base + i] : 0.f;
                        }
                        q = make_float4(e4[0], e4[1], e4[2], e4[3]);
                    }
                    bad |= !(q.x >= 0.f) | !(q.y >= 0.f) | !(q.z >= 0.f) | !(q.w >= 0.f);
                    float a0 = pow_alpha(q.x, P.alpha, P.alpha_one), a1 = pow_alpha(q.y, P.alpha, P.alpha_one);
                    float a2 = pow_alpha(q.z, P.alpha, P.alpha_one), a3 = pow_alpha(q.w, P.alpha, P.alpha_one);
                    if (!full) {  // padding beyond n contributes 0 (p^0 would be 1)
                        a0 = i0 < valid ? a0 : 0.f;
                        a1 = i0 + 1 < valid ? a1 : 0.f;
                        a2 = i0 + 2 < valid ? a2 : 0.f;
                        a3 = i0 + 3 < valid ? a3 : 0.f;
                    }
                    v[s * LANE_ITEMS + 4 * h + 0] = a0;
                    v[s * LANE_ITEMS + 4 * h + 1] = a1;
                    v[s * LANE_ITEMS + 4 * h + 2] = a2;
                    v[s * LANE_ITEMS + 4 * h + 3] = a3;
                }
            }
            if (__any_sync(PER_FULL_MASK, bad) && lane == 0) atomicOr(P.status, ST_VALUE);

            // ---- warp-local monotone scan ------------------------------------
            float carry = 0.f;
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
                float r[LANE_ITEMS];
                r[0] = v[s * LANE_ITEMS];
#pragma unroll
                for (int e = 1; e < LANE_ITEMS; ++e) r[e] = r[e - 1] + v[s * LANE_ITEMS + e];
                float x = r[LANE_ITEMS - 1];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const float y = __shfl_up_sync(PER_FULL_MASK, x, d);
                    if (lane >= d) x += y;
                }
                float ex = __shfl_up_sync(PER_FULL_MASK, x, 1);
                if (lane == 0) ex = 0.f;
                const float base = carry + ex;
#pragma unroll
                for (int e = 0; e < LANE_ITEMS; ++e) r[e] = base + r[e];
                float mx = r[LANE_ITEMS - 1];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const float y = __shfl_up_sync(PER_FULL_MASK, mx, d);
                    if (lane >= d) mx = fmaxf(mx, y);
                }
                float pm = __shfl_up_sync(PER_FULL_MASK, mx, 1);
                if (lane == 0) pm = carry;
#pragma unroll
                for (int e = 0; e < LANE_ITEMS; ++e) v[s * LANE_ITEMS + e] = fmaxf(r[e], pm);
                carry = __shfl_sync(PER_FULL_MASK, mx, 31);
            }
            float* wtot = s_wtot[it & 1];
            if (lane == 0) wtot[warp] = carry;
            __syncthreads();
            float off = 0.f;
            for (int w = 0; w < warp; ++w) off = off + wtot[w];
            // park the tile-local values in the stage buffer until the carry is known
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int i0 = warp * WCHUNK + s * 256 + lane * LANE_ITEMS + 4 * h;
                    *reinterpret_cast<float4*>(buf + i0) =
                        make_float4(off + v[s * LANE_ITEMS + 4 * h], off + v[s * LANE_ITEMS + 4 * h + 1],
                                    off + v[s * LANE_ITEMS + 4 * h + 2], off + v[s * LANE_ITEMS + 4 * h + 3]);
                }
            }
            if (warp == 0) {
                float agg = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) agg = agg + wtot[w];
                if (lane == 0) {
                    s_agg[it & 1] = agg;
                    const unsigned long long word = (static_cast<unsigned long long>(tag_agg) << 32) |
                                                    __float_as_uint(agg);
                    if (t == 0) {  // tile 0's inclusive prefix is its own sum
                        bool err = false;
                        publish(S.inc, tag_agg + 1u, to_fixed(agg, err));
                    }
                    *reinterpret_cast<volatile unsigned long long*>(S.aggw + t) =
                        t == 0 ? (word + (1ull << 32)) : word;
                }
                __syncwarp();
                group_arrive(S, t, P.num_tiles, tag_agg, lane, P.status);
            }
        }

        // ---- finish the pending tile: lookback, carry, store, refill --------
        if (pend_slot >= 0) {
            const int ps = pend_slot;
            const int64_t tile_base = static_cast<int64_t>(pend_t) * TILE;
            const int64_t valid = P.n - tile_base < TILE ? P.n - tile_base : TILE;
            const bool full = valid == TILE;
            if (warp == 0) {
                bool range_err = false;
                const float agg = s_agg[(it - 1) & 1];
                const u128 a_fix = to_fixed(agg, range_err);
                const u128 excl = pend_t == 0 ? static_cast<u128>(0) : lookback(S, pend_t, tag_agg, lane, P.status);
                if (lane == 0) {
                    if (pend_t != 0) {
                        publish(S.inc + 4 * static_cast<int64_t>(pend_t), tag_agg + 1u, excl + a_fix);
                        const unsigned long long word = (static_cast<unsigned long long>(tag_agg + 1u) << 32) |
                                                        __float_as_uint(agg);
                        *reinterpret_cast<volatile unsigned long long*>(S.aggw + pend_t) = word;
                    }
                    const double d0 = fixed_to_double(excl);
                    const double d1 = fixed_to_double(excl + a_fix);
                    const float hi = __double2float_rn(d0);
                    s_carry[0] = hi;
                    s_carry[1] = __double2float_rn(d0 - static_cast<double>(hi));
                    s_carry[2] = hi;                     // fl32(E_t)
                    s_carry[3] = __double2float_rn(d1);  // fl32(E_{t+1})
                    if (range_err) atomicOr(P.status, ST_RANGE);
                }
            }
            __syncthreads();
            const float hi = s_carry[0], lo = s_carry[1], sig_lo = s_carry[2], sig_hi = s_carry[3];
            const float* buf = s_buf + ps * TILE;
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int i0 = warp * WCHUNK + s * 256 + lane * LANE_ITEMS + 4 * h;
                    const float4 loc = *reinterpret_cast<const float4*>(buf + i0);
                    float o[4] = {hi + (lo + loc.x), hi + (lo + loc.y), hi + (lo + loc.z), hi + (lo + loc.w)};
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[e] = fminf(fmaxf(o[e], sig_lo), sig_hi);
                    if (full || i0 + 3 < valid) {
                        st_f4(P.cdf + tile_base + i0, make_float4(o[0], o[1], o[2], o[3]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (i0 + e < valid) P.cdf[tile_base + i0 + e] = o[e];
                    }
                }
            }
            __syncthreads();  // pending buffer, s_carry and s_wtot free again
            if (threadIdx.x == 0) {
                const unsigned t2 = atomicAdd(P.ctrs + CTR_SCAN_TICKET, 1u);
                s_ticket[ps] = t2;
                if (t2 < P.num_tiles) load_tile<TILE>(P, t2, s_buf + ps * TILE, &s_bar[ps]);
            }
            __syncthreads();
        }
        if (!have) break;
        pend_slot = st;
        pend_t = t;
    }

    // ---- the last CTA to finish resets the counters for the next call --------
    if (threadIdx.x == 0) {
        const unsigned done = atomicAdd(P.ctrs + CTR_SCAN_DONE, 1u);
        if (done == gridDim.x - 1u) {
            P.ctrs[CTR_SCAN_TICKET] = 0u;
            P.ctrs[CTR_SCAN_DONE] = 0u;
            unsigned next = epoch + 1u;
            if (next >= (1u << 30)) {  // epoch wrap: clear all scan state once (counters keep
                // their multiples of 32)
                const int64_t words = 4 * P.desc_tiles + P.desc_tiles + 4 * (P.desc_tiles / 32 + 1);
                for (int64_t i = 0; i < words; ++i) P.desc[i] = 0ull;
                next = 1u;
            }
            P.ctrs[CTR_SCAN_EPOCH] = next;
        }
    }
}

// ---- small inputs: one thread-block cluster, DSMEM exchange ----------------
//
// For n <= kClusterMax * TILE_C the whole array fits one cluster: CTA r of
// the cluster scans tile r in registers (same per-warp monotone scan as
// above), publishes its exact tile sum in its own shared memory, and after
// one cluster barrier reads the sums of CTAs 0..r-1 through distributed
// shared memory.  The exact 128-bit sum makes the carry independent of order;
// the clamp bounds fl32(E_r), fl32(E_r + a_r) keep the CDF monotone.  No
// global scratch, no atomics, no lookback.

__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ unsigned long long dsmem_ld_u64(const void* local_ptr, unsigned rank) {
    unsigned remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local_ptr)), "r"(rank));
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(remote) : "memory");
    return v;
}

constexpr int kClusterThreads = 512;
constexpr int kClusterItems = 32;                       // per thread
constexpr int kClusterTile = kClusterThreads * kClusterItems;  // 16384
constexpr int kClusterMax = 16;

__global__ void __launch_bounds__(kClusterThreads, 1) build_cdf_cluster_kernel(ScanParams P) {
    constexpr int ITEMS = kClusterItems;
    constexpr int LANE_ITEMS = 8;
    constexpr int SUB = ITEMS / LANE_ITEMS;
    constexpr int WCHUNK = 32 * ITEMS;
    constexpr int WARPS = kClusterThreads / 32;
    __shared__ float s_wtot[WARPS];
    __shared__ __align__(16) unsigned long long s_agg[2];
    __shared__ float s_carry[4];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned r = cluster_rank();
    const int64_t tile_base = static_cast<int64_t>(r) * kClusterTile;
    int64_t valid = P.n - tile_base;
    valid = valid < 0 ? 0 : (valid > kClusterTile ? kClusterTile : valid);
    const bool full = valid == kClusterTile;

    float v[ITEMS];
    bool bad = false;
#pragma unroll
    for (int s = 0; s < SUB; ++s) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i0 = warp * WCHUNK + s * 256 + lane * LANE_ITEMS + 4 * h;
            float4 q;
            if (full || i0 + 3 < valid) {
                q = ld_f4(P.p + tile_base + i0);
            } else {
                q.x = i0 < valid ? P.p[tile_base + i0] : 0.f;
                q.y = i0 + 1 < valid ? P.p[tile_base + i0 + 1] : 0.f;
                q.z = i0 + 2 < valid ? P.p[tile_base + i0 + 2] : 0.f;
                q.w = i0 + 3 < valid ? P.p[tile_base + i0 + 3] : 0.f;
            }
            bad |= !(q.x >= 0.f) | !(q.y >= 0.f) | !(q.z >= 0.f) | !(q.w >= 0.f);
            float a0 = pow_alpha(q.x, P.alpha, P.alpha_one), a1 = pow_alpha(q.y, P.alpha, P.alpha_one);
            float a2 = pow_alpha(q.z, P.alpha, P.alpha_one), a3 = pow_alpha(q.w, P.alpha, P.alpha_one);
            if (!full) {
                a0 = i0 < valid ? a0 : 0.f;
                a1 = i0 + 1 < valid ? a1 : 0.f;
                a2 = i0 + 2 < valid ? a2 : 0.f;
                a3 = i0 + 3 < valid ? a3 : 0.f;
            }
            v[s * LANE_ITEMS + 4 * h + 0] = a0;
            v[s * LANE_ITEMS + 4 * h + 1] = a1;
            v[s * LANE_ITEMS + 4 * h + 2] = a2;
            v[s * LANE_ITEMS + 4 * h + 3] = a3;
        }
    }
    if (__any_sync(PER_FULL_MASK, bad) && lane == 0) atomicOr(P.status, ST_VALUE);

    float carry = 0.f;
#pragma unroll
    for (int s = 0; s < SUB; ++s) {
        float rr[LANE_ITEMS];
        rr[0] = v[s * LANE_ITEMS];
#pragma unroll
        for (int e = 1; e < LANE_ITEMS; ++e) rr[e] = rr[e - 1] + v[s * LANE_ITEMS + e];
        float x = rr[LANE_ITEMS - 1];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float y = __shfl_up_sync(PER_FULL_MASK, x, d);
            if (lane >= d) x += y;
        }
        float ex = __shfl_up_sync(PER_FULL_MASK, x, 1);
        if (lane == 0) ex = 0.f;
        const float base = carry + ex;
#pragma unroll
        for (int e = 0; e < LANE_ITEMS; ++e) rr[e] = base + rr[e];
        float mx = rr[LANE_ITEMS - 1];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float y = __shfl_up_sync(PER_FULL_MASK, mx, d);
            if (lane >= d) mx = fmaxf(mx, y);
        }
        float pm = __shfl_up_sync(PER_FULL_MASK, mx, 1);
        if (lane == 0) pm = carry;
#pragma unroll
        for (int e = 0; e < LANE_ITEMS; ++e) v[s * LANE_ITEMS + e] = fmaxf(rr[e], pm);
        carry = __shfl_sync(PER_FULL_MASK, mx, 31);
    }
    if (lane == 0) s_wtot[warp] = carry;
    __syncthreads();
    float off = 0.f;
    for (int w = 0; w < warp; ++w) off = off + s_wtot[w];
    bool range_err = false;
    if (threadIdx.x == 0) {
        float agg = 0.f;
        for (int w = 0; w < WARPS; ++w) agg = agg + s_wtot[w];
        const u128 a_fix = to_fixed(agg, range_err);
        s_agg[0] = static_cast<unsigned long long>(a_fix);
        s_agg[1] = static_cast<unsigned long long>(a_fix >> 64);
    }
    cluster_sync();  // every CTA's tile sum is published in its shared memory
    if (warp == 0) {
        // lane q < r reads CTA q's sum: one parallel round of DSMEM loads
        u128 mine = 0;
        if (static_cast<unsigned>(lane) < r) {
            const unsigned long long lo = dsmem_ld_u64(&s_agg[0], lane);
            const unsigned long long hi = dsmem_ld_u64(&s_agg[1], lane);
            mine = (static_cast<u128>(hi) << 64) | lo;
        }
        const u128 excl = warp_sum_u128(mine);
        if (lane == 0) {
        const u128 a_fix = (static_cast<u128>(s_agg[1]) << 64) | s_agg[0];
        const double d0 = fixed_to_double(excl);
        const double d1 = fixed_to_double(excl + a_fix);
        const float hi = __double2float_rn(d0);
        s_carry[0] = hi;
        s_carry[1] = __double2float_rn(d0 - static_cast<double>(hi));
        s_carry[2] = hi;
        s_carry[3] = __double2float_rn(d1);
        if (range_err) atomicOr(P.status, ST_RANGE);
        }
    }
    __syncthreads();
    const float hi = s_carry[0], lo = s_carry[1], sig_lo = s_carry[2], sig_hi = s_carry[3];
#pragma unroll
    for (int s = 0; s < SUB; ++s) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i0 = warp * WCHUNK + s * 256 + lane * LANE_ITEMS + 4 * h;
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float loc = off + v[s * LANE_ITEMS + 4 * h + e];
                o[e] = fminf(fmaxf(hi + (lo + loc), sig_lo), sig_hi);
            }
            if (full || i0 + 3 < valid) {
                st_f4(P.cdf + tile_base + i0, make_float4(o[0], o[1], o[2], o[3]));
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (i0 + e < valid) P.cdf[tile_base + i0 + e] = o[e];
            }
        }
    }
    cluster_sync();  // keep shared memory alive until every CTA has read it
}

// Launches the cluster path when n fits one cluster the GPU can schedule;
// returns PER_ERR_STATE (nothing launched) otherwise.
per_status launch_scan_cluster(ScanParams P, cudaStream_t s) {
    const int64_t ctas = (P.n + kClusterTile - 1) / kClusterTile;
    if (ctas > kClusterMax) return PER_ERR_STATE;
    static int max_ok = -1;  // largest cluster size verified schedulable
    if (max_ok < 0) {
        if (cudaFuncSetAttribute(build_cdf_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
            cudaGetLastError();
            max_ok = 8;
        } else {
            max_ok = 1;
            for (int c = kClusterMax; c >= 1; c >>= 1) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(c);
                cfg.blockDim = dim3(kClusterThreads);
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = c;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int nclusters = 0;
                if (cudaOccupancyMaxActiveClusters(&nclusters, build_cdf_cluster_kernel, &cfg) == cudaSuccess &&
                    nclusters > 0) {
                    max_ok = c;
                    break;
                }
                cudaGetLastError();
            }
        }
    }
    if (ctas > max_ok) return PER_ERR_STATE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kClusterThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ctas);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, build_cdf_cluster_kernel, P);
    per_note_launch();
    return cuda_status(e);
}

// Launch: a persistent grid of as many CTAs as can be resident at once
// (never more CTAs than tiles).
template <int ITEMS, int STAGES>
per_status launch_scan(ScanParams P, int num_sms, cudaStream_t s) {
    static_assert(ITEMS % 8 == 0, "8 consecutive items per lane per sub-chunk");
    constexpr int TILE = kThreads * ITEMS;
    const size_t smem = static_cast<size_t>(STAGES) * TILE * sizeof(float);
    static int per_sm = 0;
    if (per_sm == 0) {
        if (cudaFuncSetAttribute(build_cdf_kernel<ITEMS, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, build_cdf_kernel<ITEMS, STAGES>, kThreads,
                                                          smem) != cudaSuccess)
            return PER_ERR_CUDA;
        if (per_sm < 1) per_sm = 1;
    }
    const int64_t tiles = (P.n + TILE - 1) / TILE;
    if (tiles > P.desc_tiles) return PER_ERR_ARG;
    P.num_tiles = static_cast<unsigned>(tiles);
    int64_t grid = static_cast<int64_t>(num_sms) * per_sm;
    if (grid > tiles) grid = tiles;
    build_cdf_kernel<ITEMS, STAGES><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(P);
    per_note_launch();
    return cuda_status(cudaGetLastError());
}

// Tile size: 4096 items for large inputs (fewer lookback steps per byte);
// 2048 items when that would leave SMs without a tile.
per_status scan_dispatch(ScanParams P, int num_sms, cudaStream_t s) {
    if (P.n <= static_cast<int64_t>(kClusterMax) * kClusterTile) {
        const per_status st = launch_scan_cluster(P, s);
        if (st != PER_ERR_STATE) return st;
    }
    const int64_t big_tiles = (P.n + 4095) / 4096;
    if (big_tiles >= 2 * static_cast<int64_t>(num_sms)) return launch_scan<16, 3>(P, num_sms, s);
    return launch_scan<8, 3>(P, num_sms, s);
}

}  // namespace

per_status launch_build_cdf(per_ctx* ctx, cudaStream_t s) {
    ScanParams P;
    P.p = ctx->prio;
    P.cdf = ctx->cdf;
    P.n = ctx->size;
    P.alpha = ctx->alpha;
    P.alpha_one = ctx->alpha == 1.0f;
    P.desc = ctx->scan_desc;
    P.desc_tiles = ctx->scan_desc_tiles;
    P.ctrs = ctx->ctrs;
    P.status = ctx->status;
    P.num_tiles = 0;
    return scan_dispatch(P, ctx->num_sms, s);
}

// ====================================================================
// Allocation-free variant of build_cdf (per_build_cdf_noalloc).
//
// Some callers cannot call cudaMalloc: code that runs inside another
// framework's operator or callback, where the host application owns every
// byte of device memory through its own pool, or a latency-critical loop in
// which cudaMalloc's implicit device synchronisation is not acceptable.  This
// entry point runs the same scan kernel as per_build_cdf, but keeps its
// lookback descriptors and tile counters in the file-scope array below
// instead of in a context, so the caller only passes the priorities and the
// output CDF and nothing is ever allocated.
//
// The array is part of the library image: every GPU that loads the library
// holds it (about 165 KiB) until the process exits.  All calls on a device
// share it and it keeps the previous call's contents (its counters are left
// ready for the next call by the kernel itself), so two calls whose kernels
// overlap on the GPU -- different streams without ordering between them --
// race on it and give wrong results.  Serialise calls per device.
// ====================================================================

namespace {

constexpr int64_t kNoAllocMaxN = int64_t(1) << 24;  // 16,777,216 items
constexpr int64_t kNoAllocMaxTiles = 4096;          // tiles of >= 4096 items at the max size
constexpr int kNoAllocCtrWords = 8;                 // 16 x u32 counters
constexpr int kNoAllocMaxDevices = 64;

}  // namespace

constexpr int64_t kNoAllocStateWords = 5 * kNoAllocMaxTiles + 4 * (kNoAllocMaxTiles / 32 + 1) +
                                       (kNoAllocMaxTiles / 32 + 2) / 2 + 1;  // == scan_state_words(4096)
static __device__ __align__(256) unsigned long long
    g_noalloc_scratch[kNoAllocStateWords + kNoAllocCtrWords + 8];

namespace {

std::mutex g_noalloc_mu;
unsigned long long* g_noalloc_ptr[kNoAllocMaxDevices] = {};
int g_noalloc_sms[kNoAllocMaxDevices] = {};

// Zero the descriptors and counters and start the epoch at 1 (a zero tag
// means "never written").
__global__ void noalloc_init_kernel(unsigned long long* scratch) {
    const int words = static_cast<int>(kNoAllocStateWords) + kNoAllocCtrWords + 8;
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
        // code the array's name is only a host-side stand-in -- and clear it.
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
            if (cudaGetLastError() != cudaSuccess) return PER_ERR_CUDA;
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
    P.desc = scratch;
    P.desc_tiles = kNoAllocMaxTiles;
    P.ctrs = reinterpret_cast<unsigned*>(scratch + kNoAllocStateWords);
    P.status = d_status ? d_status : reinterpret_cast<int*>(scratch + kNoAllocStateWords + kNoAllocCtrWords);
    P.num_tiles = 0;
    // same kernel and tile choice as per_build_cdf; at most 4096 tiles for n <= 2^24
    return scan_dispatch(P, g_noalloc_sms[dev], s);
}
