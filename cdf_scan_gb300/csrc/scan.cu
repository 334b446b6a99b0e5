// scan.cu -- build_cdf: cdf[i] = sum_{j<=i} p_j^alpha in one pass over HBM.
//
// Method (PufferLib PR #615, section 1 "Parallel build_cdf": an inclusive
// prefix sum of the priorities rebuilt once per minibatch update, monotone,
// deterministic, allocation- and sync-free).  The two-level block scan and
// the serial kernel described there are prior art; this is a single-pass
// scan with an exact, chain-free lookback:
//
//  * A co-resident grid of G CTAs (cooperative launch); CTA c scans tiles
//    c, c+G, c+2G, ... through a 4-stage ring of 1-D bulk copies (TMA)
//    completing on mbarriers.
//  * p^alpha is applied as a tile leaves shared memory.
//  * Inside a tile: each warp scans its contiguous chunk with a thread-serial
//    pass over 8 values plus warp shuffles, repairs the 1-ulp dips fp32
//    reassociation can leave between lanes with an exact max-scan, and the
//    warp chunks are chained by a left fold (each warp starts at the previous
//    warp's last value), so local values are monotone by construction.
//  * Across tiles the carry is exact: a tile's fp32 sum becomes a 128-bit
//    fixed-point integer (60 fractional bits).  A dedicated lookback warp
//    forms the exclusive prefix of tile t as the CTA's own previous inclusive
//    prefix plus the exact sum of the G-1 tile sums published in between --
//    integers, so the carry is the same whatever order they arrive in and the
//    result is bit-reproducible run to run.
//  * Each tile turns its exact carry E_t into fp32 hi + lo and writes
//    clamp(hi + (lo + local), fl32(E_t), fl32(E_{t+1})): the clamp bounds are
//    monotone in t, so the whole CDF is non-decreasing.
//  * Tile sums are published as one 64-bit word (32-bit epoch tag | fp32
//    bits); a reader accepts a word only with the current call's tag, so
//    stale words never need clearing.  The last CTA advances the epoch.

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
    int pow_mode;  // 0: x^alpha, 1: alpha == 1, 2: alpha == 0
    unsigned long long* desc;
    int64_t desc_tiles;
    unsigned* ctrs;
    int* status;
    unsigned num_tiles;
    float* coarse;  // every kCoarseStride-th CDF value (or nullptr)
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

// Correctly rounded (to nearest, ties to even) fp32 value of the fixed-point
// number x; monotone in x.  x < 2^104 here (values below 2^44), so the result
// is a normal float.
__device__ __forceinline__ float fixed_to_float(u128 x) {
    if (x == 0) return 0.f;
    const uint64_t hi = static_cast<uint64_t>(x >> 64), lo = static_cast<uint64_t>(x);
    const int lz = hi ? __clzll(static_cast<long long>(hi)) : 64 + __clzll(static_cast<long long>(lo));
    const u128 y = x << lz;  // leading one at bit 127
    const uint64_t top = static_cast<uint64_t>(y >> 64);
    const bool rest = static_cast<uint64_t>(y) != 0;
    uint32_t m = static_cast<uint32_t>(top >> 40);  // 24 bits, leading one included
    const uint64_t below = top & ((1ull << 40) - 1);
    const uint64_t half = 1ull << 39;
    if (below > half || (below == half && (rest || (m & 1u)))) ++m;
    // value = m * 2^(67 - lz - 23); the leading one of m lands in the exponent
    // field, and a rounding carry to 2^24 bumps the exponent by one
    return __uint_as_float((static_cast<uint32_t>(193 - lz) << 23) + m);
}

// The exact carry E as fp32 hi + lo (hi = fl32(E), lo = fl32(E - hi)).
__device__ __forceinline__ void fixed_to_float2(u128 E, float& hi, float& lo) {
    hi = fixed_to_float(E);
    bool unused = false;
    const u128 h = to_fixed(hi, unused);
    lo = E >= h ? fixed_to_float(E - h) : -fixed_to_float(h - E);
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

// ---- scan state in global memory ---------------------------------------------
// One word per tile: aggw[t] = (2*epoch << 32) | fp32 bits of the tile sum,
// written once per call when the tile has been scanned locally.  A reader
// accepts it only with the current call's tag, so stale words never need
// clearing.
struct ScanState {
    unsigned long long* aggw;
};

__device__ __forceinline__ ScanState scan_state(const ScanParams& P) {
    ScanState S;
    S.aggw = P.desc;
    return S;
}

// Exact sum of the published aggregates of tiles [lo, hi), computed by one
// warp (lane l takes tiles lo + l + 32q).  A poll issues all of a lane's loads
// before looking at any; a word is converted and added once, when its tag
// shows the current call, and later polls only wait for the missing ones.
// Gives up after kWaitLimitNs (ST_TIMEOUT) and returns what it has.
constexpr int kLookQ = 16;  // aggregates per lane per chunk (512 tiles)

__device__ u128 sum_aggregates(const ScanState& S, int64_t lo, int64_t hi, unsigned tag_agg, int lane,
                               int* status) {
    u128 acc = 0;
    uint64_t t0 = 0;
    for (int64_t j0 = lo; j0 < hi; j0 += 32 * kLookQ) {
        unsigned pending = 0;
#pragma unroll
        for (int q = 0; q < kLookQ; ++q)
            if (j0 + lane + 32 * q < hi) pending |= 1u << q;
        for (;;) {
            unsigned long long w[kLookQ];
#pragma unroll
            for (int q = 0; q < kLookQ; ++q)
                w[q] = (pending >> q) & 1u ? ld_relaxed_u64(S.aggw + j0 + lane + 32 * q) : 0ull;
#pragma unroll
            for (int q = 0; q < kLookQ; ++q) {
                if (((pending >> q) & 1u) && static_cast<unsigned>(w[q] >> 32) == tag_agg) {
                    bool err = false;  // range errors are flagged by the tile's owner
                    acc += to_fixed(__uint_as_float(static_cast<unsigned>(w[q])), err);
                    pending &= ~(1u << q);
                }
            }
            if (!__any_sync(PER_FULL_MASK, pending != 0u)) break;
            const uint64_t now = global_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitNs) {
                if (lane == 0) atomicOr(status, ST_TIMEOUT);
                return warp_sum_u128(acc);
            }
            __nanosleep(128);
        }
    }
    return warp_sum_u128(acc);
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

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Barrier among the compute warps only (the lookback warp never joins it).
template <int N>
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory"); }

// Persistent, warp-specialised scan over a co-resident grid of G CTAs (the
// launch is cooperative, so all of them run at once).  CTA c scans tiles
// c, c + G, c + 2G, ... (round k = its k-th tile), so the CTAs sweep the array
// one round at a time.  Each CTA runs WARPS compute warps plus one lookback
// warp:
//   * compute warps: wait for the stage's bulk copy, apply p^alpha, scan the
//     tile locally, park the tile-local values in the stage buffer, publish
//     the tile aggregate and signal `parked`; two tiles behind, wait for that
//     tile's carry, write its CDF values and refill its stage with the tile
//     STAGES rounds ahead;
//   * lookback warp: for each of the CTA's tiles in order, wait `parked`, run
//     the lookback, publish the tile's inclusive prefix, signal `carried`.
// A lookback waits only on tiles of earlier rounds or earlier tiles of the
// same round, so the scan always makes progress.
template <int ITEMS, int STAGES, int WARPS, int MINB>
__global__ void __launch_bounds__(WARPS * 32 + 32, MINB) build_cdf_kernel(ScanParams P) {
    static_assert(STAGES >= 4, "one stage scanning, two awaiting their carry, at least one loading");
    constexpr int THREADS = WARPS * 32;
    constexpr int LAG = 2;
    constexpr int TILE = THREADS * ITEMS;
    constexpr int LANE_ITEMS = 8;             // consecutive items per lane per sub-chunk
    constexpr int SUB = ITEMS / LANE_ITEMS;   // sub-chunks per warp
    constexpr int WCHUNK = 32 * ITEMS;        // items per warp
    extern __shared__ __align__(128) float s_buf[];  // STAGES x TILE
    __shared__ __align__(8) uint64_t s_full[STAGES], s_parked[STAGES], s_carried[STAGES];
    __shared__ float s_agg[STAGES];
    __shared__ float s_carry[STAGES][4];
    __shared__ float s_wtot[2][WARPS];
    __shared__ unsigned s_epoch;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t G = gridDim.x;
    const int64_t c = blockIdx.x;
    const ScanState S = scan_state(P);
    if (threadIdx.x == 0) {
        s_epoch = ld_relaxed_u32(P.ctrs + CTR_SCAN_EPOCH);
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(&s_full[st], 1);
            mbar_init(&s_parked[st], 1);
            mbar_init(&s_carried[st], 1);
            const int64_t t = c + st * G;
            if (t < P.num_tiles) load_tile<TILE>(P, static_cast<unsigned>(t), s_buf + st * TILE, &s_full[st]);
        }
    }
    __syncthreads();
    const unsigned epoch = s_epoch;
    const unsigned tag_agg = 2u * epoch;

    if (warp == WARPS) {
        // ======================= lookback warp ================================
        u128 run = 0;  // inclusive prefix of this CTA's previous tile
        for (int k = 0;; ++k) {
            const int64_t t = c + k * G;
            if (t >= P.num_tiles) break;
            const int st = k % STAGES;
            if (!mbar_wait_bounded(&s_parked[st], static_cast<unsigned>(k / STAGES) & 1u))
                if (lane == 0) atomicOr(P.status, ST_TIMEOUT);
            const float agg = s_agg[st];
            bool range_err = false;
            const u128 a_fix = to_fixed(agg, range_err);
            // exclusive prefix = previous own prefix + the tiles in between
            const u128 excl = run + sum_aggregates(S, k == 0 ? 0 : t - G + 1, t, tag_agg, lane, P.status);
            run = excl + a_fix;
            if (lane == 0) {
                float hi, lo;
                fixed_to_float2(excl, hi, lo);
                s_carry[st][0] = hi;
                s_carry[st][1] = lo;
                s_carry[st][2] = hi;                             // fl32(E_t)
                s_carry[st][3] = fixed_to_float(excl + a_fix);   // fl32(E_{t+1})
                if (range_err) atomicOr(P.status, ST_RANGE);
                mbar_arrive(&s_carried[st]);
            }
        }
    } else {
        // ======================= compute warps ================================
        // Writes the CDF values of the CTA's k-th tile once its carry is known,
        // then refills its stage with the tile STAGES rounds ahead.
        auto emit = [&](int k) {
            const int ps = k % STAGES;
            const int64_t pt = c + k * G;
            if (!mbar_wait_bounded(&s_carried[ps], static_cast<unsigned>(k / STAGES) & 1u))
                atomicOr(P.status, ST_TIMEOUT);
            const int64_t tile_base = pt * TILE;
            const int64_t valid = P.n - tile_base < TILE ? P.n - tile_base : TILE;
            const bool full = valid == TILE;
            const float hi = s_carry[ps][0], lo = s_carry[ps][1];
            const float sig_lo = s_carry[ps][2], sig_hi = s_carry[ps][3];
            const float* buf = s_buf + ps * TILE;
            float o[SUB * 2][4];
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int i0 = warp * WCHUNK + s * 256 + lane * LANE_ITEMS + 4 * h;
                    const float4 loc = *reinterpret_cast<const float4*>(buf + i0);
                    o[2 * s + h][0] = hi + (lo + loc.x);
                    o[2 * s + h][1] = hi + (lo + loc.y);
                    o[2 * s + h][2] = hi + (lo + loc.z);
                    o[2 * s + h][3] = hi + (lo + loc.w);
                }
            }
            // values are monotone along the warp's chunk: clamp only if its
            // first or last value falls outside [fl32(E_t), fl32(E_{t+1})]
            const float wfirst = __shfl_sync(PER_FULL_MASK, o[0][0], 0);
            const float wlast = __shfl_sync(PER_FULL_MASK, o[SUB * 2 - 1][3], 31);
            if (!(wfirst >= sig_lo && wlast <= sig_hi)) {
#pragma unroll
                for (int j = 0; j < SUB * 2; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[j][e] = fminf(fmaxf(o[j][e], sig_lo), sig_hi);
            }
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int i0 = warp * WCHUNK + s * 256 + lane * LANE_ITEMS + 4 * h;
                    const float* oo = o[2 * s + h];
                    if (full || i0 + 3 < valid) {
                        st_f4(P.cdf + tile_base + i0, make_float4(oo[0], oo[1], oo[2], oo[3]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (i0 + e < valid) P.cdf[tile_base + i0 + e] = oo[e];
                    }
                    // coarse[j] = cdf[min(64j + 63, n - 1)].  In a full tile the
                    // entries are the items 64j + 63 (n - 1 is one of them when it
                    // ends the tile): the last item of the second half of every
                    // eighth lane.  A ragged tile checks each item.
                    static_assert(LANE_ITEMS == 8 && kCoarseStride == 64, "coarse lane rule");
                    if (P.coarse) {
                        if (full) {
                            if (h == 1 && (lane & 7) == 7)
                                P.coarse[(tile_base + i0 + 3) / kCoarseStride] = oo[3];
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int64_t g = tile_base + i0 + e;
                                if (g < P.n && ((g & (kCoarseStride - 1)) == kCoarseStride - 1 || g == P.n - 1))
                                    P.coarse[g / kCoarseStride] = oo[e];
                            }
                        }
                    }
                }
            }
            compute_sync<THREADS>();  // the stage was read by everyone
            if (threadIdx.x == 0) {
                const int64_t t2 = pt + STAGES * G;
                if (t2 < P.num_tiles) load_tile<TILE>(P, static_cast<unsigned>(t2), s_buf + ps * TILE, &s_full[ps]);
            }
        };

        // the CTA's tiles: k = 0 .. K-1; iteration k scans tile k and emits k - LAG
        const int K = c < P.num_tiles ? static_cast<int>((P.num_tiles - 1 - c) / G) + 1 : 0;
        for (int k = 0; k < K + LAG; ++k) {
          if (k < K) {
            const int64_t t = c + k * G;
            const int st = k % STAGES;
            if (!mbar_wait_bounded(&s_full[st], static_cast<unsigned>(k / STAGES) & 1u))
                atomicOr(P.status, ST_TIMEOUT);
            float* buf = s_buf + st * TILE;
            const int64_t tile_base = t * TILE;
            const int64_t valid = P.n - tile_base < TILE ? P.n - tile_base : TILE;
            const int bulk = static_cast<int>(valid & ~int64_t(3));
            const bool full = valid == TILE;

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
                    const float4 pa = pow4_alpha(q, P.alpha, P.pow_mode, bad);
                    float a0 = pa.x, a1 = pa.y, a2 = pa.z, a3 = pa.w;
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
            float* wtot = s_wtot[k & 1];
            if (lane == 0) wtot[warp] = carry;
            compute_sync<THREADS>();
            float off = 0.f;
            for (int w = 0; w < warp; ++w) off = off + wtot[w];
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
            if (threadIdx.x == 0) {
                float agg = 0.f;
                for (int w = 0; w < WARPS; ++w) agg = agg + wtot[w];
                s_agg[st] = agg;
                *reinterpret_cast<volatile unsigned long long*>(S.aggw + t) =
                    (static_cast<unsigned long long>(tag_agg) << 32) | __float_as_uint(agg);
                mbar_arrive(&s_parked[st]);
            }
          }
          if (k >= LAG) emit(k - LAG);
        }
    }
    __syncthreads();

    // ---- the last CTA to finish advances the epoch for the next call ---------
    if (threadIdx.x == 0) {
        const unsigned done = atomicAdd(P.ctrs + CTR_SCAN_DONE, 1u);
        if (done == gridDim.x - 1u) {
            P.ctrs[CTR_SCAN_DONE] = 0u;
            unsigned next = epoch + 1u;
            if (next >= (1u << 30)) {  // epoch wrap: clear all scan state once
                for (int64_t i = 0; i < P.desc_tiles; ++i) P.desc[i] = 0ull;
                next = 1u;
            }
            P.ctrs[CTR_SCAN_EPOCH] = next;
        }
    }
}

// ---- one wave of tiles: every tile's CTA resident at once ------------------
//
// For inputs that fit one wave of co-resident CTAs (cooperative launch), CTA c
// scans tile c (THREADS x 8 items) entirely in registers: the same per-warp
// monotone scan as above (thread-serial over 8 items, warp shuffles, exact
// max-scan repair, left fold across warps), publishes the tile's fp32 sum as
// one tagged word, and one warp sums the words of tiles 0..c-1 exactly
// (128-bit fixed point) while the other warps finish their local values.  No
// shared-memory ring, no second pass: the data never leaves registers.

template <int THREADS>
__global__ void __launch_bounds__(THREADS) build_cdf_wave_kernel(ScanParams P) {
    constexpr int ITEMS = 8;
    constexpr int WARPS = THREADS / 32;
    constexpr int TILE = THREADS * ITEMS;
    __shared__ float s_wtot[WARPS];
    __shared__ float4 s_carry;
    __shared__ unsigned s_epoch;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t c = blockIdx.x;
    const int64_t base = c * TILE;
    const int i0 = warp * (32 * ITEMS) + lane * ITEMS;  // this lane's first item in the tile
    if (threadIdx.x == 0) s_epoch = ld_relaxed_u32(P.ctrs + CTR_SCAN_EPOCH);

    float v[ITEMS];
    if (base + i0 + ITEMS <= P.n) {
        const float4 a = ld_f4(P.p + base + i0), b = ld_f4(P.p + base + i0 + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < ITEMS; ++e) v[e] = base + i0 + e < P.n ? P.p[base + i0 + e] : 0.f;
    }
    bool bad = false;
    pow_alpha_n<ITEMS>(v, P.alpha, P.pow_mode, bad, [&](int e) {
        return base + i0 + e < P.n ? P.p[base + i0 + e] : 0.f;
    });
    if (base + i0 + ITEMS > P.n) {  // padding beyond n contributes 0 (p^0 would be 1)
#pragma unroll
        for (int e = 0; e < ITEMS; ++e)
            if (base + i0 + e >= P.n) v[e] = 0.f;
    }
    if (__any_sync(PER_FULL_MASK, bad) && lane == 0) atomicOr(P.status, ST_VALUE);

    // warp-local inclusive scan, monotone across lanes
#pragma unroll
    for (int e = 1; e < ITEMS; ++e) v[e] = v[e - 1] + v[e];
    float x = v[ITEMS - 1];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(PER_FULL_MASK, x, d);
        if (lane >= d) x += y;
    }
    float ex = __shfl_up_sync(PER_FULL_MASK, x, 1);
    if (lane == 0) ex = 0.f;
#pragma unroll
    for (int e = 0; e < ITEMS; ++e) v[e] = ex + v[e];
    float mx = v[ITEMS - 1];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(PER_FULL_MASK, mx, d);
        if (lane >= d) mx = fmaxf(mx, y);
    }
    float pm = __shfl_up_sync(PER_FULL_MASK, mx, 1);
    if (lane == 0) pm = 0.f;
#pragma unroll
    for (int e = 0; e < ITEMS; ++e) v[e] = fmaxf(v[e], pm);
    if (lane == 31) s_wtot[warp] = mx;
    __syncthreads();
    const unsigned tag_agg = 2u * s_epoch;

    // publish the tile sum, then gather the carry (warp 0) while every warp
    // applies its left-fold offset
    float agg = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) agg = agg + s_wtot[w];
    if (threadIdx.x == 0)
        *reinterpret_cast<volatile unsigned long long*>(P.desc + c) =
            (static_cast<unsigned long long>(tag_agg) << 32) | __float_as_uint(agg);
    if (warp == 0) {
        const u128 excl = sum_aggregates(scan_state(P), 0, c, tag_agg, lane, P.status);
        if (lane == 0) {
            bool range_err = false;
            const u128 a_fix = to_fixed(agg, range_err);
            float hi, lo;
            fixed_to_float2(excl, hi, lo);
            s_carry = make_float4(hi, lo, hi, fixed_to_float(excl + a_fix));
            if (range_err) atomicOr(P.status, ST_RANGE);
        }
    }
    float off = 0.f;
    for (int w = 0; w < warp; ++w) off = off + s_wtot[w];
    __syncthreads();
    const float4 cy = s_carry;
    float o[ITEMS];
#pragma unroll
    for (int e = 0; e < ITEMS; ++e) o[e] = fminf(fmaxf(cy.x + (cy.y + (off + v[e])), cy.z), cy.w);
    if (base + i0 + ITEMS <= P.n) {
        st_f4(P.cdf + base + i0, make_float4(o[0], o[1], o[2], o[3]));
        st_f4(P.cdf + base + i0 + 4, make_float4(o[4], o[5], o[6], o[7]));
    } else {
#pragma unroll
        for (int e = 0; e < ITEMS; ++e)
            if (base + i0 + e < P.n) P.cdf[base + i0 + e] = o[e];
    }
    if (P.coarse) {  // coarse[j] = cdf[min(64j + 63, n - 1)]
        static_assert(ITEMS == 8 && kCoarseStride == 64, "coarse lane rule assumes 8 items per lane");
        if (base + i0 + ITEMS < P.n) {
            // n - 1 lies beyond this lane, so its entries are the items 64j + 63:
            // only the last item of every eighth lane can be one
            if ((lane & 7) == 7) P.coarse[(base + i0 + ITEMS - 1) / kCoarseStride] = o[ITEMS - 1];
        } else {
#pragma unroll
            for (int e = 0; e < ITEMS; ++e) {
                const int64_t g = base + i0 + e;
                if (g < P.n && ((g & (kCoarseStride - 1)) == kCoarseStride - 1 || g == P.n - 1))
                    P.coarse[g / kCoarseStride] = o[e];
            }
        }
    }

    // ---- the last CTA to finish advances the epoch for the next call ---------
    if (threadIdx.x == 0) {
        const unsigned done = atomicAdd(P.ctrs + CTR_SCAN_DONE, 1u);
        if (done == gridDim.x - 1u) {
            P.ctrs[CTR_SCAN_DONE] = 0u;
            unsigned next = s_epoch + 1u;
            if (next >= (1u << 30)) {  // epoch wrap: clear all scan state once
                for (int64_t i = 0; i < P.desc_tiles; ++i) P.desc[i] = 0ull;
                next = 1u;
            }
            P.ctrs[CTR_SCAN_EPOCH] = next;
        }
    }
}

// Launches the one-wave kernel when every tile's CTA can be resident at once;
// returns PER_ERR_STATE (nothing launched) otherwise.
template <int THREADS>
per_status launch_scan_wave(ScanParams P, int num_sms, cudaStream_t s) {
    constexpr int TILE = THREADS * 8;
    static int per_sm = 0;
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, build_cdf_wave_kernel<THREADS>, THREADS, 0) !=
            cudaSuccess)
            return PER_ERR_CUDA;
        if (per_sm < 1) per_sm = 1;
    }
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

// Launch: a persistent grid of as many CTAs as can be resident at once
// (never more CTAs than tiles).
template <int ITEMS, int STAGES, int WARPS, int MINB>
per_status launch_scan(ScanParams P, int num_sms, cudaStream_t s) {
    static_assert(ITEMS % 8 == 0, "8 consecutive items per lane per sub-chunk");
    constexpr int TILE = WARPS * 32 * ITEMS;
    const size_t smem = static_cast<size_t>(STAGES) * TILE * sizeof(float);
    static int per_sm = 0;
    if (per_sm == 0) {
        if (cudaFuncSetAttribute(build_cdf_kernel<ITEMS, STAGES, WARPS, MINB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, build_cdf_kernel<ITEMS, STAGES, WARPS, MINB>,
                                                          WARPS * 32 + 32, smem) != cudaSuccess)
            return PER_ERR_CUDA;
        if (per_sm < 1) per_sm = 1;
    }
    const int64_t tiles = (P.n + TILE - 1) / TILE;
    if (tiles > P.desc_tiles) return PER_ERR_ARG;
    P.num_tiles = static_cast<unsigned>(tiles);
    int64_t grid = static_cast<int64_t>(num_sms) * per_sm;
    if (grid > tiles) grid = tiles;
    // cooperative: every CTA of the grid is resident at once (the static tile
    // stride relies on it)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(WARPS * 32 + 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, build_cdf_kernel<ITEMS, STAGES, WARPS, MINB>, P);
    per_note_launch();
    return cuda_status(e);
}

// Tile size: 4096 items for large inputs (fewer lookback steps per byte);
// 2048 items when that would leave SMs without a tile.
per_status scan_dispatch(ScanParams P, int num_sms, cudaStream_t s) {
    // one wave of 2048-item tiles for small inputs, of 4096-item tiles up to
    // what the GPU can hold at once, then the persistent ring
    if (P.n <= int64_t(1) << 19) {
        const per_status st = launch_scan_wave<256>(P, num_sms, s);
        if (st != PER_ERR_STATE) return st;
    }
    {
        const per_status st = launch_scan_wave<512>(P, num_sms, s);
        if (st != PER_ERR_STATE) return st;
    }
    const int64_t big_tiles = (P.n + 4095) / 4096;
    if (big_tiles >= 2 * static_cast<int64_t>(num_sms)) return launch_scan<16, 4, 8, 3>(P, num_sms, s);
    return launch_scan<8, 4, 8, 3>(P, num_sms, s);
}

}  // namespace

per_status launch_build_cdf(per_ctx* ctx, cudaStream_t s) {
    ScanParams P;
    P.p = ctx->prio;
    P.cdf = ctx->cdf;
    P.n = ctx->size;
    P.alpha = ctx->alpha;
    P.alpha_one = ctx->alpha == 1.0f;
    P.pow_mode = ctx->alpha == 1.0f ? 1 : (ctx->alpha == 0.0f ? 2 : 0);
    P.desc = ctx->scan_desc;
    P.desc_tiles = ctx->scan_desc_tiles;
    P.ctrs = ctx->ctrs;
    P.status = ctx->status;
    P.num_tiles = 0;
    P.coarse = ctx->coarse;
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
// holds it (about 33 KiB) until the process exits.  All calls on a device
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

constexpr int64_t kNoAllocStateWords = kNoAllocMaxTiles + 1;  // == scan_state_words(4096)
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
    P.pow_mode = alpha == 1.0f ? 1 : (alpha == 0.0f ? 2 : 0);
    P.desc = scratch;
    P.desc_tiles = kNoAllocMaxTiles;
    P.ctrs = reinterpret_cast<unsigned*>(scratch + kNoAllocStateWords);
    P.status = d_status ? d_status : reinterpret_cast<int*>(scratch + kNoAllocStateWords + kNoAllocCtrWords);
    P.num_tiles = 0;
    P.coarse = nullptr;
    // same kernel and tile choice as per_build_cdf; at most 4096 tiles for n <= 2^24
    return scan_dispatch(P, g_noalloc_sms[dev], s);
}
