// scan_core.cuh -- pieces of build_cdf shared by the scan kernels (scan.cu)
// and the fused PER step (step.cu): exact 128-bit fixed-point carries, the
// tagged tile-sum words and their exact lookback, and the one-wave tile scan.
// Method: PufferLib PR #615, section 1 "Parallel build_cdf" (an inclusive
// prefix sum of p^alpha rebuilt once per minibatch update, monotone and
// deterministic).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kFracBits = 60;
typedef unsigned __int128 u128;

struct ScanParams {
    const float* __restrict__ p;
    float* __restrict__ cdf;
    int64_t n;
    float alpha;
    bool alpha_one;
    int pow_mode;  // 0: x^alpha, 1: alpha == 1, 2: alpha == 0
    float pow_lim; // pow_limit(alpha)
    bool cdf_v8;   // cdf is 32-byte aligned (256-bit stores)
    unsigned long long* desc;
    int64_t desc_tiles;
    unsigned* ctrs;
    int* status;
    unsigned num_tiles;
    float* coarse;  // every kCoarseStride-th CDF value (or nullptr)
    // streaming kernel only: one tagged record per tile, kRecStride words
    // apart (rec_tiles of them)
    unsigned long long* rec = nullptr;
    int64_t rec_tiles = 0;
    // fault injection for tests (per_debug_drop_tile): the tile whose carry
    // word (one-wave kernels) or record (streaming kernel) this call
    // withholds, or -1
    int64_t drop_tile = -1;
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
// One word per tile (kDescStride apart, each in its own 128-byte line):
// aggw[t * kDescStride] = (2*epoch << 32) | fp32 bits of the tile sum,
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

// With `below`, also the sum over tiles [lo, split) and, in *before, the fp32
// sum word of tile split - 1 (when split > lo).
__device__ u128 sum_aggregates(const ScanState& S, int64_t lo, int64_t hi, unsigned tag_agg, int lane,
                               int* status, int64_t split = -1, u128* below = nullptr, float* before = nullptr) {
    u128 acc = 0, acc_below = 0;  // acc_below: the tiles before `split` (when `below` is given)
    float pv = 0.f;               // the word of tile split - 1, on the lane that reads it
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
                w[q] = (pending >> q) & 1u ? ld_relaxed_u64(S.aggw + (j0 + lane + 32 * q) * kDescStride) : 0ull;
#pragma unroll
            for (int q = 0; q < kLookQ; ++q) {
                if (((pending >> q) & 1u) && static_cast<unsigned>(w[q] >> 32) == tag_agg) {
                    bool err = false;  // range errors are flagged by the tile's owner
                    const u128 a = to_fixed(__uint_as_float(static_cast<unsigned>(w[q])), err);
                    acc += a;
                    if (j0 + lane + 32 * q < split) acc_below += a;
                    if (j0 + lane + 32 * q == split - 1) pv = __uint_as_float(static_cast<unsigned>(w[q]));
                    pending &= ~(1u << q);
                }
            }
            if (!__any_sync(PER_FULL_MASK, pending != 0u)) break;
            // lane 0's clock for the whole warp, so every lane takes the same branch
            const uint64_t now = __shfl_sync(PER_FULL_MASK, global_ns(), 0);
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitNs) {
                if (lane == 0) atomicOr(status, ST_TIMEOUT);
                break;
            }
            __nanosleep(128);
        }
    }
    if (below) *below = warp_sum_u128(acc_below);
    if (before && split > lo) *before = __shfl_sync(PER_FULL_MASK, pv, static_cast<int>((split - 1 - lo) & 31));
    return warp_sum_u128(acc);
}


// The next call's epoch; on wrap every tile word is cleared once.
__device__ __forceinline__ void advance_scan_epoch(const ScanParams& P, unsigned epoch) {
    unsigned next = epoch + 1u;
    if (next >= (1u << 30)) {
        for (int64_t i = 0; i < P.desc_tiles; ++i) P.desc[i * kDescStride] = 0ull;
        for (int64_t i = 0; i < P.rec_tiles * kRecStride; ++i) P.rec[i] = 0ull;
        next = 1u;
    }
    P.ctrs[CTR_SCAN_EPOCH] = next;
}

// ---- one wave of tiles: every tile's CTA resident at once ------------------
//
// For inputs that fit one wave of co-resident CTAs, the CTA that owns tile c
// (THREADS x 8 items) scans it entirely in registers: a monotone per-warp
// scan (thread-serial over 8 items, warp shuffles, an exact max-scan that
// repairs the 1-ulp dips fp32 reassociation can leave between lanes, a left
// fold across warps), publishes the tile's fp32 sum as one tagged word
// (32-bit epoch tag | fp32 bits, so stale words never need clearing), and one
// warp sums the words of tiles 0..c-1 exactly (128-bit fixed point, so the
// carry is the same whatever order they arrive in) while the other warps
// finish their local values.  Each tile writes
// clamp(hi + (lo + local), fl32(E_c), fl32(E_{c+1})) with E_c its exact carry
// as fp32 hi + lo; the clamp bounds are monotone in c, so the CDF is
// non-decreasing.  `src` points at the tile's first priority (global memory,
// or a shared-memory copy); when `s_out` is not null the tile's CDF values
// are also left there (shared memory, TILE floats).  The CDF's last value
// cdf[n-1] is the correctly rounded exact total fl32(E_G) (the last tile's
// upper clamp bound).  When `s_bounds` is not null (shared memory, 3
// floats), warp 0 also sums the words of every tile (P.num_tiles of them)
// and leaves there, without waiting for any other tile's local scan:
//   [0] the previous tile's last CDF value (c > 0): a full tile's last local
//       value is its fp32 sum word (both are the same left fold of the warp
//       totals), so it is clamp(hi' + (lo' + a_{c-1}), fl32(E_{c-1}),
//       fl32(E_c)) with E_{c-1} = E_c - a_{c-1}, as that tile writes it;
//   [1] this tile's last CDF value, the same way;
//   [2] T = cdf[n-1] = fl32(E_G).
// Returns the epoch the tile was tagged with; the caller advances it once
// every tile is done (advance_scan_epoch).

template <int THREADS>
__device__ __forceinline__ unsigned wave_scan_tile(const ScanParams& P, int64_t c, const float* src,
                                                   float* s_out, float* s_bounds = nullptr) {
    constexpr int ITEMS = 8;
    constexpr int WARPS = THREADS / 32;
    constexpr int TILE = THREADS * ITEMS;
    __shared__ float s_wtot[WARPS];
    __shared__ float4 s_carry;
    __shared__ unsigned s_epoch;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t base = c * TILE;
    const int i0 = warp * (32 * ITEMS) + lane * ITEMS;  // this lane's first item in the tile
    if (threadIdx.x == 0) s_epoch = ld_relaxed_u32(P.ctrs + CTR_SCAN_EPOCH);

    float v[ITEMS];
    if (base + i0 + ITEMS <= P.n) {
        const float4 a = ld_f4(src + i0), b = ld_f4(src + i0 + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < ITEMS; ++e) v[e] = base + i0 + e < P.n ? src[i0 + e] : 0.f;
    }
    bool bad = false;
    pow_alpha_n<ITEMS>(v, P.alpha, P.pow_lim, P.pow_mode, bad,
                       [&](int e) { return base + i0 + e < P.n ? src[i0 + e] : 0.f; });
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
    if (threadIdx.x == 0 && c != P.drop_tile)
        *reinterpret_cast<volatile unsigned long long*>(P.desc + c * kDescStride) =
            (static_cast<unsigned long long>(tag_agg) << 32) | __float_as_uint(agg);
    if (warp == 0) {
        u128 excl = 0, total = 0;
        float a_prev = 0.f;
        if (s_bounds)  // every tile's word: the total, and the tiles before c on the way
            total = sum_aggregates(scan_state(P), 0, P.num_tiles, tag_agg, lane, P.status, c, &excl, &a_prev);
        else
            excl = sum_aggregates(scan_state(P), 0, c, tag_agg, lane, P.status);
        // the conversions to fp32 run side by side on lanes 0-3 (the u128
        // values are the same on every lane): lane 0 the carry E_c, lane 1
        // E_{c+1}, lane 2 the total, lane 3 E_{c-1} = E_c - a_{c-1}
        bool range_err = false, unused = false;
        const u128 a_fix = to_fixed(agg, range_err);
        const u128 x = lane == 1 ? excl + a_fix
                     : lane == 2 ? total
                     : lane == 3 ? excl - to_fixed(a_prev, unused) : excl;
        float xh, xl;
        fixed_to_float2(x, xh, xl);
        const float hi = __shfl_sync(PER_FULL_MASK, xh, 0), lo = __shfl_sync(PER_FULL_MASK, xl, 0);
        const float e_next = __shfl_sync(PER_FULL_MASK, xh, 1);
        const float T = __shfl_sync(PER_FULL_MASK, xh, 2);
        const float hp = __shfl_sync(PER_FULL_MASK, xh, 3), lp = __shfl_sync(PER_FULL_MASK, xl, 3);
        if (lane == 0) {
            s_carry = make_float4(hi, lo, hi, e_next);
            if (s_bounds) {
                if (c > 0) s_bounds[0] = fminf(fmaxf(hp + (lp + a_prev), hp), hi);
                s_bounds[1] = base + TILE >= P.n ? T : fminf(fmaxf(hi + (lo + agg), hi), e_next);
                s_bounds[2] = T;
            }
            if (range_err) atomicOr(P.status, ST_RANGE);
        }
    }
    float off = 0.f;
    for (int w = 0; w < warp; ++w) off = off + s_wtot[w];
    __syncthreads();
    const float4 cy = s_carry;
    float o[ITEMS];
#pragma unroll
    for (int e = 0; e < ITEMS; ++e) {
        o[e] = fminf(fmaxf(cy.x + (cy.y + (off + v[e])), cy.z), cy.w);
        if (base + i0 + e == P.n - 1) o[e] = cy.w;  // the last value is fl32(E_G) exactly
    }
    if (s_out) {  // the tile's CDF values for the caller (shared memory)
        *reinterpret_cast<float4*>(s_out + i0) = make_float4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<float4*>(s_out + i0 + 4) = make_float4(o[4], o[5], o[6], o[7]);
    }
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

    return s_epoch;
}
}  // namespace
