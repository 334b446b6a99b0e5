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

// Exclusive prefix (exact) of tile t >= 1, computed by one warp.
__device__ u128 lookback(const unsigned long long* desc, int64_t t, unsigned tag_agg, int lane, int* status) {
    u128 excl = 0;
    int64_t j = t - 1;  // lane l examines tile j - l
    unsigned spins = 0;
    for (;;) {
        const int64_t tile = j - lane;
        int st;
        u128 val;
        unsigned first_inc;
        bool timed_out = false;
        for (;;) {
            val = 0;
            st = (tile >= 0) ? read_desc(desc + 4 * tile, tag_agg, val) : 2;  // before tile 0: nothing
            unsigned inc = __ballot_sync(PER_FULL_MASK, st == 2);
            unsigned inv = __ballot_sync(PER_FULL_MASK, st == 0);
            first_inc = inc ? static_cast<unsigned>(__ffs(inc) - 1) : 32u;
            unsigned need = first_inc >= 32u ? PER_FULL_MASK : ((1u << first_inc) - 1u);
            if ((inv & need) == 0u) break;
            if (++spins > kSpinLimit) {
                timed_out = true;
                if (lane == 0) atomicOr(status, ST_TIMEOUT);
                break;
            }
            __nanosleep(spins < 32 ? 64 : 256);
        }
        u128 contrib = (static_cast<unsigned>(lane) <= first_inc && st != 0) ? val : static_cast<u128>(0);
        excl += warp_sum_u128(contrib);
        if (first_inc < 32u || timed_out) break;
        j -= 32;
    }
    return excl;
}

template <int ITEMS>
__global__ void __launch_bounds__(kThreads) build_cdf_kernel(ScanParams P) {
    constexpr int S = ITEMS / 4;
    constexpr int TILE = kThreads * ITEMS;
    __shared__ float s_wtot[kWarps];
    __shared__ unsigned s_tile, s_epoch;
    __shared__ float s_carry[4];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        s_epoch = ld_relaxed_u32(P.ctrs + CTR_SCAN_EPOCH);
        s_tile = atomicAdd(P.ctrs + CTR_SCAN_TICKET, 1u);
    }
    __syncthreads();
    const int64_t t = s_tile;
    const unsigned epoch = s_epoch;
    const int64_t tile_base = t * TILE;
    const int64_t wbase = tile_base + static_cast<int64_t>(warp) * 32 * ITEMS;
    const bool full = tile_base + TILE <= P.n;

    // ---- load + p^alpha ---------------------------------------------------
    float v[ITEMS];
    bool bad = false;
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const int64_t i0 = wbase + s * 128 + lane * 4;
        float4 q;
        if (full || i0 + 3 < P.n) {
            q = ld_f4(P.p + i0);
        } else {
            q.x = i0 < P.n ? P.p[i0] : 0.f;
            q.y = i0 + 1 < P.n ? P.p[i0 + 1] : 0.f;
            q.z = i0 + 2 < P.n ? P.p[i0 + 2] : 0.f;
            q.w = i0 + 3 < P.n ? P.p[i0 + 3] : 0.f;
        }
        bad |= !(q.x >= 0.f) | !(q.y >= 0.f) | !(q.z >= 0.f) | !(q.w >= 0.f);
        float a0 = pow_alpha(q.x, P.alpha, P.alpha_one), a1 = pow_alpha(q.y, P.alpha, P.alpha_one);
        float a2 = pow_alpha(q.z, P.alpha, P.alpha_one), a3 = pow_alpha(q.w, P.alpha, P.alpha_one);
        if (!full) {  // padding beyond n contributes 0 (p^0 would be 1)
            a0 = i0 < P.n ? a0 : 0.f;
            a1 = i0 + 1 < P.n ? a1 : 0.f;
            a2 = i0 + 2 < P.n ? a2 : 0.f;
            a3 = i0 + 3 < P.n ? a3 : 0.f;
        }
        v[4 * s + 0] = a0;
        v[4 * s + 1] = a1;
        v[4 * s + 2] = a2;
        v[4 * s + 3] = a3;
    }
    if (__any_sync(PER_FULL_MASK, bad) && lane == 0) atomicOr(P.status, ST_VALUE);

    // ---- warp-local monotone scan -----------------------------------------
    float carry = 0.f;
#pragma unroll
    for (int s = 0; s < S; ++s) {
        float r0 = v[4 * s];
        float r1 = r0 + v[4 * s + 1];
        float r2 = r1 + v[4 * s + 2];
        float r3 = r2 + v[4 * s + 3];
        float x = r3;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            float y = __shfl_up_sync(PER_FULL_MASK, x, d);
            if (lane >= d) x += y;
        }
        float ex = __shfl_up_sync(PER_FULL_MASK, x, 1);
        if (lane == 0) ex = 0.f;
        const float base = carry + ex;
        float q0 = base + r0, q1 = base + r1, q2 = base + r2, q3 = base + r3;
        float mx = q3;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            float y = __shfl_up_sync(PER_FULL_MASK, mx, d);
            if (lane >= d) mx = fmaxf(mx, y);
        }
        float pm = __shfl_up_sync(PER_FULL_MASK, mx, 1);
        if (lane == 0) pm = carry;
        v[4 * s + 0] = fmaxf(q0, pm);
        v[4 * s + 1] = fmaxf(q1, pm);
        v[4 * s + 2] = fmaxf(q2, pm);
        v[4 * s + 3] = fmaxf(q3, pm);
        carry = __shfl_sync(PER_FULL_MASK, mx, 31);
    }
    if (lane == 0) s_wtot[warp] = carry;
    __syncthreads();

    // ---- warp chunks chained by a left fold; tile aggregate ----------------
    float off = 0.f;
    for (int w = 0; w < warp; ++w) off = off + s_wtot[w];

    if (warp == 0) {
        float agg = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) agg = agg + s_wtot[w];
        bool range_err = false;
        const u128 a_fix = to_fixed(agg, range_err);
        const unsigned tag_agg = 2u * epoch;
        unsigned long long* mine = P.desc + 4 * t;
        u128 excl = 0;
        if (t == 0) {
            if (lane == 0) publish(mine, tag_agg + 1u, a_fix);
        } else {
            if (lane == 0) publish(mine, tag_agg, a_fix);
            excl = lookback(P.desc, t, tag_agg, lane, P.status);
            if (lane == 0) publish(mine, tag_agg + 1u, excl + a_fix);
        }
        if (lane == 0) {
            const double d0 = fixed_to_double(excl);
            const double d1 = fixed_to_double(excl + a_fix);
            const float hi = __double2float_rn(d0);
            const float lo = __double2float_rn(d0 - static_cast<double>(hi));
            s_carry[0] = hi;
            s_carry[1] = lo;
            s_carry[2] = hi;                     // fl32(E_t)
            s_carry[3] = __double2float_rn(d1);  // fl32(E_{t+1})
            if (range_err) atomicOr(P.status, ST_RANGE);
        }
    }
    __syncthreads();

    // ---- apply the carry, clamp, store -------------------------------------
    const float hi = s_carry[0], lo = s_carry[1], sig_lo = s_carry[2], sig_hi = s_carry[3];
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const int64_t i0 = wbase + s * 128 + lane * 4;
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float loc = off + v[4 * s + e];
            const float raw = hi + (lo + loc);
            o[e] = fminf(fmaxf(raw, sig_lo), sig_hi);
        }
        if (full || i0 + 3 < P.n) {
            st_f4(P.cdf + i0, make_float4(o[0], o[1], o[2], o[3]));
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (i0 + e < P.n) P.cdf[i0 + e] = o[e];
        }
    }

    // ---- the last CTA to finish resets the counters for the next call ------
    if (threadIdx.x == 0) {
        unsigned done = atomicAdd(P.ctrs + CTR_SCAN_DONE, 1u);
        if (done == P.num_tiles - 1u) {
            P.ctrs[CTR_SCAN_TICKET] = 0u;
            P.ctrs[CTR_SCAN_DONE] = 0u;
            unsigned next = epoch + 1u;
            if (next >= (1u << 30)) {  // epoch wrap: clear every descriptor once
                for (int64_t i = 0; i < 4 * P.desc_tiles; ++i) P.desc[i] = 0ull;
                next = 1u;
            }
            P.ctrs[CTR_SCAN_EPOCH] = next;
        }
    }
}

template <int ITEMS>
per_status launch_items(per_ctx* ctx, cudaStream_t s) {
    constexpr int TILE = kThreads * ITEMS;
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
    const int64_t tiles = (ctx->size + TILE - 1) / TILE;
    P.num_tiles = static_cast<unsigned>(tiles);
    build_cdf_kernel<ITEMS><<<static_cast<unsigned>(tiles), kThreads, 0, s>>>(P);
    per_note_launch();
    return cuda_status(cudaGetLastError());
}

}  // namespace

// Tile size: 4096 items for large inputs (fewer lookback steps, more bytes in
// flight per CTA); 1024 items when that would leave SMs idle.
per_status launch_build_cdf(per_ctx* ctx, cudaStream_t s) {
    const int64_t big_tiles = (ctx->size + 4095) / 4096;
    if (big_tiles >= 4 * static_cast<int64_t>(ctx->num_sms)) return launch_items<16>(ctx, s);
    return launch_items<4>(ctx, s);
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
// holds it (128 KiB + 128 B) until the process exits.  All calls on a device
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

static __device__ __align__(256) unsigned long long
    g_noalloc_scratch[4 * kNoAllocMaxTiles + kNoAllocCtrWords + 8];

namespace {

std::mutex g_noalloc_mu;
unsigned long long* g_noalloc_ptr[kNoAllocMaxDevices] = {};
int g_noalloc_sms[kNoAllocMaxDevices] = {};

// Zero the descriptors and counters and start the epoch at 1 (a zero tag
// means "never written").
__global__ void noalloc_init_kernel(unsigned long long* scratch) {
    const int words = 4 * kNoAllocMaxTiles + kNoAllocCtrWords + 8;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < words; i += gridDim.x * blockDim.x) scratch[i] = 0ull;
}

__global__ void noalloc_epoch_kernel(unsigned* ctrs) { ctrs[CTR_SCAN_EPOCH] = 1u; }

template <int ITEMS>
per_status noalloc_launch(ScanParams P, cudaStream_t s) {
    constexpr int TILE = kThreads * ITEMS;
    const int64_t tiles = (P.n + TILE - 1) / TILE;
    P.num_tiles = static_cast<unsigned>(tiles);
    build_cdf_kernel<ITEMS><<<static_cast<unsigned>(tiles), kThreads, 0, s>>>(P);
    per_note_launch();
    return cuda_status(cudaGetLastError());
}

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
            noalloc_epoch_kernel<<<1, 1, 0, s>>>(reinterpret_cast<unsigned*>(p + 4 * kNoAllocMaxTiles));
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
    P.ctrs = reinterpret_cast<unsigned*>(scratch + 4 * kNoAllocMaxTiles);
    P.status = d_status ? d_status : reinterpret_cast<int*>(scratch + 4 * kNoAllocMaxTiles + kNoAllocCtrWords);
    P.num_tiles = 0;
    // same tile choice as per_build_cdf; at most 4096 tiles for n <= 2^24
    const int64_t big_tiles = (n + 4095) / 4096;
    if (big_tiles >= 4 * static_cast<int64_t>(g_noalloc_sms[dev])) return noalloc_launch<16>(P, s);
    return noalloc_launch<4>(P, s);
}
