// common.cuh -- device helpers: relaxed/acquire memory accesses, mbarrier +
// bulk-copy (TMA) wrappers, bounded waits, Philox4x32-10, thresholds.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#define PER_FULL_MASK 0xffffffffu

// Upper bound on polling iterations of a device-side spin on global memory.
// Each poll sleeps ~0.25-1 us, so such a wait gives up after roughly one to a
// few seconds and records ST_TIMEOUT instead of hanging.
constexpr unsigned kSpinLimit = 1u << 22;

// ---- memory access --------------------------------------------------------

__device__ __forceinline__ void ld_relaxed_v2(const unsigned long long* p, unsigned long long& a,
                                              unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ void st_relaxed_v2(unsigned long long* p, unsigned long long a, unsigned long long b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

// 32-byte relaxed accesses (sm_100+): each 64-bit word is single-copy atomic
// on its own, the four together are not (readers check a tag in every word).
__device__ __forceinline__ void ld_relaxed_v4(const unsigned long long* p, unsigned long long& a,
                                              unsigned long long& b, unsigned long long& c, unsigned long long& d) {
    asm volatile("ld.relaxed.gpu.global.v4.u64 {%0, %1, %2, %3}, [%4];"
                 : "=l"(a), "=l"(b), "=l"(c), "=l"(d)
                 : "l"(p)
                 : "memory");
}
__device__ __forceinline__ void st_relaxed_v4(unsigned long long* p, unsigned long long a, unsigned long long b,
                                              unsigned long long c, unsigned long long d) {
    asm volatile("st.relaxed.gpu.global.v4.u64 [%0], {%1, %2, %3, %4};" ::"l"(p), "l"(a), "l"(b), "l"(c), "l"(d)
                 : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ float4 ld_f4(const float* p) { return *reinterpret_cast<const float4*>(p); }

__device__ __forceinline__ void st_f4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// 256-bit store of v[0..7] (p 32-byte aligned).
__device__ __forceinline__ void st_f8(float* p, const float* v) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(v[0]), "f"(v[1]),
                 "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
}

// ---- mbarrier + bulk copy (global -> shared, completes on an mbarrier) ------

__device__ __forceinline__ unsigned smem_addr(const void* p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Plain (non-multicast) 1-D bulk copy; dst/src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that may suspend the thread in hardware for up to `ns`
// nanoseconds while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait_for(uint64_t* bar, unsigned parity, unsigned ns) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Every device-side wait gives up after this long and records ST_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Bounded wait for phase `parity` of an mbarrier: the thread sleeps in
// hardware between checks.  A bulk copy from valid global memory always
// completes, so the limit is a safety net: on expiry the caller records
// ST_TIMEOUT.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_for(bar, parity, 20000u)) return true;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Barrier across a co-resident grid (cooperative launch).  `ticket` holds
// (generation << 32) | arrivals.  Each CTA adds one arrival; the CTA whose
// arrival completes the grid moves the word to (generation + 1, 0) with one
// more atomic, and the others wait for the generation to change.  The count
// is back at 0 after every barrier, so launches of any grid size can share
// the word.  The wait is bounded (kWaitLimitNs; ST_TIMEOUT).  Writes before
// the barrier are visible to every CTA after it (fence + acquire).  On
// timeout it sets `timeout_bit` in *status and returns false (the same on
// every thread of the CTA); the word is then left mid-barrier and must be
// cleared before the next launch (per_check does).
__device__ __forceinline__ bool grid_barrier(unsigned long long* ticket, int* status, int timeout_bit) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned long long G = gridDim.x;
        const unsigned long long old = atomicAdd(ticket, 1ull);
        int ok = 1;
        if ((old & 0xffffffffull) == G - 1ull) {
            atomicAdd(ticket, (1ull << 32) - G);  // arrivals G -> 0, generation + 1
        } else {
            const unsigned gen = static_cast<unsigned>(old >> 32);
            uint64_t t0 = 0;
            while (static_cast<unsigned>(ld_acquire_u64(ticket) >> 32) == gen) {
                const uint64_t now = global_ns();
                if (t0 == 0) {
                    t0 = now;
                } else if (now - t0 > kWaitLimitNs) {
                    atomicOr(status, timeout_bit);
                    ok = 0;
                    break;
                }
                __nanosleep(64);
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// ---- Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) ----------------------
// First output word for counter (ctr64 lo, ctr64 hi, 0, 0) under key
// (seed lo, seed hi).

__device__ __forceinline__ uint32_t philox_word(uint64_t seed, uint64_t ctr64) {
    uint32_t c0 = static_cast<uint32_t>(ctr64), c1 = static_cast<uint32_t>(ctr64 >> 32);
    uint32_t c2 = 0u, c3 = 0u;
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t m0 = 0xD2511F53u, m1 = 0xCD9E8D57u;
        uint32_t hi0 = __umulhi(m0, c0), lo0 = m0 * c0;
        uint32_t hi1 = __umulhi(m1, c2), lo1 = m1 * c2;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c0;
}

// U in (0, 1]: ((x >> 8) + 1) * 2^-24 (exact).
__device__ __forceinline__ float u01_open_closed(uint64_t seed, uint64_t ctr) {
    return __uint2float_rn((philox_word(seed, ctr) >> 8) + 1u) * 5.9604644775390625e-8f;
}

// U in [0, 1): (x >> 8) * 2^-24 (exact).
__device__ __forceinline__ float u01_closed_open(uint64_t seed, uint64_t ctr) {
    return __uint2float_rn(philox_word(seed, ctr) >> 8) * 5.9604644775390625e-8f;
}

// Stratified threshold u_k = fl32(fl32(fl32(k + U) / B) * T), no contraction.
__device__ __forceinline__ float stratified_threshold(int k, float U, float fB, float T) {
    float a = __fadd_rn(__int2float_rn(k), U);
    float b = __fdiv_rn(a, fB);
    return __fmul_rn(b, T);
}

// ---- x^alpha ---------------------------------------------------------------
// x^alpha = 2^(alpha * log2 x), with x = m * 2^e (m in [1, 2)):
//   alpha*e is split exactly into p + pe (fma gives the product's rounding
//   error), n = rint(p), and the small remainder r = (p - n) + (pe + alpha *
//   log2 m) goes through the hardware base-2 exponential; the result is
//   2^r * 2^n.  Hardware lg2/ex2 approximations (PTX lg2.approx / ex2.approx)
//   bound the error to a few ulp for alpha in [0, 1]; zero, subnormal,
//   infinite, negative and NaN inputs take CUDA's powf (C pow semantics).

__device__ __forceinline__ float hw_lg2(float x) {
    float y;
    asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float hw_ex2(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Flush-to-zero forms: a subnormal input of lg2 reads as 0 (result -inf) and
// a subnormal result of ex2 becomes 0.  Callers keep both out of their
// domain (pow_alpha_n below).
__device__ __forceinline__ float hw_lg2_ftz(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float hw_ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Inputs that are not positive normal floats (zero, subnormal, infinite,
// negative, NaN) take CUDA's powf; kept out of line so the fast path stays
// small at every call site.  `bad` is set for negative and NaN inputs.
static __device__ __noinline__ float pow_special(float x, float alpha, bool* bad) {
    if (!(x >= 0.f)) *bad = true;
    return powf(x, alpha);
}

__device__ __forceinline__ float pow_fast(float x, float alpha, bool& bad) {
    const unsigned bits = __float_as_uint(x);
    if (bits - 0x00800000u >= 0x7f000000u) return pow_special(x, alpha, &bad);
    // e = unbiased exponent as a float, without an int->float conversion:
    // 2^23 + biased exponent, minus 2^23 + 127
    const float e = __fsub_rn(__uint_as_float(0x4B000000u | (bits >> 23)), 8388735.0f);
    const float m = __uint_as_float((bits & 0x007fffffu) | 0x3f800000u);  // [1, 2)
    const float f = hw_lg2(m);                                             // [0, 1)
    const float p = __fmul_rn(alpha, e);
    const float pe = __fmaf_rn(alpha, e, -p);  // alpha*e - p exactly
    // n = rint(p) by the 1.5*2^23 magic-number addition; its low bits give n
    const float big = __fadd_rn(p, 12582912.0f);
    const float n = __fsub_rn(big, 12582912.0f);
    const int ni = static_cast<int>(__float_as_uint(big) - 0x4B400000u);
    const float r = __fadd_rn(__fsub_rn(p, n), __fmaf_rn(alpha, f, pe));
    const float y = hw_ex2(r);
    if (ni > 126 || ni < -126) return ldexpf(y, ni);
    return __fmul_rn(y, __uint_as_float(static_cast<unsigned>(ni + 127) << 23));  // y * 2^n
}

// pow_fast out of line, for the rare inputs outside the direct range below.
static __device__ __noinline__ float pow_split(float x, float alpha) {
    bool bad = false;
    return pow_fast(x, alpha, bad);
}

// max(|a|, b) that returns NaN when either input is NaN.
__device__ __forceinline__ float absmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(fabsf(a)), "f"(b));
    return d;
}

// v[e] <- v[e]^alpha in place (the scan's hot path).  For |log2 x| < lim,
// x^alpha = ex2(alpha * lg2(x)) directly: the hardware lg2 (absolute error
// ~2^-22.6), the fp32 rounding of L = lg2(x) (<= 2^-21 for |L| < 16), the
// rounding of alpha*L (<= 2^-21) and the hardware ex2 (~2^-22.5 relative)
// bound the relative error by ~1e-6.  `lim` = min(16, 120/alpha) (pow_limit)
// keeps x and the result normal floats, so the flush-to-zero forms of lg2
// and ex2 are exact stand-ins for the full ones there.  One range test covers
// all N values; any other input -- tiny, huge, zero, subnormal (lg2 reads it
// as 0), infinite, negative, NaN (the NaN-propagating max fails the test) --
// takes pow_fast's exact exponent split, and negative or NaN inputs set
// `bad`.  mode: 0 = x^alpha, 1 = alpha == 1 (x), 2 = alpha == 0 (1).
template <int N, class Fetch>
__device__ __forceinline__ void pow_alpha_n(float (&v)[N], float alpha, float lim, int mode, bool& bad,
                                            Fetch fetch) {
    if (mode != 0) {
        bool ok = true;
#pragma unroll
        for (int e = 0; e < N; ++e) ok = ok && v[e] >= 0.f;
        if (!ok) bad = true;
        if (mode == 2) {
#pragma unroll
            for (int e = 0; e < N; ++e) v[e] = 1.f;
        }
        return;
    }
    // v <- lg2(v) in place; the rare slow path re-reads the inputs via fetch(e)
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = hw_lg2_ftz(v[e]);
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < N; ++e) m = absmax_nan(v[e], m);
    if (m < lim) {
#pragma unroll
        for (int e = 0; e < N; ++e) v[e] = hw_ex2_ftz(__fmul_rn(alpha, v[e]));
        return;
    }
#pragma unroll
    for (int e = 0; e < N; ++e) {
        const float x = fetch(e);
        if (!(x >= 0.f)) bad = true;
        v[e] = fabsf(v[e]) < lim ? hw_ex2_ftz(__fmul_rn(alpha, v[e])) : pow_split(x, alpha);
    }
}

// Range bound of pow_alpha_n's direct path for exponent alpha > 0: with
// |lg2 x| < lim, |alpha * lg2 x| < 120, so x^alpha stays a normal float.
inline __host__ __device__ float pow_limit(float alpha) {
    return alpha > 7.5f ? 120.f / alpha : 16.f;
}

// ---- packed fp32 pairs (sm_100+ f32x2 arithmetic; per-lane IEEE rounding,
// the same results as two scalar operations) ---------------------------------
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// v[e] <- k + v[e] for an even count of values
template <int N>
__device__ __forceinline__ void add_each(float k, float* v) {
    const unsigned long long k2 = f2_pack(k, k);
#pragma unroll
    for (int e = 0; e < N; e += 2) f2_unpack(f2_add(k2, f2_pack(v[e], v[e + 1])), v[e], v[e + 1]);
}

// max / min of three (max propagates NaN)
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// pow_alpha_n's rule (mode 0) for the N values a lane holds, with one range
// test for the whole warp: when every lane's lg2 values lie in (-lim, lim)
// the direct path runs without a divergent branch; otherwise each value
// takes pow_alpha_n's per-value decision (fetch(e) re-reads input e).  All
// 32 lanes must call it together.  N even.
template <int N, class Fetch>
__device__ __forceinline__ void pow_alpha_warp(float (&v)[N], float alpha, float lim, bool& bad, Fetch fetch) {
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = hw_lg2_ftz(v[e]);
    float mx = max3_nan(v[0], v[1], v[1]), mn = min3(v[0], v[1], v[1]);
#pragma unroll
    for (int e = 2; e + 1 < N; e += 2) {
        mx = max3_nan(mx, v[e], v[e + 1]);
        mn = min3(mn, v[e], v[e + 1]);
    }
    if (__all_sync(PER_FULL_MASK, mx < lim && mn > -lim)) {
        const unsigned long long a2 = f2_pack(alpha, alpha);
#pragma unroll
        for (int e = 0; e < N; e += 2) {
            float p0, p1;
            f2_unpack(f2_mul(a2, f2_pack(v[e], v[e + 1])), p0, p1);
            v[e] = hw_ex2_ftz(p0);
            v[e + 1] = hw_ex2_ftz(p1);
        }
        return;
    }
#pragma unroll
    for (int e = 0; e < N; ++e) {
        const float x = fetch(e);
        if (!(x >= 0.f)) bad = true;
        v[e] = fabsf(v[e]) < lim ? hw_ex2_ftz(__fmul_rn(alpha, v[e])) : pow_split(x, alpha);
    }
}

// Accurate power (CUDA powf), for quantities with a tight error budget.
__device__ __forceinline__ float pow_accurate(float x, float alpha, bool identity) {
    return identity ? x : powf(x, alpha);
}
