// resample.cu -- row-batched systematic resampling (POPCORNBENCH particle
// filter, reference forward: logsumexp-normalised weights, exp, cumsum along
// the particle axis, u_j = (j + U_b)/P with one U_b per row, searchsorted
// (right=False), clamp to P-1).
//
// A cluster of K <= 8 CTAs (512 threads each) per row, CTA k owning a
// contiguous segment of whole 4096-particle chunks, so that a batch of 256
// rows spreads evenly over the SMs; three passes over the segment -- the
// last two served by L2 -- with two exchanges between the cluster's CTAs in
// distributed shared memory (the row maximum; the segments' exact totals,
// whose exclusive prefix is the segment's carry):
//   1. the row maximum m;
//   2. the exact total Q of q_i = fix40(exp(lw_i - m)) (40 fractional bits,
//      64-bit integer sums: order-independent);
//   3. an exact 64-bit integer scan of the same q_i (8 consecutive particles
//      per lane, warp shuffles, a block scan per chunk of 4096 particles),
//      c_i = f(E_i) * fl32(1 / Q), f a monotone fp32 rounding of E
//      (u64_to_f32) -- so c is monotone in the exact prefix E_i.  Every
//      particle i computes n(c_i) = #{j : u_j <= c_i} in closed form (a guess
//      from c*P - U corrected by a couple of exact threshold evaluations) and
//      owns outputs [n(c_{i-1}), n(c_i)) -- exactly the outputs whose
//      lower_bound lands on i, the last particle's run extending to P (the
//      clamp).  The outputs are written in blocks of 4096 starting at the
//      chunk's first output (rounded down to 8): each non-empty run puts its
//      particle at its first output in shared memory, and a block-wide prefix
//      max fills every output with the particle whose run covers it (16-byte
//      stores; no per-output search).
// exp is the hardware ex2 of (lw - m) * log2(e): its relative error (~2^-22)
// stays far inside the CDF tolerance.  Segments of up to 16,384 particles
// (the usual case) are staged in shared memory, so the row is read once and
// exp runs once per particle; longer segments read the row in each pass.  For a power-of-two P the threshold
// division is an exact multiplication by 2^-k.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kLane = 8;                   // consecutive particles per lane per chunk
constexpr int kBatch = 8;                  // float4 loads in flight per thread in passes 1 and 2
constexpr int kChunk = kThreads * kLane;   // 4096
constexpr int kWarpBlock = 32 * kLane;     // outputs per warp per output block (256)
static_assert(kWarps * kWarpBlock == kChunk, "the warps' staging rows tile one block of kChunk");
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplit = 8;      // CTAs per row at most (one cluster, the portable size limit)
constexpr int kMinSegChunks = 4;  // chunks per CTA below which splitting needs a spare wave
// Segments of at most kStageMax particles are staged in shared memory (64 KiB,
// two CTAs per SM): pass 1 copies the log-weights there, pass 2 replaces
// them by w = exp(x - m), and pass 3 reads w back, so the row is read from
// global memory once and exp runs once per particle.  Longer segments (and
// the resample step, which runs three CTAs per SM) read the row in every
// pass and compute exp twice.
constexpr int kStageMax = 4 * kChunk;
static_assert(kStageMax == kThreads * 4 * kBatch, "one pass-1 iteration covers a staged segment");

struct ResampleParams {
    const float* logw;  // may also be out_logw
    int P;
    uint64_t seed, offset;
    const float* __restrict__ u_rows;
    int32_t* __restrict__ out;
    float* __restrict__ out_cdf;
    // the rest of the particle filter's resample step (or null): the
    // resampled particles' states and the reset log-weights
    const float* __restrict__ state;  // [rows][P][D]
    int D;
    float* __restrict__ out_state;    // [rows][P][D]
    float* out_logw;                  // [rows][P] (may be logw itself)
    float reset;                      // fl32(-log P)
    int seg;                          // particles per CTA of a row's cluster (a multiple of kChunk)
    bool staged;                      // the segment lives in shared memory (seg <= kStageMax)
};

// Threshold u_j = fl32(fl32(j + U) / P); for a power of two P the division is
// the exact product with inv_p = 2^-k.
__device__ __forceinline__ float row_threshold(int j, float U, float fP, float inv_p, bool pow2) {
    const float a = __fadd_rn(__int2float_rn(j), U);
    return pow2 ? __fmul_rn(a, inv_p) : __fdiv_rn(a, fP);
}

// #{ j in [0, P) : u_j <= c }.
__device__ __forceinline__ int count_le(float c, float U, int P, float fP, float inv_p, bool pow2) {
    const float g = __fsub_rn(__fmul_rn(c, fP), U);
    int j;
    if (!(g >= 0.f)) j = -1;
    else if (g >= fP) j = P - 1;
    else j = static_cast<int>(g);
    while (j + 1 < P && row_threshold(j + 1, U, fP, inv_p, pow2) <= c) ++j;
    while (j >= 0 && row_threshold(j, U, fP, inv_p, pow2) > c) --j;
    return j + 1;
}

// count_le for a power-of-two P without loops.  u_j <= c exactly when
// fl32(j + U) <= C = c * P (both products by a power of two are exact).  With
// f = floor(C): every j <= f - 1 counts, since fl32(j + U) <= j + 1 <= C (j + 1
// is exact below 2^24, U < 1, and rounding to nearest cannot pass the
// representable j + 1); every j >= f + 1 does not, since fl32(j + U) >= j > C.
// So one exact test, at j = f, settles the count: n = f + [fl32(F + U) <= C]
// with F = floor(C) in floats (exact), clamped to [0, P].  NaN gives 0.  (A
// second test at j = f - 1, always true, went out: 95.0-95.6 -> 94.6 us.)
__device__ __forceinline__ int count_le_pow2(float c, float U, int P, float fP) {
    const float C = __fmul_rn(c, fP);
    const float F = floorf(C);
    int n = __float2int_rz(F);
    if (__fadd_rn(F, U) <= C) ++n;
    return min(max(n, 0), P);
}

// w = exp(x - m) as the hardware ex2 of (x - m) * log2(e); -inf gives 0.
// The flush-to-zero form (one instruction) differs from the other only for
// a subnormal argument (x within ~1e-38 of m, the result 1 either way up to
// the approximation) or a result below 2^-126, which fix40w maps to 0 in
// both: 97.8 against 98.9 us for the resample.
__device__ __forceinline__ float exp_rel(float x, float m) {
    return hw_ex2_ftz(__fmul_rn(__fsub_rn(x, m), kLog2e));
}

// floor(w * 2^40) for w in [0, 1], from the float's exponent and mantissa
// (no 64-bit conversion): w * 2^40 = mant * 2^sh with sh = e - 110 <= 17, so
// it is (mant >> -sh) for sh < 0 (0 from sh <= -24: below 2^-40, zero,
// subnormal) and mant * 2^sh otherwise -- one 32 x 32 -> 64-bit multiply
// instead of 64-bit shifts (resample 100.8 -> 96.8 us; the same value for
// every float in [0, 1], checked exhaustively against the shift form).
__device__ __forceinline__ unsigned long long fix40w(float w) {
    const unsigned bits = __float_as_uint(w);
    const int sh = static_cast<int>(bits >> 23) - 110;
    const unsigned mant = (bits & 0x7fffffu) | 0x800000u;
    const unsigned sl = static_cast<unsigned>(max(sh, 0));            // <= 17 for w <= 1
    const unsigned sr = static_cast<unsigned>(min(max(-sh, 0), 31));  // mant < 2^24: 0 from 24 on
    unsigned p2;  // 2^sl; PTX shl clamps the shift, so a NaN or inf w (sl > 31) gives 0
    asm("shl.b32 %0, %1, %2;" : "=r"(p2) : "r"(1u), "r"(sl));
    return static_cast<unsigned long long>(mant >> sr) * p2;
}

// Monotone fp32 value of E < 2^56: the high half (below 2^24) is exact in
// fp32, the low half is rounded once, and one fused multiply-add combines
// them; a carry into the high half can never make the result decrease.
__device__ __forceinline__ float u64_to_f32(unsigned long long E) {
    const float hi = __uint2float_rn(static_cast<unsigned>(E >> 32));
    const float lo = __uint2float_rn(static_cast<unsigned>(E));
    return __fmaf_rn(hi, 4294967296.0f, lo);
}

__device__ __forceinline__ unsigned long long warp_incl_u64(unsigned long long x, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long y = __shfl_up_sync(PER_FULL_MASK, x, d);
        if (lane >= d) x += y;
    }
    return x;
}

// STEP: the whole resample step (states copied, log-weights reset).  Its state
// copy is memory-bound and gains from a third CTA per SM (40 registers, a few
// spilled); the indices alone run faster at two (62 registers, no spills).
// POW2: P is a power of two, so the threshold count is count_le_pow2's one
// test, compiled in instead of chosen per particle (95 -> 90.7 us at
// 256 x 65536; the step 206 -> 203 us).  STAGED: the segment lives in shared
// memory (the index kernel's usual case); compiled in, it drops the unstaged
// path's loads and registers (90.8 -> 88.6 us; the step, never staged, 203
// -> 199 us with fewer spills).
template <bool STEP, bool POW2, bool STAGED>
__global__ void __launch_bounds__(kThreads, STEP ? 3 : 2) resample_kernel(ResampleParams R) {
    __shared__ float s_f[kWarps];
    __shared__ unsigned long long s_u[kWarps];
    __shared__ float s_cmax;                // this segment's maximum, read by the cluster
    __shared__ unsigned long long s_cq;     // this segment's exact total, read by the cluster
    __shared__ float s_rmax;
    __shared__ unsigned long long s_rq[2];  // the row's total; the segments' before this one
    __shared__ unsigned long long s_cw[2][kWarps];  // per chunk (by parity): the warps' inclusive totals
    __shared__ __align__(16) int s_stage[kChunk];  // one block of outputs (per warp: kWarpBlock of them): run starts, then filled
    __shared__ int s_wmax[kWarps];                  // resample step only: the block-wide max-scan
    __shared__ int s_range[2];                      // resample step only: the chunk's outputs [j_lo, j_hi)
    extern __shared__ __align__(16) float s_seg[];  // the staged segment (kStageMax floats when STAGED)
    cg::cluster_group cluster = cg::this_cluster();
    const int K = static_cast<int>(cluster.num_blocks()), k = static_cast<int>(cluster.block_rank());
    const int b = blockIdx.x / K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int P = R.P;
    const int s0 = k * R.seg, s1 = min(P, s0 + R.seg);  // this CTA's particles (s0 < s1)
    const float* row = R.logw + static_cast<size_t>(b) * P;
    int32_t* orow = R.out + static_cast<size_t>(b) * P;

    // ---- 1: row maximum (kBatch loads in flight per thread) -----------------
    float m = -INFINITY;
    for (int i0 = s0 + threadIdx.x * 4; i0 < s1; i0 += kThreads * 4 * kBatch) {
        float4 q[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + u * kThreads * 4;
            q[u] = i < s1 ? ld_f4(row + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
        if (STAGED) {  // the whole segment, -inf past its end (one iteration)
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                *reinterpret_cast<float4*>(s_seg + (i0 - s0) + u * kThreads * 4) = q[u];
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) m = fmaxf(m, fmaxf(fmaxf(q[u].x, q[u].y), fmaxf(q[u].z, q[u].w)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(PER_FULL_MASK, m, o));
    if (lane == 0) s_f[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mk = s_f[0];
        for (int w = 1; w < kWarps; ++w) mk = fmaxf(mk, s_f[w]);
        s_cmax = mk;
    }
    cluster.sync();  // every segment's maximum is visible to the cluster
    if (warp == 0) {
        float mr = lane < K ? *cluster.map_shared_rank(&s_cmax, lane) : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mr = fmaxf(mr, __shfl_xor_sync(PER_FULL_MASK, mr, o));
        if (lane == 0) s_rmax = mr;
    }
    __syncthreads();
    const float rmax = s_rmax;

    // ---- 2: exact total -------------------------------------------------------------
    unsigned long long acc = 0ull;
    for (int i0 = s0 + threadIdx.x * 4; i0 < s1; i0 += kThreads * 4 * kBatch) {
        float4 q[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + u * kThreads * 4;
            if (STAGED)  // this thread's own pass-1 stores
                q[u] = *reinterpret_cast<const float4*>(s_seg + (i0 - s0) + u * kThreads * 4);
            else
                q[u] = i < s1 ? ld_f4(row + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const float4 w = make_float4(exp_rel(q[u].x, rmax), exp_rel(q[u].y, rmax), exp_rel(q[u].z, rmax),
                                         exp_rel(q[u].w, rmax));
            if (STAGED) *reinterpret_cast<float4*>(s_seg + (i0 - s0) + u * kThreads * 4) = w;
            acc += fix40w(w.x) + fix40w(w.y) + fix40w(w.z) + fix40w(w.w);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(PER_FULL_MASK, acc, o);
    if (lane == 0) s_u[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long qk = 0ull;
        for (int w = 0; w < kWarps; ++w) qk += s_u[w];
        s_cq = qk;
    }
    cluster.sync();  // every segment's total is visible to the cluster (and every maximum read)
    if (warp == 0) {
        const unsigned long long qr = lane < K ? *cluster.map_shared_rank(&s_cq, lane) : 0ull;
        const unsigned long long incl = warp_incl_u64(qr, lane);
        const unsigned long long all = __shfl_sync(PER_FULL_MASK, incl, 31);
        const unsigned long long before = __shfl_sync(PER_FULL_MASK, incl - qr, k);
        if (lane == 0) {
            s_rq[0] = all;
            s_rq[1] = before;
        }
    }
    // the cluster's CTAs may not leave while a peer can still read their
    // totals: arrive here, wait before the exit
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    __syncthreads();
    const unsigned long long Q = s_rq[0];
    // c = fl32(E) * fl32(1 / Q): monotone in E, c(Q) ~= 1
    const float inv = __fdiv_rn(1.0f, u64_to_f32(Q));
    const float fP = static_cast<float>(P);
    const float inv_p = __fdiv_rn(1.0f, fP);
    const float U = R.u_rows ? R.u_rows[b] : u01_closed_open(R.seed, R.offset + static_cast<uint64_t>(b));

    // ---- 3: scan, then the outputs of each chunk ----------------------------------
    // unstaged: the next chunk's loads are issued before the current chunk is
    // processed; staged: w comes from shared memory (written before the
    // barriers above)
    float4 nxt[kLane / 4];
#pragma unroll
    for (int h = 0; h < kLane / 4; ++h) {
        const int i = s0 + threadIdx.x * kLane + 4 * h;
        nxt[h] = !STAGED && i < s1 ? ld_f4(row + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    unsigned long long carry = s_rq[1];  // the exact total of the segments before this one
    for (int c0 = s0; c0 < s1; c0 += kChunk) {
        const int i0 = c0 + threadIdx.x * kLane;
        float4 cur[kLane / 4];
        if (STAGED) {
#pragma unroll
            for (int h = 0; h < kLane / 4; ++h)
                cur[h] = *reinterpret_cast<const float4*>(s_seg + (i0 - s0) + 4 * h);
        } else {
#pragma unroll
            for (int h = 0; h < kLane / 4; ++h) {
                const float4 x = nxt[h];
                cur[h] = make_float4(exp_rel(x.x, rmax), exp_rel(x.y, rmax), exp_rel(x.z, rmax), exp_rel(x.w, rmax));
                const int i = i0 + kChunk + 4 * h;
                nxt[h] = i < s1 ? ld_f4(row + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
        }
        unsigned long long r[kLane];
        unsigned long long run = 0ull;
#pragma unroll
        for (int h = 0; h < kLane / 4; ++h) {
            run += fix40w(cur[h].x);
            r[4 * h] = run;
            run += fix40w(cur[h].y);
            r[4 * h + 1] = run;
            run += fix40w(cur[h].z);
            r[4 * h + 2] = run;
            run += fix40w(cur[h].w);
            r[4 * h + 3] = run;
        }
        const unsigned long long x = warp_incl_u64(run, lane);
        const int par = ((c0 - s0) / kChunk) & 1;
        if (lane == 31) s_cw[par][warp] = x;
        // One barrier per chunk: every warp scans the kWarps warp totals itself
        // (instead of warp 0 scanning them between two barriers).  A warp
        // writes this parity's slots again two chunks later, past the next
        // chunk's barrier, which every warp reaches only after its reads here.
        __syncthreads();
        const unsigned long long t = lane < kWarps ? s_cw[par][lane] : 0ull;
        const unsigned long long wi = warp_incl_u64(t, lane);
        const unsigned long long wb = __shfl_sync(PER_FULL_MASK, wi, warp > 0 ? warp - 1 : 0);
        const unsigned long long before_w = warp > 0 ? wb : 0ull;
        const unsigned long long base = carry + before_w + (x - run);  // E before this lane's first particle
        carry += __shfl_sync(PER_FULL_MASK, wi, kWarps - 1);
        float cv[kLane];
#pragma unroll
        for (int e = 0; e < kLane; ++e) cv[e] = __fmul_rn(u64_to_f32(base + r[e]), inv);
        if (R.out_cdf && i0 < P) {
            float* crow = R.out_cdf + static_cast<size_t>(b) * P + i0;
            st_f4(crow, make_float4(cv[0], cv[1], cv[2], cv[3]));
            if (i0 + 4 < P) st_f4(crow + 4, make_float4(cv[4], cv[5], cv[6], cv[7]));
        }
        // run ends: particle i owns outputs [n(c_{i-1}), n(c_i)), the last
        // particle's run extending to P (the clamp)
        auto n_of = [&](float c) {
            if constexpr (POW2) return count_le_pow2(c, U, P, fP);
            else return count_le(c, U, P, fP, inv_p, false);
        };
        int start = 0;  // n(c) of the particle before this lane's first
        if (i0 >= P) start = P;
        else if (i0 > 0) start = n_of(__fmul_rn(u64_to_f32(base), inv));
        int nend[kLane];
        int prev = start;
#pragma unroll
        for (int e = 0; e < kLane; ++e) {
            const int i = i0 + e;
            int n = prev;
            if (i < P) n = (i == P - 1) ? P : max(n_of(cv[e]), prev);
            nend[e] = n;
            prev = n;
        }
        if constexpr (STEP) {
            // The resample step copies a state row per output, which gains
            // from all warps copying at once: the chunk's outputs [j_lo, j_hi)
            // -- from its first particle's run start to its last particle's
            // run end -- go out in block-wide blocks of kChunk.
            if (threadIdx.x == 0) s_range[0] = start;
            if (threadIdx.x == kThreads - 1) s_range[1] = c0 + kChunk >= P ? P : nend[kLane - 1];
            __syncthreads();
            const int j_lo = s_range[0], j_hi = s_range[1];
            // outputs in blocks of kChunk from the chunk's first output (rounded
            // down to 8, so that a thread's 8 outputs start 32-byte aligned): a
            // chunk of about kChunk outputs mostly needs one block.  Each
            // non-empty run writes its particle at its first output, and a
            // prefix max fills every output with the particle whose run covers it
            int started = -1;  // the last particle started in earlier blocks
            for (int b0 = j_lo & ~(kLane - 1); b0 < j_hi; b0 += kChunk) {
                const int t0 = threadIdx.x * kLane;  // this thread's outputs in the block: b0 + t0 .. + 7
                *reinterpret_cast<int4*>(s_stage + t0) = make_int4(-1, -1, -1, -1);
                *reinterpret_cast<int4*>(s_stage + t0 + 4) = make_int4(-1, -1, -1, -1);
                __syncthreads();
                int a = start;
#pragma unroll
                for (int e = 0; e < kLane; ++e) {
                    if (nend[e] > a && a >= b0 && a < b0 + kChunk) s_stage[a - b0] = i0 + e;
                    a = nend[e];
                }
                __syncthreads();
                const int4 v0 = *reinterpret_cast<const int4*>(s_stage + t0);
                const int4 v1 = *reinterpret_cast<const int4*>(s_stage + t0 + 4);
                int v[kLane] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int e = 1; e < kLane; ++e) v[e] = max(v[e], v[e - 1]);
                int x = v[kLane - 1];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(PER_FULL_MASK, x, d);
                    if (lane >= d) x = max(x, y);
                }
                if (lane == 31) s_wmax[warp] = x;
                int before = __shfl_up_sync(PER_FULL_MASK, x, 1);
                if (lane == 0) before = -1;
                __syncthreads();
                // the maxima of the warps before this one and of all warps: one
                // max-scan over the kWarps warp maxima (lane w holds warp w's)
                int wm = lane < kWarps ? s_wmax[lane] : -1;
#pragma unroll
                for (int d = 1; d < kWarps; d <<= 1) {
                    const int y = __shfl_up_sync(PER_FULL_MASK, wm, d);
                    if (lane >= d) wm = max(wm, y);
                }
                const int wb_in = __shfl_sync(PER_FULL_MASK, wm, warp > 0 ? warp - 1 : 0);
                const int wb = max(started, warp > 0 ? wb_in : -1);
                const int all = max(started, __shfl_sync(PER_FULL_MASK, wm, kWarps - 1));
                before = max(before, wb);
#pragma unroll
                for (int e = 0; e < kLane; ++e) v[e] = max(v[e], before);
                const int j0 = b0 + t0;
                if (j0 >= j_lo && j0 + kLane <= j_hi) {  // written once: evict-first stores
                    __stcs(reinterpret_cast<int4*>(orow + j0), make_int4(v[0], v[1], v[2], v[3]));
                    __stcs(reinterpret_cast<int4*>(orow + j0 + 4), make_int4(v[4], v[5], v[6], v[7]));
                } else {
#pragma unroll
                    for (int e = 0; e < kLane; ++e)
                        if (j0 + e >= j_lo && j0 + e < j_hi) orow[j0 + e] = v[e];
                }
                if (R.out_state) {
                    // the block's particles in shared memory, then their states
                    // copied by consecutive threads for consecutive outputs
                    // (coalesced: neighbouring outputs hold neighbouring particles).
                    // States are read and written once: evict-first loads and
                    // stores, so that they do not push the rows' log-weights,
                    // which the row's later passes read again, out of L2.
                    __syncthreads();  // every thread has read s_stage
                    *reinterpret_cast<int4*>(s_stage + t0) = make_int4(v[0], v[1], v[2], v[3]);
                    *reinterpret_cast<int4*>(s_stage + t0 + 4) = make_int4(v[4], v[5], v[6], v[7]);
                    __syncthreads();
                    const int D = R.D;
                    const float* srow = R.state + static_cast<size_t>(b) * P * D;
                    float* drow = R.out_state + static_cast<size_t>(b) * P * D;
                    for (int t = threadIdx.x; t < kChunk; t += kThreads) {
                        const int j = b0 + t;
                        if (j < j_lo || j >= j_hi) continue;
                        const int i = s_stage[t];
                        if ((D & 3) == 0) {
                            for (int d = 0; d < D; d += 4)
                                __stcs(reinterpret_cast<float4*>(drow + static_cast<size_t>(j) * D + d),
                                       __ldcs(reinterpret_cast<const float4*>(srow + static_cast<size_t>(i) * D + d)));
                        } else {
                            for (int d = 0; d < D; ++d)
                                __stcs(drow + static_cast<size_t>(j) * D + d, __ldcs(srow + static_cast<size_t>(i) * D + d));
                        }
                    }
                }
                started = all;
                __syncthreads();  // s_stage and s_wmax are reused by the next block
            }
        } else {
            // the warp's outputs [w_lo, w_hi): from its first particle's run start
            // to its last particle's run end.  They are written in blocks of 256
            // from w_lo rounded down to 8 (so that a lane's 8 outputs start
            // 32-byte aligned; a warp's ~256 outputs mostly need one block): each
            // non-empty run puts its particle at its first output in the warp's
            // staging row, and a warp prefix max fills every output with the
            // particle whose run covers it.  Only the warp synchronises.
            const int w_lo = __shfl_sync(PER_FULL_MASK, start, 0);
            const int w_hi = __shfl_sync(PER_FULL_MASK, nend[kLane - 1], 31);
            int* stage = s_stage + warp * kWarpBlock;
            const int t0 = lane * kLane;  // this lane's outputs in a block: b0 + t0 .. + 7
            int started = -1;             // the last particle started in earlier blocks
            for (int b0 = w_lo & ~(kLane - 1); b0 < w_hi; b0 += kWarpBlock) {
                *reinterpret_cast<int4*>(stage + t0) = make_int4(-1, -1, -1, -1);
                *reinterpret_cast<int4*>(stage + t0 + 4) = make_int4(-1, -1, -1, -1);
                __syncwarp();
                int a = start;
#pragma unroll
                for (int e = 0; e < kLane; ++e) {
                    if (nend[e] > a && a >= b0 && a < b0 + kWarpBlock) stage[a - b0] = i0 + e;
                    a = nend[e];
                }
                __syncwarp();
                const int4 v0 = *reinterpret_cast<const int4*>(stage + t0);
                const int4 v1 = *reinterpret_cast<const int4*>(stage + t0 + 4);
                int v[kLane] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int e = 1; e < kLane; ++e) v[e] = max(v[e], v[e - 1]);
                int x = v[kLane - 1];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(PER_FULL_MASK, x, d);
                    if (lane >= d) x = max(x, y);
                }
                int before = __shfl_up_sync(PER_FULL_MASK, x, 1);
                if (lane == 0) before = -1;
                before = max(before, started);
                started = max(started, __shfl_sync(PER_FULL_MASK, x, 31));
#pragma unroll
                for (int e = 0; e < kLane; ++e) v[e] = max(v[e], before);
                const int j0 = b0 + t0;
                if (j0 >= w_lo && j0 + kLane <= w_hi) {  // written once: evict-first stores
                    __stcs(reinterpret_cast<int4*>(orow + j0), make_int4(v[0], v[1], v[2], v[3]));
                    __stcs(reinterpret_cast<int4*>(orow + j0 + 4), make_int4(v[4], v[5], v[6], v[7]));
                } else {
#pragma unroll
                    for (int e = 0; e < kLane; ++e)
                        if (j0 + e >= w_lo && j0 + e < w_hi) orow[j0 + e] = v[e];
                }
                __syncwarp();  // the staging row is reused by the next block
            }
        }
    }
    if (R.out_logw) {  // every read of the segment's log-weights is done: the reset may overwrite them
        float* lrow = R.out_logw + static_cast<size_t>(b) * P;
        const float4 r4 = make_float4(R.reset, R.reset, R.reset, R.reset);
        for (int i = s0 + threadIdx.x * 4; i < s1; i += kThreads * 4) __stcs(reinterpret_cast<float4*>(lrow + i), r4);
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace

per_status launch_resample(const float* logw, int rows, int P, uint64_t seed, uint64_t offset,
                           const float* u_rows, int32_t* out, float* out_cdf, const float* state, int D,
                           float* out_state, float* out_logw, float reset, cudaStream_t s) {
    ResampleParams R;
    R.logw = logw;
    R.P = P;
    R.seed = seed;
    R.offset = offset;
    R.u_rows = u_rows;
    R.out = out;
    R.out_cdf = out_cdf;
    R.state = state;
    R.D = D;
    R.out_state = out_state;
    R.out_logw = out_logw;
    R.reset = reset;
    // K <= kMaxSplit CTAs per row, each a whole number of chunks, none
    // empty.  Splitting evens out the SMs' loads when rows outnumber them,
    // but short segments (fewer than kMinSegChunks chunks) only pay off when
    // the split rows still fit one wave of resident CTAs: the passes over a
    // short segment are latency-bound, so extra waves of them cost more than
    // the imbalance they remove.
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PER_ERR_CUDA;
    const bool step = state != nullptr;
    const int64_t slots = (step ? 3 : 2) * static_cast<int64_t>(sms);  // resident CTAs per SM, as launch_bounds
    const int chunks = (P + kChunk - 1) / kChunk;
    int K = min(kMaxSplit, chunks);
    while (K > 1 && (chunks + K - 1) / K < kMinSegChunks && static_cast<int64_t>(rows) * K > slots) --K;
    const int seg_chunks = (chunks + K - 1) / K;
    K = (chunks + seg_chunks - 1) / seg_chunks;
    R.seg = seg_chunks * kChunk;
    R.staged = !step && R.seg <= kStageMax;
    const size_t smem = R.staged ? kStageMax * sizeof(float) : 0;
    if (R.staged) {
        static DeviceCache cache;
        const int ok = device_cached(cache, [&]() {
            return cudaFuncSetAttribute(resample_kernel<false, true, true>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem)) == cudaSuccess &&
                           cudaFuncSetAttribute(resample_kernel<false, false, true>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                static_cast<int>(smem)) == cudaSuccess
                       ? 1 : 2;
        });
        if (ok != 1) return PER_ERR_CUDA;
    }
    if (static_cast<int64_t>(rows) * K > 0x7fffffffll) return PER_ERR_ARG;  // grid limit
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows) * static_cast<unsigned>(K));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(K);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool pow2 = (P & (P - 1)) == 0;
    auto go = [&](auto kernel) { return cudaLaunchKernelEx(&cfg, kernel, R); };
    cudaError_t e;
    if (step)
        e = pow2 ? go(resample_kernel<true, true, false>) : go(resample_kernel<true, false, false>);
    else if (R.staged)
        e = pow2 ? go(resample_kernel<false, true, true>) : go(resample_kernel<false, false, true>);
    else
        e = pow2 ? go(resample_kernel<false, true, false>) : go(resample_kernel<false, false, false>);
    per_note_launch();
    return cuda_status(e);
}
