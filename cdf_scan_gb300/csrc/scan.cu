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
//  * Larger inputs: build_cdf_2p_kernel, two passes per L2-sized segment --
//    slice sums from HBM, one exact exchange of chunk sums per segment, then
//    slice scans re-read from L2 -- with a producer warp streaming tiles
//    through a ring of 1-D bulk copies (TMA) on mbarriers.
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

// ---- two passes per segment: reduce, exchange, scan from L2 ----------------
//
// For inputs larger than one wave.  The tiles are cut into segments of at most
// kSegMaxTiles tiles (64 MiB of fp32 at 4096-item tiles), small enough that a
// segment read from HBM is still in L2 when it is read a second time.  Inside
// segment s, CTA c owns a contiguous chunk of the segment's tiles and makes
// two passes over it.  A tile is WARPS slices of 32 x ITEMS items, one per
// compute warp, and the slice is the unit of the exact carries:
//   pass 1: p^alpha and a fixed-order sum per slice (fp32);
//   exchange: the chunk's exact sum (128-bit fixed point) goes to a slot; after
//     a grid barrier every CTA adds the slots up (its exclusive prefix and the
//     segment total) and turns E = prefix + the chunk's earlier slice sums
//     into the carries (hi, lo, fl32(E), fl32(E')) of its slices, E' being
//     the next slice's E;
//   pass 2: re-reads the chunk (from L2), scans each slice with the monotone
//     per-warp scan of the kernels above, and writes
//     clamp(hi + (lo + local), fl32(E), fl32(E')) from registers.
// The clamp bounds come from the exact pass-1 sums, so the CDF is
// non-decreasing across slices, tiles and chunks, and no carry depends on
// timing: the result is bit-reproducible.  Compute warps never wait for each
// other inside a pass; a producer warp refills each stage of the ring of
// bulk copies once all compute warps have released it (mbarriers), and the
// one cross-CTA dependency is the grid barrier per segment.

constexpr int64_t kSegMaxTiles = 4096;  // tiles per segment (64 MiB at 4096 items)
constexpr int kChunkMax = 32;           // tiles per CTA per segment (one lane per tile)

// Barrier among the compute warps only (the producer warp never joins it).
template <int N>
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

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

// Inclusive scan of one run (8 consecutive items per lane, lanes in order)
// continuing from `carry`, the last value of the slice so far: thread-serial
// over the lane's items, shuffles across the lanes, and an exact max-scan
// that removes the dips fp32 reassociation can leave between lanes.  On
// return `carry` is the run's last value.
__device__ __forceinline__ void scan_run(float (&v)[8], float& carry, int lane) {
    float r[8];
    r[0] = v[0];
#pragma unroll
    for (int e = 1; e < 8; ++e) r[e] = r[e - 1] + v[e];
    float x = r[7];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(PER_FULL_MASK, x, d);
        if (lane >= d) x += y;
    }
    float ex = __shfl_up_sync(PER_FULL_MASK, x, 1);
    if (lane == 0) ex = 0.f;
    const float base = carry + ex;
    add_each<8>(base, r);
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
// cy = (hi, lo, fl32(E), fl32(E')), clamped to [fl32(E), fl32(E')] when the
// run's first or last value falls outside (the values are monotone along the
// run), and its coarse-index entries; item n-1 gets fl32(E') itself, the
// correctly rounded exact total.  FAST: full tile, 32-byte aligned cdf.
template <bool FAST, int TILE>
__device__ __forceinline__ void emit_run(const ScanParams& P, float (&v)[8], float4 cy, int64_t tile_base, int i0,
                                         int valid, int lane) {
    add_each<8>(cy.y, v);
    add_each<8>(cy.x, v);
    const float first = __shfl_sync(PER_FULL_MASK, v[0], 0);
    const float last = __shfl_sync(PER_FULL_MASK, v[7], 31);
    if (!(first >= cy.z && last <= cy.w)) {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = fminf(fmaxf(v[e], cy.z), cy.w);
    }
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

// The chunks of a CTA of the two-pass kernel and the sequence of bulk copies
// it consumes: for each segment its chunk's tiles twice (pass 1, then pass 2).
struct TwoPassLoads {
    int64_t T, S, nseg;
    int G, c;
    int64_t s = 0, j = 0, lo = 0, len = 0;
    int pass = 0;
    bool done = false;

    __device__ int64_t seg_count(int64_t sg) const { return T - sg * S < S ? T - sg * S : S; }
    __device__ int64_t chunk_lo(int64_t sg) const { return sg * S + c * seg_count(sg) / G; }
    __device__ int64_t chunk_len(int64_t sg) const { return sg * S + (c + 1) * seg_count(sg) / G - chunk_lo(sg); }
    __device__ void start() {
        lo = chunk_lo(0);
        len = chunk_len(0);
    }
    // the tile of the next copy; false once the sequence is exhausted
    __device__ bool next(int64_t& tile) {
        while (!done && j >= len) {
            j = 0;
            if (pass == 0) {
                pass = 1;
            } else {
                pass = 0;
                if (++s >= nseg) {
                    done = true;
                } else {
                    lo = chunk_lo(s);
                    len = chunk_len(s);
                }
            }
        }
        if (done) return false;
        tile = lo + j++;
        return true;
    }
};

// Layout of the two-pass kernel's exchange words (ScanParams::xsum):
// slots[2][kScanMaxGrid][2] | totals[2][2] | ready.  Parity = segment & 1.
constexpr int64_t kXsumTotals = 4 * kScanMaxGrid;
constexpr int64_t kXsumReady = kXsumTotals + 4;

// Exchange of the two-pass kernel, run by the compute warps of every CTA of
// the co-resident grid once per segment, after each CTA has written its
// chunk's exact sum to slots[c].  The CTA that arrives last at `ticket`
// turns the slots into exclusive prefixes in place with one block-wide scan
// (O(G) reads in all, instead of every CTA reading every slot), writes the
// segment total and publishes `ready`; every CTA waits for `ready`
// (bounded: ST_TIMEOUT) and reads its own prefix and the total into
// ex / tot (all compute threads).
template <int WARPS>
__device__ __forceinline__ void exchange_prefix(const ScanParams& P, int64_t sg, int c, int G, u128& ex, u128& tot) {
    constexpr int THREADS = WARPS * 32;
    constexpr int Q = kScanMaxGrid / THREADS;
    static_assert(kScanMaxGrid % THREADS == 0, "slots per thread");
    __shared__ unsigned long long s_gen;
    __shared__ int s_last;
    __shared__ unsigned long long s_part[WARPS][2];
    __shared__ unsigned long long s_res[4];
    unsigned long long* slots = P.xsum + (sg & 1) * kScanMaxGrid * 2;
    unsigned long long* total = P.xsum + kXsumTotals + (sg & 1) * 2;
    unsigned long long* ready = P.xsum + kXsumReady;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    compute_sync<THREADS>();
    if (threadIdx.x == 0) {
        __threadfence();  // this CTA's slot before its arrival
        // (a CTA chosen by per_debug_drop_tile only reads the ticket: its
        // arrival is lost, so nobody is last and every wait for `ready`
        // runs out)
        const unsigned long long t = c == P.drop_tile ? ld_relaxed_u64(P.ticket) : atomicAdd(P.ticket, 1ull);
        s_gen = t / static_cast<unsigned long long>(G) + 1ull;
        s_last = c != P.drop_tile && (t % static_cast<unsigned long long>(G)) == static_cast<unsigned long long>(G - 1);
        if (s_last) __threadfence();  // every CTA's slot is visible from here on
    }
    compute_sync<THREADS>();
    const unsigned long long gen = s_gen;
    if (s_last) {
        u128 x[Q];
        u128 run = 0;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int k = threadIdx.x * Q + q;
            unsigned long long a = 0ull, b = 0ull;
            if (k < G) ld_relaxed_v2(slots + 2 * k, a, b);
            x[q] = (static_cast<u128>(b) << 64) | a;
        }
#pragma unroll
        for (int q = 0; q < Q; ++q) {  // thread-local exclusive prefixes
            const u128 v = x[q];
            x[q] = run;
            run += v;
        }
        const u128 incl = warp_scan_u128(run, lane);
        if (lane == 31) {
            s_part[warp][0] = static_cast<unsigned long long>(incl);
            s_part[warp][1] = static_cast<unsigned long long>(incl >> 64);
        }
        compute_sync<THREADS>();
        u128 off = incl - run, all = 0;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            const u128 pw = (static_cast<u128>(s_part[w][1]) << 64) | s_part[w][0];
            if (w < warp) off += pw;
            all += pw;
        }
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int k = threadIdx.x * Q + q;
            const u128 e = off + x[q];
            if (k < G) st_relaxed_v2(slots + 2 * k, static_cast<unsigned long long>(e), static_cast<unsigned long long>(e >> 64));
        }
        if (threadIdx.x == 0)
            st_relaxed_v2(total, static_cast<unsigned long long>(all), static_cast<unsigned long long>(all >> 64));
        compute_sync<THREADS>();
        if (threadIdx.x == 0) {
            __threadfence();
            st_release_u64(ready, gen);
        }
    }
    if (threadIdx.x == 0) {
        uint64_t t0 = 0;
        while (ld_acquire_u64(ready) < gen) {
            const uint64_t now = global_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitNs) {
                atomicOr(P.status, ST_TIMEOUT);
                break;
            }
            __nanosleep(32);
        }
        ld_relaxed_v2(slots + 2 * c, s_res[0], s_res[1]);
        ld_relaxed_v2(total, s_res[2], s_res[3]);
    }
    compute_sync<THREADS>();
    ex = (static_cast<u128>(s_res[1]) << 64) | s_res[0];
    tot = (static_cast<u128>(s_res[3]) << 64) | s_res[2];
}

template <int ITEMS, int STAGES, int WARPS, int MINB>
__global__ void __launch_bounds__(WARPS * 32 + 32, MINB) build_cdf_2p_kernel(ScanParams P) {
    constexpr int THREADS = WARPS * 32;  // compute threads; one more warp produces
    constexpr int TILE = THREADS * ITEMS;
    constexpr int RUNS = ITEMS / 8;
    static_assert(ITEMS % 8 == 0, "runs of 8 consecutive items per lane");
    extern __shared__ __align__(128) float s_buf[];  // STAGES x TILE
    __shared__ __align__(8) uint64_t s_full[STAGES], s_empty[STAGES];
    __shared__ float s_agg[kChunkMax * WARPS];              // slice sums of the chunk
    __shared__ float4 s_carry[kChunkMax * WARPS];           // slice carries
    __shared__ volatile int s_abort;                        // a wait ran out: stop waiting

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    TwoPassLoads L;
    L.T = P.num_tiles;
    L.S = P.seg_tiles;
    L.nseg = (L.T + L.S - 1) / L.S;
    L.G = G;
    L.c = c;
    L.start();
    if (threadIdx.x == 0) {
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(&s_full[st], 1);
            mbar_init(&s_empty[st], WARPS);
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // bounded wait; after the first expiry in the CTA nobody waits any more
    auto wait = [&](uint64_t* bar, unsigned parity) {
        if (s_abort) return;
        if (!mbar_wait_bounded(bar, parity)) {
            s_abort = 1;
            atomicOr(P.status, ST_TIMEOUT);
        }
    };

    if (warp == WARPS) {
        // ======================= producer warp ================================
        if (lane == 0) {
            for (uint64_t q = 0;; ++q) {
                int64_t t;
                if (!L.next(t)) break;
                const int st = static_cast<int>(q % STAGES);
                if (q >= STAGES) wait(&s_empty[st], static_cast<unsigned>(q / STAGES - 1) & 1u);
                if (s_abort) break;
                load_tile<TILE>(P, static_cast<unsigned>(t), s_buf + st * TILE, &s_full[st]);
            }
        }
    } else {
        // ======================= compute warps ================================
        u128 base = 0;   // exact total of the earlier segments
        uint64_t q = 0;  // copies consumed
        const int ibase = warp * 32 * ITEMS + lane * 8;  // this lane's first item of run 0
        bool bad = false;
        for (int64_t sg = 0; sg < L.nseg; ++sg) {
            const int64_t lo = L.chunk_lo(sg);
            const int m = static_cast<int>(L.chunk_len(sg));

            // ---- pass 1: slice sums ---------------------------------------
            for (int j = 0; j < m; ++j, ++q) {
                const int st = static_cast<int>(q % STAGES);
                wait(&s_full[st], static_cast<unsigned>(q / STAGES) & 1u);
                const int64_t tile_base = (lo + j) * TILE;
                const int valid = static_cast<int>(P.n - tile_base < TILE ? P.n - tile_base : TILE);
                const float* buf = s_buf + st * TILE;
                float sum = 0.f;
                if (valid == TILE && P.pow_mode != 2) {
                    // full tile: the slice's values at once, one range test
                    float v[ITEMS];
                    slice_values<ITEMS>(P, buf, ibase, v, bad);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s_empty[st]);
                    unsigned long long acc = f2_pack(v[0], v[1]);
#pragma unroll
                    for (int e = 2; e < ITEMS; e += 2) acc = f2_add(acc, f2_pack(v[e], v[e + 1]));
                    float a0, a1;
                    f2_unpack(acc, a0, a1);
                    sum = a0 + a1;
                } else {
#pragma unroll
                    for (int r = 0; r < RUNS; ++r) {
                        float v[8];
                        run_values<TILE>(P, buf, tile_base, valid, ibase + r * 256, v, bad);
#pragma unroll
                        for (int e = 0; e < 8; ++e) sum += v[e];
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s_empty[st]);
                }
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(PER_FULL_MASK, sum, d);
                if (lane == 0) s_agg[j * WARPS + warp] = sum;
            }

            // ---- exchange: chunk sums -> prefixes -> carries of the slices ---
            // Before the barrier, from this CTA's sums alone: lane j of warp w
            // holds the exact prefix of slice (j, w) within the chunk and the
            // next slice's (kChunkMax == 32: one lane per tile).
            static_assert(kChunkMax == 32, "one lane per tile of the chunk");
            compute_sync<THREADS>();  // s_agg complete
            u128 loc = 0, loc_next = 0;
            {
                u128 tsum = 0, before = 0;  // tile j's sum; its slices before this warp's
                bool range_err = false;
                if (lane < m) {
#pragma unroll
                    for (int w = 0; w < WARPS; ++w) {
                        const u128 f = to_fixed(s_agg[lane * WARPS + w], range_err);
                        if (w < warp) before += f;
                        if (w == warp) loc_next = f;
                        tsum += f;
                    }
                }
                if (range_err && warp == 0) atomicOr(P.status, ST_RANGE);
                const u128 incl = warp_scan_u128(tsum, lane);
                loc = incl - tsum + before;
                loc_next += loc;
                if (warp == 0 && lane == 31)  // the chunk's exact sum
                    st_relaxed_v2(P.xsum + (sg & 1) * kScanMaxGrid * 2 + 2 * c,
                                  static_cast<unsigned long long>(incl), static_cast<unsigned long long>(incl >> 64));
            }
            {
                u128 ex, tot;
                exchange_prefix<WARPS>(P, sg, c, G, ex, tot);
                if (lane < m) {  // carry of this warp's slice of tile `lane`
                    float hi, lo2;
                    fixed_to_float2(base + ex + loc, hi, lo2);
                    s_carry[lane * WARPS + warp] = make_float4(hi, lo2, hi, fixed_to_float(base + ex + loc_next));
                }
                base += tot;
            }
            compute_sync<THREADS>();  // s_agg is free for the next segment

            // ---- pass 2: slice scans, written with their carries -------------
            for (int j = 0; j < m; ++j, ++q) {
                const int st = static_cast<int>(q % STAGES);
                wait(&s_full[st], static_cast<unsigned>(q / STAGES) & 1u);
                const int64_t tile_base = (lo + j) * TILE;
                const int valid = static_cast<int>(P.n - tile_base < TILE ? P.n - tile_base : TILE);
                const bool full = valid == TILE;
                const float* buf = s_buf + st * TILE;
                const float4 cy = s_carry[j * WARPS + warp];
                float carry = 0.f;
                if (full && P.pow_mode != 2 && P.cdf_v8) {
                    // full tile: the slice's values at once, then run by run
                    float v[ITEMS];
                    bool unused = false;
                    slice_values<ITEMS>(P, buf, ibase, v, unused);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s_empty[st]);
#pragma unroll
                    for (int r = 0; r < RUNS; ++r) {
                        float(&u)[8] = *reinterpret_cast<float(*)[8]>(v + 8 * r);
                        scan_run(u, carry, lane);
                        emit_run<true, TILE>(P, u, cy, tile_base, ibase + r * 256, TILE, lane);
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < RUNS; ++r) {
                        float v[8];
                        bool unused = false;
                        run_values<TILE>(P, buf, tile_base, valid, ibase + r * 256, v, unused);
                        if (r == RUNS - 1) {  // the stage has been read
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&s_empty[st]);
                        }
                        scan_run(v, carry, lane);
                        emit_run<false, TILE>(P, v, cy, tile_base, ibase + r * 256, valid, lane);
                    }
                }
            }
        }
        if (__any_sync(PER_FULL_MASK, bad) && lane == 0) atomicOr(P.status, ST_VALUE);
    }

    // ---- the last CTA to finish rearms the barrier ticket for the next call --
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned done = atomicAdd(P.ctrs + CTR_SCAN_DONE, 1u);
        if (done == gridDim.x - 1u) {
            P.ctrs[CTR_SCAN_DONE] = 0u;
            *P.ticket = 0ull;
            P.xsum[kXsumReady] = 0ull;
        }
    }
}

// Launch of the two-pass kernel: one co-resident wave (cooperative) of at most
// kScanMaxGrid CTAs; segments of equal size, at most kSegMaxTiles tiles and at
// most kChunkMax tiles per CTA.
template <int ITEMS, int STAGES, int WARPS, int MINB>
per_status launch_scan_2p(ScanParams P, int num_sms, cudaStream_t s) {
    constexpr int TILE = WARPS * 32 * ITEMS;
    const size_t smem = static_cast<size_t>(STAGES) * TILE * sizeof(float);
    if (!P.xsum || !P.ticket) return PER_ERR_STATE;
    static DeviceCache cache;
    const int per_sm = device_cached(cache, [&]() {
        int b = 0;
        if (cudaFuncSetAttribute(build_cdf_2p_kernel<ITEMS, STAGES, WARPS, MINB>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, build_cdf_2p_kernel<ITEMS, STAGES, WARPS, MINB>,
                                                          WARPS * 32 + 32, smem) != cudaSuccess)
            return 0;
        return b;  // 0: the kernel does not fit an SM (a launch error)
    });
    if (per_sm == 0) return PER_ERR_CUDA;
    const int64_t tiles = (P.n + TILE - 1) / TILE;
    if (tiles > 0xffffffffll) return PER_ERR_ARG;
    P.num_tiles = static_cast<unsigned>(tiles);
    int64_t grid = static_cast<int64_t>(num_sms) * per_sm;
    if (grid > tiles) grid = tiles;
    if (grid > kScanMaxGrid) grid = kScanMaxGrid;
    const int64_t seg_max = kSegMaxTiles < kChunkMax * grid ? kSegMaxTiles : kChunkMax * grid;
    const int64_t nseg = (tiles + seg_max - 1) / seg_max;
    P.seg_tiles = (tiles + nseg - 1) / nseg;
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
    const cudaError_t e = cudaLaunchKernelEx(&cfg, build_cdf_2p_kernel<ITEMS, STAGES, WARPS, MINB>, P);
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
// the GPU holds at once, then the two-pass kernel.
per_status scan_dispatch(ScanParams P, int num_sms, cudaStream_t s) {
    if (P.n <= int64_t(1) << 19) {
        const per_status st = launch_scan_wave<256>(P, num_sms, s);
        if (st != PER_ERR_STATE) return st;
    }
    {
        const per_status st = launch_scan_wave<512>(P, num_sms, s);
        if (st != PER_ERR_STATE) return st;
    }
    return launch_scan_2p<16, 4, 8, 3>(P, num_sms, s);
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
    P.xsum = ctx->scan_xsum;
    P.ticket = ctx->tickets + TK_SCAN;
    P.seg_tiles = 0;
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
// entry point runs the same scan kernel as per_build_cdf, but keeps its
// lookback words, chunk sums, barrier ticket and counters in the file-scope
// array below instead of in a context, so the caller only passes the
// priorities and the output CDF and nothing is ever allocated.
//
// The array is part of the library image: every GPU that loads the library
// holds it (about 160 KiB) until the process exits.  All calls on a device
// share it and it keeps the previous call's contents: the kernels leave their
// counters, ticket and ready word at rest for the next call even after a
// bounded wait ran out, and their tile words carry a per-call tag, so
// nothing needs re-arming.  Two calls whose kernels overlap on the GPU --
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
// layout (64-bit words): lookback words | counters | status | chunk sums
// (16-byte aligned) | barrier ticket
constexpr int64_t kNoAllocXsumOff = (kNoAllocStateWords + kNoAllocCtrWords + 8 + 1) & ~int64_t(1);
constexpr int64_t kNoAllocTicketOff = kNoAllocXsumOff + kScanXsumWords;
constexpr int64_t kNoAllocWords = kNoAllocTicketOff + 2;
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
    P.xsum = scratch + kNoAllocXsumOff;
    P.ticket = scratch + kNoAllocTicketOff;
    P.seg_tiles = 0;
    P.drop_tile = -1;
    // same kernels and tile choice as per_build_cdf: the one-wave kernels use
    // at most kMaxWaveTiles tile words (launch_scan_wave checks), and larger
    // inputs go to the two-pass kernel, whose exchange words do not depend
    // on n
    return scan_dispatch(P, g_noalloc_sms[dev], s);
}
