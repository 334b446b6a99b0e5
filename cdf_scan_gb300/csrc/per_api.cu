// per_api.cu -- the C ABI declared in include/per.h: context lifetime,
// argument checking (before any launch) and dispatch to the kernels.
#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "internal.h"

namespace {

std::atomic<uint64_t> g_launches{0};

constexpr int64_t kMaxCapacity = int64_t(1) << 30;
constexpr int64_t kPad = 16384;  // buffer padding: vector loads of a ragged tail stay in bounds
constexpr int64_t kMaxRowBytes = int64_t(1) << 20;  // per_gather / per_step_gather row size limit

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T>
cudaError_t alloc_zero(T** p, size_t count, cudaStream_t s) {
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T));
    if (e != cudaSuccess) {
        *p = nullptr;
        return e;
    }
    return cudaMemsetAsync(*p, 0, count * sizeof(T), s);
}

void free_ctx(per_ctx* c) {
    if (!c) return;
    cudaFree(c->prio);
    cudaFree(c->cdf);
    cudaFree(c->tree);
    cudaFree(c->scan_desc);
    cudaFree(c->winner);
    cudaFree(c->ctrs);
    cudaFree(c->status);
    cudaFree(c->coarse);
    cudaFree(c->sample_bounds);
    cudaFree(c->tickets);
    cudaFree(c->slots);
    cudaFree(c->scan_rec);
    cudaFree(c->step_min);
    cudaFree(c->rank_keys0);
    cudaFree(c->rank_keys1);
    cudaFree(c->rank_vals1);
    cudaFree(c->rank_order);
    cudaFree(c->rank_of);
    cudaFree(c->rank_counts);
    cudaFree(c->rank_totals);
    cudaFree(c->rank_q);
    cudaFree(c->rank_cdf);
    cudaFree(c->rank_coarse);
    std::free(c);
}

}  // namespace

void per_note_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

extern "C" {

uint64_t per_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* per_status_str(per_status s) {
    switch (s) {
        case PER_OK: return "PER_OK";
        case PER_ERR_ARG: return "PER_ERR_ARG: invalid argument";
        case PER_ERR_CUDA: return "PER_ERR_CUDA: CUDA call or launch failed";
        case PER_ERR_OOM: return "PER_ERR_OOM: device allocation failed";
        case PER_ERR_TIMEOUT: return "PER_ERR_TIMEOUT: a bounded device wait ran out";
        case PER_ERR_EMPTY: return "PER_ERR_EMPTY: nothing to sample (size or total is zero)";
        case PER_ERR_STATE: return "PER_ERR_STATE: structure not enabled in this context";
        case PER_ERR_RANGE: return "PER_ERR_RANGE: a tile sum exceeded the exact-carry range";
        case PER_ERR_VALUE: return "PER_ERR_VALUE: negative/NaN priority or index out of range";
    }
    return "PER_ERR_UNKNOWN";
}

per_status per_create(per_ctx** out, int64_t capacity, float alpha, uint32_t flags, void* stream) {
    if (!out) return PER_ERR_ARG;
    *out = nullptr;
    if (capacity < 1 || capacity > kMaxCapacity || !(alpha >= 0.f) || alpha > 1e30f) return PER_ERR_ARG;
    if (flags == 0 || (flags & ~(PER_SCAN | PER_TREE | PER_RANK)) != 0) return PER_ERR_ARG;
    if ((flags & PER_RANK) && (flags != PER_RANK || capacity > kRankMaxN)) return PER_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    per_ctx* c = static_cast<per_ctx*>(std::calloc(1, sizeof(per_ctx)));
    if (!c) return PER_ERR_OOM;
    if (cudaGetDevice(&c->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
        std::free(c);
        return PER_ERR_CUDA;
    }
    c->capacity = capacity;
    c->alloc_n = (capacity + kPad - 1) / kPad * kPad + kPad;
    c->log2_cap = 0;
    while ((int64_t(1) << c->log2_cap) < capacity) ++c->log2_cap;
    c->cap_pow2 = int64_t(1) << c->log2_cap;
    c->size = 0;
    c->alpha = alpha;
    c->flags = flags;
    c->scan_desc_tiles = std::min<int64_t>((c->alloc_n + 1023) / 1024, kMaxWaveTiles);
    c->drop_tile = -1;
    c->scan_rec_tiles = scan_rec_tiles(c->alloc_n);
    c->coarse_n = c->alloc_n / kCoarseStride + 1;
    // the sampler's CTAs: at most max(B / 1024, n / 4096) + 1 of them
    c->sample_bounds_n = std::max<int64_t>(int64_t(1) << 14, c->alloc_n / 4096) + 2;
    c->slot_n = 16 * c->num_sms;
    bool ok = alloc_zero(&c->prio, c->alloc_n, s) == cudaSuccess &&
              alloc_zero(&c->winner, static_cast<size_t>(capacity), s) == cudaSuccess &&
              alloc_zero(&c->ctrs, NUM_CTRS, s) == cudaSuccess &&
              alloc_zero(&c->status, 1, s) == cudaSuccess &&
              alloc_zero(&c->tickets, NUM_TICKETS, s) == cudaSuccess &&
              alloc_zero(&c->slots, static_cast<size_t>(c->slot_n), s) == cudaSuccess;
    if (ok && (flags & PER_SCAN))
        ok = alloc_zero(&c->cdf, c->alloc_n, s) == cudaSuccess &&
             alloc_zero(&c->coarse, static_cast<size_t>(c->coarse_n), s) == cudaSuccess &&
             alloc_zero(&c->sample_bounds, 2 * static_cast<size_t>(c->sample_bounds_n), s) == cudaSuccess &&
             alloc_zero(&c->scan_desc, static_cast<size_t>(scan_state_words(c->scan_desc_tiles)), s) == cudaSuccess &&
             alloc_zero(&c->scan_rec, static_cast<size_t>(c->scan_rec_tiles * kRecStride), s) == cudaSuccess &&
             alloc_zero(&c->step_min, 3, s) == cudaSuccess;
    if (ok && (flags & PER_TREE)) ok = alloc_zero(&c->tree, 2 * static_cast<size_t>(c->cap_pow2) + 16, s) == cudaSuccess;
    if (ok && (flags & PER_RANK)) {
        const size_t cap = static_cast<size_t>(capacity);
        ok = alloc_zero(&c->rank_keys0, cap, s) == cudaSuccess && alloc_zero(&c->rank_keys1, cap, s) == cudaSuccess &&
             alloc_zero(&c->rank_vals1, cap, s) == cudaSuccess && alloc_zero(&c->rank_order, cap, s) == cudaSuccess &&
             alloc_zero(&c->rank_of, cap, s) == cudaSuccess &&
             alloc_zero(&c->rank_counts, static_cast<size_t>(rank_count_words(capacity)), s) == cudaSuccess &&
             alloc_zero(&c->rank_totals, static_cast<size_t>(kRadixDigits), s) == cudaSuccess &&
             alloc_zero(&c->rank_q, c->alloc_n, s) == cudaSuccess &&
             alloc_zero(&c->rank_cdf, c->alloc_n, s) == cudaSuccess &&
             alloc_zero(&c->rank_coarse, static_cast<size_t>(c->coarse_n), s) == cudaSuccess &&
             (c->sample_bounds || alloc_zero(&c->sample_bounds, 2 * static_cast<size_t>(c->sample_bounds_n), s) == cudaSuccess) &&
             (c->scan_desc || alloc_zero(&c->scan_desc, static_cast<size_t>(scan_state_words(c->scan_desc_tiles)), s) == cudaSuccess) &&
             (c->scan_rec || alloc_zero(&c->scan_rec, static_cast<size_t>(c->scan_rec_tiles * kRecStride), s) == cudaSuccess);
    }
    if (ok) {
        // epochs start at 1 (0 marks "never written"); the IS-weight minimum
        // starts above every non-negative float.
        unsigned init[NUM_CTRS] = {0};
        init[CTR_SCAN_EPOCH] = 1u;
        init[CTR_UPD_EPOCH] = 1u;
        init[CTR_ISW_MIN] = 0xffffffffu;
        const unsigned step_init[3] = {0u, 0x7f800000u, 0x7f800000u};  // call 0; +inf, +inf
        ok = cudaMemcpyAsync(c->ctrs, init, sizeof(init), cudaMemcpyHostToDevice, s) == cudaSuccess &&
             (!c->step_min ||
              cudaMemcpyAsync(c->step_min, step_init, sizeof(step_init), cudaMemcpyHostToDevice, s) == cudaSuccess) &&
             cudaStreamSynchronize(s) == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();
        free_ctx(c);
        return PER_ERR_OOM;
    }
    *out = c;
    return PER_OK;
}

per_status per_destroy(per_ctx* ctx) {
    if (!ctx) return PER_OK;
    cudaError_t e = cudaDeviceSynchronize();
    free_ctx(ctx);
    return cuda_status(e);
}

per_status per_set_size(per_ctx* ctx, int64_t n) {
    if (!ctx || n < 0 || n > ctx->capacity) return PER_ERR_ARG;
    ctx->size = n;
    return PER_OK;
}

int64_t per_size(const per_ctx* ctx) { return ctx ? ctx->size : -1; }
int64_t per_capacity_pow2(const per_ctx* ctx) { return ctx ? ctx->cap_pow2 : -1; }
const float* per_priorities_ptr(const per_ctx* ctx) { return ctx ? ctx->prio : nullptr; }
const float* per_cdf_ptr(const per_ctx* ctx) { return ctx ? ctx->cdf : nullptr; }
const float* per_tree_ptr(const per_ctx* ctx) { return ctx ? ctx->tree : nullptr; }
const int32_t* per_rank_order_ptr(const per_ctx* ctx) { return ctx ? ctx->rank_order : nullptr; }
const float* per_rank_cdf_ptr(const per_ctx* ctx) { return ctx ? ctx->rank_cdf : nullptr; }

per_status per_set_priorities(per_ctx* ctx, const float* d_prio, int64_t n, void* stream) {
    if (!ctx || n < 0 || n > ctx->capacity || (n > 0 && (!d_prio || !aligned16(d_prio)))) return PER_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (n > 0 && cudaMemcpyAsync(ctx->prio, d_prio, static_cast<size_t>(n) * sizeof(float),
                                 cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return PER_ERR_CUDA;
    if (cudaMemsetAsync(ctx->prio + n, 0, static_cast<size_t>(ctx->alloc_n - n) * sizeof(float), s) != cudaSuccess)
        return PER_ERR_CUDA;
    ctx->size = n;
    if (ctx->flags & PER_TREE) return launch_tree_from_prio(ctx, s);
    return PER_OK;
}

per_status per_update(per_ctx* ctx, const int32_t* d_idx, const float* d_prio, int32_t n, void* stream) {
    if (!ctx || n < 0 || (n > 0 && (!d_idx || !d_prio))) return PER_ERR_ARG;
    if (n == 0) return PER_OK;
    return launch_update(ctx, d_idx, d_prio, n, static_cast<cudaStream_t>(stream));
}

per_status per_build_cdf(per_ctx* ctx, void* stream) {
    if (!ctx) return PER_ERR_ARG;
    if (!(ctx->flags & PER_SCAN)) return PER_ERR_STATE;
    if (ctx->size < 1) return PER_ERR_EMPTY;
    return launch_build_cdf(ctx, static_cast<cudaStream_t>(stream));
}

per_status per_sample(per_ctx* ctx, int32_t B, uint64_t seed, uint64_t offset, int mode, const float* d_u01,
                      int32_t* d_out_idx, void* stream) {
    if (!ctx || B < 1 || B > (1 << 24) || !d_out_idx) return PER_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (mode == static_cast<int>(PER_SCAN)) {
        if (!(ctx->flags & PER_SCAN)) return PER_ERR_STATE;
        if (ctx->size < 1) return PER_ERR_EMPTY;
        return launch_sample_scan(ctx, B, seed, offset, d_u01, d_out_idx, s);
    }
    if (mode == static_cast<int>(PER_TREE) || mode == static_cast<int>(PER_TREE | PER_IID)) {
        if (!(ctx->flags & PER_TREE)) return PER_ERR_STATE;
        return launch_sample_tree(ctx, B, seed, offset, d_u01, (mode & PER_IID) != 0, d_out_idx, s);
    }
    if (mode == static_cast<int>(PER_RANK)) {
        if (!(ctx->flags & PER_RANK)) return PER_ERR_STATE;
        if (ctx->size < 1) return PER_ERR_EMPTY;
        if (ctx->rank_sorted_n != ctx->size) return PER_ERR_STATE;  // per_rank_build first
        return launch_sample_scan(ctx, B, seed, offset, d_u01, d_out_idx, s);
    }
    return PER_ERR_ARG;
}

per_status per_rank_build(per_ctx* ctx, void* stream) {
    if (!ctx) return PER_ERR_ARG;
    if (!(ctx->flags & PER_RANK)) return PER_ERR_STATE;
    if (ctx->size < 1) return PER_ERR_EMPTY;
    return launch_rank_build(ctx, static_cast<cudaStream_t>(stream));
}

per_status per_is_weights(per_ctx* ctx, const int32_t* d_idx, int32_t B, float beta, float* d_out_w, void* stream) {
    if (!ctx || B < 1 || !d_idx || !d_out_w || !(beta >= 0.f) || beta > 1e30f) return PER_ERR_ARG;
    if ((ctx->flags & PER_RANK) && (ctx->size < 1 || ctx->rank_sorted_n != ctx->size)) return PER_ERR_STATE;
    return launch_is_weights(ctx, d_idx, B, beta, d_out_w, static_cast<cudaStream_t>(stream));
}

per_status per_sample_weighted(per_ctx* ctx, int32_t B, uint64_t seed, uint64_t offset, int mode,
                               const float* d_u01, float beta, int32_t* d_out_idx, float* d_out_w, void* stream) {
    if (!ctx || B < 1 || B > (1 << 24) || !d_out_idx || !d_out_w || !(beta >= 0.f) || beta > 1e30f)
        return PER_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool scan_only = mode == static_cast<int>(PER_SCAN) && ctx->flags == PER_SCAN;
    const bool rank = mode == static_cast<int>(PER_RANK) && ctx->flags == PER_RANK && ctx->rank_sorted_n == ctx->size;
    if ((scan_only || rank) && ctx->size >= 1) {
        const per_status st = launch_sample_scan_weighted(ctx, B, seed, offset, d_u01, beta, d_out_idx, d_out_w, s);
        if (st != PER_ERR_STATE) return st;
    }
    const per_status st = per_sample(ctx, B, seed, offset, mode, d_u01, d_out_idx, stream);
    if (st != PER_OK) return st;
    return per_is_weights(ctx, d_out_idx, B, beta, d_out_w, stream);
}

per_status per_gather(per_ctx* ctx, const void* d_rows, int64_t row_bytes, const int32_t* d_idx, int32_t B,
                      void* d_out, void* stream) {
    if (!ctx || !d_rows || !d_idx || !d_out || B < 1 || row_bytes < 16 || row_bytes > kMaxRowBytes ||
        (row_bytes & 15) != 0 || !aligned16(d_rows) || !aligned16(d_out))
        return PER_ERR_ARG;
    return launch_gather(ctx, d_rows, row_bytes, d_idx, B, d_out, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// per_step, with the copy of the sampled rows when d_rows is not NULL.
per_status step_impl(per_ctx* ctx, const int32_t* d_upd_idx, const float* d_upd_prio, int32_t n_upd, int32_t B,
                     uint64_t seed, uint64_t offset, int mode, const float* d_u01, float beta, int32_t* d_out_idx,
                     float* d_out_w, const void* d_rows, int64_t row_bytes, void* d_out_rows, void* stream) {
    if (!ctx || n_upd < 0 || (n_upd > 0 && (!d_upd_idx || !d_upd_prio))) return PER_ERR_ARG;
    if (B < 1 || B > (1 << 24) || !d_out_idx || !d_out_w || !(beta >= 0.f) || beta > 1e30f) return PER_ERR_ARG;
    if (mode != static_cast<int>(PER_SCAN) && mode != static_cast<int>(PER_TREE) &&
        mode != static_cast<int>(PER_TREE | PER_IID) && mode != static_cast<int>(PER_RANK))
        return PER_ERR_ARG;
    if (d_rows && (!d_out_rows || row_bytes < 16 || row_bytes > kMaxRowBytes || (row_bytes & 15) != 0 ||
                   !aligned16(d_rows) || !aligned16(d_out_rows)))
        return PER_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (mode == static_cast<int>(PER_SCAN) && ctx->flags == PER_SCAN && ctx->size >= 1) {
        const per_status st = launch_step(ctx, d_upd_idx, d_upd_prio, n_upd, B, seed, offset, d_u01, beta, d_out_idx,
                                          d_out_w, d_rows, row_bytes, d_out_rows, s);
        if (st != PER_ERR_STATE) return st;
    }
    per_status st = per_update(ctx, d_upd_idx, d_upd_prio, n_upd, stream);
    if (st != PER_OK) return st;
    if (ctx->flags & PER_SCAN) {
        st = per_build_cdf(ctx, stream);
        if (st != PER_OK) return st;
    }
    if (ctx->flags & PER_RANK) {
        st = per_rank_build(ctx, stream);
        if (st != PER_OK) return st;
    }
    st = per_sample_weighted(ctx, B, seed, offset, mode, d_u01, beta, d_out_idx, d_out_w, stream);
    if (st != PER_OK || !d_rows) return st;
    return launch_gather(ctx, d_rows, row_bytes, d_out_idx, B, d_out_rows, s);
}

}  // namespace

extern "C" {

per_status per_step(per_ctx* ctx, const int32_t* d_upd_idx, const float* d_upd_prio, int32_t n_upd, int32_t B,
                    uint64_t seed, uint64_t offset, int mode, const float* d_u01, float beta, int32_t* d_out_idx,
                    float* d_out_w, void* stream) {
    return step_impl(ctx, d_upd_idx, d_upd_prio, n_upd, B, seed, offset, mode, d_u01, beta, d_out_idx, d_out_w,
                     nullptr, 0, nullptr, stream);
}

per_status per_step_gather(per_ctx* ctx, const int32_t* d_upd_idx, const float* d_upd_prio, int32_t n_upd, int32_t B,
                           uint64_t seed, uint64_t offset, int mode, const float* d_u01, float beta,
                           int32_t* d_out_idx, float* d_out_w, const void* d_rows, int64_t row_bytes,
                           void* d_out_rows, void* stream) {
    if (!d_rows) return PER_ERR_ARG;
    return step_impl(ctx, d_upd_idx, d_upd_prio, n_upd, B, seed, offset, mode, d_u01, beta, d_out_idx, d_out_w,
                     d_rows, row_bytes, d_out_rows, stream);
}

per_status per_total(per_ctx* ctx, int mode, float* d_out, void* stream) {
    if (!ctx || !d_out) return PER_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const float* src = nullptr;
    if (mode == static_cast<int>(PER_TREE)) {
        if (!(ctx->flags & PER_TREE)) return PER_ERR_STATE;
        src = ctx->tree + 1;
    } else if (mode == static_cast<int>(PER_SCAN)) {
        if (!(ctx->flags & PER_SCAN)) return PER_ERR_STATE;
        if (ctx->size < 1) return PER_ERR_EMPTY;
        src = ctx->cdf + ctx->size - 1;
    } else if (mode == static_cast<int>(PER_RANK)) {
        if (!(ctx->flags & PER_RANK)) return PER_ERR_STATE;
        if (ctx->size < 1) return PER_ERR_EMPTY;
        if (ctx->rank_q_n != ctx->size) return PER_ERR_STATE;
        src = ctx->rank_cdf + ctx->size - 1;
    } else {
        return PER_ERR_ARG;
    }
    return cuda_status(cudaMemcpyAsync(d_out, src, sizeof(float), cudaMemcpyDeviceToDevice, s));
}

per_status per_total_host(per_ctx* ctx, int mode, float* h_out, void* stream) {
    if (!ctx || !h_out) return PER_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const float* src = nullptr;
    if (mode == static_cast<int>(PER_TREE)) {
        if (!(ctx->flags & PER_TREE)) return PER_ERR_STATE;
        src = ctx->tree + 1;
    } else if (mode == static_cast<int>(PER_SCAN)) {
        if (!(ctx->flags & PER_SCAN)) return PER_ERR_STATE;
        if (ctx->size < 1) return PER_ERR_EMPTY;
        src = ctx->cdf + ctx->size - 1;
    } else if (mode == static_cast<int>(PER_RANK)) {
        if (!(ctx->flags & PER_RANK)) return PER_ERR_STATE;
        if (ctx->size < 1) return PER_ERR_EMPTY;
        if (ctx->rank_q_n != ctx->size) return PER_ERR_STATE;
        src = ctx->rank_cdf + ctx->size - 1;
    } else {
        return PER_ERR_ARG;
    }
    if (cudaMemcpyAsync(h_out, src, sizeof(float), cudaMemcpyDeviceToHost, s) != cudaSuccess) return PER_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(s));
}

per_status per_debug_drop_tile(per_ctx* ctx, int64_t tile) {
    if (!ctx || tile < -1) return PER_ERR_ARG;
    ctx->drop_tile = tile;
    return PER_OK;
}

per_status per_check(per_ctx* ctx, void* stream) {
    if (!ctx) return PER_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = 0;
    if (cudaMemcpyAsync(&st, ctx->status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(ctx->status, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return PER_ERR_CUDA;
    if (st & ST_TIMEOUT) {
        // a grid barrier may have been left short of arrivals: restart the
        // ticket counts so the next call's barriers line up again
        if (cudaMemsetAsync(ctx->tickets, 0, NUM_TICKETS * sizeof(unsigned long long), s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return PER_ERR_CUDA;
        return PER_ERR_TIMEOUT;
    }
    if (st & ST_RANGE) return PER_ERR_RANGE;
    if (st & ST_VALUE) return PER_ERR_VALUE;
    if (st & ST_EMPTY) return PER_ERR_EMPTY;
    return PER_OK;
}

per_status per_resample(const float* d_logw, int32_t rows, int32_t P, uint64_t seed, uint64_t offset,
                        const float* d_u_rows, int32_t* d_out_idx, float* d_out_cdf, void* stream) {
    if (!d_logw || !d_out_idx || rows < 1 || P < 4 || (P & 3) != 0 || P > (1 << 23)) return PER_ERR_ARG;
    if (!aligned16(d_logw) || !aligned16(d_out_idx) || (d_out_cdf && !aligned16(d_out_cdf))) return PER_ERR_ARG;
    return launch_resample(d_logw, rows, P, seed, offset, d_u_rows, d_out_idx, d_out_cdf, nullptr, 0, nullptr,
                           nullptr, 0.f, static_cast<cudaStream_t>(stream));
}

per_status per_resample_step(const float* d_logw, const float* d_state, int32_t rows, int32_t P, int32_t D,
                             uint64_t seed, uint64_t offset, const float* d_u_rows, int32_t* d_out_idx,
                             float* d_out_state, float* d_out_logw, void* stream) {
    if (!d_logw || !d_out_idx || !d_state || !d_out_state || rows < 1 || P < 4 || (P & 3) != 0 || P > (1 << 23) ||
        D < 1 || D > 4096)
        return PER_ERR_ARG;
    if (!aligned16(d_logw) || !aligned16(d_out_idx) || !aligned16(d_state) || !aligned16(d_out_state) ||
        (d_out_logw && !aligned16(d_out_logw)))
        return PER_ERR_ARG;
    const float reset = static_cast<float>(-std::log(static_cast<double>(P)));
    return launch_resample(d_logw, rows, P, seed, offset, d_u_rows, d_out_idx, nullptr, d_state, D, d_out_state,
                           d_out_logw, reset, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
