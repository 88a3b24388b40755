// In-place KV-cache append for sm_103a: the cache update that precedes
// attention when new tokens arrive (Kimi K2 "KV cache" update step, where the
// new keys and values are concatenated after the cached ones along the
// sequence axis).  Here the cache is preallocated with a fixed capacity, so
// the concatenation is a copy of the new rows into place:
//   k_cache[b, h, start_b + t, :] = k_new[b, h, t, :]   for t < Tn
//   v_cache[b, h, start_b + t, :] = v_new[b, h, t, :]
// Each (b, h) contributes one contiguous span of Tn*384 key bytes and one of
// Tn*256 value bytes on both sides, so the copy is a stream of 16-byte
// vectors: pure HBM traffic (read + write of Tn*640 bytes per (b, h)).
#define MLA_FILE_ID 5   // site ids of the bounds-checked debug build
#include "common.cuh"
#include "kernels.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;               // 16-byte vectors in flight per thread
constexpr int kKVec = kDqk * 2 / 16;     // 24 vectors per key row
constexpr int kVVec = kDv * 2 / 16;      // 16 vectors per value row

struct AppendParams {
    const uint4* k_new;
    const uint4* v_new;
    uint4* k_cache;
    uint4* v_cache;
    const int64_t* start;
    int64_t start_all, cap;
    int BH, H, Tn;
    int* status;
};

// Vector r of the span of (b, h): the key rows first, then the value rows.
__device__ __forceinline__ void copy_span(const AppendParams& p, int bh, int64_t s, int r,
                                          int kspan, int span, uint4& x, bool load) {
    if (r >= span) return;
    // the destination rows s .. s+Tn-1 of (b, h) lie inside the capacity
    MLA_CHECK(bh >= 0 && bh < p.BH && s >= 0 && s + p.Tn <= p.cap && r >= 0, p.status);
    if (r < kspan) {
        if (load) x = __ldcs(p.k_new + int64_t(bh) * kspan + r);
        else p.k_cache[(int64_t(bh) * p.cap + s) * kKVec + r] = x;
    } else {
        const int rv = r - kspan;
        if (load) x = __ldcs(p.v_new + int64_t(bh) * p.Tn * kVVec + rv);
        else p.v_cache[(int64_t(bh) * p.cap + s) * kVVec + rv] = x;
    }
}

__device__ __forceinline__ bool start_ok(const AppendParams& p, int bh, int64_t* s) {
    *s = p.start ? p.start[bh / p.H] : p.start_all;
    return *s >= 0 && *s + p.Tn <= p.cap;
}

// Long spans (a prefill chunk): grid.x tiles one (b, h) span of Tn*40
// vectors and grid.y walks the (b, h).  Short spans (a decode token, 40
// vectors): one flat index over every (b, h) so that no thread idles.
__global__ void __launch_bounds__(kThreads) cache_append_kernel(const AppendParams p, int flat) {
    const int kspan = p.Tn * kKVec, span = p.Tn * (kKVec + kVVec);
    uint4 x[kUnroll];
    if (flat) {
        const int64_t total = int64_t(p.BH) * span;
        const int64_t i0 = int64_t(blockIdx.x) * (kThreads * kUnroll) + threadIdx.x;
        int bh[kUnroll], r[kUnroll];
        int64_t s[kUnroll];
        bool ok[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = i0 + u * kThreads;
            bh[u] = int(i / span);
            r[u] = int(i - int64_t(bh[u]) * span);
            ok[u] = i < total && start_ok(p, bh[u], &s[u]);
            if (i < total && !ok[u] && r[u] == 0) report(p.status, kStInvalid);
            if (ok[u]) copy_span(p, bh[u], s[u], r[u], kspan, span, x[u], true);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (ok[u]) copy_span(p, bh[u], s[u], r[u], kspan, span, x[u], false);
        return;
    }
    const int r0 = blockIdx.x * (kThreads * kUnroll) + threadIdx.x;
    for (int bh = blockIdx.y; bh < p.BH; bh += gridDim.y) {
        int64_t s;
        if (!start_ok(p, bh, &s)) {
            if (threadIdx.x == 0 && blockIdx.x == 0) report(p.status, kStInvalid);
            continue;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            copy_span(p, bh, s, r0 + u * kThreads, kspan, span, x[u], true);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            copy_span(p, bh, s, r0 + u * kThreads, kspan, span, x[u], false);
    }
}

}  // namespace

cudaError_t launch_cache_append(const AppendArgs& a, const DeviceInfo& dev, const KernelTimer& tm,
                                cudaStream_t st) {
    AppendParams p{reinterpret_cast<const uint4*>(a.k_new), reinterpret_cast<const uint4*>(a.v_new),
                   reinterpret_cast<uint4*>(a.k_cache), reinterpret_cast<uint4*>(a.v_cache),
                   a.start, a.start_all, a.cap, a.B * a.H, a.H, a.Tn, dev.status};
    const int span = a.Tn * (kKVec + kVVec);
    const int per_cta = kThreads * kUnroll;
    const int64_t total = int64_t(p.BH) * span;
    const bool flat = span < per_cta && (total + per_cta - 1) / per_cta < (int64_t(1) << 31);
    const dim3 grid = flat ? dim3(unsigned((total + per_cta - 1) / per_cta))
                           : dim3((span + per_cta - 1) / per_cta, p.BH < 65535 ? p.BH : 65535);
    if (tm.begin) cudaEventRecord(tm.begin, st);
    cache_append_kernel<<<grid, kThreads, 0, st>>>(p, flat ? 1 : 0);
    if (tm.end) cudaEventRecord(tm.end, st);
    return cudaGetLastError();
}

}  // namespace mla
