// C ABI of the library (declared in include/mla.h): host-side argument
// validation, workspace sizing, the per-device status word, and dispatch to
// the kernel launchers.  Nothing here allocates device memory.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/mla.h"
#include "kernels.h"

namespace {

// Device status: the first error a kernel recorded, and (bounds-checked
// debug build) the site of a failed check.  One per device context.
__device__ int g_status[2];

thread_local std::string t_err;
std::atomic<long long> g_wait_limit_ns{2000000000LL};
std::atomic<int> g_stall_stage{-1};
std::atomic<int> g_sparse_chunk{0};
std::atomic<int> g_prefill_ctas{0};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
mla::DeviceInfo g_dev[kMaxDevices];
unsigned long long g_dev_ctx[kMaxDevices];   // context the cached facts belong to

mla_status fail(mla_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
mla_status fail(mla_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_err = buf;
    return s;
}

mla_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device facts and the status word address for the current device; set up
// on first use in each context of the device (a device reset creates a new
// context, in which the status word has a new address).
mla_status device_info(mla::DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(MLA_ERR_UNSUPPORTED, "device %d", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    mla::DeviceInfo& d = g_dev[dev];
    const unsigned long long ctx = mla::current_context_id();
    if (d.status == nullptr || ctx == 0 || ctx != g_dev_ctx[dev]) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return fail(MLA_ERR_UNSUPPORTED,
                        "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                        major, minor);
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
        d.status = static_cast<int*>(p);
        g_dev_ctx[dev] = mla::current_context_id();   // the lookup made one current
    }
    *out = d;
    return MLA_OK;
}

mla::Knobs knobs() {
    return mla::Knobs{g_wait_limit_ns.load(), g_stall_stage.load(), g_sparse_chunk.load(),
                      g_prefill_ctas.load()};
}

// ----- kernel timing (instrumentation) -----
std::atomic<bool> g_timing{false};
std::mutex g_tm_mu;
struct TimerPool {
    std::vector<mla::KernelTimer> ev;
    size_t used = 0;
};
constexpr int kOps = 10;  // MLA_OP_PREFILL .. MLA_OP_GATHER_PROBE
TimerPool g_pool[kOps];

// Next event pair for `op` when timing is on, else an empty timer.
mla::KernelTimer take_timer(int op) {
    mla::KernelTimer t;
    if (!g_timing.load() || op < 0 || op >= kOps) return t;
    std::lock_guard<std::mutex> lk(g_tm_mu);
    TimerPool& p = g_pool[op];
    if (p.used == p.ev.size()) {
        mla::KernelTimer n;
        if (cudaEventCreate(&n.begin) != cudaSuccess) return t;
        if (cudaEventCreate(&n.end) != cudaSuccess) {
            cudaEventDestroy(n.begin);
            return t;
        }
        p.ev.push_back(n);
    }
    return p.ev[p.used++];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE(cond, code, ...) \
    do {                         \
        if (!(cond)) return fail(code, __VA_ARGS__); \
    } while (0)

mla_status check_ws(void* ws, size_t have, size_t need) {
    if (need == 0) return MLA_OK;
    REQUIRE(ws != nullptr, MLA_ERR_WORKSPACE, "workspace of %zu bytes required, got NULL", need);
    REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, MLA_ERR_WORKSPACE,
            "workspace must be 256-byte aligned");
    REQUIRE(have >= need, MLA_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", have, need);
    return MLA_OK;
}

mla_status check_decode_common(const void* q, const void* k, const void* v, const void* cu,
                               const void* gate, const void* out, int B, int H, int max_len) {
    REQUIRE(q && k && v && cu && out, MLA_ERR_INVALID_ARG, "null tensor pointer");
    REQUIRE(B >= 1 && H >= 1 && max_len >= 1, MLA_ERR_INVALID_ARG,
            "need B >= 1, H >= 1, max length >= 1 (got %d, %d, %d)", B, H, max_len);
    REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out) &&
                (gate == nullptr || aligned16(gate)) && (reinterpret_cast<uintptr_t>(cu) & 7u) == 0,
            MLA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    REQUIRE(int64_t(B) * H * ((int64_t(max_len) + 63) / 64) < (int64_t(1) << 31),
            MLA_ERR_UNSUPPORTED, "B*H*max_len too large for one call");
    return MLA_OK;
}

}  // namespace

extern "C" {

const char* mla_last_error(void) { return t_err.c_str(); }

mla_status mla_debug_set(int knob, long long value) {
    switch (knob) {
        case MLA_DEBUG_WAIT_LIMIT_NS:
            g_wait_limit_ns.store(value > 0 ? value : 2000000000LL);
            return MLA_OK;
        case MLA_DEBUG_STALL_STAGE:
            g_stall_stage.store(value >= 0 && value < (1LL << 30) ? int(value) : -1);
            return MLA_OK;
        case MLA_DEBUG_SPARSE_CHUNK:
            if (value != 0 && (value < 64 || value > 2048 || (value & (value - 1))))
                return fail(MLA_ERR_INVALID_ARG, "sparse chunk must be 0 or a power of two in [64, 2048]");
            g_sparse_chunk.store(int(value));
            return MLA_OK;
        case MLA_DEBUG_PREFILL_CTAS:
            if (value < 0 || value > 2)
                return fail(MLA_ERR_INVALID_ARG, "prefill CTAs per MMA must be 0, 1 or 2");
            g_prefill_ctas.store(int(value));
            return MLA_OK;
        default:
            return fail(MLA_ERR_INVALID_ARG, "unknown debug knob %d", knob);
    }
}

size_t mla_workspace_size(int op, int B, int H, int max_seqlen, int topk) {
    switch (op) {
        case MLA_OP_PREFILL:
        case MLA_OP_CACHE_APPEND:
            return 0;
        case MLA_OP_DECODE:
            if (B < 1 || H < 1 || max_seqlen < 1) return 0;
            return mla::plan_decode(B, H, max_seqlen, false).total;
        case MLA_OP_SPARSE_DECODE:
            if (B < 1 || H < 1 || topk < 1 || topk > mla::kMaxTopk) return 0;
            return mla::plan_decode(B, H, topk, true, g_sparse_chunk.load()).total;
        case MLA_OP_INDEX_TOPK:
            if (B < 1 || max_seqlen < 1 || max_seqlen > (1 << 24)) return 0;
            return mla::plan_index(B, max_seqlen).total;
        case MLA_OP_INDEX_TOPK_FP8:
            if (B < 1 || max_seqlen < 1 || max_seqlen > (1 << 24)) return 0;
            return mla::plan_index(B, max_seqlen, true).total;
        case MLA_OP_PREFILL_INDEX_TOPK:
            if (B < 1 || max_seqlen < B || max_seqlen >= (1 << 24)) return 0;
            return mla::prefill_index_ws(B, max_seqlen);
        case MLA_OP_SPARSE_PREFILL_LATENT:
        case MLA_OP_LATENT_DECODE: {
            if (B < 1 || H < 16 || H > 96 || H % 16 != 0) return 0;
            mla::DeviceInfo d;
            if (device_info(&d) != MLA_OK) return 0;
            return mla::plan_latent(B, H, d.sms).total;
        }
        default:
            return 0;
    }
}

mla_status mla_timing_enable(int on) {
    g_timing.store(on != 0);
    return MLA_OK;
}

mla_status mla_timing_read(int op, double* total_ms, long long* launches) {
    REQUIRE(op >= 0 && op < kOps && total_ms && launches, MLA_ERR_INVALID_ARG,
            "mla_timing_read: bad op or null output");
    std::lock_guard<std::mutex> lk(g_tm_mu);
    TimerPool& p = g_pool[op];
    double sum = 0.0;
    for (size_t i = 0; i < p.used; ++i) {
        cudaError_t e = cudaEventSynchronize(p.ev[i].end);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
        float ms = 0.f;
        e = cudaEventElapsedTime(&ms, p.ev[i].begin, p.ev[i].end);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
        sum += ms;
    }
    *total_ms = sum;
    *launches = static_cast<long long>(p.used);
    p.used = 0;
    return MLA_OK;
}

mla_status mla_check_device_status(mla_stream stream) {
    mla::DeviceInfo d;
    mla_status s = device_info(&d);
    if (s != MLA_OK) return s;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int w[2] = {0, 0};
    e = cudaMemcpyFromSymbol(w, g_status, sizeof w);
    if (e != cudaSuccess) return cuda_fail(e, "read status");
    const int zero[2] = {0, 0};
    e = cudaMemcpyToSymbol(g_status, zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "clear status");
    const int v = w[0];
    switch (v) {
        case 0: return MLA_OK;
        case MLA_ERR_TIMEOUT: return fail(MLA_ERR_TIMEOUT, "a device pipeline wait ran out");
        case MLA_ERR_BAD_INDEX:
            return fail(MLA_ERR_BAD_INDEX, "a selected position lies outside its sequence");
        case MLA_ERR_INVALID_ARG:
            return fail(MLA_ERR_INVALID_ARG, "a sequence length is outside [1, max_seqlen]");
        case MLA_ERR_CHECK: {
            static const char* const files[] = {"?", "decode.cu", "prefill.cu", "indexer.cu",
                                                "latent.cu", "cache.cu", "probe.cu"};
            const int id = w[1] / 100000, line = w[1] % 100000;
            return fail(MLA_ERR_CHECK, "bounds check failed at %s:%d",
                        files[id >= 0 && id <= 6 ? id : 0], line);
        }
        default: return fail(static_cast<mla_status>(v), "device status %d", v);
    }
}

mla_status mla_decode(const mla_bf16* q, const mla_bf16* k, const mla_bf16* v,
                      const int64_t* cu_seqlens, int B, int H, int max_seqlen,
                      const mla_bf16* gate, mla_bf16* out, float scale, void* ws,
                      size_t ws_bytes, mla_stream stream) {
    mla_status s = check_decode_common(q, k, v, cu_seqlens, gate, out, B, H, max_seqlen);
    if (s != MLA_OK) return s;
    REQUIRE(scale > 0.f && scale < 1e30f, MLA_ERR_INVALID_ARG, "scale must be positive finite");
    const mla::DecodePlan pl = mla::plan_decode(B, H, max_seqlen, false);
    if ((s = check_ws(ws, ws_bytes, pl.total)) != MLA_OK) return s;
    mla::DeviceInfo d;
    if ((s = device_info(&d)) != MLA_OK) return s;
    mla::DecodeArgs a{q, k, v, mla::SeqLayout{cu_seqlens}, nullptr, gate, out, B, H, max_seqlen, 0, scale,
                      ws, ws_bytes};
    cudaError_t e = mla::launch_decode(a, pl, false, d, knobs(), take_timer(MLA_OP_DECODE),
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_decode launch");
}

mla_status dsa_sparse_decode(const mla_bf16* q, const mla_bf16* k, const mla_bf16* v,
                             const int64_t* cu_seqlens, const int32_t* topk_idx, int topk,
                             int B, int H, const mla_bf16* gate, mla_bf16* out, float scale,
                             void* ws, size_t ws_bytes, mla_stream stream) {
    mla_status s = check_decode_common(q, k, v, cu_seqlens, gate, out, B, H, topk > 0 ? topk : 1);
    if (s != MLA_OK) return s;
    REQUIRE(topk_idx != nullptr && (reinterpret_cast<uintptr_t>(topk_idx) & 3u) == 0,
            MLA_ERR_INVALID_ARG, "topk_idx must be a 4-byte aligned device pointer");
    REQUIRE(topk >= 1 && topk <= mla::kMaxTopk, MLA_ERR_UNSUPPORTED,
            "topk must be in [1, %d] (got %d)", mla::kMaxTopk, topk);
    REQUIRE(scale > 0.f && scale < 1e30f, MLA_ERR_INVALID_ARG, "scale must be positive finite");
    const mla::DecodePlan pl = mla::plan_decode(B, H, topk, true, g_sparse_chunk.load());
    if ((s = check_ws(ws, ws_bytes, pl.total)) != MLA_OK) return s;
    mla::DeviceInfo d;
    if ((s = device_info(&d)) != MLA_OK) return s;
    mla::DecodeArgs a{q, k, v, mla::SeqLayout{cu_seqlens}, topk_idx, gate, out, B, H, 1 << 30, topk, scale,
                      ws, ws_bytes};
    cudaError_t e = mla::launch_decode(a, pl, true, d, knobs(), take_timer(MLA_OP_SPARSE_DECODE),
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "dsa_sparse_decode launch");
}

mla_status mla_prefill(const mla_bf16* q, const mla_bf16* k, const mla_bf16* v,
                       const mla_bf16* gate, mla_bf16* out, int B, int H, int Tq, int Tk,
                       float scale, void* ws, size_t ws_bytes, mla_stream stream) {
    (void)ws;
    (void)ws_bytes;
    REQUIRE(q && k && v && out, MLA_ERR_INVALID_ARG, "null tensor pointer");
    REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out) &&
                (gate == nullptr || aligned16(gate)),
            MLA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    REQUIRE(B >= 1 && H >= 1 && Tq >= 1 && Tk >= Tq, MLA_ERR_INVALID_ARG,
            "need B >= 1, H >= 1, 1 <= Tq <= Tk (got B=%d H=%d Tq=%d Tk=%d)", B, H, Tq, Tk);
    REQUIRE(int64_t(B) * H * Tk < (int64_t(1) << 31) &&
                int64_t(B) * H * ((Tq + 127) / 128) < (int64_t(1) << 31),
            MLA_ERR_UNSUPPORTED, "B*H*Tk too large for one call");
    REQUIRE(scale > 0.f && scale < 1e30f, MLA_ERR_INVALID_ARG, "scale must be positive finite");
    mla::DeviceInfo d;
    mla_status s = device_info(&d);
    if (s != MLA_OK) return s;
    mla::PrefillArgs a{q, k, v, gate, out, B, H, Tq, Tk, Tk, scale};
    cudaError_t e = mla::launch_prefill(a, d, knobs(), take_timer(MLA_OP_PREFILL),
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_prefill launch");
}

// Host checks of an append of Tn rows per (b, h) into [B,H,cap,D] caches.
static mla_status check_append(const void* kn, const void* vn, const void* kc, const void* vc,
                               const void* start, int B, int H, int Tn, int cap) {
    REQUIRE(kn && vn && kc && vc, MLA_ERR_INVALID_ARG, "null tensor pointer");
    REQUIRE(aligned16(kn) && aligned16(vn) && aligned16(kc) && aligned16(vc) &&
                (reinterpret_cast<uintptr_t>(start) & 7u) == 0,
            MLA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    REQUIRE(B >= 1 && H >= 1 && Tn >= 1 && cap >= 1, MLA_ERR_INVALID_ARG,
            "need B, H, Tn, kv_capacity >= 1 (got %d, %d, %d, %d)", B, H, Tn, cap);
    REQUIRE(int64_t(Tn) * 40 < (int64_t(1) << 31) && int64_t(B) * H < (int64_t(1) << 31),
            MLA_ERR_UNSUPPORTED, "Tn or B*H too large for one call");
    return MLA_OK;
}

static mla_status enqueue_append(const mla_bf16* k_new, const mla_bf16* v_new, mla_bf16* k_cache,
                                 mla_bf16* v_cache, const int64_t* start, int64_t start_all,
                                 int B, int H, int Tn, int cap, const mla::DeviceInfo& d,
                                 cudaStream_t st) {
    mla::AppendArgs a{k_new, v_new, k_cache, v_cache, start, start_all, B, H, Tn, cap};
    cudaError_t e = mla::launch_cache_append(a, d, take_timer(MLA_OP_CACHE_APPEND), st);
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "cache append launch");
}

mla_status mla_cache_append(const mla_bf16* k_new, const mla_bf16* v_new, mla_bf16* k_cache,
                            mla_bf16* v_cache, const int64_t* start, int64_t start_all, int B,
                            int H, int Tn, int kv_capacity, mla_stream stream) {
    mla_status s = check_append(k_new, v_new, k_cache, v_cache, start, B, H, Tn, kv_capacity);
    if (s != MLA_OK) return s;
    REQUIRE(start != nullptr || (start_all >= 0 && start_all + Tn <= kv_capacity),
            MLA_ERR_INVALID_ARG, "start_all + Tn must lie in [0, kv_capacity] (got %lld + %d, %d)",
            static_cast<long long>(start_all), Tn, kv_capacity);
    mla::DeviceInfo d;
    if ((s = device_info(&d)) != MLA_OK) return s;
    return enqueue_append(k_new, v_new, k_cache, v_cache, start, start_all, B, H, Tn, kv_capacity,
                          d, static_cast<cudaStream_t>(stream));
}

mla_status mla_prefill_chunk(const mla_bf16* q, const mla_bf16* k_new, const mla_bf16* v_new,
                             mla_bf16* k_cache, mla_bf16* v_cache, const mla_bf16* gate,
                             mla_bf16* out, int B, int H, int Tq, int P, int kv_capacity,
                             float scale, void* ws, size_t ws_bytes, mla_stream stream) {
    (void)ws;
    (void)ws_bytes;
    mla_status s = check_append(k_new, v_new, k_cache, v_cache, nullptr, B, H, Tq, kv_capacity);
    if (s != MLA_OK) return s;
    REQUIRE(q && out, MLA_ERR_INVALID_ARG, "null tensor pointer");
    REQUIRE(aligned16(q) && aligned16(out) && (gate == nullptr || aligned16(gate)),
            MLA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    REQUIRE(P >= 0 && int64_t(P) + Tq <= kv_capacity, MLA_ERR_INVALID_ARG,
            "need 0 <= P and P + Tq <= kv_capacity (got P=%d Tq=%d capacity=%d)", P, Tq,
            kv_capacity);
    REQUIRE(int64_t(B) * H * ((Tq + 127) / 128) < (int64_t(1) << 31), MLA_ERR_UNSUPPORTED,
            "B*H*Tq too large for one call");
    REQUIRE(scale > 0.f && scale < 1e30f, MLA_ERR_INVALID_ARG, "scale must be positive finite");
    mla::DeviceInfo d;
    if ((s = device_info(&d)) != MLA_OK) return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((s = enqueue_append(k_new, v_new, k_cache, v_cache, nullptr, P, B, H, Tq, kv_capacity, d,
                            st)) != MLA_OK)
        return s;
    mla::PrefillArgs a{q, k_cache, v_cache, gate, out, B, H, Tq, P + Tq, kv_capacity, scale};
    cudaError_t e = mla::launch_prefill(a, d, knobs(), take_timer(MLA_OP_PREFILL), st);
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_prefill_chunk launch");
}

mla_status mla_decode_cached(const mla_bf16* q, const mla_bf16* k_new, const mla_bf16* v_new,
                             mla_bf16* k_cache, mla_bf16* v_cache, const int64_t* cache_seqlens,
                             int B, int H, int kv_capacity, int max_seqlen, const mla_bf16* gate,
                             mla_bf16* out, float scale, void* ws, size_t ws_bytes,
                             mla_stream stream) {
    mla_status s = check_decode_common(q, k_cache, v_cache, cache_seqlens, gate, out, B, H,
                                       max_seqlen);
    if (s != MLA_OK) return s;
    REQUIRE((k_new == nullptr) == (v_new == nullptr), MLA_ERR_INVALID_ARG,
            "k_new and v_new must both be given or both be NULL");
    REQUIRE(max_seqlen <= kv_capacity, MLA_ERR_INVALID_ARG,
            "max_seqlen (%d) exceeds kv_capacity (%d)", max_seqlen, kv_capacity);
    if (k_new) {
        s = check_append(k_new, v_new, k_cache, v_cache, cache_seqlens, B, H, 1, kv_capacity);
        if (s != MLA_OK) return s;
    }
    REQUIRE(scale > 0.f && scale < 1e30f, MLA_ERR_INVALID_ARG, "scale must be positive finite");
    const mla::DecodePlan pl = mla::plan_decode(B, H, max_seqlen, false);
    if ((s = check_ws(ws, ws_bytes, pl.total)) != MLA_OK) return s;
    mla::DeviceInfo d;
    if ((s = device_info(&d)) != MLA_OK) return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (k_new && (s = enqueue_append(k_new, v_new, k_cache, v_cache, cache_seqlens, 0, B, H, 1,
                                     kv_capacity, d, st)) != MLA_OK)
        return s;
    mla::SeqLayout seq;
    seq.lens = cache_seqlens;
    seq.cap = kv_capacity;
    seq.add = k_new ? 1 : 0;
    mla::DecodeArgs a{q, k_cache, v_cache, seq, nullptr, gate, out, B, H, max_seqlen, 0, scale,
                      ws, ws_bytes};
    cudaError_t e = mla::launch_decode(a, pl, false, d, knobs(), take_timer(MLA_OP_DECODE), st);
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_decode_cached launch");
}

// Shared body of the bf16 and FP8 latent decode entry points.
static mla_status latent_decode_common(const mla_bf16* q, const mla_bf16* ckv, const uint8_t* rec,
                                       const int64_t* cu_seqlens, int64_t total_positions, int B,
                                       int H, int max_seqlen, const mla_bf16* w_kc,
                                       const mla_bf16* w_vc, const mla_bf16* gate, mla_bf16* out,
                                       float scale, void* ws, size_t ws_bytes, mla_stream stream) {
    const void* cache = rec ? static_cast<const void*>(rec) : static_cast<const void*>(ckv);
    mla_status s = check_decode_common(q, cache, w_kc, cu_seqlens, gate, out, B, H, max_seqlen);
    if (s != MLA_OK) return s;
    REQUIRE(w_vc != nullptr && aligned16(w_vc), MLA_ERR_INVALID_ARG,
            "w_vc must be a 16-byte aligned device pointer");
    REQUIRE(H >= 16 && H <= 96 && H % 16 == 0, MLA_ERR_UNSUPPORTED,
            "H must be a multiple of 16 in [16, 96] (got %d)", H);
    REQUIRE(total_positions >= 0 && total_positions < (int64_t(1) << 31), MLA_ERR_UNSUPPORTED,
            "total_positions must be in [0, 2^31)");
    REQUIRE(B <= 65535 * 16, MLA_ERR_UNSUPPORTED, "B too large for one call");
    REQUIRE(scale > 0.f && scale < 1e30f, MLA_ERR_INVALID_ARG, "scale must be positive finite");
    mla::DeviceInfo d;
    if ((s = device_info(&d)) != MLA_OK) return s;
    const mla::LatentPlan pl = mla::plan_latent(B, H, d.sms);
    if ((s = check_ws(ws, ws_bytes, pl.total)) != MLA_OK) return s;
    mla::LatentArgs a{q, ckv, cu_seqlens, w_kc, w_vc, gate, out, B, H, max_seqlen,
                      total_positions, scale, ws};
    a.rec = rec;
    cudaError_t e = mla::launch_latent_decode(a, pl, d, knobs(), take_timer(MLA_OP_LATENT_DECODE),
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "latent decode launch");
}

mla_status mla_decode_latent(const mla_bf16* q, const mla_bf16* ckv, const int64_t* cu_seqlens,
                             int64_t total_positions, int B, int H, int max_seqlen,
                             const mla_bf16* w_kc, const mla_bf16* w_vc, const mla_bf16* gate,
                             mla_bf16* out, float scale, void* ws, size_t ws_bytes,
                             mla_stream stream) {
    return latent_decode_common(q, ckv, nullptr, cu_seqlens, total_positions, B, H, max_seqlen,
                                w_kc, w_vc, gate, out, scale, ws, ws_bytes, stream);
}

mla_status mla_decode_latent_fp8(const mla_bf16* q, const uint8_t* rec, const int64_t* cu_seqlens,
                                 int64_t total_positions, int B, int H, int max_seqlen,
                                 const mla_bf16* w_kc, const mla_bf16* w_vc, const mla_bf16* gate,
                                 mla_bf16* out, float scale, void* ws, size_t ws_bytes,
                                 mla_stream stream) {
    REQUIRE(rec != nullptr, MLA_ERR_INVALID_ARG, "null record pointer");
    return latent_decode_common(q, nullptr, rec, cu_seqlens, total_positions, B, H, max_seqlen,
                                w_kc, w_vc, gate, out, scale, ws, ws_bytes, stream);
}

mla_status mla_quantize_latent_cache(const mla_bf16* ckv, uint8_t* rec, int64_t N,
                                     mla_stream stream) {
    REQUIRE(N >= 0, MLA_ERR_INVALID_ARG, "N must be >= 0");
    if (N == 0) return MLA_OK;
    REQUIRE(ckv && rec, MLA_ERR_INVALID_ARG, "null pointer");
    REQUIRE(aligned16(ckv) && aligned16(rec), MLA_ERR_INVALID_ARG, "misaligned pointer");
    REQUIRE(N < (int64_t(1) << 31), MLA_ERR_UNSUPPORTED, "N too large for one call");
    cudaError_t e = mla::launch_quantize_latent(ckv, rec, N, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_quantize_latent_cache launch");
}

static mla_status sparse_prefill_common(const mla_bf16* q, const mla_bf16* ckv, const uint8_t* rec,
                                        const int32_t* topk_idx, int Tq, int Tk, int topk, int H,
                                        const mla_bf16* w_kc, const mla_bf16* w_vc,
                                        const mla_bf16* gate, mla_bf16* out, float scale, void* ws,
                                        size_t ws_bytes, mla_stream stream) {
    const void* cache = rec ? static_cast<const void*>(rec) : static_cast<const void*>(ckv);
    REQUIRE(q && cache && topk_idx && w_kc && w_vc && out, MLA_ERR_INVALID_ARG, "null pointer");
    REQUIRE(aligned16(q) && aligned16(cache) && aligned16(w_kc) && aligned16(w_vc) &&
                aligned16(out) && (gate == nullptr || aligned16(gate)) &&
                (reinterpret_cast<uintptr_t>(topk_idx) & 3u) == 0,
            MLA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    REQUIRE(H >= 16 && H <= 96 && H % 16 == 0, MLA_ERR_UNSUPPORTED,
            "H must be a multiple of 16 in [16, 96] (got %d)", H);
    REQUIRE(topk >= 1 && topk <= mla::kMaxTopk, MLA_ERR_UNSUPPORTED,
            "topk must be in [1, %d] (got %d)", mla::kMaxTopk, topk);
    REQUIRE(Tq >= 1 && Tk >= Tq, MLA_ERR_INVALID_ARG, "need 1 <= Tq <= Tk (got Tq=%d Tk=%d)",
            Tq, Tk);
    REQUIRE(int64_t(Tq) * H < (int64_t(1) << 31) && Tq <= 65535 * 128, MLA_ERR_UNSUPPORTED,
            "Tq too large for one call");
    REQUIRE(scale > 0.f && scale < 1e30f, MLA_ERR_INVALID_ARG, "scale must be positive finite");
    mla::DeviceInfo d;
    mla_status s = device_info(&d);
    if (s != MLA_OK) return s;
    const mla::LatentPlan pl = mla::plan_latent(Tq, H, d.sms);
    if ((s = check_ws(ws, ws_bytes, pl.total)) != MLA_OK) return s;
    mla::LatentArgs a{q, ckv, nullptr, w_kc, w_vc, gate, out, Tq, H, Tk, Tk, scale, ws};
    a.idx = topk_idx;
    a.topk = topk;
    a.P = Tk - Tq;
    a.rec = rec;
    cudaError_t e = mla::launch_latent_decode(a, pl, d, knobs(), take_timer(MLA_OP_LATENT_DECODE),
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "mla_sparse_prefill_latent launch");
}

mla_status dsa_prefill_index_topk(const mla_bf16* index_q, const mla_bf16* index_k,
                                  const float* w, int Tq, int Tk, int NH, int topk,
                                  int32_t* topk_idx, float* topk_scores, void* ws,
                                  size_t ws_bytes, mla_stream stream) {
    REQUIRE(index_q && index_k && w && topk_idx, MLA_ERR_INVALID_ARG, "null pointer");
    REQUIRE(aligned16(index_q) && aligned16(index_k), MLA_ERR_INVALID_ARG,
            "index_q and index_k must be 16-byte aligned");
    REQUIRE((reinterpret_cast<uintptr_t>(w) & 3u) == 0 &&
                (reinterpret_cast<uintptr_t>(topk_idx) & 3u) == 0 &&
                (reinterpret_cast<uintptr_t>(topk_scores) & 3u) == 0,
            MLA_ERR_INVALID_ARG, "misaligned w or outputs");
    REQUIRE(NH == mla::kIndexHeads, MLA_ERR_UNSUPPORTED, "NH must be 32 (got %d)", NH);
    REQUIRE(topk >= 1 && topk <= mla::kMaxTopk, MLA_ERR_UNSUPPORTED,
            "topk must be in [1, %d] (got %d)", mla::kMaxTopk, topk);
    REQUIRE(Tq >= 1 && Tk >= Tq && Tk < (1 << 24), MLA_ERR_INVALID_ARG,
            "need 1 <= Tq <= Tk < 2^24 (got Tq=%d Tk=%d)", Tq, Tk);
    REQUIRE(int64_t(Tq) * mla::kIndexHeads < (int64_t(1) << 31), MLA_ERR_UNSUPPORTED,
            "Tq too large for one call");
    mla_status s = check_ws(ws, ws_bytes, mla::prefill_index_ws(Tq, Tk));
    if (s != MLA_OK) return s;
    mla::DeviceInfo d;
    if ((s = device_info(&d)) != MLA_OK) return s;
    mla::PrefillIndexArgs a{index_q, index_k, w, Tq, Tk, topk, topk_idx, topk_scores, ws};
    cudaError_t e = mla::launch_prefill_index_topk(a, d, knobs(),
                                                   take_timer(MLA_OP_PREFILL_INDEX_TOPK),
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "dsa_prefill_index_topk launch");
}

mla_status dsa_quantize_index_keys(const mla_bf16* index_k, uint8_t* k8, float* kscale, int64_t N,
                                   mla_stream stream) {
    REQUIRE(N >= 0, MLA_ERR_INVALID_ARG, "N must be >= 0");
    if (N == 0) return MLA_OK;
    REQUIRE(index_k && k8 && kscale, MLA_ERR_INVALID_ARG, "null pointer");
    REQUIRE(aligned16(index_k) && aligned16(k8) && (reinterpret_cast<uintptr_t>(kscale) & 3u) == 0,
            MLA_ERR_INVALID_ARG, "misaligned pointer");
    REQUIRE(N < (int64_t(1) << 34), MLA_ERR_UNSUPPORTED, "N too large for one call");
    cudaError_t e = mla::launch_quantize_rows_e4m3(index_k, k8, kscale, N, mla::kIndexDim,
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "dsa_quantize_index_keys launch");
}

mla_status dsa_index_topk_fp8(const mla_bf16* index_q, const uint8_t* k8, const float* kscale,
                              const float* w, const int64_t* cu_seqlens, int B, int NH,
                              int64_t total_keys, int max_seqlen, int topk, int32_t* topk_idx,
                              float* topk_scores, void* ws, size_t ws_bytes, mla_stream stream) {
    REQUIRE(index_q && k8 && kscale && w && cu_seqlens && topk_idx, MLA_ERR_INVALID_ARG,
            "null pointer");
    REQUIRE(aligned16(index_q) && aligned16(k8), MLA_ERR_INVALID_ARG,
            "index_q and k8 must be 16-byte aligned");
    REQUIRE((reinterpret_cast<uintptr_t>(w) & 3u) == 0 &&
                (reinterpret_cast<uintptr_t>(kscale) & 3u) == 0 &&
                (reinterpret_cast<uintptr_t>(topk_idx) & 3u) == 0 &&
                (reinterpret_cast<uintptr_t>(topk_scores) & 3u) == 0 &&
                (reinterpret_cast<uintptr_t>(cu_seqlens) & 7u) == 0,
            MLA_ERR_INVALID_ARG, "misaligned w, kscale, cu_seqlens or outputs");
    REQUIRE(NH == mla::kIndexHeads, MLA_ERR_UNSUPPORTED, "NH must be 32 (got %d)", NH);
    REQUIRE(topk >= 1 && topk <= mla::kMaxTopk, MLA_ERR_UNSUPPORTED,
            "topk must be in [1, %d] (got %d)", mla::kMaxTopk, topk);
    REQUIRE(B >= 1 && B <= 65535, MLA_ERR_INVALID_ARG, "B must be in [1, 65535]");
    REQUIRE(max_seqlen >= 1 && max_seqlen <= (1 << 24), MLA_ERR_UNSUPPORTED,
            "max_seqlen must be in [1, 2^24]");
    REQUIRE(total_keys >= 0 && total_keys < (int64_t(1) << 31), MLA_ERR_UNSUPPORTED,
            "total_keys must be in [0, 2^31)");
    const mla::IndexPlan pl = mla::plan_index(B, max_seqlen, true);
    mla_status s = check_ws(ws, ws_bytes, pl.total);
    if (s != MLA_OK) return s;
    mla::DeviceInfo d;
    if ((s = device_info(&d)) != MLA_OK) return s;
    mla::IndexArgs a{index_q, nullptr, w, cu_seqlens, B, max_seqlen, topk, total_keys,
                     topk_idx, topk_scores, ws};
    mla::IndexFp8Args f{k8, kscale};
    cudaError_t e = mla::launch_index_topk_fp8(a, f, pl, d, knobs(),
                                               take_timer(MLA_OP_INDEX_TOPK_FP8),
                                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "dsa_index_topk_fp8 launch");
}

mla_status mla_sparse_prefill_latent(const mla_bf16* q, const mla_bf16* ckv,
                                     const int32_t* topk_idx, int Tq, int Tk, int topk, int H,
                                     const mla_bf16* w_kc, const mla_bf16* w_vc,
                                     const mla_bf16* gate, mla_bf16* out, float scale, void* ws,
                                     size_t ws_bytes, mla_stream stream) {
    return sparse_prefill_common(q, ckv, nullptr, topk_idx, Tq, Tk, topk, H, w_kc, w_vc, gate, out,
                                 scale, ws, ws_bytes, stream);
}

mla_status mla_sparse_prefill_latent_fp8(const mla_bf16* q, const uint8_t* rec,
                                         const int32_t* topk_idx, int Tq, int Tk, int topk, int H,
                                         const mla_bf16* w_kc, const mla_bf16* w_vc,
                                         const mla_bf16* gate, mla_bf16* out, float scale,
                                         void* ws, size_t ws_bytes, mla_stream stream) {
    REQUIRE(rec != nullptr, MLA_ERR_INVALID_ARG, "null record pointer");
    return sparse_prefill_common(q, nullptr, rec, topk_idx, Tq, Tk, topk, H, w_kc, w_vc, gate, out,
                                 scale, ws, ws_bytes, stream);
}

mla_status dsa_index_topk(const mla_bf16* index_q, const mla_bf16* index_k, const float* w,
                          const int64_t* cu_seqlens, int B, int NH, int64_t total_keys,
                          int max_seqlen, int topk, int32_t* topk_idx, float* topk_scores,
                          void* ws, size_t ws_bytes, mla_stream stream) {
    REQUIRE(index_q && index_k && w && cu_seqlens && topk_idx, MLA_ERR_INVALID_ARG,
            "null pointer");
    REQUIRE(aligned16(index_q) && aligned16(index_k), MLA_ERR_INVALID_ARG,
            "index_q and index_k must be 16-byte aligned");
    REQUIRE((reinterpret_cast<uintptr_t>(w) & 3u) == 0 &&
                (reinterpret_cast<uintptr_t>(topk_idx) & 3u) == 0 &&
                (reinterpret_cast<uintptr_t>(topk_scores) & 3u) == 0 &&
                (reinterpret_cast<uintptr_t>(cu_seqlens) & 7u) == 0,
            MLA_ERR_INVALID_ARG, "misaligned w, cu_seqlens or outputs");
    REQUIRE(NH == mla::kIndexHeads, MLA_ERR_UNSUPPORTED, "NH must be 32 (got %d)", NH);
    REQUIRE(topk >= 1 && topk <= mla::kMaxTopk, MLA_ERR_UNSUPPORTED,
            "topk must be in [1, %d] (got %d)", mla::kMaxTopk, topk);
    REQUIRE(B >= 1 && B <= 65535, MLA_ERR_INVALID_ARG, "B must be in [1, 65535]");
    REQUIRE(max_seqlen >= 1 && max_seqlen <= (1 << 24), MLA_ERR_UNSUPPORTED,
            "max_seqlen must be in [1, 2^24]");
    REQUIRE(total_keys >= 0 && total_keys < (int64_t(1) << 31), MLA_ERR_UNSUPPORTED,
            "total_keys must be in [0, 2^31)");
    const mla::IndexPlan pl = mla::plan_index(B, max_seqlen);
    mla_status s = check_ws(ws, ws_bytes, pl.total);
    if (s != MLA_OK) return s;
    mla::DeviceInfo d;
    if ((s = device_info(&d)) != MLA_OK) return s;
    mla::IndexArgs a{index_q, index_k, w, cu_seqlens, B, max_seqlen, topk, total_keys,
                     topk_idx, topk_scores, ws};
    cudaError_t e = mla::launch_index_topk(a, pl, d, knobs(), take_timer(MLA_OP_INDEX_TOPK),
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "dsa_index_topk launch");
}

}  // extern "C"

// ---- helpers shared with other entry-point files (see abi_util.h) ----
#include "abi_util.h"

namespace mla {

mla_status set_error(mla_status s, const char* msg) { return fail(s, "%s", msg); }

mla_status current_device(DeviceInfo* out) { return device_info(out); }

Knobs current_knobs() { return knobs(); }

mla_status check_decode_args(const void* q, const void* k, const void* v, const void* cu,
                             const void* gate, const void* out, int B, int H, int max_len,
                             float scale) {
    mla_status s = check_decode_common(q, k, v, cu, gate, out, B, H, max_len);
    if (s != MLA_OK) return s;
    REQUIRE(scale > 0.f && scale < 1e30f, MLA_ERR_INVALID_ARG, "scale must be positive finite");
    return MLA_OK;
}

}  // namespace mla

extern "C" int mla_gather_probe_blocks(void) {
    mla::DeviceInfo d;
    return device_info(&d) == MLA_OK ? mla::gather_probe_blocks(d) : 0;
}

extern "C" mla_status mla_gather_probe(const mla_bf16* k, const mla_bf16* v,
                                       const int64_t* cu_seqlens, const int32_t* topk_idx,
                                       int topk, int B, int H, uint32_t* sink,
                                       mla_stream stream) {
    REQUIRE(k && v && cu_seqlens && topk_idx && sink, MLA_ERR_INVALID_ARG, "null pointer");
    REQUIRE(aligned16(k) && aligned16(v), MLA_ERR_INVALID_ARG,
            "cache pointers must be 16-byte aligned");
    REQUIRE(B >= 1 && H >= 1 && topk >= 1 && topk <= mla::kMaxTopk, MLA_ERR_INVALID_ARG,
            "need B >= 1, H >= 1, 1 <= topk <= %d", mla::kMaxTopk);
    mla::DeviceInfo d;
    mla_status s = device_info(&d);
    if (s != MLA_OK) return s;
    cudaError_t e = mla::launch_gather_probe(k, v, cu_seqlens, topk_idx, topk, B, H, sink, d,
                                             take_timer(MLA_OP_GATHER_PROBE),
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "gather probe launch");
}
