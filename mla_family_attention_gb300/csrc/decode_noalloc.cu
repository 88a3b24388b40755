// Gated MLA decode for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory for a workspace: a plugin
// running inside a host runtime that owns every device allocation, or a
// latency-critical loop that must not call cudaMalloc because it implicitly
// synchronises the device.  mla_decode_noalloc serves them: it runs the same
// split-KV decode kernels as mla_decode, but takes its scratch (the chunk
// partials and the work-item table) from a fixed-size array compiled into
// this library instead of a caller workspace.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds its MLA_NOALLOC_SCRATCH_BYTES until the process exits.  Host
// code cannot use the variable's name as a device address; the first call
// on each device (with that device current) looks the address up with
// cudaGetSymbolAddress and caches it with the id of the context it belongs
// to.  After a device reset the device has a new context, in which the
// array lives elsewhere, so the next call looks the address up again.
//
// Every call shares the one array, and it keeps the previous call's
// contents.  Nothing in it has to start at zero: the decode kernels write
// every partial and table entry they later read.  Calls whose kernels
// overlap on the GPU (different streams, or different host threads without
// ordering) race on the array.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "abi_util.h"
#include "kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDev];
unsigned long long g_scratch_ctx[kMaxDev];

// Device address of the scratch array on the current device (set up once
// per context of the device).
mla_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return mla::set_error(MLA_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDev) return mla::set_error(MLA_ERR_UNSUPPORTED, "device ordinal");
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    const unsigned long long ctx = mla::current_context_id();
    if (g_scratch_ptr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return mla::set_error(MLA_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed");
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = mla::current_context_id();
    }
    *out = g_scratch_ptr[dev];
    return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_decode_noalloc(const mla_bf16* q, const mla_bf16* k,
                                         const mla_bf16* v, const int64_t* cu_seqlens, int B,
                                         int H, int max_seqlen, const mla_bf16* gate,
                                         mla_bf16* out, float scale, mla_stream stream) {
    mla_status s = mla::check_decode_args(q, k, v, cu_seqlens, gate, out, B, H, max_seqlen,
                                          scale);
    if (s != MLA_OK) return s;
    const mla::DecodePlan pl = mla::plan_decode(B, H, max_seqlen, false);
    if (pl.total > MLA_NOALLOC_SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "mla_decode_noalloc needs %zu bytes of scratch for B=%d H=%d max_seqlen=%d; "
                 "the built-in scratch holds %zu bytes",
                 pl.total, B, H, max_seqlen, static_cast<size_t>(MLA_NOALLOC_SCRATCH_BYTES));
        return mla::set_error(MLA_ERR_WORKSPACE, msg);
    }
    mla::DeviceInfo d;
    if ((s = mla::current_device(&d)) != MLA_OK) return s;
    void* scratch = nullptr;
    if ((s = scratch_address(&scratch)) != MLA_OK) return s;
    mla::DecodeArgs a{q, k, v, mla::SeqLayout{cu_seqlens}, nullptr, gate, out, B, H, max_seqlen, 0, scale,
                      scratch, MLA_NOALLOC_SCRATCH_BYTES};
    cudaError_t e = mla::launch_decode(a, pl, false, d, mla::current_knobs(), mla::KernelTimer{},
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : mla::set_error(MLA_ERR_CUDA, cudaGetErrorString(e));
}
