// Device helpers shared by the library's kernels: mbarrier pipelines with
// bounded waits, bulk (TMA) copies, bf16 unpacking and the device status word.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

// Device status codes (the same values as mla_status in include/mla.h).
enum : int { kStInvalid = 1, kStTimeout = 5, kStBadIndex = 6, kStCheck = 7 };

// First error wins; later ones are dropped until the host clears the word.
__device__ __forceinline__ void report(int* status, int code) { atomicCAS(status, 0, code); }

// Bounds-checked debug build.  Compiled with -DMLA_CHECKS, MLA_CHECK(cond,
// status) tests a kernel's own index arithmetic (ring slots, TMEM columns,
// swizzled shared-memory offsets, histogram bins, output positions) and, when
// the condition fails, records MLA_ERR_CHECK in the status word and the site
// (file id * 100000 + line) in the word after it; nothing traps.  Without
// MLA_CHECKS the macro compiles to nothing.  Each kernel file defines
// MLA_FILE_ID before including this header.
#ifndef MLA_FILE_ID
#define MLA_FILE_ID 0
#endif
__device__ __forceinline__ void check_failed(int* status, int site) {
    if (atomicCAS(status, 0, kStCheck) == 0) atomicExch(status + 1, site);
}
#ifdef MLA_CHECKS
#define MLA_CHECK(cond, status)                                                   \
    do {                                                                          \
        if (!(cond)) ::mla::check_failed((status), MLA_FILE_ID * 100000 + __LINE__); \
    } while (0)
#else
#define MLA_CHECK(cond, status) \
    do {                        \
    } while (0)
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// True once the phase with the given parity has completed.  try_wait may
// suspend the thread for a hardware-defined interval, so a loop over it does
// not spin hot.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait: false when `limit_ns` elapsed before the phase completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit_ns) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_test(bar, parity)) {
        if (static_cast<long long>(global_ns() - t0) > limit_ns) return false;
    }
    return true;
}

// The same wait by every lane of a converged warp (the MMA-issuing and TMA
// roles run as whole warps); the result is the same in every lane.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, long long limit_ns) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit_ns));
}

// A whole-warp wait that gives up at once when another role has set *abort
// after a failure of its own.
__device__ __forceinline__ bool warp_wait_abortable(uint64_t* bar, uint32_t parity,
                                                    long long limit_ns, volatile int* abort) {
    const bool ok = mbar_test(bar, parity) || (!*abort && mbar_wait(bar, parity, limit_ns));
    return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// Bulk copies (TMA, non-tensor): global -> shared, completion counted in bytes
// on an mbarrier.  Both addresses 16-byte aligned, size a multiple of 16.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------------------
// Arithmetic helpers
// ---------------------------------------------------------------------------
// bf16 pair packed in a 32-bit word -> the two fp32 values (exact).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 2^x on the special-function unit; 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// tanh on the special-function unit (relative error about 2^-11).
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// sigmoid(g) = (1 + tanh(g/2)) / 2: one special-function operation and an
// FMA, instead of an exponential and an IEEE division (whose ~20
// instructions dominated the gate epilogues).  The error, below 2^-11 of
// the gate, is well under the bf16 output step (2^-8 relative).
__device__ __forceinline__ float sigmoidf_fast(float g) {
    return fmaf(0.5f, tanh_approx(0.5f * g), 0.5f);
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 16-byte global -> shared copy through L2 (bypassing L1).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
                 : "memory");
}

// One arrival on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic
// stream serialization may start while the previous kernel of the stream
// finishes; grid_dep_wait blocks until that grid has completed and its
// writes are visible (a no-op under a normal launch), so it precedes every
// read of the previous kernel's results.  grid_dep_trigger, issued once a
// CTA's work is done, lets the next kernel start launching early; its own
// grid_dep_wait still waits for this grid to complete.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace mla
