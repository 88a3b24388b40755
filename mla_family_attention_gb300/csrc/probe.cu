// Measurement aid: a plain gather of the rows the sparse decode reads.
//
// dsa_sparse_decode reads, for every sequence b, head h and selection entry
// e, a 384-byte key row and a 256-byte value row at a position the top-k
// chose, scattered over that head's cache region.  This kernel reads exactly
// those rows with plain 16-byte loads and no arithmetic but an XOR of the
// words (so no load is dead), giving an achievable gather rate against
// which the sparse decode's rate is judged.  Work is ordered like the sparse
// decode's (sequence, head, entry), so concurrent blocks gather from the same
// few heads' regions.
#include <cuda_runtime.h>

#define MLA_FILE_ID 6   // site ids of the bounds-checked debug build
#include "common.cuh"
#include "kernels.h"

namespace mla {
namespace {

constexpr int kChunks = (kDqk + kDv) * 2 / 16;   // 40 16-byte chunks per (key, value) pair
constexpr int kRowsPerPass = 8;                   // entries a block covers in one pass
constexpr int kPasses = 4;                        // loads in flight per thread
constexpr int kProbeThreads = kRowsPerPass * kChunks;              // 320
constexpr int kEntriesPerBlock = kRowsPerPass * kPasses;           // 32

// Block = (sequence b, head h, 32 consecutive selection entries); thread
// (entry lane e, chunk c) reads chunk c of the (key, value) pair of entries
// e, e+8, e+16, e+24: four independent 16-byte loads per thread, every
// 40-thread group covering one row pair with consecutive chunks.
__global__ void __launch_bounds__(kProbeThreads) gather_probe_kernel(
    const uint4* k, const uint4* v, const int64_t* cu, const int32_t* idx, int topk, int B,
    int H, int groups, uint32_t* sink) {
    const int c = threadIdx.x % kChunks, el = threadIdx.x / kChunks;
    uint32_t x = 0;
    for (int64_t blk = blockIdx.x; blk < int64_t(B) * H * groups; blk += gridDim.x) {
        const int g = int(blk % groups);
        const int64_t bh = blk / groups;
        const int h = int(bh % H), b = int(bh / H);
        const int64_t T = cu[b + 1] - cu[b];
        const int64_t base = cu[b] * H + int64_t(h) * T;
        uint4 r[kPasses];
#pragma unroll
        for (int q = 0; q < kPasses; ++q) {
            const int e = g * kEntriesPerBlock + el + kRowsPerPass * q;
            const int s = e < topk ? idx[int64_t(b) * topk + e] : -1;
            r[q] = make_uint4(0, 0, 0, 0);
            if (s >= 0 && s < T) {
                const int64_t row = base + s;
                r[q] = c < 24 ? __ldcs(k + row * 24 + c) : __ldcs(v + row * 16 + (c - 24));
            }
        }
#pragma unroll
        for (int q = 0; q < kPasses; ++q) x ^= r[q].x ^ r[q].y ^ r[q].z ^ r[q].w;
    }
    __shared__ uint32_t wx[kProbeThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, o);
    if ((threadIdx.x & 31) == 0) wx[threadIdx.x >> 5] = x;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int w = 0; w < kProbeThreads / 32; ++w) t ^= wx[w];
        sink[blockIdx.x] = t;
    }
}

}  // namespace

int gather_probe_blocks(const DeviceInfo& dev) { return dev.sms * 6; }

cudaError_t launch_gather_probe(const uint16_t* k, const uint16_t* v, const int64_t* cu,
                                const int32_t* idx, int topk, int B, int H, uint32_t* sink,
                                const DeviceInfo& dev, const KernelTimer& tm, cudaStream_t st) {
    if (tm.begin) cudaEventRecord(tm.begin, st);
    const int groups = (topk + kEntriesPerBlock - 1) / kEntriesPerBlock;
    gather_probe_kernel<<<gather_probe_blocks(dev), kProbeThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v), cu, idx, topk, B,
        H, groups, sink);
    if (tm.end) cudaEventRecord(tm.end, st);
    return cudaGetLastError();
}

}  // namespace mla
