// K3.1 Gated DSA indexer score and top-k for sm_103a.
//
// What it computes (K3.1 Gated DSA post, eqs. (5) and (6)):
//   score[b,s] = sum_{h<32} w[b,h] * max(0, q^I[b,h] . k^I[b,s])   for s < T_b
//   S_b        = the min(topk, T_b) positions of largest score, ranked by
//                (score descending, position ascending), returned ascending
// with the eq. (5) constant already folded into w by the caller.  When
// T_b <= topk every position is kept and no score is computed (the post's
// short-context shortcut).
//
// Scoring (dsa_score_kernel).  The index keys are read once from HBM: 256 B
// per position, against 2*32*128 = 8,192 flops per position (32 flop/B), so
// on CUDA cores the kernel would be ALU bound well below HBM speed; the
// 32-head dot products therefore run on the tensor cores as one
// M=128 (positions) x N=32 (index heads) x K=128 tcgen05.mma tile per 128
// positions, accumulating in TMEM:
//   warp 0  TMA producer: 128 key rows (two 64-feature swizzled boxes) and the
//           sequence's 32 index queries into a 4-stage shared-memory ring;
//   warp 1  allocates 64 TMEM columns (two 32-column accumulators) and one
//           lane issues the eight K=16 MMAs per tile, committing to mbarriers;
//   warps 2-5 read the accumulator (thread = position, 32 columns = heads),
//           apply ReLU and the head weights, write the fp32 score and count it
//           in a 2048-bin histogram of its top 11 order-preserving key bits.
// Tiles are assigned to CTAs in contiguous ranges so the histogram of one
// sequence is flushed to global memory a few times, not per tile.
//
// Top-k (dsa_topk_kernel, one CTA per sequence).  An exact radix select on
// order-preserving 32-bit keys: the first 11 bits come from the histogram the
// scoring pass built, two more passes over the (L2-resident) scores find the
// next 11 and the last 10 bits of the k-th key, and a final pass in position
// order keeps every key above it plus the lowest positions among keys equal
// to it, writing the output in ascending position order directly.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kTile = 128;                                   // positions per MMA tile
constexpr int kIStages = 4;
constexpr int kAHalf = kTile * 64 * 2;                       // 16 KB: 128 rows x 128 B
constexpr int kBHalf = kIndexHeads * 64 * 2;                 // 4 KB: 32 rows x 128 B
constexpr int kStageBytes = 2 * kAHalf + 2 * kBHalf;         // 40 KB
constexpr int kBins = 2048;
constexpr int kScoreThreads = 6 * 32;
constexpr uint32_t kTmemCols = 64;
constexpr size_t kScoreSmem = 1024 + size_t(kIStages) * kStageBytes + kBins * 4 + 256;
constexpr uint32_t kIdesc = idesc_bf16_f32(128, kIndexHeads, false, false);

struct ScoreParams {
    const float* w;
    const int64_t* cu;
    const int* tile_start;   // [B+1]
    float* scores;           // [B][max_seqlen]
    unsigned* hist;          // [B][2048]
    int B, max_seqlen;
    long long wait_ns;
    int* status;
};

__device__ __forceinline__ uint32_t okey(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int tile_owner(const int* tile_start, int B, int t) {
    int lo = 0, hi = B;   // largest b with tile_start[b] <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tile_start[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kScoreThreads, 1)
    dsa_score_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap qmap, const ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned* hist = reinterpret_cast<unsigned*>(smem + kIStages * kStageBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(hist + kBins);
    uint64_t* empty = full + kIStages;
    uint64_t* tfull = empty + kIStages;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = p.tile_start[p.B];
    const int t_begin = int((int64_t(n_tiles) * blockIdx.x) / gridDim.x);
    const int t_end = int((int64_t(n_tiles) * (blockIdx.x + 1)) / gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kIStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0;
    if (warp == 1) tmem_alloc(tmem_holder, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&qmap);
            const uint64_t stream_policy = l2_evict_first_policy();
            int filled[kIStages] = {0, 0, 0, 0};
            for (int t = t_begin, j = 0; t < t_end; ++t, ++j) {
                const int slot = j % kIStages, round = j / kIStages;
                if (*abort_flag) break;
                if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, p.wait_ns)) {
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                    break;
                }
                const int b = tile_owner(p.tile_start, p.B, t);
                const int row = int(p.cu[b]) + (t - p.tile_start[b]) * kTile;
                uint8_t* st = smem + slot * kStageBytes;
                mbar_arrive_expect_tx(&full[slot], kStageBytes);
                tma_load_2d_hint(st, &kmap, 0, row, &full[slot], stream_policy);
                tma_load_2d_hint(st + kAHalf, &kmap, 64, row, &full[slot], stream_policy);
                tma_load_2d(st + 2 * kAHalf, &qmap, 0, b * kIndexHeads, &full[slot]);
                tma_load_2d(st + 2 * kAHalf + kBHalf, &qmap, 64, b * kIndexHeads, &full[slot]);
                filled[slot] = round + 1;
            }
            for (int s = 0; s < kIStages; ++s)
                if (filled[s] > 0 && !mbar_wait(&full[s], (filled[s] - 1) & 1, p.wait_ns))
                    report(p.status, kStTimeout);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer -------------------------------
        if (lane == 0) {
            int last_acc = -1, last_phase = 0;
            for (int t = t_begin, j = 0; t < t_end; ++t, ++j) {
                const int slot = j % kIStages, acc = j & 1;
                if (*abort_flag) break;
                if (!mbar_wait(&full[slot], (j / kIStages) & 1, p.wait_ns) ||
                    (j >= 2 && !mbar_wait(&tempty[acc], ((j >> 1) - 1) & 1, p.wait_ns))) {
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(smem + slot * kStageBytes);
                const uint32_t b0 = a0 + 2 * kAHalf;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = smem_desc_sw128(a0 + (kk >> 2) * kAHalf + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(b0 + (kk >> 2) * kBHalf + (kk & 3) * 32, 16, 1024);
                    mma_bf16_ss(tmem + acc * 32, ad, bd, kIdesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(&empty[slot]);
                mma_commit(&tfull[acc]);
                last_acc = acc;
                last_phase = (j >> 1) & 1;
            }
            // the accumulator must not be released while an MMA still writes it
            if (last_acc >= 0 && !mbar_wait(&tfull[last_acc], last_phase, p.wait_ns))
                report(p.status, kStTimeout);
        }
    } else {
        // ------------------------------- epilogue --------------------------------
        const int quad = warp & 3;                 // TMEM lanes 32*quad .. 32*quad+31
        const int r = quad * 32 + lane;            // position within the tile
        int cur_b = -1;
        for (int t = t_begin, j = 0; t < t_end; ++t, ++j) {
            const int acc = j & 1;
            const int b = tile_owner(p.tile_start, p.B, t);
            if (b != cur_b) {
                if (cur_b >= 0) {                  // flush the previous sequence's bins
                    named_bar_sync(1, 128);
                    for (int i = threadIdx.x - 64; i < kBins; i += 128) {
                        const unsigned c = hist[i];
                        if (c) {
                            atomicAdd(&p.hist[size_t(cur_b) * kBins + i], c);
                            hist[i] = 0;
                        }
                    }
                    named_bar_sync(1, 128);
                }
                cur_b = b;
            }
            // After a timeout every warp keeps walking the tile list without
            // touching TMEM, so all four warps meet the same named barriers.
            bool ok = !*abort_flag;
            if (ok && !mbar_wait(&tfull[acc], (j >> 1) & 1, p.wait_ns)) {
                report(p.status, kStTimeout);
                *abort_flag = 1;
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) continue;
            tc_fence_after();
            float d[32];
            tmem_ld32(tmem + (uint32_t(quad * 32) << 16) + acc * 32, d);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);

            const float* wb = p.w + size_t(b) * kIndexHeads;
            float s = 0.f;
#pragma unroll
            for (int h = 0; h < kIndexHeads; ++h) s = fmaf(__ldg(wb + h), fmaxf(d[h], 0.f), s);
            s += 0.0f;                             // -0 -> +0: equal scores compare equal
            const int64_t T = p.cu[b + 1] - p.cu[b];
            const int pos = (t - p.tile_start[b]) * kTile + r;
            if (pos < T) {
                p.scores[size_t(b) * p.max_seqlen + pos] = s;
                atomicAdd(&hist[okey(s) >> 21], 1u);
            }
        }
        named_bar_sync(1, 128);
        if (cur_b >= 0) {
            for (int i = threadIdx.x - 64; i < kBins; i += 128) {
                const unsigned c = hist[i];
                if (c) atomicAdd(&p.hist[size_t(cur_b) * kBins + i], c);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Tiles per sequence: ceil(T_b/128) when T_b > topk, 0 when every position
// is kept anyway.  Sequences outside [0, max_seqlen] or past total_keys are
// reported and get no tiles.
__global__ void __launch_bounds__(1024) dsa_tiles_kernel(const int64_t* cu, int B, int max_seqlen,
                                                         int64_t total_keys, int topk,
                                                         int* tile_start, int* status) {
    __shared__ int warp_sums[32];
    const int per = (B + blockDim.x - 1) / blockDim.x;
    const int b0 = min(B, int(threadIdx.x) * per), b1 = min(B, b0 + per);
    auto tiles_of = [&](int b) -> int {
        const int64_t T = cu[b + 1] - cu[b];
        if (T < 0 || T > max_seqlen || cu[b] < 0 || cu[b + 1] > total_keys) {
            report(status, kStInvalid);
            return 0;
        }
        return T > topk ? int((T + kTile - 1) / kTile) : 0;
    };
    int local = 0;
    for (int b = b0; b < b1; ++b) local += tiles_of(b);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < int(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        warp_sums[lane] = v;
    }
    __syncthreads();
    int run = incl - local + (warp > 0 ? warp_sums[warp - 1] : 0);
    for (int b = b0; b < b1; ++b) {
        tile_start[b] = run;
        const int64_t T = cu[b + 1] - cu[b];
        if (!(T < 0 || T > max_seqlen || cu[b] < 0 || cu[b + 1] > total_keys))
            run += T > topk ? int((T + kTile - 1) / kTile) : 0;
    }
    if (threadIdx.x == blockDim.x - 1) tile_start[B] = run;
}

// Block-wide exclusive prefix sum over 1024 threads; *total gets the sum.
__device__ __forceinline__ int block_excl_scan(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int x = sh[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        sh[lane] = x;
    }
    __syncthreads();
    const int r = incl - v + (warp > 0 ? sh[warp - 1] : 0);
    *total = sh[31];
    __syncthreads();
    return r;
}

// Bin holding the K-th largest key given a histogram (bins ordered by key):
// count(bins above) < K <= count(bins at or above).
__device__ __forceinline__ void find_bin(const unsigned* hist, int nbins, int K, int* sh,
                                         int* out_bin, int* out_above) {
    const int per = nbins / 1024;                  // 1 or 2 bins per thread
    const int hi = nbins - 1 - int(threadIdx.x) * per;
    int local = 0;
    for (int i = 0; i < per; ++i) local += int(hist[hi - i]);
    int total;
    const int above = block_excl_scan(local, sh, &total);
    if (above < K && K <= above + local) {
        int cum = above;
        for (int i = 0; i < per; ++i) {
            const int c = int(hist[hi - i]);
            if (cum + c >= K) {
                sh[32] = hi - i;
                sh[33] = cum;
                break;
            }
            cum += c;
        }
    }
    __syncthreads();
    *out_bin = sh[32];
    *out_above = sh[33];
    __syncthreads();
}

constexpr int kSelPer = 16;                        // positions per thread per collect tile

__global__ void __launch_bounds__(1024) dsa_topk_kernel(const float* scores, const unsigned* ghist,
                                                        const int64_t* cu, int max_seqlen,
                                                        int64_t total_keys, int topk,
                                                        int32_t* out_idx, float* out_scores,
                                                        int* status) {
    __shared__ unsigned hist[kBins];
    __shared__ int sh[40];
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    int32_t* oi = out_idx + size_t(b) * topk;
    float* os = out_scores ? out_scores + size_t(b) * topk : nullptr;
    const int64_t T64 = cu[b + 1] - cu[b];
    const bool valid = !(T64 < 0 || T64 > max_seqlen || cu[b] < 0 || cu[b + 1] > total_keys);
    const int T = valid ? int(T64) : 0;
    const float* s = scores + size_t(b) * max_seqlen;
    if (T <= topk) {                               // every position is kept
        for (int i = tid; i < topk; i += blockDim.x) {
            oi[i] = i < T ? i : -1;
            if (os) os[i] = -INFINITY;
        }
        return;
    }
    const int K = topk;
    // ---- level 1: top 11 key bits, histogram built by the scoring pass ----
    for (int i = tid; i < kBins; i += blockDim.x) hist[i] = ghist[size_t(b) * kBins + i];
    __syncthreads();
    int bin1, above1;
    find_bin(hist, kBins, K, sh, &bin1, &above1);
    // ---- level 2: next 11 bits among keys in bin1 ----
    for (int i = tid; i < kBins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < T; i += blockDim.x) {
        const uint32_t k = okey(s[i]);
        if ((k >> 21) == uint32_t(bin1)) atomicAdd(&hist[(k >> 10) & 2047u], 1u);
    }
    __syncthreads();
    int bin2, above2;
    find_bin(hist, kBins, K - above1, sh, &bin2, &above2);
    // ---- level 3: last 10 bits ----
    const uint32_t pre = (uint32_t(bin1) << 11) | uint32_t(bin2);
    for (int i = tid; i < kBins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < T; i += blockDim.x) {
        const uint32_t k = okey(s[i]);
        if ((k >> 10) == pre) atomicAdd(&hist[k & 1023u], 1u);
    }
    __syncthreads();
    int bin3, above3;
    find_bin(hist, 1024, K - above1 - above2, sh, &bin3, &above3);
    const uint32_t kth = (pre << 10) | uint32_t(bin3);
    const int need_eq = K - above1 - above2 - above3;          // >= 1
    const bool all_eq = int(hist[bin3]) == need_eq;            // no tie to break
    __syncthreads();
    // ---- collect in position order ----
    int out_base = 0, eq_base = 0;
    for (int t0 = 0; t0 < T; t0 += 1024 * kSelPer) {
        const int i0 = t0 + tid * kSelPer;
        uint32_t gt = 0, eq = 0;
#pragma unroll
        for (int u = 0; u < kSelPer; ++u) {
            if (i0 + u < T) {
                const uint32_t k = okey(s[i0 + u]);
                gt |= uint32_t(k > kth) << u;
                eq |= uint32_t(k == kth) << u;
            }
        }
        uint32_t sel = gt | eq;
        if (!all_eq) {
            int eq_total;
            const int eq_before = eq_base + block_excl_scan(__popc(eq), sh, &eq_total);
            uint32_t keep = 0;
            int r = eq_before;
            for (uint32_t m = eq; m; m &= m - 1, ++r)
                if (r < need_eq) keep |= m & (~m + 1);
            sel = gt | keep;
            eq_base += eq_total;
        }
        int sel_total;
        int o = out_base + block_excl_scan(__popc(sel), sh, &sel_total);
        for (uint32_t m = sel; m; m &= m - 1, ++o) {
            const int pos = i0 + (__ffs(m) - 1);
            oi[o] = pos;
            if (os) os[o] = s[pos];
        }
        out_base += sel_total;
    }
    if (out_base != K) report(status, kStInvalid);   // cannot happen for finite scores
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

IndexPlan plan_index(int B, int max_seqlen) {
    IndexPlan p{};
    p.scores_off = 0;
    p.hist_off = align256(size_t(B) * max_seqlen * 4);
    p.tiles_off = p.hist_off + align256(size_t(B) * kBins * 4);
    p.total = p.tiles_off + align256(size_t(B + 1) * 4);
    return p;
}

cudaError_t launch_index_topk(const IndexArgs& a, const IndexPlan& pl, const DeviceInfo& dev,
                              const Knobs& kn, const KernelTimer& tm, cudaStream_t st) {
    static_assert(kScoreSmem <= 227 * 1024, "shared memory budget");
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    float* scores = reinterpret_cast<float*>(ws + pl.scores_off);
    unsigned* hist = reinterpret_cast<unsigned*>(ws + pl.hist_off);
    int* tiles = reinterpret_cast<int*>(ws + pl.tiles_off);

    CUtensorMap kmap, qmap;
    const uint64_t rows = a.total_keys > 0 ? uint64_t(a.total_keys) : 1;
    cudaError_t e = encode_tmap_2d_bf16(&kmap, a.index_k, kIndexDim, rows, kIndexDim * 2, 64, kTile);
    if (e != cudaSuccess) return e;
    e = encode_tmap_2d_bf16(&qmap, a.index_q, kIndexDim, uint64_t(a.B) * kIndexHeads,
                            kIndexDim * 2, 64, kIndexHeads);
    if (e != cudaSuccess) return e;

    e = cudaMemsetAsync(hist, 0, size_t(a.B) * kBins * 4, st);
    if (e != cudaSuccess) return e;
    dsa_tiles_kernel<<<1, 1024, 0, st>>>(a.cu, a.B, a.max_seqlen, a.total_keys, a.topk, tiles,
                                         dev.status);
    e = cudaFuncSetAttribute(dsa_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kScoreSmem));
    if (e != cudaSuccess) return e;
    ScoreParams p{a.w, a.cu, tiles, scores, hist, a.B, a.max_seqlen, kn.wait_limit_ns, dev.status};
    if (tm.begin) cudaEventRecord(tm.begin, st);
    dsa_score_kernel<<<dev.sms, kScoreThreads, kScoreSmem, st>>>(kmap, qmap, p);
    if (tm.end) cudaEventRecord(tm.end, st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dsa_topk_kernel<<<a.B, 1024, 0, st>>>(scores, hist, a.cu, a.max_seqlen, a.total_keys, a.topk,
                                          a.topk_idx, a.topk_scores, dev.status);
    return cudaGetLastError();
}

}  // namespace mla
