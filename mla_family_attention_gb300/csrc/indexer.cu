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
//   warp 0  TMA producer: 128 key rows (two 64-feature swizzled boxes) per
//           shared-memory ring stage, and each sequence's 32 index queries;
//   warp 1  allocates 128 TMEM columns (four 32-column accumulators) and one
//           lane issues the eight K=16 MMAs per tile, committing to mbarriers;
//   warps 2-17, four groups of four warps, one group per accumulator: read it
//           (thread = position, 32 columns = heads), apply ReLU and the head
//           weights, write the fp32 score and count it in a 2048-bin
//           histogram of its top 11 order-preserving key bits.
// Each CTA starts on a home sequence and claims tiles two at a time from
// per-sequence counters (home first, then the following sequences), so the
// CTAs finish together although their rates differ; home bins are counted
// in shared memory and added to the global histogram once, at the end, the
// bins of tiles claimed elsewhere directly.  The FP8 variant reads 128 e4m3
// codes per position and applies the key's scale in the epilogue.
//
// Top-k: dsa_topk_regs_kernel for sequences of at most 8 x 16,384
// positions (each thread's 16 order keys stay in registers; the keys sharing
// the k-th key's 22-bit prefix are ranked by ballots), else
// dsa_topk_cluster_kernel, a cluster of eight CTAs per sequence.  Both are an
// exact radix select on order-preserving 32-bit keys: the first 11 bits come
// from the histogram the scoring pass built, a pass over the (L2-resident)
// scores held in shared memory finds the next 11 bits of the k-th key (and,
// only when that bin holds more keys than are still needed, another pass the
// last 10), the CTAs sum their bins through distributed shared memory, and a
// final pass in position order keeps every key above the k-th plus the
// lowest positions among keys equal to it, writing the output in ascending
// position order directly.
//
// The tile-list, scoring and top-k kernels are launched as programmatic
// dependents of one another: each waits on the device before it touches
// global memory, and does its set-up while its predecessor drains.
#include <algorithm>

#include <cuda.h>
#include <cuda_fp8.h>

#define MLA_FILE_ID 3   // site ids of the bounds-checked debug build
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kTile = 128;                                   // positions per MMA tile
#ifndef MLA_INDEX_STAGES
#define MLA_INDEX_STAGES 6
#endif
constexpr int kIStages = MLA_INDEX_STAGES;
// The TMA producer prefetches into L2 the key rows of the next chunk it has
// claimed (bf16 keys; 0 = none): 2-4 tiles ahead of its loads.  With
// contiguous ranges, 4 tiles ahead had taken the scoring kernel from 49.6
// to 46.7 us on B=8, T=131072, and 8 and 16 ahead were slower (the
// prefetches share the TMA unit with the loads); FP8 keys gained nothing,
// so their producer prefetches nothing.
#ifndef MLA_INDEX_PREFETCH
#define MLA_INDEX_PREFETCH 1
#endif
// Tiles per claim.  The scoring CTAs take their tiles from per-sequence
// counters, two at a time: each starts on a home sequence (the one holding
// tile c*n/G, so ~n/G tiles per CTA) and moves to the following sequences
// once it is used up.  With fixed contiguous ranges the 152 CTAs finished
// between 38.5 and 43.4 us (B=8, T=131072): their rates differ by ~10 %.
constexpr int kClaim = 2;
constexpr int kAHalf = kTile * 64 * 2;                       // 16 KB: 128 rows x 128 B
constexpr int kBHalf = kIndexHeads * 64 * 2;                 // 4 KB: 32 rows x 128 B
constexpr int kStageBytes = 2 * kAHalf;                      // 32 KB of index keys
constexpr int kQBytes = 2 * kBHalf;                          // 8 KB: one sequence's queries
constexpr int kBins = 2048;
constexpr int kEpiGroups = 4;                               // epilogue groups of four warps (one per accumulator)
constexpr int kScoreThreads = (2 + 4 * kEpiGroups) * 32;
constexpr int kEpiThreads = 128 * kEpiGroups;
constexpr int kAcc = 4;                                      // TMEM accumulators (32 columns each)
constexpr uint32_t kTmemCols = 32 * kAcc;
constexpr uint32_t kIdesc = idesc_bf16_f32(128, kIndexHeads, false, false);
constexpr uint32_t kIdescF8 = idesc_e4m3_f32(128, kIndexHeads);

// Per-variant tile sizes: bf16 keys are two 64-feature boxes (256 B per
// position), e4m3 keys one 128-byte box (128 B per position).
// FP8 tiles are half the size, so the FP8 ring has twice the stages (the
// same bytes in flight, which is what keeps HBM busy).
template <bool kFp8>
struct ScoreCfg {
    static constexpr int kStage = kFp8 ? kTile * 128 : kStageBytes;
    static constexpr int kStages = kFp8 ? 2 * kIStages : kIStages;
    static constexpr int kQ = kFp8 ? kIndexHeads * 128 : kQBytes;
    // barriers: 2*kStages ring + 2*kAcc accumulator + 2 query + kAcc tile
    // notices, then the TMEM address and the abort flag; then the tile of
    // each ring stage and of each accumulator (int2 each)
    static constexpr size_t kBarBytes = (2 * kStages + 3 * kAcc + 2) * 8 + 16;
    static constexpr size_t kSmem = 1024 + size_t(kStages) * kStage + 2 * kQ + kBins * 4 + kBarBytes +
                                    (kStages + kAcc) * 8;
};

struct ScoreParams {
    const void* keys;        // the key rows the tensor map reads (for L2 prefetches)
    int64_t total_keys;
    const float* w;          // head weights (FP8: with the query scales folded in)
    const float* kscale;     // FP8: per-position key scale, else null
    const int64_t* cu;
    const int* tile_start;   // [B+1]
    int* claim;              // [B] tiles of each sequence claimed so far (zeroed by the tiles kernel)
    float* scores;           // [B][stride]
    unsigned* hist;          // [B][2048]
    int B, stride;
    long long wait_ns;
    int* status;
};

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2_bytes(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

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

template <bool kFp8>
__global__ void __launch_bounds__(kScoreThreads, 1)
    dsa_score_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap qmap, const ScoreParams p) {
    using C = ScoreCfg<kFp8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* qbuf = smem + C::kStages * C::kStage;              // [2] query tiles
    unsigned* hist = reinterpret_cast<unsigned*>(qbuf + 2 * C::kQ);
    uint64_t* full = reinterpret_cast<uint64_t*>(hist + kBins);
    uint64_t* empty = full + C::kStages;
    uint64_t* tfull = empty + C::kStages;
    uint64_t* tempty = tfull + kAcc;
    uint64_t* qfull = tempty + kAcc;
    uint64_t* tnote = qfull + 2;                                // [kAcc] accumulator's tile known
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tnote + kAcc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    // (tile, sequence) of each ring stage (tile -1: no more tiles) and of
    // each accumulator, written by the producer and the MMA warp
    int2* stage_tile = reinterpret_cast<int2*>(tmem_holder + 4);
    int2* acc_tile = stage_tile + C::kStages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        grid_dep_trigger();
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
            mbar_init(&tnote[a], 1);
        }
        mbar_init(&qfull[0], 1);
        mbar_init(&qfull[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0;
    if (warp == 1) tmem_alloc(tmem_holder, kTmemCols);
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&qmap);
    }
    // everything above is set-up; the tile list, the cleared histograms and
    // claim counters come from the tiles kernel
    grid_dep_wait();
    const int n_tiles = p.tile_start[p.B];
    // home sequence: the one holding tile c*n/G (its level-1 bins are kept in
    // shared memory; tiles of other sequences add theirs to global memory)
    const int home = n_tiles > 0
        ? tile_owner(p.tile_start, p.B, int((int64_t(n_tiles) * blockIdx.x) / gridDim.x))
        : 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            const uint64_t stream_policy = l2_evict_first_policy();
            // Queries are loaded once per sequence into one of two buffers; a
            // buffer is refilled only after the MMAs of the last tile that read
            // it have completed (the commit of that tile's stage).
            int filled[C::kStages];
            for (int i = 0; i < C::kStages; ++i) filled[i] = 0;
            int qfilled[2] = {0, 0}, last_use[2] = {-1, -1};
            int cur_b = -1, seg = 0, row0 = 0;   // row0: first key row of sequence cur_b
            // claims: chunk = (first tile, tiles, sequence); seq is the
            // sequence of the latest claim
            int seq = home;
            auto ntiles = [&](int b) { return p.tile_start[b + 1] - p.tile_start[b]; };
            // Blocking claim from seq onwards (cyclically): the claim counters
            // of eight sequences are read at once, the first one with tiles
            // left is claimed; a claim that lost the race probes again.
            auto claim_next = [&]() -> int3 {
                for (int attempt = 0; attempt < 4 * p.B + 4; ++attempt) {
                    int found = -1;
                    for (int k0 = 0; k0 < p.B && found < 0; k0 += 8) {
                        int c[8], nt[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            int b = seq + k0 + k;
                            b -= b >= p.B ? p.B : 0;
                            const bool in = k0 + k < p.B;
                            c[k] = in ? *reinterpret_cast<volatile int*>(p.claim + b) : 0;
                            nt[k] = in ? ntiles(b) : 0;
                        }
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            if (found < 0 && c[k] < nt[k]) {
                                found = seq + k0 + k;
                                found -= found >= p.B ? p.B : 0;
                            }
                    }
                    if (found < 0) break;
                    seq = found;
                    const int base = int(atomicAdd(reinterpret_cast<unsigned*>(p.claim + seq),
                                                   unsigned(kClaim)));
                    if (base < ntiles(seq))
                        return make_int3(p.tile_start[seq] + base, min(kClaim, ntiles(seq) - base),
                                         seq);
                }
                return make_int3(0, 0, -1);
            };
            auto prefetch_chunk = [&](int3 ch) {
                if (kFp8 || MLA_INDEX_PREFETCH == 0 || ch.y <= 0) return;
                const int64_t r0 = int64_t(p.cu[ch.z]) + int64_t(ch.x - p.tile_start[ch.z]) * kTile;
                int64_t r1 = r0 + int64_t(ch.y) * kTile;
                if (r1 > p.cu[ch.z + 1]) r1 = p.cu[ch.z + 1];
                if (r1 > r0 && r0 >= 0 && r1 <= p.total_keys)
                    prefetch_l2_bytes(static_cast<const uint8_t*>(p.keys) + r0 * (C::kStage / kTile),
                                      uint32_t((r1 - r0) * (C::kStage / kTile)));
            };
            // The first 2*kClaim tiles of each CTA need no claim: CTA c is the
            // r-th of the CTAs homed on sequence h and takes tiles 4r..4r+3 of
            // it (the tiles kernel started h's counter past them).
            int3 cur = make_int3(0, 0, -1), nxt = make_int3(0, 0, -1);
            if (n_tiles > 0) {
                const int64_t G = gridDim.x, n = n_tiles;
                const int r = int(blockIdx.x) - int((int64_t(p.tile_start[home]) * G + n - 1) / n);
                const int nt = ntiles(home), f0 = 2 * kClaim * r;
                if (f0 < nt) cur = make_int3(p.tile_start[home] + f0, min(kClaim, nt - f0), home);
                if (f0 + kClaim < nt)
                    nxt = make_int3(p.tile_start[home] + f0 + kClaim, min(kClaim, nt - f0 - kClaim),
                                    home);
            }
            if (cur.y == 0) {
                cur = claim_next();
                nxt = cur.y > 0 ? claim_next() : make_int3(0, 0, -1);
            } else if (nxt.y == 0) {
                nxt = claim_next();
            }
            int j = 0;
            bool ok = true;
            while (ok && cur.y > 0) {
                // the claim after nxt, in flight while cur's tiles are issued
                const bool pending = nxt.y > 0;
                const unsigned pend =
                    pending ? atomicAdd(reinterpret_cast<unsigned*>(p.claim + seq), unsigned(kClaim))
                            : 0u;
                prefetch_chunk(nxt);
                for (int t = cur.x; t < cur.x + cur.y; ++t, ++j) {
                    const int slot = j % C::kStages, round = j / C::kStages;
                    if (*abort_flag) { ok = false; break; }
                    if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, p.wait_ns)) {
                        report(p.status, kStTimeout);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    const int b = cur.z;
                    if (b != cur_b) {
                        const int qb = seg & 1;
                        const int lu = last_use[qb];
                        if (lu >= 0 && j - lu < C::kStages &&
                            !mbar_wait(&empty[lu % C::kStages], (lu / C::kStages) & 1, p.wait_ns)) {
                            report(p.status, kStTimeout);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&qfull[qb], C::kQ);
                        tma_load_2d(qbuf + qb * C::kQ, &qmap, 0, b * kIndexHeads, &qfull[qb]);
                        if (!kFp8)
                            tma_load_2d(qbuf + qb * C::kQ + kBHalf, &qmap, 64, b * kIndexHeads,
                                        &qfull[qb]);
                        qfilled[qb] = (seg >> 1) + 1;
                        cur_b = b;
                        row0 = int(p.cu[b]) - p.tile_start[b] * kTile;
                        ++seg;
                    }
                    last_use[(seg - 1) & 1] = j;
                    const int row = row0 + t * kTile;
                    MLA_CHECK(slot < C::kStages && row >= 0, p.status);
                    stage_tile[slot] = make_int2(t, b);
                    uint8_t* st = smem + slot * C::kStage;
                    mbar_arrive_expect_tx(&full[slot], C::kStage);
                    tma_load_2d_hint(st, &kmap, 0, row, &full[slot], stream_policy);
                    if (!kFp8)
                        tma_load_2d_hint(st + kAHalf, &kmap, 64, row, &full[slot], stream_policy);
                    filled[slot] = round + 1;
                }
                if (!ok) break;
                int3 after = make_int3(0, 0, -1);
                if (pending) {
                    if (int(pend) < ntiles(seq))
                        after = make_int3(p.tile_start[seq] + int(pend),
                                          min(kClaim, ntiles(seq) - int(pend)), seq);
                    else
                        after = claim_next();
                }
                cur = nxt;
                nxt = after;
            }
            if (ok) {
                // no more tiles: the stage after the last one carries tile -1
                const int slot = j % C::kStages, round = j / C::kStages;
                if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, p.wait_ns)) {
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                } else {
                    stage_tile[slot] = make_int2(-1, -1);
                    mbar_arrive(&full[slot]);
                    filled[slot] = round + 1;
                }
            }
            for (int i = 0; i < C::kStages; ++i)
                if (filled[i] > 0 && !mbar_wait(&full[i], (filled[i] - 1) & 1, p.wait_ns))
                    report(p.status, kStTimeout);
            for (int i = 0; i < 2; ++i)
                if (qfilled[i] > 0 && !mbar_wait(&qfull[i], (qfilled[i] - 1) & 1, p.wait_ns))
                    report(p.status, kStTimeout);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer -------------------------------
        // Takes each stage's tile from the producer, hands it on to the
        // epilogue group of the stage's accumulator (acc_tile + tnote), and
        // after the last tile posts "no more tiles" to all four groups.
        if (lane == 0) {
            int last_acc = -1, last_phase = 0;
            int cur_b = -1, seg = 0;
            for (int j = 0;; ++j) {
                const int slot = j % C::kStages, acc = j % kAcc;
                if (*abort_flag) break;
                if (!mbar_wait(&full[slot], (j / C::kStages) & 1, p.wait_ns)) {
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                    break;
                }
                const int2 tb = stage_tile[slot];
                if (tb.x < 0) {                           // no more tiles
                    for (int k = 0; k < kAcc; ++k) {
                        const int jj = j + k, a = jj % kAcc;
                        if (jj >= kAcc && !mbar_wait(&tempty[a], ((jj / kAcc) - 1) & 1, p.wait_ns)) {
                            report(p.status, kStTimeout);
                            *abort_flag = 1;
                            break;
                        }
                        acc_tile[a] = make_int2(-1, -1);
                        mbar_arrive(&tnote[a]);
                    }
                    break;
                }
                bool ok = true;
                if (tb.y != cur_b) {                      // this sequence's queries
                    ok = mbar_wait(&qfull[seg & 1], (seg >> 1) & 1, p.wait_ns);
                    cur_b = tb.y;
                    ++seg;
                }
                if (!ok ||
                    (j >= kAcc && !mbar_wait(&tempty[acc], ((j / kAcc) - 1) & 1, p.wait_ns))) {
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                    break;
                }
                acc_tile[acc] = tb;
                mbar_arrive(&tnote[acc]);
                tc_fence_after();
                const uint32_t a0 = smem_u32(smem + slot * C::kStage);
                const uint32_t b0 = smem_u32(qbuf + ((seg - 1) & 1) * C::kQ);
                if (kFp8) {
                    // one 128-byte row per position: four K = 32 steps of 32 bytes
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
                        const uint64_t bd = smem_desc_sw128(b0 + kk * 32, 16, 1024);
                        mma_f8_ss(tmem + acc * 32, ad, bd, kIdescF8, kk > 0 ? 1u : 0u);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad =
                            smem_desc_sw128(a0 + (kk >> 2) * kAHalf + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd =
                            smem_desc_sw128(b0 + (kk >> 2) * kBHalf + (kk & 3) * 32, 16, 1024);
                        mma_bf16_ss(tmem + acc * 32, ad, bd, kIdesc, kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit(&empty[slot]);
                mma_commit(&tfull[acc]);
                last_acc = acc;
                last_phase = (j / kAcc) & 1;
            }
            // the accumulator must not be released while an MMA still writes it
            if (last_acc >= 0 && !mbar_wait(&tfull[last_acc], last_phase, p.wait_ns))
                report(p.status, kStTimeout);
        }
    } else {
        // ------------------------------- epilogue --------------------------------
        // kEpiGroups groups of four warps take turns: group g the tiles of
        // accumulator g (steps j = g, g + kEpiGroups, ...), each told by the
        // MMA warp which tile its next step holds.  Scores of the home
        // sequence are counted in the shared histogram (added to global
        // memory once, at the end); those of other sequences directly in
        // global memory.
        const int grp = (warp - 2) >> 2;
        const int quad = warp & 3;                 // TMEM lanes 32*quad .. 32*quad+31
        const int r = quad * 32 + lane;            // position within the tile
        const int acc = grp;
        int cur_b = -1, T = 0, tstart = 0;
        int64_t kbase = 0;                         // first key row of the current sequence
        float wr[kIndexHeads];                     // head weights of the current sequence
        for (int j = grp;; j += kEpiGroups) {
            const uint32_t par = (j / kAcc) & 1;
            bool ok = !*abort_flag && mbar_wait(&tnote[acc], par, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0 && !*abort_flag) {
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                }
                break;
            }
            const int2 tb = acc_tile[acc];
            if (tb.x < 0) break;                   // no more tiles
            const int t = tb.x, b = tb.y;
            if (b != cur_b) {
                cur_b = b;
                kbase = p.cu[b];
                T = int(p.cu[b + 1] - kbase);
                tstart = p.tile_start[b];
#pragma unroll
                for (int h = 0; h < kIndexHeads; ++h) wr[h] = __ldg(p.w + size_t(b) * kIndexHeads + h);
            }
            const int pos = (t - tstart) * kTile + r;
            const bool in = pos < T;
            // FP8: the key scale is loaded before the accumulator wait so its
            // latency overlaps it
            const float ksc = (kFp8 && in) ? __ldg(p.kscale + kbase + pos) : 1.f;
            ok = mbar_wait(&tfull[acc], par, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) {
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            MLA_CHECK(acc < kAcc && uint32_t(acc * 32 + 32) <= kTmemCols && r < kTile, p.status);
            float d[32];
            tmem_ld32(tmem + (uint32_t(quad * 32) << 16) + acc * 32, d);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);

            float s = 0.f;
#pragma unroll
            for (int h = 0; h < kIndexHeads; ++h) s = fmaf(wr[h], fmaxf(d[h], 0.f), s);
            if (kFp8) s *= ksc;
            s += 0.0f;                             // -0 -> +0: equal scores compare equal
            MLA_CHECK(!in || (pos >= 0 && pos < p.stride && b < p.B), p.status);
            if (in) p.scores[size_t(b) * p.stride + pos] = s;
            // histogram of the top 11 key bits, one atomic per distinct bin per warp
            const unsigned mask = __ballot_sync(0xffffffffu, in);
            if (in) {
                const unsigned bin = okey(s) >> 21;
                MLA_CHECK(bin < unsigned(kBins), p.status);
                const unsigned peers = __match_any_sync(mask, bin);
                if (lane == __ffs(peers) - 1) {
                    if (b == home)
                        atomicAdd(&hist[bin], unsigned(__popc(peers)));
                    else
                        atomicAdd(&p.hist[size_t(b) * kBins + bin], unsigned(__popc(peers)));
                }
            }
        }
        named_bar_sync(1, kEpiThreads);
        if (n_tiles > 0) {
            for (int i = threadIdx.x - 64; i < kBins; i += kEpiThreads) {
                const unsigned c = hist[i];
                if (c) atomicAdd(&p.hist[size_t(home) * kBins + i], c);
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
// Blocks after the first clear the level-1 histograms the scoring pass adds
// into (B x 2048 counters).  Block 0 also starts each sequence's claim
// counter past the tiles the G scoring CTAs homed on it take without a
// claim (2 * kClaim each; CTA c is homed on the sequence holding tile
// floor(c * n / G), so the CTAs homed on b are ceil(start_b * G / n) ..
// ceil(start_{b+1} * G / n) - 1).
__global__ void __launch_bounds__(1024) dsa_tiles_kernel(const int64_t* cu, int B, int max_seqlen,
                                                         int64_t total_keys, int topk,
                                                         int* tile_start, unsigned* hist,
                                                         int* claim, int G, int* status) {
    __shared__ int warp_sums[32];
    if (threadIdx.x == 0) grid_dep_trigger();
    grid_dep_wait();
    if (blockIdx.x > 0) {
        const size_t n = size_t(B) * kBins;
        for (size_t i = size_t(blockIdx.x - 1) * blockDim.x + threadIdx.x; i < n;
             i += size_t(gridDim.x - 1) * blockDim.x)
            hist[i] = 0;
        return;
    }
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
    const int64_t n = warp_sums[31];               // all tiles
    auto first_cta = [&](int64_t t) { return n > 0 ? (t * G + n - 1) / n : int64_t(0); };
    for (int b = b0; b < b1; ++b) {
        tile_start[b] = run;
        const int64_t T = cu[b + 1] - cu[b];
        int nt = 0;
        if (!(T < 0 || T > max_seqlen || cu[b] < 0 || cu[b + 1] > total_keys))
            nt = T > topk ? int((T + kTile - 1) / kTile) : 0;
        const int64_t homed = nt > 0 ? first_cta(run + nt) - first_cta(run) : 0;
        claim[b] = int(min(int64_t(nt), homed * 2 * kClaim));
        run += nt;
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

// Distributed shared memory: the address of `p` in cluster CTA `rank`, and
// remote add / store / load through it.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}

__device__ __forceinline__ void dsmem_add(uint32_t addr, unsigned v) {
    asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned dsmem_ld(uint32_t addr) {
    unsigned v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Bin holding the K-th largest key given a histogram (bins ordered by key):
// count(bins above) < K <= count(bins at or above).  With own > 0 the
// histogram is a cluster total kept by owners: bin i in CTA i / own.  Each
// thread then fetches its bins from their owner and leaves a copy in its own
// `hist`, so the whole total can be read locally after the call.
__device__ __forceinline__ void find_bin(unsigned* hist, int nbins, int K, int* sh,
                                         int* out_bin, int* out_above, int own = 0,
                                         uint32_t rank = 0) {
    const int per = nbins / 1024;                  // 1 or 2 bins per thread
    const int hi = nbins - 1 - int(threadIdx.x) * per;
    unsigned c2[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 2; ++i)
        if (i < per) {
            const uint32_t r = own ? uint32_t((hi - i) / own) : rank;
            c2[i] = r != rank ? dsmem_ld(dsmem_addr(&hist[hi - i], r)) : hist[hi - i];
        }
    int local = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i)
        if (i < per) {
            if (own && uint32_t((hi - i) / own) != rank) hist[hi - i] = c2[i];
            local += int(c2[i]);
        }
    int total;
    const int above = block_excl_scan(local, sh, &total);
    if (above < K && K <= above + local) {
        int cum = above;
        for (int i = 0; i < per; ++i) {
            const int c = int(c2[i]);
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

constexpr int kSelPer = 16;                        // positions per thread per pass step
constexpr int kStep = 1024 * kSelPer;              // positions per CTA per pass step
#ifndef MLA_TOPK_CLUSTER
#define MLA_TOPK_CLUSTER 8
#endif
constexpr int kCluster = MLA_TOPK_CLUSTER;         // CTAs cooperating on one sequence

// Load this thread's 16 consecutive scores (positions i0..i0+15, rows padded
// to 16 bytes so the float4 reads stay inside the row).
__device__ __forceinline__ void load16(const float* s, int i0, int T, float (&v)[kSelPer]) {
    const float4* s4 = reinterpret_cast<const float4*>(s);
#pragma unroll
    for (int u = 0; u < kSelPer / 4; ++u) {
        const float4 x = (i0 + 4 * u) < T ? s4[(i0 >> 2) + u] : make_float4(0.f, 0.f, 0.f, 0.f);
        v[4 * u] = x.x;
        v[4 * u + 1] = x.y;
        v[4 * u + 2] = x.z;
        v[4 * u + 3] = x.w;
    }
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of all CTAs of the cluster; orders shared-memory writes before
// the barrier with reads (local or remote) after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of cluster_sync, for work that can run between them.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

struct TopkParams {
    const float* scores;     // [B][stride]
    const unsigned* hist1;   // [B][2048]  top 11 key bits (built by the scoring pass)
    const int64_t* cu;
    int max_seqlen, stride, topk;
    int64_t total_keys;
    int32_t* out_idx;
    float* out_scores;
    int* status;
};

__device__ __forceinline__ int seq_len(const TopkParams& p, int b) {
    const int64_t T = p.cu[b + 1] - p.cu[b];
    const bool ok = !(T < 0 || T > p.max_seqlen || p.cu[b] < 0 || p.cu[b + 1] > p.total_keys);
    return ok ? int(T) : 0;
}


// Keys that share the k-th key's 22-bit prefix are ranked one against another
// when there are at most kCand of them (the usual case: a handful).
constexpr int kCand = 256;
constexpr size_t kTopkSmem = size_t(kStep) * 4 + (kBins + 1024 + kBins + kBins) * 4 +
                             2 * kCluster * 4 + size_t(kCluster) * kCand * 8 + kCluster * 4 +
                             kCand * 4;

// Top-k of one sequence per cluster of eight CTAs; CTA r owns positions
// [r*span, (r+1)*span) and keeps them in shared memory when they fit (one
// 16,384-position step; otherwise every pass re-reads its steps from L2).
// Level 1 of the radix select (top 11 key bits) comes with the scores; level 2
// histograms the next 11 bits of the keys inside the level-1 bin.  Bin i of
// the level-2 cluster total is kept by CTA i / (bins / cluster size): each CTA
// adds its partial bins into the owners' totals with remote (distributed
// shared memory) atomics, one per nonzero bin, and after a cluster barrier
// every CTA reads the whole total back from the owners, so all CTAs find the
// same bin.  The keys above its 22-bit prefix are kept; of the keys sharing
// it (the candidates, usually a handful), the larger ones are kept, lower
// positions first among equal keys.  Up to kCand candidates are exchanged
// with their positions and ranked in every CTA; with more, a third 10-bit
// level (same scheme) finds the exact k-th key, and a count exchange follows.
// Each CTA then writes its kept positions at their place in the ascending
// output.  Three cluster barriers, four when level 3 runs.
// (cluster size set at launch: 16 is a non-portable size)
__global__ void __launch_bounds__(1024) dsa_topk_cluster_kernel(const TopkParams p) {
    extern __shared__ float4 topk_dyn[];
    // scores of one step: element u of thread t (position t0 + 16t + u) at
    // vals[u*1024 + t], so a warp's accesses hit 32 different banks
    float* vals = reinterpret_cast<float*>(topk_dyn);
    unsigned* sum2 = reinterpret_cast<unsigned*>(vals + kStep);   // [2048] cluster totals
    unsigned* sum3 = sum2 + kBins;                                // [1024] cluster totals
    unsigned* hist1 = sum3 + 1024;                                // [2048] level 1
    unsigned* part = hist1 + kBins;                               // [2048] this CTA's bins
    int* cnts = reinterpret_cast<int*>(part + kBins);             // [kCluster][2]
    uint32_t* ckey = reinterpret_cast<uint32_t*>(cnts + 2 * kCluster);  // [kCluster][kCand]
    int* cpos = reinterpret_cast<int*>(ckey + kCluster * kCand);         // [kCluster][kCand]
    int* ccnt = cpos + kCluster * kCand;                                 // [kCluster]
    int* ckeep = ccnt + kCluster;                                        // [kCand]
    __shared__ int sh[40];
    const int b = blockIdx.y;
    const uint32_t rank = cluster_rank();
    const int tid = threadIdx.x;
    if (tid == 0) grid_dep_trigger();
    grid_dep_wait();                                // the scores and level-1 bins
    int32_t* oi = p.out_idx + size_t(b) * p.topk;
    float* os = p.out_scores ? p.out_scores + size_t(b) * p.topk : nullptr;
    const int T = seq_len(p, b);                    // the same for the whole cluster
    if (T <= p.topk) {                              // every position is kept
        if (rank == 0)
            for (int i = tid; i < p.topk; i += blockDim.x) {
                oi[i] = i < T ? i : -1;
                if (os) os[i] = -INFINITY;
            }
        return;
    }
    const int K = p.topk;
    const int span = ((T + kCluster - 1) / kCluster + kSelPer - 1) / kSelPer * kSelPer;
    const int lo = int(rank) * span, hi = min(T, lo + span);
    const bool resident = hi - lo <= kStep;
    const float* s = p.scores + size_t(b) * p.stride;

    // Load step [t0, t0+kStep) of this CTA's range into shared memory.
    auto stage = [&](int t0) {
        float v[kSelPer];
        const int i0 = t0 + tid * kSelPer;
        load16(s, i0, hi, v);
#pragma unroll
        for (int u = 0; u < kSelPer; ++u) vals[u * 1024 + tid] = v[u];
        MLA_CHECK((kSelPer - 1) * 1024 + tid < kStep, p.status);
    };
    // level-1 bins and this CTA's scores: both loads are issued before either
    // is stored, so their latencies overlap
    static_assert(kBins == 2 * 1024, "two level-1 bins per thread");
    unsigned hv[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) hv[k] = p.hist1[size_t(b) * kBins + tid + k * 1024];
    if (resident) stage(lo);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        sum2[tid + k * 1024] = 0;
        hist1[tid + k * 1024] = hv[k];
    }
    sum3[tid] = 0;
    if (tid == 0) sh[36] = 0;                       // this CTA's candidate count
    __syncthreads();
    cluster_arrive();                               // (1) every CTA's totals are zero ...
    int bin1, above1;
    find_bin(hist1, kBins, K, sh, &bin1, &above1);

    // One refinement level: partial bins of the keys with top bits == pre
    // (and, per thread, the number of keys whose top bits are above pre),
    // then added into the owners' totals.
    int n_above = 0;
    auto hist_level = [&](int shift, int nb, uint32_t pre) {
        n_above = 0;
        for (int i = tid; i < nb; i += blockDim.x) part[i] = 0;
        __syncthreads();
        for (int t0 = lo; t0 < hi; t0 += kStep) {
            if (!resident) {
                stage(t0);
                __syncthreads();
            }
            const int i0 = t0 + tid * kSelPer;
#pragma unroll
            for (int u = 0; u < kSelPer; ++u) {
                if (i0 + u < hi) {
                    const uint32_t k = okey(vals[u * 1024 + tid]);
                    const uint32_t top = k >> (shift + (nb == 1024 ? 10 : 11));
                    if (top == pre)
                        atomicAdd(&part[(k >> shift) & uint32_t(nb - 1)], 1u);
                    n_above += top > pre;
                }
            }
            if (!resident) __syncthreads();
        }
        __syncthreads();
    };
    auto push_level = [&](int nb, unsigned* total) {
        const int own = nb / kCluster;
        for (int i = tid; i < nb; i += blockDim.x) {
            const unsigned c = part[i];
            if (c) dsmem_add(dsmem_addr(&total[i], uint32_t(i / own)), c);
        }
    };
    hist_level(10, kBins, uint32_t(bin1));
    cluster_wait();                                 // (1) ... before anyone adds into them
    push_level(kBins, sum2);
    cluster_sync();                                 // (2) level-2 totals at their owners
    int bin2, above2;
    find_bin(sum2, kBins, K - above1, sh, &bin2, &above2, kBins / kCluster, rank);
    MLA_CHECK(bin1 >= 0 && bin1 < kBins && bin2 >= 0 && bin2 < kBins, p.status);
    const uint32_t pre = (uint32_t(bin1) << 11) | uint32_t(bin2);
    // Keys are compared by their top 32 - kshift bits from here on: kth is
    // the k-th key's prefix, need_eq the number of keys sharing it that are
    // kept.  The totals are the same in every CTA, so the whole cluster takes
    // the same branch below.
    uint32_t kth = pre;
    int kshift = 10;
    int need_eq = K - above1 - above2;
    const int n_c = int(sum2[bin2]);                // keys of the sequence with prefix pre
    const bool cand = n_c <= kCand;
    int gt_before = 0, eq_before = 0, keep_before = 0;
    // This CTA's keys above the 22-bit prefix: those above bin1 plus its
    // level-2 bins above bin2 (`part` still holds its level-2 counts).
    auto count_above = [&]() {
        int gt = n_above;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int i = tid + k * 1024;
            if (i > bin2) gt += int(part[i]);
        }
        int tg;
        block_excl_scan(gt, sh, &tg);
        return tg;
    };
    if (cand) {
        // The few keys with prefix pre are sent, with their positions, to
        // every CTA (CTA r's into rows r of ckey / cpos), and so is this
        // CTA's count of keys above; after one barrier each CTA ranks the
        // candidates itself (larger key first, then lower position) and keeps
        // the first need_eq.
        const int tg = count_above();
        for (int t0 = lo; t0 < hi; t0 += kStep) {
            if (!resident) {
                __syncthreads();
                stage(t0);
                __syncthreads();
            }
            const int i0 = t0 + tid * kSelPer;
#pragma unroll
            for (int u = 0; u < kSelPer; ++u)
                if (i0 + u < hi) {
                    const uint32_t k = okey(vals[u * 1024 + tid]);
                    if ((k >> 10) == pre) {
                        const int j = atomicAdd(&sh[36], 1);
                        MLA_CHECK(j < kCand, p.status);
                        if (j < kCand)
                            for (uint32_t r = 0; r < kCluster; ++r) {
                                dsmem_st(dsmem_addr(&ckey[rank * kCand + j], r), int(k));
                                dsmem_st(dsmem_addr(&cpos[rank * kCand + j], r), i0 + u);
                            }
                    }
                }
        }
        __syncthreads();
        if (tid < kCluster) {
            dsmem_st(dsmem_addr(&ccnt[rank], uint32_t(tid)), min(sh[36], kCand));
            dsmem_st(dsmem_addr(&cnts[2 * rank], uint32_t(tid)), tg);
        }
        for (int i = tid; i < kCand; i += blockDim.x) ckeep[i] = 0;
        if (tid == 0) sh[37] = sh[38] = 0;
        cluster_sync();                             // (3) candidates and counts everywhere; last remote access
        for (int i = tid; i < kCluster * kCand; i += blockDim.x) {
            const int r = i / kCand;
            if (i - r * kCand >= ccnt[r]) continue;
            const uint32_t ki = ckey[i];
            const int pi = cpos[i];
            int before = 0, order = 0;              // rank, and rank by position alone
            for (int r2 = 0; r2 < kCluster; ++r2)
                for (int j = 0; j < ccnt[r2]; ++j) {
                    const uint32_t kj = ckey[r2 * kCand + j];
                    const int pj = cpos[r2 * kCand + j];
                    before += kj > ki || (kj == ki && pj < pi);
                    order += pj < pi;
                }
            const bool kept = before < need_eq;
            MLA_CHECK(order < kCand, p.status);
            if (order < kCand) ckeep[order] = kept;
            if (pi < lo) {
                atomicAdd(&sh[37], 1);
                if (kept) atomicAdd(&sh[38], 1);
            }
        }
        for (int r = 0; r < int(rank); ++r) gt_before += cnts[2 * r];
        __syncthreads();
        eq_before = sh[37];
        keep_before = sh[38];
    } else {
        // Many keys share the prefix: a third 10-bit level when the bin holds
        // more keys than are still needed, then the counts of this CTA's
        // keys above and equal to the k-th one go to every CTA.
        if (n_c != need_eq) {
            hist_level(0, 1024, pre);
            push_level(1024, sum3);
            cluster_sync();                         // (3) level-3 totals at their owners
            int bin3, above3;
            find_bin(sum3, 1024, K - above1 - above2, sh, &bin3, &above3, 1024 / kCluster, rank);
            MLA_CHECK(bin3 >= 0 && bin3 < 1024, p.status);
            kth = (pre << 10) | uint32_t(bin3);
            kshift = 0;
            need_eq -= above3;
        }
    }
    const bool all_eq = int(kshift ? n_c : sum3[kth & 1023u]) == need_eq;

    if (!cand) {
        // counts of this CTA's range, written into every CTA
        int tg, te;
        if (kshift) {                               // level 3 skipped
            tg = count_above();
            te = int(part[bin2]);
        } else {
            int gt = 0, eq = 0;
            for (int t0 = lo; t0 < hi; t0 += kStep) {
                if (!resident) {
                    __syncthreads();
                    stage(t0);
                    __syncthreads();
                }
                const int i0 = t0 + tid * kSelPer;
#pragma unroll
                for (int u = 0; u < kSelPer; ++u)
                    if (i0 + u < hi) {
                        const uint32_t k = okey(vals[u * 1024 + tid]);
                        gt += k > kth;
                        eq += k == kth;
                    }
            }
            block_excl_scan(gt, sh, &tg);
            block_excl_scan(eq, sh, &te);
        }
        if (tid < kCluster) {
            dsmem_st(dsmem_addr(&cnts[2 * rank], uint32_t(tid)), tg);
            dsmem_st(dsmem_addr(&cnts[2 * rank + 1], uint32_t(tid)), te);
        }
        cluster_sync();                             // (4) all counts everywhere; last remote access
        for (uint32_t r = 0; r < rank; ++r) {
            gt_before += cnts[2 * r];
            eq_before += cnts[2 * r + 1];
        }
        keep_before = min(eq_before, need_eq);      // equal keys are kept lowest position first
    }

    // emit in position order
    int out = gt_before + keep_before, eq_seen = eq_before;
    for (int t0 = lo; t0 < hi; t0 += kStep) {
        if (!resident) {
            __syncthreads();
            stage(t0);
            __syncthreads();
        }
        const int i0 = t0 + tid * kSelPer;
        uint32_t g = 0, e = 0;
#pragma unroll
        for (int u = 0; u < kSelPer; ++u)
            if (i0 + u < hi) {
                const uint32_t k = okey(vals[u * 1024 + tid]) >> kshift;
                g |= uint32_t(k > kth) << u;
                e |= uint32_t(k == kth) << u;
            }
        uint32_t keep = e;
        if (!all_eq) {                              // which of the keys equal to the k-th are kept
            int e_total;
            int r = eq_seen + block_excl_scan(__popc(e), sh, &e_total);
            keep = 0;
            for (uint32_t m = e; m; m &= m - 1, ++r) {
                MLA_CHECK(!cand || r < kCand, p.status);
                if (cand ? (r < kCand && ckeep[r] != 0) : r < need_eq) keep |= m & (~m + 1);
            }
            eq_seen += e_total;
        }
        const uint32_t take = g | keep;
        int total;
        int o = out + block_excl_scan(__popc(take), sh, &total);
        for (uint32_t m = take; m; m &= m - 1, ++o) {
            const int u = __ffs(m) - 1;
            if (o < K) {
                oi[o] = i0 + u;
                if (os) os[o] = vals[u * 1024 + tid];
            } else {
                report(p.status, kStInvalid);       // cannot happen for consistent counts
            }
        }
        out += total;
    }
}

// Inverse of okey: the score whose order key is k.
__device__ __forceinline__ float okey_inv(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Bin search with two block barriers: every warp scans its bins (taken from
// the top, `per` per thread), the 32 warp sums go through shared memory, and
// each warp forms its own prefix from them.  The bin holding the K-th largest
// key, the count of the bins above it and its own count go to sh[32..34]
// (1 <= K <= total is the caller's to ensure).  With own > 0 the histogram is
// a cluster total kept by owners (bin i in CTA i / own).  Uses sh[0..34].
__device__ __forceinline__ void find_bin_fast(const unsigned* hist, int nbins, int K, int* sh,
                                              int own, uint32_t rank) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = nbins / 1024;                  // 1 or 2 bins per thread
    const int hi = nbins - 1 - int(threadIdx.x) * per;
    unsigned c2[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 2; ++i)
        if (i < per) {
            const uint32_t r = own ? uint32_t((hi - i) / own) : rank;
            c2[i] = r != rank ? dsmem_ld(dsmem_addr(&hist[hi - i], r)) : hist[hi - i];
        }
    const int local = int(c2[0] + c2[1]);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    const int ws = sh[lane];
    int wincl = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wincl, o);
        if (lane >= o) wincl += y;
    }
    const int above = __shfl_sync(0xffffffffu, wincl - ws, warp) + incl - local;
    if (above < K && K <= above + local) {
        const bool first = above + int(c2[0]) >= K;
        sh[32] = first ? hi : hi - 1;
        sh[33] = first ? above : above + int(c2[0]);
        sh[34] = int(first ? c2[0] : c2[1]);
    }
    __syncthreads();
}

// Sum over the block of one value per thread (two warp reductions around one
// barrier); `slot` is a shared word cleared before the previous barrier.
__device__ __forceinline__ int block_sum(int v, int* slot) {
    const int w = __reduce_add_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0 && w) atomicAdd(slot, w);
    __syncthreads();
    return *slot;
}

#ifndef MLA_TOPK_RCLUSTER
#define MLA_TOPK_RCLUSTER 8
#endif
constexpr int kRC = MLA_TOPK_RCLUSTER;             // CTAs per sequence
constexpr int kRPer = 16 * 8 / kRC;                // positions per thread
constexpr int kRStep = 1024 * kRPer;               // positions per CTA
static_assert(kRPer == 8 || kRPer == 16, "8 or 16 CTAs per sequence");
constexpr int kRCand = 64;                         // candidates ranked one against another
struct RegsSmem {
    unsigned hist1[kBins];                         // level 1 (from the scoring pass)
    unsigned sum2[kBins];                          // level-2 cluster totals (owners + copies)
    unsigned part[kBins];                          // this CTA's level-2 (then level-3) bins
    unsigned sum3[1024];                           // level-3 cluster totals
    uint32_t kept[kRStep / 32];                     // kept candidates of this range, by position
    uint32_t ckey[kRC * kRCand];              // candidates of CTA r in row r
    int cpos[kRC * kRCand];
    int ccnt[kRC];
    int cnts[2 * kRC];                        // counts of every CTA's range
};

// Top-k of one sequence of at most 8 x 16,384 positions per cluster of eight
// CTAs (the same selection as dsa_topk_cluster_kernel).  Each thread holds the
// order keys of its 16 positions in registers from the first load to the
// output, so no pass re-reads them:
//   level 1: the bin from the scoring pass's histogram (while the scores load);
//   level 2: this CTA's histogram of the level-1 bin's keys, added into the
//     owners' totals (remote atomics), one barrier, the bin from the totals;
//   the keys above the 22-bit prefix are kept; those sharing it (at most
//     kRCand, else level 3 below) go with their positions to every CTA, and
//     so does this CTA's count of keys above; after one barrier every CTA
//     ranks the candidates (larger key first, lower position first among
//     equal keys) and keeps the first need_eq;
//   output: one block scan over the kept positions of each thread.
// With more candidates, a 10-bit level 3 finds the exact k-th key and a
// count exchange gives each CTA its offsets (two more barriers).
__global__ void __launch_bounds__(1024) dsa_topk_regs_kernel(const TopkParams p) {
    extern __shared__ uint4 regs_dyn[];
    RegsSmem& S = *reinterpret_cast<RegsSmem*>(regs_dyn);
    __shared__ int sh[48];
    const int b = blockIdx.y;
    const uint32_t rank = cluster_rank();
    const int tid = threadIdx.x;
    if (tid == 0) grid_dep_trigger();
    grid_dep_wait();                                // the scores and level-1 bins
    int32_t* oi = p.out_idx + size_t(b) * p.topk;
    float* os = p.out_scores ? p.out_scores + size_t(b) * p.topk : nullptr;
    auto span_of = [](int n) { return ((n + kRC - 1) / kRC + kRPer - 1) / kRPer * kRPer; };
    // This thread's level-1 bins and 16 scores are requested together with
    // the sequence length: the scores for the span of a sequence of
    // max_seqlen positions (re-read below when the length gives another),
    // inside the row's padded stride; past the length they are masked.
    unsigned hv[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) hv[k] = p.hist1[size_t(b) * kBins + tid + k * 1024];
    const float4* s4 = reinterpret_cast<const float4*>(p.scores + size_t(b) * p.stride);
    float v[kRPer];
    auto load_scores = [&](int first) {
#pragma unroll
        for (int q = 0; q < kRPer / 4; ++q) {
            const float4 x = first + 4 * q + 4 <= p.stride ? s4[(first >> 2) + q]
                                                            : make_float4(0.f, 0.f, 0.f, 0.f);
            v[4 * q] = x.x;
            v[4 * q + 1] = x.y;
            v[4 * q + 2] = x.z;
            v[4 * q + 3] = x.w;
        }
    };
    const int span_g = span_of(p.max_seqlen);
    load_scores(int(rank) * span_g + tid * kRPer);
    const int T = seq_len(p, b);                    // the same for the whole cluster
    if (T <= p.topk) {                              // every position is kept
        if (rank == 0)
            for (int i = tid; i < p.topk; i += blockDim.x) {
                oi[i] = i < T ? i : -1;
                if (os) os[i] = -INFINITY;
            }
        return;
    }
    const int K = p.topk;
    const int span = span_of(T);
    const int lo = int(rank) * span, hi = min(T, lo + span);
    MLA_CHECK(span <= kRStep, p.status);
    const int i0 = lo + tid * kRPer;              // this thread's first position
    if (span != span_g) load_scores(i0);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        S.hist1[tid + k * 1024] = hv[k];
        S.sum2[tid + k * 1024] = 0;
        S.part[tid + k * 1024] = 0;
    }
    S.sum3[tid] = 0;
    if (tid < kRStep / 32) S.kept[tid] = 0;
    if (tid < 8) sh[40 + tid] = 0;                  // counters
    __syncthreads();
    cluster_arrive();                               // (1) every CTA's totals are zero ...
    find_bin_fast(S.hist1, kBins, K, sh, 0, rank);
    const int bin1 = sh[32], above1 = sh[33];
    uint32_t key[kRPer];
#pragma unroll
    for (int u = 0; u < kRPer; ++u) key[u] = okey(v[u]);
    // positions past the end: only in the thread that holds the end
    constexpr uint32_t kAll = (1u << kRPer) - 1u;
    const uint32_t valid = hi - i0 >= kRPer ? kAll : (hi > i0 ? (1u << (hi - i0)) - 1u : 0u);
    // level 2: the next 11 bits of the keys in bin1; in1 / g1 mark this
    // thread's keys in and above bin1
    uint32_t in1 = 0, g1 = 0;
#pragma unroll
    for (int u = 0; u < kRPer; ++u) {
        const uint32_t top = key[u] >> 21;
        const bool in = top == uint32_t(bin1) && ((valid >> u) & 1u);
        if (in) atomicAdd(&S.part[(key[u] >> 10) & (kBins - 1)], 1u);
        in1 |= uint32_t(in) << u;
        g1 |= uint32_t(top > uint32_t(bin1)) << u;
    }
    g1 &= valid;
    __syncthreads();
    cluster_wait();                                 // (1) ... before anyone adds into them
    {
        constexpr int own = kBins / kRC;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int i = tid + k * 1024;
            const unsigned c = S.part[i];
            if (c) dsmem_add(dsmem_addr(&S.sum2[i], uint32_t(i / own)), c);
        }
    }
    cluster_sync();                                 // (2) level-2 totals at their owners
    find_bin_fast(S.sum2, kBins, K - above1, sh, kBins / kRC, rank);
    const int bin2 = sh[32], above2 = sh[33], n_c = sh[34];
    MLA_CHECK(bin1 >= 0 && bin1 < kBins && bin2 >= 0 && bin2 < kBins, p.status);
    const uint32_t pre = (uint32_t(bin1) << 11) | uint32_t(bin2);
    int need_eq = K - above1 - above2;              // keys with prefix pre that are kept
    int gt_before = 0, keep_before = 0;
    uint32_t take;
    if (n_c <= kRCand) {
        // keys above the prefix (g) and sharing it (e): the keys above bin1,
        // and those of bin1 by their level-2 bin
        uint32_t g = g1, e = 0;
        if (in1) {
#pragma unroll
            for (int u = 0; u < kRPer; ++u)
                if ((in1 >> u) & 1u) {
                    const uint32_t l2 = (key[u] >> 10) & (kBins - 1);
                    g |= uint32_t(l2 > uint32_t(bin2)) << u;
                    e |= uint32_t(l2 == uint32_t(bin2)) << u;
                }
        }
        if (e) {
#pragma unroll
            for (int u = 0; u < kRPer; ++u)       // this CTA's candidates into its own row
                if ((e >> u) & 1u) {
                    const int j = atomicAdd(&sh[41], 1);
                    MLA_CHECK(j < kRCand, p.status);
                    if (j < kRCand) {
                        S.ckey[rank * kRCand + j] = key[u];
                        S.cpos[rank * kRCand + j] = i0 + u;
                    }
                }
        }
        const int tg = block_sum(__popc(g), &sh[40]);
        const int mine = min(sh[41], kRCand);
        // the row, its length and the count of keys above go to the other
        // CTAs, one remote store pair per thread
        if (tid < kRC * mine) {
            const uint32_t r = uint32_t(tid % kRC);
            const int j = tid / kRC;
            if (r != rank) {
                dsmem_st(dsmem_addr(&S.ckey[rank * kRCand + j], r), int(S.ckey[rank * kRCand + j]));
                dsmem_st(dsmem_addr(&S.cpos[rank * kRCand + j], r), S.cpos[rank * kRCand + j]);
            }
        }
        if (tid < kRC) {
            dsmem_st(dsmem_addr(&S.ccnt[rank], uint32_t(tid)), mine);
            dsmem_st(dsmem_addr(&S.cnts[2 * rank], uint32_t(tid)), tg);
        }
        cluster_sync();                             // (3) candidates and counts everywhere; last remote access
        // every CTA's candidate count and count of keys above, read at once
        int cc[kRC];
        int n = 0;
#pragma unroll
        for (int r = 0; r < kRC; ++r) {
            cc[r] = S.ccnt[r];
            n += cc[r];
            gt_before += r < int(rank) ? S.cnts[2 * r] : 0;
        }
        MLA_CHECK(n == n_c, p.status);
        // candidate c: entry c of the rows taken in order
        auto cand = [&](int c, uint32_t* k, int* pos) {
            int r = 0;
#pragma unroll
            for (int q = 0; q < kRC; ++q)
                if (r == q && c >= cc[q]) {
                    c -= cc[q];
                    r = q + 1;
                }
            const int i = min(r, kRC - 1) * kRCand + c;
            *k = S.ckey[i];
            *pos = S.cpos[i];
        };
        // warp w ranks candidates w and w + 32: lane l compares them with
        // candidates l and l + 32 (larger key first, then lower position)
        const int lane = tid & 31, warp = tid >> 5;
        for (int c = warp; c < n; c += 32) {
            uint32_t kc, kj;
            int pc, pj;
            cand(c, &kc, &pc);
            int before = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = lane + 32 * h;
                bool beats = false;
                if (j < n) {
                    cand(j, &kj, &pj);
                    beats = kj > kc || (kj == kc && pj < pc);
                }
                before += __popc(__ballot_sync(0xffffffffu, beats));
            }
            if (lane == 0 && before < need_eq) {
                if (pc < lo) {
                    atomicAdd(&sh[42], 1);
                } else if (pc < hi) {
                    MLA_CHECK(pc - lo < kRStep, p.status);
                    atomicOr(&S.kept[(pc - lo) >> 5], 1u << ((pc - lo) & 31));
                }
            }
        }
        __syncthreads();
        keep_before = sh[42];
        take = g | (e & ((S.kept[(tid * kRPer) >> 5] >> ((tid * kRPer) & 31)) & kAll));
    } else {
        // level 3 over the keys with prefix pre (part's level-2 counts were
        // read by the pushes before barrier (2))
        S.part[tid] = 0;
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kRPer; ++u)
            if (((in1 >> u) & 1u) && ((key[u] >> 10) & (kBins - 1)) == uint32_t(bin2))
                atomicAdd(&S.part[key[u] & 1023u], 1u);
        __syncthreads();
        {
            constexpr int own = 1024 / kRC;
            const unsigned c = S.part[tid];
            if (c) dsmem_add(dsmem_addr(&S.sum3[tid], uint32_t(tid / own)), c);
        }
        cluster_sync();                             // (3) level-3 totals at their owners
        find_bin_fast(S.sum3, 1024, need_eq, sh, 1024 / kRC, rank);
        const int bin3 = sh[32], above3 = sh[33], n_eq = sh[34];
        MLA_CHECK(bin3 >= 0 && bin3 < 1024, p.status);
        const uint32_t kth = (pre << 10) | uint32_t(bin3);
        need_eq -= above3;
        uint32_t g = 0, e = 0;
#pragma unroll
        for (int u = 0; u < kRPer; ++u) {
            g |= uint32_t(key[u] > kth) << u;
            e |= uint32_t(key[u] == kth) << u;
        }
        g &= valid;
        e &= valid;
        const int tg = block_sum(__popc(g), &sh[43]);
        const int te = block_sum(__popc(e), &sh[44]);
        if (tid < kRC) {
            dsmem_st(dsmem_addr(&S.cnts[2 * rank], uint32_t(tid)), tg);
            dsmem_st(dsmem_addr(&S.cnts[2 * rank + 1], uint32_t(tid)), te);
        }
        cluster_sync();                             // (4) all counts everywhere; last remote access
        int eq_before = 0;
        for (uint32_t r = 0; r < rank; ++r) {
            gt_before += S.cnts[2 * r];
            eq_before += S.cnts[2 * r + 1];
        }
        keep_before = min(eq_before, need_eq);
        take = g | e;
        if (n_eq != need_eq) {                      // equal keys: lowest positions first
            int e_total;
            int r = eq_before + block_excl_scan(__popc(e), sh, &e_total);
            uint32_t keep = 0;
            for (uint32_t m = e; m; m &= m - 1, ++r)
                if (r < need_eq) keep |= m & (~m + 1);
            take = g | keep;
        }
    }
    // output: this thread's kept positions at their place in ascending order
    int total;
    int o = gt_before + keep_before + block_excl_scan(__popc(take), sh, &total);
    if (take) {
#pragma unroll
        for (int u = 0; u < kRPer; ++u)
            if ((take >> u) & 1u) {
                if (o < K) {
                    oi[o] = i0 + u;
                    if (os) os[o] = okey_inv(key[u]);
                } else {
                    report(p.status, kStInvalid);   // cannot happen for consistent counts
                }
                ++o;
            }
    }
}

// ---------------------------------------------------------------------------
// DSA prefill: every token of a prompt scores its own visible history and
// keeps its own top-k (DSA post, eqs. (5), (6) per token; complexity section).
// Token i (position P+i, P = Tk - Tq) sees positions 0..P+i.
//
// Scoring (dsa_prefill_score_kernel): one CTA per block of 8 tokens, heavy
// (late) blocks first.  The block's 8 x 32 index queries are the N = 256
// columns of a tcgen05 tile (B operand, resident), 128 index keys the M rows
// (A operand, streamed by TMA through a 4-stage ring); two 256-column TMEM
// accumulators alternate.  Eight epilogue warps each take 32 keys x 4 tokens:
// ReLU per head, the token's head weights, the sum over the 32 heads, and a
// coalesced store of the visible scores.
// ---------------------------------------------------------------------------
constexpr int kPQ = 8;                               // tokens per CTA
constexpr int kPN = kPQ * kIndexHeads;               // 256 MMA columns
constexpr int kPStages = 4;
constexpr int kPQHalf = kPN * 64 * 2;                // 32 KB: 256 rows x 128 B
constexpr int kPThreads = 10 * 32;
constexpr size_t kPScoreSmem =
    1024 + 2 * size_t(kPQHalf) + size_t(kPStages) * kStageBytes + kPN * 4 + 256;
constexpr uint32_t kPIdesc = idesc_bf16_f32(128, kPN, false, false);

struct PrefillScoreParams {
    const float* w;          // [Tq][32]
    float* scores;           // [Tq][stride]
    int Tq, Tk, stride;
    long long wait_ns;
    int* status;
};

__global__ void __launch_bounds__(kPThreads, 1)
    dsa_prefill_score_kernel(const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap qmap,
                             const PrefillScoreParams p) {
    extern __shared__ uint8_t psm_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(psm_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* qsm = sm;                                        // [2][256 rows][64]
    uint8_t* ring = sm + 2 * kPQHalf;                         // [stages][2][128 rows][64]
    float* wsm = reinterpret_cast<float*>(ring + kPStages * kStageBytes);   // [8][32]
    uint64_t* full = reinterpret_cast<uint64_t*>(wsm + kPN);
    uint64_t* empty = full + kPStages;
    uint64_t* afull = empty + kPStages;                       // [2] MMA -> epilogue
    uint64_t* aempty = afull + 2;                             // [2] epilogue -> MMA
    uint64_t* qfull = aempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(qfull + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nqb = (p.Tq + kPQ - 1) / kPQ;
    const int qb = nqb - 1 - int(blockIdx.x);                 // heavy blocks first
    const int i0 = qb * kPQ;
    const int P = p.Tk - p.Tq;
    const int last_key = P + min(i0 + kPQ - 1, p.Tq - 1);
    const int ntiles = last_key / kTile + 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&afull[i], 1);
            mbar_init(&aempty[i], 8);
        }
        mbar_init(qfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < kPN; i += blockDim.x) {
        const int t = i0 + i / kIndexHeads;
        wsm[i] = t < p.Tq ? p.w[int64_t(t) * kIndexHeads + (i % kIndexHeads)] : 0.f;
    }
    if (warp == 1) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&qmap);
            mbar_arrive_expect_tx(qfull, 2 * kPQHalf);
            for (int hf = 0; hf < 2; ++hf)
                tma_load_2d(qsm + hf * kPQHalf, &qmap, hf * 64, i0 * kIndexHeads, qfull);
            int filled[kPStages] = {0, 0, 0, 0};
            for (int j = 0; j < ntiles; ++j) {
                const int st = j % kPStages, r = j / kPStages;
                if (*abort_flag) break;
                if (r > 0 && !mbar_wait(&empty[st], (r - 1) & 1, p.wait_ns)) {
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[st], kStageBytes);
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_2d(ring + st * kStageBytes + hf * kAHalf, &kmap, hf * 64, j * kTile,
                                &full[st]);
                filled[st] = r + 1;
            }
            for (int i = 0; i < kPStages; ++i)
                if (filled[i] > 0 && !mbar_wait(&full[i], (filled[i] - 1) & 1, p.wait_ns))
                    report(p.status, kStTimeout);
            if (!mbar_wait(qfull, 0, p.wait_ns)) report(p.status, kStTimeout);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = mbar_wait(qfull, 0, p.wait_ns);
            const uint32_t qa = smem_u32(qsm), ra = smem_u32(ring);
            for (int j = 0; ok && j < ntiles; ++j) {
                const int st = j % kPStages, acc = j & 1;
                if (*abort_flag) { ok = false; break; }
                if (j >= 2 && !mbar_wait(&aempty[acc], ((j - 2) >> 1) & 1, p.wait_ns)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(&full[st], (j / kPStages) & 1, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = smem_desc_sw128(
                        ra + st * kStageBytes + (kk >> 2) * kAHalf + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd =
                        smem_desc_sw128(qa + (kk >> 2) * kPQHalf + (kk & 3) * 32, 16, 1024);
                    mma_bf16_ss(tmem + acc * kPN, ad, bd, kPIdesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(&empty[st]);
                mma_commit(&afull[acc]);
            }
            if (!ok) {
                report(p.status, kStTimeout);
                *abort_flag = 1;
            }
            // drain: wait for the last tile's MMAs before TMEM is released
            if (ntiles > 0) mbar_wait(&afull[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, p.wait_ns);
        }
    } else {
        // epilogue: warp w reads TMEM lanes of quadrant w%4 (keys) and the
        // columns of tokens 4*half..4*half+3 of the block
        const int quad = warp & 3, half = (warp - 2) >> 2;
        for (int j = 0; j < ntiles; ++j) {
            const int acc = j & 1;
            if (!*abort_flag && !mbar_wait(&afull[acc], (j >> 1) & 1, p.wait_ns)) {
                report(p.status, kStTimeout);
                *abort_flag = 1;
            }
            tc_fence_after();
            const int key = j * kTile + quad * 32 + lane;
            float sc[4];
#pragma unroll
            for (int tq = 0; tq < 4; ++tq) {
                const int col = (half * 4 + tq) * kIndexHeads;
                float v[32];
                tmem_ld32(tmem + (uint32_t(quad * 32) << 16) + acc * kPN + col, v);
                tmem_ld_wait();
                float a = 0.f;
#pragma unroll
                for (int hh = 0; hh < kIndexHeads; ++hh) a = fmaf(wsm[col + hh], fmaxf(v[hh], 0.f), a);
                sc[tq] = a;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&aempty[acc]);
#pragma unroll
            for (int tq = 0; tq < 4; ++tq) {
                const int i = i0 + half * 4 + tq;
                if (i < p.Tq && key <= P + i) p.scores[int64_t(i) * p.stride + key] = sc[tq];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// Per-token top-k (dsa_prefill_topk_kernel): one CTA of 1024 threads per
// token row, rows walked heavy-first by a persistent grid.  The same exact
// radix select as the decode top-k (11 + 11 + 10 key bits, then a pass in
// position order keeping the keys above the k-th and the lowest positions
// among keys equal to it), on one CTA: the row's visible scores stay in
// shared memory when they fit (16,384 positions), else each pass re-reads
// them from L2.
struct PrefillTopkParams {
    const float* scores;     // [Tq][stride]
    int Tq, Tk, stride, topk;
    int32_t* out_idx;        // [Tq][topk]
    float* out_scores;       // [Tq][topk] or null
    int* status;
};

constexpr size_t kPTopkSmem = size_t(kStep) * 4 + kBins * 4;

__global__ void __launch_bounds__(1024) dsa_prefill_topk_kernel(const PrefillTopkParams p) {
    extern __shared__ float4 ptopk_dyn[];
    float* vals = reinterpret_cast<float*>(ptopk_dyn);      // vals[u*1024 + tid]
    unsigned* hist = reinterpret_cast<unsigned*>(vals + kStep);
    __shared__ int sh[40];
    const int tid = threadIdx.x;
    const int P = p.Tk - p.Tq;
    const int K = p.topk;
    for (int rr = blockIdx.x; rr < p.Tq; rr += gridDim.x) {
        const int row = p.Tq - 1 - rr;
        const int n = P + row + 1;                           // visible positions
        int32_t* oi = p.out_idx + size_t(row) * K;
        float* os = p.out_scores ? p.out_scores + size_t(row) * K : nullptr;
        if (n <= K) {                                        // every position is kept
            for (int i = tid; i < K; i += blockDim.x) {
                oi[i] = i < n ? i : -1;
                if (os) os[i] = -INFINITY;
            }
            continue;
        }
        const float* s = p.scores + size_t(row) * p.stride;
        const bool resident = n <= kStep;
        auto stage = [&](int t0) {
            float v[kSelPer];
            load16(s, t0 + tid * kSelPer, n, v);
#pragma unroll
            for (int u = 0; u < kSelPer; ++u) vals[u * 1024 + tid] = v[u];
        MLA_CHECK((kSelPer - 1) * 1024 + tid < kStep, p.status);
        };
        __syncthreads();                                    // previous row fully consumed
        if (resident) stage(0);
        // histogram over the keys whose bits above `shift + width` equal `pre`
        auto level = [&](int shift, int nb, int width, uint32_t pre, bool all) {
            for (int i = tid; i < nb; i += blockDim.x) hist[i] = 0;
            __syncthreads();
            for (int t0 = 0; t0 < n; t0 += kStep) {
                if (!resident) {
                    stage(t0);
                    __syncthreads();
                }
                const int i0 = t0 + tid * kSelPer;
#pragma unroll
                for (int u = 0; u < kSelPer; ++u)
                    if (i0 + u < n) {
                        const uint32_t k = okey(vals[u * 1024 + tid]);
                        if (all || (k >> (shift + width)) == pre)
                            atomicAdd(&hist[(k >> shift) & uint32_t(nb - 1)], 1u);
                    }
                if (!resident) __syncthreads();
            }
            __syncthreads();
        };
        level(21, kBins, 11, 0, true);
        int bin1, above1;
        find_bin(hist, kBins, K, sh, &bin1, &above1);
        level(10, kBins, 11, uint32_t(bin1), false);
        int bin2, above2;
        find_bin(hist, kBins, K - above1, sh, &bin2, &above2);
        const uint32_t pre = (uint32_t(bin1) << 11) | uint32_t(bin2);
        level(0, 1024, 10, pre, false);
        int bin3, above3;
        find_bin(hist, 1024, K - above1 - above2, sh, &bin3, &above3);
        const uint32_t kth = (pre << 10) | uint32_t(bin3);
        const int need_eq = K - above1 - above2 - above3;
        const bool all_eq = int(hist[bin3]) == need_eq;
        // emit in position order
        int out = 0, eq_seen = 0;
        for (int t0 = 0; t0 < n; t0 += kStep) {
            if (!resident) {
                __syncthreads();
                stage(t0);
                __syncthreads();
            }
            const int i0 = t0 + tid * kSelPer;
            uint32_t g = 0, e = 0;
#pragma unroll
            for (int u = 0; u < kSelPer; ++u)
                if (i0 + u < n) {
                    const uint32_t k = okey(vals[u * 1024 + tid]);
                    g |= uint32_t(k > kth) << u;
                    e |= uint32_t(k == kth) << u;
                }
            uint32_t keep = e;
            if (!all_eq) {
                int e_total;
                int r = eq_seen + block_excl_scan(__popc(e), sh, &e_total);
                keep = 0;
                for (uint32_t m = e; m; m &= m - 1, ++r)
                    if (r < need_eq) keep |= m & (~m + 1);
                eq_seen += e_total;
            }
            const uint32_t take = g | keep;
            int total;
            int o = out + block_excl_scan(__popc(take), sh, &total);
            for (uint32_t m = take; m; m &= m - 1, ++o) {
                const int u = __ffs(m) - 1;
                if (o < K) {
                    oi[o] = i0 + u;
                    if (os) os[o] = vals[u * 1024 + tid];
                } else {
                    report(p.status, kStInvalid);
                }
            }
            out += total;
        }
    }
}

// ---------------------------------------------------------------------------
// E4M3 quantisation (the FP8 index key of the DSA post's cache section: 128
// one-byte features and one fp32 scale per position).  One warp per row of
// 128 values, four per lane: amax by shuffles, scale = amax/448, codes =
// e4m3(x * (448/amax)) rounded to nearest even with saturation.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE,
                                                              __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE,
                                                              __NV_E4M3);
    return uint32_t(lo) | (uint32_t(hi) << 16);
}

// codes [rows][128], scale [rows]; `wq`/`w`: when given, wq[row] = w[row] * scale
// (the index queries' scales folded into the head weights).
__global__ void __launch_bounds__(256) quantize_rows128_kernel(const uint16_t* x, uint8_t* codes,
                                                               float* scale, int64_t rows,
                                                               const float* w, float* wq) {
    const int lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const uint2 v = *reinterpret_cast<const uint2*>(x + row * 128 + lane * 4);
    const float f0 = bf_lo(v.x), f1 = bf_hi(v.x), f2 = bf_lo(v.y), f3 = bf_hi(v.y);
    float amax = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    uint32_t c = 0;
    float sc = 0.f;
    if (amax > 0.f) {
        const float inv = 448.0f / amax;
        sc = amax / 448.0f;
        c = e4m3x4(f0 * inv, f1 * inv, f2 * inv, f3 * inv);
    }
    *reinterpret_cast<uint32_t*>(codes + row * 128 + lane * 4) = c;
    if (lane == 0) {
        scale[row] = sc;
        if (wq) wq[row] = w[row] * sc;
    }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Score rows start on 16-byte boundaries so the top-k passes can load float4.
int score_stride(int max_seqlen) { return (max_seqlen + 3) & ~3; }

}  // namespace

IndexPlan plan_index(int B, int max_seqlen, bool fp8) {
    // scores | level-1 histograms | tile table | claim counters | FP8: query
    // codes, scales, folded weights
    IndexPlan p{};
    p.scores_off = 0;
    p.hist_off = align256(size_t(B) * score_stride(max_seqlen) * 4);
    p.tiles_off = p.hist_off + align256(size_t(B) * kBins * 4);
    p.claims_off = p.tiles_off + align256(size_t(B + 1) * 4);
    p.total = p.claims_off + align256(size_t(B) * 4);
    if (fp8) {
        p.q8_off = p.total;
        p.qs_off = p.q8_off + align256(size_t(B) * kIndexHeads * 128);
        p.wq_off = p.qs_off + align256(size_t(B) * kIndexHeads * 4);
        p.total = p.wq_off + align256(size_t(B) * kIndexHeads * 4);
    }
    return p;
}

cudaError_t launch_quantize_rows_e4m3(const uint16_t* x, uint8_t* codes, float* scale,
                                      int64_t rows, int cols, cudaStream_t st) {
    if (cols != 128) return cudaErrorInvalidValue;
    if (rows == 0) return cudaSuccess;
    quantize_rows128_kernel<<<unsigned((rows + 7) / 8), 256, 0, st>>>(x, codes, scale, rows,
                                                                       nullptr, nullptr);
    return cudaGetLastError();
}

// Tile list (and cleared level-1 bins), scores, top-k: three kernels, each
// launched programmatically dependent on the one before it, so it is placed
// on the SMs its predecessor leaves and does its set-up while that
// predecessor finishes; every one waits on the device (grid_dep_wait) before
// it touches global memory.
template <bool kFp8>
static cudaError_t launch_score_topk(const IndexArgs& a, const CUtensorMap& kmap,
                                     const CUtensorMap& qmap, const ScoreParams& p,
                                     const DeviceInfo& dev, const KernelTimer& tm,
                                     cudaStream_t st) {
    const int zero_blocks = int(std::min<int64_t>(1024, (int64_t(a.B) * kBins + 16383) / 16384));
    cudaError_t e = launch_after_prev(dsa_tiles_kernel, dim3(1 + zero_blocks), dim3(1024), 0, st,
                                      a.cu, a.B, a.max_seqlen, a.total_keys, a.topk,
                                      const_cast<int*>(p.tile_start), p.hist, p.claim, dev.sms,
                                      dev.status);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dsa_score_kernel<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(ScoreCfg<kFp8>::kSmem));
    if (e != cudaSuccess) return e;
    if (tm.begin) cudaEventRecord(tm.begin, st);
    e = launch_after_prev(dsa_score_kernel<kFp8>, dim3(dev.sms), dim3(kScoreThreads),
                          ScoreCfg<kFp8>::kSmem, st, kmap, qmap, p);
    if (tm.end) cudaEventRecord(tm.end, st);
    if (e != cudaSuccess) return e;
    TopkParams tp{p.scores, p.hist, a.cu, a.max_seqlen, p.stride, a.topk,
                  a.total_keys, a.topk_idx, a.topk_scores, dev.status};
    // every CTA's range fits in registers (16 positions a thread) up to
    // 8 x 16,384 positions; longer sequences take the general kernel
    const bool regs = int64_t(a.max_seqlen) <= int64_t(kRC) * kRStep;
    void (*const topk_kernel)(TopkParams) = regs ? dsa_topk_regs_kernel : dsa_topk_cluster_kernel;
    const size_t topk_smem = regs ? sizeof(RegsSmem) : kTopkSmem;
    const int cluster = regs ? kRC : kCluster;
    e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(topk_smem));
    if (e != cudaSuccess) return e;
    if (cluster > 8) {
        e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    {
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cluster, a.B);
        cfg.blockDim = dim3(1024);
        cfg.dynamicSmemBytes = topk_smem;
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, topk_kernel, tp);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_index_topk(const IndexArgs& a, const IndexPlan& pl, const DeviceInfo& dev,
                              const Knobs& kn, const KernelTimer& tm, cudaStream_t st) {
    static_assert(ScoreCfg<false>::kSmem <= 227 * 1024 && ScoreCfg<true>::kSmem <= 227 * 1024,
                  "shared memory budget");
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    float* scores = reinterpret_cast<float*>(ws + pl.scores_off);
    unsigned* hist = reinterpret_cast<unsigned*>(ws + pl.hist_off);
    int* tiles = reinterpret_cast<int*>(ws + pl.tiles_off);
    int* claims = reinterpret_cast<int*>(ws + pl.claims_off);

    CUtensorMap kmap, qmap;
    const uint64_t rows = a.total_keys > 0 ? uint64_t(a.total_keys) : 1;
    cudaError_t e = encode_tmap_2d_bf16(&kmap, a.index_k, kIndexDim, rows, kIndexDim * 2, 64, kTile);
    if (e != cudaSuccess) return e;
    e = encode_tmap_2d_bf16(&qmap, a.index_q, kIndexDim, uint64_t(a.B) * kIndexHeads,
                            kIndexDim * 2, 64, kIndexHeads);
    if (e != cudaSuccess) return e;

    ScoreParams p{a.index_k, a.total_keys, a.w, nullptr, a.cu, tiles, claims, scores, hist, a.B,
                  score_stride(a.max_seqlen), kn.wait_limit_ns, dev.status};
    return launch_score_topk<false>(a, kmap, qmap, p, dev, tm, st);
}

size_t prefill_index_ws(int Tq, int Tk) {
    return align256(size_t(Tq) * score_stride(Tk) * 4);
}

cudaError_t launch_prefill_index_topk(const PrefillIndexArgs& a, const DeviceInfo& dev,
                                      const Knobs& kn, const KernelTimer& tm, cudaStream_t st) {
    static_assert(kPScoreSmem <= 227 * 1024, "shared memory budget");
    float* scores = static_cast<float*>(a.ws);
    CUtensorMap kmap, qmap;
    cudaError_t e = encode_tmap_2d_bf16(&kmap, a.index_k, kIndexDim, uint64_t(a.Tk),
                                        kIndexDim * 2, 64, kTile);
    if (e != cudaSuccess) return e;
    e = encode_tmap_2d_bf16(&qmap, a.index_q, kIndexDim, uint64_t(a.Tq) * kIndexHeads,
                            kIndexDim * 2, 64, kPN);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dsa_prefill_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kPScoreSmem));
    if (e != cudaSuccess) return e;
    PrefillScoreParams sp{a.w, scores, a.Tq, a.Tk, score_stride(a.Tk), kn.wait_limit_ns,
                          dev.status};
    if (tm.begin) cudaEventRecord(tm.begin, st);
    dsa_prefill_score_kernel<<<(a.Tq + kPQ - 1) / kPQ, kPThreads, kPScoreSmem, st>>>(kmap, qmap,
                                                                                   sp);
    if (tm.end) cudaEventRecord(tm.end, st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dsa_prefill_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kPTopkSmem));
    if (e != cudaSuccess) return e;
    PrefillTopkParams tp{scores, a.Tq, a.Tk, score_stride(a.Tk), a.topk, a.topk_idx, a.topk_scores,
                         dev.status};
    const int grid = a.Tq < 2 * dev.sms ? a.Tq : 2 * dev.sms;
    dsa_prefill_topk_kernel<<<grid, 1024, kPTopkSmem, st>>>(tp);
    return cudaGetLastError();
}

cudaError_t launch_index_topk_fp8(const IndexArgs& a, const IndexFp8Args& f, const IndexPlan& pl,
                                  const DeviceInfo& dev, const Knobs& kn, const KernelTimer& tm,
                                  cudaStream_t st) {
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    float* scores = reinterpret_cast<float*>(ws + pl.scores_off);
    unsigned* hist = reinterpret_cast<unsigned*>(ws + pl.hist_off);
    int* tiles = reinterpret_cast<int*>(ws + pl.tiles_off);
    int* claims = reinterpret_cast<int*>(ws + pl.claims_off);
    uint8_t* q8 = ws + pl.q8_off;
    float* qs = reinterpret_cast<float*>(ws + pl.qs_off);
    float* wq = reinterpret_cast<float*>(ws + pl.wq_off);
    // queries: one scale per (sequence, head), folded into that head's weight
    const int64_t qrows = int64_t(a.B) * kIndexHeads;
    quantize_rows128_kernel<<<unsigned((qrows + 7) / 8), 256, 0, st>>>(a.index_q, q8, qs, qrows,
                                                                        a.w, wq);
    CUtensorMap kmap, qmap;
    const uint64_t rows = a.total_keys > 0 ? uint64_t(a.total_keys) : 1;
    cudaError_t e = encode_tmap_2d_u8(&kmap, f.k8, 128, rows, 128, 128, kTile);
    if (e != cudaSuccess) return e;
    e = encode_tmap_2d_u8(&qmap, q8, 128, uint64_t(qrows), 128, 128, kIndexHeads);
    if (e != cudaSuccess) return e;
    ScoreParams p{f.k8, a.total_keys, wq, f.kscale, a.cu, tiles, claims, scores, hist, a.B,
                  score_stride(a.max_seqlen), kn.wait_limit_ns, dev.status};
    return launch_score_topk<true>(a, kmap, qmap, p, dev, tm, st);
}

}  // namespace mla
