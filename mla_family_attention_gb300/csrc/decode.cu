// Split-KV gated MLA decode and DSA sparse decode for sm_103a.
//
// What it computes (Kimi K3 MLA forward in decode mode; K3.1 Gated DSA post,
// eqs. (9) and (10)): for every sequence b and head h,
//   z = sum_s softmax_s(scale * q.k_s) v_s over the visible positions s
//   out[b, h*128+d] = z_d * sigmoid(gate[b, h*128+d])
// where the visible positions are all T_b cached positions (decode) or the
// selected ones (sparse decode).
//
// Design.  Decode reads 640 bytes (a 384-byte key row and a 256-byte value
// row) per position and head and does 320 multiply-adds on them: about one
// flop per byte, so the kernel is bound by HBM bandwidth and the work is done
// on the CUDA cores.  A persistent grid of one CTA per SM walks a list of work
// items, each a chunk of up to `chunk` positions of one (sequence, head):
//   - warp 0 is the producer: one elected lane issues bulk (TMA) copies of
//     64 contiguous key rows and value rows per pipeline stage into shared
//     memory (four stages), completing on an mbarrier; for sparse decode four
//     producer warps gather the selected rows with 16-byte cp.async copies
//     (a bulk copy per 384- or 256-byte row is too small to keep HBM busy),
//     each thread arriving on the stage's mbarrier when its copies land;
//   - eight consumer warps split each stage into 8-lane groups, one position
//     per group at a time: every lane dots 24 query features with its three
//     16-byte slices of the key row, three xor-shuffles finish the score,
//     and an online softmax (running max and sum in the log2 domain) folds
//     the position's value slice into 16 accumulators per lane;
//   - at the end of an item the 32 group states are merged (shuffles, then
//     shared memory) into one unnormalised partial (acc[128], max, sum)
//     written to the workspace.
// A second kernel merges the partials of each (b,h) by log-sum-exp in a fixed
// order and applies the sigmoid gate, so results do not depend on timing.
//
// Every wait on an mbarrier is bounded; when one runs out the kernel records
// MLA_ERR_TIMEOUT in the status word, skips the rest of its work, waits (again
// bounded) for the copies it has in flight and returns.
#include <cuda_bf16.h>

#define MLA_FILE_ID 1   // site ids of the bounds-checked debug build
#include "common.cuh"
#include "kernels.h"

namespace mla {
namespace {

constexpr int kKRow = kDqk * 2;                 // 384 bytes
constexpr int kVRow = kDv * 2;                  // 256 bytes
constexpr int kDenseSP = 64;                    // positions per dense pipeline stage
#ifndef MLA_SPARSE_STAGE_POS
#define MLA_SPARSE_STAGE_POS 64                 // positions per sparse pipeline stage
#endif
#ifndef MLA_SPARSE_PRODUCER_WARPS
#define MLA_SPARSE_PRODUCER_WARPS 8             // gathering warps of the sparse decode
#endif
#ifndef MLA_SPARSE_CONSUMER_WARPS
#define MLA_SPARSE_CONSUMER_WARPS 8             // consumer warps of the sparse decode
#endif
// Dense decode: one producer warp (bulk copies).  Sparse decode: four
// producer warps (16-byte cp.async gathers), completing on the same barrier.
// Dense decode: four stages of 64 streamed positions (160 KB; B=32, H=96,
// T=8192 measured 7.49 / 7.52 / 6.92 TB/s with 3 / 4 / 5 stages).  Sparse
// decode: about 200 KB in smaller stages, because gathered rows take longer
// to arrive and a stage is only complete when its slowest row has landed.
#ifndef MLA_DENSE_STAGES
#define MLA_DENSE_STAGES 4
#endif
template <bool kSparse>
struct Roles {
    static constexpr int kProducerWarps = kSparse ? MLA_SPARSE_PRODUCER_WARPS : 1;
    static constexpr int kPT = 32 * kProducerWarps;            // producer threads
    static constexpr int kConsumerWarps = kSparse ? MLA_SPARSE_CONSUMER_WARPS : 8;
    static constexpr int kGroups = kConsumerWarps * 4;       // 8-lane groups
    static constexpr int kThreads = 32 * (kProducerWarps + kConsumerWarps);
    static constexpr int kFullArrivals = kSparse ? 32 * kProducerWarps : 1;
    static constexpr int kSP = kSparse ? MLA_SPARSE_STAGE_POS : kDenseSP;
    static constexpr int kStages = kSparse ? (200 * 1024) / (kSP * (kDqk + kDv) * 2) : MLA_DENSE_STAGES;
    static constexpr int kKStage = kSP * kDqk * 2;
    static constexpr int kVStage = kSP * kDv * 2;
    static constexpr int kPPG = kSP / kGroups;                // positions per group per stage
    static constexpr int kMergeFloats = kConsumerWarps * (kDv + 2);
};

constexpr float kLog2e = 1.4426950408889634f;

template <bool kSparse>
constexpr size_t smem_bytes() {
    using R = Roles<kSparse>;
    return size_t(R::kStages) * (R::kKStage + R::kVStage + kKRow) + R::kMergeFloats * 4 +
           2 * R::kStages * 8 + 16;
}

static_assert((Roles<true>::kSP * 24) % Roles<true>::kPT == 0 &&
                  (Roles<true>::kSP * 16) % Roles<true>::kPT == 0,
              "a stage's key and value pieces must split evenly over the producer threads");
static_assert(Roles<true>::kPPG * Roles<true>::kGroups == Roles<true>::kSP &&
                  Roles<false>::kPPG * Roles<false>::kGroups == Roles<false>::kSP &&
                  Roles<true>::kConsumerWarps >= 4,
              "stage must split evenly over groups; the merge takes four warps");

struct Params {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    SeqLayout seq;
    const int32_t* idx;      // sparse: [B,topk]
    int B, H, chunk, max_chunks, topk, max_seqlen;
    const int* item_start;   // dense: [B+1]
    float* part_acc;         // [slots][128]
    float* part_ml;          // [slots][2]
    float scale_log2;
    long long wait_ns;
    int stall_stage;
    int* status;
};

struct Item {
    int b, h, c;
    int64_t row0;   // cache row of position 0 of (b, h)
    int T;          // T_b
    int e0, e1;     // range of positions (dense) or index entries (sparse)
    int nst;        // pipeline stages in the item
};

template <bool kSparse>
__device__ __forceinline__ int stage_entry(const Item& w, int k) {
    return w.e0 + k * Roles<kSparse>::kSP;
}

// Work item `it` -> (b, h, chunk).  Dense items come from the prefix table
// item_start, heads fastest: concurrent CTAs stream different heads'
// contiguous chunks.  Sparse items are a (b, h, chunk) grid, chunk fastest:
// the selected rows of one head are scattered over its whole cache region
// (dozens of 2 MB pages), so concurrent CTAs share a few heads' pages
// instead of each walking its own head's pages (translation-cache reach).
template <bool kSparse>
__device__ __forceinline__ Item item_of(const Params& p, int it) {
    Item r;
    if (kSparse) {
        const int nch = (p.topk + p.chunk - 1) / p.chunk;
        r.b = it / (p.H * nch);
        const int rem = it - r.b * p.H * nch;
        r.h = rem / nch;
        r.c = rem - r.h * nch;
        r.T = static_cast<int>(p.seq.len(r.b));
        r.row0 = p.seq.row0(r.b, r.h, p.H, r.T);
        r.e0 = r.c * p.chunk;
        r.e1 = min(p.topk, r.e0 + p.chunk);
        r.nst = (r.e1 - r.e0 + Roles<kSparse>::kSP - 1) / Roles<kSparse>::kSP;
    } else {
        int lo = 0, hi = p.B;   // largest b with item_start[b] <= it
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.item_start[mid] <= it) lo = mid; else hi = mid;
        }
        r.b = lo;
        r.T = static_cast<int>(p.seq.len(r.b));
        const int rem = it - p.item_start[r.b];
        r.c = rem / p.H;
        r.h = rem - r.c * p.H;
        r.row0 = p.seq.row0(r.b, r.h, p.H, r.T);
        r.e0 = r.c * p.chunk;
        r.e1 = min(r.T, r.e0 + p.chunk);
        r.nst = (r.e1 - r.e0 + Roles<kSparse>::kSP - 1) / Roles<kSparse>::kSP;
    }
    return r;
}

template <bool kSparse>
__device__ __forceinline__ int total_items(const Params& p) {
    if (kSparse) return p.B * p.H * ((p.topk + p.chunk - 1) / p.chunk);
    return p.item_start[p.B];
}

__device__ __forceinline__ bool valid_pos(int s, int T) { return s >= 0 && s < T; }

template <bool kSparse>
__global__ void __launch_bounds__(Roles<kSparse>::kThreads, 1)
    decode_partial_kernel(const Params p) {
    using R = Roles<kSparse>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* ks = smem;                                        // [stages][64][384]
    uint8_t* vs = smem + R::kStages * R::kKStage;                    // [stages][64][256]
    uint8_t* qs = vs + R::kStages * R::kVStage;                // [stages][384]: query row of
                                                               // the item a stage starts
    float* red = reinterpret_cast<float*>(qs + R::kStages * kKRow);   // [8][130]
    uint64_t* full = reinterpret_cast<uint64_t*>(red + R::kMergeFloats);
    uint64_t* empty = full + R::kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + R::kStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < R::kStages; ++s) {
            mbar_init(&full[s], R::kFullArrivals);
            mbar_init(&empty[s], R::kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
        grid_dep_trigger();
    }
    grid_dep_wait();   // the item table (dense) or the selections (sparse) of earlier kernels
    __syncthreads();

    const int n_items = total_items<kSparse>(p);

    if (!kSparse && warp == 0) {
        // ------------------------- producer (dense) -------------------------
        const uint64_t policy = l2_evict_first_policy();
        int it = 0;                    // pipeline stages issued (or skipped) so far
        int filled[R::kStages];           // stage count of the last real fill per slot (+1)
        for (int s = 0; s < R::kStages; ++s) filled[s] = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const Item w = item_of<kSparse>(p, item);
            for (int st = 0; st < w.nst; ++st, ++it) {
                const int e = stage_entry<kSparse>(w, st);
                const int slot = it % R::kStages;
                const int round = it / R::kStages;
                if (*abort_flag) { ok = false; break; }
                if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, p.wait_ns)) {
                    if (lane == 0) report(p.status, kStTimeout);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                if (it == p.stall_stage) continue;   // test hook: withhold this stage
                const int n = min(R::kSP, w.e1 - e);
                MLA_CHECK(slot < R::kStages && n >= 1 && n <= R::kSP && w.row0 >= 0, p.status);
                if (lane == 0) {
                    const int64_t row = w.row0 + e;
                    mbar_arrive_expect_tx(&full[slot], n * (kKRow + kVRow) + (st == 0 ? kKRow : 0));
                    if (st == 0)                      // the item's query row rides along
                        bulk_load(qs + slot * kKRow, p.q + (int64_t(w.b) * p.H + w.h) * kDqk,
                                  kKRow, &full[slot], policy);
                    bulk_load(ks + slot * R::kKStage, p.k + row * kDqk, n * kKRow, &full[slot],
                              policy);
                    bulk_load(vs + slot * R::kVStage, p.v + row * kDv, n * kVRow, &full[slot],
                              policy);
                }
                filled[slot] = round + 1;
            }
        }
        // Drain: every copy this CTA issued lands before the CTA may exit.
        for (int s = 0; s < R::kStages; ++s) {
            if (filled[s] > 0 && !mbar_wait(&full[s], (filled[s] - 1) & 1, p.wait_ns)) {
                if (lane == 0) report(p.status, kStTimeout);
            }
        }
        return;
    }
    if (kSparse && warp < R::kProducerWarps) {
        // ------------------------ producers (sparse) ------------------------
        // kPT threads gather the selected rows in 16-byte pieces: a stage holds
        // 64 x 24 key pieces and 64 x 16 value pieces; consecutive threads take
        // consecutive pieces of a row.  Each thread's copies complete with one
        // arrival on the stage's barrier (expected count kPT).
        const int pt = threadIdx.x;
        const uint8_t* kb = reinterpret_cast<const uint8_t*>(p.k);
        const uint8_t* vb = reinterpret_cast<const uint8_t*>(p.v);
        int it = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const Item w = item_of<kSparse>(p, item);
            const int64_t rbase = w.row0;
            for (int st = 0; st < w.nst; ++st, ++it) {
                const int e = stage_entry<kSparse>(w, st);
                const int slot = it % R::kStages;
                const int round = it / R::kStages;
                if (*abort_flag) { ok = false; break; }
                // Selections of this stage are loaded before waiting for the
                // slot, so their latency hides behind the wait.
                const int n = min(R::kSP, w.e1 - e);
                const int32_t* ix = p.idx + int64_t(w.b) * p.topk + e;
                int selk[R::kSP * 24 / R::kPT], selv[R::kSP * 16 / R::kPT];
#pragma unroll
                for (int i = 0; i < R::kSP * 24 / R::kPT; ++i) {
                    const int j = (pt + R::kPT * i) / 24;
                    selk[i] = j < n ? ix[j] : -1;
                }
#pragma unroll
                for (int i = 0; i < R::kSP * 16 / R::kPT; ++i) {
                    const int j = (pt + R::kPT * i) >> 4;
                    selv[i] = j < n ? ix[j] : -1;
                }
                if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, p.wait_ns)) {
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                if (it == p.stall_stage) continue;   // test hook: withhold this stage
                if (st == 0 && pt < 24)               // the item's query row rides along
                    cp_async16(qs + slot * kKRow + pt * 16,
                               reinterpret_cast<const uint8_t*>(p.q) +
                                   (int64_t(w.b) * p.H + w.h) * kKRow + pt * 16);
#pragma unroll
                for (int i = 0; i < R::kSP * 24 / R::kPT; ++i) {
                    const int c = pt + R::kPT * i, j = c / 24, off = (c - j * 24) * 16;
                    MLA_CHECK(slot < R::kStages && j < R::kSP && off + 16 <= kKRow, p.status);
                    if (valid_pos(selk[i], w.T))
                        cp_async16(ks + slot * R::kKStage + j * kKRow + off,
                                   kb + (rbase + selk[i]) * kKRow + off);
                    else if (selk[i] < -1 || selk[i] >= w.T)
                        report(p.status, kStBadIndex);
                }
#pragma unroll
                for (int i = 0; i < R::kSP * 16 / R::kPT; ++i) {
                    const int c = pt + R::kPT * i, j = c >> 4, off = (c & 15) * 16;
                    MLA_CHECK(j < R::kSP && off + 16 <= kVRow, p.status);
                    if (valid_pos(selv[i], w.T))
                        cp_async16(vs + slot * R::kVStage + j * kVRow + off,
                                   vb + (rbase + selv[i]) * kVRow + off);
                }
                cp_async_arrive_noinc(&full[slot]);
            }
        }
        cp_async_wait_all();   // nothing this thread started is still in flight at exit
        return;
    }

    // ------------------------------ consumers ------------------------------
    const int cw = warp - R::kProducerWarps;   // consumer warp 0..7
    const int g = cw * 4 + (lane >> 3);      // group 0..31
    const int j = lane & 7;                  // lane within the group
    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const Item w = item_of<kSparse>(p, item);
        // query slices of this lane (features 8j.., 64+8j.., 128+8j..), read
        // from the first stage of the item once it has landed
        float qf[24];
        float m = -INFINITY, l = 0.f, acc[16];
#pragma unroll
        for (int d = 0; d < 16; ++d) acc[d] = 0.f;

        for (int st = 0; st < w.nst; ++st, ++it) {
            const int e = stage_entry<kSparse>(w, st);
            const int slot = it % R::kStages;
            const int round = it / R::kStages;
            // Which of this group's positions hold data: known before the
            // wait (sparse: the selection is read while the copies land).
            const int n = min(R::kSP, w.e1 - e);
            bool ok[R::kPPG];
#pragma unroll
            for (int r = 0; r < R::kPPG; ++r) {
                const int pos = g + R::kGroups * r;
                ok[r] = pos < n;
                if (kSparse && ok[r])
                    ok[r] = valid_pos(p.idx[int64_t(w.b) * p.topk + e + pos], w.T);
            }
            bool have = !*abort_flag;
            if (have && !mbar_wait(&full[slot], round & 1, p.wait_ns)) {
                if (lane == 0) report(p.status, kStTimeout);
                *abort_flag = 1;
                have = false;
            }
            have = __all_sync(0xffffffffu, have);
            if (have && st == 0) {
                const uint4* qp = reinterpret_cast<const uint4*>(qs + slot * kKRow);
#pragma unroll
                for (int c = 0; c < 3; ++c) {
                    const uint4 u = qp[c * 8 + j];
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        qf[c * 8 + 2 * t] = bf_lo(wd[t]) * p.scale_log2;
                        qf[c * 8 + 2 * t + 1] = bf_hi(wd[t]) * p.scale_log2;
                    }
                }
            }
            if (have) {
                const uint8_t* kst = ks + slot * R::kKStage;
                const uint8_t* vst = vs + slot * R::kVStage;
                float s[R::kPPG];
#pragma unroll
                for (int r = 0; r < R::kPPG; ++r) {
                    const int pos = g + R::kGroups * r;
                    MLA_CHECK(pos < R::kSP && slot < R::kStages, p.status);
                    float dot = 0.f;
                    if (ok[r]) {
                        const uint8_t* kr = kst + pos * kKRow;
#pragma unroll
                        for (int c = 0; c < 3; ++c) {
                            const uint4 u =
                                *reinterpret_cast<const uint4*>(kr + (c * 8 + j) * 16);
                            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                dot = fmaf(qf[c * 8 + 2 * t], bf_lo(wd[t]), dot);
                                dot = fmaf(qf[c * 8 + 2 * t + 1], bf_hi(wd[t]), dot);
                            }
                        }
                    }
                    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
                    dot += __shfl_xor_sync(0xffffffffu, dot, 4);
                    s[r] = ok[r] ? dot : -INFINITY;
                }
                float mn = m;
#pragma unroll
                for (int r = 0; r < R::kPPG; ++r) mn = fmaxf(mn, s[r]);
                if (mn != -INFINITY) {
                    const float alpha = ex2(m - mn);    // m = -inf -> 0
                    l *= alpha;
#pragma unroll
                    for (int d = 0; d < 16; ++d) acc[d] *= alpha;
#pragma unroll
                    for (int r = 0; r < R::kPPG; ++r) {
                        if (ok[r]) {
                            const float pr = ex2(s[r] - mn);
                            l += pr;
                            const uint8_t* vr = vst + (g + R::kGroups * r) * kVRow;
#pragma unroll
                            for (int c = 0; c < 2; ++c) {
                                const uint4 u =
                                    *reinterpret_cast<const uint4*>(vr + (c * 8 + j) * 16);
                                const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                                for (int t = 0; t < 4; ++t) {
                                    acc[c * 8 + 2 * t] = fmaf(pr, bf_lo(wd[t]), acc[c * 8 + 2 * t]);
                                    acc[c * 8 + 2 * t + 1] =
                                        fmaf(pr, bf_hi(wd[t]), acc[c * 8 + 2 * t + 1]);
                                }
                            }
                        }
                    }
                    m = mn;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }

        // ---- merge the 4 groups of this warp (butterfly over lanes 8, 16) ----
#pragma unroll
        for (int off = 8; off <= 16; off <<= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
            const float mn = fmaxf(m, m2);
            const float a1 = mn == -INFINITY ? 0.f : ex2(m - mn);
            const float a2 = mn == -INFINITY ? 0.f : ex2(m2 - mn);
            l = l * a1 + l2 * a2;
#pragma unroll
            for (int d = 0; d < 16; ++d) {
                const float o = __shfl_xor_sync(0xffffffffu, acc[d], off);
                acc[d] = acc[d] * a1 + o * a2;
            }
            m = mn;
        }
        // lanes 0..7 hold the warp's state: features 8j..8j+7 and 64+8j..64+8j+7
        float* rw = red + cw * (kDv + 2);
        if (lane < 8) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                rw[8 * j + t] = acc[t];
                rw[64 + 8 * j + t] = acc[8 + t];
            }
        }
        if (lane == 0) {
            rw[kDv] = m;
            rw[kDv + 1] = l;
        }
        named_bar_sync(1, 32 * R::kConsumerWarps);
        const bool aborted = *abort_flag != 0;
        if (cw < 4 && !aborted) {
            const int d = cw * 32 + lane;     // one feature per thread
            float mx = -INFINITY;
#pragma unroll
            for (int u = 0; u < R::kConsumerWarps; ++u) mx = fmaxf(mx, red[u * (kDv + 2) + kDv]);
            float a = 0.f, ls = 0.f;
            if (mx != -INFINITY) {
#pragma unroll
                for (int u = 0; u < R::kConsumerWarps; ++u) {
                    const float wgt = ex2(red[u * (kDv + 2) + kDv] - mx);
                    a += wgt * red[u * (kDv + 2) + d];
                    ls += wgt * red[u * (kDv + 2) + kDv + 1];
                }
            }
            MLA_CHECK(w.b >= 0 && w.b < p.B && w.h >= 0 && w.h < p.H && w.c >= 0 &&
                          w.c < p.max_chunks && d < kDv, p.status);
            const int64_t slotid = (int64_t(w.b) * p.H + w.h) * p.max_chunks + w.c;
            p.part_acc[slotid * kDv + d] = a;
            if (d == 0) {
                p.part_ml[slotid * 2] = mx;
                p.part_ml[slotid * 2 + 1] = ls;
            }
        }
        named_bar_sync(1, 32 * R::kConsumerWarps);
    }
}

// Per-sequence work-item prefix: item_start[b] = sum_{b'<b} H*ceil(T_b'/chunk).
// A sequence with T_b outside [1, max_seqlen] gets no items and is reported.
__global__ void __launch_bounds__(1024) decode_items_kernel(const SeqLayout seq, int B, int H,
                                                            int chunk, int max_seqlen,
                                                            int* item_start, int* status) {
    __shared__ int warp_sums[32];
    if (threadIdx.x == 0) grid_dep_trigger();
    grid_dep_wait();
    const int per = (B + blockDim.x - 1) / blockDim.x;
    const int b0 = min(B, int(threadIdx.x) * per), b1 = min(B, b0 + per);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
        const int64_t T = seq.len(b);
        if (T < 1 || T > max_seqlen) { report(status, kStInvalid); continue; }
        local += H * int((T + chunk - 1) / chunk);
    }
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
        warp_sums[lane] = v;   // inclusive over warps
    }
    __syncthreads();
    int run = incl - local + (warp > 0 ? warp_sums[warp - 1] : 0);
    for (int b = b0; b < b1; ++b) {
        item_start[b] = run;
        const int64_t T = seq.len(b);
        if (T >= 1 && T <= max_seqlen) run += H * int((T + chunk - 1) / chunk);
    }
    if (threadIdx.x == blockDim.x - 1) item_start[B] = run;
}

// One warp per (b,h): log-sum-exp merge of the chunk partials, then the gate.
__global__ void __launch_bounds__(256) decode_merge_kernel(
    const float* part_acc, const float* part_ml, const SeqLayout seq, const uint16_t* gate,
    uint16_t* out, int B, int H, int chunk, int max_chunks, int max_seqlen, int sparse_topk,
    int* status) {
    if (threadIdx.x == 0) grid_dep_trigger();
    grid_dep_wait();                           // the partial kernel's chunk states
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= B * H) return;
    const int b = gw / H;
    const int64_t T = seq.len(b);
    if (T < 1 || T > max_seqlen) return;        // reported by the item pass
    const int span = sparse_topk > 0 ? sparse_topk : int(T);
    const int nch = (span + chunk - 1) / chunk;
    MLA_CHECK(nch >= 1 && nch <= max_chunks, status);
    const int64_t s0 = int64_t(gw) * max_chunks;
    // Chunks go 32 at a time: lane c holds chunk c's (max, sum), and every
    // lane's accumulator loads of the 32 chunks are issued together.
    float mx = -INFINITY;
    for (int c = lane; c < nch; c += 32) mx = fmaxf(mx, part_ml[(s0 + c) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float a[4] = {0.f, 0.f, 0.f, 0.f}, L = 0.f;
    if (mx != -INFINITY) {
        for (int c0 = 0; c0 < nch; c0 += 32) {
            const int cnt = min(32, nch - c0);
            float wl = 0.f;
            if (lane < cnt) {
                const float2 ml = *reinterpret_cast<const float2*>(part_ml + (s0 + c0 + lane) * 2);
                wl = ex2(ml.x - mx);
                L += wl * ml.y;
            }
            const float* base = part_acc + (s0 + c0) * kDv + lane * 4;
#pragma unroll 8
            for (int u = 0; u < cnt; ++u) {
                const float wgt = __shfl_sync(0xffffffffu, wl, u);
                const float4 pa = *reinterpret_cast<const float4*>(base + u * kDv);
                a[0] += wgt * pa.x;
                a[1] += wgt * pa.y;
                a[2] += wgt * pa.z;
                a[3] += wgt * pa.w;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    }
    const float inv = L > 0.f ? 1.0f / L : 0.f;
    const int64_t o = int64_t(gw) * kDv + lane * 4;
    uint32_t packed[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        float z0 = a[2 * t] * inv, z1 = a[2 * t + 1] * inv;
        if (gate) {
            const uint32_t gw2 = *reinterpret_cast<const uint32_t*>(gate + o + 2 * t);
            z0 *= sigmoidf_fast(bf_lo(gw2));
            z1 *= sigmoidf_fast(bf_hi(gw2));
        }
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(z0, z1);
        packed[t] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint2*>(out + o) = make_uint2(packed[0], packed[1]);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

DecodePlan plan_decode(int B, int H, int max_len, bool sparse, int sparse_chunk) {
    // Dense: largest chunk (<= 1024, >= one stage) that still gives >= 2432
    // work items (16 per SM on a 152-SM part) when every sequence is max_len
    // long.  Sparse: `sparse_chunk` entries (a power of two, one stage at
    // least), 256 unless the test knob sets it (a sweep over 64..2048 on the
    // B=8, T=131072 workload peaked at 256).
    DecodePlan pl{};
    int chunk = 1024;
    auto items = [&](int c) { return int64_t(B) * H * ((int64_t(max_len) + c - 1) / c); };
    while (chunk > kDenseSP && items(chunk) < 2432) chunk >>= 1;
    if (sparse) chunk = sparse_chunk > 0 ? sparse_chunk : 256;
    pl.chunk = chunk;
    pl.max_chunks = int((int64_t(max_len) + chunk - 1) / chunk);
    const size_t slots = size_t(B) * H * pl.max_chunks;
    pl.acc_off = 0;
    pl.ml_off = align256(slots * kDv * 4);
    pl.items_off = pl.ml_off + align256(slots * 2 * 4);
    pl.total = pl.items_off + (sparse ? 0 : align256(size_t(B + 1) * 4));
    return pl;
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& pl, bool sparse,
                          const DeviceInfo& dev, const Knobs& kn, const KernelTimer& tm,
                          cudaStream_t st) {
    static_assert(smem_bytes<true>() <= 227 * 1024 && smem_bytes<false>() <= 227 * 1024,
                  "shared memory budget");
    Params p{};
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.seq = a.seq;
    p.idx = a.idx;
    p.B = a.B;
    p.H = a.H;
    p.chunk = pl.chunk;
    p.max_chunks = pl.max_chunks;
    p.topk = a.topk;
    p.max_seqlen = a.max_seqlen;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    p.part_acc = reinterpret_cast<float*>(ws + pl.acc_off);
    p.part_ml = reinterpret_cast<float*>(ws + pl.ml_off);
    p.item_start = sparse ? nullptr : reinterpret_cast<int*>(ws + pl.items_off);
    p.scale_log2 = a.scale * kLog2e;
    p.wait_ns = kn.wait_limit_ns;
    p.stall_stage = kn.stall_stage;
    p.status = dev.status;

    cudaError_t e;
    int grid = dev.sms;
    if (sparse) {
        const int items = a.B * a.H * ((a.topk + pl.chunk - 1) / pl.chunk);
        grid = items < grid ? items : grid;
        e = cudaFuncSetAttribute(decode_partial_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem_bytes<true>()));
        if (e != cudaSuccess) return e;
        if (tm.begin) cudaEventRecord(tm.begin, st);
        e = launch_after_prev(decode_partial_kernel<true>, dim3(grid), dim3(Roles<true>::kThreads),
                              smem_bytes<true>(), st, p);
        if (tm.end) cudaEventRecord(tm.end, st);
    } else {
        e = launch_after_prev(decode_items_kernel, dim3(1), dim3(1024), 0, st, a.seq, a.B, a.H,
                              pl.chunk, a.max_seqlen, const_cast<int*>(p.item_start), dev.status);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(decode_partial_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem_bytes<false>()));
        if (e != cudaSuccess) return e;
        if (tm.begin) cudaEventRecord(tm.begin, st);
        e = launch_after_prev(decode_partial_kernel<false>, dim3(grid),
                              dim3(Roles<false>::kThreads), smem_bytes<false>(), st, p);
        if (tm.end) cudaEventRecord(tm.end, st);
    }
    if (e != cudaSuccess) return e;
    // Every kernel of the call is launched programmatically dependent on the
    // one before it and waits on the device before touching global memory.
    const int warps = a.B * a.H;
    e = launch_after_prev(decode_merge_kernel, dim3((warps + 7) / 8), dim3(256), 0, st,
                          static_cast<const float*>(p.part_acc), static_cast<const float*>(p.part_ml),
                          a.seq, a.gate, a.out, a.B, a.H, pl.chunk, pl.max_chunks,
                          sparse ? (1 << 30) : a.max_seqlen, sparse ? a.topk : 0, dev.status);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mla
