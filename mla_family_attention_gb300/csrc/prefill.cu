// Causal gated MLA prefill on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes (Kimi K3 MLA forward; Kimi K2 "Latent attention > KV
// cache" score line; K3.1 Gated DSA post eqs. (9), (10)): for every sequence
// b, head h and new token i (absolute position Tk-Tq+i),
//   z = sum_{j <= Tk-Tq+i} softmax_j(scale * q_i . k_j) v_j
//   out[b, i, h*128+d] = z_d * sigmoid(gate[b, i, h*128+d])   (gate optional)
//
// Design (one CTA per 128-row query tile of one (b, h); CTAs ordered head by
// head so concurrent CTAs share K/V in L2, heavy causal tiles first):
//   * TMEM (512 columns): three 128-column score buffers S0/S1/S2 and the
//     128-column output O.  The softmax writes P (bf16) back over the first
//     64 columns of its score buffer, so P.V reads its A operand from TMEM.
//     The query tile (192 features, 48 KB) stays in shared memory for the
//     whole CTA as Q.K^T's A operand; keeping it in TMEM instead (96
//     columns) left room for only two score buffers and measured 2-3 %
//     slower.
//   * warp 0: TMA producer for the query tile, a 2-stage key ring (three
//     64-feature boxes of 128 keys, 128-byte swizzle) and a 2-stage value
//     ring;
//   * warp 1: owns TMEM; one lane issues S_j = Q K_j^T; warp 10: one lane
//     issues O += P_j V_j.  tcgen05.mma blocks the issuing thread until the
//     pipe accepts it, so with two issuing threads one's barrier waits and
//     commits overlap the other's MMAs; the next scores are computed while
//     the softmax of the current tile runs.  S_{j+3} reuses the buffer whose
//     P_j the P.V of tile j reads, so it waits for that P.V to complete;
//   * warps 2-9: two threads per query row, each owning 64 of the tile's 128
//     key columns (and 64 of the 128 output features).  They load their half
//     of the row's scores, apply the causal / length mask on tiles that need
//     it, swap partial maxima through shared memory, and update the running
//     maximum lazily: O (in TMEM) is rescaled only when a row maximum grows by
//     more than 2^8, otherwise exponentials use the stale maximum (values up
//     to 2^8 are exact enough in bf16 and fp32).  At the end they normalise
//     O, apply the sigmoid gate and store bf16 rows.
// A second shape of the same kernel (kPair) runs query tiles 2i and 2i+1 of
// a head on a cluster of two CTAs: the even CTA issues M = 256 MMAs
// (tcgen05 cta_group::2) over both SMs' TMEM, each CTA loads half of every
// key and value tile, the odd CTA forwards its load completions and its
// softmax arrivals to the even CTA's barriers, and the MMA commits arrive on
// both CTAs' barriers (multicast).  It halves the MMA instructions and the
// key/value bytes per SM, but the cross-SM handoffs lengthen every key
// tile's score -> softmax -> P.V chain, which is what bounds this kernel,
// and it measured slower (982 vs 1,343 TFLOP/s at H=96, T=16384), so the
// one-CTA shape is the default.
// All waits are bounded; a timeout sets MLA_ERR_TIMEOUT, the roles stop, the
// MMA lane waits for its last commit, and TMEM is released before exit.
#include <cuda_bf16.h>

#define MLA_FILE_ID 2   // site ids of the bounds-checked debug build
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kBM = 128;                       // query rows per CTA
constexpr int kBN = 128;                       // keys per KV tile
constexpr int kSoftmaxWarps = 8;               // two per TMEM lane quadrant
constexpr int kPvWarp = 2 + kSoftmaxWarps;     // the P.V issuing warp, after the softmax warps
constexpr int kPThreads = (kPvWarp + 1) * 32;
constexpr uint32_t kCols = 512;
constexpr int kNB = 3;                        // score buffers
constexpr uint32_t kColS = 0, kColO = 384;     // S_i at kColS + 128 i
constexpr int kQBox = kBM * 128;               // 128 query rows x 64 features
constexpr int kQTile = 3 * kQBox;              // the query tile, 48 KB
constexpr float kRescaleLog2 = 8.f;

// Tile geometry.  One CTA (kPair = false): each CTA loads whole 128-key
// tiles (three 64-feature key boxes of 128 rows, two 64-feature value
// boxes).  A CTA pair (kPair = true, M = 256 MMAs): each CTA loads half of
// every tile's B operand — keys 64*rank..64*rank+63 of the Q.K^T tile and
// value features 64*rank..64*rank+63 of the P.V tile — so each SM's shared
// memory carries half the key and value bytes, and the even CTA issues one
// MMA for both SMs' 128 query rows.
template <bool kPair>
struct PCfg {
    static constexpr int kKRows = kPair ? 64 : 128;                 // key rows per CTA per tile
    static constexpr int kKBox = kKRows * 128;                      // 64 features x kKRows
    static constexpr int kKTile = 3 * kKBox;
    static constexpr int kVBox = kBN * 128;                         // 128 keys x 64 features
    static constexpr int kVBoxes = kPair ? 1 : 2;
    static constexpr int kVTile = kVBoxes * kVBox;
    static constexpr int kKStages = kPair ? 3 : 2, kVStages = kPair ? 3 : 2;
    static constexpr int kRows = kPair ? 256 : 128;                 // MMA M
    static constexpr int kArrivals = kSoftmaxWarps * (kPair ? 2 : 1);
    static constexpr size_t kSmem = 1024 + size_t(kKStages) * kKTile + size_t(kVStages) * kVTile +
                                    kQTile + 512 + (2 * 2 * kBM * 2 + 2 * kBM) * 4;
    static constexpr uint32_t kIdescQK = idesc_bf16_f32(kRows, 128, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(kRows, 128, false, true);
};

struct PrefillParams {
    const uint16_t* q;      // [B,H,Tq,192]
    const uint16_t* gate;   // [B,Tq,H*128] or null
    uint16_t* out;          // [B,Tq,H*128]
    int B, H, Tq, Tk, n_qt;
    float scale_log2;
    long long wait_ns;
    int* status;
};

// Prefetch the 128-byte line holding `p` into L2.
__device__ __forceinline__ void prefetch_l2_line(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <bool kPair>
__global__ void __launch_bounds__(kPThreads, 1)
    mla_prefill_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap,
                       const __grid_constant__ CUtensorMap qmap, const PrefillParams p) {
    using C = PCfg<kPair>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ksm = smem;                                        // [KS][key tile]
    uint8_t* vsm = smem + C::kKStages * C::kKTile;              // [VS][value tile]
    uint8_t* qsm = vsm + C::kVStages * C::kVTile;               // [3][16 KB] query tile
    uint64_t* bars = reinterpret_cast<uint64_t*>(qsm + kQTile);
    uint64_t* kfull = bars;                                     // TMA -> MMA (this CTA's half)
    uint64_t* kempty = kfull + C::kKStages;                     // MMA -> TMA
    uint64_t* vfull = kempty + C::kKStages;
    uint64_t* vempty = vfull + C::kVStages;
    uint64_t* kpeer = vempty + C::kVStages;                     // pair: odd CTA's key half landed
    uint64_t* vpeer = kpeer + C::kKStages;                      // pair: odd CTA's value half landed
    uint64_t* sfull = vpeer + C::kVStages;                      // [3] MMA -> softmax
    uint64_t* pfull = sfull + kNB;                              // [3] softmax -> MMA
    uint64_t* odone = pfull + kNB;                              // MMA -> softmax (each P.V)
    uint64_t* ofinal = odone + 1;                               // MMA -> epilogue
    uint64_t* qready = ofinal + 1;                              // TMA -> MMA (this CTA's queries)
    uint64_t* qpeer = qready + 1;                               // pair: odd CTA's queries landed
    uint64_t* qkdone = qpeer + 1;                               // Q.K^T lane's drain
    uint64_t* sfree = qkdone + 1;                               // [3] P.V -> Q.K^T (buffer's P read)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sfree + kNB);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    // row-half exchange between the two softmax warps of a quadrant:
    // [parity][half][row] partial maxima and the halves' ok flags, and a
    // separate [half][row] slot for the final row sums
    float* xmax = reinterpret_cast<float*>(smem + C::kKStages * C::kKTile +
                                           C::kVStages * C::kVTile + kQTile + 512);
    int* xok = reinterpret_cast<int*>(xmax + 2 * 2 * kBM);
    float* xsum = reinterpret_cast<float*>(xok + 2 * 2 * kBM);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Head-major order: the CTAs running at one time share one or two heads'
    // keys and values in L2 (one head's cache is 10 MB at T=16384, all heads'
    // 1 GB); within a head, heavy (late) causal tiles go first.  A pair
    // takes query tiles 2i (even CTA) and 2i+1 (odd CTA) of one head.
    const uint32_t rank = kPair ? pair_rank() : 0u;
    const bool leader = rank == 0;
    int bh, qt, qt_last;
    if (kPair) {
        const int n_qp = (p.n_qt + 1) / 2;
        const int pair = int(blockIdx.x) >> 1;
        bh = pair / n_qp;
        const int qp = n_qp - 1 - (pair - bh * n_qp);
        qt = 2 * qp + int(rank);
        qt_last = 2 * qp + 1;
    } else {
        bh = int(blockIdx.x) / p.n_qt;
        qt = p.n_qt - 1 - (int(blockIdx.x) - bh * p.n_qt);
        qt_last = qt;
    }
    const int b = bh / p.H, h = bh - b * p.H;
    const int P0 = p.Tk - p.Tq;                                 // cached positions before the new tokens
    const int q0 = qt * kBM;
    // last key any row of the tile (of the pair) sees; both CTAs of a pair
    // walk the same key tiles
    const int kmax = P0 + min(qt_last * kBM + kBM - 1, p.Tq - 1);
    const int n_kv = min((p.Tk + kBN - 1) / kBN, kmax / kBN + 1);
    const int n_full = min((P0 + q0 + 1) / kBN, p.Tk / kBN);    // tiles visible to every row

    // One CTA per tile (no pair): thread 0, the TMA producer, requests the
    // query tile and the first key and value tiles as soon as their barriers
    // exist, before the CTA-wide set-up barrier (the loads then overlap the
    // TMEM allocation); a short prompt's whole run is a few such latencies.
    const bool early = !kPair && n_kv > 0;
    // Launched as a programmatic dependent of the stream's previous kernel:
    // the set-up below (barriers, TMEM) may overlap that kernel's tail, and
    // every thread waits for it (grid_dep_wait) before touching global
    // memory, since it may have written the inputs.  The next kernel may be
    // placed as soon as this one starts.
    if (threadIdx.x == 0) {
        grid_dep_trigger();
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        tma_prefetch_desc(&qmap);
        for (int i = 0; i < C::kKStages; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kempty[i], 1);
            mbar_init(&kpeer[i], 1);
        }
        for (int i = 0; i < C::kVStages; ++i) {
            mbar_init(&vfull[i], 1);
            mbar_init(&vempty[i], 1);
            mbar_init(&vpeer[i], 1);
        }
        for (int i = 0; i < kNB; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&pfull[i], C::kArrivals);
            mbar_init(&sfree[i], 1);
        }
        mbar_init(odone, 1);
        mbar_init(ofinal, 1);
        mbar_init(qready, 1);
        mbar_init(qpeer, 1);
        mbar_init(qkdone, 1);
        *abort_flag = 0;
        fence_mbar_init();
        grid_dep_wait();
        if (early) {
            mbar_arrive_expect_tx(qready, kQTile);
            for (int c = 0; c < 3; ++c)
                tma_load_3d(qsm + c * kQBox, &qmap, c * 64, q0, bh, qready);
            mbar_arrive_expect_tx(&kfull[0], C::kKTile);
            for (int c = 0; c < 3; ++c)
                tma_load_3d(ksm + c * C::kKBox, &kmap, c * 64, 0, bh, &kfull[0]);
            mbar_arrive_expect_tx(&vfull[0], C::kVTile);
            for (int c = 0; c < C::kVBoxes; ++c)
                tma_load_3d(vsm + c * C::kVBox, &vmap, c * 64, 0, bh, &vfull[0]);
        }
    }
    if (warp == 1) {
        if (kPair) tmem_alloc_pair(tmem_holder, kCols);
        else tmem_alloc(tmem_holder, kCols);
    }
    grid_dep_wait();
    tc_fence_before();
    if (kPair) pair_sync();     // both CTAs' barriers exist before either signals the other
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // waits on barriers the other CTA of a pair arrives on acquire at cluster scope
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        return kPair ? mbar_wait_cluster(bar, parity, p.wait_ns) : mbar_wait(bar, parity, p.wait_ns);
    };
    // arrivals for the MMA lanes land on the even CTA's barriers
    auto arrive_mma = [&](uint64_t* bar) {
        if (kPair) mbar_arrive_cluster(pair_addr(bar, 0));
        else mbar_arrive(bar);
    };
    auto commit_both = [&](uint64_t* bar) {
        if (kPair) mma_commit_pair(bar, uint16_t(3));
        else mma_commit(bar);
    };
    auto commit_self = [&](uint64_t* bar) {
        if (kPair) mma_commit_pair(bar, uint16_t(1));
        else mma_commit(bar);
    };

    if (warp == 0) {
        // --------------------------------- TMA ---------------------------------
        // The whole warp walks the tiles and waits; one elected lane issues.
        {
            int kf[C::kKStages] = {}, vf[C::kVStages] = {};
            const int krow0 = kPair ? 64 * int(rank) : 0;       // this CTA's key rows of a tile
            if (early) {
                kf[0] = vf[0] = 1;                              // requested before the set-up barrier
            } else if (elect_one()) {
                // this CTA's 128 query rows (rows at or past Tq arrive as zeros)
                mbar_arrive_expect_tx(qready, kQTile);
                for (int c = 0; c < 3; ++c)
                    tma_load_3d(qsm + c * kQBox, &qmap, c * 64, q0, bh, qready);
            }
            __syncwarp();
            for (int j = early ? 1 : 0; j < n_kv; ++j) {
                if (*abort_flag) break;
                const int ks = j % C::kKStages, kr = j / C::kKStages;
                MLA_CHECK(ks < C::kKStages && (ks + 1) * C::kKTile <= C::kKStages * C::kKTile,
                          p.status);
                if (kr > 0 && !__all_sync(0xffffffffu, wait(&kempty[ks], (kr - 1) & 1))) {
                    if (elect_one()) {
                        report(p.status, kStTimeout);
                        *abort_flag = 1;
                    }
                    break;
                }
                // keys j*128.. of (b, h); rows at or past Tk arrive as zeros
                const int y = j * kBN;
                if (elect_one()) {
                    mbar_arrive_expect_tx(&kfull[ks], C::kKTile);
                    for (int c = 0; c < 3; ++c)
                        tma_load_3d(ksm + ks * C::kKTile + c * C::kKBox, &kmap, c * 64, y + krow0,
                                    bh, &kfull[ks]);
                }
                __syncwarp();
                kf[ks] = kr + 1;
                const int vs = j % C::kVStages, vr = j / C::kVStages;
                if (vr > 0 && !__all_sync(0xffffffffu, wait(&vempty[vs], (vr - 1) & 1))) {
                    if (elect_one()) {
                        report(p.status, kStTimeout);
                        *abort_flag = 1;
                    }
                    break;
                }
                MLA_CHECK(vs < C::kVStages && y >= 0, p.status);
                if (elect_one()) {
                    mbar_arrive_expect_tx(&vfull[vs], C::kVTile);
                    for (int c = 0; c < C::kVBoxes; ++c)
                        tma_load_3d(vsm + vs * C::kVTile + c * C::kVBox, &vmap,
                                    kPair ? 64 * int(rank) : c * 64, y, bh, &vfull[vs]);
                }
                __syncwarp();
                vf[vs] = vr + 1;
            }
            for (int i = 0; i < C::kKStages; ++i)
                if (kf[i] > 0 && !warp_wait(&kfull[i], (kf[i] - 1) & 1, p.wait_ns) && elect_one())
                    report(p.status, kStTimeout);
            for (int i = 0; i < C::kVStages; ++i)
                if (vf[i] > 0 && !warp_wait(&vfull[i], (vf[i] - 1) & 1, p.wait_ns) && elect_one())
                    report(p.status, kStTimeout);
            if (!warp_wait(qready, 0, p.wait_ns) && elect_one()) report(p.status, kStTimeout);
        }
    } else if (kPair && !leader && (warp == 1 || warp == kPvWarp)) {
        // ------------- odd CTA of a pair: tell the MMA lanes its halves landed -------------
        if (lane == 0) {
            const bool keys = warp == 1;
            const int stages = keys ? C::kKStages : C::kVStages;
            uint64_t* full = keys ? kfull : vfull;
            const uint32_t peer = pair_addr(keys ? kpeer : vpeer, 0);
            if (keys) {                                     // the query tile first
                if (mbar_wait(qready, 0, p.wait_ns)) {
                    mbar_arrive_cluster(pair_addr(qpeer, 0));
                } else {
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                }
            }
            for (int j = 0; j < n_kv; ++j) {
                if (*abort_flag) break;
                const int st = j % stages;
                if (!mbar_wait(&full[st], (j / stages) & 1, p.wait_ns)) {
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_cluster(peer + uint32_t(st * 8));
            }
        }
    } else if (warp == 1) {
        // ------------------------------ Q.K^T MMAs ------------------------------
        // The whole warp waits; one elected lane issues each MMA and commit.
        {
            bool ok = __all_sync(0xffffffffu,
                                 mbar_wait(qready, 0, p.wait_ns) && (!kPair || wait(qpeer, 0)));
            bool issued = false;
            for (int j = 0; ok && j < n_kv; ++j) {
                if (*abort_flag) { ok = false; break; }
                const int ks = j % C::kKStages;
                // S_j = Q K_j^T into score buffer j%3 (A = queries in shared
                // memory), once the keys landed (both halves for a pair) and
                // P_{j-3}, in that buffer, has been consumed (a barrier per
                // buffer: its next phase needs S_j, so the parity cannot run
                // two phases ahead of this wait)
                const int sb = j % kNB;
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&kfull[ks], (j / C::kKStages) & 1, p.wait_ns) &&
                                    (!kPair || wait(&kpeer[ks], (j / C::kKStages) & 1)) &&
                                    (j < kNB ||
                                     mbar_wait(&sfree[sb], ((j - kNB) / kNB) & 1, p.wait_ns)))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t kb = smem_u32(ksm + ks * C::kKTile);
                const uint32_t qb = smem_u32(qsm);
                MLA_CHECK(kColS + uint32_t(sb) * 128 + 128 <= kColO, p.status);
                const uint32_t d = tmem + kColS + uint32_t(sb) * 128;
#pragma unroll
                for (int kk = 0; kk < 12; ++kk) {
                    const uint64_t ad =
                        smem_desc_sw128(qb + (kk >> 2) * kQBox + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd =
                        smem_desc_sw128(kb + (kk >> 2) * C::kKBox + (kk & 3) * 32, 16, 1024);
                    if (elect_one()) {
                        if (kPair)
                            mma_bf16_ss_pair(d, ad, bd, C::kIdescQK, kk > 0 ? 1u : 0u);
                        else
                            mma_bf16_ss(d, ad, bd, C::kIdescQK, kk > 0 ? 1u : 0u);
                    }
                }
                if (elect_one()) commit_both(&kempty[ks]);
                if (elect_one()) commit_both(&sfull[sb]);
                __syncwarp();
                issued = true;
            }
            if (!ok && elect_one()) {
                report(p.status, kStTimeout);
                *abort_flag = 1;
            }
            if (elect_one()) commit_self(qkdone);
            __syncwarp();
            if (issued && !warp_wait(qkdone, 0, p.wait_ns) && elect_one())
                report(p.status, kStTimeout);
        }
    } else if (warp == kPvWarp) {
        // ------------------------------- P.V MMAs -------------------------------
        // The whole warp waits; one elected lane issues each MMA and commit.
        {
            bool ok = true, issued = false;
            for (int j = 0; ok && j < n_kv; ++j) {
                if (*abort_flag) { ok = false; break; }
                const int vs = j % C::kVStages;
                const int sb = j % kNB;
                if (!__all_sync(0xffffffffu,
                                wait(&pfull[sb], (j / kNB) & 1) &&
                                    mbar_wait(&vfull[vs], (j / C::kVStages) & 1, p.wait_ns) &&
                                    (!kPair || wait(&vpeer[vs], (j / C::kVStages) & 1)))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // O += P_j V_j (A = probabilities in TMEM, B = values, MN-major)
                const uint32_t vb = smem_u32(vsm + vs * C::kVTile);
                const uint32_t a = tmem + kColS + uint32_t(sb) * 128;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t bd = smem_desc_sw128(vb + kk * 2048, C::kVBox, 1024);
                    if (elect_one()) {
                        if (kPair)
                            mma_bf16_ts_pair(tmem + kColO, a + kk * 8, bd, C::kIdescPV,
                                             (j > 0 || kk > 0) ? 1u : 0u);
                        else
                            mma_bf16_ts(tmem + kColO, a + kk * 8, bd, C::kIdescPV,
                                        (j > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                if (elect_one()) commit_both(&vempty[vs]);
                if (elect_one()) commit_self(&sfree[sb]);
                if (elect_one()) commit_both(odone);
                __syncwarp();
                issued = true;
            }
            if (!ok && elect_one()) {
                report(p.status, kStTimeout);
                *abort_flag = 1;
            }
            if (elect_one()) commit_both(ofinal);   // also releases the epilogue after an abort
            __syncwarp();
            if (issued && !warp_wait(ofinal, 0, p.wait_ns) && elect_one())
                report(p.status, kStTimeout);
        }
    } else {
        // ------------------------- softmax / epilogue --------------------------
        // Warps 2..9: warp w serves TMEM lane quadrant w%4 (rows 32*quad..),
        // and column half `half` of those rows (keys 64*half..64*half+63 of
        // every tile, output features likewise).  The two warps of a quadrant
        // swap partial row maxima (and their ok flags, so they stop together)
        // through shared memory once per tile.
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const int bar_id = 1 + quad;                        // named barrier of the pair
        const int r = quad * 32 + lane;                     // row within the tile
        const int row = q0 + r;                             // query index
        const int qa = P0 + row;                            // absolute position
        const uint32_t lane_off = uint32_t(quad * 32) << 16;
        // this thread's output row and its 64 gate logits (128 bytes): the
        // logits are prefetched into L2 now, so the epilogue's loads of them
        // do not wait on HBM after the last P.V
        const size_t orow = (size_t(b) * p.Tq + size_t(row < p.Tq ? row : 0)) * p.H + h;
        const uint4* g = p.gate ? reinterpret_cast<const uint4*>(p.gate + orow * kDv) + half * 8
                                : nullptr;
        // A prompt of one key tile leaves the second key stage unused: the
        // logits are copied there (cp.async) at once, 128 bytes a thread;
        // otherwise they are prefetched into L2 now and loaded before the
        // last P.V wait.  Either way their sigmoids are computed while the
        // last P.V runs (a sigmoid is a tanh on the special-function unit,
        // ~1 us for a CTA's 16,384).
        const bool gate_smem = !kPair && n_kv == 1 && g && row < p.Tq;
        uint8_t* gsm = ksm + C::kKTile + size_t(half * kBM + r) * 128;
        MLA_CHECK(!gate_smem || C::kKStages >= 2 && (2 * kBM) * 128 <= C::kKTile, p.status);
        if (gate_smem) {
#pragma unroll
            for (int k = 0; k < 8; ++k) cp_async16(gsm + 16 * k, g + k);
        } else if (g && row < p.Tq) {
            prefetch_l2_line(g);
        }
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int buf = j % kNB;
            const int par = j & 1;                          // row-half exchange slot
            ok = ok && !*abort_flag;
            if (ok && !wait(&sfull[buf], (j / kNB) & 1)) {
                report(p.status, kStTimeout);
                *abort_flag = 1;
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);
            const uint32_t sb = tmem + lane_off + kColS + uint32_t(buf) * 128;
            // this thread's 64 score columns and its 64 output columns lie
            // inside its buffer and inside O
            MLA_CHECK(buf < kNB && kColS + uint32_t(buf) * 128 + half * 64 + 64 <= kColO &&
                          kColO + half * 64 + 64 <= kCols && r < kBM,
                      p.status);
            float s[64];
            float mloc = -INFINITY;
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float t[32];
                    tmem_ld32(sb + half * 64 + c * 32, t);
#pragma unroll
                    for (int u = 0; u < 32; ++u) s[c * 32 + u] = t[u];
                }
                tmem_ld_wait();
                if (j >= n_full) {                          // causal / length mask
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int key = j * kBN + half * 64 + c;
                        if (key > qa || key >= p.Tk) s[c] = -INFINITY;
                    }
                }
                float mx[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) mx[u] = s[u];
#pragma unroll
                for (int c = 8; c < 64; ++c) mx[c & 7] = fmaxf(mx[c & 7], s[c]);
                mloc = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            }
            // swap with the other half of the row (double-buffered by tile parity)
            xmax[(par * 2 + half) * kBM + r] = mloc;
            xok[(par * 2 + half) * kBM + r] = ok;
            named_bar_sync(bar_id, 64);
            const float mo = xmax[(par * 2 + (half ^ 1)) * kBM + r];
            ok = __all_sync(0xffffffffu, ok && xok[(par * 2 + (half ^ 1)) * kBM + r] != 0);
            if (!ok) break;                                  // both warps of the pair
            const float mt = fmaxf(mloc, mo) * p.scale_log2; // scale > 0 keeps the order
            // lazy rescale: only when the row maximum grows by more than 2^8
            const bool need = mt > m_used + kRescaleLog2;
            const float m_new = need ? mt : m_used;
            const float factor = need ? ex2(m_used - m_new) : 1.f;     // m_used=-inf -> 0
            if (__any_sync(0xffffffffu, need && j > 0)) {
                bool o_ok = wait(odone, (j - 1) & 1);                   // P_{j-1} V_{j-1} landed
                o_ok = __all_sync(0xffffffffu, o_ok);
                if (o_ok) {
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        float o[32];
                        tmem_ld32(tmem + lane_off + kColO + half * 64 + c * 32, o);
                        tmem_ld_wait();
                        uint32_t w[32];
#pragma unroll
                        for (int u = 0; u < 32; ++u) w[u] = __float_as_uint(o[u] * factor);
                        tmem_st32(tmem + lane_off + kColO + half * 64 + c * 32, w);
                    }
                } else {                                    // both halves stop next tile
                    report(p.status, kStTimeout);
                    *abort_flag = 1;
                }
            }
            l *= factor;
            m_used = m_new;
            const float nme = m_used == -INFINITY ? 0.f : -m_used;
            // P_j (bf16) over columns 32*half.. of the score buffer
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t w[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float p0 = ex2(fmaf(s[c * 32 + 2 * u], p.scale_log2, nme));
                    const float p1 = ex2(fmaf(s[c * 32 + 2 * u + 1], p.scale_log2, nme));
                    ls[u & 3] += p0 + p1;
                    w[u] = pack_bf16(p0, p1);
                }
                tmem_st16(tmem + lane_off + kColS + uint32_t(buf) * 128 + half * 32 + c * 16, w);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_mma(&pfull[buf]);
        }
        // ---- epilogue: O / l * sigmoid(gate) -> bf16 ----
        // the gate logits are loaded before the wait for the last P.V, so
        // their latency overlaps it
        // the 64 gates, while the last P.V runs
        uint4 gl[8];
        if (gate_smem) {
            cp_async_wait_all();
#pragma unroll
            for (int k = 0; k < 8; ++k) gl[k] = *reinterpret_cast<const uint4*>(gsm + 16 * k);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                gl[k] = (g && row < p.Tq) ? __ldg(g + k) : make_uint4(0u, 0u, 0u, 0u);
        }
        float sg[64];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t gg[4] = {gl[k].x, gl[k].y, gl[k].z, gl[k].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sg[8 * k + 2 * e] = g ? sigmoidf_fast(bf_lo(gg[e])) : 1.f;
                sg[8 * k + 2 * e + 1] = g ? sigmoidf_fast(bf_hi(gg[e])) : 1.f;
            }
        }
        bool fin = ok && wait(ofinal, 0);
        fin = __all_sync(0xffffffffu, fin);
        if (!fin && ok) report(p.status, kStTimeout);
        xsum[half * kBM + r] = l;                           // row sum = both halves
        named_bar_sync(bar_id, 64);
        const float lt = l + xsum[(half ^ 1) * kBM + r];
        if (fin) {
            tc_fence_after();
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kDv) + half * 8;
            float o[64];
            tmem_ld32(tmem + lane_off + kColO + half * 64, *reinterpret_cast<float(*)[32]>(o));
            tmem_ld32(tmem + lane_off + kColO + half * 64 + 32,
                      *reinterpret_cast<float(*)[32]>(o + 32));
            tmem_ld_wait();
            if (row < p.Tq) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    float z[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) z[e] = o[u * 8 + e] * inv * sg[u * 8 + e];
                    dst[u] = make_uint4(pack_bf16(z[0], z[1]), pack_bf16(z[2], z[3]),
                                        pack_bf16(z[4], z[5]), pack_bf16(z[6], z[7]));
                }
            }
        }
    }
    tc_fence_before();
    // A pair's CTAs leave together: neither exits while the other (or the
    // MMAs the even one issued) may still touch its barriers, shared memory
    // or TMEM.  Every wait above is bounded, so every thread arrives here.
    if (kPair) pair_sync();
    else __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        if (kPair) tmem_dealloc_pair(tmem, kCols);
        else tmem_dealloc(tmem, kCols);
    }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const DeviceInfo& dev, const Knobs& kn,
                           const KernelTimer& tm, cudaStream_t st) {
    static_assert(PCfg<false>::kSmem <= 227 * 1024 && PCfg<true>::kSmem <= 227 * 1024,
                  "shared memory budget");
    const bool pair = kn.prefill_ctas == 2;
    // [B*H][Tk][D] views of the [B,H,kv_cap,D] caches: a tile that runs past
    // Tk reads zeros, never the unused capacity or the next head's rows.
    CUtensorMap kmap, vmap;
    const uint64_t bhs = uint64_t(a.B) * a.H, cap = uint64_t(a.kv_cap);
    cudaError_t e = encode_tmap_3d_bf16(&kmap, a.k, kDqk, a.Tk, bhs, kDqk * 2, cap * kDqk * 2, 64,
                                        pair ? PCfg<true>::kKRows : PCfg<false>::kKRows);
    if (e != cudaSuccess) return e;
    e = encode_tmap_3d_bf16(&vmap, a.v, kDv, a.Tk, bhs, kDv * 2, cap * kDv * 2, 64, kBN);
    if (e != cudaSuccess) return e;
    // [B*H][Tq][192] view of the queries: rows past Tq read as zeros
    CUtensorMap qmap;
    e = encode_tmap_3d_bf16(&qmap, a.q, kDqk, a.Tq, bhs, kDqk * 2, uint64_t(a.Tq) * kDqk * 2, 64,
                            kBM);
    if (e != cudaSuccess) return e;
    PrefillParams p{a.q, a.gate, a.out, a.B, a.H, a.Tq, a.Tk, (a.Tq + kBM - 1) / kBM,
                    a.scale * 1.4426950408889634f, kn.wait_limit_ns, dev.status};
    if (!pair) {
        e = cudaFuncSetAttribute(mla_prefill_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(PCfg<false>::kSmem));
        if (e != cudaSuccess) return e;
        const int grid = p.n_qt * a.B * a.H;
        if (tm.begin) cudaEventRecord(tm.begin, st);
        e = launch_after_prev(mla_prefill_kernel<false>, dim3(grid), dim3(kPThreads),
                              PCfg<false>::kSmem, st, kmap, vmap, qmap, p);
        if (tm.end) cudaEventRecord(tm.end, st);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    e = cudaFuncSetAttribute(mla_prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(PCfg<true>::kSmem));
    if (e != cudaSuccess) return e;
    // clusters of two CTAs: query tiles 2i and 2i+1 of one head (the odd
    // CTA of the last pair of an odd tile count has no rows to store)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * ((p.n_qt + 1) / 2) * a.B * a.H);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = PCfg<true>::kSmem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (tm.begin) cudaEventRecord(tm.begin, st);
    e = cudaLaunchKernelEx(&cfg, mla_prefill_kernel<true>, kmap, vmap, qmap, p);
    if (tm.end) cudaEventRecord(tm.end, st);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mla
