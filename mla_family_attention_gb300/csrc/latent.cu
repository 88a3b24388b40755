// Absorbed-latent gated MLA decode for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes (K3.1 Gated DSA post, eqs. (7)-(10), and its remark that
// inference absorbs W^K into the query and applies W^V after attention): the
// cache holds per position the normalised latent c_s (512 features) and the
// shared key r_s (64); head h's key is [W^K_h c_s ; r_s] and its value
// W^V_h c_s.  For the one query of sequence b and head h,
//   q~_h = [W^K_h^T q_h[0:128] ; q_h[128:192]]                 (576 features)
//   z~_h = sum_s softmax_s(scale * q~_h . [c_s ; r_s]) c_s     (512 features)
//   out[b, h*128+d] = (W^V_h z~_h)_d * sigmoid(gate[b, h*128+d])
// which equals attention over the expanded keys and values exactly (up to
// rounding) while reading 1,152 cache bytes per position instead of 61,440.
//
// Kernels, in launch order:
//   1. latent_absorb_kernel: q~ = W^K-absorbed queries, bf16, into workspace.
//   2. latent_sched_kernel: splits the sequences' 64-position tiles evenly over
//      one CTA per SM (a CTA's range may span sequences); every (CTA,
//      sequence) piece is a segment with its own partial result.
//   3. mla_latent_kernel (one CTA per SM):
//      * S = Q~ K^T on the tensor cores with the heads as the M dimension
//        (M = 128 rows, rows past H ignored), 64 keys as N, 576 features as K;
//        Q~ stays in shared memory for the whole segment;
//      * softmax per head row (two threads per row), lazily rescaled: the
//        accumulator is rescaled only when a row maximum grows by 2^8;
//      * O^T += C^T P^T with the latent features as M (four 128-row blocks),
//        the heads as N and the 64 keys as K; O^T (512 x H fp32) lives in
//        TMEM next to two 64-column score buffers;
//      * a six-slot ring of 16 KB slots carries each tile as five units
//        (the 64 shared-key features, then four 128-feature latent blocks),
//        filled by TMA tile loads of a decode sequence's contiguous rows, by
//        16-byte cp.async copies of a prompt token's selected rows (sparse
//        prefill) or by producer threads converting FP8 records; the latent
//        blocks stay until P.V has used them, so every cache byte is read
//        once.  S of the next tile is computed on its first two units while
//        the softmax of the current tile runs.
//   4. latent_fixup_kernel: per head, log-sum-exp merge of the segments of
//      the sequences that span CTAs, into the normalised z~.
//   5. latent_out_kernel: out = (W^V_h z~) * sigmoid(gate), a tensor-core
//      GEMM per head over all sequences.
// Every wait is bounded; a timeout records MLA_ERR_TIMEOUT, the roles stop
// (the softmax warps keep walking their barriers), in-flight copies and MMAs
// are waited for, and TMEM is released before exit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#define MLA_FILE_ID 4   // site ids of the bounds-checked debug build
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kLT = 64;                          // keys per tile
constexpr int kMaxH = 96;                        // TMEM: 2*64 score + 4*H output columns
constexpr int kHalf = kLT * 64 * 2;              // 8 KB: 64 keys x 64 features
constexpr int kSlot = 2 * kHalf;                 // 16 KB ring slot
constexpr int kSlots = 6;
constexpr int kFills = 5;                        // ring fills per tile
constexpr int kQBytes = (8 * kMaxH + 128) * 128; // nine [H x 64] blocks + rows read past them
constexpr int kPBytes = kMaxH * 128;             // P: [H rows][64 keys] bf16
// Where a tile's rows come from: tiled TMA loads of 64 contiguous cache rows
// (decode), 16-byte cp.async copies of the selected rows (sparse prefill), or
// FP8 records converted to bf16 by the producer threads.
enum Src { kSrcTma = 0, kSrcGather = 1, kSrcFp8 = 2 };
// Warp roles: 0 TMA producer, 1 Q.K^T MMA issue, 2-9 softmax and epilogue,
// then the P.V MMA issue warp; the gather and FP8 variants have 128 producer
// threads instead of the TMA warp (warp 0 and warps 10-12), so their P.V
// warp is warp 13.  tcgen05.mma issue blocks the issuing thread until the
// tensor pipe takes the instruction, so every barrier wait or commit of an
// issuing thread idles the pipe; two issuing warps hide each other's waits.
template <int kSrc>
constexpr int kPvWarp = kSrc == kSrcTma ? 10 : 13;
template <int kSrc>
constexpr int kThreadsOf = (kPvWarp<kSrc> + 1) * 32;
constexpr int kRec = 656;                        // FP8 record: 512 codes, 4 fp32 scales, 64 bf16
constexpr int kColO = 2 * kLT;                   // O^T columns start after the score buffers
constexpr float kRescaleLog2 = 8.f;
// FP8 records are prefetched into L2 this many tiles ahead of the producer
// threads' loads (1 measured best of 0, 1, 2, 4, 8, 12; the TMA path measured
// best with no prefetch: bulk prefetches share the TMA unit with its loads).
constexpr int kAheadFp8 = 1;
constexpr size_t kExtra = (2 * 2 * 128 + 2 * 128 + 128 + 128) * 4 + 256;
constexpr size_t kLatSmem = 1024 + kQBytes + kPBytes + size_t(kSlots) * kSlot + kExtra;
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kLT, false, false);

// Work split written by latent_sched_kernel: n tiles in all, `per` tiles
// per CTA, the number of sequences that span CTAs, the tile prefix, the
// partial-slot prefix (nonzero only for spanning sequences), and their list.
struct Sched {
    const int* base;
    __device__ int n() const { return base[0]; }
    __device__ int per() const { return base[1]; }
    __device__ int nmulti() const { return base[2]; }
    __device__ const int* ts() const { return base + 3; }
    __device__ const int* seg(int B) const { return base + 3 + (B + 1); }
    __device__ const int* mlist(int B) const { return base + 3 + 2 * (B + 1); }
};

struct LatParams {
    const int* sched;
    const int64_t* cu;       // decode: [B+1] packed positions of each sequence
    const int32_t* idx;      // sparse prefill: [B][topk] selections, else null
    int topk, P;             // sparse prefill: selection width; cached positions before token 0
    const uint16_t* ckv;     // the latent cache (the gather producer reads its selected rows)
    int64_t total;           // rows of ckv
    float* part;             // [slots][H][512] unnormalised O of segments of spanning sequences
    float* ml;               // [slots][H][2]: max (log2 units), sum
    uint16_t* zbuf;          // [B][H][512] bf16 normalised latent outputs
    const uint8_t* rec;      // FP8 cache: [total][656] records, else null
    int B, H;
    float scale_log2;
    long long wait_ns;
    int* status;
};

__device__ __forceinline__ bool bar_or(int id, int threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(r)
        : "r"(uint32_t(pred)), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

// Bulk prefetch of `bytes` (multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// A "sequence" of the latent kernel: a decode sequence (rows row0..row0+T-1
// of the cache) or one prompt token of a sparse prefill (the first T entries
// of its selection, positions below vis).
struct SeqDesc {
    int64_t row0;
    int T, vis;
};

__device__ __forceinline__ SeqDesc seq_desc(const LatParams& p, int b) {
    if (p.idx) {
        const int vis = p.P + b + 1;
        return SeqDesc{0, min(p.topk, vis), vis};
    }
    const int64_t r0 = p.cu[b];
    return SeqDesc{r0, int(p.cu[b + 1] - r0), 0};
}

// Selection entry e of token b (sparse prefill), -1 past the token's count.
__device__ __forceinline__ int sel_raw(const LatParams& p, int b, const SeqDesc& sd, int e) {
    return e < sd.T ? __ldg(p.idx + int64_t(b) * p.topk + e) : -1;
}

// Cache row of a selection entry and whether it names a visible position;
// padding and invalid entries read row 0 and are masked by the softmax.
__device__ __forceinline__ int sel_row(const LatParams& p, const SeqDesc& sd, int v, bool* valid) {
    *valid = v >= 0 && v < sd.vis;
    if (!*valid && (v < -1 || v >= sd.vis)) report(p.status, kStBadIndex);
    return *valid ? v : 0;
}

// Walks a CTA's tile range [t0, t1) sequence by sequence.
struct Cursor {
    const int* ts;
    int b = 0;
    __device__ void seek(int t, int B) {
        int lo = 0, hi = B;                      // largest b with ts[b] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (ts[mid] <= t) lo = mid; else hi = mid;
        }
        b = lo;
    }
    __device__ void advance(int t) {
        while (t >= ts[b + 1]) ++b;
    }
};

template <int kSrc>
__global__ void __launch_bounds__(kThreadsOf<kSrc>, 1)
    mla_latent_kernel(const __grid_constant__ CUtensorMap cmap,
                      const __grid_constant__ CUtensorMap qmap, const LatParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* qs = smem;                                  // Q~: block kb at kb*H*128
    uint8_t* ps = qs + kQBytes;                          // P (B operand of P.V)
    uint8_t* ring = ps + kPBytes;
    float* xmax = reinterpret_cast<float*>(ring + kSlots * kSlot);   // [2][2][128]
    float* xsum = xmax + 2 * 2 * 128;                                // [2][128]
    float* fsm = xsum + 2 * 128;                                     // [128]
    float* inv_l = fsm + 128;                                        // [128]
    uint64_t* full = reinterpret_cast<uint64_t*>(inv_l + 128);
    uint64_t* empty = full + kSlots;
    uint64_t* sfull = empty + kSlots;      // [2] MMA -> softmax
    uint64_t* sfree = sfull + 2;           // [2] softmax -> MMA
    uint64_t* pfull = sfree + 2;           // softmax -> MMA
    uint64_t* qfull = pfull + 1;           // TMA -> MMA (Q~ of a segment)
    uint64_t* qfree = qfull + 1;           // MMA -> TMA (a segment's Q.K^T done)
    uint64_t* ofinal = qfree + 1;          // MMA -> epilogue (a segment's P.V done)
    uint64_t* oread = ofinal + 1;          // epilogue -> MMA (O^T read out)
    uint64_t* pfree = oread + 1;           // P.V of a tile done: P and O^T free
    uint64_t* mdone = pfree + 1;           // [2] each issuing warp's drain before TMEM release
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mdone + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H, B = p.B;
    const Sched sch{p.sched};
    const int n = sch.n(), per = sch.per();
    const int* ts = sch.ts();
    const int* seg = sch.seg(B);
    const bool sparse = p.idx != nullptr;
    const int c = blockIdx.x;
    const int t0 = min(n, c * per), t1 = min(n, t0 + per);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&full[i], kSrc == kSrcTma ? 1 : 128);   // else every producer thread arrives
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sfree[i], 8);
        }
        mbar_init(pfull, 8);
        mbar_init(qfull, 1);
        mbar_init(qfree, 1);
        mbar_init(ofinal, 1);
        mbar_init(oread, 8);
        mbar_init(pfree, 1);
        mbar_init(&mdone[0], 1);
        mbar_init(&mdone[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    grid_dep_wait();                                     // the work split and absorbed queries

    auto fail = [&]() {
        report(p.status, kStTimeout);
        *abort_flag = 1;
    };

    const bool producer_warp = warp == 0 || (warp >= 10 && warp < 13);
    if (kSrc == kSrcFp8 && producer_warp) {
        // -------------------- FP8 producer (128 threads) --------------------
        // Thread ptid converts row ptid/2 of each fill, half ptid&1: 64 e4m3
        // codes times their group scale into 64 bf16 features (or 32 bf16
        // shared-key features), stored in the same 128-byte swizzled layout
        // the TMA boxes have; every thread arrives on the fill's barrier.
        const int ptid = warp == 0 ? lane : (warp - 9) * 32 + lane;
        const int r = ptid >> 1, hf = ptid & 1;
        if (t0 < t1) {
            int nseg = 0, fill = 0;
            Cursor cur{ts}, ahead{ts};
            cur.seek(t0, B);
            ahead.seek(t0, B);
            auto prefetch_tile = [&](int t) {
                ahead.advance(t);
                const int64_t r0 = p.cu[ahead.b] + int64_t(t - ts[ahead.b]) * kLT;
                const int64_t r1 = min(r0 + kLT, p.total);
                if (r1 > r0) prefetch_l2(p.rec + r0 * kRec, uint32_t((r1 - r0) * kRec));
            };
            if (!sparse && ptid == 0)
                for (int t = t0; t < min(t1, t0 + kAheadFp8); ++t) prefetch_tile(t);
            bool ok = true;
            for (int t = t0; t < t1 && ok; ++t) {
                if (!sparse && ptid == 0 && t + kAheadFp8 < t1) prefetch_tile(t + kAheadFp8);
                cur.advance(t);
                const int b = cur.b;
                const SeqDesc sd = seq_desc(p, b);
                if (t == t0 || t == ts[b]) {
                    if (ptid == 0) {
                        if (nseg > 0 && !mbar_wait(qfree, (nseg - 1) & 1, p.wait_ns)) {
                            fail();
                        } else {
                            mbar_arrive_expect_tx(qfull, 9 * H * 128);
                            for (int kb = 0; kb < 9; ++kb)
                                tma_load_2d(qs + kb * H * 128, &qmap, kb * 64, b * H, qfull);
                        }
                    }
                    ++nseg;
                }
                const int e0 = (t - ts[b]) * kLT;
                int64_t grow;
                if (sparse) {
                    bool v;
                    grow = sel_row(p, sd, sel_raw(p, b, sd, e0 + r), &v);
                } else {
                    grow = sd.row0 + e0 + r;
                }
                const bool inb = grow < p.total;
                const uint8_t* src = p.rec + (inb ? grow : 0) * kRec;
                const uint32_t rowoff = (r >> 3) * 1024 + (r & 7) * 128;
                // this thread's 320 bytes of the tile (shared key, 4 x 64 codes)
                // and the 4 group scales, loaded together so one latency covers
                // the tile's five fills
                uint4 v[kFills][4];
                float4 sc4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int i = 0; i < kFills; ++i) {
                    const uint4* s4 = reinterpret_cast<const uint4*>(
                        i == 0 ? src + 512 + 16 + hf * 64 : src + 128 * (i - 1) + 64 * hf);
#pragma unroll
                    for (int q = 0; q < 4; ++q) v[i][q] = inb ? __ldg(s4 + q) : make_uint4(0, 0, 0, 0);
                }
                if (inb) sc4 = __ldg(reinterpret_cast<const float4*>(src + 512));
                const float scs[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
#pragma unroll
                for (int i = 0; i < kFills; ++i, ++fill) {
                    const int slot = fill % kSlots, round = fill / kSlots;
                    if (*abort_flag) { ok = false; break; }
                    if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, p.wait_ns)) {
                        fail();
                        ok = false;
                        break;
                    }
                    uint8_t* dst = ring + slot * kSlot;
                    if (i == 0) {                      // shared key: bf16 copy, 64 bytes
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4*>(dst + rowoff + (((hf * 4 + q) ^ (r & 7)) << 4)) =
                                v[0][q];
                    } else {                           // latent features 128u + 64hf ..
                        const float sc = scs[i - 1];
                        uint8_t* hrow = dst + hf * kHalf + rowoff;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t cw[4] = {v[i][q].x, v[i][q].y, v[i][q].z, v[i][q].w};
                            uint32_t o[8];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                                    __nv_fp8x2_storage_t(cw[k] & 0xffffu), __NV_E4M3);
                                const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
                                    __nv_fp8x2_storage_t(cw[k] >> 16), __NV_E4M3);
                                const float2 fl = __half22float2(*reinterpret_cast<const __half2*>(&lo));
                                const float2 fh = __half22float2(*reinterpret_cast<const __half2*>(&hi));
                                o[2 * k] = pack2(fl.x * sc, fl.y * sc);
                                o[2 * k + 1] = pack2(fh.x * sc, fh.y * sc);
                            }
                            *reinterpret_cast<uint4*>(hrow + (((2 * q) ^ (r & 7)) << 4)) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                            *reinterpret_cast<uint4*>(hrow + (((2 * q + 1) ^ (r & 7)) << 4)) =
                                make_uint4(o[4], o[5], o[6], o[7]);
                        }
                    }
                    fence_async_smem();
                    mbar_arrive(&full[slot]);
                }
            }
            if (ptid == 0 && nseg > 0 && !mbar_wait(qfull, (nseg - 1) & 1, p.wait_ns))
                report(p.status, kStTimeout);
        }
    } else if (kSrc == kSrcGather && producer_warp) {
        // ------------------- cp.async gather (128 threads) -------------------
        // Thread ptid copies 16-byte chunk ptid&7 of tile rows 8k + ptid/16:
        // of feature half (ptid/8)&1 of a latent block (k = 0..7), or of the
        // shared key for the rows whose k%2 is that half.  Eight lanes cover
        // one 128-byte row segment, so a warp request reads whole lines.  A
        // thread's copies arrive on the fill's barrier as they land; nothing
        // waits for them here but the drain at exit.  The selection entries
        // of the next tile are loaded while the current one is copied.
        const int ptid = warp == 0 ? lane : (warp - 9) * 32 + lane;
        const int rr = ptid >> 4, hf = (ptid >> 3) & 1, ch = ptid & 7;
        const uint32_t sw = uint32_t(rr * 128 + ((ch ^ rr) << 4));   // row 8k+rr, swizzled chunk
        if (t0 < t1) {
            int nseg = 0, fill = 0;
            Cursor cur{ts}, nxt{ts};
            cur.seek(t0, B);
            nxt.seek(t0, B);
            int nraw[8];
            auto load_sel = [&](int t) {
                nxt.advance(t);
                const SeqDesc s1 = seq_desc(p, nxt.b);
                const int e = (t - ts[nxt.b]) * kLT + rr;
#pragma unroll
                for (int k = 0; k < 8; ++k) nraw[k] = sel_raw(p, nxt.b, s1, e + 8 * k);
            };
            load_sel(t0);
            const uint8_t* base = reinterpret_cast<const uint8_t*>(p.ckv) + ch * 16;
            bool ok = true;
            for (int t = t0; t < t1 && ok; ++t) {
                cur.advance(t);
                const int b = cur.b;
                const SeqDesc sd = seq_desc(p, b);
                int grow[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    bool v;
                    grow[k] = sel_row(p, sd, nraw[k], &v);
                }
                if (t + 1 < t1) load_sel(t + 1);
                if (t == t0 || t == ts[b]) {
                    if (ptid == 0) {
                        if (nseg > 0 && !mbar_wait(qfree, (nseg - 1) & 1, p.wait_ns)) {
                            fail();
                        } else {
                            mbar_arrive_expect_tx(qfull, 9 * H * 128);
                            for (int kb = 0; kb < 9; ++kb)
                                tma_load_2d(qs + kb * H * 128, &qmap, kb * 64, b * H, qfull);
                        }
                    }
                    ++nseg;
                }
                for (int i = 0; i < kFills; ++i, ++fill) {
                    const int slot = fill % kSlots, round = fill / kSlots;
                    if (*abort_flag) { ok = false; break; }
                    if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, p.wait_ns)) {
                        fail();
                        ok = false;
                        break;
                    }
                    uint8_t* dst = ring + slot * kSlot + sw;
                    MLA_CHECK(slot < kSlots && sw + 7 * 1024 + 16 <= uint32_t(kHalf), p.status);
                    if (i == 0) {                      // shared-key features 512..575
#pragma unroll
                        for (int m = 0; m < 4; ++m)
                            cp_async16(dst + (2 * m + hf) * 1024,
                                       base + int64_t(grow[2 * m + hf]) * (kCkv * 2) + kLatent * 2);
                    } else {                           // latent features 128(i-1) + 64hf ..
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            cp_async16(dst + hf * kHalf + k * 1024,
                                       base + int64_t(grow[k]) * (kCkv * 2) + (128 * (i - 1) + 64 * hf) * 2);
                    }
                    cp_async_arrive_noinc(&full[slot]);
                }
            }
            cp_async_wait_all();   // nothing this thread started is still in flight at exit
            if (ptid == 0 && nseg > 0 && !mbar_wait(qfull, (nseg - 1) & 1, p.wait_ns))
                report(p.status, kStTimeout);
        }
    } else if (warp == 0) {
        // ------------------------------- TMA -------------------------------
        // Decode: the whole warp walks the tiles and waits on the ring; one
        // elected lane issues the tiled loads of 64 contiguous cache rows.
        // (An L2 prefetch of the next tiles measured slower at every distance
        // tried: it competes with these loads for the TMA unit.)
        if (t0 < t1) {
            if (elect_one()) {
                tma_prefetch_desc(&cmap);
                tma_prefetch_desc(&qmap);
            }
            const uint64_t policy = l2_evict_first_policy();
            int filled[kSlots];
            for (int s = 0; s < kSlots; ++s) filled[s] = 0;
            int nseg = 0, fill = 0;
            Cursor cur{ts};
            cur.seek(t0, B);
            bool ok = true;
            for (int t = t0; t < t1 && ok; ++t) {
                cur.advance(t);
                const int b = cur.b;
                if (t == t0 || t == ts[b]) {
                    // q~ of sequence b, once the previous segment's Q.K^T is done
                    if (nseg > 0 && !warp_wait(qfree, (nseg - 1) & 1, p.wait_ns)) {
                        if (elect_one()) fail();
                        break;
                    }
                    if (elect_one()) {
                        mbar_arrive_expect_tx(qfull, 9 * H * 128);
                        for (int kb = 0; kb < 9; ++kb)
                            tma_load_2d(qs + kb * H * 128, &qmap, kb * 64, b * H, qfull);
                    }
                    __syncwarp();
                    ++nseg;
                }
                const int row = int(p.cu[b]) + (t - ts[b]) * kLT;
                for (int i = 0; i < kFills; ++i, ++fill) {
                    const int slot = fill % kSlots, round = fill / kSlots;
                    if (*abort_flag) { ok = false; break; }
                    if (round > 0 && !warp_wait(&empty[slot], (round - 1) & 1, p.wait_ns)) {
                        if (elect_one()) fail();
                        ok = false;
                        break;
                    }
                    uint8_t* dst = ring + slot * kSlot;
                    MLA_CHECK(slot < kSlots && row >= 0, p.status);
                    if (elect_one()) {
                        if (i == 0) {          // shared-key features 512..575
                            mbar_arrive_expect_tx(&full[slot], kHalf);
                            tma_load_2d_hint(dst, &cmap, kLatent, row, &full[slot], policy);
                        } else {               // latent features 128*(i-1) .. +127
                            mbar_arrive_expect_tx(&full[slot], kSlot);
                            tma_load_2d_hint(dst, &cmap, 128 * (i - 1), row, &full[slot], policy);
                            tma_load_2d_hint(dst + kHalf, &cmap, 128 * (i - 1) + 64, row,
                                             &full[slot], policy);
                        }
                    }
                    __syncwarp();
                    filled[slot] = round + 1;
                }
            }
            for (int s = 0; s < kSlots; ++s)
                if (filled[s] > 0 && !warp_wait(&full[s], (filled[s] - 1) & 1, p.wait_ns) &&
                    elect_one())
                    report(p.status, kStTimeout);
            if (nseg > 0 && !warp_wait(qfull, (nseg - 1) & 1, p.wait_ns) && elect_one())
                report(p.status, kStTimeout);
        }
    } else if (warp == 1) {
        // ---------------------------- Q.K^T MMAs ----------------------------
        // The whole warp, in order: for each tile, the five fills' S (+)= Q~
        // K^T into the tile's score buffer; every lane waits, one elected
        // lane issues each MMA and commit.  Descriptors are built once and
        // advanced by their 16-byte address units; the ring slot and phase
        // advance with the fills.
        if (t0 < t1) {
            const uint64_t qdesc = smem_desc_sw128(smem_u32(qs), 16, 1024);     // Q~, K-major
            const uint64_t kdesc = smem_desc_sw128(smem_u32(ring), 16, 1024);   // keys, K-major
            const uint32_t qblk = uint32_t(H) * 8;       // one [H x 64] block of Q~
            constexpr uint32_t kSlotU = kSlot >> 4, kHalfU = kHalf >> 4;
            bool ok = true;
            int slot = 0;                                // ring slot of the next fill
            uint32_t phase = 0;                          // and the parity of its phase
            auto wait_bar = [&](uint64_t* bar, uint32_t par) -> bool {
                return warp_wait_abortable(bar, par, p.wait_ns, abort_flag);
            };
            Cursor cur{ts};
            cur.seek(t0, B);
            int nseg = 0;
            for (int t = t0; t < t1 && ok; ++t) {
                const int j = t - t0;
                cur.advance(t);
                const int b = cur.b;
                const bool first = (t == t0 || t == ts[b]);
                const bool last = (t + 1 == t1 || t + 1 == ts[b + 1]);
                if (j >= 2 && !wait_bar(&sfree[j & 1], ((j - 2) >> 1) & 1)) {
                    ok = false;
                    break;
                }
                if (first) {
                    if (!wait_bar(qfull, nseg & 1)) { ok = false; break; }
                    ++nseg;
                }
                const uint32_t d = tmem + uint32_t(j & 1) * kLT;
                for (int i = 0; i < kFills; ++i) {
                    if (!wait_bar(&full[slot], phase)) { ok = false; break; }
                    // cp.async writes come through the generic proxy: order
                    // them before the tensor core's reads of the slot
                    if (kSrc == kSrcGather) fence_async_smem();
                    tc_fence_after();
                    const uint64_t b0 = kdesc + uint32_t(slot) * kSlotU;
                    MLA_CHECK(slot < kSlots && (8 * H + 128) * 128 <= kQBytes &&
                                  uint32_t(j & 1) * kLT + kLT <= uint32_t(kColO),
                              p.status);
                    if (i == 0) {                        // shared-key features
                        const uint64_t a0 = qdesc + 8 * qblk;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            if (elect_one())
                                mma_bf16_ss(d, a0 + 2 * kk, b0 + 2 * kk, kIdescQK, kk > 0 ? 1u : 0u);
                        if (elect_one()) mma_commit(&empty[slot]);
                    } else {                             // latent block i-1
                        const uint64_t a0 = qdesc + uint32_t(2 * (i - 1)) * qblk;
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                if (elect_one())
                                    mma_bf16_ss(d, a0 + hf * qblk + 2 * kk,
                                                b0 + hf * kHalfU + 2 * kk, kIdescQK, 1u);
                    }
                    __syncwarp();
                    if (++slot == kSlots) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (last && elect_one()) mma_commit(qfree);
                if (elect_one()) mma_commit(&sfull[j & 1]);
                __syncwarp();
            }
            if (!ok && elect_one()) fail();
            if (elect_one()) mma_commit(&mdone[0]);
            __syncwarp();
            if (!warp_wait(&mdone[0], 0, p.wait_ns) && elect_one()) report(p.status, kStTimeout);
        }
    } else if (warp == kPvWarp<kSrc>) {
        // ----------------------------- P.V MMAs -----------------------------
        // O^T += C^T P^T for each tile once its probabilities are written;
        // the latent blocks' ring slots are released as their MMAs finish.
        // A tile's P.V follows its softmax, which followed its Q.K^T, so the
        // slots' Q.K^T reads are complete when these commits free them.
        // Whole warp, one elected lane issuing (as for Q.K^T).
        if (t0 < t1) {
            const uint32_t idesc_pv = idesc_bf16_f32(128, H, true, false);
            const uint64_t cdesc = smem_desc_sw128(smem_u32(ring), kHalf, 1024);  // C^T, MN-major
            const uint64_t pdesc = smem_desc_sw128(smem_u32(ps), 16, 1024);     // P, K-major
            constexpr uint32_t kSlotU = kSlot >> 4;
            bool ok = true;
            auto wait_bar = [&](uint64_t* bar, uint32_t par) -> bool {
                return warp_wait_abortable(bar, par, p.wait_ns, abort_flag);
            };
            Cursor cur{ts};
            cur.seek(t0, B);
            int s1 = 1;          // ring slot of the current tile's first latent block
            int pv_seg = 0;      // segments whose first P.V has been issued
            for (int t = t0; t < t1 && ok; ++t) {
                const int j = t - t0;
                cur.advance(t);
                const int b = cur.b;
                const bool first = (t == t0 || t == ts[b]);
                const bool last = (t + 1 == t1 || t + 1 == ts[b + 1]);
                if (!wait_bar(pfull, j & 1)) { ok = false; break; }
                if (first) {
                    // the previous segment's O^T has been read out
                    if (pv_seg > 0 && !wait_bar(oread, (pv_seg - 1) & 1)) { ok = false; break; }
                    ++pv_seg;
                }
                if (kSrc == kSrcGather) fence_async_smem();
                tc_fence_after();
                int sl = s1;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint64_t a0 = cdesc + uint32_t(sl) * kSlotU;
                    MLA_CHECK(sl < kSlots && kColO + uint32_t((u + 1) * H) <= 512u, p.status);
                    const uint32_t d = tmem + kColO + uint32_t(u * H);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (elect_one())
                            mma_bf16_ss(d, a0 + 128 * k, pdesc + 2 * k, idesc_pv,
                                        (first && k == 0) ? 0u : 1u);
                    if (elect_one()) mma_commit(&empty[sl]);
                    if (++sl == kSlots) sl = 0;
                }
                if (elect_one()) mma_commit(pfree);
                if (last && elect_one()) mma_commit(ofinal);
                __syncwarp();
                s1 += kFills;
                if (s1 >= kSlots) s1 -= kSlots;
            }
            if (!ok && elect_one()) {
                fail();
                mma_commit(ofinal);
            }
            if (elect_one()) mma_commit(&mdone[1]);
            __syncwarp();
            if (!warp_wait(&mdone[1], 0, p.wait_ns) && elect_one()) report(p.status, kStTimeout);
        }
    } else {
        // ------------------------- softmax / epilogue ------------------------
        // Warp w serves TMEM lane quadrant w%4 (head rows 32*quad..) and key
        // columns 32*half.. of each tile; for O^T it serves the same lanes
        // (latent features) of output blocks 2*half and 2*half+1.
        const int quad = warp & 3, half = (warp - 2) >> 2;
        const int r = quad * 32 + lane;
        const bool real = r < H;
        const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);
        float m = 0.f, l = 0.f;
        int nseg = -1;
        Cursor cur{ts}, nxt{ts};
        int nraw = -1;                        // sparse: this lane's entry of the next tile
        if (t0 < t1) {
            cur.seek(t0, B);
            nxt.seek(t0, B);
            if (sparse)
                nraw = sel_raw(p, nxt.b, seq_desc(p, nxt.b), (t0 - ts[nxt.b]) * kLT + half * 32 + lane);
        }
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (mbar_test(bar, parity) || *abort_flag) return;
            if (!mbar_wait(bar, parity, p.wait_ns)) fail();
        };
        for (int t = t0; t < t1; ++t) {
            const int j = t - t0;
            cur.advance(t);
            const int b = cur.b;
            const int raw = nraw;
            if (sparse && t + 1 < t1) {
                nxt.advance(t + 1);
                nraw = sel_raw(p, nxt.b, seq_desc(p, nxt.b),
                               (t + 1 - ts[nxt.b]) * kLT + half * 32 + lane);
            }
            const bool first = (t == t0 || t == ts[b]);
            const bool last = (t + 1 == t1 || t + 1 == ts[b + 1]);
            if (first) ++nseg;
            const SeqDesc sd = seq_desc(p, b);
            const int key0 = (t - ts[b]) * kLT + half * 32;
            // keys of this warp's 32 columns that take part in the softmax
            uint32_t valid;
            if (sparse) {
                bool v;
                sel_row(p, sd, raw, &v);
                valid = __ballot_sync(0xffffffffu, v);
            } else {
                const int nk = sd.T - key0;
                valid = nk >= 32 ? 0xffffffffu : (nk <= 0 ? 0u : (1u << nk) - 1u);
            }
            const int sb = j & 1;
            wait(&sfull[sb], (j >> 1) & 1);
            tc_fence_after();
            float s[32];
            tmem_ld32(lane_base + sb * kLT + half * 32, s);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfree[sb]);
            float lm = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float x = (valid >> i) & 1u ? s[i] * p.scale_log2 : -INFINITY;
                s[i] = x;
                lm = fmaxf(lm, x);
            }
            // A segment's first tile sets the running maxima; later tiles
            // rescale only when a row maximum grows past the slack, which a
            // thread can see from its own half of the row, so the halves'
            // maxima are exchanged only on those tiles.
            const bool need = first || (real && lm > m + kRescaleLog2);
            // the previous tile's P.V is done before O^T is rescaled or P rewritten
            if (j > 0) wait(pfree, (j - 1) & 1);
            tc_fence_after();
            if (bar_or(2, 256, need)) {
                xmax[(sb * 2 + half) * 128 + r] = lm;
                named_bar_sync(1, 256);
                const float rm = fmaxf(xmax[(sb * 2) * 128 + r], xmax[(sb * 2 + 1) * 128 + r]);
                if (first) {
                    m = real ? rm : 0.f;
                    l = 0.f;
                } else {
                    // rescale O^T columns (heads) of the rows whose maximum grew
                    float f = 1.f;
                    if (real && rm > m + kRescaleLog2) {
                        f = ex2(m - rm);
                        m = rm;
                        l *= f;
                    }
                    if (half == 0) fsm[r] = f;
                    named_bar_sync(1, 256);
                    for (int uu = 0; uu < 2; ++uu) {
                        const uint32_t base = lane_base + kColO + (2 * half + uu) * H;
                        for (int c0 = 0; c0 < H; c0 += 16) {
                            float v[16];
                            tmem_ld16(base + c0, v);
                            tmem_ld_wait();
                            uint32_t w[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[i] * fsm[c0 + i]);
                            tmem_st16(base + c0, w);
                        }
                    }
                    tmem_st_wait();
                }
            }
            // probabilities, bf16, into P row r (128-byte swizzled K-major rows)
            uint32_t w[16];
            float ps_sum = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float a = ex2(s[2 * i] - m), bq = ex2(s[2 * i + 1] - m);
                ps_sum += a + bq;
                w[i] = pack2(a, bq);
            }
            l += ps_sum;
            MLA_CHECK(!real || (r >> 3) * 1024 + (r & 7) * 128 + 128 <= kPBytes, p.status);
            if (real) {
                uint8_t* row = ps + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<uint4*>(row + (((half * 4 + q4) ^ (r & 7)) << 4)) =
                        make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pfull);
            if (last) {
                // segment done: row sums; a sequence wholly inside this CTA
                // writes its normalised output z~ (bf16), a spanning one its
                // partial (O^T, m, l) for the fixup pass
                xsum[half * 128 + r] = l;
                named_bar_sync(1, 256);
                const float L = xsum[r] + xsum[128 + r];
                const bool single = seg[b + 1] == seg[b];
                const int slot = single ? 0 : seg[b] + (c - ts[b] / per);
                if (half == 0) {
                    inv_l[r] = L > 0.f ? 1.f / L : 0.f;
                    if (!single && real) {
                        p.ml[(int64_t(slot) * H + r) * 2] = m;
                        p.ml[(int64_t(slot) * H + r) * 2 + 1] = L;
                    }
                }
                named_bar_sync(1, 256);
                wait(ofinal, nseg & 1);
                tc_fence_after();
                for (int uu = 0; uu < 2; ++uu) {
                    const int u = 2 * half + uu, dim = u * 128 + quad * 32 + lane;
                    MLA_CHECK(dim < kLatent && b < B && kColO + uint32_t((u + 1) * H) <= 512u,
                              p.status);
                    for (int c0 = 0; c0 < H; c0 += 16) {
                        float v[16];
                        tmem_ld16(lane_base + kColO + u * H + c0, v);
                        tmem_ld_wait();
                        if (single) {
                            uint16_t* dst = p.zbuf + int64_t(b) * H * kLatent + dim;
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const __nv_bfloat16 x = __float2bfloat16_rn(v[i] * inv_l[c0 + i]);
                                dst[int64_t(c0 + i) * kLatent] = *reinterpret_cast<const uint16_t*>(&x);
                            }
                        } else {
                            float* dst = p.part + int64_t(slot) * H * kLatent + dim;
#pragma unroll
                            for (int i = 0; i < 16; ++i) dst[int64_t(c0 + i) * kLatent] = v[i];
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(oread);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0) grid_dep_trigger();
}

// q~[b,h,0:512] = W^K_h^T q[b,h,0:128] and q~[b,h,512:576] = q[b,h,128:192],
// as tensor-core GEMMs D[j, b] = sum_d W^K_h[d, j] q[b, h, d] with the latent
// features as M (A = W^K_h, MN-major), the sequences as N (B = queries,
// K-major) and K = 128.  Work items are (head, block of kAbN sequences) in
// head-major order; each CTA takes a contiguous range of them, so it loads a
// head's W^K (128 x 512, 128 KB in eight boxes) once per head it visits and
// streams the query blocks through two stages.  Per item, four M=128 GEMMs
// (the four 128-feature blocks of j, eight K=16 MMAs each) fill one of two
// 256-column TMEM buffers while four epilogue warps convert and store the
// other.  Roles: warp 0 TMA, warp 1 MMA issue (whole warp, one elected lane
// issuing), warps 2-9 epilogue (thread = latent feature within a block; the
// two warps of a TMEM lane quadrant take two feature blocks each).
constexpr int kAbN = 64;                                  // sequences per item
constexpr int kAbWBytes = 4 * 2 * 16384;                  // W^K_h: 4 blocks x two 64-j boxes
constexpr int kAbQStage = 2 * kAbN * 128;                 // 64 sequences x 128 d
constexpr size_t kAbsorbSmem = 1024 + kAbWBytes + 2 * kAbQStage + 128;
constexpr uint32_t kIdescAbs = idesc_bf16_f32(128, kAbN, true, false);

constexpr int kAbThreads = 10 * 32;
__global__ void __launch_bounds__(kAbThreads, 1) latent_absorb_kernel(
    const __grid_constant__ CUtensorMap wkmap, const __grid_constant__ CUtensorMap qmap,
    const uint16_t* q, uint16_t* qt, const uint16_t* wv, int B, int H, int nblk,
    long long wait_ns, int* status) {
    // the work split launched next reads none of this kernel's output
    if (threadIdx.x == 0) grid_dep_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* wsm = sm;                                    // [4 blocks][2 halves][128 d][64 j]
    uint8_t* qsm = sm + kAbWBytes;                        // [2 stages][2 halves][kAbN b][64 d]
    uint64_t* bars = reinterpret_cast<uint64_t*>(qsm + 2 * kAbQStage);
    uint64_t* wfull = bars;                               // W^K of the current head landed
    uint64_t* wfree = bars + 1;                           // MMAs of the previous head done
    uint64_t* qfull = bars + 2;                           // [2]
    uint64_t* qempty = bars + 4;                          // [2]
    uint64_t* tfull = bars + 6;                           // [2] MMA -> epilogue
    uint64_t* tempty = bars + 8;                          // [2] epilogue -> MMA
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 10);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int items = H * nblk;
    const int i0 = int((int64_t(items) * blockIdx.x) / gridDim.x);
    const int i1 = int((int64_t(items) * (blockIdx.x + 1)) / gridDim.x);
    if (threadIdx.x == 0) {
        mbar_init(wfull, 1);
        mbar_init(wfree, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 8);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    auto fail = [&]() {
        report(status, kStTimeout);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ------------------------------- TMA -------------------------------
        if (lane == 0) {
            tma_prefetch_desc(&wkmap);
            tma_prefetch_desc(&qmap);
            int cur_h = -1, nheads = 0, wfilled = 0;
            int qf[2] = {0, 0};
            for (int it = i0, k = 0; it < i1; ++it, ++k) {
                if (*abort_flag) break;
                const int h = it / nblk, blk = it - h * nblk;
                if (h != cur_h) {
                    // the previous head's MMAs read W^K before it is replaced
                    if (nheads > 0 && !mbar_wait(wfree, (nheads - 1) & 1, wait_ns)) {
                        fail();
                        break;
                    }
                    mbar_arrive_expect_tx(wfull, kAbWBytes);
                    for (int jb = 0; jb < 4; ++jb)
                        for (int hf = 0; hf < 2; ++hf)
                            tma_load_2d(wsm + jb * 32768 + hf * 16384, &wkmap, jb * 128 + hf * 64,
                                        h * 128, wfull);
                    // W^V rows of this head, into L2 for the output projection
                    for (int qq = 0; qq < 4; ++qq)
                        prefetch_l2(wv + (int64_t(h) * kDv + qq * 32) * kLatent, 32 * kLatent * 2);
                    cur_h = h;
                    ++nheads;
                    wfilled = nheads;
                }
                const int s = k & 1;
                if (k >= 2 && !mbar_wait(&qempty[s], ((k >> 1) - 1) & 1, wait_ns)) {
                    fail();
                    break;
                }
                mbar_arrive_expect_tx(&qfull[s], kAbQStage);
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_3d(qsm + s * kAbQStage + hf * kAbN * 128, &qmap, hf * 64, h,
                                blk * kAbN, &qfull[s]);
                qf[s] = (k >> 1) + 1;
            }
            for (int s = 0; s < 2; ++s)
                if (qf[s] > 0 && !mbar_wait(&qfull[s], (qf[s] - 1) & 1, wait_ns))
                    report(status, kStTimeout);
            if (wfilled > 0 && !mbar_wait(wfull, (wfilled - 1) & 1, wait_ns))
                report(status, kStTimeout);
        }
    } else if (warp == 1) {
        // ------------------------------- MMA -------------------------------
        bool ok = true;
        int cur_h = -1, nheads = 0, last_u = -1, last_par = 0;
        const uint32_t wa = smem_u32(wsm), qa = smem_u32(qsm);
        for (int it = i0, k = 0; it < i1 && ok; ++it, ++k) {
            const int h = it / nblk;
            if (h != cur_h) {
                if (nheads > 0 && elect_one()) mma_commit(wfree);   // previous head's reads
                __syncwarp();
                if (!warp_wait_abortable(wfull, nheads & 1, wait_ns, abort_flag)) { ok = false; break; }
                cur_h = h;
                ++nheads;
            }
            const int s = k & 1, u = k & 1;
            if (!warp_wait_abortable(&qfull[s], (k >> 1) & 1, wait_ns, abort_flag) ||
                (k >= 2 && !warp_wait_abortable(&tempty[u], ((k >> 1) - 1) & 1, wait_ns, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int jb = 0; jb < 4; ++jb) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = smem_desc_sw128(wa + jb * 32768 + kk * 2048, 16384, 1024);
                    const uint64_t bd = smem_desc_sw128(
                        qa + s * kAbQStage + (kk >> 2) * kAbN * 128 + (kk & 3) * 32, 16, 1024);
                    if (elect_one())
                        mma_bf16_ss(tmem + uint32_t(u * 256 + jb * kAbN), ad, bd, kIdescAbs,
                                    kk > 0 ? 1u : 0u);
                }
            }
            if (elect_one()) mma_commit(&qempty[s]);
            if (elect_one()) mma_commit(&tfull[u]);
            __syncwarp();
            last_u = u;
            last_par = (k >> 1) & 1;
        }
        if (!ok && elect_one()) fail();
        // the accumulators must not be released while an MMA still writes them
        if (last_u >= 0 && !warp_wait(&tfull[last_u], last_par, wait_ns) && elect_one())
            report(status, kStTimeout);
    } else {
        // ----------------------------- epilogue -----------------------------
        // warp w: TMEM lanes 32*(w%4).. = latent features 32*(w%4).. of the
        // feature blocks 2*jh and 2*jh+1 (jh = (w-2)/4); 64 columns (one
        // block's 64 sequences) loaded per wait
        const int quad = warp & 3, jh = (warp - 2) >> 2;
        const int et = threadIdx.x - 64;                  // 0..255
        for (int it = i0, k = 0; it < i1; ++it, ++k) {
            const int h = it / nblk, blk = it - h * nblk;
            const int u = k & 1;
            bool ok = !*abort_flag && mbar_wait(&tfull[u], (k >> 1) & 1, wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0 && !*abort_flag) fail();
                break;
            }
            tc_fence_after();
            const int b0 = blk * kAbN;
#pragma unroll 1
            for (int jj = 0; jj < 2; ++jj) {
                const int jb = 2 * jh + jj;
                const int j = jb * 128 + quad * 32 + lane;
                float v[kAbN];
#pragma unroll
                for (int c0 = 0; c0 < kAbN; c0 += 16)
                    tmem_ld16(tmem + (uint32_t(quad * 32) << 16) + uint32_t(u * 256 + jb * kAbN + c0),
                              *reinterpret_cast<float(*)[16]>(v + c0));
                tmem_ld_wait();
                uint16_t* dst = qt + (int64_t(b0) * H + h) * kCkv + j;
#pragma unroll
                for (int i = 0; i < kAbN; ++i)
                    if (b0 + i < B) {
                        const __nv_bfloat16 x = __float2bfloat16_rn(v[i]);
                        dst[int64_t(i) * H * kCkv] = *reinterpret_cast<const uint16_t*>(&x);
                    }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[u]);
            // the 64 shared-key features pass through: eight 16-byte pieces per
            // sequence, all loads issued before the stores
            uint4 x[kAbN * 8 / 256];
#pragma unroll
            for (int e = 0; e < kAbN * 8 / 256; ++e) {
                const int i = et + 256 * e, b = b0 + (i >> 3);
                if (b < B)
                    x[e] = *reinterpret_cast<const uint4*>(q + (int64_t(b) * H + h) * kDqk + 128 +
                                                           (i & 7) * 8);
            }
#pragma unroll
            for (int e = 0; e < kAbN * 8 / 256; ++e) {
                const int i = et + 256 * e, b = b0 + (i >> 3);
                if (b < B)
                    *reinterpret_cast<uint4*>(qt + (int64_t(b) * H + h) * kCkv + kLatent + (i & 7) * 8) =
                        x[e];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}


// Block-wide exclusive scan of one int per thread (1024 threads); returns the
// exclusive prefix and writes the total to *total.
__device__ int block_scan_excl(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int s = lane < int(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    const int excl = incl - v + (warp > 0 ? warp_sums[warp - 1] : 0);
    *total = warp_sums[31];
    __syncthreads();
    return excl;
}

// The work split.  Tiles per sequence: ceil(T_b / 64) (decode: T_b from the
// packed lengths, 0 when outside [1, max_seqlen], which is reported; sparse
// prefill: T_b = min(topk, P+b+1) selection entries).  n tiles in all, `per`
// = ceil(n / G) per CTA; a sequence whose tiles span several CTAs gets one
// partial slot per CTA (seg prefix) and a place in the fixup list.
__global__ void __launch_bounds__(1024) latent_sched_kernel(const int64_t* cu, const int32_t* idx,
                                                            int topk, int P, int B,
                                                            int max_seqlen, int G, int* sched,
                                                            int* status) {
    __shared__ int warp_sums[32];
    int* ts = sched + 3;
    int* seg = ts + B + 1;
    int* mlist = seg + B + 1;
    const int per_thr = (B + blockDim.x - 1) / blockDim.x;
    const int b0 = min(B, int(threadIdx.x) * per_thr), b1 = min(B, b0 + per_thr);
    auto tiles = [&](int b) -> int {
        if (idx) return (min(topk, P + b + 1) + kLT - 1) / kLT;
        const int64_t T = cu[b + 1] - cu[b];
        return (T >= 1 && T <= max_seqlen) ? int((T + kLT - 1) / kLT) : 0;
    };
    int local = 0;
    for (int b = b0; b < b1; ++b) {
        if (!idx) {
            const int64_t T = cu[b + 1] - cu[b];
            if (T < 1 || T > max_seqlen) report(status, kStInvalid);
        }
        local += tiles(b);
    }
    int n;
    int run = block_scan_excl(local, warp_sums, &n);
    for (int b = b0; b < b1; ++b) {
        ts[b] = run;
        run += tiles(b);
    }
    if (threadIdx.x == 0) ts[B] = n;
    const int per = max(1, (n + G - 1) / G);
    __syncthreads();
    auto nseg = [&](int b) -> int {
        const int nt = ts[b + 1] - ts[b];
        if (nt == 0) return 0;
        const int clo = ts[b] / per, chi = (ts[b] + nt - 1) / per;
        return chi > clo ? chi - clo + 1 : 0;
    };
    local = 0;
    int lm = 0;
    for (int b = b0; b < b1; ++b) {
        local += nseg(b);
        lm += nseg(b) > 0;
    }
    int nslots;
    run = block_scan_excl(local, warp_sums, &nslots);
    int nmulti;
    int mrun = block_scan_excl(lm, warp_sums, &nmulti);
    for (int b = b0; b < b1; ++b) {
        seg[b] = run;
        const int k = nseg(b);
        run += k;
        if (k > 0) mlist[mrun++] = b;
    }
    if (threadIdx.x == 0) {
        seg[B] = nslots;
        sched[0] = n;
        sched[1] = per;
        sched[2] = nmulti;
    }
    // runs beside the absorption (it reads none of its output); finishing
    // only after it lets the attention kernel's wait cover both
    grid_dep_wait();
    if (threadIdx.x == 0) grid_dep_trigger();
}

// Fixup: the sequences whose tiles spanned several CTAs.  Warp w of CTA
// (h, y) takes list entry 8y+w, merges its segments' (O, m, l) by
// log-sum-exp and writes the normalised z~ (bf16) like a single-CTA
// sequence.  Lane holds latent features 2*lane + 64*k (k < 8); the segments'
// maxima and sums are read by the lanes in parallel, then the partial rows
// are independent weighted sums, loaded two segments at a time.
__global__ void __launch_bounds__(256) latent_fixup_kernel(const float* part, const float* ml,
                                                           const int* sched_base, uint16_t* zbuf,
                                                           int B, int H) {
    grid_dep_wait();                             // the attention kernel's partials
    const Sched sch{sched_base};
    const int h = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = blockIdx.y * 8 + warp;
    if (k >= sch.nmulti()) return;
    const int b = sch.mlist(B)[k];
    const int* seg = sch.seg(B);
    const int s0 = seg[b], ns = seg[b + 1] - s0;
    float M = -INFINITY, L = 0.f;                // lane-local over segments lane, lane+32, ...
    for (int i = lane; i < ns; i += 32) {
        const float2 v = *reinterpret_cast<const float2*>(ml + (int64_t(s0 + i) * H + h) * 2);
        const float Mn = fmaxf(M, v.x);
        L = L * ex2(M - Mn) + v.y * ex2(v.x - Mn);
        M = Mn;
    }
    float Mw = M;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Mw = fmaxf(Mw, __shfl_xor_sync(0xffffffffu, Mw, o));
    L = M == -INFINITY ? 0.f : L * ex2(M - Mw);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float z[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) z[q] = 0.f;
    for (int i0 = 0; i0 < ns; i0 += 2) {
        float2 pv[2][8];
        float wgt[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = min(i0 + q, ns - 1);
            const float* row = part + (int64_t(s0 + i) * H + h) * kLatent + 2 * lane;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) pv[q][kk] = *reinterpret_cast<const float2*>(row + 64 * kk);
            wgt[q] = i0 + q < ns ? ex2(ml[(int64_t(s0 + i) * H + h) * 2] - Mw) * inv : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                z[2 * kk] = fmaf(wgt[q], pv[q][kk].x, z[2 * kk]);
                z[2 * kk + 1] = fmaf(wgt[q], pv[q][kk].y, z[2 * kk + 1]);
            }
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>(zbuf + (int64_t(b) * H + h) * kLatent + 2 * lane);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) dst[32 * kk] = pack2(z[2 * kk], z[2 * kk + 1]);
    if (lane == 0) grid_dep_trigger();
}

// Output projection and gate: for head h and 128 sequences (rows),
//   out[b, h*128+d] = sigmoid(gate[b, h*128+d]) * sum_j z~[b,h,j] W^V_h[d,j]
// as a tensor-core GEMM with the sequences as M (A = z~ rows, K-major), the
// 128 output features as N (B = W^V_h, K-major) and K = 512 latent features,
// streamed in eight 64-feature blocks through a four-stage ring.
// kN output features per CTA: 128 (a head's all) for large batches; for a
// batch of at most 128 sequences the head's features are split over two
// CTAs (N = 64) so twice as many SMs stream W^V.
constexpr int kOutStages = 4;
template <int kN>
constexpr int kOutStageOf = 16384 + kN * 128;    // z~ block (128 rows) + W^V block
template <int kN>
constexpr size_t kOutSmemOf = 1024 + size_t(kOutStages) * kOutStageOf<kN> + 128;

template <int kN>
__global__ void __launch_bounds__(192) latent_out_kernel(
    const __grid_constant__ CUtensorMap zmap, const __grid_constant__ CUtensorMap wvmap,
    const int* sched_base, const uint16_t* gate, uint16_t* out, int B, int H, int zrows,
    long long wait_ns, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int kOutStage = kOutStageOf<kN>;
    constexpr uint32_t kIdescOut = idesc_bf16_f32(128, kN, false, false);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + kOutStages * kOutStage);
    uint64_t* empty = full + kOutStages;
    uint64_t* done = empty + kOutStages;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);
    const int h = blockIdx.x, b0 = blockIdx.y * 128, n0 = blockIdx.z * kN;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int* ts = Sched{sched_base}.ts();
    if (threadIdx.x == 0) {
        for (int i = 0; i < kOutStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_holder, kN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    grid_dep_wait();                                     // z~ from the attention and fixup kernels
    if (warp == 0 && lane == 0) {
        int filled[kOutStages] = {0, 0, 0, 0};
        for (int kb = 0; kb < 8; ++kb) {
            const int st = kb % kOutStages, r = kb / kOutStages;
            if (r > 0 && !mbar_wait(&empty[st], (r - 1) & 1, wait_ns)) {
                report(status, kStTimeout);
                break;
            }
            mbar_arrive_expect_tx(&full[st], kN * 128 + zrows * 128);
            tma_load_3d(sm + st * kOutStage, &zmap, kb * 64, h, b0, &full[st]);
            tma_load_2d(sm + st * kOutStage + 16384, &wvmap, kb * 64, h * kDv + n0, &full[st]);
            filled[st] = r + 1;
        }
        for (int i = 0; i < kOutStages; ++i)
            if (filled[i] > 0 && !mbar_wait(&full[i], (filled[i] - 1) & 1, wait_ns))
                report(status, kStTimeout);
    } else if (warp == 1 && lane == 0) {
        const uint32_t sa = smem_u32(sm);
        bool ok = true;
        for (int kb = 0; kb < 8 && ok; ++kb) {
            const int st = kb % kOutStages;
            if (!mbar_wait(&full[st], (kb / kOutStages) & 1, wait_ns)) {
                report(status, kStTimeout);
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = smem_desc_sw128(sa + st * kOutStage + kk * 32, 16, 1024);
                const uint64_t bd = smem_desc_sw128(sa + st * kOutStage + 16384 + kk * 32, 16, 1024);
                mma_bf16_ss(tmem, ad, bd, kIdescOut, (kb > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&empty[st]);
        }
        mma_commit(done);
    } else if (warp >= 2) {
        // thread = sequence row (TMEM lane), kN output features; the gate
        // logits are loaded first so their latency overlaps the GEMM
        const int quad = warp & 3, b = b0 + quad * 32 + lane;
        const bool live = b < B && ts[b + 1] > ts[b];
        uint4 g[kN / 8];
        const uint4* g4 = reinterpret_cast<const uint4*>(gate + (int64_t(b) * H + h) * kDv + n0);
#pragma unroll
        for (int q = 0; q < kN / 8; ++q) g[q] = (live && gate) ? __ldg(g4 + q) : make_uint4(0, 0, 0, 0);
        if (!mbar_wait(done, 0, wait_ns) && lane == 0) report(status, kStTimeout);
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < kN; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + (uint32_t(quad * 32) << 16) + c0, v);
            tmem_ld_wait();
            if (!live) continue;
            uint32_t w[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 gq = g[c0 / 8 + q];
                const uint32_t gg[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = v[8 * q + 2 * e], c = v[8 * q + 2 * e + 1];
                    w[4 * q + e] = gate ? pack2(a * sigmoidf_fast(bf_lo(gg[e])),
                                                c * sigmoidf_fast(bf_hi(gg[e])))
                                        : pack2(a, c);
                }
            }
            uint4* o4 = reinterpret_cast<uint4*>(out + (int64_t(b) * H + h) * kDv + n0 + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q) o4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, kN);
}

// FP8 latent records: one warp per cache row.  Group g (features 128g..) is
// quantised like the index keys (scale = amax/448, codes e4m3(x * 448/amax),
// nearest even, saturating; a zero group has scale 0); record bytes: codes
// 0..511, scales 512..527, the 64 bf16 shared-key features 528..655.
__global__ void __launch_bounds__(256) quantize_latent_kernel(const uint16_t* ckv, uint8_t* rec,
                                                              int64_t rows) {
    const int lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const uint16_t* x = ckv + row * kCkv;
    uint8_t* o = rec + row * kRec;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint2 v = *reinterpret_cast<const uint2*>(x + g * 128 + lane * 4);
        const float f0 = bf_lo(v.x), f1 = bf_hi(v.x), f2 = bf_lo(v.y), f3 = bf_hi(v.y);
        float amax = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        uint32_t c = 0;
        float sc = 0.f;
        if (amax > 0.f) {
            const float inv = 448.0f / amax;
            sc = amax / 448.0f;
            const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                make_float2(f0 * inv, f1 * inv), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                make_float2(f2 * inv, f3 * inv), __NV_SATFINITE, __NV_E4M3);
            c = uint32_t(lo) | (uint32_t(hi) << 16);
        }
        *reinterpret_cast<uint32_t*>(o + g * 128 + lane * 4) = c;
        if (lane == 0) *reinterpret_cast<float*>(o + 512 + 4 * g) = sc;
    }
    *reinterpret_cast<uint32_t*>(o + 528 + lane * 4) =
        *reinterpret_cast<const uint32_t*>(x + 512 + lane * 2);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

LatentPlan plan_latent(int B, int H, int sms) {
    LatentPlan pl{};
    pl.ctas = sms;
    const size_t slots = 2 * size_t(sms);        // segments of sequences spanning CTAs
    pl.qt_off = 0;
    pl.sched_off = pl.qt_off + align256(size_t(B) * H * kCkv * 2);
    pl.part_off = pl.sched_off + align256((3 + 2 * size_t(B + 1) + sms) * 4);
    pl.ml_off = pl.part_off + align256(slots * H * kLatent * 4);
    pl.z_off = pl.ml_off + align256(slots * H * 2 * 4);
    pl.total = pl.z_off + align256(size_t(B) * H * kLatent * 2);
    return pl;
}

cudaError_t launch_latent_decode(const LatentArgs& a, const LatentPlan& pl, const DeviceInfo& dev,
                                 const Knobs& kn, const KernelTimer& tm, cudaStream_t st) {
    static_assert(kLatSmem <= 227 * 1024, "shared memory budget");
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    uint16_t* qt = reinterpret_cast<uint16_t*>(ws + pl.qt_off);
    int* sched = reinterpret_cast<int*>(ws + pl.sched_off);
    float* part = reinterpret_cast<float*>(ws + pl.part_off);
    float* ml = reinterpret_cast<float*>(ws + pl.ml_off);
    uint16_t* zbuf = reinterpret_cast<uint16_t*>(ws + pl.z_off);

    // W^K as [H*128 rows (h, d)][512], W^V likewise; queries as [B][H][192]
    CUtensorMap wkmap, wvmap, q3map, cmap, qmap, zmap;
    cudaError_t e = encode_tmap_2d_bf16(&wkmap, a.w_kc, kLatent, uint64_t(a.H) * 128, kLatent * 2,
                                        64, 128);
    if (e != cudaSuccess) return e;
    const bool small = a.B <= 128;               // one sequence block: split each head's features
    e = encode_tmap_2d_bf16(&wvmap, a.w_vc, kLatent, uint64_t(a.H) * kDv, kLatent * 2, 64,
                            small ? 64 : 128);
    if (e != cudaSuccess) return e;
    e = encode_tmap_3d_bf16(&q3map, a.q, kDqk, a.H, a.B, kDqk * 2, uint64_t(a.H) * kDqk * 2, 64,
                            1, kAbN);
    if (e != cudaSuccess) return e;
    const int src = a.rec ? kSrcFp8 : a.idx ? kSrcGather : kSrcTma;
    if (src == kSrcTma) {
        e = encode_tmap_2d_bf16(&cmap, a.ckv, kCkv, uint64_t(a.total), kCkv * 2, 64, kLT);
        if (e != cudaSuccess) return e;
    } else {                                  // rows are read by the producer threads
        cmap = wkmap;
    }
    e = encode_tmap_2d_bf16(&qmap, qt, kCkv, uint64_t(a.B) * a.H, kCkv * 2, 64, a.H);
    if (e != cudaSuccess) return e;
    const int zrows = a.B < 128 ? (a.B + 15) / 16 * 16 : 128;   // rows a z~ box carries
    e = encode_tmap_3d_bf16(&zmap, zbuf, kLatent, a.H, a.B, kLatent * 2,
                            uint64_t(a.H) * kLatent * 2, 64, 1, zrows);
    if (e != cudaSuccess) return e;

    e = cudaFuncSetAttribute(latent_absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kAbsorbSmem));
    if (e != cudaSuccess) return e;
    const int nblk = (a.B + kAbN - 1) / kAbN;
    latent_absorb_kernel<<<std::min(a.H * nblk, dev.sms), kAbThreads, kAbsorbSmem, st>>>(
        wkmap, q3map, a.q, qt, a.w_vc, a.B, a.H, nblk, kn.wait_limit_ns, dev.status);
    // the four kernels after the absorption are launched programmatically
    // dependent: each may start while its predecessor finishes and waits on
    // the device for that predecessor's results
    e = launch_after_prev(latent_sched_kernel, dim3(1), dim3(1024), 0, st, a.cu, a.idx, a.topk, a.P,
                          a.B, a.max_seqlen, pl.ctas, sched, dev.status);
    if (e != cudaSuccess) return e;
    const void* kern = src == kSrcFp8      ? reinterpret_cast<const void*>(mla_latent_kernel<kSrcFp8>)
                       : src == kSrcGather ? reinterpret_cast<const void*>(mla_latent_kernel<kSrcGather>)
                                           : reinterpret_cast<const void*>(mla_latent_kernel<kSrcTma>);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kLatSmem));
    if (e != cudaSuccess) return e;
    LatParams p{sched, a.cu, a.idx, a.topk, a.P, a.ckv, a.total, part, ml, zbuf, a.rec, a.B, a.H,
                a.scale * 1.4426950408889634f, kn.wait_limit_ns, dev.status};
    if (tm.begin) cudaEventRecord(tm.begin, st);
    if (src == kSrcFp8)
        e = launch_after_prev(mla_latent_kernel<kSrcFp8>, dim3(pl.ctas), dim3(kThreadsOf<kSrcFp8>),
                              kLatSmem, st, cmap, qmap, p);
    else if (src == kSrcGather)
        e = launch_after_prev(mla_latent_kernel<kSrcGather>, dim3(pl.ctas),
                              dim3(kThreadsOf<kSrcGather>), kLatSmem, st, cmap, qmap, p);
    else
        e = launch_after_prev(mla_latent_kernel<kSrcTma>, dim3(pl.ctas), dim3(kThreadsOf<kSrcTma>),
                              kLatSmem, st, cmap, qmap, p);
    if (tm.end) cudaEventRecord(tm.end, st);
    if (e != cudaSuccess) return e;
    // the fixup list holds at most min(B, CTAs) sequences
    e = launch_after_prev(latent_fixup_kernel, dim3(a.H, (min(a.B, pl.ctas) + 7) / 8), dim3(256), 0,
                          st, static_cast<const float*>(part), static_cast<const float*>(ml),
                          static_cast<const int*>(sched), zbuf, a.B, a.H);
    if (e != cudaSuccess) return e;
    if (small) {
        e = cudaFuncSetAttribute(latent_out_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(kOutSmemOf<64>));
        if (e != cudaSuccess) return e;
        e = launch_after_prev(latent_out_kernel<64>, dim3(a.H, 1, 2), dim3(192), kOutSmemOf<64>, st,
                              zmap, wvmap, static_cast<const int*>(sched), a.gate, a.out, a.B, a.H,
                              zrows, kn.wait_limit_ns, dev.status);
    } else {
        e = cudaFuncSetAttribute(latent_out_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(kOutSmemOf<128>));
        if (e != cudaSuccess) return e;
        e = launch_after_prev(latent_out_kernel<128>, dim3(a.H, (a.B + 127) / 128, 1), dim3(192),
                              kOutSmemOf<128>, st, zmap, wvmap, static_cast<const int*>(sched),
                              a.gate, a.out, a.B, a.H, zrows, kn.wait_limit_ns, dev.status);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_quantize_latent(const uint16_t* ckv, uint8_t* rec, int64_t rows,
                                   cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    quantize_latent_kernel<<<unsigned((rows + 7) / 8), 256, 0, st>>>(ckv, rec, rows);
    return cudaGetLastError();
}

}  // namespace mla
