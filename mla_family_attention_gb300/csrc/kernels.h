// Internal launch interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Host-side validation happens in api.cu; these launchers
// only enqueue work and return the CUDA launch error.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mla {

constexpr int kDqk = 192;   // 128 content + 64 shared key features
constexpr int kDv = 128;    // value features
constexpr int kIndexHeads = 32;
constexpr int kIndexDim = 128;
constexpr int kMaxTopk = 2048;

struct DeviceInfo {
    int sms = 0;
    int* status = nullptr;  // device status word
};

struct Knobs {
    long long wait_limit_ns;
    int stall_stage;
    int sparse_chunk;   // 0 = default
    int prefill_ctas;   // CTAs per MMA in the prefill: 0 = default (1), 1 or 2
};

// Optional event pair recorded around an operation's dominant kernel.
struct KernelTimer {
    cudaEvent_t begin = nullptr, end = nullptr;
};

#ifdef __CUDACC__
// Launch with programmatic stream serialization: the kernel may begin while
// the previous kernel of the stream finishes, so it calls grid_dep_wait
// before it reads that kernel's results.
template <typename... P, typename... A>
inline cudaError_t launch_after_prev(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t st, A&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
}
#endif

// ------------------------------ decode ------------------------------------
// Where sequence b's cache lives.  Packed (cap == 0): [H, T_b, D] at
// position offset cu[b], T_b = cu[b+1] - cu[b].  Fixed capacity (cap > 0):
// [B, H, cap, D], T_b = lens[b] + add.
struct SeqLayout {
    const int64_t* cu = nullptr;
    const int64_t* lens = nullptr;
    int64_t cap = 0;
    int add = 0;
#ifdef __CUDACC__
    __device__ __forceinline__ int64_t len(int b) const {
        return cap > 0 ? lens[b] + add : cu[b + 1] - cu[b];
    }
    // Row (in units of one position's features) of position 0 of (b, h).
    __device__ __forceinline__ int64_t row0(int b, int h, int H, int64_t T) const {
        return cap > 0 ? (int64_t(b) * H + h) * cap : cu[b] * H + int64_t(h) * T;
    }
#endif
};

struct DecodeArgs {
    const uint16_t* q;       // [B,H,192]
    const uint16_t* k;       // cache keys, laid out as `seq` says
    const uint16_t* v;       // cache values
    SeqLayout seq;
    const int32_t* idx;      // sparse only: [B,topk]
    const uint16_t* gate;    // [B,H*128] or null
    uint16_t* out;           // [B,H*128]
    int B, H, max_seqlen, topk;
    float scale;
    void* ws;
    size_t ws_bytes;
};

// Work decomposition shared by workspace sizing and launch.
struct DecodePlan {
    int chunk;           // positions (dense) or index entries (sparse) per work item
    int max_chunks;      // work items per (b,h) at most
    size_t acc_off, ml_off, items_off, total;  // workspace layout in bytes
};

DecodePlan plan_decode(int B, int H, int max_len, bool sparse, int sparse_chunk = 0);
cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& p, bool sparse,
                          const DeviceInfo& dev, const Knobs& kn, const KernelTimer& tm,
                          cudaStream_t st);

// Unique id of the CUDA context current on this thread, 0 if there is none
// (or the driver cannot tell).  Device addresses of the library's __device__
// variables are valid for one context: a device reset makes a new one.
unsigned long long current_context_id();

// --------------------------- TMA tensor maps ------------------------------
// 2-D bf16 map over a row-major [outer][inner] array with 128-byte swizzle.
cudaError_t encode_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                                uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);

// 3-D bf16 map over [outer][mid][inner] with 128-byte swizzle; rows with
// mid >= `mid` read as zeros.
cudaError_t encode_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid,
                                uint64_t outer, uint64_t mid_bytes, uint64_t outer_bytes,
                                uint32_t box_inner, uint32_t box_mid, uint32_t box_outer = 1);

// 2-D 8-bit map over a row-major [outer][inner] byte array, 128-byte swizzle.
cudaError_t encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);

// ---------------------------- DSA indexer --------------------------------
struct IndexArgs {
    const uint16_t* index_q;   // [B,32,128]
    const uint16_t* index_k;   // packed [total_keys,128]
    const float* w;            // [B,32]
    const int64_t* cu;         // [B+1]
    int B, max_seqlen, topk;
    int64_t total_keys;
    int32_t* topk_idx;         // [B,topk]
    float* topk_scores;        // [B,topk] or null
    void* ws;
};

struct IndexPlan {
    size_t scores_off, hist_off, tiles_off, claims_off, total;
    size_t q8_off = 0, qs_off = 0, wq_off = 0;   // FP8 variant only
};

IndexPlan plan_index(int B, int max_seqlen, bool fp8 = false);
// FP8 index keys: k8 [total_keys,128] e4m3 codes and kscale [total_keys]
// fp32 (132 bytes per position); the queries are quantised per (b, head)
// inside, their scales folded into the head weights.
struct IndexFp8Args {
    const uint8_t* k8;
    const float* kscale;
};
cudaError_t launch_index_topk_fp8(const IndexArgs& a, const IndexFp8Args& f, const IndexPlan& p,
                                  const DeviceInfo& dev, const Knobs& kn, const KernelTimer& tm,
                                  cudaStream_t st);
// Quantise rows of `cols` bf16 values to e4m3 codes with one fp32 scale per
// row: scale = amax/448, code = e4m3(x * (448/amax)) (round to nearest even,
// saturating); an all-zero row gets scale 0 and zero codes.
cudaError_t launch_quantize_rows_e4m3(const uint16_t* x, uint8_t* codes, float* scale,
                                      int64_t rows, int cols, cudaStream_t st);
cudaError_t launch_index_topk(const IndexArgs& a, const IndexPlan& p, const DeviceInfo& dev,
                              const Knobs& kn, const KernelTimer& tm, cudaStream_t st);

// ----------------------------- DSA prefill ---------------------------------
struct PrefillIndexArgs {
    const uint16_t* index_q;   // [Tq,32,128]
    const uint16_t* index_k;   // [Tk,128]
    const float* w;            // [Tq,32]
    int Tq, Tk, topk;
    int32_t* topk_idx;         // [Tq,topk]
    float* topk_scores;        // [Tq,topk] or null
    void* ws;                  // prefill_index_ws(Tq, Tk) bytes: fp32 score rows
};

size_t prefill_index_ws(int Tq, int Tk);
cudaError_t launch_prefill_index_topk(const PrefillIndexArgs& a, const DeviceInfo& dev,
                                      const Knobs& kn, const KernelTimer& tm, cudaStream_t st);

// ------------------------------ prefill -----------------------------------
struct PrefillArgs {
    const uint16_t* q;       // [B,H,Tq,192]
    const uint16_t* k;       // [B,H,kv_cap,192]; positions 0..Tk-1 used
    const uint16_t* v;       // [B,H,kv_cap,128]
    const uint16_t* gate;    // [B,Tq,H*128] or null
    uint16_t* out;           // [B,Tq,H*128]
    int B, H, Tq, Tk, kv_cap;
    float scale;
};

cudaError_t launch_prefill(const PrefillArgs& a, const DeviceInfo& dev, const Knobs& kn,
                           const KernelTimer& tm, cudaStream_t st);

// ---------------------------- cache append --------------------------------
struct AppendArgs {
    const uint16_t* k_new;   // [B,H,Tn,192]
    const uint16_t* v_new;   // [B,H,Tn,128]
    uint16_t* k_cache;       // [B,H,cap,192]
    uint16_t* v_cache;       // [B,H,cap,128]
    const int64_t* start;    // device [B] or null (then `start_all`)
    int64_t start_all;
    int B, H, Tn;
    int64_t cap;
};

cudaError_t launch_cache_append(const AppendArgs& a, const DeviceInfo& dev, const KernelTimer& tm,
                                cudaStream_t st);

// ------------------------ absorbed-latent decode ---------------------------
constexpr int kLatent = 512;               // latent features c_s
constexpr int kCkv = kLatent + 64;         // cached per position: c_s ++ r_s

struct LatentArgs {
    const uint16_t* q;       // [B,H,192] expanded-form queries (sparse prefill: B = tokens)
    const uint16_t* ckv;     // packed [total,576]
    const int64_t* cu;       // decode: [B+1]; null for sparse prefill
    const uint16_t* w_kc;    // [H,128,512]
    const uint16_t* w_vc;    // [H,128,512]
    const uint16_t* gate;    // [B,H*128] or null
    uint16_t* out;           // [B,H*128]
    int B, H, max_seqlen;
    int64_t total;
    float scale;
    void* ws;
    const int32_t* idx = nullptr;   // sparse prefill: [B][topk] selections
    int topk = 0, P = 0;            // sparse prefill: selection width, cached positions
    const uint8_t* rec = nullptr;   // FP8 cache: [total][656] records instead of ckv
};

struct LatentPlan {
    int ctas;                 // attention CTAs (one per SM)
    size_t qt_off, sched_off, part_off, ml_off, z_off, total;
};

LatentPlan plan_latent(int B, int H, int sms);
// FP8 latent records [rows][656] from bf16 latent rows [rows][576].
cudaError_t launch_quantize_latent(const uint16_t* ckv, uint8_t* rec, int64_t rows,
                                   cudaStream_t st);
cudaError_t launch_latent_decode(const LatentArgs& a, const LatentPlan& p, const DeviceInfo& dev,
                                 const Knobs& kn, const KernelTimer& tm, cudaStream_t st);

// --------------------------- measurement aid ---------------------------
// Plain gather of the rows dsa_sparse_decode reads (XOR-reduced into one
// word per CTA of `sink`, gather_probe_blocks(dev) words).
int gather_probe_blocks(const DeviceInfo& dev);
cudaError_t launch_gather_probe(const uint16_t* k, const uint16_t* v, const int64_t* cu,
                                const int32_t* idx, int topk, int B, int H, uint32_t* sink,
                                const DeviceInfo& dev, const KernelTimer& tm, cudaStream_t st);

}  // namespace mla
