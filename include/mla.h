/*
 * mla.h - C ABI of the GB300 (sm_103a) Gated MLA / Gated DSA attention library.
 *
 * The library computes the attention core of Kimi K3's Gated MLA layer and of
 * its K3.1 Gated DSA variant, below the modules the pages show:
 *
 *   - Kimi K3 modeling code, MLA forward: per-head queries and cached keys of
 *     192 features (128 content + 64 shared key part, unrotated, identical for
 *     every head), cached values of 128 features, scale 192^-1/2
 *     ("self.scaling"), causal ("is_causal = True"), then the output reshaped
 *     to [B,T,H*128] and multiplied by sigmoid of the gate logits before
 *     o_proj.
 *   - Kimi K2 "Latent attention > KV cache" page: the same layout with 64
 *     heads, the last 64 key features a pre-rotated rotary key, no gate.
 *   - K3.1 Gated DSA post, eqs. (5), (6), (9), (10): a 32-head ReLU-weighted
 *     index score over the cached index keys, the top min(2048, t) positions,
 *     and gated MLA over those positions only.
 *
 * Conventions for every entry point:
 *   - bf16 tensors are passed as raw 16-bit patterns (mla_bf16).
 *   - Every pointer is DEVICE memory owned by the caller, contiguous, and
 *     16-byte aligned; the library never allocates, frees or keeps a pointer
 *     after the call returns.  Scratch memory is the caller's workspace
 *     `ws` of at least mla_workspace_size(...) bytes, 256-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream): they validate arguments on the host, enqueue kernels
 *     and return.  They never synchronise.  Calls that share a workspace must
 *     be ordered (same stream or events); overlapping calls on one workspace
 *     race.
 *   - Errors: a non-MLA_OK status means nothing was enqueued (except
 *     MLA_ERR_CUDA after a launch failure); mla_last_error() returns a
 *     message for the calling thread.  Faults that only the GPU can see
 *     (a cache length outside [1, max_seqlen], a selected index outside the
 *     sequence, a pipeline wait that ran out) never trap: the kernel skips
 *     the offending work, records a code in a device status word, and
 *     mla_check_device_status() reports it.
 *   - Positions are 0-based (the DSA post counts from 1).
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mla_bf16;   /* bfloat16 bit pattern */
typedef void* mla_stream;    /* cudaStream_t */

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer */
    MLA_ERR_UNSUPPORTED = 2,  /* a shape the kernels do not implement */
    MLA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    MLA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    MLA_ERR_TIMEOUT = 5,      /* a device-side pipeline wait ran out (device status) */
    MLA_ERR_BAD_INDEX = 6,    /* a selected position outside its sequence (device status) */
    MLA_ERR_CHECK = 7         /* bounds-checked debug build (-DMLA_CHECKS) only: a kernel's
                                 own index or offset check failed (device status; the
                                 message names the source file and line) */
} mla_status;

/* Operation ids for mla_workspace_size. */
enum {
    MLA_OP_PREFILL = 0,
    MLA_OP_DECODE = 1,
    MLA_OP_INDEX_TOPK = 2,
    MLA_OP_SPARSE_DECODE = 3,
    MLA_OP_CACHE_APPEND = 4,
    MLA_OP_LATENT_DECODE = 5,
    MLA_OP_PREFILL_INDEX_TOPK = 6,
    MLA_OP_SPARSE_PREFILL_LATENT = 7,
    MLA_OP_INDEX_TOPK_FP8 = 8,
    MLA_OP_GATHER_PROBE = 9     /* timing only (mla_gather_probe); no workspace */
};

/*
 * Causal gated MLA prefill (Kimi K3 MLA forward; Kimi K2 score line
 * attn_weights = matmul(q, k^T) * softmax_scale; DSA post eq. (9), (10)).
 *
 *   q    [B,H,Tq,192]  queries (128 content ++ 64 shared-key partner)
 *   k    [B,H,Tk,192]  cached keys including the Tq new ones at the end
 *   v    [B,H,Tk,128]  cached values
 *   gate [B,Tq,H*128]  gate logits, or NULL for no gate (K2 shape)
 *   out  [B,Tq,H*128]  out[b,i,h*128+d] = z[b,h,i,d] * sigmoid(gate[b,i,h*128+d])
 *
 * Query i is at absolute position Tk-Tq+i and sees keys j <= Tk-Tq+i
 * (bottom-right aligned causal mask; Tq == Tk is an empty-cache prefill).
 * Requires 1 <= Tq <= Tk, H >= 1, B >= 1.  Softmax and gate in fp32, one
 * rounding to bf16 at the output.
 */
mla_status mla_prefill(const mla_bf16* q, const mla_bf16* k, const mla_bf16* v,
                       const mla_bf16* gate, mla_bf16* out, int B, int H, int Tq, int Tk,
                       float scale, void* ws, size_t ws_bytes, mla_stream stream);

/*
 * Split-KV gated MLA decode: one query per sequence over a packed cache
 * (Kimi K3 MLA forward in decode mode; DSA post eq. (9), (10)).
 *
 *   q          [B,H,192]
 *   k          packed: sequence b is [H, T_b, 192] starting at element cu[b]*H*192
 *   v          packed: sequence b is [H, T_b, 128] starting at element cu[b]*H*128
 *   cu_seqlens [B+1] int64 on the device, cu[0] = 0, T_b = cu[b+1]-cu[b]
 *   gate       [B,H*128] logits or NULL
 *   out        [B,H*128]
 *
 * Every cached position is visible (the current token is already in the
 * cache).  Each sequence must have 1 <= T_b <= max_seqlen; a sequence that
 * violates this is skipped (its output is left untouched) and the device
 * status records MLA_ERR_INVALID_ARG.  A uniform cache [B,H,T,D] is the case
 * cu[b] = b*T.  Partial results of position chunks are merged by
 * log-sum-exp in a fixed order, so reruns are bitwise identical.
 */
mla_status mla_decode(const mla_bf16* q, const mla_bf16* k, const mla_bf16* v,
                      const int64_t* cu_seqlens, int B, int H, int max_seqlen,
                      const mla_bf16* gate, mla_bf16* out, float scale,
                      void* ws, size_t ws_bytes, mla_stream stream);

/*
 * mla_decode for callers that cannot allocate device memory.  The pages have
 * no counterpart to this entry point: it exists for callers with no device
 * allocator of their own, such as a plugin inside a host runtime that owns
 * every device allocation, or a latency-critical loop that must not call
 * cudaMalloc (which synchronises the device).
 *
 * Same arguments, layouts and results as mla_decode, without ws/ws_bytes:
 * the scratch comes from one fixed array of MLA_NOALLOC_SCRATCH_BYTES inside
 * the library, which every GPU that loads the library holds until the
 * process exits.  The call allocates and frees nothing.
 *   - Rejects, with MLA_ERR_WORKSPACE and a message, any (B, H, max_seqlen)
 *     whose scratch need, mla_workspace_size(MLA_OP_DECODE, ...), exceeds
 *     the array (B=32, H=96, max_seqlen=8192 needs about 12.8 MB and fits).
 *   - The first call on each device, with that device current, looks up the
 *     array's device address; make that first call before any stream
 *     capture.  The address belongs to the device's current context: after
 *     a device reset (a new context) the next call looks it up again, so
 *     make that call before any capture too.
 *   - Every call shares the array and it keeps the last call's contents;
 *     nothing in it needs to start at zero.  Calls whose kernels overlap on
 *     the GPU race on the array: order them (one stream, or events).
 */
#define MLA_NOALLOC_SCRATCH_BYTES (16u << 20)
mla_status mla_decode_noalloc(const mla_bf16* q, const mla_bf16* k, const mla_bf16* v,
                              const int64_t* cu_seqlens, int B, int H, int max_seqlen,
                              const mla_bf16* gate, mla_bf16* out, float scale,
                              mla_stream stream);

/*
 * In-place KV-cache append (the Kimi K2 "KV cache" update: new keys and
 * values concatenated after the cached ones on the sequence axis, here
 * written into a cache preallocated with a fixed capacity).
 *
 *   k_new   [B,H,Tn,192]        keys of the Tn new tokens
 *   v_new   [B,H,Tn,128]        their values
 *   k_cache [B,H,kv_capacity,192]  written in place:
 *           k_cache[b,h,s_b+t,:] = k_new[b,h,t,:] for t < Tn
 *   v_cache [B,H,kv_capacity,128]  likewise
 *   start   [B] int64 on the device (s_b = start[b], per-sequence lengths of
 *           a ragged batch), or NULL to use s_b = start_all for every b
 *
 * Other cache positions are not touched.  Requires B, H, Tn >= 1,
 * Tn*40 < 2^31, 0 <= start_all and start_all + Tn <= kv_capacity when start
 * is NULL; a sequence whose device start breaks that bound is skipped and
 * the device status records MLA_ERR_INVALID_ARG.  The new rows must not
 * overlap the cache.  No workspace.
 */
mla_status mla_cache_append(const mla_bf16* k_new, const mla_bf16* v_new, mla_bf16* k_cache,
                            mla_bf16* v_cache, const int64_t* start, int64_t start_all, int B,
                            int H, int Tn, int kv_capacity, mla_stream stream);

/*
 * Chunked prefill: Tq new tokens after P cached ones (Kimi K3 MLA forward with
 * a non-empty cache).  Appends k_new/v_new at positions P..P+Tq-1 of the
 * fixed-capacity caches (as mla_cache_append with start_all = P), then runs
 * causal gated attention of the Tq queries over cache positions 0..P+Tq-1:
 * query i (absolute position P+i) sees keys j <= P+i.
 *
 *   q       [B,H,Tq,192]     k_new [B,H,Tq,192]    v_new [B,H,Tq,128]
 *   k_cache [B,H,kv_capacity,192]   v_cache [B,H,kv_capacity,128]
 *   gate    [B,Tq,H*128] or NULL     out [B,Tq,H*128]
 *
 * Feeding a prompt in chunks (P = 0, c, 2c, ...) gives the same rows as one
 * mla_prefill over the whole prompt.  Cache positions at or past P+Tq are
 * never read, so the unused capacity may hold anything.  Requires
 * 0 <= P, 1 <= Tq, P+Tq <= kv_capacity.  No workspace.
 */
mla_status mla_prefill_chunk(const mla_bf16* q, const mla_bf16* k_new, const mla_bf16* v_new,
                             mla_bf16* k_cache, mla_bf16* v_cache, const mla_bf16* gate,
                             mla_bf16* out, int B, int H, int Tq, int P, int kv_capacity,
                             float scale, void* ws, size_t ws_bytes, mla_stream stream);

/*
 * Decode step over fixed-capacity caches [B,H,kv_capacity,D] with a ragged
 * batch (sequence b holds cache_seqlens[b] positions).
 *
 *   q             [B,H,192]
 *   k_new, v_new  [B,H,1,192] / [B,H,1,128] of the current token, or both
 *                 NULL.  When given they are first appended at position
 *                 cache_seqlens[b] (as mla_cache_append) and the query sees
 *                 T_b = cache_seqlens[b] + 1 positions; when NULL it sees
 *                 T_b = cache_seqlens[b] (the token is already cached).
 *   k_cache, v_cache  [B,H,kv_capacity,192] / [B,H,kv_capacity,128]
 *   cache_seqlens [B] int64 on the device; not modified (the caller
 *                 advances it after the step)
 *   gate, out     as in mla_decode
 *
 * Same arithmetic, work split and results as mla_decode on the equivalent
 * packed cache.  Requires 1 <= T_b <= max_seqlen <= kv_capacity; a sequence
 * outside that is skipped with MLA_ERR_INVALID_ARG in the device status.
 * Workspace: mla_workspace_size(MLA_OP_DECODE, B, H, max_seqlen, 0).
 */
mla_status mla_decode_cached(const mla_bf16* q, const mla_bf16* k_new, const mla_bf16* v_new,
                             mla_bf16* k_cache, mla_bf16* v_cache, const int64_t* cache_seqlens,
                             int B, int H, int kv_capacity, int max_seqlen, const mla_bf16* gate,
                             mla_bf16* out, float scale, void* ws, size_t ws_bytes,
                             mla_stream stream);

/*
 * Gated MLA decode over the absorbed 576-feature latent cache (DSA post,
 * eqs. (7)-(10), and its remark that inference absorbs W^K into the query
 * side and applies W^V after attention).  Position s of a sequence caches
 * c_s (512 normalised latent features) followed by r_s (64 shared key
 * features); head h's key is [W^K_h c_s ; r_s] and its value W^V_h c_s.
 *
 *   q          [B,H,192]  expanded-form queries (128 content ++ 64 shared)
 *   ckv        packed [total_positions,576]: sequence b is rows
 *              cu[b]..cu[b+1]-1 (total_positions = rows the allocation holds)
 *   cu_seqlens [B+1] int64 on the device
 *   w_kc       [H,128,512] W^K (row d, latent feature j)
 *   w_vc       [H,128,512] W^V
 *   gate, out  as in mla_decode
 *
 * Result: the same as mla_decode over the expanded keys and values, up to
 * rounding (the absorbed query W^K_h^T q[0:128] is rounded to bf16).  Reads
 * 1,152 cache bytes per position instead of 61,440.  Requires H a multiple
 * of 16 in [16, 96], 1 <= T_b <= max_seqlen (else the sequence is skipped
 * with MLA_ERR_INVALID_ARG in the device status, output untouched) and
 * total_positions < 2^31.  Workspace: mla_workspace_size(
 * MLA_OP_LATENT_DECODE, B, H, max_seqlen, 0) bytes (absorbed queries, the
 * work split, and per-segment partial results); it depends on the current
 * device's SM count.
 */
mla_status mla_decode_latent(const mla_bf16* q, const mla_bf16* ckv, const int64_t* cu_seqlens,
                             int64_t total_positions, int B, int H, int max_seqlen,
                             const mla_bf16* w_kc, const mla_bf16* w_vc, const mla_bf16* gate,
                             mla_bf16* out, float scale, void* ws, size_t ws_bytes,
                             mla_stream stream);

/*
 * FP8 latent cache (DSA post, cache section: the fp8_ds_mla record is 512
 * bytes of FP8 latent, 4 fp32 scales and 64 bf16 shared-key features, 656
 * bytes per position).  Record layout: bytes 0..511 the e4m3 codes of latent
 * features 0..511, in four groups of 128 with one scale each (scale =
 * amax/448, code = e4m3(x * 448/amax) rounded to nearest even, saturating,
 * computed in fp32; a zero group has scale 0); bytes 512..527 the four fp32
 * scales; bytes 528..655 the 64 bf16 shared-key features unchanged.
 *
 * mla_quantize_latent_cache writes the records rec [N,656] of N latent rows
 * ckv [N,576] bf16.  mla_decode_latent_fp8 and mla_sparse_prefill_latent_fp8
 * are mla_decode_latent and mla_sparse_prefill_latent over such records (the
 * row arguments count records); the kernels convert each record back to
 * bf16 features (code x scale, rounded to bf16) on the way into shared
 * memory, so the arithmetic after that is the bf16 path's.
 */
mla_status mla_quantize_latent_cache(const mla_bf16* ckv, uint8_t* rec, int64_t N,
                                     mla_stream stream);
mla_status mla_decode_latent_fp8(const mla_bf16* q, const uint8_t* rec, const int64_t* cu_seqlens,
                                 int64_t total_positions, int B, int H, int max_seqlen,
                                 const mla_bf16* w_kc, const mla_bf16* w_vc, const mla_bf16* gate,
                                 mla_bf16* out, float scale, void* ws, size_t ws_bytes,
                                 mla_stream stream);
mla_status mla_sparse_prefill_latent_fp8(const mla_bf16* q, const uint8_t* rec,
                                         const int32_t* topk_idx, int Tq, int Tk, int topk, int H,
                                         const mla_bf16* w_kc, const mla_bf16* w_vc,
                                         const mla_bf16* gate, mla_bf16* out, float scale,
                                         void* ws, size_t ws_bytes, mla_stream stream);

/*
 * DSA indexer score and top-k (DSA post eqs. (5) and (6)).
 *
 *   index_q     [B,NH,128]  index queries (NH must be 32)
 *   index_k     [total_keys,128] packed index keys: sequence b's keys are rows
 *               cu[b]..cu[b+1]-1; total_keys is the number of rows the
 *               allocation holds (the kernels never read past it)
 *   w           [B,NH] fp32 head weights, with the eq. (5) constant
 *               1/(sqrt(32)*sqrt(128)) already folded in by the caller
 *   topk_idx    [B,topk] int32 out: the min(topk, T_b) positions of largest
 *               score_s = sum_h w_h * max(0, q_h . k_s), ranked by (score
 *               descending, position ascending), written in ascending
 *               position order and padded with -1.  When T_b <= topk every
 *               position is returned and no score is computed.
 *   topk_scores [B,topk] fp32 out (score of each returned position; -inf on
 *               padding and when T_b <= topk) or NULL
 *
 * Requires 1 <= topk <= 2048, NH == 32, 1 <= max_seqlen <= 2^24 and
 * total_keys < 2^31.  A sequence with T_b outside [0, max_seqlen] or rows
 * past total_keys gets an all -1 output and MLA_ERR_INVALID_ARG in the
 * device status.  Workspace: mla_workspace_size(MLA_OP_INDEX_TOPK, B, 0,
 * max_seqlen, topk) bytes (fp32 scores, histograms, tile table, per-sequence
 * tile claim counters).
 */
mla_status dsa_index_topk(const mla_bf16* index_q, const mla_bf16* index_k, const float* w,
                          const int64_t* cu_seqlens, int B, int NH, int64_t total_keys,
                          int max_seqlen, int topk, int32_t* topk_idx, float* topk_scores,
                          void* ws, size_t ws_bytes, mla_stream stream);

/*
 * DSA prefill indexer: index score and top-k for every token of a prompt
 * (DSA post, eqs. (5) and (6) applied per token; its complexity section:
 * every token scores its whole visible history).  Token i of the Tq new
 * tokens sits at position Tk-Tq+i and sees positions 0..Tk-Tq+i.
 *
 *   index_q     [Tq,NH,128] index queries (NH must be 32)
 *   index_k     [Tk,128]    index keys of the sequence (cached ones first)
 *   w           [Tq,NH]     fp32 head weights (eq. (5) constant folded in)
 *   topk_idx    [Tq,topk]   int32 out: per token, the min(topk, visible)
 *               positions of largest score ranked by (score descending,
 *               position ascending), ascending, -1 padded
 *   topk_scores [Tq,topk]   fp32 out or NULL (-inf on padding and on rows
 *               that keep every visible position)
 *
 * Requires 1 <= Tq <= Tk < 2^24, 1 <= topk <= 2048, NH == 32.  Workspace:
 * mla_workspace_size(MLA_OP_PREFILL_INDEX_TOPK, Tq, 0, Tk, topk) bytes (the
 * fp32 score rows, Tq x Tk rounded up).
 */
mla_status dsa_prefill_index_topk(const mla_bf16* index_q, const mla_bf16* index_k,
                                  const float* w, int Tq, int Tk, int NH, int topk,
                                  int32_t* topk_idx, float* topk_scores, void* ws,
                                  size_t ws_bytes, mla_stream stream);

/*
 * DSA sparse prefill over the absorbed latent cache: every prompt token
 * attends over its own selection (DSA post, eqs. (9), (10) on S_t, with the
 * keys and values of eq. (8) absorbed as in mla_decode_latent).  Token i of
 * the Tq new tokens sits at position Tk-Tq+i.
 *
 *   q        [Tq,H,192]  expanded-form queries
 *   ckv      [Tk,576]    latent cache of the sequence (c_s ++ r_s per position)
 *   topk_idx [Tq,topk]   int32 selections (dsa_prefill_index_topk's output):
 *            token i uses its first min(topk, Tk-Tq+i+1) entries; -1 entries
 *            are skipped; an entry outside [0, Tk-Tq+i] is skipped and
 *            recorded as MLA_ERR_BAD_INDEX in the device status
 *   w_kc, w_vc [H,128,512]; gate [Tq,H*128] or NULL; out [Tq,H*128]
 *
 * Requires H a multiple of 16 in [16, 96], 1 <= Tq <= Tk < 2^31,
 * 1 <= topk <= 2048.  Workspace: mla_workspace_size(
 * MLA_OP_SPARSE_PREFILL_LATENT, Tq, H, Tk, topk) bytes.
 */
mla_status mla_sparse_prefill_latent(const mla_bf16* q, const mla_bf16* ckv,
                                     const int32_t* topk_idx, int Tq, int Tk, int topk, int H,
                                     const mla_bf16* w_kc, const mla_bf16* w_vc,
                                     const mla_bf16* gate, mla_bf16* out, float scale, void* ws,
                                     size_t ws_bytes, mla_stream stream);

/*
 * FP8 index keys (DSA post, cache section: the default FP8 index key is 128
 * bytes of data plus a 4-byte scale per position).  The two parts are kept
 * as separate arrays so every 128-byte row stays 16-byte aligned.
 *
 * dsa_quantize_index_keys writes, for each of the N rows of index_k
 * [N,128] bf16, the e4m3 codes k8 [N,128] and the fp32 scale kscale [N]:
 *   scale = amax / 448, code = e4m3(x * (448 / amax)) rounded to nearest
 *   even with saturation (computed in fp32); an all-zero row gets scale 0.
 * dsa_index_topk_fp8 is dsa_index_topk over such keys: the index queries are
 * quantised the same way per (sequence, head) inside and their scales folded
 * into the head weights, the 32-head dot products run as e4m3 x e4m3
 * tensor-core products with fp32 accumulation, and each position's score is
 * multiplied by its key scale.  Same outputs, tie rule and status behaviour
 * as dsa_index_topk.  Workspace: mla_workspace_size(MLA_OP_INDEX_TOPK_FP8,
 * B, 0, max_seqlen, topk) bytes.
 */
mla_status dsa_quantize_index_keys(const mla_bf16* index_k, uint8_t* k8, float* kscale, int64_t N,
                                   mla_stream stream);
mla_status dsa_index_topk_fp8(const mla_bf16* index_q, const uint8_t* k8, const float* kscale,
                              const float* w, const int64_t* cu_seqlens, int B, int NH,
                              int64_t total_keys, int max_seqlen, int topk, int32_t* topk_idx,
                              float* topk_scores, void* ws, size_t ws_bytes, mla_stream stream);

/*
 * Gated MLA over the selected positions only (DSA post eqs. (9), (10)); all
 * H heads of a sequence share its selection.
 *
 *   q, k, v, cu_seqlens, gate, out as in mla_decode
 *   topk_idx [B,topk] int32 positions within each sequence; -1 entries are
 *            skipped; an entry >= T_b or < -1 is skipped and recorded as
 *            MLA_ERR_BAD_INDEX in the device status.  The order of the
 *            entries does not matter.  A sequence with no valid entry gets a
 *            zero output.
 */
mla_status dsa_sparse_decode(const mla_bf16* q, const mla_bf16* k, const mla_bf16* v,
                             const int64_t* cu_seqlens, const int32_t* topk_idx, int topk,
                             int B, int H, const mla_bf16* gate, mla_bf16* out, float scale,
                             void* ws, size_t ws_bytes, mla_stream stream);

/*
 * Bytes of workspace an operation needs (a multiple of 256; 0 if none).
 * `op` is one of MLA_OP_*; arguments an operation does not use are ignored
 * (prefill and cache_append: none needed; decode: B, H, max_seqlen;
 * index_topk: B, max_seqlen; sparse_decode: B, H, topk; latent_decode: B, H;
 * prefill_index_topk: B = Tq, max_seqlen = Tk; sparse_prefill_latent: B = Tq, H;
 * index_topk_fp8: B, max_seqlen).  Returns 0 for invalid arguments.
 */
size_t mla_workspace_size(int op, int B, int H, int max_seqlen, int topk);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device: MLA_OK, or the first MLA_ERR_TIMEOUT /
 * MLA_ERR_BAD_INDEX / MLA_ERR_INVALID_ARG a kernel recorded since the last
 * check.  MLA_ERR_CUDA if the synchronisation itself failed.
 */
mla_status mla_check_device_status(mla_stream stream);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* mla_last_error(void);

/*
 * Test hooks for the device-side failure paths (never needed in normal use).
 *   MLA_DEBUG_WAIT_LIMIT_NS: limit of every pipeline wait in ns (default 2e9;
 *                            value <= 0 restores the default).
 *   MLA_DEBUG_STALL_STAGE:   when >= 0, the decode producer withholds the copy
 *                            of that pipeline stage of each CTA, so the wait
 *                            for it runs out and the kernel returns
 *                            MLA_ERR_TIMEOUT through the device status
 *                            (default -1 = off).
 *   MLA_DEBUG_SPARSE_CHUNK:  index entries per sparse-decode work item (a
 *                            power of two in [64, 2048]; 0 = default 256).
 *                            Changes the sparse-decode workspace size, so
 *                            query mla_workspace_size after setting it.
 *   MLA_DEBUG_PREFILL_CTAS:  CTAs that share each tensor-core MMA of the
 *                            prefill: 1 = one CTA per 128-row query tile,
 *                            2 = a pair of CTAs (two SMs) per M = 256 MMA;
 *                            0 = default (1: the pair's cross-SM handoffs
 *                            lengthen each key tile's dependency chain).
 * Returns MLA_OK or MLA_ERR_INVALID_ARG for an unknown knob or bad value.
 */
enum { MLA_DEBUG_WAIT_LIMIT_NS = 1, MLA_DEBUG_STALL_STAGE = 2, MLA_DEBUG_SPARSE_CHUNK = 3,
       MLA_DEBUG_PREFILL_CTAS = 4 };
mla_status mla_debug_set(int knob, long long value);

/*
 * Kernel timing (instrumentation for roofline figures).  While enabled, every
 * call records a CUDA event pair on its stream around its dominant kernel
 * (decode: the split-KV partial kernel; sparse decode: the same kernel in
 * gather mode; index_topk: the scoring kernel; prefill: the attention
 * kernel; cache_append: the copy kernel, also when a chunked prefill or a
 * cached decode step appends; latent_decode: the latent attention kernel;
 * prefill_index_topk: the prefill scoring kernel; sparse_prefill_latent: the
 * latent attention kernel, counted under MLA_OP_LATENT_DECODE; index_topk_fp8:
 * the FP8 scoring kernel).  mla_timing_read synchronises those events, returns the summed
 * kernel time in milliseconds and the number of launches of operation `op`
 * (MLA_OP_*) since the last read, and resets the count.  Events are created
 * on first use and reused; no device memory is allocated.
 */
mla_status mla_timing_enable(int on);
mla_status mla_timing_read(int op, double* total_ms, long long* launches);

/*
 * Measurement aid; the pages have no counterpart.  Gathers, with plain
 * 16-byte loads and no arithmetic, exactly the rows dsa_sparse_decode reads
 * for the same arguments: for every sequence b, head h and entry e with
 * 0 <= topk_idx[b,e] < T_b, the 384-byte key row and 256-byte value row of
 * that position in the packed cache (k, v, cu_seqlens as in
 * dsa_sparse_decode).  Entries outside [0, T_b) are skipped.  The words read
 * are XOR-reduced into one 32-bit value per CTA in `sink` (device memory of
 * at least mla_gather_probe_blocks() words, caller-owned), so the rate it
 * reaches (timed under MLA_OP_GATHER_PROBE) is what a gather of these rows
 * can achieve on this GPU, the ceiling against which the sparse decode's
 * rate is read.  Asynchronous on `stream`; MLA_ERR_INVALID_ARG for null or
 * misaligned pointers or bad sizes.
 */
int mla_gather_probe_blocks(void);
mla_status mla_gather_probe(const mla_bf16* k, const mla_bf16* v, const int64_t* cu_seqlens,
                            const int32_t* topk_idx, int topk, int B, int H, uint32_t* sink,
                            mla_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */
