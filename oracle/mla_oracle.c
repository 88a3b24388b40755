/*
 * Plain fp64 CPU oracle for Gated MLA / Gated DSA attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file.  The library's GPU path never
 * calls it, includes it or shares any code with it.
 *
 * Every function is written from the definitions on the pages, with no
 * blocking, fusion or reordering beyond what those definitions state:
 *
 *  - Scores: s_j = (q . k_j) * scale, scale = q_head_dim^-1/2 = 192^-1/2
 *    (Kimi K3 modeling code, MLA __init__ "self.scaling"; Kimi K2 "Latent
 *    attention > KV cache" page, attn_weights = matmul(q, k^T) * softmax_scale;
 *    K3.1 Gated DSA post, eq. (9)).
 *  - Causal mask: a query at absolute position P+i (P = Tk - Tq cached
 *    positions before the new tokens) sees keys j <= P+i; decode sees every
 *    cached position, the current token included (K3 MLA "is_causal = True";
 *    K3.1 post eq. (5) "s <= t", eq. (6) and its note that t counts the
 *    current token).
 *  - Softmax over the visible positions, two passes (max, then normalise),
 *    then z = sum_j p_j v_j (K3.1 post, eq. (9)).
 *  - Output gate: out[b,t,h*128+d] = z[b,h,t,d] * sigmoid(g[b,t,h*128+d]),
 *    i.e. the attention output reshaped to [B,T,H*128] (channel h*128+d,
 *    Concat_h) times the sigmoid of the gate logits, before o_proj (K3 MLA
 *    forward, "attn_output * g_proj(x).sigmoid()"; K3.1 post, eq. (10)).
 *  - Index score: I_s = sum_h w_h * ReLU(q^I_h . k^I_s) (K3.1 post, eq. (5));
 *    the constant 1/(sqrt(32)*sqrt(128)) is folded into w by the caller, as the
 *    post says vLLM does.
 *  - Top-k: S = the min(topk, T) visible positions of largest score
 *    (K3.1 post, eq. (6)); ranking by (score descending, position ascending);
 *    returned in ascending position order, padded with -1.  When T <= topk
 *    every position is kept (the post's short-context remark).
 *  - Sparse gated MLA: eq. (9) restricted to S, then the gate of eq. (10).
 *
 * Readings where the pages are silent: an empty visible set (all indices -1)
 * gives z = 0; the gate is omitted when no gate tensor is given.
 *
 * All tensors are fp64 arrays, contiguous, in the library's layouts:
 *   prefill  q [B,H,Tq,Dqk], k [B,H,Tk,Dqk], v [B,H,Tk,Dv],
 *            gate/out [B,Tq,H*Dv]
 *   decode   q [B,H,Dqk]; packed k: sequence b holds [H,T_b,Dqk] starting at
 *            element cu[b]*H*Dqk (v likewise with Dv); gate/out [B,H*Dv]
 *   indexer  index_q [B,NH,Di], packed index_k [cu[B],Di], w [B,NH],
 *            scores packed [cu[B]]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double dot(const double* a, const double* b, int n) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/*
 * Softmax attention of one query over n keys.  Key j is row pos[j] of kbase
 * (row j when pos is NULL).  Writes z[Dv]; if p is not NULL, also the
 * probabilities p[n].  Returns 0, or -1 when scratch cannot be allocated.
 */
static int attend(const double* q, const double* kbase, const double* vbase,
                  const int64_t* pos, int64_t n, int Dqk, int Dv, double scale,
                  double* z, double* p) {
    for (int d = 0; d < Dv; ++d) z[d] = 0.0;
    if (n <= 0) return 0;
    double* s = (double*)malloc((size_t)n * sizeof(double));
    if (!s) return -1;
    for (int64_t j = 0; j < n; ++j) {
        int64_t r = pos ? pos[j] : j;
        s[j] = dot(q, kbase + r * Dqk, Dqk) * scale;
    }
    double m = s[0];
    for (int64_t j = 1; j < n; ++j) if (s[j] > m) m = s[j];
    double denom = 0.0;
    for (int64_t j = 0; j < n; ++j) denom += exp(s[j] - m);
    for (int64_t j = 0; j < n; ++j) {
        int64_t r = pos ? pos[j] : j;
        double pj = exp(s[j] - m) / denom;
        if (p) p[j] = pj;
        const double* vr = vbase + r * Dv;
        for (int d = 0; d < Dv; ++d) z[d] += pj * vr[d];
    }
    free(s);
    return 0;
}

static void gate_store(const double* z, const double* g, double* out, int Dv) {
    for (int d = 0; d < Dv; ++d) out[d] = g ? z[d] * sigmoid(g[d]) : z[d];
}

int orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Causal prefill with bottom-right alignment (query i sees keys j <= Tk-Tq+i). */
int orc_mla_prefill(const double* q, const double* k, const double* v, const double* gate,
                    double* out, int B, int H, int Tq, int Tk, int Dqk, int Dv, double scale) {
    if (B < 1 || H < 1 || Tq < 1 || Tk < Tq || Dqk < 1 || Dv < 1) return 1;
    int err = 0;
    const int64_t P = (int64_t)Tk - Tq;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : err)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            double* z = (double*)malloc((size_t)Dv * sizeof(double));
            if (!z) { err |= 1; continue; }
            const double* kb = k + ((int64_t)b * H + h) * Tk * Dqk;
            const double* vb = v + ((int64_t)b * H + h) * Tk * Dv;
            for (int i = 0; i < Tq; ++i) {
                const double* qi = q + (((int64_t)b * H + h) * Tq + i) * Dqk;
                int64_t n = P + i + 1;                       /* keys 0..P+i are visible */
                err |= attend(qi, kb, vb, NULL, n, Dqk, Dv, scale, z, NULL) ? 1 : 0;
                int64_t o = (((int64_t)b * Tq + i) * H + h) * Dv;   /* [B,Tq,H*Dv] */
                gate_store(z, gate ? gate + o : NULL, out + o, Dv);
            }
            free(z);
        }
    return err ? 2 : 0;
}

/* Decode: one query per sequence, every cached position visible. */
int orc_mla_decode(const double* q, const double* k, const double* v, const int64_t* cu,
                   int B, int H, int Dqk, int Dv, const double* gate, double* out,
                   double scale) {
    if (B < 1 || H < 1 || Dqk < 1 || Dv < 1 || Dv > 1024) return 1;
    for (int b = 0; b < B; ++b) if (cu[b + 1] - cu[b] < 1) return 1;
    int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : err)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            double z[1024];
            const int64_t T = cu[b + 1] - cu[b];
            const double* kb = k + (cu[b] * H + (int64_t)h * T) * Dqk;
            const double* vb = v + (cu[b] * H + (int64_t)h * T) * Dv;
            const double* qb = q + ((int64_t)b * H + h) * Dqk;
            err |= attend(qb, kb, vb, NULL, T, Dqk, Dv, scale, z, NULL) ? 1 : 0;
            int64_t o = ((int64_t)b * H + h) * Dv;
            gate_store(z, gate ? gate + o : NULL, out + o, Dv);
        }
    return err ? 2 : 0;
}

/* Probabilities of one attention row over n contiguous keys (for invariant tests). */
int orc_attention_probs(const double* q, const double* k, const double* v, int64_t n,
                        int Dqk, int Dv, double scale, double* z, double* p) {
    return attend(q, k, v, NULL, n, Dqk, Dv, scale, z, p) ? 2 : 0;
}

/* Index scores I_s = sum_h w_h * max(0, q_h . k_s) for every cached position s. */
int orc_dsa_index_scores(const double* iq, const double* ik, const double* w,
                         const int64_t* cu, int B, int NH, int Di, double* scores) {
    if (B < 1 || NH < 1 || Di < 1) return 1;
    for (int b = 0; b < B; ++b) {
        const int64_t T = cu[b + 1] - cu[b];
#pragma omp parallel for schedule(static)
        for (int64_t s = 0; s < T; ++s) {
            const double* ks = ik + (cu[b] + s) * Di;
            double acc = 0.0;
            for (int h = 0; h < NH; ++h) {
                double zh = dot(iq + ((int64_t)b * NH + h) * Di, ks, Di);
                acc += w[(int64_t)b * NH + h] * (zh > 0.0 ? zh : 0.0);
            }
            scores[cu[b] + s] = acc;
        }
    }
    return 0;
}

typedef struct { double score; int64_t pos; } ranked;

static int by_rank(const void* a, const void* b) {
    const ranked* x = (const ranked*)a;
    const ranked* y = (const ranked*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

static int by_value(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Top-k by full sort; idx [B,topk] ascending, -1 padded. */
int orc_dsa_topk(const double* scores, const int64_t* cu, int B, int topk, int32_t* idx) {
    if (B < 1 || topk < 1) return 1;
    for (int b = 0; b < B; ++b) {
        const int64_t T = cu[b + 1] - cu[b];
        int32_t* row = idx + (int64_t)b * topk;
        for (int i = 0; i < topk; ++i) row[i] = -1;
        if (T <= 0) continue;
        int64_t kk = T < topk ? T : topk;
        ranked* r = (ranked*)malloc((size_t)T * sizeof(ranked));
        if (!r) return 2;
        for (int64_t s = 0; s < T; ++s) { r[s].score = scores[cu[b] + s]; r[s].pos = s; }
        qsort(r, (size_t)T, sizeof(ranked), by_rank);
        for (int64_t i = 0; i < kk; ++i) row[i] = (int32_t)r[i].pos;
        qsort(row, (size_t)kk, sizeof(int32_t), by_value);
        free(r);
    }
    return 0;
}

/* Gated MLA over the selected positions only (entries < 0 are skipped). */
int orc_dsa_sparse_decode(const double* q, const double* k, const double* v,
                          const int64_t* cu, const int32_t* idx, int topk, int B, int H,
                          int Dqk, int Dv, const double* gate, double* out, double scale) {
    if (B < 1 || H < 1 || topk < 1 || Dqk < 1 || Dv < 1 || Dv > 1024) return 1;
    for (int b = 0; b < B; ++b) {
        const int64_t T = cu[b + 1] - cu[b];
        for (int i = 0; i < topk; ++i) {
            int32_t s = idx[(int64_t)b * topk + i];
            if (s >= T || s < -1) return 3;
        }
    }
    int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : err)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            double z[1024];
            const int64_t T = cu[b + 1] - cu[b];
            int64_t* pos = (int64_t*)malloc((size_t)topk * sizeof(int64_t));
            if (!pos) { err |= 1; continue; }
            int64_t n = 0;
            for (int i = 0; i < topk; ++i) {
                int32_t s = idx[(int64_t)b * topk + i];
                if (s >= 0) pos[n++] = s;
            }
            const double* kb = k + (cu[b] * H + (int64_t)h * T) * Dqk;
            const double* vb = v + (cu[b] * H + (int64_t)h * T) * Dv;
            const double* qb = q + ((int64_t)b * H + h) * Dqk;
            err |= attend(qb, kb, vb, pos, n, Dqk, Dv, scale, z, NULL) ? 1 : 0;
            int64_t o = ((int64_t)b * H + h) * Dv;
            gate_store(z, gate ? gate + o : NULL, out + o, Dv);
            free(pos);
        }
    return err ? 2 : 0;
}
