/*
 * Plain CPU oracle for the MoE layer's local data path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA path.
 *
 * Everything here is the slow, literal definition:
 *   - floating point accumulates in fp64 (inputs may be fp32, bf16 or fp64);
 *   - loops follow the order in which the method is stated, with no blocking,
 *     fusion or reordering;
 *   - bf16 rounding points (where the bf16 pipeline stores an intermediate
 *     tensor) are applied only when the caller asks for them.
 *
 * Sources (page title, section):
 *   [EP]    "Expert Parallelism (EP)", llm-infra-atlas, section 1 (MoE layer
 *           forward path: gating logits x.W_g^T, top-k + score function,
 *           tokens_per_expert, permute, grouped fc1 -> act -> fc2,
 *           unpermute with top-k weighted reduce), section 2 (layout
 *           contract: expert-contiguous segments aligned to the GEMM M tile),
 *           section 3 (DeepSeek-V3-style group-limited routing: a token may
 *           only reach topk_group expert groups), section 5 (permute /
 *           unpermute symmetry).
 *   [ETP]   "Expert Tensor Parallel design" (HyperParallel issue 104),
 *           section 4.3 (GroupedExperts w1/w3 [E,H,D], w2 [E,D,H]; shards on
 *           dim 1 and dim 2).
 *   [NCCL32] "NCCL course 32: TP, PP, EP/MoE and multi-dim process groups",
 *           section "Tensor Parallel matrix split" (F.linear computes X.W^T,
 *           row-parallel partial outputs sum to the full output).
 *   SwiGLU expert FFN_e(v) = w2_e . (SiLU(w1_e . v) (*) (w3_e . v)) is the
 *   expert function named for this layer; SiLU(z) = z / (1 + exp(-z)).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element type codes for inputs */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };
/* score functions */
enum { ORC_SOFTMAX = 0, ORC_SIGMOID = 1 };
/* layouts */
enum { ORC_CONTIGUOUS = 0, ORC_MASKED = 1 };
/* rounding points (bit flags): where the bf16 pipeline stores a bf16 tensor */
enum { ORC_ROUND_H = 1, ORC_ROUND_Y = 2 };
/* return codes */
enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_CAPACITY = 3, ORC_BAD_ROUTING = 6 };

/* ------------------------------------------------------------------ */
/* element access and rounding                                          */
/* ------------------------------------------------------------------ */

/* bf16 is the upper 16 bits of an IEEE binary32 value. */
static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *p, int dtype, size_t i)
{
    switch (dtype) {
    case ORC_F32: return (double)((const float *)p)[i];
    case ORC_BF16: return bf16_bits_to_double(((const uint16_t *)p)[i]);
    default: return ((const double *)p)[i];
    }
}

/*
 * Round a double to the nearest bf16 value, ties to even.  bf16 keeps 8
 * significant bits (1 implicit + 7 stored) and the binary32 exponent range.
 * Below the smallest normal (2^-126) the spacing is fixed at 2^-133.
 */
double oracle_round_bf16(double v)
{
    if (!isfinite(v) || v == 0.0) return v;
    const double min_normal = ldexp(1.0, -126);
    const double max_finite = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    double out;
    if (fabs(v) < min_normal) {
        out = ldexp(nearbyint(ldexp(v, 133)), -133);
    } else {
        int e;
        double m = frexp(v, &e); /* v = m * 2^e, 0.5 <= |m| < 1 */
        out = ldexp(nearbyint(ldexp(m, 8)), e - 8);
    }
    if (fabs(out) > max_finite) return copysign(INFINITY, v);
    return out;
}

void oracle_round_bf16_array(long n, const double *in, double *out)
{
    for (long i = 0; i < n; ++i) out[i] = oracle_round_bf16(in[i]);
}

double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------------------------ */
/* a tiny thread pool: split [0, n) into contiguous chunks              */
/* ------------------------------------------------------------------ */

typedef void (*range_fn)(void *ctx, long lo, long hi);
typedef struct { range_fn fn; void *ctx; long lo, hi; } range_job;

static void *range_trampoline(void *arg)
{
    range_job *j = (range_job *)arg;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

static void parallel_for(long n, int nthreads, range_fn fn, void *ctx)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((long)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    if (nthreads == 1) { fn(ctx, 0, n); return; }
    pthread_t th[256];
    range_job jobs[256];
    long chunk = (n + nthreads - 1) / nthreads;
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        long lo = (long)i * chunk, hi = lo + chunk < n ? lo + chunk : n;
        if (lo >= hi) break;
        jobs[i].fn = fn; jobs[i].ctx = ctx; jobs[i].lo = lo; jobs[i].hi = hi;
        if (pthread_create(&th[i], NULL, range_trampoline, &jobs[i]) != 0) {
            fn(ctx, lo, hi); /* run inline if a thread cannot start */
            jobs[i].fn = NULL;
        }
        started = i + 1;
    }
    for (int i = 0; i < started; ++i)
        if (jobs[i].fn) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------ */
/* router: gating logits  ([EP] section 1: logits = x . W_g^T, [T,E])   */
/* ------------------------------------------------------------------ */

typedef struct {
    int T, D, E, xdt, wdt;
    const void *x, *wg;
    const double *bias;
    double *logits;
} logits_ctx;

static void logits_range(void *c, long lo, long hi)
{
    logits_ctx *p = (logits_ctx *)c;
    for (long t = lo; t < hi; ++t)
        for (int e = 0; e < p->E; ++e) {
            double acc = 0.0;
            for (int d = 0; d < p->D; ++d)
                acc += load_elem(p->x, p->xdt, (size_t)t * p->D + d) *
                       load_elem(p->wg, p->wdt, (size_t)e * p->D + d);
            if (p->bias) acc += p->bias[e];
            p->logits[(size_t)t * p->E + e] = acc;
        }
}

/* logits[t,e] = sum_d x[t,d] * wg[e,d] (+ bias[e]), accumulated in fp64. */
void oracle_router_logits(int T, int D, int E, const void *x, int xdt,
                          const void *wg, int wdt, const double *bias,
                          double *logits, int nthreads)
{
    logits_ctx c = {T, D, E, xdt, wdt, x, wg, bias, logits};
    parallel_for(T, nthreads, logits_range, &c);
}

/* ------------------------------------------------------------------ */
/* top-k selection                                                       */
/* ------------------------------------------------------------------ */

/*
 * Selection order on the fp32 key l: a comes before b when l_a > l_b, or
 * when they are equal and a < b (ties go to the lower expert index).  NaN
 * sorts after every number, -inf included; two NaNs tie by index.  -0 and +0
 * compare equal, so they tie by index as well.
 */
static int key_before(float la, int a, float lb, int b)
{
    int na = isnan(la), nb = isnan(lb);
    if (na || nb) {
        if (na && nb) return a < b;
        return nb; /* the non-NaN one comes first */
    }
    if (la > lb) return 1;
    if (la < lb) return 0;
    return a < b;
}

/*
 * topk_idx[t, j] = the j-th expert in selection order, j < k.  Plain
 * selection: k passes over all E experts, each taking the best remaining.
 * Returns ORC_BAD_ROUTING if any logit is NaN (the selection is still made).
 */
int oracle_topk(int T, int E, int k, const float *logits, int32_t *topk_idx)
{
    if (k < 1 || k > E) return ORC_BAD_ARG;
    int status = ORC_OK;
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    if (!taken) return ORC_BAD_ARG;
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int e = 0; e < E; ++e)
            if (isnan(l[e])) status = ORC_BAD_ROUTING;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || key_before(l[e], e, l[best], best)) best = e;
            }
            taken[best] = 1;
            topk_idx[(size_t)t * k + j] = best;
        }
    }
    free(taken);
    return status;
}

/*
 * Group-limited top-k ([EP] section 3: DeepSeek-V3-style group-limited
 * routing splits the experts into groups and lets each token reach only
 * topk_group of them, which bounds the all-to-all fan-out).
 *
 * The pages do not say how a group is scored.  Reading taken here: the E
 * experts form n_group equal groups of consecutive indices; a group's score
 * is the sum of its m = k / topk_group best keys, taken in selection order
 * and added in fp32 (the precision in which the kernel takes the same
 * decision); groups are ranked by that score, ties to the lower group index
 * and NaN last, as for keys; the top-k is then the plain selection over the
 * experts of the topk_group best groups.  n_group <= 1 is plain top-k.
 * Returns ORC_BAD_ARG for an unusable grouping, ORC_BAD_ROUTING on a NaN key.
 */
static int score_before(float sa, int a, float sb, int b)
{
    return key_before(sa, a, sb, b);
}

int oracle_topk_grouped(int T, int E, int k, int n_group, int topk_group, const float *logits,
                        int32_t *topk_idx)
{
    if (n_group <= 1) return oracle_topk(T, E, k, logits, topk_idx);
    if (E % n_group != 0 || topk_group < 1 || topk_group > n_group || k < topk_group ||
        k > topk_group * (E / n_group) || k > E)
        return ORC_BAD_ARG;
    const int gs = E / n_group, m = k / topk_group;
    int status = ORC_OK;
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    unsigned char *gsel = (unsigned char *)malloc((size_t)n_group);
    float *gscore = (float *)malloc(sizeof(float) * (size_t)n_group);
    if (!taken || !gsel || !gscore) {
        free(taken);
        free(gsel);
        free(gscore);
        return ORC_BAD_ARG;
    }
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        for (int e = 0; e < E; ++e)
            if (isnan(l[e])) status = ORC_BAD_ROUTING;
        /* group scores */
        memset(taken, 0, (size_t)E);
        for (int g = 0; g < n_group; ++g) {
            float sum = 0.f;
            for (int i = 0; i < m; ++i) {
                int best = -1;
                for (int e = g * gs; e < (g + 1) * gs; ++e) {
                    if (taken[e]) continue;
                    if (best < 0 || key_before(l[e], e, l[best], best)) best = e;
                }
                taken[best] = 1;
                sum += l[best];
            }
            gscore[g] = sum;
        }
        /* the topk_group best groups */
        memset(gsel, 0, (size_t)n_group);
        for (int r = 0; r < topk_group; ++r) {
            int best = -1;
            for (int g = 0; g < n_group; ++g) {
                if (gsel[g]) continue;
                if (best < 0 || score_before(gscore[g], g, gscore[best], best)) best = g;
            }
            gsel[best] = 1;
        }
        /* plain selection restricted to the chosen groups */
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e] || !gsel[e / gs]) continue;
                if (best < 0 || key_before(l[e], e, l[best], best)) best = e;
            }
            taken[best] = 1;
            topk_idx[(size_t)t * k + j] = best;
        }
    }
    free(taken);
    free(gsel);
    free(gscore);
    return status;
}


/*
 * Routing weights for the selected experts ([EP] section 1: "top-k +
 * score_func -> probs").  Scores from the fp32 key l:
 *   softmax: p_e = exp(l_e - max_e' l_e') / sum_e' exp(l_e' - max)
 *            (over all E experts)
 *   sigmoid: p_e = 1 / (1 + exp(-l_e))
 * Weight of slot j: w_j = p[idx_j], or p[idx_j] / sum_i p[idx_i] when
 * renormalising over the selected k.
 */
void oracle_topk_weights(int T, int E, int k, const float *logits,
                         const int32_t *topk_idx, int score, int renorm,
                         double *topk_w)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    if (!p) return;
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        if (score == ORC_SOFTMAX) {
            double m = -INFINITY;
            for (int e = 0; e < E; ++e)
                if ((double)l[e] > m) m = (double)l[e];
            double z = 0.0;
            for (int e = 0; e < E; ++e) z += exp((double)l[e] - m);
            for (int e = 0; e < E; ++e) p[e] = exp((double)l[e] - m) / z;
        } else {
            for (int e = 0; e < E; ++e) p[e] = 1.0 / (1.0 + exp(-(double)l[e]));
        }
        double s = 0.0;
        for (int j = 0; j < k; ++j) s += p[topk_idx[(size_t)t * k + j]];
        for (int j = 0; j < k; ++j) {
            double w = p[topk_idx[(size_t)t * k + j]];
            topk_w[(size_t)t * k + j] = renorm ? w / s : w;
        }
    }
    free(p);
}

/* ------------------------------------------------------------------ */
/* layout: tokens_per_expert, segment offsets, permutation               */
/* ------------------------------------------------------------------ */

/* rows needed by the layout (same formula the library documents). */
long oracle_rows_alloc(int T, int k, int E_local, int layout, int align_m,
                       int capacity)
{
    if (layout == ORC_MASKED) return (long)E_local * capacity;
    long kl = k < E_local ? k : E_local;
    return (long)T * kl + (long)E_local * (align_m - 1);
}

/*
 * Slot (t, j) of a caller-supplied routing table takes part in the layout
 * when its expert id lies in [0, E) and no earlier slot of the same token
 * names the same expert.  A token reaches each expert at most once ([EP]
 * section 1: top-k picks k distinct experts); an id outside [0, E) or a
 * repeated id is a contract violation, and that slot is left out.
 */
static int slot_valid(const int32_t *row, int j, int E)
{
    int e = row[j];
    if (e < 0 || e >= E) return 0;
    for (int q = 0; q < j; ++q)
        if (row[q] == e) return 0;
    return 1;
}

/*
 * tokens_per_expert over all E experts ([EP] section 1, "preprocess"),
 * counting the valid slots only.
 * Segment offsets over the local range [e_first, e_first + E_local):
 *   contiguous: each segment padded up to a multiple of align_m
 *               ([EP] section 2: segments aligned to the GEMM M tile);
 *   masked:     segment i starts at i * capacity ([EP] sections 2 and 6,
 *               "masked" per-expert buffers of fixed capacity).
 * Inside a segment, rows hold the routed tokens in ascending token order.
 * row_of[t, j] is that row (or -1 when expert idx[t,j] is not local, the
 * slot is not valid, or the token was dropped); token_of_row[r] is the token
 * in row r, or -1 for padding rows.
 *
 * Contract violations still produce the whole layout:
 *   - a masked expert with more than `capacity` tokens keeps its first
 *     `capacity` tokens in token order and drops the rest (row_of = -1);
 *     tokens_per_expert still counts every routed token; the return value
 *     is ORC_CAPACITY;
 *   - an invalid slot (see slot_valid) is neither counted nor placed; the
 *     return value is ORC_BAD_ROUTING unless a capacity overflow also
 *     happened (ORC_CAPACITY is reported first).
 */
int oracle_layout(int T, int k, int E, int e_first, int E_local, int layout,
                  int align_m, int capacity, const int32_t *topk_idx,
                  int32_t *cnt, int32_t *seg_off, int32_t *row_of,
                  int32_t *token_of_row, long rows_alloc)
{
    if (E_local < 0 || e_first < 0 || e_first + E_local > E || align_m < 1 ||
        (layout == ORC_MASKED && capacity < 0))
        return ORC_BAD_ARG;
    int bad = 0, over = 0;
    for (int e = 0; e < E; ++e) cnt[e] = 0;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            const int32_t *row = topk_idx + (size_t)t * k;
            if (slot_valid(row, j, E)) cnt[row[j]] += 1;
            else bad = 1;
        }
    seg_off[0] = 0;
    for (int i = 0; i < E_local; ++i) {
        int c = cnt[e_first + i];
        if (layout == ORC_MASKED) {
            if (c > capacity) over = 1;
            seg_off[i + 1] = (i + 1) * capacity;
        } else {
            int padded = (c + align_m - 1) / align_m * align_m;
            seg_off[i + 1] = seg_off[i] + padded;
        }
    }
    if ((long)seg_off[E_local] > rows_alloc) return ORC_BAD_ARG;
    for (long r = 0; r < rows_alloc; ++r) token_of_row[r] = -1;
    for (long i = 0; i < (long)T * k; ++i) row_of[i] = -1;
    for (int i = 0; i < E_local; ++i) {
        int e = e_first + i, n = 0;
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j) {
                const int32_t *row = topk_idx + (size_t)t * k;
                if (row[j] != e || !slot_valid(row, j, E)) continue;
                if (layout == ORC_MASKED && n >= capacity) continue;  /* dropped */
                int r = seg_off[i] + n;
                row_of[(size_t)t * k + j] = r;
                token_of_row[r] = t;
                n += 1;
            }
    }
    if (over) return ORC_CAPACITY;
    if (bad) return ORC_BAD_ROUTING;
    return ORC_OK;
}

/* dispatch permute: x_perm[r] = x[token_of_row[r]] for every filled row. */
void oracle_permute_rows(long rows, int D, int elem_bytes, const void *x,
                         const int32_t *token_of_row, void *x_perm)
{
    size_t rb = (size_t)D * elem_bytes;
    for (long r = 0; r < rows; ++r) {
        int t = token_of_row[r];
        if (t >= 0)
            memcpy((char *)x_perm + (size_t)r * rb, (const char *)x + (size_t)t * rb, rb);
    }
}

/* ------------------------------------------------------------------ */
/* expert FFN                                                            */
/* ------------------------------------------------------------------ */

/*
 * One expert on one input vector v[D] (weights in the F.linear [out, in]
 * convention, [NCCL32] "Tensor Parallel matrix split"; shapes from [ETP]
 * section 4.3, here for one expert and one H shard of width Hl):
 *   a[h] = SiLU(sum_d w1[h,d] v[d]) * (sum_d w3[h,d] v[d])     h < Hl
 *   y[d] = sum_h w2[d,h] a[h]                                   d < D
 * `rounding` selects where values are rounded to bf16: ORC_ROUND_H rounds a
 * (stored as the bf16 h tensor), ORC_ROUND_Y rounds y.
 */
static void expert_ffn(int D, int Hl, const void *w1, const void *w3,
                       const void *w2, int wdt, const double *v,
                       int rounding, double *a, double *y)
{
    for (int h = 0; h < Hl; ++h) {
        double g = 0.0, u = 0.0;
        for (int d = 0; d < D; ++d) {
            g += load_elem(w1, wdt, (size_t)h * D + d) * v[d];
            u += load_elem(w3, wdt, (size_t)h * D + d) * v[d];
        }
        double act = oracle_silu(g) * u;
        a[h] = (rounding & ORC_ROUND_H) ? oracle_round_bf16(act) : act;
    }
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int h = 0; h < Hl; ++h)
            acc += load_elem(w2, wdt, (size_t)d * Hl + h) * a[h];
        y[d] = (rounding & ORC_ROUND_Y) ? oracle_round_bf16(acc) : acc;
    }
}

void oracle_expert_ffn(int D, int Hl, const void *w1, const void *w3,
                       const void *w2, int wdt, const double *v,
                       int rounding, double *y)
{
    double *a = (double *)malloc(sizeof(double) * (size_t)(Hl > 0 ? Hl : 1));
    if (!a) return;
    expert_ffn(D, Hl, w1, w3, w2, wdt, v, rounding, a, y);
    free(a);
}

/*
 * Per-token brute force, no permutation at all ([EP] section 1, the whole
 * layer for one token):  out[t] = sum_j w[t,j] * FFN_{idx[t,j]}(x[t]),
 * summed in slot order j = 0..k-1, skipping experts outside the local
 * range [e_first, e_first + E_local) (their contribution belongs to another
 * shard).  Weights of local expert i are w1s[i], w3s[i], w2s[i]; a NULL
 * entry is allowed for experts no listed token uses.
 */
typedef struct {
    int D, Hl, k, e_first, E_local, xdt, wdt, rounding;
    const void *x;
    const void *const *w1s, *const *w3s, *const *w2s;
    const int32_t *tokens, *topk_idx;
    const double *topk_w;
    double *out;
    int *missing;
} tokens_ctx;

static void tokens_range(void *c, long lo, long hi)
{
    tokens_ctx *p = (tokens_ctx *)c;
    double *v = (double *)malloc(sizeof(double) * (size_t)p->D);
    double *y = (double *)malloc(sizeof(double) * (size_t)p->D);
    double *a = (double *)malloc(sizeof(double) * (size_t)(p->Hl > 0 ? p->Hl : 1));
    if (!v || !y || !a) { free(v); free(y); free(a); *p->missing = 1; return; }
    for (long i = lo; i < hi; ++i) {
        int t = p->tokens[i];
        double *o = p->out + (size_t)i * p->D;
        for (int d = 0; d < p->D; ++d) {
            o[d] = 0.0;
            v[d] = load_elem(p->x, p->xdt, (size_t)t * p->D + d);
        }
        for (int j = 0; j < p->k; ++j) {
            int e = p->topk_idx[(size_t)t * p->k + j] - p->e_first;
            if (e < 0 || e >= p->E_local) continue;
            if (!p->w1s[e] || !p->w3s[e] || !p->w2s[e]) { *p->missing = 1; continue; }
            expert_ffn(p->D, p->Hl, p->w1s[e], p->w3s[e], p->w2s[e], p->wdt, v,
                       p->rounding, a, y);
            double w = p->topk_w[(size_t)t * p->k + j];
            for (int d = 0; d < p->D; ++d) o[d] += w * y[d];
        }
    }
    free(v); free(y); free(a);
}

int oracle_moe_tokens(int ntok, const int32_t *tokens, int D, int Hl, int k,
                      int e_first, int E_local, const void *x, int xdt,
                      const void *const *w1s, const void *const *w3s,
                      const void *const *w2s, int wdt, const int32_t *topk_idx,
                      const double *topk_w, int rounding, double *out,
                      int nthreads)
{
    int missing = 0;
    tokens_ctx c = {D, Hl, k, e_first, E_local, xdt, wdt, rounding, x,
                    w1s, w3s, w2s, tokens, topk_idx, topk_w, out, &missing};
    parallel_for(ntok, nthreads, tokens_range, &c);
    return missing ? ORC_BAD_ARG : ORC_OK;
}

/* ------------------------------------------------------------------ */
/* grouped form over the permuted layout                                  */
/* ------------------------------------------------------------------ */

/*
 * First grouped GEMM with the SwiGLU gate, row by row over each local
 * expert's filled rows [seg_off[i], seg_off[i] + cnt_local[i]):
 *   h[r, c] = SiLU(sum_d x_perm[r,d] w1_i[c,d]) * (sum_d x_perm[r,d] w3_i[c,d])
 * Rows outside the filled ranges are left untouched.
 */
typedef struct {
    int D, Hl, E_local, xdt, wdt, rounding, which;
    const int32_t *seg_off, *cnt_local;
    const void *in;
    const void *const *wa, *const *wb;
    double *out;
} grouped_ctx;

static void grouped_range(void *c, long lo, long hi)
{
    grouped_ctx *p = (grouped_ctx *)c;
    for (long i = lo; i < hi; ++i) {
        if (!p->wa[i] || (p->which == 1 && !p->wb[i])) continue;
        for (int n = 0; n < p->cnt_local[i]; ++n) {
            long r = (long)p->seg_off[i] + n;
            if (p->which == 1) {
                for (int c2 = 0; c2 < p->Hl; ++c2) {
                    double g = 0.0, u = 0.0;
                    for (int d = 0; d < p->D; ++d) {
                        double xv = load_elem(p->in, p->xdt, (size_t)r * p->D + d);
                        g += xv * load_elem(p->wa[i], p->wdt, (size_t)c2 * p->D + d);
                        u += xv * load_elem(p->wb[i], p->wdt, (size_t)c2 * p->D + d);
                    }
                    double act = oracle_silu(g) * u;
                    p->out[(size_t)r * p->Hl + c2] =
                        (p->rounding & ORC_ROUND_H) ? oracle_round_bf16(act) : act;
                }
            } else {
                for (int d = 0; d < p->D; ++d) {
                    double acc = 0.0;
                    for (int c2 = 0; c2 < p->Hl; ++c2)
                        acc += load_elem(p->in, p->xdt, (size_t)r * p->Hl + c2) *
                               load_elem(p->wa[i], p->wdt, (size_t)d * p->Hl + c2);
                    p->out[(size_t)r * p->D + d] =
                        (p->rounding & ORC_ROUND_Y) ? oracle_round_bf16(acc) : acc;
                }
            }
        }
    }
}

void oracle_grouped_gemm1_swiglu(int D, int Hl, int E_local,
                                 const int32_t *seg_off, const int32_t *cnt_local,
                                 const void *x_perm, int xdt,
                                 const void *const *w1s, const void *const *w3s,
                                 int wdt, int rounding, double *h, int nthreads)
{
    grouped_ctx c = {D, Hl, E_local, xdt, wdt, rounding, 1, seg_off, cnt_local,
                     x_perm, w1s, w3s, h};
    parallel_for(E_local, nthreads, grouped_range, &c);
}

/* Second grouped GEMM: y[r, d] = sum_c h[r, c] w2_i[d, c] over filled rows. */
void oracle_grouped_gemm2(int D, int Hl, int E_local, const int32_t *seg_off,
                          const int32_t *cnt_local, const void *h, int hdt,
                          const void *const *w2s, int wdt, int rounding,
                          double *y, int nthreads)
{
    grouped_ctx c = {D, Hl, E_local, hdt, wdt, rounding, 2, seg_off, cnt_local,
                     h, w2s, NULL, y};
    parallel_for(E_local, nthreads, grouped_range, &c);
}

/*
 * Unpermute with the top-k weighted reduce ([EP] section 1, combine
 * post-process):  out[t] = sum_j w[t,j] * y_perm[row_of[t,j]], j in slot
 * order, skipping row_of = -1 (expert not local).
 */
void oracle_unpermute_combine(int T, int k, int D, const void *y_perm, int ydt,
                              const int32_t *row_of, const double *topk_w,
                              double *out)
{
    for (int t = 0; t < T; ++t) {
        double *o = out + (size_t)t * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int j = 0; j < k; ++j) {
            int r = row_of[(size_t)t * k + j];
            if (r < 0) continue;
            double w = topk_w[(size_t)t * k + j];
            for (int d = 0; d < D; ++d)
                o[d] += w * load_elem(y_perm, ydt, (size_t)r * D + d);
        }
    }
}

/* ------------------------------------------------------------------ */
/* backward of the layer (fp64 throughout)                               */
/* ------------------------------------------------------------------ */

/*
 * The layer written once more entirely in fp64, as the function that the
 * backward below differentiates ([EP] section 1 forward path; [EP] section 5:
 * the backward mirrors it -- combine-bwd is a dispatch, dispatch-bwd a
 * combine -- and the expert weights get m-grouped dgrad / k-grouped wgrad):
 *   l = x.wg^T + b                         (fp64, no fp32 key here)
 *   S = top-k of l (same order and grouping rules as the fp32 selection)
 *   w_j = score weights of l over S (softmax over all E or sigmoid, renorm)
 *   out[t] = sum_j w_j FFN_{S_j}(x[t])
 * The selection is piecewise constant: it carries no gradient.
 */
static int before64(double a, int ia, double b, int ib)
{
    int na = isnan(a), nb = isnan(b);
    if (na || nb) {
        if (na && nb) return ia < ib;
        return nb;
    }
    if (a > b) return 1;
    if (a < b) return 0;
    return ia < ib;
}

static void select64(int E, int k, int n_group, int topk_group, const double *l, int32_t *idx)
{
    unsigned char taken[1024], gsel[1024];
    double gscore[1024];
    const int grouped = n_group > 1;
    const int gs = grouped ? E / n_group : E;
    if (grouped) {
        const int m = k / topk_group;
        memset(taken, 0, (size_t)E);
        for (int g = 0; g < n_group; ++g) {
            double sum = 0.0;
            for (int i = 0; i < m; ++i) {
                int best = -1;
                for (int e = g * gs; e < (g + 1) * gs; ++e)
                    if (!taken[e] && (best < 0 || before64(l[e], e, l[best], best))) best = e;
                taken[best] = 1;
                sum += l[best];
            }
            gscore[g] = sum;
        }
        memset(gsel, 0, (size_t)n_group);
        for (int r = 0; r < topk_group; ++r) {
            int best = -1;
            for (int g = 0; g < n_group; ++g)
                if (!gsel[g] && (best < 0 || before64(gscore[g], g, gscore[best], best))) best = g;
            gsel[best] = 1;
        }
    }
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e] || (grouped && !gsel[e / gs])) continue;
            if (best < 0 || before64(l[e], e, l[best], best)) best = e;
        }
        taken[best] = 1;
        idx[j] = best;
    }
}

/* softmax over all E (p_all) or sigmoid scores, then the k weights */
static void weights64(int E, int k, const double *l, const int32_t *idx, int score, int renorm,
                      double *p_all, double *w)
{
    if (score == ORC_SOFTMAX) {
        double m = -INFINITY, z = 0.0;
        for (int e = 0; e < E; ++e) if (l[e] > m) m = l[e];
        for (int e = 0; e < E; ++e) z += exp(l[e] - m);
        for (int e = 0; e < E; ++e) p_all[e] = exp(l[e] - m) / z;
    } else {
        for (int e = 0; e < E; ++e) p_all[e] = 1.0 / (1.0 + exp(-l[e]));
    }
    double s = 0.0;
    for (int j = 0; j < k; ++j) s += p_all[idx[j]];
    for (int j = 0; j < k; ++j) w[j] = renorm ? p_all[idx[j]] / s : p_all[idx[j]];
}

static int backward_args_ok(int D, int H, int E, int k, int n_group, int topk_group)
{
    if (D < 1 || H < 1 || E < 1 || E > 1024 || k < 1 || k > E) return 0;
    if (n_group > 1 && (E % n_group || topk_group < 1 || topk_group > n_group ||
                        k < topk_group || k > topk_group * (E / n_group)))
        return 0;
    return 1;
}

int oracle_moe_forward64(int T, int D, int H, int E, int k, const double *x, const double *wg,
                         const double *bias, const double *w1, const double *w3,
                         const double *w2, int score, int renorm, int n_group, int topk_group,
                         double *out, int32_t *topk_idx)
{
    if (!backward_args_ok(D, H, E, k, n_group, topk_group)) return ORC_BAD_ARG;
    double *l = malloc(sizeof(double) * E), *p = malloc(sizeof(double) * E);
    double *w = malloc(sizeof(double) * k), *a = malloc(sizeof(double) * H);
    double *y = malloc(sizeof(double) * D);
    if (!l || !p || !w || !a || !y) { free(l); free(p); free(w); free(a); free(y); return ORC_BAD_ARG; }
    for (int t = 0; t < T; ++t) {
        const double *xt = x + (size_t)t * D;
        for (int e = 0; e < E; ++e) {
            double s = bias ? bias[e] : 0.0;
            for (int d = 0; d < D; ++d) s += xt[d] * wg[(size_t)e * D + d];
            l[e] = s;
        }
        int32_t *idx = topk_idx + (size_t)t * k;
        select64(E, k, n_group, topk_group, l, idx);
        weights64(E, k, l, idx, score, renorm, p, w);
        double *o = out + (size_t)t * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int j = 0; j < k; ++j) {
            const int e = idx[j];
            expert_ffn(D, H, w1 + (size_t)e * H * D, w3 + (size_t)e * H * D,
                       w2 + (size_t)e * D * H, ORC_F64, xt, 0, a, y);
            for (int d = 0; d < D; ++d) o[d] += w[j] * y[d];
        }
    }
    free(l); free(p); free(w); free(a); free(y);
    return ORC_OK;
}

/*
 * Gradients of L = sum_t <dout[t], out[t]> for the layer above.  Per token,
 * with g = w1_e x, u = w3_e x, a = SiLU(g), h = a * u, y_j = w2_e h:
 *   dw_j  = <dout, y_j>                 (the combine's backward: a dot per slot)
 *   dy    = w_j dout                    (combine-bwd = dispatch, [EP] section 5)
 *   dh    = w2_e^T dy;  du = dh * a;  dg = dh * u * SiLU'(g),
 *           SiLU'(g) = s (1 + g (1 - s)),  s = 1 / (1 + exp(-g))
 *   dx   += w1_e^T dg + w3_e^T du       (dispatch-bwd = combine over the slots)
 *   dw2_e += dy h^T,  dw1_e += dg x^T,  dw3_e += du x^T
 * Router, with dl = dL/dl over all E:
 *   softmax:           dl_e = p_e (G_e - sum_j dw_j p_{S_j}),  G_e = dw_j if e = S_j
 *   softmax, renorm:   dl_{S_j} = w_j (dw_j - sum_i dw_i w_i), 0 elsewhere
 *   sigmoid:           dl_{S_j} = dw_j s_j (1 - s_j)
 *   sigmoid, renorm:   dl_{S_j} = (dw_j - sum_i dw_i w_i) / sum_i s_i * s_j (1 - s_j)
 *   dbias += dl,  dwg += dl x^T,  dx += wg^T dl.
 * Outputs are overwritten (dx [T,D], dwg [E,D], dbias [E], dw1/dw3 [E,H,D],
 * dw2 [E,D,H]); topk_idx receives the selection used.
 */
int oracle_moe_backward(int T, int D, int H, int E, int k, const double *x, const double *wg,
                        const double *bias, const double *w1, const double *w3,
                        const double *w2, int score, int renorm, int n_group, int topk_group,
                        const double *dout, double *dx, double *dwg, double *dbias, double *dw1,
                        double *dw3, double *dw2, int32_t *topk_idx)
{
    if (!backward_args_ok(D, H, E, k, n_group, topk_group)) return ORC_BAD_ARG;
    memset(dx, 0, sizeof(double) * (size_t)T * D);
    memset(dwg, 0, sizeof(double) * (size_t)E * D);
    memset(dbias, 0, sizeof(double) * (size_t)E);
    memset(dw1, 0, sizeof(double) * (size_t)E * H * D);
    memset(dw3, 0, sizeof(double) * (size_t)E * H * D);
    memset(dw2, 0, sizeof(double) * (size_t)E * D * H);
    double *l = malloc(sizeof(double) * E), *p = malloc(sizeof(double) * E);
    double *dl = malloc(sizeof(double) * E), *w = malloc(sizeof(double) * k);
    double *dw = malloc(sizeof(double) * k), *g = malloc(sizeof(double) * H);
    double *u = malloc(sizeof(double) * H), *hh = malloc(sizeof(double) * H);
    double *dh = malloc(sizeof(double) * H), *y = malloc(sizeof(double) * D);
    double *dy = malloc(sizeof(double) * D);
    if (!l || !p || !dl || !w || !dw || !g || !u || !hh || !dh || !y || !dy) {
        free(l); free(p); free(dl); free(w); free(dw); free(g); free(u); free(hh); free(dh);
        free(y); free(dy);
        return ORC_BAD_ARG;
    }
    for (int t = 0; t < T; ++t) {
        const double *xt = x + (size_t)t * D;
        const double *go = dout + (size_t)t * D;
        double *gx = dx + (size_t)t * D;
        for (int e = 0; e < E; ++e) {
            double s = bias ? bias[e] : 0.0;
            for (int d = 0; d < D; ++d) s += xt[d] * wg[(size_t)e * D + d];
            l[e] = s;
        }
        int32_t *idx = topk_idx + (size_t)t * k;
        select64(E, k, n_group, topk_group, l, idx);
        weights64(E, k, l, idx, score, renorm, p, w);
        /* experts */
        for (int j = 0; j < k; ++j) {
            const int e = idx[j];
            const double *W1 = w1 + (size_t)e * H * D, *W3 = w3 + (size_t)e * H * D;
            const double *W2 = w2 + (size_t)e * D * H;
            for (int c = 0; c < H; ++c) {
                double gs = 0.0, us = 0.0;
                for (int d = 0; d < D; ++d) {
                    gs += W1[(size_t)c * D + d] * xt[d];
                    us += W3[(size_t)c * D + d] * xt[d];
                }
                g[c] = gs;
                u[c] = us;
                hh[c] = oracle_silu(gs) * us;
            }
            double dwj = 0.0;
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int c = 0; c < H; ++c) acc += W2[(size_t)d * H + c] * hh[c];
                y[d] = acc;
                dwj += go[d] * acc;
                dy[d] = w[j] * go[d];
            }
            dw[j] = dwj;
            for (int c = 0; c < H; ++c) {
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += W2[(size_t)d * H + c] * dy[d];
                dh[c] = acc;
            }
            double *G1 = dw1 + (size_t)e * H * D, *G3 = dw3 + (size_t)e * H * D;
            double *G2 = dw2 + (size_t)e * D * H;
            for (int d = 0; d < D; ++d)
                for (int c = 0; c < H; ++c) G2[(size_t)d * H + c] += dy[d] * hh[c];
            for (int c = 0; c < H; ++c) {
                const double s = 1.0 / (1.0 + exp(-g[c]));
                const double dgc = dh[c] * u[c] * s * (1.0 + g[c] * (1.0 - s));
                const double duc = dh[c] * oracle_silu(g[c]);
                for (int d = 0; d < D; ++d) {
                    gx[d] += W1[(size_t)c * D + d] * dgc + W3[(size_t)c * D + d] * duc;
                    G1[(size_t)c * D + d] += dgc * xt[d];
                    G3[(size_t)c * D + d] += duc * xt[d];
                }
            }
        }
        /* router */
        for (int e = 0; e < E; ++e) dl[e] = 0.0;
        double dot = 0.0;
        for (int j = 0; j < k; ++j) dot += dw[j] * w[j];
        if (score == ORC_SOFTMAX && !renorm) {
            double sp = 0.0;
            for (int j = 0; j < k; ++j) sp += dw[j] * p[idx[j]];
            for (int e = 0; e < E; ++e) dl[e] = -p[e] * sp;
            for (int j = 0; j < k; ++j) dl[idx[j]] += p[idx[j]] * dw[j];
        } else if (score == ORC_SOFTMAX) {
            for (int j = 0; j < k; ++j) dl[idx[j]] = w[j] * (dw[j] - dot);
        } else if (!renorm) {
            for (int j = 0; j < k; ++j) dl[idx[j]] = dw[j] * p[idx[j]] * (1.0 - p[idx[j]]);
        } else {
            double ssum = 0.0;
            for (int j = 0; j < k; ++j) ssum += p[idx[j]];
            for (int j = 0; j < k; ++j)
                dl[idx[j]] = (dw[j] - dot) / ssum * p[idx[j]] * (1.0 - p[idx[j]]);
        }
        for (int e = 0; e < E; ++e) {
            if (dl[e] == 0.0) continue;
            dbias[e] += dl[e];
            for (int d = 0; d < D; ++d) {
                dwg[(size_t)e * D + d] += dl[e] * xt[d];
                gx[d] += wg[(size_t)e * D + d] * dl[e];
            }
        }
    }
    free(l); free(p); free(dl); free(w); free(dw); free(g); free(u); free(hh); free(dh);
    free(y); free(dy);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* FP8 e4m3 dispatch (the FP8 next step of the pages: e4m3 dispatched      */
/* activations with scales feeding an FP8 grouped GEMM)                     */
/* ------------------------------------------------------------------ */

/*
 * The e4m3 format ("fn" variant): 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities; exponent field 15 with mantissa 7 is NaN,
 * so the largest finite value is 1.75 * 2^8 = 448.  Exponent field 0 holds
 * the subnormals m/8 * 2^-6.
 */
double oracle_e4m3_value(int code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/*
 * Nearest e4m3 code of a binary32 value, ties to the even mantissa, values
 * beyond the largest finite magnitude saturated to +-448, NaN to 0x7f.
 * Every step is exact in double: the input has 24 significant bits.
 */
int oracle_e4m3_encode(float vf)
{
    double v = (double)vf;
    if (v != v) return 0x7f;
    int sign = v < 0.0 || (v == 0.0 && signbit(v)) ? 0x80 : 0;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7e;
    if (a < ldexp(1.0, -6)) {                 /* subnormal range, step 2^-9 */
        double m = rint(a / ldexp(1.0, -9)); /* rint: nearest, ties to even */
        return sign | (int)m;                 /* m = 8 is the code of 2^-6 */
    }
    int e2;
    frexp(a, &e2);                            /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                           /* a in [2^e, 2^(e+1)) */
    double mf = rint((a / ldexp(1.0, e) - 1.0) * 8.0);
    if (mf == 8.0) { mf = 0.0; e += 1; }
    int field = e + 7;
    if (field > 15 || (field == 15 && mf == 7.0)) return sign | 0x7e;
    return sign | (field << 3) | (int)mf;
}

/*
 * Row-wise quantisation (the reading taken for the scale granularity): for
 * each row r of src [rows, cols] (binary32 values, e.g. bf16 activations or
 * weights widened exactly), amax = max_c |src[r,c]|, scale[r] = amax / 448
 * computed in binary32 (1 when amax is 0), and dst[r,c] = e4m3 code of the
 * binary32 quotient src[r,c] / scale[r].  The dequantised value is
 * scale[r] * e4m3_value(dst[r,c]).
 */
void oracle_quantize_rows_e4m3(long rows, int cols, const float *src, uint8_t *dst, float *scale)
{
    for (long r = 0; r < rows; ++r) {
        const float *x = src + (size_t)r * cols;
        float amax = 0.0f;
        for (int c = 0; c < cols; ++c) {
            float a = fabsf(x[c]);
            if (a > amax) amax = a;
        }
        volatile float s = amax > 0.0f ? amax / 448.0f : 1.0f;  /* one binary32 division */
        scale[r] = s;
        for (int c = 0; c < cols; ++c) {
            volatile float q = x[c] / s;                         /* binary32 quotient */
            dst[(size_t)r * cols + c] = (uint8_t)oracle_e4m3_encode(q);
        }
    }
}
