/*
 * Plain CPU oracle for the batched composite multi-LoRA delta.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The product path
 * (the CUDA library and its Python binding) never calls it, and this file
 * shares no code, header, table or constant with that path.
 *
 * What it computes, in fp64 from the exact bf16 / fp32 input values:
 *
 *   y_t  <-  bf16_rne( y_t + sum_{(i, alpha) in P(t)} alpha * (x_t . A_i[:, :k_i]) . B_i[:k_i, :] )
 *
 * Sources:
 *  - composite delta  dW = sum_i alpha_i * B_i A_i^T, one serving path for
 *    static (per request) and dynamic (per token) weights: DyMerge-LoRA
 *    summary page, "Core idea" (paper Sec. 3.1, M1);
 *  - deferred (post-merge) fusion of all token-LoRA pairs of a batch, which
 *    must equal pre-merging: same page, "One-minute summary" and "Core idea"
 *    (paper Sec. 4.3), "How far to trust it" (Sec. 5.4);
 *  - one LoRA pair W' = W + A B, applied to one projection: ELORA page,
 *    Sec. 1.2 (Eq. 1) and Sec. 1.3 (Eq. 2);
 *  - retained effective rank k_m: the live directions are a sorted prefix of
 *    the factors: LoRAForge summary page, "Key contributions" and
 *    "Approach" (1);
 *  - mapping tuples reordered by LoRA id so that one CTA sees one adapter's
 *    tokens together: DyMerge-LoRA page, "Core idea" (paper Sec. 4.3,
 *    Algorithm 2, Figure 8).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - row form y += (x A) B with A: d_in x r, B: r x d_out;
 *  - the mapping is a stable order by adapter id: ties keep CSR order
 *    (token ascending, then list position);
 *  - an id outside [0, capacity), an unregistered slot (rank < 0) or a rank
 *    above r_max is an error: the pair contributes nothing and a status bit
 *    is set; malformed CSR offsets make the whole batch contribute nothing;
 *  - the result is rounded once, to nearest-even bf16.
 *
 * Status bits: 1 = id out of range, 2 = malformed offsets,
 *              4 = unregistered slot, 8 = rank above r_max.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_BAD_ID 1
#define ORC_BAD_OFFSETS 2
#define ORC_UNREGISTERED 4
#define ORC_BAD_RANK 8

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value to the nearest bf16 (8 significant bits, exponent range
 * of fp32, subnormal quantum 2^-133), ties to even.  Returns the bit pattern. */
uint16_t orc_round_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    int e;
    frexp(a, &e);          /* a = m * 2^e, 0.5 <= m < 1 */
    int q = e - 8;         /* spacing of bf16 numbers around a */
    if (q < -133)
        q = -133;          /* subnormal range: fixed spacing */
    double r = nearbyint(ldexp(a, -q)); /* default mode: nearest, ties to even */
    double res = ldexp(r, q);
    if (res >= 0x1p128)
        return (uint16_t)(sign | 0x7F80);
    float f = (float)res;  /* exact: res has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* Checks that offsets is a CSR row pointer for P pairs. */
static int offsets_ok(int T, int P, const int32_t *offsets)
{
    if (offsets[0] != 0 || offsets[T] != P)
        return 0;
    for (int t = 0; t < T; ++t)
        if (offsets[t + 1] < offsets[t])
            return 0;
    return 1;
}

/*
 * The delta itself.  y_out (bf16 bits, T x d_out) and, when non-NULL,
 * acc_out (fp64, T x d_out, the value before rounding).  ranks[a] is the
 * retained rank of slot a, or -1 for an unregistered slot.  Returns the
 * status bits.  threads <= 0: all available.
 */
int orc_delta_apply(int T, int P, int d_in, int d_out, int r_max, int capacity,
                    const int32_t *offsets, const int32_t *ids, const float *alpha,
                    const uint16_t *x, const uint16_t *A, const uint16_t *B,
                    const int32_t *ranks, const uint16_t *y_in,
                    uint16_t *y_out, double *acc_out, int threads)
{
    int status = 0;
    int live = offsets_ok(T, P, offsets);
    if (!live)
        status |= ORC_BAD_OFFSETS;
#ifdef _OPENMP
    if (threads <= 0)
        threads = omp_get_max_threads();
#pragma omp parallel num_threads(threads) reduction(| : status)
#endif
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)d_out);
        double *s = (double *)malloc(sizeof(double) * (size_t)d_out);
        double *z = (double *)malloc(sizeof(double) * (size_t)(r_max > 0 ? r_max : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int t = 0; t < T; ++t) {
            for (int c = 0; c < d_out; ++c)
                acc[c] = bf16_to_double(y_in[(size_t)t * d_out + c]);
            int p0 = live ? offsets[t] : 0, p1 = live ? offsets[t + 1] : 0;
            for (int p = p0; p < p1; ++p) {
                int a = ids[p];
                if (a < 0 || a >= capacity) {
                    status |= ORC_BAD_ID;
                    continue;
                }
                int k = ranks[a];
                if (k < 0) {
                    status |= ORC_UNREGISTERED;
                    continue;
                }
                if (k > r_max) {
                    status |= ORC_BAD_RANK;
                    continue;
                }
                double al = (double)alpha[p];
                const uint16_t *Aa = A + (size_t)a * d_in * r_max;
                const uint16_t *Ba = B + (size_t)a * r_max * d_out;
                /* z_j = sum_d x[t, d] * A_a[d, j], j < k */
                for (int j = 0; j < k; ++j) {
                    double zj = 0.0;
                    for (int d = 0; d < d_in; ++d)
                        zj += bf16_to_double(x[(size_t)t * d_in + d]) *
                              bf16_to_double(Aa[(size_t)d * r_max + j]);
                    z[j] = zj;
                }
                /* s_c = sum_{j<k} z_j * B_a[j, c]  (j ascending for every c) */
                for (int c = 0; c < d_out; ++c)
                    s[c] = 0.0;
                for (int j = 0; j < k; ++j)
                    for (int c = 0; c < d_out; ++c)
                        s[c] += z[j] * bf16_to_double(Ba[(size_t)j * d_out + c]);
                for (int c = 0; c < d_out; ++c)
                    acc[c] += al * s[c];
            }
            for (int c = 0; c < d_out; ++c) {
                y_out[(size_t)t * d_out + c] = orc_round_bf16(acc[c]);
                if (acc_out)
                    acc_out[(size_t)t * d_out + c] = acc[c];
            }
        }
        free(acc);
        free(s);
        free(z);
    }
    return status;
}

typedef struct {
    int32_t adapter;
    int32_t src;
} orc_key;

static int cmp_key(const void *pa, const void *pb)
{
    const orc_key *a = (const orc_key *)pa, *b = (const orc_key *)pb;
    if (a->adapter != b->adapter)
        return a->adapter < b->adapter ? -1 : 1;
    return a->src < b->src ? -1 : (a->src > b->src);
}

/*
 * The mapping: pairs in CSR order p = 0..P-1 become tuples
 * (tok, adapter, alpha, src = p), ordered by (adapter, p).  Pairs with an id
 * outside [0, capacity) are left out (pos = -1).  Outputs:
 *   s_tok, s_adapter, s_alpha, s_src   [P_valid]  the ordered tuples
 *   pos                                [P]        p -> ordered position or -1
 *   seg_adapter [U], seg_start [U+1]   distinct adapters, ascending
 *   counts[0] = U, counts[1] = P_valid
 * Returns the status bits.  Malformed offsets give an empty mapping.
 */
int orc_build_mapping(int T, int P, int capacity, const int32_t *offsets,
                      const int32_t *ids, const float *alpha,
                      int32_t *s_tok, int32_t *s_adapter, float *s_alpha, int32_t *s_src,
                      int32_t *pos, int32_t *seg_adapter, int32_t *seg_start, int32_t *counts)
{
    int status = 0;
    for (int p = 0; p < P; ++p)
        pos[p] = -1;
    counts[0] = counts[1] = 0;
    seg_start[0] = 0;
    if (!offsets_ok(T, P, offsets))
        return ORC_BAD_OFFSETS;

    int32_t *tok = (int32_t *)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    orc_key *keys = (orc_key *)malloc(sizeof(orc_key) * (size_t)(P > 0 ? P : 1));
    for (int t = 0; t < T; ++t)
        for (int p = offsets[t]; p < offsets[t + 1]; ++p)
            tok[p] = t;
    int n = 0;
    for (int p = 0; p < P; ++p) {
        if (ids[p] < 0 || ids[p] >= capacity) {
            status |= ORC_BAD_ID;
            continue;
        }
        keys[n].adapter = ids[p];
        keys[n].src = p;
        ++n;
    }
    /* keys are unique (src differs), so any correct sort gives this order */
    qsort(keys, (size_t)n, sizeof(orc_key), cmp_key);
    int U = 0;
    for (int q = 0; q < n; ++q) {
        int p = keys[q].src;
        s_tok[q] = tok[p];
        s_adapter[q] = keys[q].adapter;
        s_alpha[q] = alpha[p];
        s_src[q] = p;
        pos[p] = q;
        if (q == 0 || keys[q].adapter != keys[q - 1].adapter) {
            seg_adapter[U] = keys[q].adapter;
            seg_start[U] = q;
            ++U;
        }
    }
    seg_start[U] = n;
    counts[0] = U;
    counts[1] = n;
    free(tok);
    free(keys);
    return status;
}

/*
 * MoE-LoRA gating that produces the pair lists (DyMerge-LoRA page, code
 * release notes / Appendix A: per-token adapter weights from padded,
 * masked candidate lists, batched gate logits, top-k, renormalised).
 *
 * orc_gate_logits: logits[t][e] = sum_d x[t][d] * Wg[req[t]][e][d], fp64.
 *   x bf16 [T][d_in]; Wg bf16 [R][E][d_in] (a router per request); req[t]
 *   the request of token t.
 */
void orc_gate_logits(int T, int E, int d_in, const uint16_t *x, const uint16_t *Wg, const int32_t *req,
                     double *logits)
{
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            const uint16_t *w = Wg + ((size_t)req[t] * E + e) * d_in;
            double s = 0.0;
            for (int d = 0; d < d_in; ++d)
                s += bf16_to_double(x[(size_t)t * d_in + d]) * bf16_to_double(w[d]);
            logits[(size_t)t * E + e] = s;
        }
}

/*
 * orc_gate_topk: per token t, the candidates e with cand[t][e] >= 0 are
 * ranked by logit, largest first, equal logits by the lower e; the first
 * top_k are kept and weighted by the softmax over all candidates
 * renormalised over the kept ones, alpha_i = exp(l_i) / sum_kept exp(l_j)
 * (the full softmax denominator cancels), computed in fp64 from the given
 * fp32 logits and rounded to fp32.  Every token emits exactly top_k pairs
 * (offsets[t] = t * top_k): a token with fewer valid candidates repeats its
 * best one with alpha = 0; a token with none emits ids -1 (alpha 0).
 * Returns the number of tokens without any valid candidate.
 */
int orc_gate_topk(int T, int E, int top_k, const float *logits, const int32_t *cand, int32_t *offsets, int32_t *ids,
                  float *alpha)
{
    int empty = 0;
    int *taken = (int *)malloc(sizeof(int) * (size_t)(E > 0 ? E : 1));
    int *sel = (int *)malloc(sizeof(int) * (size_t)(top_k > 0 ? top_k : 1));
    for (int t = 0; t <= T; ++t)
        offsets[t] = t * top_k;
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        const int32_t *c = cand + (size_t)t * E;
        for (int e = 0; e < E; ++e)
            taken[e] = 0;
        int n = 0;
        for (int i = 0; i < top_k; ++i) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (c[e] >= 0 && !taken[e] && (best < 0 || l[e] > l[best]))
                    best = e; /* strict >: the lower e wins a tie */
            if (best < 0)
                break;
            taken[best] = 1;
            sel[n++] = best;
        }
        int32_t *id = ids + (size_t)t * top_k;
        float *al = alpha + (size_t)t * top_k;
        if (n == 0) {
            ++empty;
            for (int i = 0; i < top_k; ++i) {
                id[i] = -1;
                al[i] = 0.0f;
            }
            continue;
        }
        double mx = (double)l[sel[0]], den = 0.0;
        for (int i = 0; i < n; ++i)
            den += exp((double)l[sel[i]] - mx);
        for (int i = 0; i < top_k; ++i) {
            if (i < n) {
                id[i] = c[sel[i]];
                al[i] = (float)(exp((double)l[sel[i]] - mx) / den);
            } else {
                id[i] = c[sel[0]];
                al[i] = 0.0f;
            }
        }
    }
    free(taken);
    free(sel);
    return empty;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
