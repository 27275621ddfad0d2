/*
 * sv_oracle.c -- plain, slow, sequential float64 oracle for batched
 * speculative-decoding verification and confidence scheduling.
 *
 * TEST INFRASTRUCTURE ONLY. The CUDA library never calls, links or loads this
 * file, and this file shares no code, header or constant with it. Only the
 * tests, the smoke check and the CPU-baseline leg of the benchmark use it.
 *
 * Every step is written the way the method is stated, one element at a time,
 * in float64: no blocking, no fusion, no reordering. Inputs arrive as the exact
 * fp32 or bf16 values the GPU sees; both widen to float64 without rounding.
 *
 * Sources (web pages on DSpark, cited by title and section):
 *  [DD]  "DSpark Deep Dive: How DeepSeek Squeezed an 85% Speedup Out of
 *        Inference Without Touching a Single Model Weight" (fuyuan7.com)
 *  [GD]  "DSpark Guide: Confidence Speculative Decoding in LLMs" (aifetchly)
 *  [TP]  perchy.ai "Technology", engine 01 "Verified by the target"
 *  [SN]  "DSpark shows why fast AI inference is a scheduling problem, not a
 *        model trick" (seventnews.com)
 *
 * Readings taken where the pages are silent or garbled are listed next to the
 * code that takes them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Return codes (oracle-local; the CUDA library has its own). */
#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_INPUT (-5)

/* Per-request flags written by oracle_verify. */
#define ORC_FLAG_ACCEPT_TIE 1     /* |u - min(1,p/q)| < 1e-5 at a tested position */
#define ORC_FLAG_CDF_EDGE 2       /* terminal uniform within 1e-5 of a bucket edge */
#define ORC_FLAG_TINY_PROB 4      /* p(x) and q(x) both below 1e-30 at a test     */
#define ORC_FLAG_SMALL_RESIDUAL 8 /* residual mass below 1e-5 at the rejection    */
#define ORC_FLAG_INVALID 16       /* request rejected as invalid input            */

#define NEAR_TIE 1e-5

/* ------------------------------------------------------------------------ */
/* Input widening: fp32 is widened by a cast, bf16 by placing its 16 bits in  */
/* the high half of an fp32 word (bf16 is the top half of an IEEE binary32).  */
/* ------------------------------------------------------------------------ */
static double logit_at(const void *base, int dtype, size_t i) {
    if (dtype == 0) return (double)((const float *)base)[i];
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* A row is a valid logit row when it has no NaN, no +inf, and at least one
 * finite entry (-inf entries are allowed: they are masked tokens). Returns the
 * row maximum through *max_out, and the lowest index attaining it. */
static int row_scan(const void *base, int dtype, size_t off, int V, double *max_out,
                    int *argmax_out) {
    double m = -INFINITY;
    int am = 0;
    for (int v = 0; v < V; v++) {
        double z = logit_at(base, dtype, off + (size_t)v);
        if (isnan(z)) return -1;
        if (z > m) { /* strict: ties keep the lowest index */
            m = z;
            am = v;
        }
    }
    if (!isfinite(m)) return -1; /* +inf present, or every entry -inf */
    *max_out = m;
    *argmax_out = am;
    return 0;
}

/* Softmax at temperature T > 0 [DD "The Speculative Decoding Solution":
 * target and draft probabilities are softmax of the logits; the temperature
 * divides the logits]. p_v = exp((z_v - M)/T) / sum_w exp((z_w - M)/T),
 * with M the row maximum and the sum taken left to right. */
static void row_softmax(const void *base, int dtype, size_t off, int V, double T, double M,
                        double *p) {
    double S = 0.0;
    for (int v = 0; v < V; v++) {
        p[v] = exp((logit_at(base, dtype, off + (size_t)v) - M) / T);
        S += p[v];
    }
    for (int v = 0; v < V; v++) p[v] /= S;
}

/* Inverse CDF over non-negative weights w[0..V) at uniform u in [0,1):
 * Z = sum of w (left to right); the sample is the smallest v with
 * u*Z < w[0] + ... + w[v]. A bucket of zero weight can never be chosen.
 * Also reports how close u*Z came to the chosen bucket's edges, in units of
 * Z, for near-tie flagging. Returns -1 when Z is not positive. */
static int inverse_cdf(const double *w, int V, double u, double *Z_out, double *edge_gap) {
    double Z = 0.0;
    for (int v = 0; v < V; v++) Z += w[v];
    *Z_out = Z;
    if (!(Z > 0.0)) return -1;
    double target = u * Z;
    double cum = 0.0;
    for (int v = 0; v < V; v++) {
        double lo = cum;
        cum += w[v];
        if (target < cum) {
            double g_lo = (target - lo) / Z, g_hi = (cum - target) / Z;
            *edge_gap = g_lo < g_hi ? g_lo : g_hi;
            return v;
        }
    }
    /* Not reachable for u < 1: the last partial sum equals Z exactly. */
    *edge_gap = 0.0;
    return V - 1;
}

/* ======================================================================== */
/* Confidence scheduling                                                    */
/* ======================================================================== */

typedef struct {
    double s;  /* prefix survival probability S_{b,k} */
    int k;     /* position in the block (0-based) */
    int b;     /* request */
    int floor; /* 1 when this is a guaranteed floor position (ranks first) */
} orc_cand;

/* Rank order for the budget trim: floor positions first (when the budget can
 * honour one per request), then survival descending, then position ascending,
 * then request ascending. */
static int cand_order(const void *pa, const void *pb) {
    const orc_cand *a = (const orc_cand *)pa, *b = (const orc_cand *)pb;
    if (a->floor != b->floor) return a->floor ? -1 : 1;
    if (a->s != b->s) return a->s > b->s ? -1 : 1;
    if (a->k != b->k) return a->k < b->k ? -1 : 1;
    return (a->b > b->b) - (a->b < b->b);
}

/*
 * oracle_schedule: verify lengths from per-position draft confidences.
 *
 *  1. Prefix survival S_{b,k} = c_{b,0} * ... * c_{b,k}, a running product
 *     left to right in float64 [GD "2. Confidence-Scheduled Dynamic
 *     Verification": C_k = prod_{i<=k} p_i; [SN]: "prefix survival
 *     probability"; [GD] "Hands-On Implementation": cum_prob *= p_accept].
 *  2. tau-truncation: L0_b = number of positions with S_{b,k} >= tau, at
 *     least 1, at most K [GD: K* = max{k in [1,K] : C_k >= tau}; the sketch
 *     in "Hands-On Implementation" truncates at the first C_k < tau with a
 *     floor of 1; [DD "The Full Scheduling Pipeline"]: 1 <= L <= K].
 *  3. Budget trim: when sum_b L0_b exceeds token_budget, keep the
 *     token_budget best positions in the order of cand_order among the
 *     tau-survivors, so the lowest marginal-survival positions go first
 *     [DD "The Optimization Logic": a slot is better spent on another
 *     request's more confident token]. Reading: when token_budget >= B each
 *     request keeps its floor position; when token_budget < B the floor
 *     positions compete like the others and a request may get 0.
 *     out_len[b] = number of kept positions of request b (a prefix, because
 *     S is non-increasing along the block and ties go to the smaller k).
 *
 * conf: [B,K] float32 in [0,1]. out_len: [B]. out_surv: [B,K] or NULL.
 * out_l0: [B] or NULL (lengths after step 2). Returns ORC_ERR_INPUT (and all
 * out_len = 0) when any confidence is NaN or outside [0,1].
 */
int oracle_schedule(const float *conf, int B, int K, float tau, long long token_budget,
                    int32_t *out_len, double *out_surv, int32_t *out_l0) {
    if (B < 0 || K < 1 || token_budget < 0 || !(tau >= 0.0f && tau <= 1.0f)) return ORC_ERR_ARG;
    for (int b = 0; b < B; b++) out_len[b] = 0;
    if (B == 0) return ORC_OK;
    for (long long i = 0; i < (long long)B * K; i++)
        if (!(conf[i] >= 0.0f && conf[i] <= 1.0f)) return ORC_ERR_INPUT;

    double *S = (double *)malloc(sizeof(double) * (size_t)B * K);
    int *L0 = (int *)malloc(sizeof(int) * (size_t)B);
    long long total = 0;
    for (int b = 0; b < B; b++) {
        double run = 1.0;
        int n = 0;
        for (int k = 0; k < K; k++) {
            run = run * (double)conf[(size_t)b * K + k];
            S[(size_t)b * K + k] = run;
            if (run >= (double)tau) n = k + 1; /* S is non-increasing: count = last index */
        }
        if (n < 1) n = 1;
        L0[b] = n;
        total += n;
    }
    if (out_surv) memcpy(out_surv, S, sizeof(double) * (size_t)B * K);
    if (out_l0)
        for (int b = 0; b < B; b++) out_l0[b] = L0[b];

    if (total <= token_budget) {
        for (int b = 0; b < B; b++) out_len[b] = L0[b];
    } else {
        orc_cand *c = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)total);
        int floor_first = token_budget >= B;
        size_t n = 0;
        for (int b = 0; b < B; b++)
            for (int k = 0; k < L0[b]; k++) {
                c[n].s = S[(size_t)b * K + k];
                c[n].k = k;
                c[n].b = b;
                c[n].floor = floor_first && k == 0;
                n++;
            }
        qsort(c, n, sizeof(orc_cand), cand_order);
        for (long long i = 0; i < token_budget; i++) out_len[c[i].b]++;
        free(c);
    }
    free(S);
    free(L0);
    return ORC_OK;
}

/* ======================================================================== */
/* Verification                                                             */
/* ======================================================================== */

/*
 * One request of oracle_verify (see below). Writes row b of the outputs.
 */
static int verify_one(const void *tgt, const void *drf, int dtype, const int32_t *tok,
                      const int32_t *vlen, const double *u, int b, int K, int V, double T,
                      int32_t *out_tok, int32_t *out_acc, double *out_p, double *out_q,
                      int32_t *out_flags, double *out_margin, double *p, double *q, double *r) {
    const int L = vlen[b];
    double margin = INFINITY; /* smallest decision margin seen (diagnostic) */
    if (out_margin) out_margin[b] = INFINITY;
    int32_t *ot = out_tok + (size_t)b * (K + 1);
    for (int k = 0; k <= K; k++) ot[k] = -1;
    for (int k = 0; k < K; k++) {
        if (out_p) out_p[(size_t)b * K + k] = NAN;
        if (out_q) out_q[(size_t)b * K + k] = NAN;
    }
    out_flags[b] = 0;
    out_acc[b] = -1;

    /* Validation of everything this request reads. */
    if (L < 0 || L > K) goto invalid;
    for (int k = 0; k < L; k++)
        if (tok[(size_t)b * K + k] < 0 || tok[(size_t)b * K + k] >= V) goto invalid;
    const size_t trow0 = (size_t)b * (K + 1), drow0 = (size_t)b * K;
    double Mt[33], Md[33];
    int At[33], Ad[33];
    for (int k = 0; k <= L; k++)
        if (row_scan(tgt, dtype, (trow0 + k) * (size_t)V, V, &Mt[k], &At[k])) goto invalid;
    if (T > 0.0) {
        for (int k = 0; k < L; k++)
            if (row_scan(drf, dtype, (drow0 + k) * (size_t)V, V, &Md[k], &Ad[k])) goto invalid;
        for (int k = 0; k < L; k++)
            if (!(u[(size_t)b * (K + 1) + k] >= 0.0 && u[(size_t)b * (K + 1) + k] < 1.0))
                goto invalid;
        if (!(u[(size_t)b * (K + 1) + K] >= 0.0 && u[(size_t)b * (K + 1) + K] < 1.0)) goto invalid;
    }

    if (T == 0.0) {
        /* Greedy verification: at T=0 rejection sampling reduces to argmax
         * matching. Accept x_k iff it is the lowest-index argmax of target row
         * k; the terminal token is the argmax of the first mismatching row, or
         * of row L when every draft matches. */
        int j = 0;
        while (j < L && tok[(size_t)b * K + j] == At[j]) j++;
        for (int k = 0; k < j; k++) ot[k] = tok[(size_t)b * K + k];
        ot[j] = At[j];
        out_acc[b] = j;
        return 0;
    }

    /* Diagnostics: p_k(x_k), q_k(x_k) for every drafted position k < L. */
    if (out_p || out_q) {
        for (int k = 0; k < L; k++) {
            int x = tok[(size_t)b * K + k];
            row_softmax(tgt, dtype, (trow0 + k) * (size_t)V, V, T, Mt[k], p);
            row_softmax(drf, dtype, (drow0 + k) * (size_t)V, V, T, Md[k], q);
            if (out_p) out_p[(size_t)b * K + k] = p[x];
            if (out_q) out_q[(size_t)b * K + k] = q[x];
        }
    }

    /* Rejection sampling [DD "The Speculative Decoding Solution"; GD "1. The
     * Mathematics of Suffix Decay"]: at each drafted position accept x_k with
     * probability min(1, p_k(x_k)/q_k(x_k)) using the test u_k < p/q written
     * division-free as u_k * q < p (strict, as the pages' random() < ratio);
     * stop at the first rejection. */
    int j = L;
    for (int k = 0; k < L; k++) {
        const int x = tok[(size_t)b * K + k];
        row_softmax(tgt, dtype, (trow0 + k) * (size_t)V, V, T, Mt[k], p);
        row_softmax(drf, dtype, (drow0 + k) * (size_t)V, V, T, Md[k], q);
        const double uk = u[(size_t)b * (K + 1) + k];
        const double px = p[x], qx = q[x];
        /* Near-tie bookkeeping (the decision itself is the line after). */
        double ratio = qx > 0.0 ? (px / qx < 1.0 ? px / qx : 1.0) : (px > 0.0 ? 1.0 : 0.0);
        if (fabs(uk - ratio) < NEAR_TIE) out_flags[b] |= ORC_FLAG_ACCEPT_TIE;
        if (fabs(uk - ratio) < margin) margin = fabs(uk - ratio);
        if (px < 1e-30 && qx < 1e-30) out_flags[b] |= ORC_FLAG_TINY_PROB;
        if (uk * qx < px) {
            ot[k] = x;
            continue;
        }
        /* First rejection: sample from normalize(max(0, p - q)) by inverse
         * CDF on the request's last uniform u_{b,K} [DD "The Speculative
         * Decoding Solution": "sample from adjusted distribution"; the page's
         * residual line subtracts a list of scalars from a vector, read here
         * as the full distributions p and q]. */
        j = k;
        for (int v = 0; v < V; v++) r[v] = p[v] - q[v] > 0.0 ? p[v] - q[v] : 0.0;
        double Z, gap;
        const double uK = u[(size_t)b * (K + 1) + K];
        int y = inverse_cdf(r, V, uK, &Z, &gap);
        if (Z < NEAR_TIE) out_flags[b] |= ORC_FLAG_SMALL_RESIDUAL;
        if (y < 0) {
            /* Reading: no residual mass left (p == q up to rounding); fall
             * back to sampling the target distribution itself. */
            y = inverse_cdf(p, V, uK, &Z, &gap);
        }
        if (gap < NEAR_TIE) out_flags[b] |= ORC_FLAG_CDF_EDGE;
        if (out_margin) out_margin[b] = gap < margin ? gap : margin;
        ot[j] = y;
        out_acc[b] = j;
        return 0;
    }

    /* Every drafted token accepted: sample the bonus token from p_L with
     * u_{b,K} (standard method of Leviathan et al. and Chen et al., which the
     * Deep Dive cites; its pseudocode stops before this step). */
    {
        row_softmax(tgt, dtype, (trow0 + L) * (size_t)V, V, T, Mt[L], p);
        double Z, gap;
        int y = inverse_cdf(p, V, u[(size_t)b * (K + 1) + K], &Z, &gap);
        if (gap < NEAR_TIE) out_flags[b] |= ORC_FLAG_CDF_EDGE;
        if (out_margin) out_margin[b] = gap < margin ? gap : margin;
        ot[L] = y;
        out_acc[b] = L;
    }
    return 0;

invalid:
    for (int k = 0; k <= K; k++) ot[k] = -1;
    out_acc[b] = -1;
    out_flags[b] = ORC_FLAG_INVALID;
    return -1;
}

/*
 * oracle_verify_u64: batched verification with float64 uniforms.
 *
 *  target: [B, K+1, V] logits (dtype 0 = fp32, 1 = bf16 bits).
 *  draft:  [B, K, V] logits, same dtype (unused at T=0; may be NULL then).
 *  tok:    [B, K] draft tokens x_{b,k}.   vlen: [B] verify lengths L_b.
 *  u:      [B, K+1]: u_{b,k} drives the accept test at position k, u_{b,K}
 *          drives the terminal (residual or bonus) sample. Unused at T=0.
 *  T:      temperature; 0 = greedy argmax verification.
 *  out_tok [B, K+1]: accepted drafts, then the terminal token, then -1.
 *  out_acc [B]: number of accepted drafts j (or -1 for an invalid request).
 *  out_p, out_q [B, K] or NULL: p_k(x_k), q_k(x_k) for k < L_b (T > 0).
 *  out_flags [B]: ORC_FLAG_* bits.
 *  out_margin [B] or NULL (T > 0): the smallest decision margin of the request,
 *  the quantity the near-tie flags threshold: min over tested positions of
 *  |u_k - min(1, p/q)| and the terminal sample's distance to its nearest CDF edge
 *  (normalised units). A diagnostic; no decision depends on it.
 *  nthreads: OpenMP threads over requests (requests are independent, so the
 *  result does not depend on it).
 * Returns ORC_OK, ORC_ERR_ARG, or ORC_ERR_INPUT if any request was invalid.
 */
int oracle_verify_u64m(const void *target, const void *draft, int dtype, const int32_t *tok,
                       const int32_t *vlen, const double *u, int B, int K, int V, double T,
                       int32_t *out_tok, int32_t *out_acc, double *out_p, double *out_q,
                       int32_t *out_flags, double *out_margin, int nthreads) {
    if (B < 0 || K < 1 || K > 32 || V < 1 || (dtype != 0 && dtype != 1) || !(T >= 0.0) ||
        !isfinite(T))
        return ORC_ERR_ARG;
    if (B == 0) return ORC_OK;
    if (!target || !tok || !vlen || !out_tok || !out_acc || !out_flags) return ORC_ERR_ARG;
    if (T > 0.0 && (!draft || !u)) return ORC_ERR_ARG;
    int n_invalid = 0;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads) reduction(+ : n_invalid)
#endif
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *q = (double *)malloc(sizeof(double) * (size_t)V);
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int b = 0; b < B; b++)
            if (verify_one(target, draft, dtype, tok, vlen, u, b, K, V, T, out_tok, out_acc, out_p,
                           out_q, out_flags, out_margin, p, q, r))
                n_invalid++;
        free(p);
        free(q);
        free(r);
    }
    return n_invalid ? ORC_ERR_INPUT : ORC_OK;
}

/* oracle_verify_u64m without the margin output. */
int oracle_verify_u64(const void *target, const void *draft, int dtype, const int32_t *tok,
                      const int32_t *vlen, const double *u, int B, int K, int V, double T,
                      int32_t *out_tok, int32_t *out_acc, double *out_p, double *out_q,
                      int32_t *out_flags, int nthreads) {
    return oracle_verify_u64m(target, draft, dtype, tok, vlen, u, B, K, V, T, out_tok, out_acc,
                              out_p, out_q, out_flags, NULL, nthreads);
}

/* Same as oracle_verify_u64m with the float32 uniforms of the C-ABI, widened
 * exactly to float64. */
int oracle_verify_m(const void *target, const void *draft, int dtype, const int32_t *tok,
                    const int32_t *vlen, const float *u, int B, int K, int V, float T,
                    int32_t *out_tok, int32_t *out_acc, double *out_p, double *out_q,
                    int32_t *out_flags, double *out_margin, int nthreads) {
    double *u64 = NULL;
    if (u && B > 0) {
        u64 = (double *)malloc(sizeof(double) * (size_t)B * (K + 1));
        for (size_t i = 0; i < (size_t)B * (K + 1); i++) u64[i] = (double)u[i];
    }
    int rc = oracle_verify_u64m(target, draft, dtype, tok, vlen, u64, B, K, V, (double)T,
                                out_tok, out_acc, out_p, out_q, out_flags, out_margin, nthreads);
    free(u64);
    return rc;
}

/* oracle_verify_m without the margin output. */
int oracle_verify(const void *target, const void *draft, int dtype, const int32_t *tok,
                  const int32_t *vlen, const float *u, int B, int K, int V, float T,
                  int32_t *out_tok, int32_t *out_acc, double *out_p, double *out_q,
                  int32_t *out_flags, int nthreads) {
    return oracle_verify_m(target, draft, dtype, tok, vlen, u, B, K, V, T, out_tok, out_acc,
                           out_p, out_q, out_flags, NULL, nthreads);
}
