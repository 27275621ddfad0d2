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
/* Steps 1-3 on confidences already widened (or calibrated) to float64, against
 * the float64 threshold th. */
static void schedule_core(const double *c, int B, int K, double th, long long token_budget,
                          int32_t *out_len, double *out_surv, int32_t *out_l0) {
    double *S = (double *)malloc(sizeof(double) * (size_t)B * K);
    int *L0 = (int *)malloc(sizeof(int) * (size_t)B);
    long long total = 0;
    for (int b = 0; b < B; b++) {
        double run = 1.0;
        int n = 0;
        for (int k = 0; k < K; k++) {
            run = run * c[(size_t)b * K + k];
            S[(size_t)b * K + k] = run;
            if (run >= th) n = k + 1; /* S is non-increasing: count = last index */
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
        orc_cand *cd = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)total);
        int floor_first = token_budget >= B;
        size_t n = 0;
        for (int b = 0; b < B; b++)
            for (int k = 0; k < L0[b]; k++) {
                cd[n].s = S[(size_t)b * K + k];
                cd[n].k = k;
                cd[n].b = b;
                cd[n].floor = floor_first && k == 0;
                n++;
            }
        qsort(cd, n, sizeof(orc_cand), cand_order);
        for (long long i = 0; i < token_budget; i++) out_len[cd[i].b]++;
        free(cd);
    }
    free(S);
    free(L0);
}

int oracle_schedule(const float *conf, int B, int K, float tau, long long token_budget,
                    int32_t *out_len, double *out_surv, int32_t *out_l0) {
    if (B < 0 || K < 1 || token_budget < 0 || !(tau >= 0.0f && tau <= 1.0f)) return ORC_ERR_ARG;
    for (int b = 0; b < B; b++) out_len[b] = 0;
    if (B == 0) return ORC_OK;
    for (long long i = 0; i < (long long)B * K; i++)
        if (!(conf[i] >= 0.0f && conf[i] <= 1.0f)) return ORC_ERR_INPUT;
    double *c = (double *)malloc(sizeof(double) * (size_t)B * K);
    for (long long i = 0; i < (long long)B * K; i++) c[i] = (double)conf[i];
    schedule_core(c, B, K, (double)tau, token_budget, out_len, out_surv, out_l0);
    free(c);
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
         * Decoding Solution": after a rejection the token is drawn from the
         * residual of the two distributions; the page's residual line
         * subtracts a list of scalars from a vector, read here as the full
         * distributions p and q]. */
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

/* ======================================================================== */
/* Calibration prologue, load-aware threshold, and the online calibration  */
/* loop                                                                      */
/* ======================================================================== */

/*
 * Sequential temperature scaling of one confidence [DD "Sequential Temperature
 * Scaling"]: the raw score is mapped to a logit, divided by the temperature of
 * its draft position, and mapped back through the sigmoid,
 *     c' = sigmoid(logit(c) / T_k),  logit(c) = ln(c / (1 - c)).
 * The end points are fixed (c = 0 -> 0, c = 1 -> 1) for every T > 0.
 */
static double calibrate_one(double c, double T) {
    if (c <= 0.0) return 0.0;
    if (c >= 1.0) return 1.0;
    double z = (log(c) - log1p(-c)) / T;
    return 1.0 / (1.0 + exp(-z));
}

/*
 * Load-aware threshold [GD "Dynamic Verification Scheduling Algorithm", steps 1
 * and 2]: load factor LF = 0.6 * Q / Q_max + 0.4 * M_gpu / M_max, then
 * tau = tau_min + (tau_max - tau_min) * LF^2. Reading: the page states LF in
 * [0, 1]; a load beyond its maximum is clamped to 1.
 * load: {Q, Q_max, M_gpu, M_max} as float32 (widened exactly).
 * Returns -1 when a load value is NaN/inf or negative, or a maximum is not > 0.
 */
static double load_tau(const float *load, double tau_min, double tau_max) {
    double Q = load[0], Qmax = load[1], M = load[2], Mmax = load[3];
    if (!(isfinite(Q) && isfinite(Qmax) && isfinite(M) && isfinite(Mmax))) return -1.0;
    if (Q < 0.0 || M < 0.0 || !(Qmax > 0.0) || !(Mmax > 0.0)) return -1.0;
    double lf = 0.6 * (Q / Qmax) + 0.4 * (M / Mmax);
    if (lf > 1.0) lf = 1.0;
    return tau_min + (tau_max - tau_min) * (lf * lf);
}

double oracle_load_tau(const float *load, double tau_min, double tau_max) {
    return load_tau(load, tau_min, tau_max);
}

/*
 * oracle_schedule_ex: the schedule of oracle_schedule run on calibrated
 * confidences, optionally with the load-aware threshold [DD "The Full Scheduling
 * Pipeline": raw scores -> online calibration -> scheduler with the GPU's load].
 *
 *  temps [K] float32 > 0, or NULL for no calibration (c' = c).
 *  load [4] {Q, Q_max, M_gpu, M_max}, or NULL to use tau as given.
 *  out_cal [B,K] float32 or NULL: c' rounded to float32.
 *  out_tau: the threshold used (float64), or NULL.
 * Steps 1-3 of oracle_schedule then run on c' in float64: S_{b,k} =
 * c'_{b,0} * ... * c'_{b,k}, compared with the float64 threshold.
 * Returns ORC_ERR_INPUT (and out_len = 0) for a confidence outside [0,1], a
 * temperature that is not a positive finite number, or an invalid load.
 */
int oracle_schedule_ex(const float *conf, const float *temps, const float *load, float tau,
                       float tau_min, float tau_max, int B, int K, long long token_budget,
                       int32_t *out_len, double *out_surv, int32_t *out_l0, float *out_cal,
                       double *out_tau) {
    if (B < 0 || K < 1 || token_budget < 0) return ORC_ERR_ARG;
    if (!(tau >= 0.0f && tau <= 1.0f) || !(tau_min >= 0.0f && tau_min <= 1.0f) ||
        !(tau_max >= 0.0f && tau_max <= 1.0f))
        return ORC_ERR_ARG;
    for (int b = 0; b < B; b++) out_len[b] = 0;
    double th = (double)tau;
    int bad = 0;
    if (load) {
        th = load_tau(load, (double)tau_min, (double)tau_max);
        if (th < 0.0) bad = 1;
    }
    if (out_tau) *out_tau = th;
    if (temps)
        for (int k = 0; k < K; k++)
            if (!(isfinite(temps[k]) && temps[k] > 0.0f)) bad = 1;
    for (long long i = 0; i < (long long)B * K; i++)
        if (!(conf[i] >= 0.0f && conf[i] <= 1.0f)) bad = 1;
    if (bad) return ORC_ERR_INPUT;
    if (B == 0) return ORC_OK;

    double *c = (double *)malloc(sizeof(double) * (size_t)B * K);
    for (int b = 0; b < B; b++)
        for (int k = 0; k < K; k++) {
            size_t i = (size_t)b * K + k;
            c[i] = temps ? calibrate_one((double)conf[i], (double)temps[k]) : (double)conf[i];
            if (out_cal) out_cal[i] = (float)c[i];
        }
    schedule_core(c, B, K, th, token_budget, out_len, out_surv, out_l0);
    free(c);
    return ORC_OK;
}

/*
 * Calibration window statistics [DD "The Calibration Loop in Practice"]. Over a
 * window of verification rounds, per draft position i: the mean calibrated
 * confidence and the fraction of tokens at position i that were accepted; and,
 * for the expected calibration error [DD "The Raw Confidence Problem": the average
 * gap between predicted confidence and observed acceptance], the same two
 * quantities per confidence bin.
 *
 * Reading: a position counts when the verifier tested it, i.e. k < L_b and k <= j_b
 * (j_b = accepted count; positions after the first rejection were never tested);
 * it was accepted when k < j_b. Requests with j_b < 0 (invalid) do not count. The
 * bins are ORC_CALIB_BINS equal-width bins of c' over [0, 1] (the last one closed).
 *
 * stats layout (float64): [3*K] per position (sum of c', tested, accepted), then
 * [3*ORC_CALIB_BINS] per bin (tested, sum of c', accepted).
 */
#define ORC_CALIB_BINS 10

static int calib_bin(float c) {
    int bin = (int)floor((double)c * ORC_CALIB_BINS);
    if (bin < 0) bin = 0;
    if (bin > ORC_CALIB_BINS - 1) bin = ORC_CALIB_BINS - 1;
    return bin;
}

int oracle_calib_observe(const float *conf_cal, const int32_t *vlen, const int32_t *acc, int B,
                         int K, double *stats) {
    if (B < 0 || K < 1) return ORC_ERR_ARG;
    double *bins = stats + 3 * (size_t)K;
    for (int b = 0; b < B; b++) {
        int L = vlen[b], j = acc[b];
        if (j < 0 || L < 0 || L > K) continue;
        for (int k = 0; k < L && k <= j; k++) {
            float c = conf_cal[(size_t)b * K + k];
            int a = k < j;
            stats[3 * k + 0] += (double)c;
            stats[3 * k + 1] += 1.0;
            stats[3 * k + 2] += (double)a;
            int bin = calib_bin(c);
            bins[3 * bin + 0] += 1.0;
            bins[3 * bin + 1] += (double)c;
            bins[3 * bin + 2] += (double)a;
        }
    }
    return ORC_OK;
}

/*
 * Window update [DD "The Calibration Loop in Practice"]: for each position with
 * at least one tested token, error = mean c' - acceptance rate and
 * T_k <- T_k + lr * error (an overconfident position gets a higher temperature,
 * [DD "Online Adaptation"]). Reading: the temperature is kept at or above
 * temp_floor > 0 so that the scaling stays defined. The new T_k is rounded to
 * float32. ECE = sum over bins of (n_bin / N) * |acceptance_bin - mean c'_bin| =
 * sum_bins |accepted_bin - sum c'_bin| / N (0 when N = 0). The statistics are then
 * reset for the next window.
 */
int oracle_calib_update(double *stats, float *temps, int K, double lr, double temp_floor,
                        double *ece_out) {
    if (K < 1 || !(temp_floor > 0.0)) return ORC_ERR_ARG;
    for (int k = 0; k < K; k++) {
        double n = stats[3 * k + 1];
        if (n > 0.0) {
            double err = stats[3 * k + 0] / n - stats[3 * k + 2] / n;
            double t = (double)temps[k] + lr * err;
            float tf = (float)t;
            if ((double)tf < temp_floor) tf = (float)temp_floor;
            temps[k] = tf;
        }
    }
    const double *bins = stats + 3 * (size_t)K;
    double N = 0.0, gap = 0.0;
    for (int i = 0; i < ORC_CALIB_BINS; i++) {
        N += bins[3 * i + 0];
        gap += fabs(bins[3 * i + 2] - bins[3 * i + 1]);
    }
    if (ece_out) *ece_out = N > 0.0 ? gap / N : 0.0;
    for (size_t i = 0; i < 3 * (size_t)K + 3 * ORC_CALIB_BINS; i++) stats[i] = 0.0;
    return ORC_OK;
}

/* Exposed for the pins: one calibrated value. */
double oracle_calibrate(double c, double T) { return calibrate_one(c, T); }

/* ======================================================================== */
/* Markov logit-bias head (drafting side)                                    */
/* ======================================================================== */

/* Round a float64 value to bf16 (round to nearest, ties to even) and return its
 * bit pattern; |x| must be finite and within bf16 range. */
static uint16_t to_bf16_rne(double x) {
    if (x == 0.0) return signbit(x) ? 0x8000u : 0u;
    int e;
    double m = frexp(fabs(x), &e);           /* |x| = m * 2^e, m in [0.5, 1) */
    double scaled = ldexp(m, 8);             /* 8 significant bits: bf16 keeps 8 (1 implicit + 7) */
    double lo = floor(scaled), frac = scaled - lo;
    double q;
    if (frac > 0.5 || (frac == 0.5 && fmod(lo, 2.0) != 0.0)) q = lo + 1.0;
    else q = lo;
    double r = ldexp(q, e - 8);
    float rf = (float)r;                      /* exact: r has 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &rf, sizeof bits);
    if (x < 0) bits |= 0x80000000u;
    return (uint16_t)(bits >> 16);
}

static double bf16_value(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * oracle_markov_draft: the semi-autoregressive sampling loop of [GD "1. The Markov
 * Logit-Bias Head" and "Hands-On Implementation"]. For each request b and position
 * k = 0..K-1, with y_{-1} = prev[b]:
 *     L'_{b,k} = L_{b,k} + U (Vm[y_{k-1}, :])^T      (a [V] vector; U, Vm are [V, r])
 *     y_k      = argmax_v L'_{b,k}[v]  (lowest index on ties)
 * The correction is formed in float64 from the bf16 inputs (exact products, sums in
 * index order), L + correction is rounded once to bf16 (to nearest, ties to even) and
 * stored; the argmax is taken over the stored bf16 values. Reading: greedy drafting,
 * as the sketch's argmax; the corrected logits keep the dtype of the raw ones because
 * they are the draft logits the verifier reads.
 *
 * L: [B,K,V] bf16 bits; U, Vm: [V,r] bf16 bits; prev: [B] in [0,V).
 * out_corr: [B,K,V] bf16 bits; out_tok: [B,K].
 * out_edge (or NULL): [B,K] the smallest distance, in units of the bf16 spacing at the
 *   value, between an exact L + correction and a bf16 rounding midpoint, over the row's
 *   elements (a diagnostic for comparing against a kernel with fp32 sums).
 * out_gap (or NULL): [B,K] the gap between the row's largest and second largest
 *   exact L + correction values, relative to the largest magnitude (diagnostic).
 * Returns ORC_ERR_INPUT if a prev token is out of range.
 */
int oracle_markov_draft(const uint16_t *L, const uint16_t *U, const uint16_t *Vm,
                        const int32_t *prev, int B, int K, int V, int r, uint16_t *out_corr,
                        int32_t *out_tok, double *out_edge, double *out_gap) {
    if (B < 0 || K < 1 || V < 1 || r < 1) return ORC_ERR_ARG;
    for (int b = 0; b < B; b++)
        if (prev[b] < 0 || prev[b] >= V) return ORC_ERR_INPUT;
    /* Requests are independent: OpenMP threads take whole requests, so the result
     * does not depend on the thread count. */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int b = 0; b < B; b++) {
        double *x = (double *)malloc(sizeof(double) * (size_t)r);
        int y = prev[b];
        for (int k = 0; k < K; k++) {
            for (int j = 0; j < r; j++) x[j] = bf16_value(Vm[(size_t)y * r + j]);
            size_t row = ((size_t)b * K + k) * (size_t)V;
            int best = -1;
            double bestv = 0.0, edge = INFINITY, top1 = -INFINITY, top2 = -INFINITY, amax = 0.0;
            for (int v = 0; v < V; v++) {
                double c = 0.0;
                for (int j = 0; j < r; j++) c += bf16_value(U[(size_t)v * r + j]) * x[j];
                double z = bf16_value(L[row + v]) + c;
                uint16_t h = to_bf16_rne(z);
                out_corr[row + v] = h;
                double stored = bf16_value(h);
                if (best < 0 || stored > bestv) {
                    best = v;
                    bestv = stored;
                }
                /* diagnostics: distance of z to the nearest rounding midpoint */
                if (z != 0.0) {
                    int e;
                    frexp(fabs(z), &e);
                    double spacing = ldexp(1.0, e - 8);
                    double t = fabs(z) / spacing;
                    double d = fabs((t - floor(t)) - 0.5);
                    if (d < edge) edge = d;
                }
                if (z > top1) {
                    top2 = top1;
                    top1 = z;
                } else if (z > top2) {
                    top2 = z;
                }
                if (fabs(z) > amax) amax = fabs(z);
            }
            out_tok[(size_t)b * K + k] = best;
            if (out_edge) out_edge[(size_t)b * K + k] = edge;
            if (out_gap) out_gap[(size_t)b * K + k] = amax > 0 ? (top1 - top2) / amax : 0.0;
            y = best;
        }
        free(x);
    }
    return ORC_OK;
}

/* ======================================================================== */
/* Throughput-curve scheduling                                               */
/* ======================================================================== */

/* The throughput curve at x tokens: linear between its points (x ascending), flat
 * beyond its first and last points. */
static double curve_at(const float *cx, const float *cy, int n, double x) {
    if (x <= (double)cx[0]) return (double)cy[0];
    for (int i = 1; i < n; i++) {
        if (x <= (double)cx[i]) {
            double x0 = cx[i - 1], x1 = cx[i], y0 = cy[i - 1], y1 = cy[i];
            return y0 + (y1 - y0) * ((x - x0) / (x1 - x0));
        }
    }
    return (double)cy[n - 1];
}

static int desc_double(const void *pa, const void *pb) {
    double a = *(const double *)pa, b = *(const double *)pb;
    return (a < b) - (a > b);
}

/*
 * oracle_schedule_curve: the verify budget chosen from a throughput curve
 * [DD "The Throughput Curve", "The Optimization Logic"]. Reading: a verified token of
 * survival S adds S expected accepted tokens; a step of B requests verifying N drafted
 * tokens runs B + N tokens through the target at T(B + N) tokens/s (the curve) and
 * emits B + A(N) tokens on average, A(N) the sum of the survivals of the N positions
 * kept (the best N in the budget-trim order). The budget is the smallest N maximising
 * the goodput G(N) = (B + A(N)) * T(B + N) / (B + N) over N_lo <= N <= N_hi, with
 * N_hi = min(sum L0, token_budget) and N_lo = B when token_budget >= B (each request
 * keeps its floor position), else 0; then the trim of oracle_schedule runs with it.
 * At small batches, where T grows with the batch, adding a token raises G and every
 * tau-survivor is verified; where T is flat, low-survival tokens lower it.
 *
 * conf/temps/load/tau...: as oracle_schedule_ex. curve_x [n_pts] ascending (tokens),
 * curve_y [n_pts] > 0 (tokens/s), float32. out_n: the chosen N; out_g: G(N).
 * Returns ORC_ERR_INPUT for an invalid curve (n_pts < 1, x not strictly ascending,
 * y <= 0 or not finite) as for the other device inputs.
 */
int oracle_schedule_curve(const float *conf, const float *temps, const float *load, float tau,
                          float tau_min, float tau_max, const float *curve_x,
                          const float *curve_y, int n_pts, int B, int K, long long token_budget,
                          int32_t *out_len, int32_t *out_n, double *out_g) {
    if (B < 0 || K < 1 || token_budget < 0 || n_pts < 1) return ORC_ERR_ARG;
    int bad = 0;
    for (int i = 0; i < n_pts; i++) {
        if (!(isfinite(curve_x[i]) && isfinite(curve_y[i]) && curve_y[i] > 0.0f)) bad = 1;
        if (i > 0 && !(curve_x[i] > curve_x[i - 1])) bad = 1;
    }
    for (int b = 0; b < B; b++) out_len[b] = 0;
    if (bad) return ORC_ERR_INPUT;
    double *S = (double *)malloc(sizeof(double) * ((size_t)B * K + 1));
    int32_t *L0 = (int32_t *)malloc(sizeof(int32_t) * ((size_t)B + 1));
    int rc = oracle_schedule_ex(conf, temps, load, tau, tau_min, tau_max, B, K, (long long)B * K,
                                out_len, S, L0, NULL, NULL);
    if (rc != ORC_OK || B == 0) {
        free(S);
        free(L0);
        return rc;
    }
    long long total = 0;
    for (int b = 0; b < B; b++) total += L0[b];
    long long n_hi = total < token_budget ? total : token_budget;
    int floors = token_budget >= B;
    long long n_lo = floors ? B : 0;
    /* competing survivals, descending (ties in any order: only their sum matters) */
    double *c = (double *)malloc(sizeof(double) * ((size_t)B * K + 1));
    size_t nc = 0;
    double a_floor = 0.0;
    for (int b = 0; b < B; b++)
        for (int k = 0; k < L0[b]; k++) {
            double s = S[(size_t)b * K + k];
            if (floors && k == 0) a_floor += s;
            else c[nc++] = s;
        }
    qsort(c, nc, sizeof(double), desc_double);
    double best_g = -1.0, a = a_floor;
    long long best_n = n_lo;
    for (long long n = n_lo; n <= n_hi; n++) {
        if (n > n_lo) a += c[n - n_lo - 1];
        double x = (double)B + (double)n;
        double g = ((double)B + a) * curve_at(curve_x, curve_y, n_pts, x) / x;
        if (g > best_g) {
            best_g = g;
            best_n = n;
        }
    }
    if (out_n) *out_n = (int32_t)best_n;
    if (out_g) *out_g = best_g;
    rc = oracle_schedule_ex(conf, temps, load, tau, tau_min, tau_max, B, K, best_n, out_len, NULL,
                            NULL, NULL, NULL);
    free(c);
    free(S);
    free(L0);
    return rc;
}

/* ======================================================================== */
/* Tree (multi-candidate) verification                                      */
/* ======================================================================== */

/*
 * The pages name tree verification without defining it: the DSpark Guide's
 * pipeline ("Deep Dive into the DSpark Architecture", step 4) forwards the
 * verified prefix "with tree / sequence mask", and its feature matrix ("3.
 * Comprehensive Technical Feature Matrix") lists "Static / Tree" verification
 * for EAGLE-3. Reading taken here, the plainest lossless one that reduces to the
 * chain of [DD "The Speculative Decoding Solution"] when every node has at most
 * one child:
 *
 *  - Request b holds a token tree of n_nodes[b] nodes. Node 0 is the committed
 *    context; node n >= 1 carries the drafted token tok[n] and has parent
 *    par[n] < n. Target row n is the target's logits after the path 0 -> n;
 *    draft row n is the drafter's logits the children of n were drawn from,
 *    each child independently (with replacement).
 *  - The walk starts at node 0. At node c the children are tested in index
 *    order against a residual distribution r that starts as p_c: child n with
 *    token x is accepted when u_n * q_c(x) < r(x) (probability
 *    min(1, r(x)/q_c(x))); the walk then moves to n. After a rejection r
 *    becomes normalize(max(0, r - q_c)), so the next child is tested against
 *    the target mass the rejected draws left uncovered.
 *  - When every child of c is rejected, the token is sampled from r by inverse
 *    CDF at u_{b,0} (for one child this is the chain's residual sample); at a
 *    leaf, from p_c (the chain's bonus token).
 *  - At T == 0: accept the first child (index order) whose token is the lowest
 *    index argmax of target row c; otherwise emit that argmax.
 *  - Rows the walk never reaches are not read, so their contents (even NaN)
 *    do not matter. A reached row that is not a valid logit row makes the
 *    request invalid, as do bad tree links, tokens or uniforms.
 *  - Reading for a residual with no mass left (p == q up to rounding): r starts
 *    again from p_c, as the chain falls back to sampling p.
 */

/* Near-tie bookkeeping of one decision at residual state (lam, W), where
 * r = max(0, p - lam*q) / W in closed form (lam = 0, W = 1 for r = p). A kernel
 * forming r from fp32 p and q carries an error in r/q of about eps*(1 + 2 lam)/W,
 * and in a CDF position of about eps*(1 + lam)/W, so the margins are divided by
 * those factors before they are compared with the window. */
static double tree_scale_test(double lam, double W) { return (1.0 + 2.0 * lam) / W; }
static double tree_scale_cdf(double lam, double W) { return (1.0 + lam) / W; }

static int tree_one(const void *tgt, const void *drf, int dtype, const int32_t *par,
                    const int32_t *tok, const int32_t *nnod, const double *u, int b, int N,
                    int V, double T, int32_t *out_tok, int32_t *out_acc, int32_t *out_path,
                    int32_t *out_flags, double *out_margin, double *p, double *q, double *r,
                    double *w) {
    const size_t base = (size_t)b * N;
    int32_t *ot = out_tok + base;
    int32_t *op = out_path ? out_path + base : NULL;
    for (int i = 0; i < N; i++) {
        ot[i] = -1;
        if (op) op[i] = -1;
    }
    out_acc[b] = -1;
    out_flags[b] = 0;
    double margin = INFINITY;
    if (out_margin) out_margin[b] = INFINITY;

    const int nn = nnod[b];
    if (nn < 1 || nn > N) goto invalid;
    for (int n = 1; n < nn; n++) {
        if (par[base + n] < 0 || par[base + n] >= n) goto invalid;
        if (tok[base + n] < 0 || tok[base + n] >= V) goto invalid;
    }
    if (T > 0.0)
        for (int n = 0; n < nn; n++)
            if (!(u[base + n] >= 0.0 && u[base + n] < 1.0)) goto invalid;

    int c = 0, depth = 0;
    for (;;) {
        double Mt, Md;
        int At, Ad;
        if (row_scan(tgt, dtype, (base + c) * (size_t)V, V, &Mt, &At)) goto invalid;
        int first_child = -1;
        for (int n = c + 1; n < nn; n++)
            if (par[base + n] == c) {
                first_child = n;
                break;
            }

        if (T == 0.0) {
            int next = -1;
            for (int n = c + 1; n < nn && next < 0; n++)
                if (par[base + n] == c && tok[base + n] == At) next = n;
            if (next < 0) {
                ot[depth] = At;
                out_acc[b] = depth;
                return 0;
            }
            ot[depth] = tok[base + next];
            if (op) op[depth] = next;
            depth++;
            c = next;
            continue;
        }

        row_softmax(tgt, dtype, (base + c) * (size_t)V, V, T, Mt, p);
        if (first_child < 0) {
            /* A leaf: the bonus token from p_c. */
            double Z, gap;
            int y = inverse_cdf(p, V, u[base], &Z, &gap);
            if (gap < NEAR_TIE) out_flags[b] |= ORC_FLAG_CDF_EDGE;
            if (gap < margin) margin = gap;
            if (out_margin) out_margin[b] = margin;
            ot[depth] = y;
            out_acc[b] = depth;
            return 0;
        }
        if (row_scan(drf, dtype, (base + c) * (size_t)V, V, &Md, &Ad)) goto invalid;
        row_softmax(drf, dtype, (base + c) * (size_t)V, V, T, Md, q);

        for (int v = 0; v < V; v++) r[v] = p[v];
        const double *wlast = p; /* weights of the terminal sample if all are rejected */
        double lam = 0.0, W = 1.0; /* r = max(0, p - lam*q) / W (diagnostics only) */
        int next = -1;
        for (int n = first_child; n < nn; n++) {
            if (par[base + n] != c) continue;
            const int x = tok[base + n];
            const double un = u[base + n];
            const double rx = r[x], qx = q[x];
            double ratio = qx > 0.0 ? (rx / qx < 1.0 ? rx / qx : 1.0) : (rx > 0.0 ? 1.0 : 0.0);
            double mg = fabs(un - ratio) / tree_scale_test(lam, W);
            if (mg < NEAR_TIE) out_flags[b] |= ORC_FLAG_ACCEPT_TIE;
            if (mg < margin) margin = mg;
            if (rx < 1e-30 && qx < 1e-30) out_flags[b] |= ORC_FLAG_TINY_PROB;
            if (un * qx < rx) {
                next = n;
                break;
            }
            /* Rejected: r <- normalize(max(0, r - q)). */
            double Z = 0.0;
            for (int v = 0; v < V; v++) {
                w[v] = r[v] - q[v] > 0.0 ? r[v] - q[v] : 0.0;
                Z += w[v];
            }
            lam += W;
            W *= Z;
            if (W < NEAR_TIE) out_flags[b] |= ORC_FLAG_SMALL_RESIDUAL;
            if (Z > 0.0) {
                for (int v = 0; v < V; v++) r[v] = w[v] / Z;
                wlast = w;
            } else {
                for (int v = 0; v < V; v++) r[v] = p[v];
                wlast = p;
                lam = 0.0;
                W = 1.0;
            }
        }
        if (next >= 0) {
            ot[depth] = tok[base + next];
            if (op) op[depth] = next;
            depth++;
            c = next;
            continue;
        }
        /* Every child rejected: sample the residual at u_{b,0}. */
        double Z, gap;
        int y = inverse_cdf(wlast, V, u[base], &Z, &gap);
        if (y < 0) y = inverse_cdf(p, V, u[base], &Z, &gap);
        gap /= tree_scale_cdf(lam, W);
        if (gap < NEAR_TIE) out_flags[b] |= ORC_FLAG_CDF_EDGE;
        if (gap < margin) margin = gap;
        if (out_margin) out_margin[b] = margin;
        ot[depth] = y;
        out_acc[b] = depth;
        return 0;
    }

invalid:
    for (int i = 0; i < N; i++) {
        ot[i] = -1;
        if (op) op[i] = -1;
    }
    out_acc[b] = -1;
    out_flags[b] = ORC_FLAG_INVALID;
    return -1;
}

/*
 * oracle_verify_tree_u64: batched tree verification with float64 uniforms.
 *
 *  target, draft: [B, N, V] logits (dtype 0 = fp32, 1 = bf16 bits); draft may be
 *    NULL at T == 0.
 *  par, tok: [B, N] parent links and drafted tokens (entry 0 of each unused).
 *  nnod: [B] nodes in use, 1..N.
 *  u: [B, N]: u[b,n] (n >= 1) drives the test of node n; u[b,0] the terminal
 *    sample. Unused at T == 0.
 *  out_tok [B, N]: tokens of the accepted path, then the terminal token, then -1.
 *  out_acc [B]: accepted drafted tokens (the path's depth), or -1 if invalid.
 *  out_path [B, N] or NULL: node index of each accepted token, then -1.
 *  out_flags [B], out_margin [B] or NULL: as oracle_verify (scaled margins).
 * Returns ORC_OK, ORC_ERR_ARG, or ORC_ERR_INPUT if any request was invalid.
 */
int oracle_verify_tree_u64(const void *target, const void *draft, int dtype,
                           const int32_t *par, const int32_t *tok, const int32_t *nnod,
                           const double *u, int B, int N, int V, double T, int32_t *out_tok,
                           int32_t *out_acc, int32_t *out_path, int32_t *out_flags,
                           double *out_margin, int nthreads) {
    if (B < 0 || N < 1 || V < 1 || (dtype != 0 && dtype != 1) || !(T >= 0.0) || !isfinite(T))
        return ORC_ERR_ARG;
    if (B == 0) return ORC_OK;
    if (!target || !par || !tok || !nnod || !out_tok || !out_acc || !out_flags)
        return ORC_ERR_ARG;
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
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int b = 0; b < B; b++)
            if (tree_one(target, draft, dtype, par, tok, nnod, u, b, N, V, T, out_tok, out_acc,
                         out_path, out_flags, out_margin, p, q, r, w))
                n_invalid++;
        free(p);
        free(q);
        free(r);
        free(w);
    }
    return n_invalid ? ORC_ERR_INPUT : ORC_OK;
}

/* oracle_verify_tree_u64 with the float32 uniforms of the C-ABI, widened exactly. */
int oracle_verify_tree(const void *target, const void *draft, int dtype, const int32_t *par,
                       const int32_t *tok, const int32_t *nnod, const float *u, int B, int N,
                       int V, float T, int32_t *out_tok, int32_t *out_acc, int32_t *out_path,
                       int32_t *out_flags, double *out_margin, int nthreads) {
    double *u64 = NULL;
    if (u && B > 0) {
        u64 = (double *)malloc(sizeof(double) * (size_t)B * N);
        for (size_t i = 0; i < (size_t)B * N; i++) u64[i] = (double)u[i];
    }
    int rc = oracle_verify_tree_u64(target, draft, dtype, par, tok, nnod, u64, B, N, V,
                                    (double)T, out_tok, out_acc, out_path, out_flags, out_margin,
                                    nthreads);
    free(u64);
    return rc;
}
