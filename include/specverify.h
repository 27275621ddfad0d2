/*
 * specverify.h -- C-ABI of libspecverify: batched, lossless verification of drafted
 * token blocks, and the confidence schedule that sets how many drafted tokens of each
 * request go to verification. GB300 (sm_103a) only.
 *
 * The method is DSpark's ("confidence-scheduled, semi-autoregressive speculative
 * decoding"). Sources, cited by page title and section:
 *  [DD] "DSpark Deep Dive: How DeepSeek Squeezed an 85% Speedup Out of Inference
 *       Without Touching a Single Model Weight" (fuyuan7.com)
 *  [GD] "DSpark Guide: Confidence Speculative Decoding in LLMs" (aifetchly)
 *  [TP] perchy.ai "Technology", engine 01, "Verified by the target"
 *
 * Conventions for every call
 *  - Pointers named *_d are DEVICE pointers owned by the caller; tensors are dense,
 *    row-major, and aligned to their element size. Nothing is allocated per call.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL means
 *    the legacy default stream). A return of SV_OK means the work was enqueued.
 *  - Arguments the host can check are checked before anything is enqueued; a bad
 *    argument returns SV_ERR_ARG / SV_ERR_SHAPE / SV_ERR_DTYPE / SV_ERR_WORKSPACE
 *    and enqueues nothing. Errors in device-resident data (NaN or +inf logits, a
 *    row of -inf, a token outside [0,V), a verify length outside [0,K], a uniform
 *    outside [0,1), a confidence outside [0,1]) cannot be seen by the host: the
 *    kernels mark the affected request (out_accepted = -1, its out_tok row = -1; or
 *    out_len = 0 for the schedule) and set a sticky bit in the workspace status
 *    word, readable with sv_get_status. Kernels never trap.
 *  - A workspace serves one call at a time: calls that share a workspace must be
 *    ordered on one stream. Calls on different workspaces may run concurrently.
 *  - Grids depend only on (B, K, V, dtype, greedy), and device-resident lengths are
 *    read on the device, so a call sequence can be captured in a CUDA graph and
 *    replayed with new data in the same buffers.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sv_status {
    SV_OK = 0,
    SV_ERR_ARG = -1,          /* null pointer, non-finite or out-of-range scalar */
    SV_ERR_SHAPE = -2,        /* B, K or V outside the supported range */
    SV_ERR_DTYPE = -3,        /* unknown sv_dtype */
    SV_ERR_CUDA = -4,         /* a CUDA runtime call failed (launch, attribute query) */
    SV_ERR_DEVICE_INPUT = -5, /* (status word) invalid device-resident data was seen */
    SV_ERR_TIMEOUT = -6,      /* (status word) a bounded device wait gave up */
    SV_ERR_WORKSPACE = -7     /* workspace missing, too small or misaligned */
} sv_status;

typedef enum sv_dtype { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Supported sizes. */
#define SV_MAX_B 4096         /* requests per verify call */
#define SV_MAX_K 32           /* drafted positions per request */
#define SV_MAX_V (1 << 24)    /* vocabulary entries */
#define SV_MAX_SCHED_B 8192   /* requests per schedule call */
#define SV_MAX_SCHED_BK 16384 /* B*K per schedule call */
#define SV_CALIB_BINS 10      /* equal-width confidence bins of the calibration error */
#define SV_MAX_MARKOV_R 256   /* rank of the Markov logit-bias head */
#define SV_MAX_CURVE 64       /* points of a throughput curve */
#define SV_MAX_CURVE_BK 8192  /* B*K of a throughput-curve schedule */
#define SV_MAX_TREE 64        /* nodes of a draft tree */

/*
 * sv_workspace_bytes: size of the device workspace needed by sv_schedule and
 * sv_verify for shapes up to (B, K, V), for either dtype (0 for an unsupported
 * shape). The caller allocates it (256-byte aligned) and zeroes it once with
 * sv_workspace_init before first use; every call leaves it ready for the next call,
 * of any shape that fits, including after device-side errors.
 */
size_t sv_workspace_bytes(int B, int K, int V);

/* Zero a workspace on `stream` (one cudaMemsetAsync). */
sv_status sv_workspace_init(void *ws_d, size_t ws_bytes, void *stream);

/*
 * sv_schedule: per-request verify lengths from per-position draft confidences.
 * [GD "2. Confidence-Scheduled Dynamic Verification"; DD "Variable-Length Drafts",
 *  "The Optimization Logic", "GPU-Resident Scheduling", "The Full Scheduling Pipeline"]
 *
 *  conf_d     [B,K] float32, c_{b,k} in [0,1]: calibrated probability that drafted
 *             token k of request b is accepted.
 *  tau        survival threshold in [0,1].
 *  token_budget  global cap (>= 0) on sum_b out_len[b] (drafted tokens sent to
 *             verification; the +1 target row per request is not counted).
 *  out_len_d  [B] int32 result L_b.
 *
 *  1. Prefix survival S_{b,k} = c_{b,0} * ... * c_{b,k}, computed left to right in
 *     float64 (the product of per-position survival, [GD] C_k).
 *  2. L0_b = max(1, #{k : S_{b,k} >= tau}) (truncate at the first C_k < tau, keep
 *     at least one token [GD "Hands-On Implementation"]; 1 <= L <= K [DD]).
 *  3. If sum_b L0_b > token_budget, keep the token_budget highest-ranked positions
 *     among the tau-survivors and drop the rest, lowest marginal survival first.
 *     Rank: guaranteed floor positions (b,0) first when token_budget >= B; then S
 *     descending, position k ascending, request b ascending. When token_budget < B
 *     the floor positions compete like the others and a request can get L_b = 0.
 *     Kept positions always form a prefix of each request's block.
 *  One CTA; a few microseconds. Device errors: a confidence outside [0,1] or NaN
 *  sets SV_ERR_DEVICE_INPUT in the status word and writes out_len = 0 everywhere.
 *  Limits: 1 <= K <= SV_MAX_K, 0 <= B <= SV_MAX_SCHED_B, B*K <= SV_MAX_SCHED_BK.
 *  The workspace needs only its 256-byte header (any size from sv_workspace_bytes).
 */
sv_status sv_schedule(const float *conf_d, int B, int K, float tau, int token_budget,
                      int32_t *out_len_d, void *ws_d, size_t ws_bytes, void *stream);

/*
 * sv_schedule_cal: sv_schedule with its two device-resident inputs from the pages'
 * scheduling pipeline [DD "The Full Scheduling Pipeline": raw confidence -> online
 * calibration -> scheduler with the GPU's load state -> verify length].
 *
 *  temps_d    [K] float32 per-position temperatures T_k (> 0, finite), or NULL for
 *             no calibration. Each confidence becomes c' = sigmoid(logit(c) / T_k)
 *             [DD "Sequential Temperature Scaling"], computed in fp32 (c = 0 and
 *             c = 1 stay fixed); the survival products then run on c' in float64.
 *  load_d     [4] float32 {Q, Q_max, M_gpu, M_max}: queue depth and GPU memory use
 *             with their maxima, or NULL to use `tau` as given. Otherwise
 *             LF = 0.6 Q/Q_max + 0.4 M_gpu/M_max, clamped to 1, and
 *             tau = tau_min + (tau_max - tau_min) LF^2, in float64
 *             [GD "Dynamic Verification Scheduling Algorithm", steps 1-2].
 *  tau_min, tau_max  in [0,1]; read only when load_d is given (the page's example
 *             range is 0.20 to 0.75).
 *  conf_cal_d [B,K] float32 out: c' (the input of sv_calib_observe), or NULL.
 *  tau_out_d  [1] float64 out: the threshold used, or NULL.
 *  Other arguments, steps 1-3, limits and the workspace: as sv_schedule. Device
 *  errors (SV_ERR_DEVICE_INPUT, out_len = 0 everywhere): a confidence outside [0,1],
 *  a temperature that is not a positive finite number, a load value that is not
 *  finite, a negative Q or M_gpu, or a maximum that is not > 0. When B == 0 nothing
 *  is enqueued and nothing is written.
 */
sv_status sv_schedule_cal(const float *conf_d, const float *temps_d, const float *load_d,
                          float tau, float tau_min, float tau_max, int B, int K,
                          int token_budget, int32_t *out_len_d, float *conf_cal_d,
                          double *tau_out_d, void *ws_d, size_t ws_bytes, void *stream);

/*
 * sv_schedule_curve: sv_schedule_cal whose budget is chosen from the target's
 * throughput curve [DD "The Throughput Curve", "The Optimization Logic"].
 *
 *  curve_d  [2 * n_pts] float32: batch sizes in tokens (strictly ascending), then the
 *           tokens/s at each (> 0); linear between points, flat beyond the ends.
 *  n_pts    1 <= n_pts <= SV_MAX_CURVE.
 *  n_out_d  [1] int32 out (or NULL): the chosen budget N; g_out_d [1] float64 out (or
 *           NULL): its goodput.
 *  A verified token of survival S adds S expected accepted tokens; a step verifying N
 *  drafted tokens of B requests runs B + N tokens at T(B + N) tokens/s and emits
 *  B + A(N) on average, A(N) the sum of the survivals kept (the best N in the trim
 *  order). N is the smallest value maximising (B + A(N)) T(B + N) / (B + N) between
 *  N_lo = B (0 when token_budget < B) and min(sum L0, token_budget), all in float64;
 *  the trim of sv_schedule then runs with budget N. Limits: as sv_schedule, and
 *  B * K <= SV_MAX_CURVE_BK. An invalid curve is a device error (SV_ERR_DEVICE_INPUT,
 *  out_len = 0).
 */
sv_status sv_schedule_curve(const float *conf_d, const float *temps_d, const float *load_d,
                            float tau, float tau_min, float tau_max, const float *curve_d,
                            int n_pts, int B, int K, int token_budget, int32_t *out_len_d,
                            float *conf_cal_d, double *tau_out_d, int32_t *n_out_d,
                            double *g_out_d, void *ws_d, size_t ws_bytes, void *stream);

/*
 * Online calibration loop [DD "The Calibration Loop in Practice", "Online
 * Adaptation"; ECE: "The Raw Confidence Problem"]. The caller owns a window buffer
 * of sv_calib_stats_len(K) float64 values (zeroed once), calls sv_calib_observe after
 * every verification round and sv_calib_update every N rounds (the page's example
 * window is about 500 rounds).
 *
 * Window layout (float64): per position k (3K values): sum of c', tested tokens,
 * accepted tokens; then per confidence bin i (3 SV_CALIB_BINS values; bin i holds
 * c' in [i/10, (i+1)/10), the last bin also 1): tested, sum of c', accepted.
 */
size_t sv_calib_stats_len(int K); /* 0 for K outside [1, SV_MAX_K] */

/*
 * sv_calib_observe: add one verification round to the window.
 *  conf_cal_d [B,K] float32 c' (sv_schedule_cal's conf_cal_d), verify_len_d [B] and
 *  accepted_d [B] (sv_verify's input and out_accepted). Position k of request b
 *  counts when it was tested, k < L_b and k <= j_b (j_b = accepted count; later
 *  positions were never tested), and as accepted when k < j_b; requests with
 *  j_b < 0 or L_b outside [0,K] are skipped. One small launch; the sums are formed
 *  in a fixed order, so repeated runs give identical windows.
 *  Limits: 0 <= B <= SV_MAX_B, 1 <= K <= SV_MAX_K. stats_d is read and written.
 */
sv_status sv_calib_observe(const float *conf_cal_d, const int32_t *verify_len_d,
                           const int32_t *accepted_d, int B, int K, double *stats_d,
                           void *stream);

/*
 * sv_calib_update: close the window. For each position k with a tested token,
 * error_k = (sum c')/tested - accepted/tested and T_k <- T_k + lr * error_k (float64,
 * rounded to float32), then T_k <- max(T_k, temp_floor) so the scaling stays defined
 * (an overconfident position gets a higher temperature). ece_d [1] float64 out (or
 * NULL): sum over bins of |accepted - sum c'| / total tested (0 for an empty window).
 * The window is then zeroed. lr finite (the pages use 0.001 to 0.01); temp_floor > 0.
 */
sv_status sv_calib_update(double *stats_d, float *temps_d, int K, float lr, float temp_floor,
                          double *ece_d, void *stream);

/*
 * sv_markov_draft: the drafter's Markov logit-bias head and greedy drafting loop
 * [GD "1. The Markov Logit-Bias Head"; GD "Hands-On Implementation"]. For k = 0..K-1
 * and every request b, with y_{-1} = prev_tok[b]:
 *     L'_{b,k} = L_{b,k} + U (Vm[y_{k-1}, :])^T       (U, Vm: [V, r] low-rank factors)
 *     y_k      = the lowest index of the largest value of L'_{b,k} (as stored)
 *
 *  logits_d    [B, K, V] bf16 raw logits of the parallel backbone.
 *  U_d, Vm_d   [V, r] bf16, r a multiple of 16 in [16, SV_MAX_MARKOV_R].
 *  prev_tok_d  [B] int32, the last token before the block (in [0, V)).
 *  corrected_d [B, K, V] bf16 out: L' (the correction in fp32 on the tensor cores,
 *              added to L in fp32 and rounded once to bf16); these are the draft
 *              logits that sv_verify reads.
 *  draft_tok_d [B, K] int32 out: y_k (-1 for a request whose prev_tok is invalid; its
 *              corrected rows are then unspecified and SV_ERR_DEVICE_INPUT is set).
 *  keys_d      [K * B] uint64 scratch (sv_markov_keys_len), overwritten.
 *  ws_d        a workspace (its status word and a counter in its header; any size
 *              from sv_workspace_bytes).
 *  After zeroing keys_d: at B <= 128 one cooperative launch runs all K positions (one
 *  CTA per SM; the CTAs meet at a grid barrier between positions, whose counter sits
 *  in the workspace header and is reset by the last launch), otherwise one launch per
 *  position; then one launch writes the tokens. Capturable in a CUDA graph. A wait
 *  that runs out (~2 s) sets SV_ERR_TIMEOUT. logits_d and corrected_d must be 16-byte
 *  aligned, U_d and Vm_d too. Limits: 0 <= B <= SV_MAX_B, 1 <= K <= SV_MAX_K,
 *  1 <= V <= SV_MAX_V.
 */
size_t sv_markov_keys_len(int B, int K); /* uint64 elements of keys_d; 0 if out of range */
sv_status sv_markov_draft(const void *logits_d, const void *U_d, const void *Vm_d,
                          const int32_t *prev_tok_d, int B, int K, int V, int r,
                          void *corrected_d, int32_t *draft_tok_d, unsigned long long *keys_d,
                          void *ws_d, size_t ws_bytes, void *stream);

/*
 * sv_verify: standard speculative rejection sampling over a batch of drafted blocks.
 * [DD "Speculative Decoding From First Principles" / "The Speculative Decoding
 *  Solution"; GD "1. The Mathematics of Suffix Decay"; TP "Verified by the target"]
 *
 *  target_d   [B, K+1, V] target logits (dtype), row k = target prediction for the
 *             position of drafted token k; row L_b is the bonus position.
 *  draft_d    [B, K, V] draft logits (dtype). Not read when temperature == 0 (may be
 *             NULL then).
 *  draft_tok_d [B, K] int32 drafted tokens x_{b,k}.
 *  verify_len_d [B] int32 L_b in [0, K] (for example sv_schedule's out_len; rows
 *             past L_b are never read, so only the verified prefix must hold data).
 *  uniforms_d [B, K+1] float32 in [0,1): u_{b,k} (k < K) drives the accept test of
 *             drafted token k; u_{b,K} drives the terminal sample. Not read when
 *             temperature == 0 (may be NULL then).
 *  temperature  T >= 0. p_k = softmax(target_k / T), q_k = softmax(draft_k / T).
 *             T == 0 selects greedy verification; otherwise 1e-6 <= T <= 1e6.
 *  out_tok_d  [B, K+1] int32: x_{b,0..j-1}, then the terminal token y, then -1.
 *  out_accepted_d [B] int32: j, the number of accepted drafted tokens (or -1).
 *
 *  Per request: accept x_k iff u_k * q_k(x_k) < p_k(x_k), i.e. with probability
 *  min(1, p/q); j = first rejected position, or L_b. If j < L_b the terminal token
 *  is the inverse-CDF sample of max(0, p_j - q_j) (normalised) at u_{b,K}: the
 *  smallest v with u*Z < r_0 + ... + r_v; if that residual has no mass left the
 *  sample is taken from p_j instead. If j == L_b it is the inverse-CDF sample of
 *  p_{L_b} at u_{b,K} (bonus token). At T == 0: accept iff x_k is the lowest-index
 *  argmax of target row k, and the terminal token is the argmax of row j. The
 *  emitted tokens follow the target distribution exactly.
 *  Arithmetic: fp32 softmax statistics; the terminal inverse CDF is accumulated in
 *  float-float (about 48 significant bits) over compensated fp32 sums.
 *  Limits: 0 <= B <= SV_MAX_B, 1 <= K <= SV_MAX_K, 1 <= V <= SV_MAX_V.
 */
sv_status sv_verify(const void *target_d, const void *draft_d, sv_dtype dtype,
                    const int32_t *draft_tok_d, const int32_t *verify_len_d,
                    const float *uniforms_d, int B, int K, int V, float temperature,
                    int32_t *out_tok_d, int32_t *out_accepted_d, void *ws_d,
                    size_t ws_bytes, void *stream);

/*
 * sv_verify_diag: sv_verify plus diagnostics (same decisions, same arguments).
 *  out_p_d, out_q_d [B, K] float32 or NULL: p_k(x_k) and q_k(x_k) for k < L_b
 *           (NaN for k >= L_b, and at T == 0).
 *  accept_count_d [K] uint32 or NULL: for each position k, atomically adds the
 *           number of requests whose drafted token k was accepted.
 *  tested_count_d [K] uint32 or NULL: adds the number of requests that tested
 *           position k (k <= j and k < L_b). accept/tested is the per-position
 *           acceptance rate the online calibration of [DD "Online Calibration"]
 *           compares against the predicted confidence.
 *  near_tie_flags_d [B] int32 or NULL: per request, the decisions that were close
 *           enough to a boundary that fp32 rounding could have changed them (the
 *           accept rule u < min(1, p/q) and the residual sample of [DD "The
 *           Speculative Decoding Solution"]); 0 for a request with none. Bits:
 *             1  an accept test at a tested position (k <= j, k < L_b) had
 *                |u_k - min(1, p/q)| < 1e-5 (min(1, p/q) read as 1 when q = 0 < p,
 *                and 0 when p = q = 0);
 *             2  the terminal sample's target u_{b,K} * Z lay within 1e-5 * Z of an
 *                edge of the chosen token's inverse-CDF bucket (Z = total weight);
 *             4  p and q were both below 1e-30 at a tested position;
 *             8  the residual max(0, p_j - q_j) had less than 1e-5 of mass;
 *            16  the request is invalid (out_accepted = -1).
 *           At T == 0: 0, or 16 for an invalid request. Computed from the kernel's own
 *           fp32 / float-float values, so a flag can differ from an exact
 *           computation's only when the exact margin is itself within about 2e-6 of
 *           the 1e-5 window.
 */
sv_status sv_verify_diag(const void *target_d, const void *draft_d, sv_dtype dtype,
                         const int32_t *draft_tok_d, const int32_t *verify_len_d,
                         const float *uniforms_d, int B, int K, int V, float temperature,
                         int32_t *out_tok_d, int32_t *out_accepted_d, float *out_p_d,
                         float *out_q_d, uint32_t *accept_count_d, uint32_t *tested_count_d,
                         int32_t *near_tie_flags_d, void *ws_d, size_t ws_bytes,
                         void *stream);

/*
 * sv_set_wait_limit: bound, in GPU clock cycles, on how long a verify call's warps
 * wait for results published by other warps (a row's partial sums, a request's
 * decision, a queued terminal job) before the call gives up: SV_ERR_TIMEOUT in the
 * status word, outputs unspecified, the workspace left ready for the next call.
 * cycles <= 0 restores the default (about 2 s). Applies to calls made afterwards in
 * this process; returns the previous bound. A testing aid: the default is far above
 * any normal wait. The library has no counterpart on the pages.
 */
long long sv_set_wait_limit(long long cycles);

/*
 * sv_verify_tree: verification of drafted token trees (multi-candidate rejection
 * sampling). The DSpark Guide names tree verification without defining it ("Deep
 * Dive into the DSpark Architecture", step 4, "tree / sequence mask"; "3.
 * Comprehensive Technical Feature Matrix", "Static / Tree"); this call takes the
 * lossless reading that reduces to sv_verify when every node has at most one child.
 *
 *  target_d   [B, N, V] target logits (dtype): row n = the target's prediction after
 *             the path from node 0 to node n (node 0 = the committed context).
 *  draft_d    [B, N, V] draft logits (dtype): row n = the distribution the children
 *             of node n were drawn from, independently. Read only for nodes with
 *             children that the walk reaches; not read at T == 0 (may be NULL then).
 *  parent_d   [B, N] int32: parent of node n (0 <= parent < n for 1 <= n < n_nodes);
 *             entry 0 is ignored.
 *  draft_tok_d [B, N] int32: the drafted token of node n >= 1; entry 0 is ignored.
 *  n_nodes_d  [B] int32 in [1, N]: nodes in use (nodes at or past it are ignored).
 *  uniforms_d [B, N] float32 in [0,1): u_{b,n} (n >= 1) drives the test of node n,
 *             u_{b,0} the terminal sample. Not read at T == 0 (may be NULL then).
 *  temperature  as sv_verify.
 *  out_tok_d  [B, N] int32: tokens of the accepted path, then the terminal token,
 *             then -1.
 *  out_accepted_d [B] int32: accepted drafted tokens (the depth of the path), or -1.
 *  out_path_d [B, N] int32 or NULL: node index of each accepted token, then -1 (the
 *             nodes whose KV entries the caller keeps).
 *  ws_d       any workspace of at least 256 bytes (only its status word is used).
 *
 *  Per request: the walk starts at node 0. At node c the children are tested in
 *  index order against a residual r that starts as p_c: child n with token x is
 *  accepted iff u_{b,n} * q_c(x) < r(x) and the walk moves to n; after a rejection
 *  r <- normalize(max(0, r - q_c)) (if no mass is left, r restarts from p_c). When
 *  every child is rejected the terminal token is the inverse-CDF sample of r at
 *  u_{b,0}; at a leaf it is sampled from p_c. At T == 0 the first child drafting the
 *  lowest-index argmax of target row c is accepted, else that argmax is emitted. The
 *  emitted tokens follow the target distribution exactly when siblings are
 *  independent draws from the parent's draft distribution.
 *  Only rows the walk reaches are read; a reached row with NaN or +inf (or all -inf),
 *  a bad parent link or token, n_nodes outside [1, N] or a uniform outside [0,1) make
 *  the request invalid: its outputs are -1 and SV_ERR_DEVICE_INPUT is set.
 *  Arithmetic: fp32 softmax statistics and weights, float-float sums and prefixes.
 *  Limits: 0 <= B <= SV_MAX_B, 1 <= N <= SV_MAX_TREE, 1 <= V <= SV_MAX_V.
 */
sv_status sv_verify_tree(const void *target_d, const void *draft_d, sv_dtype dtype,
                         const int32_t *parent_d, const int32_t *draft_tok_d,
                         const int32_t *n_nodes_d, const float *uniforms_d, int B, int N,
                         int V, float temperature, int32_t *out_tok_d,
                         int32_t *out_accepted_d, int32_t *out_path_d, void *ws_d,
                         size_t ws_bytes, void *stream);

/*
 * sv_get_status: wait for `stream`, then read the sticky status word of the
 * workspace into *status_out (SV_OK, SV_ERR_DEVICE_INPUT or SV_ERR_TIMEOUT; the most
 * severe seen since the last clear). clear != 0 resets it to SV_OK.
 * Returns SV_OK or the error of the copy.
 */
sv_status sv_get_status(void *ws_d, void *stream, int clear, int32_t *status_out);

/*
 * sv_verify_static: sv_verify for callers that cannot allocate device memory -- for
 * example a plugin whose host application owns every device allocation, or a runtime
 * that plans all its memory up front and allows no allocation afterwards. The paper
 * has no counterpart; this is a convenience of this library.
 *
 * Same arguments and results as sv_verify, without the workspace: the scratch is one
 * device array inside the library, SV_STATIC_SCRATCH_BYTES long, that every GPU which
 * loads the library holds until the process exits. Shapes whose workspace
 * (sv_workspace_bytes(B, K, V)) exceeds that size return SV_ERR_WORKSPACE without
 * doing anything. The call allocates nothing (no cudaMalloc, no cudaFree).
 *  - The first call on each device also looks up the array's device address (a
 *    host-side runtime query, made with that device current).
 *  - Every call shares the one array and keeps what the previous call left there.
 *    Each call leaves its counters and published words at zero, and the call clears
 *    the array's 256-byte header (an async memset on `stream`) before its kernel.
 *    Calls whose work overlaps on the GPU -- on different streams, or from different
 *    threads -- race on the array and must not be issued; order them on one stream.
 *  - Arguments are checked, as for sv_verify, before anything is enqueued.
 *  - The workspace status word is cleared by every call and is not readable through
 *    this entry point; invalid device data still shows as out_accepted = -1.
 */
#define SV_STATIC_SCRATCH_BYTES (16u << 20)
sv_status sv_verify_static(const void *target_d, const void *draft_d, sv_dtype dtype,
                           const int32_t *draft_tok_d, const int32_t *verify_len_d,
                           const float *uniforms_d, int B, int K, int V, float temperature,
                           int32_t *out_tok_d, int32_t *out_accepted_d, void *stream);

/* Static string for a status code. */
const char *sv_status_string(sv_status s);

/* Library version, as major*10000 + minor*100 + patch. */
int sv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
