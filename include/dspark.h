/*
 * dspark.h -- C ABI of libdspark, the GB300 (sm_103a) draft-sampling hot path of DSpark
 * (confidence-scheduled speculative decoding with semi-autoregressive generation).
 *
 * Sources cited below (page title, section / equation):
 *   [P1] "DSpark -- paper verification": section 1 (Eqs 4-8), section 4 (delta table D7, D8).
 *   [P2] "DSpark: 既要猜得连贯，也要把验证算力花在刀刃上": "设计" (Hardware-aware prefix scheduler).
 *   [P3] "DSpark: Wait It's All Autoregressive?": "A parallel backbone with autoregressive
 *        sampling", "How the Markov sampler works", "Training DSpark" (teacher forcing).
 *   [P4] "Phase-Conditioned Speculative Decoding": section 3 (Eq 7, Eq 8, Theta = tau * SPS).
 *
 * Conventions shared by every call
 *   - Pointers: every array argument is DEVICE memory owned by the caller, C-contiguous, and
 *     16-byte aligned.  The library allocates nothing and keeps no per-call global state; the
 *     only process-wide state is a per-device cache of SM count and occupancy.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Calls are asynchronous: DSPARK_OK means "validated and enqueued".
 *   - Errors: a host-detectable error returns at once with nothing enqueued.  CUDA launch
 *     failures return DSPARK_ERR_CUDA; dspark_last_error() gives the text (thread-local).
 *     Errors found on the device by the draft calls are written to a status word in the
 *     workspace and read back with dspark_get_status().
 *   - dtypes: `wdt` applies to the weights (W1, W2, w, Wj), `udt` to the activations (U, h).
 *     DSPARK_BF16 arrays hold raw bfloat16; fp32 accumulation everywhere.
 *   - Limits: 1 <= gamma <= 16, 2 <= V <= 2^24, r and d multiples of 8 (d may be 0 when the
 *     confidence head is not used), 8 <= r <= 512, T finite and > 0.
 *
 * Layouts (row-major)
 *   W1      [V][r]        embedding table of the sequential head (Eq 5 lookup)
 *   W2      [r][V]        the pages' orientation (DSPARK_W2_RV: W2 in R^{r x V}, B_k = a W2), or
 *           [V][r]        a linear layer's weight (DSPARK_W2_VR: row v holds the r coefficients
 *                         of vocab entry v); the draft calls take either (argument w2_layout):
 *                         B_k[v] = sum_j a_j W2[j][v] = sum_j a_j W2^T[v][j]
 *   Wj      [3r][2r+d]    RNN joint projection, rows [gate; candidate; output], columns
 *                         [s_{k-1}; W1[x_{k-1}]; h_k] (Eq 6, delta table D8); no bias
 *   w       [d+r]         confidence weight: w[0:d] multiplies h_k, w[d:d+r] multiplies
 *                         W1[x_{k-1}] (Eq 7); no bias
 *   U       [B][gamma][V] base logits of the parallel backbone (Eq 4)
 *   h       [B][gamma][d] backbone hidden states
 *   target  [B][gamma][V] fp32 target-model logits (Eq 8), optional
 *   x0      [B]           int32 anchor tokens (the target's last token)
 *
 * Sampling (a reading: the pages only say "sample left to right according to p_k")
 *   p_k = softmax((U_k + B_k) / T).  x_k = argmax_v (y_v + g_v), y = (U_k + B_k) / T,
 *   g_v = -ln(-ln u_v), ties to the smaller v.  u_v = (2*(bits >> 9) + 1) * 2^-24 where bits is
 *   word (v mod 4) of Philox4x32-10 (Salmon et al., SC'11) with key (lo32(seed), hi32(seed))
 *   and counter (floor(v/4), k-1, b, 0x44535052).  The same seed, shapes and inputs give the
 *   same tokens on every run: the cross-block argmax is order-independent and every sum runs in
 *   a fixed order.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSPARK_OK = 0,
  DSPARK_ERR_INVALID = 1,     /* bad argument; on the device: a token or S out of range     */
  DSPARK_ERR_WORKSPACE = 2,   /* workspace NULL, misaligned, or smaller than required        */
  DSPARK_ERR_CUDA = 3,        /* a CUDA runtime call failed; see dspark_last_error()         */
  DSPARK_ERR_TIMEOUT = 4,     /* a device-side wait between thread blocks ran out (device)   */
  DSPARK_ERR_UNSUPPORTED = 5  /* valid arguments that no kernel of the library runs            */
} dspark_status;

typedef enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 } dspark_dtype;

typedef enum { DSPARK_HEAD_MARKOV = 0, DSPARK_HEAD_RNN = 1 } dspark_head;

/* Storage of W2 ("DSpark -- paper verification", section 1, Eq 5: W2 in R^{r x V}).
 * DSPARK_W2_RV: [r][V], the pages' orientation.  DSPARK_W2_VR: [V][r], the weight of a linear
 * layer from r to V.  The tensor-core kernel with the requests on M reads either natively (an
 * MN-major or a K-major operand, the same bytes at the same speed).  The small-batch kernels
 * (B <= 4) read [V][r]: for DSPARK_W2_RV they first transpose W2 into the workspace (one more
 * launch, 2 V r element reads and writes), which the workspace must be sized for
 * (DSPARK_WS_W2_RV). */
typedef enum { DSPARK_W2_VR = 0, DSPARK_W2_RV = 1 } dspark_w2_layout;

/* dspark_workspace_bytes flags */
#define DSPARK_WS_TARGET 1 /* the calls will pass target logits (Eq 8 labels) */
#define DSPARK_WS_W2_RV 2  /* the calls will pass W2 as [r][V] (room for its transpose at B <= 4) */

/*
 * Bytes of workspace the draft calls need for this problem (`flags`: DSPARK_WS_TARGET when
 * target logits will be passed; at B > 4 that reserves room for y, B * V floats; plus
 * DSPARK_WS_W2_RV when W2 will be passed as [r][V]; at B <= 4 that reserves V * r * 4 bytes).  The
 * workspace is caller-owned device memory, 256-byte aligned, that must be ZEROED ONCE before
 * its first use; every
 * successful call leaves it ready for the next call.  One workspace serves one call at a time:
 * calls that share a workspace must be ordered (same stream, or events).  After a call whose
 * device status is not DSPARK_OK, call dspark_get_status() before reusing the workspace.
 * Returns 0 for arguments the draft calls would reject.
 */
size_t dspark_workspace_bytes(int head, int B, int gamma, int V, int r, int d, int flags);

/*
 * One semi-autoregressive draft block with the Markov head [P1 s1 Eq 4, Eq 5, Eq 7, Eq 8;
 * P3 "A parallel backbone with autoregressive sampling"].  For every request b and
 * k = 1..gamma, in one persistent launch:
 *   e = W1[x_{k-1}] (x_0 = x0[b]);  B_k = e . W2^T;  z = U[b][k] + B_k;  y = z / T;
 *   lse_k = log sum_v exp y_v;  x_k = Gumbel-max sample (see above);
 *   c_k = sigmoid(w[0:d] . h[b][k] + w[d:] . e);  S_k = prod_{i<=k} c_i;
 *   c*_k = clamp(1 - 1/2 || softmax(y) - softmax(target[b][k] / T) ||_1, 0, 1)  (Eq 8),
 *   l1_k = || softmax(y) - softmax(target[b][k] / T) ||_1.
 * W2 and U are streamed from HBM once per step.
 *   W2, w2_layout  W2 as [r][V] (DSPARK_W2_RV) or [V][r] (DSPARK_W2_VR), see dspark_w2_layout;
 *            [r][V] on the tensor-core path needs V a multiple of 8 (16-byte rows).
 *
 *   forced   NULL: step k+1 conditions on the sampled x_k.  Otherwise [B][gamma] int32
 *            teacher-forcing tokens: step k+1 conditions on forced[b][k-1] ([P3] "Training
 *            DSpark"); tokens[] still receives each step's own sample.
 *   h, w     both NULL: c and S are not computed (c, S must then be NULL).
 *   target   NULL: cstar and l1 are not computed (cstar, l1 must then be NULL).
 *   outputs  tokens, lse: [B][gamma] (required).  c, S, cstar, l1: [B][gamma] fp32 or NULL.
 *            logits: [B][gamma][V] fp32 copy of z (debugging; NULL in production).
 * Device-side errors: an anchor or forced token outside [0, V) sets DSPARK_ERR_INVALID; that
 * request's tokens become -1 and its floats NaN, other requests are unaffected.  A wait
 * between thread blocks that exceeds about one second sets DSPARK_ERR_TIMEOUT and the launch
 * returns early.  Read either with dspark_get_status().
 */
dspark_status dspark_markov_draft(int B, int gamma, int V, int r, int d, float T, uint64_t seed,
                                  dspark_dtype wdt, const void* W1, const void* W2,
                                  dspark_w2_layout w2_layout, const void* w, dspark_dtype udt,
                                  const void* U, const void* h,
                                  const int32_t* x0, const int32_t* forced, const float* target,
                                  int32_t* tokens, float* lse, float* c, float* S, float* cstar,
                                  float* l1, float* logits, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * The same block with the RNN head [P1 s1 Eq 6; delta table D8]:
 *   z_k = [s_{k-1}; W1[x_{k-1}]; h_k],  (g; c; o) = Wj z_k split in three,
 *   s_k = sigmoid(g) * s_{k-1} + (1 - sigmoid(g)) * tanh(c),  B_k = tanh(o) . W2^T.
 * B_k is built from z_k, i.e. from s_{k-1}.  s0: [B][r] fp32 initial state or NULL for zeros.
 * s_out: [B][r] fp32 final state s_gamma, or NULL.  Eq 7 is unchanged (uses W1[x_{k-1}]).
 * h is required (it feeds Eq 6, d > 0); w may be NULL (then c, S are NULL).  Weights and
 * activations must be bf16 (DSPARK_ERR_UNSUPPORTED otherwise): the h_k columns of the joint
 * projection are computed for all (b, k) up front by a tensor-core GEMM, a second launch on the
 * same stream.  All other arguments, outputs and errors as dspark_markov_draft.
 */
dspark_status dspark_rnn_draft(int B, int gamma, int V, int r, int d, float T, uint64_t seed,
                               dspark_dtype wdt, const void* W1, const void* W2,
                               dspark_w2_layout w2_layout, const void* w, const void* Wj,
                               dspark_dtype udt, const void* U, const void* h,
                               const int32_t* x0, const int32_t* forced, const float* target,
                               const float* s0, int32_t* tokens, float* lse, float* c, float* S,
                               float* cstar, float* l1, float* logits, float* s_out,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Teacher-forced confidence head [P1 s1 Eq 7; P4 s3]: for given tokens,
 *   c_k = sigmoid(w[0:d] . h[b][k] + w[d:] . W1[x_{k-1}]),  S_k = prod_{i<=k} c_i,
 * with x_0 = x0[b] and x_k = tokens[b][k-1].  Outputs c, S: [B][gamma] fp32.  A token outside
 * [0, V) makes c and S NaN from that position on (no status word; no workspace needed).
 */
dspark_status dspark_confidence(int B, int gamma, int V, int r, int d, dspark_dtype wdt,
                                const void* W1, const void* w, dspark_dtype udt, const void* h,
                                const int32_t* x0, const int32_t* tokens, float* c, float* S,
                                void* stream);

/*
 * Soft acceptance label on N independent rows [P1 s1 Eq 8, D7; P4 s3]:
 *   l1 = || softmax(draft/T) - softmax(target/T) ||_1,  cstar = clamp(1 - l1/2, 0, 1),
 * the acceptance probability of the standard speculative accept/reject rule.
 * draft_logits, target_logits: [N][V] fp32.  cstar, l1: [N] fp32 (l1 may be NULL).
 */
dspark_status dspark_tv_label(int N, int V, float T, const float* draft_logits,
                              const float* target_logits, float* cstar, float* l1, void* stream);

/*
 * Hardware-aware prefix scheduler [P2 "设计"; P4 s3 Theta = tau * SPS(B)].  Picks each
 * request's verify length len[b] in 0..gamma to maximise
 *   Theta = sps[n] * sum_b (1 + sum_{k <= len[b]} S[b][k]),  n = sum_b (len[b] + 1),
 * over legal (contiguous-prefix) choices: steps/s at n verify tokens times expected tokens per
 * step.  Ties go to fewer tokens.  S: [B][gamma] fp32 prefix survival (each row in [0, 1] and
 * non-increasing); sps: [B*(gamma+1)+1] fp64 steps/s table indexed by n.  Outputs len [B] int32,
 * theta [1] fp64.  Sums of S are exact (2^-32 fixed point); the result is bit-identical to the
 * CPU reference.  B * gamma <= 16384.  Invalid S on the device: every len[b] = -1, theta NaN.
 */
dspark_status dspark_prefix_schedule(int B, int gamma, const float* S, const double* sps,
                                     int32_t* len, double* theta, void* stream);

/*
 * Speculative verification of one draft block per request: the standard accept/reject rule,
 * whose single-step acceptance probability is Eq 8's c* [P4 s3; Leviathan, Kalman, Matias,
 * ICML 2023], with the round [P2 "Why DSpark?"] stopping at the first rejection and the target
 * adding a bonus token [P2 "Results"].  For request b, p_j = softmax(draft_logits[b][j] / T),
 * q_j = softmax(target_logits[b][j] / T):
 *   position j = 0, 1, ... accepts draft_tokens[b][j] iff ln a_j < ln q_j(x_j) - ln p_j(x_j)
 *   (probability min(1, q_j(x_j) / p_j(x_j))); at the first rejection j the correction is a
 *   Gumbel-max draw from max(0, q_j - p_j) (from q_j if that is zero everywhere); after gamma
 *   acceptances the bonus is a draw from q_gamma.
 *   a_j: word 0 of Philox4x32-10 at counter (0, j, b, 0x41434350) with the sampler's key and
 *   uniform; the draw's noise for entry v: word v mod 4 at counter (v / 4, j, b, 0x52455344).
 *   Draws are Gumbel-max in fp32 (ties to the smaller entry), like the draft sampler.
 * Arguments (device pointers, row-major, caller-owned):
 *   draft_logits   [B][gamma][V] fp32 draft logits z (the draft call's `logits` output)
 *   target_logits  [B][gamma+1][V] fp32 target logits; row gamma feeds the bonus
 *   draft_tokens   [B][gamma] int32
 *   n_accepted     [B] int32 out: accepted drafted tokens, 0..gamma (-1 for an invalid request)
 *   out_tokens     [B][gamma+1] int32 out: the accepted prefix, then the correction or bonus,
 *                  then -1
 *   workspace      dspark_verify_workspace_bytes(B, gamma, V) bytes, 256-byte aligned, zeroed
 *                  once before the first call; every call leaves it ready for the next
 * Limits: 1 <= gamma <= 16, 2 <= V <= 2^24, T finite and > 0.  Three launches on `stream`.
 * A drafted token outside [0, V) gives that request n_accepted = -1 and out_tokens -1, and sets
 * DSPARK_ERR_INVALID in the workspace status (read with dspark_get_status).
 */
size_t dspark_verify_workspace_bytes(int B, int gamma, int V);
dspark_status dspark_verify(int B, int gamma, int V, float T, uint64_t seed,
                            const float* draft_logits, const float* target_logits,
                            const int32_t* draft_tokens, int32_t* n_accepted, int32_t* out_tokens,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * The drafter's training losses and their gradients [P1 s1 Eqs 9-12; delta table D3-D7], for
 * teacher-forced draft logits.  For request b and position k = 1..gamma (row j = k - 1):
 *   p_k = softmax(draft_logits[b][j] / T), q_k = softmax(target_logits[b][j] / T) (frozen),
 *   x*_k = labels[b][j], c_k = sigmoid(conf_logits[b][j]), w_k = exp(-(k - 1) / gamma);
 *   L_ce = -sum_k w_k ln p_k(x*_k)  (Eq 9);  L_tv = sum_k w_k ||p_k - q_k||_1  (Eq 10);
 *   c*_k = clamp(1 - 1/2 ||p_k - q_k||_1, 0, 1)  (Eq 8);
 *   L_conf = -sum_k w_k [c*_k ln c_k + (1 - c*_k) ln(1 - c_k)]  (Eq 11);
 *   L = alpha_ce L_ce + alpha_tv L_tv + alpha_conf L_conf  (Eq 12; defaults 0.1, 0.9, 1.0).
 * c* is a label (no gradient through it):
 *   grad_logits[b][j][v] = (w_k / T) (alpha_ce (p_v - [v == x*]) + alpha_tv p_v (s_v - sum_u s_u p_u)),
 *   s_u = sign(p_u - q_u);  grad_conf[b][j] = alpha_conf w_k (c_k - c*_k).
 * Arguments (device pointers, row-major, caller-owned): draft_logits, target_logits
 * [B][gamma][V] fp32 (16-byte aligned); labels [B][gamma] int32; conf_logits [B][gamma] fp32.
 * Outputs, each optional (NULL skips it, at least one given): loss [B], parts [B][3]
 * (L_ce, L_tv, L_conf), grad_logits [B][gamma][V] (16-byte aligned), grad_conf [B][gamma], all
 * fp32.  workspace: dspark_draft_loss_workspace_bytes(B, gamma, V) bytes, 256-byte aligned
 * (contents need not be zero).  Limits: 1 <= gamma <= 16, 2 <= V <= 2^24, T finite and > 0.
 * A label outside [0, V) makes every output of its request NaN and sets DSPARK_ERR_INVALID in
 * the workspace status.  Three launches on `stream`, four with grad_logits
 * (dspark_draft_loss_launches).
 */
size_t dspark_draft_loss_workspace_bytes(int B, int gamma, int V);
dspark_status dspark_draft_loss(int B, int gamma, int V, float T, const float* draft_logits,
                                const float* target_logits, const int32_t* labels,
                                const float* conf_logits, float alpha_ce, float alpha_tv,
                                float alpha_conf, float* loss, float* parts, float* grad_logits,
                                float* grad_conf, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * Sequential temperature scaling of the confidence head [P4 s3: calibration that minimises the
 * expected calibration error of the cumulative product, one position at a time; P1 delta
 * table D13: a left-to-right 1-D grid search with the prefix held fixed].  N calibration blocks
 * with confidence logits conf_logits [N][gamma] fp32 and accepted lengths accepted [N] int32
 * (0..gamma, e.g. dspark_verify's n_accepted); a temperature grid [ngrid] fp32 (> 0).  For
 * k = 1..gamma, with tau_1..tau_{k-1} already chosen:
 *   S_k[n](t) = prod_{i<k} sigmoid(conf[n][i-1] / tau_i) * sigmoid(conf[n][k-1] / t),
 *   y_k[n] = [accepted[n] >= k],
 *   ECE_k(t) = sum_m |sum_{n in bin m} (S_k[n](t) - y_k[n])| / N,  bin(s) = min(bins-1, floor(s bins))
 *   (the standard equal-width-bin ECE; the page's own formula is garbled),
 *   tau_k = the first grid entry with the smallest ECE_k.
 * Outputs: tau [gamma], ece [gamma] (ECE_k at tau_k), ece_grid [gamma][ngrid] (every ECE_k(t))
 * or NULL; fp32.  Limits: 1 <= gamma <= 16, 1 <= ngrid <= 4096, 1 <= bins <= 64.  workspace:
 * dspark_sts_workspace_bytes(N, gamma, ngrid, bins) bytes, 256-byte aligned.  An accepted
 * length outside [0, gamma] or a grid entry <= 0 sets DSPARK_ERR_INVALID in the workspace
 * status.  Deterministic (fixed reduction order).  2 * gamma launches on `stream`.
 */
size_t dspark_sts_workspace_bytes(int N, int gamma, int ngrid, int bins);
dspark_status dspark_sts(int N, int gamma, const float* conf_logits, const int32_t* accepted,
                         int ngrid, const float* grid, int bins, float* tau, float* ece,
                         float* ece_grid, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The Markov draft of dspark_markov_draft for callers that cannot allocate device memory.  The
 * paper has no counterpart: this is a deployment variant of the same computation.  Callers such
 * as plugins inside another framework's memory pool, serving engines that forbid allocation on
 * their decode path, or code handed only pre-allocated input and output buffers cannot create a
 * workspace; this call keeps the draft's scratch in a 1 MiB array built into the library, which
 * every GPU that loads the library holds until the process exits.
 *   - Arguments and outputs are those of dspark_markov_draft, minus the workspace and the W2
 *     layout: W2 is [V][r] here (the [r][V] form needs a transposed copy the array cannot hold).
 *   - status: optional device int32 that receives this call's device status (DSPARK_OK, or the
 *     DSPARK_ERR_INVALID / DSPARK_ERR_TIMEOUT cases described for dspark_markov_draft), written on
 *     `stream` after the draft; NULL to skip.  It is written only when the call returns
 *     DSPARK_OK: a call rejected on the host leaves it untouched, so check the return code
 *     before reading it.
 *   - Limit: problems whose dspark_workspace_bytes(0, B, gamma, V, r, d, flags) exceeds 1 MiB are
 *     rejected with DSPARK_ERR_WORKSPACE (in practice the small-batch path, B <= 4).
 *   - The first call on each device looks up the array's device address (once per device, with
 *     that device current); make that first call before any stream capture.  The address is
 *     kept for the life of the process: after cudaDeviceReset on a device, this entry point must
 *     not be called on that device again in the same process.
 *   - Allocates nothing: each call clears the part of the array it uses (the array keeps the
 *     previous call's contents) and enqueues the draft.  All calls on a device share the one
 *     array, so calls that overlap on the GPU (different streams without ordering) race.
 */
dspark_status dspark_markov_draft_noalloc(int B, int gamma, int V, int r, int d, float T,
                                          uint64_t seed, dspark_dtype wdt, const void* W1,
                                          const void* W2, const void* w, dspark_dtype udt,
                                          const void* U, const void* h, const int32_t* x0,
                                          const int32_t* forced, const float* target,
                                          int32_t* tokens, float* lse, float* c, float* S,
                                          float* cstar, float* l1, float* logits, int32_t* status,
                                          void* stream);

/*
 * Synchronises `stream`, returns the device status word of `workspace` (the most severe error
 * any draft call recorded since the last read, DSPARK_OK if none) and resets the workspace so
 * the next call starts clean.  DSPARK_ERR_CUDA if the synchronisation itself fails.
 */
dspark_status dspark_get_status(void* workspace, size_t workspace_bytes, void* stream);

/* Text of the last host-side error on the calling thread ("" if none). */
const char* dspark_last_error(void);

/*
 * Which kernel path a draft call with these arguments takes on the current device:
 *   0 = CUDA-core dot products (B <= 4; fp32 weights, or bf16 ranks the next one cannot take),
 *   1 = tensor cores with the requests on the MMA's M dimension (bf16, any B),
 *   2 = tensor cores with the vocabulary rows on M and the B <= 4 conditioning vectors on N
 *       (bf16, r a multiple of 64 up to 256, at most 4096 vocabulary rows per SM).
 * By default 2 when it can run the arguments and B >= 3, else the first of 0, 2, 1 that can
 * (on GB300 the B <= 4 tensor-core MMA, N = 16, costs about as much as a full-width one, so it
 * overtakes the CUDA cores only from B = 3).  The environment variable
 * DSPARK_DRAFT_PATH = cuda-core | tensor | tensor-vocab, read at every call, forces one (a draft
 * call then fails with DSPARK_ERR_UNSUPPORTED if that one cannot run the arguments; other
 * values are ignored).  Negative for arguments it would reject.
 */
int dspark_draft_path(int head, int B, int V, int r, dspark_dtype wdt);

/*
 * Blocks per thread-block cluster of the draft kernel paths 0 and 2 use on the current device
 * (1 = no clusters; path 1 always 1).  Those kernels run one block per SM; the blocks of a
 * cluster merge their per-step argmax keys and (max, sum-exp) partials in distributed shared
 * memory, and one block per cluster publishes the merged result to the other clusters.
 * Clusters are used only when DSPARK_CLUSTER = 2 | 4 | 8 (read at every call) asks for them: a
 * draft call then fails with DSPARK_ERR_UNSUPPORTED if clusters of that size cannot all be
 * resident at once, one block per SM (clusters must fit inside one GPC); other values, or
 * none, mean no clusters.  On GB300 only 2-block clusters tile the 152 SMs, and there the extra
 * hop per step costs more than the halved merge saves, hence the default.  Negative for
 * arguments a draft call would reject, or without a device.
 */
int dspark_draft_cluster(int head, int B, int V, int r, dspark_dtype wdt);

/* Number of kernel launches one draft call with these arguments makes on its stream, without a
 * target (on path 1 a target adds one: its normalisers are formed by a streaming launch before
 * the draft). */
int dspark_draft_launches(int head, int B, int V, int r, dspark_dtype wdt);

/* Number of kernel launches one dspark_draft_loss call makes on its stream (with_grad: whether
 * grad_logits is given).  Negative for arguments it would reject. */
int dspark_draft_loss_launches(int B, int gamma, int V, int with_grad);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
