// dspark_oracle.cpp -- plain, slow, fp64 CPU oracle of the DSpark draft-sampling path.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, import or call this file;
// only the tests, the smoke check and the benchmark's CPU-baseline leg use it.  It shares no
// code, header, table or helper with the CUDA library: it is written from the equations on the
// pages below, in their order and notation, with no blocking, fusion or reordering beyond what
// the definitions state.  Every quantity is computed in IEEE double.
//
// Sources (page title, section / equation):
//   [P1] "DSpark -- paper verification", section 1 (Eqs 4-8), section 4 (delta table D7, D8).
//   [P2] "DSpark: 既要猜得连贯，也要把验证算力花在刀刃上", "设计" (scheduler prose), "Results".
//   [P3] "DSpark: Wait It's All Autoregressive?", "A parallel backbone with autoregressive
//        sampling" and "How the Markov sampler works".
//   [P4] "Phase-Conditioned Speculative Decoding", sections 3 and 6 (Eq 7, Eq 8, Theta = tau*SPS),
//        and its reference to Leviathan, Kalman, Matias (ICML 2023) for the accept/reject rule.
//
// Readings taken where the pages are silent (each is listed in the design notes):
//   * Temperature: p_k = softmax((U_k + B_k) / T); Eq 4 itself has no temperature.
//   * Sampler: "sample left to right according to p_k" is realised as Gumbel-max,
//     x_k = argmax_v (y_v + g_v), g_v = -ln(-ln u_v), ties to the smaller v.  u_v comes from
//     Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) with key (lo32(seed), hi32(seed)) and
//     counter (floor(v/4), k-1, b, 0x44535052); the word used is lane v mod 4, and
//     u = (2*(bits >> 9) + 1) * 2^-24, which lies strictly inside (0, 1).
//   * Storage: W1 is [V][r] (an embedding table), W2 is stored as the [V][r] weight of the
//     logit projection (row v holds the r coefficients of vocab entry v), so
//     B_k[v] = sum_j e_j * W2[v][j].  The RNN joint projection Wj is [3r][2r+d] with rows
//     [gate; candidate; output] and columns [s_{k-1}; W1[x_{k-1}]; h_k]; no biases.
//   * Eq 7 has no bias; w[0:d] multiplies h_k and w[d:d+r] multiplies W1[x_{k-1}], also for
//     the RNN head.
//   * Eq 8 is clamped to [0, 1] (delta table D7); the target distribution uses the same T.
//   * Verify (the standard speculative accept/reject rule that [P4 s3] equates with Eq 8, and the
//     round [P2 "Why DSpark?"] describes: accept the matching prefix, stop at the first
//     rejection; accepted length counts the target's bonus token [P2 "Results"]): position j
//     (0-based) accepts x_j iff ln a_j < ln q_j(x_j) - ln p_j(x_j), with a_j = word 0 of Philox
//     counter (0, j, b, 0x41434350) as above; at the first rejection j the correction is a
//     Gumbel-max sample of max(0, q_j - p_j) (of q_j if that is zero everywhere), and after
//     gamma acceptances the bonus is a Gumbel-max sample of q_gamma; both draw u_v from Philox
//     counter (floor(v/4), j, b, 0x52455344).
//   * Training losses (Eqs 9-12 [P1 s1]): p_k = softmax(zd_k / T), q_k = softmax(zt_k / T),
//     w_k = exp(-(k-1)/gamma); c*_k (Eq 8) is a label in L_conf: no gradient flows through it,
//     and the target logits are frozen [P1 s1, "the target is frozen throughout"].  The losses
//     are sums over positions (no division by sum w_k).
//   * STS calibration ([P4 s3] "sequential temperature scaling that minimises expected
//     calibration error of the cumulative product, one position at a time"; [P1 delta table
//     D13] "left-to-right 1-D grid search on the cumulative product, prefix held fixed"; the
//     ECE formula there is garbled): the standard equal-width-bin ECE with M bins,
//     ECE = sum_m |sum_{n in bin m} (S_n - y_n)| / N, bin = min(M - 1, floor(S M)); the
//     survival label of position k is y = [accepted length >= k]; the temperature grid is
//     given by the caller and ties go to the first grid entry.
//   * Scheduler (Algorithm 1 is named, not printed): choose per-request verify lengths l_b in
//     0..gamma maximising Theta = SPS(n) * sum_b (1 + sum_{k<=l_b} S_{b,k}) with
//     n = sum_b (l_b + 1); only contiguous prefixes are legal; ties go to fewer tokens.
//
// Parity pins live in tests/ (brute-force block distribution, Philox against an independent
// library implementation, closed forms of Eq 8, invariants of S_k, scheduler brute force and
// the tau(a, gamma) closed form).  Nothing here is "parity unpinned" except the two tie-break
// conventions the pages never state (the Gumbel counter packing and the scheduler's tie rule),
// which are conventions rather than results.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum { DT_F32 = 0, DT_BF16 = 1, DT_F64 = 2 };

// Read element i of an array stored as fp32, bf16 (raw 16-bit pattern) or fp64.
double load(const void* p, int dt, size_t i) {
  if (dt == DT_F32) return (double)((const float*)p)[i];
  if (dt == DT_BF16) {
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    std::memcpy(&f, &bits, 4);
    return (double)f;
  }
  return ((const double*)p)[i];
}

// Philox4x32 with 10 rounds, from the round function of Salmon et al. (SC'11):
// two 32x32->64 multiplications by the round multipliers, the high halves xor-ed with the
// other two counter words and the round key, and a Weyl-sequence key schedule.
void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)x0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    x0 = hi1 ^ x1 ^ k0;
    x1 = lo1;
    x2 = hi0 ^ x3 ^ k1;
    x3 = lo0;
    k0 += 0x9E3779B9u;  // golden-ratio Weyl increment
    k1 += 0xBB67AE85u;  // sqrt(3) - 1 Weyl increment
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

const uint32_t kNoiseTag = 0x44535052u;  // "DSPR"

// u_v in (0, 1) for request b, draft position k (1-based) and vocab entry v.
double uniform(uint64_t seed, int b, int k, int64_t v) {
  const uint32_t ctr[4] = {(uint32_t)(v >> 2), (uint32_t)(k - 1), (uint32_t)b, kNoiseTag};
  const uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  const uint32_t bits = out[v & 3];
  return (2.0 * (double)(bits >> 9) + 1.0) * std::ldexp(1.0, -24);
}

double gumbel(uint64_t seed, int b, int k, int64_t v) {
  return -std::log(-std::log(uniform(seed, b, k, v)));
}

const uint32_t kAcceptTag = 0x41434350u;    // "ACCP": acceptance uniforms of the verify rule
const uint32_t kResidualTag = 0x52455344u;  // "RESD": noise of the correction / bonus sample

// (2 * (bits >> 9) + 1) * 2^-24 for word `lane` of Philox(counter, key(seed)).
double uniform_ctr(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, int lane) {
  const uint32_t ctr[4] = {c0, c1, c2, c3};
  const uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  return (2.0 * (double)(out[lane] >> 9) + 1.0) * std::ldexp(1.0, -24);
}

double sigmoid(double x) { return 1.0 / (1.0 + std::exp(-x)); }

// log sum_v exp(y_v), with the usual max shift.
double logsumexp(const std::vector<double>& y) {
  double m = -INFINITY;
  for (double v : y) m = std::max(m, v);
  double s = 0.0;
  for (double v : y) s += std::exp(v - m);
  return m + std::log(s);
}

// Eq 8: c* = 1 - 1/2 ||p - q||_1 with p = softmax(y), q = softmax(tau); clamped to [0, 1].
void tv_label_row(const std::vector<double>& y, const std::vector<double>& tau, double* cstar,
                  double* l1) {
  const double Ld = logsumexp(y), Lt = logsumexp(tau);
  double acc = 0.0;
  for (size_t v = 0; v < y.size(); ++v) acc += std::fabs(std::exp(y[v] - Ld) - std::exp(tau[v] - Lt));
  *l1 = acc;
  *cstar = std::min(1.0, std::max(0.0, 1.0 - 0.5 * acc));
}

}  // namespace

extern "C" {

void orc_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  philox4x32_10(ctr, key, out);
}

double orc_uniform(uint64_t seed, int b, int k, int64_t v) { return uniform(seed, b, k, v); }

double orc_gumbel(uint64_t seed, int b, int k, int64_t v) { return gumbel(seed, b, k, v); }

// One semi-autoregressive draft block per selected request [P1 s1 Eq 4; P3 "A parallel
// backbone with autoregressive sampling"].  head = 0: Markov head, Eq 5.  head = 1: RNN head,
// Eq 6.  For each request b (rows[i], or i when rows is NULL) and k = 1..gamma:
//   e      = W1[x_{k-1}]                                   (x_0 = anchor, Eq 5 lookup)
//   a      = e                                             (Markov, Eq 5)
//          | tanh(W_o z_k), z_k = [s_{k-1}; e; h_k]        (RNN, Eq 6; s_0 = s0 or 0)
//   B_k[v] = sum_j a_j W2[v][j]                            (Eq 5 / Eq 6 bias)
//   z_v    = U[b][k][v] + B_k[v]                           (Eq 4 logits)
//   y_v    = z_v / T; lse = log sum exp y; p_v = exp(y_v - lse)
//   x_k    = argmax_v (y_v + g_v)                          (Gumbel-max sample of p_k)
//   c_k    = sigmoid(w[0:d].h_k + w[d:].e)                 (Eq 7), S_k = prod_{i<=k} c_i
//   c*_k   = clamp(1 - 1/2 ||p - softmax(t/T)||_1, 0, 1)   (Eq 8, when target != NULL)
// The conditioning token for step k+1 is forced[b][k] when forced != NULL (teacher forcing),
// else the sampled x_k.  Outputs are indexed [i][k-1] over the selected rows; best/best2 are the
// winning and runner-up perturbed scores y + g, tok/tok2 their vocab ids.  z_out, when given,
// receives z_v (before the temperature) as [i][k-1][v].  s_out receives s_gamma as [i][r].
// Returns 0, or 1 if an anchor or forced token lies outside [0, V).
int orc_draft(int head, int B, int gamma, int V, int r, int d, double T, uint64_t seed, int wdt,
              const void* W1, const void* W2, const void* Wj, int udt, const void* U,
              const int32_t* x0, const void* h, const void* w, const float* target,
              const double* s0, const int32_t* forced, const int32_t* rows, int nrows,
              int32_t* tok, double* best, int32_t* tok2, double* best2, double* lse, double* c,
              double* S, double* cstar, double* l1, double* z_out, double* s_out, int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
  const int n = rows ? nrows : B;
  const bool par_rows = n >= 4 * std::max(1, nthreads);  // small V, many rows: split rows
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) if (par_rows) reduction(| : bad)
  for (int i = 0; i < n; ++i) {
    const int b = rows ? rows[i] : i;
    std::vector<double> e(r), a(r), s(r, 0.0), s_next(r), y(V), tau, gsc(V), zin, u;
    if (head == 1 && s0)
      for (int j = 0; j < r; ++j) s[j] = s0[(size_t)b * r + j];
    if (target) tau.resize(V);
    double surv = 1.0;
    int prev = x0[b];
    for (int k = 1; k <= gamma; ++k) {
      const size_t bk = (size_t)b * gamma + (k - 1);
      const size_t out = (size_t)i * gamma + (k - 1);
      if (prev < 0 || prev >= V) {
        bad = 1;
        tok[out] = -1;
        continue;
      }
      for (int j = 0; j < r; ++j) e[j] = load(W1, wdt, (size_t)prev * r + j);

      if (head == 0) {
        a = e;
      } else {
        // Eq 6: z_k = [s_{k-1}; W1[x_{k-1}]; h_k]; one joint projection split in three.
        const int width = 2 * r + d;
        zin.assign(width, 0.0);
        for (int j = 0; j < r; ++j) zin[j] = s[j];
        for (int j = 0; j < r; ++j) zin[r + j] = e[j];
        for (int j = 0; j < d; ++j) zin[2 * r + j] = load(h, udt, bk * d + j);
        u.assign(3 * r, 0.0);
        for (int row = 0; row < 3 * r; ++row) {
          double acc = 0.0;
          for (int m = 0; m < width; ++m) acc += load(Wj, wdt, (size_t)row * width + m) * zin[m];
          u[row] = acc;
        }
        for (int j = 0; j < r; ++j) {
          const double gate = sigmoid(u[j]);
          const double cand = std::tanh(u[r + j]);
          s_next[j] = gate * s[j] + (1.0 - gate) * cand;
          a[j] = std::tanh(u[2 * r + j]);  // B_k uses W_o z_k, with z_k built from s_{k-1}
        }
      }

      // Eq 5 / Eq 6 bias, Eq 4 logits, temperature.
#pragma omp parallel for schedule(static) if (!par_rows)
      for (int v = 0; v < V; ++v) {
        double bias = 0.0;
        for (int j = 0; j < r; ++j) bias += a[j] * load(W2, wdt, (size_t)v * r + j);
        const double z = load(U, udt, bk * V + v) + bias;
        if (z_out) z_out[out * V + v] = z;
        y[v] = z / T;
        gsc[v] = y[v] + gumbel(seed, b, k, v);
        if (target) tau[v] = (double)target[bk * V + v] / T;
      }

      lse[out] = logsumexp(y);
      int t1 = 0, t2 = -1;
      for (int v = 1; v < V; ++v)
        if (gsc[v] > gsc[t1]) t1 = v;
      for (int v = 0; v < V; ++v)
        if (v != t1 && (t2 < 0 || gsc[v] > gsc[t2])) t2 = v;
      tok[out] = t1;
      best[out] = gsc[t1];
      tok2[out] = t2;
      best2[out] = t2 >= 0 ? gsc[t2] : -INFINITY;

      if (h && w) {  // Eq 7 and the prefix survival S_k = prod c_i
        double logit = 0.0;
        for (int j = 0; j < d; ++j) logit += load(w, wdt, j) * load(h, udt, bk * d + j);
        for (int j = 0; j < r; ++j) logit += load(w, wdt, (size_t)d + j) * e[j];
        c[out] = sigmoid(logit);
        surv *= c[out];
        S[out] = surv;
      }
      if (target) tv_label_row(y, tau, &cstar[out], &l1[out]);

      if (head == 1) s = s_next;
      prev = forced ? forced[bk] : t1;
    }
    if (head == 1 && s_out)
      for (int j = 0; j < r; ++j) s_out[(size_t)i * r + j] = s[j];
  }
  return bad;
}

// Eq 7 with teacher forcing: c_k = sigmoid(w[0:d].h_k + w[d:].W1[x_{k-1}]), S_k = prod c_i,
// where x_0 = x0[b] and x_{k} = tokens[b][k-1].  Returns 1 if a token is outside [0, V).
int orc_confidence(int B, int gamma, int V, int r, int d, int wdt, const void* W1, int udt,
                   const void* h, const void* w, const int32_t* x0, const int32_t* tokens,
                   double* c, double* S) {
  int bad = 0;
  for (int b = 0; b < B; ++b) {
    double surv = 1.0;
    for (int k = 1; k <= gamma; ++k) {
      const size_t bk = (size_t)b * gamma + (k - 1);
      const int prev = k == 1 ? x0[b] : tokens[bk - 1];
      if (prev < 0 || prev >= V) {
        bad = 1;
        c[bk] = S[bk] = NAN;
        continue;
      }
      double logit = 0.0;
      for (int j = 0; j < d; ++j) logit += load(w, wdt, j) * load(h, udt, bk * d + j);
      for (int j = 0; j < r; ++j) logit += load(w, wdt, (size_t)d + j) * load(W1, wdt, (size_t)prev * r + j);
      c[bk] = sigmoid(logit);
      surv *= c[bk];
      S[bk] = surv;
    }
  }
  return bad;
}

// Eq 8 on N independent rows: c* = clamp(1 - 1/2 ||softmax(draft/T) - softmax(target/T)||_1).
void orc_tv_label(int N, int V, double T, const float* draft, const float* target, double* cstar,
                  double* l1, int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < N; ++i) {
    std::vector<double> y(V), tau(V);
    for (int v = 0; v < V; ++v) {
      y[v] = (double)draft[(size_t)i * V + v] / T;
      tau[v] = (double)target[(size_t)i * V + v] / T;
    }
    tv_label_row(y, tau, &cstar[i], &l1[i]);
  }
}

// Speculative verification of one draft block per request: the standard accept/reject rule
// [P4 s3: c* = 1 - TV is its single-step acceptance probability; P2 "Why DSpark?": the
// matching prefix is accepted and the round stops at the first rejection; P2 "Results": the
// target contributes a bonus token].  For request b, with p_j = softmax(zd[b][j] / T) (draft,
// j = 0..gamma-1) and q_j = softmax(zt[b][j] / T) (target, j = 0..gamma):
//   for j = 0, 1, ...: accept x_j = tok[b][j] iff ln a_j < ln q_j(x_j) - ln p_j(x_j)
//   (a_j uniform, i.e. with probability min(1, q_j(x_j) / p_j(x_j)));
//   at the first rejection j: n = j, and the correction is drawn from max(0, q_j - p_j)
//   (normalised; from q_j when that is zero everywhere);
//   if all gamma are accepted: n = gamma, and the bonus is drawn from q_gamma.
// Both draws are Gumbel-max: argmax_v (ln w_v + g_v) over the entries with w_v > 0, ties to the
// smaller v.  Outputs: n_acc[b] = n; out[b][0..n-1] = the accepted tokens, out[b][n] = the
// correction or bonus, out[b][n+1..gamma] = -1.  margin[b][j] = (ln q - ln p)(x_j) - ln a_j for
// the positions tested (NaN after n); best/best2/tok2 are the winning and runner-up perturbed
// scores of the draw and the runner-up's id.  Returns 1 (and n_acc = -1) for a request with a
// drafted token outside [0, V).
int orc_verify(int B, int gamma, int V, double T, uint64_t seed, const float* zd,
               const float* zt, const int32_t* tok, int32_t* n_acc, int32_t* out,
               double* margin, double* best, double* best2, int32_t* tok2, int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
  for (int b = 0; b < B; ++b) {
    std::vector<double> y(V), tau(V), w(V);
    for (int j = 0; j <= gamma; ++j) out[(size_t)b * (gamma + 1) + j] = -1;
    for (int j = 0; j < gamma; ++j) margin[(size_t)b * gamma + j] = NAN;
    bool ok = true;
    for (int j = 0; j < gamma; ++j) ok = ok && tok[(size_t)b * gamma + j] >= 0 && tok[(size_t)b * gamma + j] < V;
    if (!ok) {
      bad = 1;
      n_acc[b] = -1;
      best[b] = best2[b] = NAN;
      tok2[b] = -1;
      continue;
    }
    int n = gamma;
    for (int j = 0; j < gamma; ++j) {
      const size_t dj = ((size_t)b * gamma + j) * V, tj = ((size_t)b * (gamma + 1) + j) * V;
      for (int v = 0; v < V; ++v) {
        y[v] = (double)zd[dj + v] / T;
        tau[v] = (double)zt[tj + v] / T;
      }
      const double Ld = logsumexp(y), Lt = logsumexp(tau);
      const int x = tok[(size_t)b * gamma + j];
      const double log_ratio = (tau[x] - Lt) - (y[x] - Ld);  // ln q_j(x) - ln p_j(x)
      const double a = uniform_ctr(seed, 0u, (uint32_t)j, (uint32_t)b, kAcceptTag, 0);
      margin[(size_t)b * gamma + j] = log_ratio - std::log(a);
      out[(size_t)b * (gamma + 1) + j] = x;
      if (!(std::log(a) < log_ratio)) {  // rejected: the correction replaces x_j
        n = j;
        bool any = false;
        for (int v = 0; v < V; ++v) {
          w[v] = std::max(0.0, std::exp(tau[v] - Lt) - std::exp(y[v] - Ld));
          any = any || w[v] > 0.0;
        }
        if (!any)
          for (int v = 0; v < V; ++v) w[v] = std::exp(tau[v] - Lt);
        break;
      }
    }
    if (n == gamma) {  // every drafted token accepted: the bonus from q_gamma
      const size_t tj = ((size_t)b * (gamma + 1) + gamma) * V;
      for (int v = 0; v < V; ++v) tau[v] = (double)zt[tj + v] / T;
      const double Lt = logsumexp(tau);
      for (int v = 0; v < V; ++v) w[v] = std::exp(tau[v] - Lt);
    }
    int t1 = -1, t2 = -1;
    double s1 = -INFINITY, s2 = -INFINITY;
    for (int v = 0; v < V; ++v) {
      if (!(w[v] > 0.0)) continue;
      const double u = uniform_ctr(seed, (uint32_t)(v >> 2), (uint32_t)n, (uint32_t)b, kResidualTag, v & 3);
      const double sc = std::log(w[v]) - std::log(-std::log(u));
      if (sc > s1) {
        t2 = t1;
        s2 = s1;
        t1 = v;
        s1 = sc;
      } else if (sc > s2) {
        t2 = v;
        s2 = sc;
      }
    }
    n_acc[b] = n;
    out[(size_t)b * (gamma + 1) + n] = t1;
    best[b] = s1;
    best2[b] = s2;
    tok2[b] = t2;
  }
  return bad;
}

// Training losses of one draft block per request [P1 s1 Eqs 9-12; delta table D3-D7].  For
// request b and k = 1..gamma (row j = k - 1), p_k = softmax(zd[b][j] / T) (draft),
// q_k = softmax(zt[b][j] / T) (frozen target), x*_k = labels[b][j], c_k = sigmoid(conf[b][j]):
//   w_k    = exp(-(k - 1) / gamma)
//   L_ce   = -sum_k w_k ln p_k(x*_k)                                             (Eq 9)
//   L_tv   =  sum_k w_k ||p_k - q_k||_1                                           (Eq 10)
//   c*_k   =  clamp(1 - 1/2 ||p_k - q_k||_1, 0, 1)                                (Eq 8)
//   L_conf = -sum_k w_k [c*_k ln c_k + (1 - c*_k) ln(1 - c_k)]                    (Eq 11)
//   L      =  a_ce L_ce + a_tv L_tv + a_conf L_conf                               (Eq 12)
// and the gradients with c* held as a label:
//   dL/dzd[b][j][v] = (w_k / T) (a_ce (p_v - [v == x*]) + a_tv p_v (s_v - sum_u s_u p_u)),
//                     s_u = sign(p_u - q_u) (0 where they are equal)
//   dL/dconf[b][j]  = a_conf w_k (c_k - c*_k).
// loss[b] = L; parts[b] = (L_ce, L_tv, L_conf); grad_z [B][gamma][V] and grad_c [B][gamma] may
// be NULL.  Returns 1 when a label lies outside [0, V); every output of that request is NaN.
int orc_draft_loss(int B, int gamma, int V, double T, const float* zd, const float* zt,
                   const int32_t* labels, const float* conf, double a_ce, double a_tv,
                   double a_conf, double* loss, double* parts, double* grad_z, double* grad_c,
                   int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int b = 0; b < B; ++b) {
    std::vector<double> y(V), tau(V), p(V), q(V);
    double Lce = 0.0, Ltv = 0.0, Lconf = 0.0;
    bool ok = true;
    for (int j = 0; j < gamma; ++j) {
      const int x = labels[(size_t)b * gamma + j];
      ok = ok && x >= 0 && x < V;
    }
    if (!ok) {  // every output of the request is NaN
      bad = 1;
      loss[b] = NAN;
      if (parts) parts[3 * (size_t)b] = parts[3 * (size_t)b + 1] = parts[3 * (size_t)b + 2] = NAN;
      for (int j = 0; j < gamma; ++j) {
        if (grad_c) grad_c[(size_t)b * gamma + j] = NAN;
        if (grad_z)
          for (int v = 0; v < V; ++v) grad_z[((size_t)b * gamma + j) * V + v] = NAN;
      }
      continue;
    }
    for (int j = 0; j < gamma; ++j) {
      const int x = labels[(size_t)b * gamma + j];
      const double wk = std::exp(-(double)j / (double)gamma);  // k = j + 1
      const size_t row = ((size_t)b * gamma + j) * V;
      for (int v = 0; v < V; ++v) {
        y[v] = (double)zd[row + v] / T;
        tau[v] = (double)zt[row + v] / T;
      }
      const double Ld = logsumexp(y), Lt = logsumexp(tau);
      double l1 = 0.0, sp = 0.0;
      for (int v = 0; v < V; ++v) {
        p[v] = std::exp(y[v] - Ld);
        q[v] = std::exp(tau[v] - Lt);
        l1 += std::fabs(p[v] - q[v]);
        sp += (p[v] > q[v] ? 1.0 : p[v] < q[v] ? -1.0 : 0.0) * p[v];
      }
      const double cstar = std::min(1.0, std::max(0.0, 1.0 - 0.5 * l1));
      const double cl = (double)conf[(size_t)b * gamma + j];
      const double c = sigmoid(cl);
      // ln c = -softplus(-l), ln(1 - c) = -softplus(l)
      const double log_c = -(std::max(-cl, 0.0) + std::log1p(std::exp(-std::fabs(cl))));
      const double log_1mc = -(std::max(cl, 0.0) + std::log1p(std::exp(-std::fabs(cl))));
      Lce += -wk * (y[x] - Ld);
      Ltv += wk * l1;
      Lconf += -wk * (cstar * log_c + (1.0 - cstar) * log_1mc);
      if (grad_z)
        for (int v = 0; v < V; ++v) {
          const double s_v = p[v] > q[v] ? 1.0 : p[v] < q[v] ? -1.0 : 0.0;
          grad_z[row + v] = wk / T * (a_ce * (p[v] - (v == x ? 1.0 : 0.0)) + a_tv * p[v] * (s_v - sp));
        }
      if (grad_c) grad_c[(size_t)b * gamma + j] = a_conf * wk * (c - cstar);
    }
    loss[b] = a_ce * Lce + a_tv * Ltv + a_conf * Lconf;
    if (parts) {
      parts[3 * (size_t)b] = Lce;
      parts[3 * (size_t)b + 1] = Ltv;
      parts[3 * (size_t)b + 2] = Lconf;
    }
  }
  return bad;
}

// Sequential temperature scaling of the confidence head [P4 s3; P1 delta table D13].  N
// calibration blocks, confidence logits conf [N][gamma], accepted lengths acc [N] (0..gamma),
// a temperature grid [ng].  For k = 1..gamma in order, with tau_1..tau_{k-1} already chosen:
//   S_k[n](t) = prod_{i<k} sigmoid(conf[n][i-1] / tau_i) * sigmoid(conf[n][k-1] / t)
//   y_k[n]    = [acc[n] >= k]
//   ECE_k(t)  = sum_m |sum_{n : bin(S_k[n](t)) = m} (S_k[n](t) - y_k[n])| / N,
//               bin(s) = min(M - 1, floor(s M))
//   tau_k     = the first grid entry with the smallest ECE_k
// Outputs tau [gamma], ece [gamma] (ECE_k at tau_k) and ece_grid [gamma][ng] (every ECE_k(t)).
// Returns 1 if an accepted length lies outside [0, gamma] or a grid entry is not > 0.
int orc_sts(int N, int gamma, const float* conf, const int32_t* acc, int ng, const float* grid,
            int M, double* tau, double* ece, double* ece_grid) {
  for (int n = 0; n < N; ++n)
    if (acc[n] < 0 || acc[n] > gamma) return 1;
  for (int g = 0; g < ng; ++g)
    if (!(grid[g] > 0.0f)) return 1;
  std::vector<double> prefix(N, 1.0), sums(M);
  for (int k = 1; k <= gamma; ++k) {
    int best_g = 0;
    for (int g = 0; g < ng; ++g) {
      const double t = (double)grid[g];
      std::fill(sums.begin(), sums.end(), 0.0);
      for (int n = 0; n < N; ++n) {
        const double S = prefix[n] * sigmoid((double)conf[(size_t)n * gamma + k - 1] / t);
        const double y = acc[n] >= k ? 1.0 : 0.0;
        const int m = std::min(M - 1, (int)std::floor(S * M));
        sums[m] += std::fabs(S - y);
      }
      double e = 0.0;
      for (int m = 0; m < M; ++m) e += std::fabs(sums[m]);
      e /= (double)N;
      ece_grid[(size_t)(k - 1) * ng + g] = e;
      if (e < ece_grid[(size_t)(k - 1) * ng + best_g]) best_g = g;
    }
    tau[k - 1] = (double)grid[best_g];
    ece[k - 1] = ece_grid[(size_t)(k - 1) * ng + best_g];
    for (int n = 0; n < N; ++n) prefix[n] *= sigmoid((double)conf[(size_t)n * gamma + k - 1] / tau[k - 1]);
  }
  return 0;
}

// Hardware-aware prefix scheduler [P2 "设计"; P4 s3 Theta = tau * SPS(B)].  Choose l_b in
// 0..gamma for every request to maximise
//     Theta(l) = sps[n] * sum_b (1 + sum_{k <= l_b} S[b][k]),   n = sum_b (l_b + 1),
// i.e. steps/s at n verify tokens times the expected tokens per step (accepted prefix plus the
// bonus token).  Because every S[b][.] is non-increasing in k, ranking all (b, k) by S
// (descending; ties to smaller k, then smaller b) and taking the top m gives, for each m, the
// largest sum among legal prefix selections with B + m tokens; scanning m = 0..B*gamma finds
// the optimum (smallest m on ties).  The sums are taken in exact fixed point
// (floor(S * 2^32) summed as integers), converted to double once, and multiplied by sps[n] in
// one IEEE multiply.  sps has B*(gamma+1)+1 entries.  Returns 1 if an S is outside [0, 1] or
// increases along a request's block (a survival curve cannot increase).
int orc_prefix_schedule(int B, int gamma, const float* S, const double* sps, int32_t* len,
                        double* theta) {
  const int M = B * gamma;
  for (int i = 0; i < M; ++i) {
    if (!(S[i] >= 0.0f && S[i] <= 1.0f)) return 1;
    if (i % gamma != 0 && S[i] > S[i - 1]) return 1;
  }
  std::vector<int> order(M);
  for (int i = 0; i < M; ++i) order[i] = i;
  std::sort(order.begin(), order.end(), [&](int p, int q) {
    if (S[p] != S[q]) return S[p] > S[q];
    const int kp = p % gamma, kq = q % gamma;
    if (kp != kq) return kp < kq;
    return p / gamma < q / gamma;
  });
  uint64_t fixed_sum = 0;
  double best = sps[B] * (double)B;
  int best_m = 0;
  for (int m = 1; m <= M; ++m) {
    fixed_sum += (uint64_t)std::floor((double)S[order[m - 1]] * 4294967296.0);
    const double tau = (double)B + (double)fixed_sum / 4294967296.0;
    const double th = sps[B + m] * tau;
    if (th > best) {
      best = th;
      best_m = m;
    }
  }
  for (int b = 0; b < B; ++b) len[b] = 0;
  for (int m = 0; m < best_m; ++m) len[order[m] / gamma] += 1;
  *theta = best;
  return 0;
}

}  // extern "C"
