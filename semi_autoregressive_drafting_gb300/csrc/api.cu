// api.cu -- the C ABI of libdspark (declared in include/dspark.h): argument validation,
// workspace layout, kernel-path selection and stream-ordered launches.  No torch types, no
// allocation; the only process-wide state is a per-device cache of SM count, shared-memory
// limit and the largest thread-block cluster that tiles every SM (filled once, under a mutex).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "dspark.h"
#include "draft.cuh"
#include "kernels.h"

using namespace dspark;

namespace {

thread_local std::string g_err;

dspark_status fail(dspark_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

dspark_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DSPARK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DevInfo {
  bool init = false;
  int sms = 0;
  int smem_optin = 0;
  int cluster = 1;  // largest of 8, 4, 2 whose clusters of one-block-per-SM blocks fill every SM
};

// Stand-in for the small-batch draft kernel when sizing clusters: it has the same one block
// per SM (all the shared memory a block may have), and is never launched.
__global__ void cluster_probe_kernel() {}

// Largest cluster size C in {8, 4, 2} with sms % C == 0 such that sms / C clusters of
// whole-SM blocks can be resident at once (clusters must fit inside one GPC, so this depends on
// how the GPCs' SMs are split); 1 if none.
int fitting_cluster(int sms, int smem_optin) {
  if (cudaFuncSetAttribute(cluster_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem_optin) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  for (int c = 8; c >= 2; c /= 2) {
    if (sms % c) continue;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = (unsigned)c;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)sms);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = (size_t)smem_optin;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)cluster_probe_kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (n * c >= sms) return c;
  }
  return 1;
}
std::mutex g_mu;
DevInfo g_dev[64];

bool dev_info(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return false;
    if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
      return false;
    d.cluster = fitting_cluster(d.sms, d.smem_optin);
    d.init = true;
  }
  *out = d;
  return true;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }
bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

struct WsLayout {
  size_t keys, hdot, ml, mlt, l1p, rnn_s, rnn_a, rnn_gh, rnn_flag, ybuf, w2t, total;
};

// flags: DSPARK_WS_TARGET reserves the y buffer the tensor-core path needs for Eq 8
WsLayout ws_layout(int head, int B, int G, int V, int r, int nCTA, int flags) {
  WsLayout L;
  size_t off = sizeof(WsHeader);
  L.keys = off;
  off = align256(off + (size_t)G * B * nCTA * 8);
  L.hdot = off;
  off = align256(off + (size_t)2 * G * B * 4);
  L.ml = off;
  off = align256(off + (size_t)G * B * nCTA * 8);
  L.mlt = off;  // per-block partials (CUDA-core path) or per-chunk target partials (tensor cores)
  off = align256(off + (size_t)G * B * std::max(nCTA, (V + 16383) / 16384) * 8);
  L.l1p = off;
  off = align256(off + (size_t)G * B * nCTA * 4);
  const bool rnn = head == 1;
  L.rnn_s = off;
  off = align256(off + (rnn ? (size_t)B * r * 4 : 0));
  L.rnn_a = off;
  off = align256(off + (rnn ? (size_t)G * B * r * 4 : 0));
  L.rnn_gh = off;
  off = align256(off + (rnn ? (size_t)kRnnMaxSplit * B * G * 3 * r * 4 : 0));
  L.rnn_flag = off;
  off = align256(off + (rnn ? (size_t)G * B * 4 : 0));
  L.ybuf = off;
  off = align256(off + ((flags & DSPARK_WS_TARGET) && B > 4 ? (size_t)B * V * 4 : 0));
  // W2 given as [r][V]: the small-batch kernels (B <= 4) read its [V][r] transpose from here
  L.w2t = off;
  off = align256(off + ((flags & DSPARK_WS_W2_RV) && B <= 4 ? (size_t)V * r * 4 : 0));
  L.total = off;
  return L;
}

bool shape_ok(int head, int B, int G, int V, int r, int d) {
  return (head == 0 || head == 1) && B >= 1 && G >= 1 && G <= 16 && V >= 2 && V <= (1 << 24) &&
         r >= 8 && r <= 512 && r % 8 == 0 && d >= 0 && d % 8 == 0 && B <= (1 << 20);
}

int slice_max_of(int V, int nCTA) {
  const int units = (V + 7) / 8;
  return ((units + nCTA - 1) / nCTA) * 8;
}

// 0: CUDA-core dot products; 1: tensor cores with requests on M; 2: tensor cores with the
// vocabulary on M.  DSPARK_DRAFT_PATH=cuda-core|tensor|tensor-vocab picks one (-1 if that one
// cannot run these arguments); otherwise 2 for B = 3 or 4, else the first of 0, 2, 1 that can.
int path_of(int head, int B, int V, int r, int w_bf16, int nCTA) {
  if (head == 1 && !w_bf16) return -1;  // the RNN pre-pass is a bf16 tensor-core GEMM
  const bool ok[3] = {draft_cc_supported(B, r, w_bf16) != 0, draft_tc_supported(B, r, w_bf16) != 0,
                      draft_tcv_supported(B, r, w_bf16, slice_max_of(V, nCTA)) != 0};
  if (const char* f = std::getenv("DSPARK_DRAFT_PATH")) {
    const int want = !std::strcmp(f, "cuda-core") ? 0 : !std::strcmp(f, "tensor") ? 1
                   : !std::strcmp(f, "tensor-vocab") ? 2 : -2;
    if (want >= 0) return ok[want] ? want : -1;
  }
  // Measured on GB300 (r = 256, V = 151936): an M = 128, N = 16 MMA costs about as much as a
  // full-width one, so the tensor cores pay off from B = 3 on; below that the CUDA cores win.
  if (ok[2] && B >= 3) return 2;
  return ok[0] ? 0 : ok[2] ? 2 : ok[1] ? 1 : -1;
}

// Blocks per cluster of the small-batch kernels (paths 0 and 2): DSPARK_CLUSTER = 2 | 4 | 8,
// read at every call, asks for clusters of that size (-1 if they cannot tile the SMs); unset,
// or 1, no clusters.  Measured on GB300 (152 SMs, where only 2-block clusters tile every SM):
// the per-step hop through the cluster's first block costs more than halving the slots every
// block polls saves (B = 1, V = 151936: 90 us per block without clusters), so clusters are not
// the default.
int cluster_of(const DevInfo& di, int nCTA) {
  if (const char* f = std::getenv("DSPARK_CLUSTER")) {
    const int want = std::atoi(f);
    if (want == 2 || want == 4 || want == 8) return nCTA % want == 0 && want <= di.cluster ? want : -1;
  }
  return 1;
}

struct DraftArgs {
  int head, B, G, V, r, d;
  float T;
  uint64_t seed;
  dspark_dtype wdt, udt;
  const void *W1, *W2;
  int w2_layout;
  const void *w, *Wj, *U, *h;
  const int32_t *x0, *forced;
  const float *target, *s0;
  int32_t* tokens;
  float *lse, *c, *S, *cstar, *l1, *logits, *s_out;
  void* ws;
  size_t ws_bytes;
  void* stream;
};

dspark_status run_draft(const DraftArgs& a) {
  g_err.clear();
  if (!shape_ok(a.head, a.B, a.G, a.V, a.r, a.d))
    return fail(DSPARK_ERR_INVALID, "bad shape B=%d gamma=%d V=%d r=%d d=%d", a.B, a.G, a.V, a.r,
                a.d);
  if (!(a.T > 0.f) || !std::isfinite(a.T)) return fail(DSPARK_ERR_INVALID, "T must be finite and > 0");
  if ((a.wdt != DSPARK_F32 && a.wdt != DSPARK_BF16) || (a.udt != DSPARK_F32 && a.udt != DSPARK_BF16))
    return fail(DSPARK_ERR_INVALID, "unknown dtype");
  if (a.w2_layout != DSPARK_W2_VR && a.w2_layout != DSPARK_W2_RV)
    return fail(DSPARK_ERR_INVALID, "unknown W2 layout %d", a.w2_layout);
  if (!a.W1 || !a.W2 || !a.U || !a.x0 || !a.tokens || !a.lse)
    return fail(DSPARK_ERR_INVALID, "W1, W2, U, x0, tokens and lse are required");
  if (!aligned(a.W1, 16) || !aligned(a.W2, 16) || !aligned(a.U, 16) ||
      (a.target && !aligned(a.target, 16)) || (a.h && !aligned(a.h, 16)) ||
      (a.Wj && !aligned(a.Wj, 16)))
    return fail(DSPARK_ERR_INVALID, "W1, W2, U, h, Wj and target must be 16-byte aligned");
  const bool conf = a.h && a.w;
  if (a.head == 1 && (a.wdt != DSPARK_BF16 || a.udt != DSPARK_BF16))
    return fail(DSPARK_ERR_UNSUPPORTED, "the RNN head runs on bf16 weights and activations");
  if (a.head == 0 && ((a.h != nullptr) != (a.w != nullptr)))
    return fail(DSPARK_ERR_INVALID, "h and w go together for the Markov head");
  if (a.head == 1 && (!a.Wj || !a.h || a.d == 0))
    return fail(DSPARK_ERR_INVALID, "the RNN head needs Wj, h and d > 0");
  if (a.head == 1 && a.h && !a.w && (a.c || a.S))
    return fail(DSPARK_ERR_INVALID, "c and S need the confidence weight w");
  if (conf && a.d == 0) return fail(DSPARK_ERR_INVALID, "confidence needs d > 0");
  if ((a.c != nullptr) != conf || (a.S != nullptr) != conf)
    return fail(DSPARK_ERR_INVALID, "c and S are given exactly when h and w are");
  if ((a.cstar != nullptr) != (a.target != nullptr) || (a.l1 != nullptr) != (a.target != nullptr))
    return fail(DSPARK_ERR_INVALID, "cstar and l1 are given exactly when target is");
  DevInfo di;
  if (!dev_info(&di)) return fail(DSPARK_ERR_CUDA, "cannot query the current device");
  const int nCTA = di.sms;
  const bool w2rv = a.w2_layout == DSPARK_W2_RV;
  const WsLayout L = ws_layout(a.head, a.B, a.G, a.V, a.r, nCTA,
                               (a.target ? DSPARK_WS_TARGET : 0) | (w2rv ? DSPARK_WS_W2_RV : 0));
  if (!a.ws || !aligned(a.ws, 256) || a.ws_bytes < L.total)
    return fail(DSPARK_ERR_WORKSPACE, "workspace must be 256-byte aligned and >= %zu bytes", L.total);
  const int w_bf16 = a.wdt == DSPARK_BF16, u_bf16 = a.udt == DSPARK_BF16;
  const int path = path_of(a.head, a.B, a.V, a.r, w_bf16, nCTA);
  if (path < 0)
    return fail(DSPARK_ERR_UNSUPPORTED, "no kernel of the library runs head=%d B=%d r=%d dtype=%d",
                a.head, a.B, a.r, (int)a.wdt);

  DraftParams p;
  std::memset(&p, 0, sizeof p);
  p.head = a.head;
  p.B = a.B;
  p.gamma = a.G;
  p.V = a.V;
  p.r = a.r;
  p.d = a.d;
  p.invT = 1.f / a.T;
  p.seed_lo = (uint32_t)(a.seed & 0xFFFFFFFFu);
  p.seed_hi = (uint32_t)(a.seed >> 32);
  for (int i = 0; i < 10; ++i) {
    p.rk0[i] = p.seed_lo + (uint32_t)i * 0x9E3779B9u;
    p.rk1[i] = p.seed_hi + (uint32_t)i * 0xBB67AE85u;
  }
  p.w_bf16 = w_bf16;
  p.u_bf16 = u_bf16;
  p.W1 = a.W1;
  p.W2 = a.W2;
  p.w = a.w;
  p.Wj = a.Wj;
  p.U = a.U;
  p.h = a.h;
  p.x0 = a.x0;
  p.forced = a.forced;
  p.target = a.target;
  p.s0 = a.s0;
  p.tokens = a.tokens;
  p.lse = a.lse;
  p.c = a.c;
  p.S = a.S;
  p.cstar = a.cstar;
  p.l1 = a.l1;
  p.logits = a.logits;
  p.s_out = a.s_out;
  uint8_t* ws = (uint8_t*)a.ws;
  p.hdr = (WsHeader*)ws;
  p.keys = (unsigned long long*)(ws + L.keys);
  p.hdot = (float*)(ws + L.hdot);
  p.ml = (float2*)(ws + L.ml);
  p.mlt = (float2*)(ws + L.mlt);
  p.l1p = (float*)(ws + L.l1p);
  p.rnn_s = (float*)(ws + L.rnn_s);
  p.rnn_a = (float*)(ws + L.rnn_a);
  p.rnn_gh = (float*)(ws + L.rnn_gh);
  p.rnn_flag = (unsigned*)(ws + L.rnn_flag);
  p.ybuf = (float*)(ws + L.ybuf);

  // Failure-path test hook: DSPARK_TEST_STUCK_WAIT = grid | mbar (read at every call) makes one
  // named wait of the draft kernel wait for a signal that never comes -- one more grid-barrier
  // arrival than there are blocks, or an mbarrier no thread arrives on -- with a 20 us limit, so
  // that the call ends with DSPARK_ERR_TIMEOUT through the kernel's ordinary unwinding.  Unset
  // (normal use), nothing changes.
  if (const char* f = std::getenv("DSPARK_TEST_STUCK_WAIT")) {
    p.test_stuck = !std::strcmp(f, "grid") ? 1 : !std::strcmp(f, "mbar") ? 2 : 0;
    p.test_wait_ns = 20000ull;
  }

  const int units = (a.V + 7) / 8;
  p.slice_max = ((units + nCTA - 1) / nCTA) * 8;
  const int ues = u_bf16 ? 2 : 4;
  p.u_bulk = ((size_t)a.V * ues) % 16 == 0 && (!a.target || ((size_t)a.V * 4) % 16 == 0);
  cudaStream_t stream = (cudaStream_t)a.stream;

  if (a.head == 1) {
    // the h_k columns of Eq 6's joint projection, for every (request, position), up front
    int ks = 0;
    cudaError_t e = launch_gemm_tc(a.h, a.d, (const __nv_bfloat16*)a.Wj + 2 * a.r, 2 * a.r + a.d,
                                   a.B * a.G, 3 * a.r, a.d, p.rnn_gh, kRnnMaxSplit, nCTA, &ks,
                                   &p.hdr->status, stream);
    if (e != cudaSuccess) return cuda_fail(e, "rnn pre-pass launch");
    p.rnn_ks = ks;
  }

  if (path == 0 || path == 2) {
    p.cl = cluster_of(di, nCTA);
    if (p.cl < 0) return fail(DSPARK_ERR_UNSUPPORTED, "DSPARK_CLUSTER: clusters of that size do not tile the SMs");
    if (w2rv) {  // these kernels read [V][r]: transpose W2 into the workspace first
      void* w2t = (uint8_t*)a.ws + L.w2t;
      cudaError_t e = launch_transpose(a.W2, w2t, a.r, a.V, w_bf16 ? 2 : 4, stream);
      if (e != cudaSuccess) return cuda_fail(e, "W2 transpose launch");
      p.W2 = w2t;
    }
    p.tcv = path == 2;
    if (p.tcv && !draft_cc_configure(p, (size_t)di.smem_optin) && !std::getenv("DSPARK_DRAFT_PATH") &&
        draft_cc_supported(a.B, a.r, w_bf16))
      p.tcv = 0;  // the per-step buffers leave too little room for the slab ring: CUDA cores
    if (!draft_cc_configure(p, (size_t)di.smem_optin))
      return fail(DSPARK_ERR_UNSUPPORTED, "vocab slice too large for shared memory");
    cudaError_t e = launch_draft_cc(p, nCTA, stream);
    if (e != cudaSuccess) return cuda_fail(e, "draft_cc launch");
  } else {
    if (a.V > (1 << 24) - 1) return fail(DSPARK_ERR_UNSUPPORTED, "V too large for the tensor-core path");
    if (w2rv && a.V % 8 != 0)
      return fail(DSPARK_ERR_UNSUPPORTED, "W2 as [r][V] on the tensor-core path needs V a multiple of 8");
    p.w2_rv = w2rv;
    if (!draft_tc_configure(p, (size_t)di.smem_optin))
      return fail(DSPARK_ERR_UNSUPPORTED, "rank too large for shared memory");
    cudaError_t e = launch_draft_tc(p, nCTA, stream);
    if (e != cudaSuccess) return cuda_fail(e, "draft_tc launch");
  }
  return DSPARK_OK;
}

}  // namespace

namespace dspark {
void set_last_error(const char* msg) { g_err = msg; }
}  // namespace dspark

extern "C" {

size_t dspark_workspace_bytes(int head, int B, int gamma, int V, int r, int d, int flags) {
  if (!shape_ok(head, B, gamma, V, r, d)) return 0;
  DevInfo di;
  if (!dev_info(&di)) return 0;
  return ws_layout(head, B, gamma, V, r, di.sms, flags).total;
}

dspark_status dspark_markov_draft(int B, int gamma, int V, int r, int d, float T, uint64_t seed,
                                  dspark_dtype wdt, const void* W1, const void* W2,
                                  dspark_w2_layout w2_layout, const void* w, dspark_dtype udt,
                                  const void* U, const void* h,
                                  const int32_t* x0, const int32_t* forced, const float* target,
                                  int32_t* tokens, float* lse, float* c, float* S, float* cstar,
                                  float* l1, float* logits, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  DraftArgs a{0,       B,      gamma,  V,      r,      d,     T,     seed,    wdt,
              udt,     W1,     W2,     (int)w2_layout,     w,      nullptr, U,    h,     x0,      forced,
              target,  nullptr, tokens, lse,   c,      S,     cstar, l1,      logits,
              nullptr, workspace, workspace_bytes, stream};
  return run_draft(a);
}

dspark_status dspark_rnn_draft(int B, int gamma, int V, int r, int d, float T, uint64_t seed,
                               dspark_dtype wdt, const void* W1, const void* W2,
                               dspark_w2_layout w2_layout, const void* w, const void* Wj,
                               dspark_dtype udt, const void* U, const void* h,
                               const int32_t* x0, const int32_t* forced, const float* target,
                               const float* s0, int32_t* tokens, float* lse, float* c, float* S,
                               float* cstar, float* l1, float* logits, float* s_out,
                               void* workspace, size_t workspace_bytes, void* stream) {
  DraftArgs a{1,      B,     gamma,  V,     r,     d,     T,      seed,      wdt,
              udt,    W1,    W2,     (int)w2_layout,     w,     Wj,    U,     h,      x0,        forced,
              target, s0,    tokens, lse,   c,     S,     cstar,  l1,        logits,
              s_out,  workspace, workspace_bytes, stream};
  return run_draft(a);
}

dspark_status dspark_confidence(int B, int gamma, int V, int r, int d, dspark_dtype wdt,
                                const void* W1, const void* w, dspark_dtype udt, const void* h,
                                const int32_t* x0, const int32_t* tokens, float* c, float* S,
                                void* stream) {
  g_err.clear();
  if (!shape_ok(0, B, gamma, V, r, d) || d == 0)
    return fail(DSPARK_ERR_INVALID, "bad shape B=%d gamma=%d V=%d r=%d d=%d", B, gamma, V, r, d);
  if (!W1 || !w || !h || !x0 || !tokens || !c || !S)
    return fail(DSPARK_ERR_INVALID, "all arrays are required");
  cudaError_t e = launch_confidence(B, gamma, V, r, d, wdt == DSPARK_BF16, W1, w,
                                    udt == DSPARK_BF16, h, x0, tokens, c, S, (cudaStream_t)stream);
  return e == cudaSuccess ? DSPARK_OK : cuda_fail(e, "confidence launch");
}

dspark_status dspark_tv_label(int N, int V, float T, const float* draft_logits,
                              const float* target_logits, float* cstar, float* l1, void* stream) {
  g_err.clear();
  if (N < 1 || V < 2 || !(T > 0.f) || !std::isfinite(T))
    return fail(DSPARK_ERR_INVALID, "bad arguments N=%d V=%d", N, V);
  if (!draft_logits || !target_logits || !cstar)
    return fail(DSPARK_ERR_INVALID, "draft_logits, target_logits and cstar are required");
  cudaError_t e = launch_tv_label(N, V, T, draft_logits, target_logits, cstar, l1,
                                  (cudaStream_t)stream);
  return e == cudaSuccess ? DSPARK_OK : cuda_fail(e, "tv_label launch");
}

dspark_status dspark_prefix_schedule(int B, int gamma, const float* S, const double* sps,
                                     int32_t* len, double* theta, void* stream) {
  g_err.clear();
  if (B < 1 || gamma < 1 || gamma > 16 || (long long)B * gamma > 16384)
    return fail(DSPARK_ERR_INVALID, "need 1 <= gamma <= 16 and B * gamma <= 16384");
  if (!S || !sps || !len || !theta) return fail(DSPARK_ERR_INVALID, "all arrays are required");
  cudaError_t e = launch_prefix_schedule(B, gamma, S, sps, len, theta, (cudaStream_t)stream);
  return e == cudaSuccess ? DSPARK_OK : cuda_fail(e, "prefix_schedule launch");
}

size_t dspark_verify_workspace_bytes(int B, int gamma, int V) {
  if (B < 1 || gamma < 1 || gamma > 16 || V < 2 || V > (1 << 24)) return 0;
  return verify_workspace_bytes(B, gamma, V);
}

dspark_status dspark_verify(int B, int gamma, int V, float T, uint64_t seed,
                            const float* draft_logits, const float* target_logits,
                            const int32_t* draft_tokens, int32_t* n_accepted, int32_t* out_tokens,
                            void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  if (B < 1 || B > (1 << 20) || gamma < 1 || gamma > 16 || V < 2 || V > (1 << 24))
    return fail(DSPARK_ERR_INVALID, "bad shape B=%d gamma=%d V=%d", B, gamma, V);
  if (!(T > 0.f) || !std::isfinite(T)) return fail(DSPARK_ERR_INVALID, "T must be finite and > 0");
  if (!draft_logits || !target_logits || !draft_tokens || !n_accepted || !out_tokens)
    return fail(DSPARK_ERR_INVALID, "all arrays are required");
  if (!aligned(draft_logits, 16) || !aligned(target_logits, 16))
    return fail(DSPARK_ERR_INVALID, "draft_logits and target_logits must be 16-byte aligned");
  const size_t need = verify_workspace_bytes(B, gamma, V);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(DSPARK_ERR_WORKSPACE, "workspace must be 256-byte aligned and >= %zu bytes", need);
  cudaError_t e = launch_verify(B, gamma, V, T, seed, draft_logits, target_logits, draft_tokens,
                                n_accepted, out_tokens, workspace, (cudaStream_t)stream);
  return e == cudaSuccess ? DSPARK_OK : cuda_fail(e, "verify launch");
}

size_t dspark_draft_loss_workspace_bytes(int B, int gamma, int V) {
  if (B < 1 || gamma < 1 || gamma > 16 || V < 2 || V > (1 << 24)) return 0;
  return loss_workspace_bytes(B, gamma, V);
}

dspark_status dspark_draft_loss(int B, int gamma, int V, float T, const float* draft_logits,
                                const float* target_logits, const int32_t* labels,
                                const float* conf_logits, float alpha_ce, float alpha_tv,
                                float alpha_conf, float* loss, float* parts, float* grad_logits,
                                float* grad_conf, void* workspace, size_t workspace_bytes,
                                void* stream) {
  g_err.clear();
  if (B < 1 || B > (1 << 20) || gamma < 1 || gamma > 16 || V < 2 || V > (1 << 24))
    return fail(DSPARK_ERR_INVALID, "bad shape B=%d gamma=%d V=%d", B, gamma, V);
  if (!(T > 0.f) || !std::isfinite(T)) return fail(DSPARK_ERR_INVALID, "T must be finite and > 0");
  if (!std::isfinite(alpha_ce) || !std::isfinite(alpha_tv) || !std::isfinite(alpha_conf))
    return fail(DSPARK_ERR_INVALID, "the loss weights must be finite");
  if (!draft_logits || !target_logits || !labels || !conf_logits)
    return fail(DSPARK_ERR_INVALID, "draft_logits, target_logits, labels and conf_logits are required");
  if (!loss && !parts && !grad_logits && !grad_conf)
    return fail(DSPARK_ERR_INVALID, "no output requested");
  if (!aligned(draft_logits, 16) || !aligned(target_logits, 16) || (grad_logits && !aligned(grad_logits, 16)))
    return fail(DSPARK_ERR_INVALID, "draft_logits, target_logits and grad_logits must be 16-byte aligned");
  const size_t need = loss_workspace_bytes(B, gamma, V);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(DSPARK_ERR_WORKSPACE, "workspace must be 256-byte aligned and >= %zu bytes", need);
  cudaError_t e = launch_loss(B, gamma, V, T, draft_logits, target_logits, labels, conf_logits,
                              alpha_ce, alpha_tv, alpha_conf, loss, parts, grad_logits, grad_conf,
                              workspace, (cudaStream_t)stream);
  return e == cudaSuccess ? DSPARK_OK : cuda_fail(e, "draft loss launch");
}

size_t dspark_sts_workspace_bytes(int N, int gamma, int ngrid, int bins) {
  if (N < 1 || gamma < 1 || gamma > 16 || ngrid < 1 || ngrid > 4096 || bins < 1 || bins > 64) return 0;
  return sts_workspace_bytes(N, gamma, ngrid, bins);
}

dspark_status dspark_sts(int N, int gamma, const float* conf_logits, const int32_t* accepted,
                         int ngrid, const float* grid, int bins, float* tau, float* ece,
                         float* ece_grid, void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  if (N < 1 || N > (1 << 26) || gamma < 1 || gamma > 16 || ngrid < 1 || ngrid > 4096 || bins < 1 ||
      bins > 64)
    return fail(DSPARK_ERR_INVALID, "bad shape N=%d gamma=%d ngrid=%d bins=%d", N, gamma, ngrid, bins);
  if (!conf_logits || !accepted || !grid || !tau || !ece)
    return fail(DSPARK_ERR_INVALID, "conf_logits, accepted, grid, tau and ece are required");
  const size_t need = sts_workspace_bytes(N, gamma, ngrid, bins);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(DSPARK_ERR_WORKSPACE, "workspace must be 256-byte aligned and >= %zu bytes", need);
  cudaError_t e = launch_sts(N, gamma, conf_logits, accepted, ngrid, grid, bins, tau, ece, ece_grid,
                             workspace, (cudaStream_t)stream);
  return e == cudaSuccess ? DSPARK_OK : cuda_fail(e, "sts launch");
}

dspark_status dspark_get_status(void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  if (!workspace || workspace_bytes < sizeof(WsHeader))
    return fail(DSPARK_ERR_WORKSPACE, "workspace missing or too small");
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned st = 0;
  e = cudaMemcpy(&st, workspace, sizeof st, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (st != 0) {
    e = cudaMemset(workspace, 0, workspace_bytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "workspace reset");
  }
  return (dspark_status)st;
}

const char* dspark_last_error(void) { return g_err.c_str(); }

int dspark_draft_path(int head, int B, int V, int r, dspark_dtype wdt) {
  if (!shape_ok(head, B, 1, V, r, 0)) return -1;
  DevInfo di;
  const int nCTA = dev_info(&di) ? di.sms : 152;  // without a device: a GB300's count
  return path_of(head, B, V, r, wdt == DSPARK_BF16, nCTA);
}

int dspark_draft_cluster(int head, int B, int V, int r, dspark_dtype wdt) {
  const int path = dspark_draft_path(head, B, V, r, wdt);
  if (path < 0) return -1;
  if (path == 1) return 1;
  DevInfo di;
  if (!dev_info(&di)) return -1;
  return cluster_of(di, di.sms);
}

int dspark_draft_loss_launches(int B, int gamma, int V, int with_grad) {
  if (B < 1 || B > (1 << 20) || gamma < 1 || gamma > 16 || V < 2 || V > (1 << 24)) return -1;
  // launch_loss: the normalisers, the |p - q| sums, the gradient (when asked) and the totals
  return with_grad ? 4 : 3;
}

int dspark_draft_launches(int head, int B, int V, int r, dspark_dtype wdt) {
  const int p = dspark_draft_path(head, B, V, r, wdt);
  if (p < 0) return -1;
  return head == 1 ? 2 : 1;  // one persistent launch (+ the RNN head's pre-pass GEMM)
}

}  // extern "C"
