// draft.cuh -- parameters and host-side launch interface of the persistent draft kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace dspark {

struct DraftParams {
  // problem
  int head;  // 0 Markov, 1 RNN
  int B, gamma, V, r, d;
  float invT;
  uint32_t seed_lo, seed_hi;
  uint32_t rk0[10], rk1[10];  // Philox round keys: seed_lo + i * 0x9E3779B9, seed_hi + i * 0xBB67AE85
  int w_bf16, u_bf16;  // dtype flags (weights / activations)
  // inputs
  const void* W1;
  const void* W2;
  const void* w;   // may be null
  const void* Wj;  // RNN only
  const void* U;
  const void* h;   // may be null (Markov without confidence)
  const int32_t* x0;
  const int32_t* forced;  // may be null
  const float* target;    // may be null
  const float* s0;        // RNN, may be null
  // outputs
  int32_t* tokens;
  float* lse;
  float* c;
  float* S;
  float* cstar;
  float* l1;
  float* logits;
  float* s_out;
  // workspace
  WsHeader* hdr;
  unsigned long long* keys;  // [gamma][B][nCTA] per-block tagged argmax keys (zero between calls)
  float* hdot;               // [2][B][gamma] Eq 7 halves: w[0:d] . h[b][k], w[d:] . W1[x_{k-1}]
  float2* ml;                // [gamma][B][nCTA] (max, sum exp) of y per block
  float2* mlt;               // [gamma][B][nCTA] same for the target
  float* l1p;                // [gamma][B][nCTA] partial L1 distances
  float* rnn_s;              // [B][r] RNN state s_k, private to the request's owner block
  float* rnn_a;              // [gamma][B][r] RNN conditioning vectors tanh(o_k)
  float* rnn_gh;             // [ks][B*gamma][3r] split-K partials of h Wj[:, 2r:]^T
  unsigned* rnn_flag;        // [gamma][B] step tags: rnn_a[k][b] is published
  int rnn_ks;                // number of split-K partial planes in rnn_gh
  float* ybuf;               // [B][V] y of the current step (tensor-core path with a target)
  // launch geometry (set by the host)
  int stage_bytes;     // bytes per ring stage (a multiple of 32 W2 rows)
  int nstages;         // ring depth
  int nres;            // W2 stages (CUDA cores) or 128x64 slabs (tensor cores) of each block's
                       // slice kept in TMEM after the first step
  int tcv;             // draft_cc: 1 = bias product on the tensor cores, vocabulary rows on M
  int nres_s;          // tensor-core variant: slabs of the slice resident in shared memory
  int slice_max;       // largest vocab slice of any block (multiple of 8)
  int u_bulk;          // 1: U/target rows are 16-byte aligned and copied with TMA bulk copies
  int tc_na;           // tensor-core path: A-operand buffers
  int tc_nu;           // tensor-core path: U tiles staged in shared memory (0 = direct loads)
  int tc_pk;           // tensor-core path: at most 64 requests, vocabulary tiles in pairs
  int w2_rv;           // tensor-core path: W2 stored [r][V] (an MN-major operand), else [V][r]
  int cl;              // draft_cc: blocks per thread-block cluster (1: no clusters); the
                       // cluster's blocks merge their per-step results in distributed shared
                       // memory and one of them publishes the cluster's, so the grid-wide merge
                       // reads gridDim / cl slots instead of gridDim
  size_t smem_bytes;
  // failure-path test hook (0 in normal use): 1 = the per-step wait between thread blocks, 2 = an
  // mbarrier wait of the epilogue warps, each made to wait for a signal that never comes, with
  // the limit test_wait_ns; the kernel then unwinds exactly as on a real timeout
  int test_stuck;
  unsigned long long test_wait_ns;
};

// Host launchers (defined in the .cu files).  Return a cudaError_t.
cudaError_t launch_draft_cc(DraftParams& p, int nblocks, cudaStream_t stream);
size_t draft_cc_smem_bytes(const DraftParams& p);
bool draft_cc_configure(DraftParams& p, size_t smem_optin);
int draft_cc_supported(int B, int r, int w_bf16);
int draft_tcv_supported(int B, int r, int w_bf16, int slice_max);
cudaError_t launch_draft_tc(DraftParams& p, int nblocks, cudaStream_t stream);
bool draft_tc_configure(DraftParams& p, size_t smem_optin);
int draft_tc_supported(int B, int r, int w_bf16);
// 2-D tensor map of a row-major bf16 matrix [rows][cols] (row stride ld elements) for TMA tile
// loads of box_rows rows x 64 columns into the 128-byte-swizzled K-major layout.
bool encode_bf16_2d(CUtensorMap* m, const void* base, int rows, int cols, int ld, int box_rows);
// 3-D tensor map of U [B][G][V] bf16 for TMA loads of box_rows requests x one position x 64
// vocabulary entries, 128-byte swizzle (V a multiple of 8).
bool encode_u_bf16_3d(CUtensorMap* m, const void* U, int B, int G, int V, int box_rows);
cudaError_t launch_gemm_tc(const void* A, int lda, const void* Bm, int ldb, int M, int N, int K,
                           float* part, int max_split, int nsm, int* ksplit_out, unsigned* status,
                           cudaStream_t stream);
constexpr int kRnnMaxSplit = 8;

}  // namespace dspark
