// sts.cu -- sequential temperature scaling (STS) of the confidence head.
//
// "Phase-Conditioned Speculative Decoding" section 3: after training, the head is calibrated by
// temperature scaling that minimises the expected calibration error of the cumulative product,
// one position at a time; "DSpark -- paper verification" (delta table D13): a left-to-right
// 1-D grid search with the prefix held fixed.  For k = 1..gamma, with tau_1..tau_{k-1} chosen:
//   S_k[n](t) = prod_{i<k} sigmoid(l[n][i-1] / tau_i) * sigmoid(l[n][k-1] / t),
//   y_k[n] = [accepted[n] >= k],
//   ECE_k(t) = sum_m |sum_{n in bin m} (S_k[n](t) - y_k[n])| / N,  bin(s) = min(M - 1, floor(s M)),
//   tau_k = the first grid entry with the smallest ECE_k.
// Two launches per position: sts_part_kernel (one block per grid entry and 2048-sample split:
// each thread keeps its 8 samples' bins and differences in registers, and the per-bin sums are
// warp and block reductions in a fixed order, so the result is deterministic), then
// sts_pick_kernel (one block: the per-bin sums over the splits, the ECE of every grid entry and
// the first minimum).  No waits between thread blocks.
#include "common.cuh"
#include "kernels.h"

namespace dspark {
namespace {

constexpr int kSThr = 256;
constexpr int kSPer = 8;                  // samples per thread
constexpr int kSSplit = kSThr * kSPer;    // samples per block
constexpr int kSMaxBins = 64;

struct StsWs {
  WsHeader* hdr;
  float* tau;    // [gamma] temperatures chosen so far
  float* part;   // [ngrid][nsplit][bins] per-bin sums of S - y
};

__host__ __device__ inline size_t sws_align(size_t x) { return (x + 255) / 256 * 256; }
__host__ __device__ inline size_t sws_layout(int N, int G, int ng, int bins, size_t* off) {
  const size_t nsplit = (size_t)((N + kSSplit - 1) / kSSplit);
  size_t o = sizeof(WsHeader);
  off[0] = o;
  o = sws_align(o + (size_t)G * sizeof(float));
  off[1] = o;
  o = sws_align(o + (size_t)ng * nsplit * bins * sizeof(float));
  return o;
}

__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + __expf(-x)); }

__global__ void __launch_bounds__(kSThr) sts_part_kernel(int N, int G, int k, const float* __restrict__ conf,
                                                         const int32_t* __restrict__ acc,
                                                         const float* __restrict__ grid, int bins,
                                                         int nsplit, StsWs ws) {
  __shared__ float red[kSThr / 32][kSMaxBins];
  const int g = blockIdx.x / nsplit, sp = blockIdx.x % nsplit;
  const float t = grid[g];
  int bin[kSPer];
  float diff[kSPer];
#pragma unroll
  for (int i = 0; i < kSPer; ++i) {
    const int n = sp * kSSplit + i * kSThr + (int)threadIdx.x;
    bin[i] = -1;
    diff[i] = 0.f;
    if (n < N) {
      float S = 1.f;
      for (int j = 0; j < k; ++j) S *= sigm(conf[(size_t)n * G + j] / ws.tau[j]);
      S *= sigm(conf[(size_t)n * G + k] / t);
      bin[i] = min(bins - 1, (int)floorf(S * (float)bins));
      const int a = acc[n];
      diff[i] = S - (a > k ? 1.f : 0.f);  // y = [accepted >= k + 1] (position k + 1)
      if (k == 0 && g == 0 && (a < 0 || a > G)) atomicMax(&ws.hdr->status, kErrInvalid);
    }
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int m = 0; m < bins; ++m) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kSPer; ++i) s += bin[i] == m ? diff[i] : 0.f;
    s = warp_sum(s);
    if (lane == 0) red[w][m] = s;
  }
  __syncthreads();
  for (int m = threadIdx.x; m < bins; m += kSThr) {
    float s = 0.f;
    for (int v = 0; v < kSThr / 32; ++v) s += red[v][m];
    ws.part[((size_t)g * nsplit + sp) * bins + m] = s;
  }
}

__global__ void __launch_bounds__(kSThr) sts_pick_kernel(int N, int k, int ng, const float* __restrict__ grid,
                                                         int bins, int nsplit, StsWs ws,
                                                         float* __restrict__ tau, float* __restrict__ ece,
                                                         float* __restrict__ ece_grid) {
  __shared__ float e_sh[kSThr];
  __shared__ int g_sh[kSThr];
  float best = INFINITY;
  int bg = 0x7FFFFFFF;
  for (int g = threadIdx.x; g < ng; g += kSThr) {  // each thread: its grid entries in order
    float e = 0.f;
    for (int m = 0; m < bins; ++m) {
      float s = 0.f;
      for (int sp = 0; sp < nsplit; ++sp) s += ws.part[((size_t)g * nsplit + sp) * bins + m];
      e += fabsf(s);
    }
    e /= (float)N;
    if (ece_grid) ece_grid[(size_t)k * ng + g] = e;
    if (e < best) {
      best = e;
      bg = g;
    }
  }
  if (k == 0)
    for (int g = threadIdx.x; g < ng; g += kSThr)
      if (!(grid[g] > 0.f)) atomicMax(&ws.hdr->status, kErrInvalid);
  e_sh[threadIdx.x] = best;
  g_sh[threadIdx.x] = bg;
  __syncthreads();
  if (threadIdx.x == 0) {  // the smallest ECE; among equal ones the first grid entry
    for (int i = 1; i < kSThr; ++i)
      if (e_sh[i] < best || (e_sh[i] == best && g_sh[i] < bg)) {
        best = e_sh[i];
        bg = g_sh[i];
      }
    if (bg >= ng) bg = 0;  // every ECE NaN (non-finite inputs): keep an index inside the grid
    ws.tau[k] = grid[bg];
    tau[k] = grid[bg];
    ece[k] = best;
  }
}

}  // namespace

size_t sts_workspace_bytes(int N, int G, int ng, int bins) {
  size_t off[2];
  return sws_layout(N, G, ng, bins, off);
}

cudaError_t launch_sts(int N, int G, const float* conf, const int32_t* acc, int ng, const float* grid,
                       int bins, float* tau, float* ece, float* ece_grid, void* workspace,
                       cudaStream_t stream) {
  size_t off[2];
  sws_layout(N, G, ng, bins, off);
  uint8_t* w = (uint8_t*)workspace;
  StsWs ws;
  ws.hdr = (WsHeader*)w;
  ws.tau = (float*)(w + off[0]);
  ws.part = (float*)(w + off[1]);
  const int nsplit = (N + kSSplit - 1) / kSSplit;
  for (int k = 0; k < G; ++k) {
    sts_part_kernel<<<(unsigned)((long long)ng * nsplit), kSThr, 0, stream>>>(N, G, k, conf, acc, grid,
                                                                              bins, nsplit, ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    sts_pick_kernel<<<1, kSThr, 0, stream>>>(N, k, ng, grid, bins, nsplit, ws, tau, ece, ece_grid);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dspark
