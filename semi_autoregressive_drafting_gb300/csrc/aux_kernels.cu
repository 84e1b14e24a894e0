// aux_kernels.cu -- the three per-round kernels that sit beside the draft loop:
//   confidence_kernel  teacher-forced Eq 7 and prefix survival S_k = prod c_i
//                      ("DSpark -- paper verification", section 1, Eq 7, section 3.2.1)
//   tv_label_kernel    Eq 8: c* = 1 - 1/2 ||softmax(d/T) - softmax(t/T)||_1, clamped
//                      ("Phase-Conditioned Speculative Decoding", section 3: c* = 1 - TV)
//   schedule_kernel    the hardware-aware prefix scheduler: per-request verify lengths that
//                      maximise SPS(n) * expected accepted tokens over legal prefixes
//                      ("DSpark: 既要猜得连贯..." design section; same page-4 section, Theta)
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {
namespace {

__device__ __forceinline__ float ldv(const void* p, size_t i, int bf16) {
  return bf16 ? __bfloat162float(((const __nv_bfloat16*)p)[i]) : ((const float*)p)[i];
}

// One warp per (request, position): logit = w[0:d].h + w[d:].W1[x_{k-1}]; a second pass turns
// the logits of a request into c and the running product S.
__global__ void confidence_logits_kernel(int B, int G, int V, int r, int d, int w_bf16,
                                         const void* W1, const void* w, int u_bf16, const void* h,
                                         const int32_t* x0, const int32_t* tokens, float* c) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= B * G) return;
  const int b = warp / G, k = warp % G;
  const int prev = k == 0 ? x0[b] : tokens[(size_t)b * G + k - 1];
  if (prev < 0 || prev >= V) {
    if (lane == 0) c[warp] = NAN;
    return;
  }
  float acc = 0.f;
  for (int j = lane; j < d; j += 32) acc += ldv(w, j, w_bf16) * ldv(h, (size_t)warp * d + j, u_bf16);
  for (int j = lane; j < r; j += 32)
    acc += ldv(w, (size_t)d + j, w_bf16) * ldv(W1, (size_t)prev * r + j, w_bf16);
  acc = warp_sum(acc);
  if (lane == 0) c[warp] = acc;  // logit for now
}

__global__ void confidence_finish_kernel(int B, int G, float* c, float* S) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  float s = 1.f;
  bool bad = false;
  for (int k = 0; k < G; ++k) {
    const size_t o = (size_t)b * G + k;
    const float logit = c[o];
    bad = bad || isnan(logit);
    const float cv = bad ? NAN : sigmoidf_acc(logit);
    s = bad ? NAN : s * cv;
    c[o] = cv;
    S[o] = s;
  }
}

// Eq 8 for one row per block: pass 1 online (max, sum-exp) of both rows, pass 2 the L1 sum.
__global__ void __launch_bounds__(512) tv_label_kernel(int V, float invT, const float* dl,
                                                       const float* tl, float* cstar, float* l1) {
  __shared__ float sm[4][16];
  const size_t base = (size_t)blockIdx.x * V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  float md = -INFINITY, ld = 0.f, mt = -INFINITY, lt = 0.f;
  for (int v = tid; v < V; v += blockDim.x) {
    lse_push(md, ld, dl[base + v] * invT);
    lse_push(mt, lt, tl[base + v] * invT);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lse_merge(md, ld, __shfl_xor_sync(~0u, md, o), __shfl_xor_sync(~0u, ld, o));
    lse_merge(mt, lt, __shfl_xor_sync(~0u, mt, o), __shfl_xor_sync(~0u, lt, o));
  }
  if (lane == 0) {
    sm[0][warp] = md;
    sm[1][warp] = ld;
    sm[2][warp] = mt;
    sm[3][warp] = lt;
  }
  __syncthreads();
  md = -INFINITY, ld = 0.f, mt = -INFINITY, lt = 0.f;
  for (int w = 0; w < nw; ++w) {
    lse_merge(md, ld, sm[0][w], sm[1][w]);
    lse_merge(mt, lt, sm[2][w], sm[3][w]);
  }
  const float Ld = md + logf(ld), Lt = mt + logf(lt);
  __syncthreads();
  float acc = 0.f;
  for (int v = tid; v < V; v += blockDim.x)
    acc += fabsf(__expf(dl[base + v] * invT - Ld) - __expf(tl[base + v] * invT - Lt));
  acc = warp_sum(acc);
  if (lane == 0) sm[0][warp] = acc;
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += sm[0][w];
    if (l1) l1[blockIdx.x] = s;
    cstar[blockIdx.x] = fminf(1.f, fmaxf(0.f, 1.f - 0.5f * s));
  }
}

// Prefix scheduler, one block.  Keys rank every (b, k) by S descending, then k, then b:
//   key = ((~bits(S)) << 32) | (k << 24) | b   sorted ascending (S >= 0, so bits order S).
// Because each S row is non-increasing, every top-m set is a union of per-request prefixes
// and the top-m sum is the best legal sum with B + m verify tokens.  The sums are exact
// (floor(S 2^32) added as integers), so Theta(m) = sps[B + m] * (B + sum 2^-32) is a single
// IEEE double multiply and the argmax (smallest m on ties) is reproducible bit for bit.
// floor(S 2^32) is taken in single precision (S 2^32 is exact in fp32 for S in [0, 1], and the
// conversion truncates), and the 2^-32 scaling is an exact multiply: the only fp64 arithmetic
// left per entry is the conversion of the sum, one add and the Theta multiply.
constexpr int kSchedThreads = 1024;

// Bitonic sort of the Mp2 keys, ascending, with the keys in registers: thread t holds keys
// [t E, t E + E).  Compare-exchange partners inside a thread are swapped in registers, partners
// in another lane of the warp come by shuffle, and only strides of 32 E or more go through
// shared memory (the same sort of 4096 keys all in shared memory took 31 us on GB300, this one
// 26 us).  Padding keys (index >= Mp2 when Mp2 < 1024) only ever meet other padding keys.
template <int E>
__device__ __forceinline__ void sort_keys(unsigned long long* keys, int Mp2) {
  const int tid = threadIdx.x;
  unsigned long long r[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = tid * E + e;
    r[e] = i < Mp2 ? keys[i] : ~0ull;
  }
  for (int size = 2; size <= Mp2; size <<= 1) {
    int stride = size >> 1;
    if (stride >= 32 * E) {  // across warps: through shared memory
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (tid * E + e < Mp2) keys[tid * E + e] = r[e];
      __syncthreads();
      for (; stride >= 32 * E; stride >>= 1) {
        for (int pi = tid; pi < Mp2 / 2; pi += kSchedThreads) {
          const int lo = 2 * pi - (pi & (stride - 1));
          const int hi = lo + stride;
          const bool up = (lo & size) == 0;
          const unsigned long long a = keys[lo], c = keys[hi];
          if ((a > c) == up) {
            keys[lo] = c;
            keys[hi] = a;
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int i = tid * E + e;
        r[e] = i < Mp2 ? keys[i] : ~0ull;
      }
      __syncthreads();  // every read done before the next size writes shared memory again
    }
    for (; stride >= E; stride >>= 1) {  // across the lanes of a warp
      const int ld = stride / E;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int i = tid * E + e;
        const unsigned long long o = __shfl_xor_sync(~0u, r[e], ld);
        const bool keep_min = ((i & stride) == 0) == ((i & size) == 0);
        r[e] = keep_min ? (o < r[e] ? o : r[e]) : (o > r[e] ? o : r[e]);
      }
    }
#pragma unroll
    for (int st = E / 2; st > 0; st >>= 1) {  // inside the thread
      if (st > (size >> 1)) continue;
#pragma unroll
      for (int e = 0; e < E; ++e)
        if ((e & st) == 0) {
          const bool up = ((tid * E + e) & size) == 0;
          const unsigned long long a = r[e], c = r[e + st];
          if ((a > c) == up) {
            r[e] = c;
            r[e + st] = a;
          }
        }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (tid * E + e < Mp2) keys[tid * E + e] = r[e];
  __syncthreads();
}

// Merge sort of the keys when each request's G keys already ascend (S non-increasing along k,
// ties to the smaller k): bottom-up rounds from runs of G, ping-ponging between two buffers.
// In each round every thread writes a contiguous share of the output: one merge-path search
// (how many of the first outputs of its pair come from the pair's first run) per pair its
// share touches, then a sequential merge.  The keys are distinct, so the order is total.
// Returns the buffer holding the sorted keys.  (For 3584 keys on GB300: 19 us, against 26 us
// for the single-block bitonic sort below, which serves when the second buffer does not fit.)
__device__ __forceinline__ unsigned long long* merge_runs(unsigned long long* src,
                                                          unsigned long long* dst, int M, int L0) {
  const int per = (M + kSchedThreads - 1) / kSchedThreads;
  for (int L = L0; L < M; L <<= 1) {
    const int L2 = 2 * L;
    int p = (int)threadIdx.x * per;
    const int pend = min(M, p + per);
    while (p < pend) {
      const int lo = (p / L2) * L2;
      const int mid = min(lo + L, M), hi = min(lo + L2, M);
      const int n1 = mid - lo, n2 = hi - mid, d = p - lo;
      int alo = max(0, d - n2), ahi = min(d, n1);
      while (alo < ahi) {
        const int am = (alo + ahi) >> 1;
        if (src[lo + am] < src[mid + d - am - 1]) alo = am + 1;
        else ahi = am;
      }
      int ia = lo + alo, ib = mid + (d - alo);
      const int seg_end = min(pend, hi);
      for (; p < seg_end; ++p) {
        const bool take_a = ib >= hi || (ia < mid && src[ia] < src[ib]);
        dst[p] = take_a ? src[ia++] : src[ib++];
      }
    }
    __syncthreads();
    unsigned long long* t = src;
    src = dst;
    dst = t;
  }
  return src;
}

template <int E>
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(int B, int G, int M, int Mp2,
                                                                 int merge, const float* S,
                                                                 const double* sps, int32_t* len,
                                                                 double* theta) {
  // [Mp2] keys, [kSchedThreads] scan scratch, then (merge) a second [M] key buffer
  extern __shared__ __align__(16) unsigned long long keys_raw[];
  unsigned long long* keys = keys_raw;
  unsigned long long* csum = keys_raw + Mp2;                   // [kSchedThreads] block sums
  __shared__ int bad;
  __shared__ double best_val[32];
  __shared__ int best_m[32];
  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  __syncthreads();
  for (int i = tid; i < Mp2; i += kSchedThreads) {
    if (i < M) {
      const float s = S[i];
      const int b = i / G, k = i - b * G;
      const bool ok = s >= 0.f && s <= 1.f && (k == 0 || s <= S[i - 1]);
      if (!ok) bad = 1;
      keys[i] = ((unsigned long long)(~__float_as_uint(s)) << 32) |
                ((unsigned long long)k << 24) | (unsigned long long)b;
    } else {
      keys[i] = ~0ull;  // padding sorts last
    }
  }
  __syncthreads();
  if (bad) {
    for (int b = tid; b < B; b += kSchedThreads) len[b] = -1;
    if (tid == 0) *theta = __longlong_as_double(0x7ff8000000000000ll);
    return;
  }
  if (merge) keys = merge_runs(keys, csum + kSchedThreads, M, G);
  else sort_keys<E>(keys, Mp2);
  const int lane = tid & 31, warp = tid >> 5;
  // fixed-point values of the sorted S, inclusive prefix sums (chunk per thread)
  const int chunk = (M + kSchedThreads - 1) / kSchedThreads;
  const int c0 = min(M, tid * chunk), c1 = min(M, c0 + chunk);
  unsigned long long run = 0;
  for (int i = c0; i < c1; ++i) {
    const float s = __uint_as_float(~(uint32_t)(keys[i] >> 32));
    run += __float2ull_rz(s * 4294967296.0f);
  }
  // exclusive prefix of the chunk sums over the block: a shuffle scan per warp, then one over
  // the 32 warp totals (integer sums: exact in any order)
  unsigned long long incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long v = __shfl_up_sync(~0u, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) csum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    unsigned long long wt = lane < kSchedThreads / 32 ? csum[lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long v = __shfl_up_sync(~0u, wt, o);
      if (lane >= o) wt += v;
    }
    csum[32 + lane] = wt;  // inclusive over warps
  }
  __syncthreads();
  const unsigned long long before_warp = warp > 0 ? csum[32 + warp - 1] : 0ull;
  __syncthreads();
  csum[tid] = before_warp + incl - run;  // exclusive prefix of this thread's chunk
  __syncthreads();
  // Theta(m) for this thread's m values; m = i + 1 covers the first i + 1 sorted entries
  double bv = -1.0;
  int bm = 0x7fffffff;
  if (tid == 0) {
    bv = sps[B] * (double)B;  // m = 0
    bm = 0;
  }
  run = csum[tid];
  for (int i = c0; i < c1; ++i) {
    const float s = __uint_as_float(~(uint32_t)(keys[i] >> 32));
    run += __float2ull_rz(s * 4294967296.0f);
    const double tau = (double)B + (double)run * 0x1p-32;
    const double th = __dmul_rn(sps[B + i + 1], tau);
    if (th > bv) {
      bv = th;
      bm = i + 1;
    }
  }
  // block argmax, smallest m on ties
  for (int o = 16; o > 0; o >>= 1) {
    const double v2 = __shfl_xor_sync(~0u, bv, o);
    const int m2 = __shfl_xor_sync(~0u, bm, o);
    if (v2 > bv || (v2 == bv && m2 < bm)) {
      bv = v2;
      bm = m2;
    }
  }
  if ((tid & 31) == 0) {
    best_val[tid >> 5] = bv;
    best_m[tid >> 5] = bm;
  }
  __syncthreads();
  if (tid == 0) {
    double v = best_val[0];
    int m = best_m[0];
    for (int w = 1; w < kSchedThreads / 32; ++w)
      if (best_val[w] > v || (best_val[w] == v && best_m[w] < m)) {
        v = best_val[w];
        m = best_m[w];
      }
    best_val[0] = v;
    best_m[0] = m;
    *theta = v;
  }
  __syncthreads();
  const int mstar = best_m[0];
  for (int b = tid; b < B; b += kSchedThreads) len[b] = 0;
  __syncthreads();
  for (int i = tid; i < mstar; i += kSchedThreads) atomicAdd(&len[(int)(keys[i] & 0xFFFFFFu)], 1);
}


// dst[c][r] = src[r][c] through a 32 x 32 shared-memory tile (one padding column, so the
// column-wise reads hit 32 different banks); 32 x 8 threads, four rows each.  The small-batch
// draft kernels read W2 as [V][r]; a caller holding the pages' [r][V] gets it transposed here.
template <typename T>
__global__ void __launch_bounds__(256) transpose_kernel(const T* __restrict__ src, T* __restrict__ dst,
                                                        int rows, int cols) {
  __shared__ T tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    const int r = r0 + ty + i, c = c0 + tx;
    if (r < rows && c < cols) tile[ty + i][tx] = src[(size_t)r * cols + c];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    const int c = c0 + ty + i, r = r0 + tx;
    if (r < rows && c < cols) dst[(size_t)c * rows + r] = tile[tx][ty + i];
  }
}

}  // namespace

cudaError_t launch_confidence(int B, int G, int V, int r, int d, int w_bf16, const void* W1,
                              const void* w, int u_bf16, const void* h, const int32_t* x0,
                              const int32_t* tokens, float* c, float* S, cudaStream_t stream) {
  const int warps = B * G;
  confidence_logits_kernel<<<(warps + 7) / 8, 256, 0, stream>>>(B, G, V, r, d, w_bf16, W1, w,
                                                                 u_bf16, h, x0, tokens, c);
  confidence_finish_kernel<<<(B + 127) / 128, 128, 0, stream>>>(B, G, c, S);
  return cudaGetLastError();
}

cudaError_t launch_tv_label(int N, int V, float T, const float* d, const float* t, float* cstar,
                            float* l1, cudaStream_t stream) {
  tv_label_kernel<<<N, 512, 0, stream>>>(V, 1.f / T, d, t, cstar, l1);
  return cudaGetLastError();
}

cudaError_t launch_prefix_schedule(int B, int G, const float* S, const double* sps, int32_t* len,
                                   double* theta, cudaStream_t stream) {
  const int M = B * G;
  int Mp2 = 2;
  while (Mp2 < M) Mp2 <<= 1;
  // the merge sort needs a second buffer of M keys; without room for it, the bitonic sort
  const int merge = (size_t)(Mp2 + kSchedThreads + M) * 8 <= (size_t)(200 << 10) ? 1 : 0;
  const size_t smem = (size_t)(Mp2 + kSchedThreads + (merge ? M : 0)) * 8;
  // keys per thread for the register sort: Mp2 / 1024, at least 1
  const int E = Mp2 <= kSchedThreads ? 1 : Mp2 / kSchedThreads;
  auto kern = E == 1 ? schedule_kernel<1> : E == 2 ? schedule_kernel<2> : E == 4 ? schedule_kernel<4>
            : E == 8 ? schedule_kernel<8> : E == 16 ? schedule_kernel<16> : nullptr;
  if (!kern) return cudaErrorInvalidValue;  // more than 16384 (b, k) keys
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<1, kSchedThreads, smem, stream>>>(B, G, M, Mp2, merge, S, sps, len, theta);
  return cudaGetLastError();
}

cudaError_t launch_transpose(const void* src, void* dst, int rows, int cols, int es, cudaStream_t stream) {
  const dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32));
  if (es == 2)
    transpose_kernel<uint16_t><<<grid, 256, 0, stream>>>((const uint16_t*)src, (uint16_t*)dst, rows, cols);
  else
    transpose_kernel<uint32_t><<<grid, 256, 0, stream>>>((const uint32_t*)src, (uint32_t*)dst, rows, cols);
  return cudaGetLastError();
}

}  // namespace dspark
