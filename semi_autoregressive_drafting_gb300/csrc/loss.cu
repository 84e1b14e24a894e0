// loss.cu -- the drafter's training losses (Eqs 9-12) and their gradients.
//
// "DSpark -- paper verification", section 1: for request b and block position k (row j = k - 1),
// p_k = softmax(zd_k / T) (draft), q_k = softmax(zt_k / T) (the frozen target), x*_k the label,
// c_k = sigmoid(l_k) the confidence, w_k = exp(-(k - 1) / gamma):
//   L_ce = -sum_k w_k ln p_k(x*_k)                                    (Eq 9)
//   L_tv =  sum_k w_k ||p_k - q_k||_1                                  (Eq 10)
//   c*_k =  clamp(1 - 1/2 ||p_k - q_k||_1, 0, 1)                       (Eq 8)
//   L_conf = -sum_k w_k [c*_k ln c_k + (1 - c*_k) ln(1 - c_k)]         (Eq 11)
//   L = a_ce L_ce + a_tv L_tv + a_conf L_conf                          (Eq 12)
// with c* held as a label, so the gradients are
//   dL/dzd_v = (w_k / T) (a_ce (p_v - [v == x*]) + a_tv p_v (s_v - sum_u s_u p_u)),
//   s_u = sign(p_u - q_u);  dL/dl_k = a_conf w_k (c_k - c*_k).
//
// Four stream-ordered launches, no waits between thread blocks (all in log2 units, y2 = z / T
// log2 e):
//   1. loss_part_kernel: (max, sum 2^(y2 - max)) of the draft and target rows of every
//      8192-entry chunk, each thread's 2 x 8 sixteen-byte loads issued at once;
//   2. loss_stat_kernel: with the merged normalisers, sum |p - q| and sum s p of every chunk;
//   3. loss_grad_kernel: dL/dzd of every chunk (skipped when not requested);
//   4. loss_final_kernel: one warp per request, one lane per position: c*, the three terms, the
//      confidence gradient, and the per-request sums.
// Each launch reads the rows once: three reads of every logit row and one gradient write.
#include "common.cuh"
#include "kernels.h"

namespace dspark {
namespace {

constexpr int kLChunk = 8192;
constexpr int kLThr = 256;
constexpr int kLPer = kLChunk / 4 / kLThr;  // 16-byte loads per thread and array: 8
constexpr float kL2e = 1.4426950408889634f;
constexpr float kLn2f = 0.6931471805599453f;

__device__ __forceinline__ float ex2l(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void merge_l2(float& m, float& l, float m2, float l2) {
  if (l2 == 0.f) return;
  if (l == 0.f) {
    m = m2;
    l = l2;
    return;
  }
  const float mm = fmaxf(m, m2);
  l = l * ex2l(m - mm) + l2 * ex2l(m2 - mm);
  m = mm;
}

struct LossWs {
  WsHeader* hdr;
  float4* part;  // [rows][nchunk] (m_d, l_d, m_t, l_t) in log2 units
  float2* stat;  // [rows][nchunk] (sum |p - q|, sum s p)
};

__host__ __device__ inline size_t lws_align(size_t x) { return (x + 255) / 256 * 256; }
__host__ __device__ inline size_t lws_layout(int B, int G, int V, size_t* off) {
  const size_t rows = (size_t)B * G, nchunk = (size_t)((V + kLChunk - 1) / kLChunk);
  size_t o = sizeof(WsHeader);
  off[0] = o;
  o = lws_align(o + rows * nchunk * sizeof(float4));
  off[1] = o;
  o = lws_align(o + rows * nchunk * sizeof(float2));
  return o;
}

// both rows' chunk: loads of the draft and target chunks into registers (aligned rows only)
struct Chunk {
  float4 d[kLPer], t[kLPer];
};
// (last: the rows' last read, streamed evict-first; otherwise the lines stay in L2 normally, so
// that the next launch, which starts with the rows this one read last, finds some of them)
template <bool LAST>
__device__ __forceinline__ void load_chunk(Chunk& c, const float* zd, const float* zt, int n4) {
#pragma unroll
  for (int u = 0; u < kLPer; ++u) {
    const int i = (int)threadIdx.x + u * kLThr;
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (LAST) {
      c.d[u] = i < n4 ? __ldcs((const float4*)zd + i) : ninf;
      c.t[u] = i < n4 ? __ldcs((const float4*)zt + i) : ninf;
    } else {
      c.d[u] = i < n4 ? __ldcg((const float4*)zd + i) : ninf;
      c.t[u] = i < n4 ? __ldcg((const float4*)zt + i) : ninf;
    }
  }
}

// warp + block sum of two floats (block of kLThr threads), result in thread 0
__device__ __forceinline__ float2 block_sum2(float a, float b, float2* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float2(a, b);
  __syncthreads();
  float2 s = make_float2(0.f, 0.f);
  if (threadIdx.x == 0)
    for (int w = 0; w < kLThr / 32; ++w) {
      s.x += red[w].x;
      s.y += red[w].y;
    }
  return s;
}

// ------------------------------------------------------------------ 1. partial normalisers
__global__ void __launch_bounds__(kLThr) loss_part_kernel(const float* __restrict__ zd,
                                                          const float* __restrict__ zt, int V,
                                                          float s2, int nchunk, float4* part) {
  __shared__ float4 red[kLThr / 32];
  const long long blk = blockIdx.x, row = blk / nchunk;
  const int ch = (int)(blk % nchunk);
  const int v0 = ch * kLChunk, v1 = min(V, v0 + kLChunk);
  const float* d = zd + row * V;
  const float* t = zt + row * V;
  float md = -INFINITY, ld = 0.f, mt = -INFINITY, lt = 0.f;
  if ((V & 3) == 0) {
    Chunk c;
    load_chunk<false>(c, d + v0, t + v0, (v1 - v0) >> 2);
    float xd = -INFINITY, xt = -INFINITY;
#pragma unroll
    for (int u = 0; u < kLPer; ++u) {
      xd = fmaxf(xd, fmaxf(fmaxf(c.d[u].x, c.d[u].y), fmaxf(c.d[u].z, c.d[u].w)));
      xt = fmaxf(xt, fmaxf(fmaxf(c.t[u].x, c.t[u].y), fmaxf(c.t[u].z, c.t[u].w)));
    }
    if (xd != -INFINITY) {  // (then xt is finite too: the same entries exist)
      md = xd * s2;
      mt = xt * s2;
#pragma unroll
      for (int u = 0; u < kLPer; ++u) {
        ld += ex2l(fmaf(c.d[u].x, s2, -md)) + ex2l(fmaf(c.d[u].y, s2, -md)) +
              ex2l(fmaf(c.d[u].z, s2, -md)) + ex2l(fmaf(c.d[u].w, s2, -md));
        lt += ex2l(fmaf(c.t[u].x, s2, -mt)) + ex2l(fmaf(c.t[u].y, s2, -mt)) +
              ex2l(fmaf(c.t[u].z, s2, -mt)) + ex2l(fmaf(c.t[u].w, s2, -mt));
      }
    }
  } else {
    for (int v = v0 + (int)threadIdx.x; v < v1; v += kLThr) {
      const float yd = d[v] * s2, yt = t[v] * s2;
      merge_l2(md, ld, yd, 1.f);
      merge_l2(mt, lt, yt, 1.f);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float a = __shfl_xor_sync(0xffffffffu, md, o), b = __shfl_xor_sync(0xffffffffu, ld, o);
    const float c2 = __shfl_xor_sync(0xffffffffu, mt, o), e = __shfl_xor_sync(0xffffffffu, lt, o);
    merge_l2(md, ld, a, b);
    merge_l2(mt, lt, c2, e);
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float4(md, ld, mt, lt);
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = -INFINITY, b = 0.f, c2 = -INFINITY, e = 0.f;
    for (int w = 0; w < kLThr / 32; ++w) {
      merge_l2(a, b, red[w].x, red[w].y);
      merge_l2(c2, e, red[w].z, red[w].w);
    }
    part[blk] = make_float4(a, b, c2, e);
  }
}

// the row's log2 normalisers (draft, target) from its chunk partials; every thread
__device__ __forceinline__ float2 row_norms(const float4* part, long long row, int nchunk) {
  float md = -INFINITY, ld = 0.f, mt = -INFINITY, lt = 0.f;
  for (int c0 = 0; c0 < nchunk; c0 += 8) {
    float4 q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      q[j] = c0 + j < nchunk ? part[row * nchunk + c0 + j] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      merge_l2(md, ld, q[j].x, q[j].y);
      merge_l2(mt, lt, q[j].z, q[j].w);
    }
  }
  return make_float2(md + __log2f(ld), mt + __log2f(lt));
}

// The same for one row per warp: lane i merges partials i, i + 32, ..., then a butterfly merge
// (commutative, so every lane ends with the same value).  One round of loads for nchunk <= 32.
__device__ __forceinline__ float2 row_norms_warp(const float4* part, long long row, int nchunk) {
  float md = -INFINITY, ld = 0.f, mt = -INFINITY, lt = 0.f;
  for (int c = (int)(threadIdx.x & 31); c < nchunk; c += 32) {
    const float4 q = part[row * nchunk + c];
    merge_l2(md, ld, q.x, q.y);
    merge_l2(mt, lt, q.z, q.w);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float a = __shfl_xor_sync(0xffffffffu, md, o), b = __shfl_xor_sync(0xffffffffu, ld, o);
    const float c2 = __shfl_xor_sync(0xffffffffu, mt, o), e = __shfl_xor_sync(0xffffffffu, lt, o);
    merge_l2(md, ld, a, b);
    merge_l2(mt, lt, c2, e);
  }
  return make_float2(md + __log2f(ld), mt + __log2f(lt));
}

__device__ __forceinline__ float sgn(float x) { return x > 0.f ? 1.f : (x < 0.f ? -1.f : 0.f); }

// ------------------------------------------------------------------ 2. |p - q| and s p sums
// (the blocks take the chunks in reverse order, so that the first ones read the rows the
// normaliser launch read last, while they are still in L2; LAST: no gradient launch follows)
template <bool LAST>
__global__ void __launch_bounds__(kLThr) loss_stat_kernel(const float* __restrict__ zd,
                                                          const float* __restrict__ zt, int V,
                                                          float s2, int nchunk, LossWs ws) {
  __shared__ float2 red[kLThr / 32];
  const long long blk = (long long)gridDim.x - 1 - blockIdx.x, row = blk / nchunk;
  const int ch = (int)(blk % nchunk);
  const int v0 = ch * kLChunk, v1 = min(V, v0 + kLChunk);
  const float* d = zd + row * V;
  const float* t = zt + row * V;
  const float2 L = row_norms_warp(ws.part, row, nchunk);
  float l1 = 0.f, sp = 0.f;
  auto acc = [&](float a, float b) {
    const float p = ex2l(fmaf(a, s2, -L.x)), q = ex2l(fmaf(b, s2, -L.y));
    l1 += fabsf(p - q);
    sp += sgn(p - q) * p;
  };
  if ((V & 3) == 0) {
    Chunk c;
    load_chunk<LAST>(c, d + v0, t + v0, (v1 - v0) >> 2);
#pragma unroll
    for (int u = 0; u < kLPer; ++u) {  // padding entries are -inf: p = q = 0 adds nothing
      acc(c.d[u].x, c.t[u].x);
      acc(c.d[u].y, c.t[u].y);
      acc(c.d[u].z, c.t[u].z);
      acc(c.d[u].w, c.t[u].w);
    }
  } else {
    for (int v = v0 + (int)threadIdx.x; v < v1; v += kLThr) acc(d[v], t[v]);
  }
  const float2 s = block_sum2(l1, sp, red);
  if (threadIdx.x == 0) ws.stat[blk] = s;
}

// ------------------------------------------------------------------ 3. dL / d draft logits
__global__ void __launch_bounds__(kLThr, 3) loss_grad_kernel(
    const float* __restrict__ zd, const float* __restrict__ zt, const int32_t* __restrict__ lab,
    int G, int V, float s2, float invT, float a_ce, float a_tv, int nchunk, LossWs ws,
    float* __restrict__ grad) {
  const long long blk = blockIdx.x, row = blk / nchunk;
  const int ch = (int)(blk % nchunk);
  const int v0 = ch * kLChunk, v1 = min(V, v0 + kLChunk);
  const float* d = zd + row * V;
  const float* t = zt + row * V;
  const int n4 = (v1 - v0) >> 2;
  Chunk c;
  if ((V & 3) == 0) load_chunk<true>(c, d + v0, t + v0, n4);  // in flight during the totals
  const int lane = (int)(threadIdx.x & 31);
  const int x = lab[row];
  float* g = grad + row * V;
  // every label of the request, one lane each (an invalid one makes all its outputs NaN)
  const long long j0 = row - row % G;
  const int lj = lane < G ? lab[j0 + lane] : 0;
  const bool ok = __all_sync(0xffffffffu, lj >= 0 && lj < V);
  if (!ok) {  // invalid request: NaN gradient (the final kernel reports it)
    for (int v = v0 + (int)threadIdx.x; v < v1; v += kLThr) g[v] = NAN;
    return;
  }
  const float2 L = row_norms_warp(ws.part, row, nchunk);
  float S = 0.f;  // sum s p over the row: lane-strided, then a butterfly (the same in every lane)
  for (int ch2 = lane; ch2 < nchunk; ch2 += 32) S += ws.stat[row * nchunk + ch2].y;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  const int k0 = (int)(row % G);  // position k - 1
  const float wT = __expf(-(float)k0 / (float)G) * invT;
  auto gv = [&](float a, float b, int v) {
    const float p = ex2l(fmaf(a, s2, -L.x)), q = ex2l(fmaf(b, s2, -L.y));
    return wT * (a_ce * (p - (v == x ? 1.f : 0.f)) + a_tv * p * (sgn(p - q) - S));
  };
  if ((V & 3) == 0) {
#pragma unroll
    for (int u = 0; u < kLPer; ++u) {
      const int i = (int)threadIdx.x + u * kLThr;
      if (i < n4) {
        const int v = v0 + 4 * i;
        __stcs((float4*)(g + v), make_float4(gv(c.d[u].x, c.t[u].x, v), gv(c.d[u].y, c.t[u].y, v + 1),
                                             gv(c.d[u].z, c.t[u].z, v + 2), gv(c.d[u].w, c.t[u].w, v + 3)));
      }
    }
  } else {
    for (int v = v0 + (int)threadIdx.x; v < v1; v += kLThr) g[v] = gv(d[v], t[v], v);
  }
}

// ------------------------------------------------------------------ 4. per-request totals
__global__ void __launch_bounds__(kLThr) loss_final_kernel(
    int B, int G, int V, float s2, const float* __restrict__ zd, const int32_t* __restrict__ lab,
    const float* __restrict__ conf, float a_ce, float a_tv, float a_conf, int nchunk, LossWs ws,
    float* __restrict__ loss, float* __restrict__ parts, float* __restrict__ gconf) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (kLThr / 32) + (threadIdx.x >> 5);
  if (b >= B) return;
  float ce = 0.f, tv = 0.f, cf = 0.f;
  bool ok = true;
  if (lane < G) {
    const long long row = (long long)b * G + lane;
    const int x = lab[row];
    ok = x >= 0 && x < V;
    if (ok) {
      const float2 L = row_norms(ws.part, row, nchunk);
      float l1 = 0.f;
      for (int c = 0; c < nchunk; ++c) l1 += ws.stat[row * nchunk + c].x;
      const float w = __expf(-(float)lane / (float)G);
      const float cstar = fminf(1.f, fmaxf(0.f, 1.f - 0.5f * l1));
      const float l = conf[row];
      // ln c = -softplus(-l), ln(1 - c) = -softplus(l)
      const float sp1 = log1pf(__expf(-fabsf(l)));
      const float log_c = -(fmaxf(-l, 0.f) + sp1), log_1mc = -(fmaxf(l, 0.f) + sp1);
      ce = -w * (fmaf(zd[row * V + x], s2, -L.x) * kLn2f);  // -w ln p(x*)
      tv = w * l1;
      cf = -w * (cstar * log_c + (1.f - cstar) * log_1mc);
      if (gconf) gconf[row] = a_conf * w * (1.f / (1.f + __expf(-l)) - cstar);
    }
  }
  const bool all_ok = __all_sync(0xffffffffu, ok);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ce += __shfl_xor_sync(0xffffffffu, ce, o);
    tv += __shfl_xor_sync(0xffffffffu, tv, o);
    cf += __shfl_xor_sync(0xffffffffu, cf, o);
  }
  if (!all_ok) {
    if (lane < G && gconf) gconf[(size_t)b * G + lane] = NAN;
    if (lane == 0) atomicMax(&ws.hdr->status, kErrInvalid);
    ce = tv = cf = NAN;
  }
  if (lane == 0) {
    if (loss) loss[b] = a_ce * ce + a_tv * tv + a_conf * cf;
    if (parts) {
      parts[3 * (size_t)b] = ce;
      parts[3 * (size_t)b + 1] = tv;
      parts[3 * (size_t)b + 2] = cf;
    }
  }
}

}  // namespace

size_t loss_workspace_bytes(int B, int G, int V) {
  size_t off[2];
  return lws_layout(B, G, V, off);
}

cudaError_t launch_loss(int B, int G, int V, float T, const float* zd, const float* zt,
                        const int32_t* lab, const float* conf, float a_ce, float a_tv, float a_conf,
                        float* loss, float* parts, float* grad_z, float* grad_c, void* workspace,
                        cudaStream_t stream) {
  size_t off[2];
  lws_layout(B, G, V, off);
  uint8_t* w = (uint8_t*)workspace;
  LossWs ws;
  ws.hdr = (WsHeader*)w;
  ws.part = (float4*)(w + off[0]);
  ws.stat = (float2*)(w + off[1]);
  const int nchunk = (V + kLChunk - 1) / kLChunk;
  const long long rows = (long long)B * G;
  const float s2 = kL2e / T;
  loss_part_kernel<<<(unsigned)(rows * nchunk), kLThr, 0, stream>>>(zd, zt, V, s2, nchunk, ws.part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (grad_z)
    loss_stat_kernel<false><<<(unsigned)(rows * nchunk), kLThr, 0, stream>>>(zd, zt, V, s2, nchunk, ws);
  else
    loss_stat_kernel<true><<<(unsigned)(rows * nchunk), kLThr, 0, stream>>>(zd, zt, V, s2, nchunk, ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (grad_z) {
    loss_grad_kernel<<<(unsigned)(rows * nchunk), kLThr, 0, stream>>>(zd, zt, lab, G, V, s2, 1.f / T,
                                                                      a_ce, a_tv, nchunk, ws, grad_z);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  loss_final_kernel<<<(B + kLThr / 32 - 1) / (kLThr / 32), kLThr, 0, stream>>>(
      B, G, V, s2, zd, lab, conf, a_ce, a_tv, a_conf, nchunk, ws, loss, parts, grad_c);
  return cudaGetLastError();
}

}  // namespace dspark
