// verify.cu -- speculative verification of a draft block: the standard accept/reject rule.
//
// "Phase-Conditioned Speculative Decoding" section 3 identifies Eq 8's c* = 1 - TV(p, q) with
// the single-step acceptance probability of this rule (Leviathan, Kalman, Matias, ICML 2023);
// "DSpark：既要猜得连贯…" ("Why DSpark?") describes the round: the matching prefix is accepted and
// the round stops at the first rejection, and its "Results" count the target's bonus token in
// the accepted length.  For request b, with p_j = softmax(zd[b][j] / T) and
// q_j = softmax(zt[b][j] / T):
//   position j accepts x_j iff ln a_j < ln q_j(x_j) - ln p_j(x_j)  (probability min(1, q/p));
//   at the first rejection j the correction is a Gumbel-max draw from max(0, q_j - p_j) (from
//   q_j when that is zero everywhere); after gamma acceptances the bonus is a draw from q_gamma.
// a_j is word 0 of Philox4x32-10 at counter (0, j, b, 'ACCP'); the draw's noise for entry v is
// word v mod 4 at counter (v / 4, j, b, 'RESD'), with the same key and uniform as the sampler.
//
// Three stream-ordered launches, no waits between thread blocks:
//   1. verify_part_kernel: (max, sum 2^(y2 - max)) of every 16384-entry chunk of every draft and
//      target row, y2 = z log2(e) / T.  Each thread issues all sixteen of its 16-byte streaming
//      loads at once; this is the bulk of the bytes (B (2 gamma + 1) V fp32) and is HBM-bound.
//   2. verify_decide_kernel: one warp per request merges the partials of its rows, takes the
//      gamma accept decisions (one lane per position), and writes the accepted prefix and the
//      normalisers of the row to draw from.
//   3. verify_draw_kernel: one block per (request, 8192-entry chunk) draws over its chunk of that
//      row with the draft sampler's exact skip (the lanes of a warp share their running best:
//      they hold the same row); the blocks of a request combine with an order-independent
//      64-bit atomicMax key, and the last one writes the correction or bonus and resets the key
//      for the next call.
#include "common.cuh"
#include "kernels.h"

namespace dspark {
namespace {

constexpr int kChunk = 16384;     // vocabulary entries per block of kernel 1
constexpr int kDrawChunk = 8192;  // vocabulary entries per block of kernel 3
constexpr int kThr = 256;
constexpr uint32_t kAcceptTag = 0x41434350u;    // "ACCP"
constexpr uint32_t kResidualTag = 0x52455344u;  // "RESD"
constexpr float kLog2eV = 1.4426950408889634f;

__device__ __forceinline__ float ex2v(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// uniform (2 (bits >> 9) + 1) 2^-24, exactly, from the mantissa bits
__device__ __forceinline__ float uni(uint32_t bits) {
  return __uint_as_float(0x3F800000u | (bits >> 9)) - 0.99999994f;
}

// merge (m, l) pairs in log2 units: l = sum 2^(y - m)
__device__ __forceinline__ void merge2(float& m, float& l, float m2, float l2) {
  if (l2 == 0.f) return;
  if (l == 0.f) {
    m = m2;
    l = l2;
    return;
  }
  const float mm = fmaxf(m, m2);
  l = l * ex2v(m - mm) + l2 * ex2v(m2 - mm);
  m = mm;
}

struct VerifyWs {
  WsHeader* hdr;
  float2* part;                // [rows][nchunk]: draft rows b*G + j, then target rows
  int* n;                      // [B] accepted count, -1 for an invalid request
  float2* L;                   // [B] (draft, target) log2 normalisers of the row to draw from
  unsigned long long* keys;    // [B][2] best key of the draw (the second is spare); zero between calls
  unsigned* count;             // [B] blocks of the draw done; zero between calls
};

__host__ __device__ inline size_t vws_align(size_t x) { return (x + 255) / 256 * 256; }

__host__ __device__ inline size_t vws_layout(int B, int G, int V, size_t* off) {
  const int nchunk = (V + kChunk - 1) / kChunk;
  const size_t rows = (size_t)B * (2 * G + 1);
  size_t o = sizeof(WsHeader);
  off[0] = o;  // part
  o = vws_align(o + rows * nchunk * sizeof(float2));
  off[1] = o;  // n
  o = vws_align(o + (size_t)B * sizeof(int));
  off[2] = o;  // L
  o = vws_align(o + (size_t)B * sizeof(float2));
  off[3] = o;  // keys
  o = vws_align(o + (size_t)B * 2 * sizeof(unsigned long long));
  off[4] = o;  // count
  o = vws_align(o + (size_t)B * sizeof(unsigned));
  return o;
}

// ------------------------------------------------------------------ 1. chunk partials
__global__ void __launch_bounds__(kThr) verify_part_kernel(const float* __restrict__ zd,
                                                           const float* __restrict__ zt,
                                                           long long nd_rows, int V, float s2,
                                                           int nchunk, float2* __restrict__ part) {
  __shared__ float2 red[kThr / 32];
  const long long blk = blockIdx.x;
  const long long row = blk / nchunk;
  const int ch = (int)(blk % nchunk);
  const float* z = row < nd_rows ? zd + row * V : zt + (row - nd_rows) * V;
  const int v0 = ch * kChunk, v1 = min(V, v0 + kChunk);
  float m = -INFINITY, l = 0.f;
  if ((V & 3) == 0) {  // rows are 16-byte aligned: the chunk's sixteen loads per thread at once
    const float4* z4 = (const float4*)(z + v0);
    const int n4 = (v1 - v0) >> 2;
    constexpr int kPer = kChunk / 4 / kThr;  // 16
    float4 q[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = (int)threadIdx.x + u * kThr;
      q[u] = i < n4 ? __ldcs(z4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < kPer; ++u) mx = fmaxf(mx, fmaxf(fmaxf(q[u].x, q[u].y), fmaxf(q[u].z, q[u].w)));
    if (mx != -INFINITY) {
      m = mx * s2;  // the scale is positive and rounding monotone: the max of z s2
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        a0 += ex2v(fmaf(q[u].x, s2, -m)) + ex2v(fmaf(q[u].y, s2, -m));
        a1 += ex2v(fmaf(q[u].z, s2, -m)) + ex2v(fmaf(q[u].w, s2, -m));
      }
      l = a0 + a1;
    }
  } else {
    for (int v = v0 + (int)threadIdx.x; v < v1; v += kThr) {
      const float y = z[v] * s2;
      if (y > m) {
        l = l * ex2v(m - y) + 1.f;
        m = y;
      } else {
        l += ex2v(y - m);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), l2 = __shfl_xor_sync(0xffffffffu, l, o);
    merge2(m, l, m2, l2);
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float2(m, l);
  __syncthreads();
  if (threadIdx.x == 0) {
    float mm = -INFINITY, ll = 0.f;
    for (int w = 0; w < kThr / 32; ++w) merge2(mm, ll, red[w].x, red[w].y);
    part[blk] = make_float2(mm, ll);
  }
}

// log2 normaliser of one row from its chunk partials (one thread; eight loads in flight)
__device__ __forceinline__ float row_lse2(const float2* part, long long row, int nchunk) {
  float m = -INFINITY, l = 0.f;
  for (int c0 = 0; c0 < nchunk; c0 += 8) {
    float2 q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      q[j] = c0 + j < nchunk ? part[row * nchunk + c0 + j] : make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) merge2(m, l, q[j].x, q[j].y);
  }
  return m + __log2f(l);
}

// ------------------------------------------------------------------ 2. decisions
__global__ void __launch_bounds__(kThr) verify_decide_kernel(
    int B, int G, int V, float s2, uint32_t seed_lo, uint32_t seed_hi,
    const float* __restrict__ zd, const float* __restrict__ zt, const int32_t* __restrict__ tok,
    VerifyWs ws, int nchunk, int32_t* __restrict__ n_acc, int32_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (kThr / 32) + (threadIdx.x >> 5);
  if (b >= B) return;
  const long long nd_rows = (long long)B * G;
  // lane j < G: position j; lane G also takes the bonus row's target normaliser
  bool ok = true, acc = true;
  float Ld = 0.f, Lt = 0.f;
  if (lane < G) {
    const int x = tok[(size_t)b * G + lane];
    ok = x >= 0 && x < V;
    Ld = row_lse2(ws.part, (long long)b * G + lane, nchunk);
    Lt = row_lse2(ws.part, nd_rows + (long long)b * (G + 1) + lane, nchunk);
    if (ok) {
      // ln a < ln q(x) - ln p(x), in log2 units
      const float lr = (zt[((size_t)b * (G + 1) + lane) * V + x] - zd[((size_t)b * G + lane) * V + x]) * s2 -
                       (Lt - Ld);
      const U4 r = philox4x32_10(0u, (uint32_t)lane, (uint32_t)b, kAcceptTag, seed_lo, seed_hi);
      acc = log2f(uni(r.x)) < lr;
    }
  } else if (lane == G) {
    Lt = row_lse2(ws.part, nd_rows + (long long)b * (G + 1) + G, nchunk);
  }
  const unsigned bad = __ballot_sync(0xffffffffu, lane < G && !ok);
  const unsigned rej = __ballot_sync(0xffffffffu, lane < G && !acc);
  const int n = bad ? -1 : (rej ? __ffs(rej) - 1 : G);
  // the normalisers of row n (the bonus row when n == G)
  const float Ldn = __shfl_sync(0xffffffffu, Ld, n < 0 ? 0 : min(n, G - 1));
  const float Ltn = __shfl_sync(0xffffffffu, Lt, n < 0 ? 0 : n);
  if (lane <= G) {
    const int x = lane < G ? tok[(size_t)b * G + lane] : 0;
    out[(size_t)b * (G + 1) + lane] = (n >= 0 && lane < n) ? x : -1;
  }
  if (lane == 0) {
    ws.n[b] = n;
    ws.L[b] = make_float2(Ldn, Ltn);
    if (n < 0) {
      n_acc[b] = -1;
      atomicMax(&ws.hdr->status, kErrInvalid);
    }
  }
}

// ------------------------------------------------------------------ 3. the draw
// Gumbel-max in log2 units: score = log2 W_v - log2(-ln u_v), W = max(0, q - p) for a
// correction (n < G), W = q for the bonus (n == G).  Exact skip, as in the draft sampler: with
// w = 1 - u (exact from the bits) and -ln u >= w, an entry with w >= 1.002 2^(log2 q_v - tb)
// scores below tb - log2(1.002) (W <= q), where tb is a score some entry of this row has
// reached; f = 1 + w - 2^-24 is read from the bits and compared with fl(1 + 1.002 2^(lq - tb)).
// Only the rare candidates take the logarithms.  The lanes of a warp hold the same row, so tb
// is the warp's running best.
__device__ __forceinline__ float gumbel_l2(uint32_t bits) { return -log2f(-logf(uni(bits))); }

// Philox round keys of the seed (rk0[i] = lo + i 0x9E3779B9, rk1[i] = hi + i 0xBB67AE85), passed
// as a kernel parameter so that the per-call rounds read them from the constant bank
struct RoundKeys {
  uint32_t rk0[10], rk1[10];
};

__global__ void __launch_bounds__(kThr) verify_draw_kernel(
    int B, int G, int V, float s2, uint32_t seed_lo, uint32_t seed_hi, const RoundKeys rk,
    const float* __restrict__ zd, const float* __restrict__ zt, VerifyWs ws, int nchunk,
    int32_t* __restrict__ n_acc, int32_t* __restrict__ out) {
  __shared__ unsigned long long kred[kThr / 32];
  __shared__ unsigned long long s_key;
  __shared__ int s_last;
  const int b = blockIdx.x / nchunk, ch = blockIdx.x % nchunk;
  const int n = ws.n[b];
  if (n < 0) return;  // invalid request: outputs were written by the decisions
  const float2 L = ws.L[b];
  const bool resid = n < G;
  const float* yr = resid ? zd + ((size_t)b * G + n) * V : nullptr;
  const float* tr = zt + ((size_t)b * (G + 1) + n) * V;
  const int v0 = ch * kDrawChunk, v1 = min(V, v0 + kDrawChunk);
  const bool vec = (V & 3) == 0;  // rows 16-byte aligned
  // counter words 1-3 (position, request, stream tag) are fixed for the row: the rounds' parts
  // that do not depend on word 0 (the vocabulary quad) are formed once
  const PhiloxFixed pfx = philox_fix((uint32_t)n, (uint32_t)b, kResidualTag, seed_lo, seed_hi);
  float best = -INFINITY, tb = -INFINITY;
  uint32_t tok = 0xFFFFFFFFu;
  // four consecutive entries per thread and iteration: one Philox call, one 16-byte load of each
  // row when the rows are aligned; the loop count is the same for every lane of the warp
  for (int base = v0; base < v1; base += 4 * kThr) {
    const int v4 = base + 4 * (int)threadIdx.x;
    if (v4 < v1) {
      float tq4[4], yq4[4];
      if (vec) {
        const float4 a = __ldcs((const float4*)(tr + v4));
        tq4[0] = a.x; tq4[1] = a.y; tq4[2] = a.z; tq4[3] = a.w;
        if (resid) {
          const float4 c = __ldcs((const float4*)(yr + v4));
          yq4[0] = c.x; yq4[1] = c.y; yq4[2] = c.z; yq4[3] = c.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          tq4[e] = v4 + e < v1 ? tr[v4 + e] : 0.f;
          yq4[e] = (resid && v4 + e < v1) ? yr[v4 + e] : 0.f;
        }
      }
      const U4 r = philox_var((uint32_t)(v4 >> 2), pfx, rk.rk0, rk.rk1);
      const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int v = v4 + e;
        const float lq = tq4[e] * s2 - L.y;
        const float f = __uint_as_float(0x3F800000u | (~wd[e] >> 9));
        if (v < v1 && f < fmaf(ex2v(lq - tb), 1.002f, 1.f)) {
          float lw = lq;
          if (resid) {
            const float lp = yq4[e] * s2 - L.x;  // q_v > p_v: log2(q - p) = lq + log2(1 - 2^(lp - lq))
            lw = lq > lp ? lq + log1pf(-ex2v(lp - lq)) * kLog2eV : -INFINITY;
          }
          const float sc = lw + gumbel_l2(wd[e]);
          if (sc > best) {
            best = sc;
            tok = (uint32_t)v;
          }
        }
      }
    }
    float wb = best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wb = fmaxf(wb, __shfl_xor_sync(0xffffffffu, wb, o));
    tb = wb;
  }
  // block maximum as an order-independent key (larger score, then smaller entry)
  unsigned long long k = tok == 0xFFFFFFFFu ? 0ull : make_key(best, tok);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long a = __shfl_xor_sync(0xffffffffu, k, o);
    k = a > k ? a : k;
  }
  if ((threadIdx.x & 31) == 0) kred[threadIdx.x >> 5] = k;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThr / 32; ++w) k = kred[w] > k ? kred[w] : k;
    if (k) atomicMax(&ws.keys[2 * b], k);
    __threadfence();
    s_last = atomicAdd(&ws.count[b], 1u) == (unsigned)nchunk - 1u;
    if (s_last) {  // every block of this request has published
      __threadfence();
      s_key = *(volatile unsigned long long*)&ws.keys[2 * b];
    }
  }
  __syncthreads();
  if (!s_last) return;
  unsigned long long f = s_key;  // the same in every thread of the block
  if (resid && f == 0ull) {
    // max(0, q - p) is zero everywhere (p and q agree to the last bit): draw from q instead,
    // over the whole row in this block (a case that the accept test makes all but impossible)
    float bq = -INFINITY;
    uint32_t tq = 0xFFFFFFFFu;
    for (int v = (int)threadIdx.x; v < V; v += kThr) {
      const U4 r = philox4x32_10((uint32_t)(v >> 2), (uint32_t)n, (uint32_t)b, kResidualTag, seed_lo, seed_hi);
      const uint32_t wv = (v & 3) == 0 ? r.x : (v & 3) == 1 ? r.y : (v & 3) == 2 ? r.z : r.w;
      const float sc = tr[v] * s2 - L.y + gumbel_l2(wv);
      if (sc > bq) {
        bq = sc;
        tq = (uint32_t)v;
      }
    }
    unsigned long long kq = tq == 0xFFFFFFFFu ? 0ull : make_key(bq, tq);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long a = __shfl_xor_sync(0xffffffffu, kq, o);
      kq = a > kq ? a : kq;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) kred[threadIdx.x >> 5] = kq;
    __syncthreads();
    if (threadIdx.x == 0)
      for (int w = 0; w < kThr / 32; ++w) f = kred[w] > f ? kred[w] : f;
  }
  if (threadIdx.x == 0) {
    out[(size_t)b * (G + 1) + n] = f ? (int32_t)key_token(f) : -1;
    n_acc[b] = n;
    ws.keys[2 * b] = 0ull;
    ws.count[b] = 0u;
  }
}

}  // namespace

size_t verify_workspace_bytes(int B, int G, int V) {
  size_t off[5];
  return vws_layout(B, G, V, off);
}

cudaError_t launch_verify(int B, int G, int V, float T, uint64_t seed, const float* zd,
                          const float* zt, const int32_t* tok, int32_t* n_acc, int32_t* out,
                          void* workspace, cudaStream_t stream) {
  size_t off[5];
  vws_layout(B, G, V, off);
  uint8_t* w = (uint8_t*)workspace;
  VerifyWs ws;
  ws.hdr = (WsHeader*)w;
  ws.part = (float2*)(w + off[0]);
  ws.n = (int*)(w + off[1]);
  ws.L = (float2*)(w + off[2]);
  ws.keys = (unsigned long long*)(w + off[3]);
  ws.count = (unsigned*)(w + off[4]);
  const int nchunk = (V + kChunk - 1) / kChunk;
  const int ndraw = (V + kDrawChunk - 1) / kDrawChunk;
  const float s2 = kLog2eV / T;
  const uint32_t lo = (uint32_t)(seed & 0xFFFFFFFFu), hi = (uint32_t)(seed >> 32);
  const long long rows = (long long)B * (2 * G + 1);
  verify_part_kernel<<<(unsigned)(rows * nchunk), kThr, 0, stream>>>(zd, zt, (long long)B * G, V, s2,
                                                                     nchunk, ws.part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  verify_decide_kernel<<<(B + kThr / 32 - 1) / (kThr / 32), kThr, 0, stream>>>(
      B, G, V, s2, lo, hi, zd, zt, tok, ws, nchunk, n_acc, out);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  RoundKeys rk;
  for (int i = 0; i < 10; ++i) {
    rk.rk0[i] = lo + (uint32_t)i * 0x9E3779B9u;
    rk.rk1[i] = hi + (uint32_t)i * 0xBB67AE85u;
  }
  verify_draw_kernel<<<(unsigned)((long long)B * ndraw), kThr, 0, stream>>>(B, G, V, s2, lo, hi, rk,
                                                                           zd, zt, ws, ndraw, n_acc,
                                                                           out);
  return cudaGetLastError();
}

}  // namespace dspark
