// rnn.cuh -- the sequential part of the RNN head (Eq 6, "DSpark -- paper verification",
// section 1; split order from the delta table, D8):
//   z_k = [s_{k-1}; W1[x_{k-1}]; h_k],  (g; c; o) = Wj z_k  (rows [gate; candidate; output]),
//   s_k = sigmoid(g) * s_{k-1} + (1 - sigmoid(g)) * tanh(c),   a_k = tanh(o),
// and B_k = a_k . W2^T is then formed like the Markov bias with a_k in place of W1[x_{k-1}].
// The h_k columns of Wj z_k were computed for all (request, position) before the loop by the
// split-K tensor-core GEMM; here one block adds the s and W1 columns for one request.
#pragma once

#include "draft.cuh"

namespace dspark {

template <int NT>
__device__ __forceinline__ void rnn_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

__device__ __forceinline__ float wj_at(const DraftParams& p, size_t i) {
  return p.w_bf16 ? __bfloat162float(((const __nv_bfloat16*)p.Wj)[i]) : ((const float*)p.Wj)[i];
}

// [s; e] part of row i of Wj z_k for rows i0 .. i0+3 of one warp: 16-byte loads of bf16 Wj, fp32
// products against this lane's chunks zc of z (chunk c = columns 8c .. 8c+7, c = lane + 32 t).
template <int CPL>
__device__ __forceinline__ void rnn_rows4(const __nv_bfloat16* W, int width, int i0, int nrows,
                                          int nch, int lane, const float (&zc)[CPL][8],
                                          float (&acc)[4]) {
  uint4 q[4][CPL];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr)
#pragma unroll
    for (int t = 0; t < CPL; ++t) {
      const int c = lane + 32 * t;
      q[rr][t] = (i0 + rr < nrows && c < nch)
                     ? *(const uint4*)(W + (size_t)(i0 + rr) * width + 8 * c)
                     : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int t = 0; t < CPL; ++t) {
      float w[8];
      Vec<__nv_bfloat16>::unpack(q[rr][t], w);
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        a0 = fmaf(w[e], zc[t][e], a0);
        a1 = fmaf(w[e + 1], zc[t][e + 1], a1);
      }
    }
    acc[rr] = a0 + a1;
  }
}

// One request's recurrent update at step ks, by the NT threads that share barrier 1.
//   s_sm [r]   in: s_{k-1}, out: s_k          e_sm [r]  W1[x_{k-1}] (fp32)
//   u_sm [3r]  scratch                        a_out [r] receives a_k = tanh(o_k)
// Sums run in a fixed order: the split-K planes of the h_k part in plane order; the [s; e] part
// lane by lane (two interleaved fp32 chains), then a butterfly across the warp.
template <int NT, int CPL>
__device__ void rnn_row_update_t(const DraftParams& p, int b, int ks, float* s_sm,
                                 const float* e_sm, float* u_sm, float* a_out, int tid) {
  const int r = p.r, width = 2 * r + p.d, nrows = 3 * r;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int NW = NT / 32;
  // the h_k columns, from the pre-pass GEMM's partial planes
  for (int i = tid; i < nrows; i += NT) {
    float gh = 0.f;
    for (int q = 0; q < p.rnn_ks; ++q)
      gh += p.rnn_gh[((size_t)q * p.B * p.gamma + (size_t)b * p.gamma + ks) * nrows + i];
    u_sm[i] = gh;
  }
  // this lane's chunks of z's first 2r columns [s_{k-1}; W1[x_{k-1}]]
  const int nch = r / 4;
  float zc[CPL][8];
#pragma unroll
  for (int t = 0; t < CPL; ++t)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = 8 * (lane + 32 * t) + e;
      zc[t][e] = j < 2 * r ? (j < r ? s_sm[j] : e_sm[j - r]) : 0.f;
    }
  rnn_bar<NT>();
  const __nv_bfloat16* W = (const __nv_bfloat16*)p.Wj;
  for (int i0 = 4 * warp; i0 < nrows; i0 += 4 * NW) {
    float acc[4];
    rnn_rows4<CPL>(W, width, i0, nrows, nch, lane, zc, acc);
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) acc[rr] = warp_sum(acc[rr]);
    if (lane == 0)
#pragma unroll
      for (int rr = 0; rr < 4; ++rr)
        if (i0 + rr < nrows) u_sm[i0 + rr] += acc[rr];
  }
  rnn_bar<NT>();
  for (int j = tid; j < r; j += NT) {
    const float g = sigmoidf_acc(u_sm[j]);
    const float c = tanhf(u_sm[r + j]);
    s_sm[j] = g * s_sm[j] + (1.f - g) * c;
    a_out[j] = tanhf(u_sm[2 * r + j]);
  }
  rnn_bar<NT>();
}

// Scalar form for weights without 16-byte aligned bf16 rows.
template <int NT>
__device__ void rnn_row_update_scalar(const DraftParams& p, int b, int ks, float* s_sm,
                                      const float* e_sm, float* u_sm, float* a_out, int tid) {
  const int r = p.r, width = 2 * r + p.d;
  const int lane = tid & 31, warp = tid >> 5;
  for (int i = warp; i < 3 * r; i += NT / 32) {
    const size_t row = (size_t)i * width;
    float acc = 0.f;
    for (int j = lane; j < 2 * r; j += 32) acc += wj_at(p, row + j) * (j < r ? s_sm[j] : e_sm[j - r]);
    acc = warp_sum(acc);
    if (lane == 0) {
      float gh = 0.f;
      for (int q = 0; q < p.rnn_ks; ++q)
        gh += p.rnn_gh[((size_t)q * p.B * p.gamma + (size_t)b * p.gamma + ks) * 3 * r + i];
      u_sm[i] = acc + gh;
    }
  }
  rnn_bar<NT>();
  for (int j = tid; j < r; j += NT) {
    const float g = sigmoidf_acc(u_sm[j]);
    const float c = tanhf(u_sm[r + j]);
    s_sm[j] = g * s_sm[j] + (1.f - g) * c;
    a_out[j] = tanhf(u_sm[2 * r + j]);
  }
  rnn_bar<NT>();
}

template <int NT>
__device__ void rnn_row_update(const DraftParams& p, int b, int ks, float* s_sm, const float* e_sm,
                               float* u_sm, float* a_out, int tid) {
  const bool vec = p.w_bf16 && ((uintptr_t)p.Wj & 15) == 0 && ((2 * p.r + p.d) & 7) == 0;
  if (vec && p.r <= 256) rnn_row_update_t<NT, 2>(p, b, ks, s_sm, e_sm, u_sm, a_out, tid);
  else if (vec && p.r <= 512) rnn_row_update_t<NT, 4>(p, b, ks, s_sm, e_sm, u_sm, a_out, tid);
  else rnn_row_update_scalar<NT>(p, b, ks, s_sm, e_sm, u_sm, a_out, tid);
}

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait until flag == tag; false when the time bound ran out.
__device__ __forceinline__ bool wait_flag(const unsigned* flag, unsigned tag) {
  if (ld_acquire(flag) == tag) return true;
  const unsigned long long t0 = globaltimer();
  while (ld_acquire(flag) != tag) {
    if (globaltimer() - t0 > kWaitLimitNs) return false;
    __nanosleep(32);
  }
  return true;
}

}  // namespace dspark
