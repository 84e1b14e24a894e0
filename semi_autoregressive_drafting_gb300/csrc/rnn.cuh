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

// One request's recurrent update at step ks, by the NT threads that share barrier 1.
//   s_sm [r]   in: s_{k-1}, out: s_k          e_sm [r]  W1[x_{k-1}] (fp32)
//   u_sm [3r]  scratch                        a_out [r] receives a_k = tanh(o_k)
// Sums run in a fixed order (lane-strided, butterfly, then the partial planes in order).
template <int NT>
__device__ void rnn_row_update(const DraftParams& p, int b, int ks, float* s_sm, const float* e_sm,
                               float* u_sm, float* a_out, int tid) {
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
