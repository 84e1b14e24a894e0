// draft_cc.cu -- persistent CUDA-core draft kernel for small batches (B <= 4).
//
// One semi-autoregressive block of the DSpark sequential head ("DSpark -- paper verification",
// section 1, Eqs 4, 5, 7, 8; "DSpark: Wait It's All Autoregressive?", "A parallel backbone with
// autoregressive sampling": the serial loop is a lookup, a small projection, an addition and
// sampling).  At small B the bias product W1[x] W2^T is a GEMV bound by HBM, so it stays on
// the CUDA cores:
//   * one thread block per SM owns a contiguous vocab slice [v0, v1) for all gamma steps;
//     its W2 rows form one contiguous block of memory, streamed through a ring of 16 KB TMA
//     bulk-copy stages.  The ring is refilled as soon as a stage is consumed, including across
//     the step boundary, so the next step's W2 bytes are in flight while the grid agrees on x_k;
//   * U_k and the target rows of the slice arrive by bulk copy one step ahead;
//   * each warp reduces 4 vocab rows x NB requests at once with a transposing shuffle
//     reduction, and the owning lane fuses +U_k, /T, the online (max, sum-exp), the Philox
//     Gumbel-max update and, with a target, the target's (max, sum-exp);
//   * the grid-wide argmax is one 64-bit atomicMax per (request, block) on an order-independent
//     key; a bounded grid barrier publishes x_k; the Eq 8 label needs both normalisers, so its
//     L1 sum runs right after the barrier from y and target values kept in shared memory.
#include "draft.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStageBytes = 16384;
constexpr int kMaxG = 16;

struct Slot {  // per owning lane, merged at the end of a step
  float best;
  uint32_t tok;
  float m, l, mt, lt;
};

struct Misc {
  int cond[4];       // conditioning token of the next step per request
  int valid[4];      // request still valid
  int xk[4];         // token sampled at the current step
  float hdot[kMaxG]; // w[0:d] . h[b][k] for the owned request
  float S_run;       // running prefix survival of the owned request
  float Ld[4], Lt[4];
  int flag;
  int last;
};

struct CCLayout {
  size_t ring, ubuf, tbuf, ybuf, ebuf, slots, misc, bars, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline CCLayout cc_layout(const DraftParams& p, int NB) {
  CCLayout L;
  const size_t ues = p.u_bf16 ? 2 : 4;
  const bool tgt = p.target != nullptr;
  size_t off = 0;
  L.ring = off;
  off += (size_t)p.nstages * kStageBytes;
  L.ubuf = off;
  off = align_up(off + 2 * NB * (size_t)p.slice_max * ues, 128);
  L.tbuf = off;
  off = align_up(off + (tgt ? 2 * NB * (size_t)p.slice_max * 4 : 0), 128);
  L.ybuf = off;
  off = align_up(off + (tgt ? NB * (size_t)p.slice_max * 4 : 0), 128);
  L.ebuf = off;
  off = align_up(off + (size_t)NB * p.r * 4, 128);
  L.slots = off;
  off = align_up(off + kWarps * 16 * sizeof(Slot), 128);
  L.misc = off;
  off = align_up(off + sizeof(Misc), 128);
  L.bars = off;
  off += (size_t)(p.nstages + 2) * 8;
  L.total = align_up(off, 128);
  return L;
}

template <int N>
struct Log2 {
  static constexpr int v = 1 + Log2<N / 2>::v;
};
template <>
struct Log2<1> {
  static constexpr int v = 0;
};

// Sum N values per lane across the warp so that lane l ends with the total of value
// index (l >> (5 - log2 N)); every other index lives in another lane.
template <int N>
__device__ __forceinline__ float transpose_reduce(float (&v)[N], int lane) {
  constexpr int L = Log2<N>::v;
#pragma unroll
  for (int step = 0; step < L; ++step) {
    const int o = 16 >> step;
    const int c = N >> step;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < c / 2; ++i) {
      const float send = upper ? v[i] : v[i + c / 2];
      const float keep = upper ? v[i + c / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
#pragma unroll
  for (int o = 16 >> L; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
  return v[0];
}

__device__ __forceinline__ float ld_act(const void* p, size_t i, int bf16) {
  return bf16 ? __bfloat162float(((const __nv_bfloat16*)p)[i]) : ((const float*)p)[i];
}

// (max, sum-exp) of all blocks' partials for one (step, request), merged by one warp in a
// fixed order (deterministic): lane-strided merge, then a butterfly.
__device__ __forceinline__ float2 warp_merge_ml(const float2* part, int n, int lane) {
  float m = -INFINITY, l = 0.f;
  for (int i = lane; i < n; i += 32) {
    const float2 q = part[i];
    lse_merge(m, l, q.x, q.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    lse_merge(m, l, m2, l2);
  }
  return make_float2(m, l);
}

__device__ __forceinline__ float warp_sum_strided(const float* part, int n, int lane) {
  float s = 0.f;
  for (int i = lane; i < n; i += 32) s += part[i];
  return warp_sum(s);
}

template <typename WT, int NB, int NCV>
__global__ void __launch_bounds__(kThreads, 1) draft_cc_kernel(const DraftParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const CCLayout Lay = cc_layout(p, NB);
  uint8_t* ring = smem + Lay.ring;
  uint8_t* ubuf = smem + Lay.ubuf;
  float* tbuf = (float*)(smem + Lay.tbuf);
  float* ybuf = (float*)(smem + Lay.ybuf);
  float* ebuf = (float*)(smem + Lay.ebuf);
  Slot* slots = (Slot*)(smem + Lay.slots);
  Misc* ms = (Misc*)(smem + Lay.misc);
  uint64_t* full = (uint64_t*)(smem + Lay.bars);
  uint64_t* ufull = full + p.nstages;

  constexpr int VEC = Vec<WT>::N;
  constexpr int NV = 4 * NB;            // values per lane in the transposing reduction
  constexpr int LNV = Log2<NV>::v;
  constexpr int OWN_MASK = (32 >> LNV) - 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nCTA = gridDim.x, cta = blockIdx.x;
  const int B = p.B, G = p.gamma, V = p.V, r = p.r;
  const bool tgt = p.target != nullptr;
  const bool conf = p.h != nullptr && p.w != nullptr;
  const int ues = p.u_bf16 ? 2 : 4;
  WsHeader* hdr = p.hdr;

  // vocab slice of this block (boundaries on multiples of 8 entries)
  const int units = (V + 7) >> 3;
  const int v0 = (int)(((long long)units * cta) / nCTA) * 8;
  const int v1 = min(V, (int)(((long long)units * (cta + 1)) / nCTA) * 8);
  const int SL = max(0, v1 - v0);
  const int SLM = p.slice_max;
  const int row_bytes = r * (int)sizeof(WT);
  const int VR = row_bytes / 16;  // 16-byte vectors per W2 row
  const int R = p.rows_per_stage;
  const int NS = p.nstages;
  const int nst = (SL + R - 1) / R;
  const int total = G * nst;
  const uint64_t pol_stream = policy_evict_first();
  const uint64_t pol_w = policy_evict_last();  // W2 is re-read every step: keep it in L2

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
    mbar_init(&ufull[0], 1);
    mbar_init(&ufull[1], 1);
    fence_mbar_init();
    ms->S_run = 1.f;
  }
  if (tid < 4) {
    const int b = tid;
    const int x = b < B ? p.x0[b] : 0;
    const bool ok = b < B && x >= 0 && x < V;
    ms->cond[b] = ok ? x : 0;
    ms->valid[b] = ok;
    if (b < B && !ok) atomicMax(&hdr->status, kErrInvalid);
  }
  __syncthreads();

  auto issue_stage = [&](int g) {
    const int s = g % nst, slot = g % NS;
    const int rows = min(R, SL - s * R);
    const uint32_t bytes = (uint32_t)(rows * row_bytes);
    mbar_expect_tx(&full[slot], bytes);
    bulk_g2s(ring + (size_t)slot * kStageBytes,
             (const uint8_t*)p.W2 + (size_t)(v0 + s * R) * row_bytes, bytes, &full[slot], pol_w);
  };
  auto issue_u = [&](int ks) {
    const int buf = ks & 1;
    const uint32_t bytes = (uint32_t)(B * SL * ues + (tgt ? B * SL * 4 : 0));
    mbar_expect_tx(&ufull[buf], bytes);
    if (SL == 0) return;
    for (int b = 0; b < B; ++b) {
      bulk_g2s(ubuf + ((size_t)(buf * NB + b) * SLM) * ues,
               (const uint8_t*)p.U + (((size_t)b * G + ks) * V + v0) * ues, (uint32_t)(SL * ues),
               &ufull[buf], pol_stream);
      if (tgt)
        bulk_g2s(tbuf + (size_t)(buf * NB + b) * SLM, p.target + ((size_t)b * G + ks) * V + v0,
                 (uint32_t)(SL * 4), &ufull[buf], pol_stream);
    }
  };

  int u_issued = 0, u_waited = 0;  // block-uniform bookkeeping of U/target fills
  if (tid == 0) {
    for (int g = 0; g < min(NS, total); ++g) issue_stage(g);
    if (p.u_bulk) {
      issue_u(0);
      if (G > 1) issue_u(1);
    }
  }
  if (p.u_bulk) u_issued = min(G, 2);

  // Eq 7, hidden half, for the owned request (request b is owned by block b)
  if (conf && cta < B) {
    for (int k = warp; k < G; k += kWarps) {
      const size_t base = ((size_t)cta * G + k) * p.d;
      float acc = 0.f;
      for (int j = lane; j < p.d; j += 32)
        acc += to_f<WT>(((const WT*)p.w)[j]) * ld_act(p.h, base + j, p.u_bf16);
      acc = warp_sum(acc);
      if (lane == 0) ms->hdot[k] = acc;
    }
  }

  int g_next = 0;  // next ring stage to consume (block-uniform)
  bool failed = false;

  for (int ks = 0; ks < G && !failed; ++ks) {
    const int buf = ks & 1;
    // (a) conditioning vectors e_b = W1[x_{k-1}] (Eq 5 lookup), fp32 in shared memory
    for (int i = tid; i < NB * r; i += kThreads) {
      const int b = i / r, j = i - b * r;
      float val = 0.f;
      if (b < B && ms->valid[b]) val = to_f<WT>(((const WT*)p.W1)[(size_t)ms->cond[b] * r + j]);
      ebuf[i] = val;
    }
    __syncthreads();
    // (b) Eq 7 and the prefix survival for the owned request
    if (conf && cta < B && warp == 0) {
      float acc = 0.f;
      for (int j = lane; j < r; j += 32)
        acc += to_f<WT>(((const WT*)p.w)[p.d + j]) * ebuf[cta * r + j];
      acc = warp_sum(acc);
      if (lane == 0) {
        const size_t o = (size_t)cta * G + ks;
        if (ms->valid[cta]) {
          const float cv = sigmoidf_acc(ms->hdot[ks] + acc);
          ms->S_run *= cv;
          p.c[o] = cv;
          p.S[o] = ms->S_run;
        } else {
          p.c[o] = NAN;
          p.S[o] = NAN;
        }
      }
    }
    // (c) this lane's slice of every e_b in registers
    float ereg[NB][NCV][VEC];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int t = 0; t < NCV; ++t) {
        const int cv = lane + 32 * t;
#pragma unroll
        for (int i = 0; i < VEC; ++i) ereg[b][t][i] = cv < VR ? ebuf[b * r + cv * VEC + i] : 0.f;
      }
    // (d) U_k (and target) rows of the slice
    if (p.u_bulk) {
      const bool ok = mbar_wait(&ufull[buf], (uint32_t)((ks >> 1) & 1));
      if (__syncthreads_or(!ok)) {
        failed = true;
        break;
      }
      u_waited = ks + 1;
    } else {
      for (int i = tid; i < B * SL; i += kThreads) {
        const int b = i / SL, vl = i - b * SL;
        const size_t src = ((size_t)b * G + ks) * V + v0 + vl;
        if (p.u_bf16)
          ((uint16_t*)ubuf)[(size_t)(buf * NB + b) * SLM + vl] = ((const uint16_t*)p.U)[src];
        else
          ((float*)ubuf)[(size_t)(buf * NB + b) * SLM + vl] = ((const float*)p.U)[src];
        if (tgt) tbuf[(size_t)(buf * NB + b) * SLM + vl] = p.target[src];
      }
      __syncthreads();
    }

    // (e) stream the slice: bias dot products, logits, sampling, normalisers
    const int idx = lane >> (5 - LNV);
    const bool owner = (lane & OWN_MASK) == 0;
    const int jr = idx / NB, bq = idx % NB;
    Slot st;
    st.best = -INFINITY;
    st.tok = 0xFFFFFFFFu;
    st.m = -INFINITY;
    st.l = 0.f;
    st.mt = -INFINITY;
    st.lt = 0.f;
    const uint8_t* ub = ubuf + (size_t)(buf * NB + bq) * SLM * ues;
    const float* tb = tbuf + (size_t)(buf * NB + bq) * SLM;
    for (int s = 0; s < nst; ++s) {
      const int g = g_next;
      const int slot = g % NS;
      const bool ok = mbar_wait(&full[slot], (uint32_t)((g / NS) & 1));
      if (__syncthreads_or(!ok)) {
        failed = true;
        break;
      }
      const int rows = min(R, SL - s * R);
      const uint8_t* stg = ring + (size_t)slot * kStageBytes;
      for (int grp = warp; grp * 4 < rows; grp += kWarps) {
        float part[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) part[i] = 0.f;
#pragma unroll
        for (int t = 0; t < NCV; ++t) {
          const int cv = lane + 32 * t;
          if (cv < VR) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (grp * 4 + j < rows) {
                const uint4 q = *(const uint4*)(stg + (size_t)(grp * 4 + j) * row_bytes + cv * 16);
                float wv[VEC];
                Vec<WT>::unpack(q, wv);
#pragma unroll
                for (int b = 0; b < NB; ++b)
#pragma unroll
                  for (int i = 0; i < VEC; ++i) part[j * NB + b] = fmaf(wv[i], ereg[b][t][i], part[j * NB + b]);
              }
            }
          }
        }
        const float bias = transpose_reduce<NV>(part, lane);
        const int row = grp * 4 + jr;
        const int v = v0 + s * R + row;
        const U4 q = philox4x32_10((uint32_t)(v >> 2), (uint32_t)ks, (uint32_t)bq, kNoiseTag,
                                   p.seed_lo, p.seed_hi);
        if (owner && bq < B && row < rows) {
          const int vl = v - v0;
          const float uval = p.u_bf16 ? __uint_as_float((uint32_t)((const uint16_t*)ub)[vl] << 16)
                                      : ((const float*)ub)[vl];
          const float z = uval + bias;
          if (p.logits) p.logits[((size_t)bq * G + ks) * V + v] = z;
          const float y = z * p.invT;
          lse_push(st.m, st.l, y);
          const float sc = y + gumbel_from_uniform(bits_to_uniform(pick(q, v & 3)));
          if (sc > st.best) {  // v grows along this lane's sequence: ties keep the smaller v
            st.best = sc;
            st.tok = (uint32_t)v;
          }
          if (tgt) {
            lse_push(st.mt, st.lt, tb[vl] * p.invT);
            ybuf[(size_t)bq * SLM + vl] = y;
          }
        }
      }
      ++g_next;
      __syncthreads();
      if (tid == 0 && g + NS < total) issue_stage(g + NS);
    }
    if (failed) break;

    // (f) block-level merge in a fixed order, then publish this block's candidate
    if (owner) slots[warp * 16 + idx] = st;
    __syncthreads();
    if (tid < B) {
      const int b = tid;
      Slot a;
      a.best = -INFINITY;
      a.tok = 0xFFFFFFFFu;
      a.m = -INFINITY;
      a.l = 0.f;
      a.mt = -INFINITY;
      a.lt = 0.f;
      for (int w = 0; w < kWarps; ++w)
        for (int j = 0; j < 4; ++j) {
          const Slot& q = slots[w * 16 + j * NB + b];
          best_merge(a.best, a.tok, q.best, q.tok);
          lse_merge(a.m, a.l, q.m, q.l);
          lse_merge(a.mt, a.lt, q.mt, q.lt);
        }
      if (SL > 0 && ms->valid[b]) atomicMax(&p.keys[(size_t)ks * B + b], make_key(a.best, a.tok));
      p.ml[((size_t)ks * B + b) * nCTA + cta] = make_float2(a.m, a.l);
      if (tgt) p.mlt[((size_t)ks * B + b) * nCTA + cta] = make_float2(a.mt, a.lt);
    }

    // (g) every block has published step ks
    if (!grid_barrier(hdr, (unsigned)(ks + 1), &ms->flag)) {
      failed = true;
      break;
    }

    // (h) x_k, next conditioning token, per-request outputs of step ks
    if (tid < B) {
      const int b = tid;
      const bool was_valid = ms->valid[b];
      const int xk = was_valid ? (int)key_token(ld_acquire64(&p.keys[(size_t)ks * B + b])) : -1;
      ms->xk[b] = xk;
      int nxt = p.forced ? p.forced[(size_t)b * G + ks] : xk;
      const bool ok = was_valid && nxt >= 0 && nxt < V;
      if (was_valid && !ok && cta == 0) atomicMax(&hdr->status, kErrInvalid);
      ms->cond[b] = ok ? nxt : 0;
      ms->valid[b] = ok;
    }
    if (cta < B && warp == 0) {  // the owned request's token and log-normaliser
      const int b = cta;
      const float2 ml = warp_merge_ml(p.ml + ((size_t)ks * B + b) * nCTA, nCTA, lane);
      if (lane == 0) {
        const int xk = (int)key_token(ld_acquire64(&p.keys[(size_t)ks * B + b]));
        const bool vb = xk >= 0 && xk < V;
        p.tokens[(size_t)b * G + ks] = vb ? xk : -1;
        p.lse[(size_t)b * G + ks] = vb ? ml.x + logf(ml.y) : NAN;
      }
    }
    if (tgt) {
      // Eq 8 second pass over the slice: needs the global normalisers of p^d and p^t
      if (warp < B) {
        const float2 a = warp_merge_ml(p.ml + ((size_t)ks * B + warp) * nCTA, nCTA, lane);
        const float2 t = warp_merge_ml(p.mlt + ((size_t)ks * B + warp) * nCTA, nCTA, lane);
        if (lane == 0) {
          ms->Ld[warp] = a.x + logf(a.y);
          ms->Lt[warp] = t.x + logf(t.y);
        }
      }
      __syncthreads();
      for (int b = 0; b < B; ++b) {
        const float Ld = ms->Ld[b], Lt = ms->Lt[b];
        float acc = 0.f;
        for (int vl = tid; vl < SL; vl += kThreads)
          acc += fabsf(__expf(ybuf[(size_t)b * SLM + vl] - Ld) -
                       __expf(tbuf[(size_t)(buf * NB + b) * SLM + vl] * p.invT - Lt));
        acc = warp_sum(acc);
        if (lane == 0) slots[warp].best = acc;
        __syncthreads();
        if (tid == 0) {
          float s = 0.f;
          for (int w = 0; w < kWarps; ++w) s += slots[w].best;
          p.l1p[((size_t)ks * B + b) * nCTA + cta] = s;
        }
        __syncthreads();
      }
      // the previous step's partial L1 sums are complete: the owner finishes Eq 8
      if (ks > 0 && cta < B && warp == 0) {
        const float s = warp_sum_strided(p.l1p + ((size_t)(ks - 1) * B + cta) * nCTA, nCTA, lane);
        if (lane == 0) {
          const size_t o = (size_t)cta * G + ks - 1;
          const bool vb = p.tokens[o] >= 0;
          p.l1[o] = vb ? s : NAN;
          p.cstar[o] = vb ? fminf(1.f, fmaxf(0.f, 1.f - 0.5f * s)) : NAN;
        }
      }
    }
    __syncthreads();
    // (i) U/target buffer `buf` is free again: fetch step ks + 2 into it
    if (p.u_bulk && ks + 2 < G) {
      if (tid == 0) issue_u(ks + 2);
      u_issued = ks + 3;
    }
  }

  if (failed) {
    // unwind: record the timeout, wait (bounded) for this block's copies still in flight
    if (tid == 0) {
      atomicMax(&hdr->status, kErrTimeout);
      const int g_end = min(total, g_next + NS);
      for (int g = g_next; g < g_end; ++g) mbar_wait(&full[g % NS], (uint32_t)((g / NS) & 1));
      for (int k = u_waited; k < u_issued; ++k) mbar_wait(&ufull[k & 1], (uint32_t)((k >> 1) & 1));
    }
    __syncthreads();
    return;
  }

  // last block out: Eq 8 of the final step, then leave the workspace ready for the next call
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&hdr->exit_count, 1u);
    ms->last = (old == (unsigned)nCTA - 1u);
  }
  __syncthreads();
  if (ms->last) {
    __threadfence();
    if (tgt && warp < B) {
      const int b = warp;
      const float s = warp_sum_strided(p.l1p + ((size_t)(G - 1) * B + b) * nCTA, nCTA, lane);
      if (lane == 0) {
        const size_t o = (size_t)b * G + G - 1;
        const bool vb = ((volatile int32_t*)p.tokens)[o] >= 0;
        p.l1[o] = vb ? s : NAN;
        p.cstar[o] = vb ? fminf(1.f, fmaxf(0.f, 1.f - 0.5f * s)) : NAN;
      }
    }
    for (int i = tid; i < G * B; i += kThreads) p.keys[i] = 0ull;
    __syncthreads();
    if (tid == 0) {
      hdr->arrive = 0;
      hdr->exit_count = 0;
      __threadfence();
    }
  }
}

template <typename WT, int NB, int NCV>
cudaError_t launch_t(DraftParams& p, int nblocks, cudaStream_t stream) {
  auto kern = draft_cc_kernel<WT, NB, NCV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)p.smem_bytes);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&p};
  return cudaLaunchCooperativeKernel((const void*)kern, dim3(nblocks), dim3(kThreads), args,
                                     p.smem_bytes, stream);
}

template <typename WT, int NCV>
cudaError_t launch_nb(DraftParams& p, int nblocks, cudaStream_t stream) {
  if (p.B <= 1) return launch_t<WT, 1, NCV>(p, nblocks, stream);
  if (p.B <= 2) return launch_t<WT, 2, NCV>(p, nblocks, stream);
  return launch_t<WT, 4, NCV>(p, nblocks, stream);
}

int nb_of(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : 4; }

}  // namespace

int draft_cc_supported(int B, int r, int w_bf16) {
  const int row_bytes = r * (w_bf16 ? 2 : 4);
  return B >= 1 && B <= 4 && row_bytes % 16 == 0 && row_bytes <= 1024;
}

size_t draft_cc_smem_bytes(const DraftParams& p) { return cc_layout(p, nb_of(p.B)).total; }

cudaError_t launch_draft_cc(DraftParams& p, int nblocks, cudaStream_t stream) {
  const int row_bytes = p.r * (p.w_bf16 ? 2 : 4);
  const int ncv = row_bytes / 16 > 32 ? 2 : 1;
  if (p.w_bf16)
    return ncv == 1 ? launch_nb<__nv_bfloat16, 1>(p, nblocks, stream)
                    : launch_nb<__nv_bfloat16, 2>(p, nblocks, stream);
  return ncv == 1 ? launch_nb<float, 1>(p, nblocks, stream) : launch_nb<float, 2>(p, nblocks, stream);
}

}  // namespace dspark
