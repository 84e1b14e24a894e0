// draft_cc.cu -- persistent CUDA-core draft kernel for small batches (B <= 4).
//
// One semi-autoregressive block of the DSpark sequential head ("DSpark -- paper verification",
// section 1, Eqs 4, 5, 7, 8; "DSpark: Wait It's All Autoregressive?", "A parallel backbone with
// autoregressive sampling": the serial loop is a lookup, a small projection, an addition and
// sampling).  At small B the bias product W1[x] W2^T is a GEMV bound by memory, so it stays on
// the CUDA cores.  Design (one cooperative launch for the whole block of gamma steps):
//   * one thread block per SM owns a contiguous vocab slice [v0, v1) for all steps; its W2 rows
//     are one contiguous block of memory, streamed through a ring of TMA bulk-copy stages by a
//     dedicated producer warp (full/empty mbarriers).  The producer does not depend on the
//     sampled tokens, so it runs ahead across step boundaries: the next step's W2 bytes are in
//     flight while the grid agrees on x_k.  W2 is fetched with an L2 evict-last policy, so the
//     steps after the first find it in L2 when it fits;
//   * U_k and target rows of the slice arrive by bulk copy ahead of their step;
//   * stages go round-robin to 8 consumer warps.  A warp takes 32/NB rows at a time, every
//     lane accumulating a 16-byte K-chunk of each row for each request (32 independent sums),
//     then one transposing shuffle reduction leaves lane l with the full dot product of
//     (row l/NB, request l%NB), and every lane fuses +U_k, /T, the online (max, sum-exp), the
//     Gumbel-max update and, with a target, the target's (max, sum-exp);
//   * the Gumbel noise of step k+1 is computed while the block waits at the grid barrier of
//     step k (it does not depend on the tokens);
//   * the grid-wide argmax is one 64-bit atomicMax per (request, block) on an order-independent
//     key; each block also prefetches its candidate's W1 row into L2 so the winner's row is
//     warm when every block gathers it after the barrier;
//   * the Eq 8 label needs both normalisers, so its L1 sum runs right after the barrier from y
//     and target values kept in shared memory.
#include "draft.cuh"

namespace dspark {
namespace {

constexpr int kCWarps = 8;                   // consumer warps
constexpr int kCThreads = kCWarps * 32;      // consumer threads (named barrier 1)
constexpr int kThreads = kCThreads + 32;     // + one producer warp
constexpr int kMaxG = 16;

struct Slot {  // running state of one (request, vocab subset)
  float best;
  uint32_t tok;
  float m, l, mt, lt;
};

struct Misc {
  int cond[4];        // conditioning token of the next step per request
  int valid[4];       // request still valid
  float hdot[kMaxG];  // w[0:d] . h[b][k] for the owned request
  float S_run;        // running prefix survival of the owned request
  float Ld[4], Lt[4];
  float red[kCWarps];
  int flag;
  int last;
  volatile int abort;
};

struct CCLayout {
  size_t ring, ubuf, tbuf, ybuf, gbuf, ebuf, wsm, slots, misc, bars, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline CCLayout cc_layout(const DraftParams& p, int NB) {
  CCLayout L;
  const size_t ues = p.u_bf16 ? 2 : 4;
  const bool tgt = p.target != nullptr;
  size_t off = 0;
  L.ring = off;
  off += (size_t)p.nstages * p.stage_bytes;
  L.ubuf = off;
  off = align_up(off + 2 * NB * (size_t)p.slice_max * ues, 128);
  L.tbuf = off;
  off = align_up(off + (tgt ? 2 * NB * (size_t)p.slice_max * 4 : 0), 128);
  L.ybuf = off;
  off = align_up(off + (tgt ? NB * (size_t)p.slice_max * 4 : 0), 128);
  L.gbuf = off;
  off = align_up(off + (size_t)NB * p.slice_max * 4, 128);
  L.ebuf = off;
  off = align_up(off + (size_t)NB * p.r * 4, 128);
  L.wsm = off;
  off = align_up(off + (size_t)p.r * 4, 128);
  L.slots = off;
  off = align_up(off + kCWarps * 4 * sizeof(Slot), 128);
  L.misc = off;
  off = align_up(off + sizeof(Misc), 128);
  L.bars = off;
  off += (size_t)(2 * p.nstages + 4) * 8;
  L.total = align_up(off, 128);
  return L;
}

// ------------------------------------------------------------------ consumer-only barriers
__device__ __forceinline__ void csync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCThreads) : "memory");
}
__device__ __forceinline__ int csync_or(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "n"(kCThreads)
      : "memory");
  return r;
}
// grid barrier among the consumer threads of every block (the producer warp never takes part)
__device__ __forceinline__ void c_grid_arrive(WsHeader* hdr) {
  csync();
  if (threadIdx.x == 0) {
    __threadfence();
    red_release_add(&hdr->arrive, 1u);
  }
}
__device__ __forceinline__ bool c_grid_wait(WsHeader* hdr, unsigned n, int* s_flag) {
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned target = n * gridDim.x;
    if (ld_acquire(&hdr->arrive) < target) {
      const unsigned long long t0 = globaltimer();
      while (ld_acquire(&hdr->arrive) < target) {
        if (globaltimer() - t0 > kWaitLimitNs) {
          ok = 0;
          break;
        }
        __nanosleep(20);
      }
    }
    __threadfence();
    *s_flag = ok;
  }
  csync();
  return *s_flag != 0;
}

// bounded mbarrier wait that also gives up when the consumers abort
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity,
                                                   volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort || globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// Sum 32 values per lane across the warp: lane l ends with the total of value index l.
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const int c = 32 >> step;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < c / 2; ++i) {
      const float send = upper ? v[i] : v[i + c / 2];
      const float keep = upper ? v[i + c / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
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

// Gumbel noise of one step for this block's slice: one Philox call per 4 vocab entries.
template <int NB>
__device__ __forceinline__ void fill_noise(float* gbuf, int SLM, int SL, int v0, int B, int ks,
                                           uint32_t s_lo, uint32_t s_hi, int tid, int nthr) {
  const int nq = (SL + 3) >> 2;
  for (int i = tid; i < NB * nq; i += nthr) {
    const int b = i / nq, q = i - b * nq;
    if (b >= B) continue;
    const int v = v0 + 4 * q;  // v0 is a multiple of 8: one counter covers v .. v+3
    const U4 r4 = philox4x32_10((uint32_t)(v >> 2), (uint32_t)ks, (uint32_t)b, kNoiseTag, s_lo, s_hi);
    const uint32_t w[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (4 * q + j < SL) gbuf[(size_t)b * SLM + 4 * q + j] = gumbel_from_uniform(bits_to_uniform(w[j]));
  }
}

__device__ __forceinline__ void slot_init(Slot& s) {
  s.best = -INFINITY;
  s.tok = 0xFFFFFFFFu;
  s.m = -INFINITY;
  s.l = 0.f;
  s.mt = -INFINITY;
  s.lt = 0.f;
}
__device__ __forceinline__ void slot_merge(Slot& a, const Slot& q) {
  best_merge(a.best, a.tok, q.best, q.tok);
  lse_merge(a.m, a.l, q.m, q.l);
  lse_merge(a.mt, a.lt, q.mt, q.lt);
}
__device__ __forceinline__ Slot slot_shfl(const Slot& s, int o) {
  Slot q;
  q.best = __shfl_xor_sync(0xffffffffu, s.best, o);
  q.tok = __shfl_xor_sync(0xffffffffu, s.tok, o);
  q.m = __shfl_xor_sync(0xffffffffu, s.m, o);
  q.l = __shfl_xor_sync(0xffffffffu, s.l, o);
  q.mt = __shfl_xor_sync(0xffffffffu, s.mt, o);
  q.lt = __shfl_xor_sync(0xffffffffu, s.lt, o);
  return q;
}

template <typename WT, int NB, int NCV>
__global__ void __launch_bounds__(kThreads, 1) draft_cc_kernel(const DraftParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const CCLayout Lay = cc_layout(p, NB);
  uint8_t* ring = smem + Lay.ring;
  uint8_t* ubuf = smem + Lay.ubuf;
  float* tbuf = (float*)(smem + Lay.tbuf);
  float* ybuf = (float*)(smem + Lay.ybuf);
  float* gbuf = (float*)(smem + Lay.gbuf);
  float* ebuf = (float*)(smem + Lay.ebuf);
  float* wsm = (float*)(smem + Lay.wsm);
  Slot* slots = (Slot*)(smem + Lay.slots);
  Misc* ms = (Misc*)(smem + Lay.misc);
  uint64_t* full = (uint64_t*)(smem + Lay.bars);
  uint64_t* empty = full + p.nstages;
  uint64_t* ufull = empty + p.nstages;
  uint64_t* uempty = ufull + 2;

  constexpr int VEC = Vec<WT>::N;
  constexpr int SR = 32 / NB;  // rows per super-group: SR rows x NB requests = 32 sums
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
  const int R = p.stage_bytes / row_bytes;  // rows per stage, a multiple of 32
  const int NS = p.nstages;
  const int nst = (SL + R - 1) / R;
  const int total = G * nst;
  const bool ubulk = p.u_bulk && SL > 0;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ufull[i], 1);
      mbar_init(&uempty[i], 1);
    }
    fence_mbar_init();
    ms->S_run = 1.f;
    ms->abort = 0;
  }
  if (tid < 4) {
    const int b = tid;
    const int x = b < B ? p.x0[b] : 0;
    const bool ok = b < B && x >= 0 && x < V;
    ms->cond[b] = ok ? x : 0;
    ms->valid[b] = ok;
    if (b < B && !ok) atomicMax(&hdr->status, kErrInvalid);
  }
  __syncthreads();  // the last block-wide barrier: from here the producer warp runs on its own

  // =========================================================== producer warp
  if (warp == kCWarps) {
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_w = policy_evict_last();  // W2 is re-read every step: keep it in L2
      int issued = 0, u_issued = 0;
      bool stop = false;
      for (int g = 0; g < total && !stop; ++g) {
        const int ks = g / nst, s = g - ks * nst;
        if (s == 0 && ubulk) {  // U_k (and target) rows of step ks
          const int buf = ks & 1;
          if (ks >= 2 &&
              !mbar_wait_or_abort(&uempty[buf], (uint32_t)(((ks - 2) >> 1) & 1), &ms->abort)) {
            stop = true;
            break;
          }
          mbar_expect_tx(&ufull[buf], (uint32_t)(B * SL * ues + (tgt ? B * SL * 4 : 0)));
          for (int b = 0; b < B; ++b) {
            bulk_g2s(ubuf + ((size_t)(buf * NB + b) * SLM) * ues,
                     (const uint8_t*)p.U + (((size_t)b * G + ks) * V + v0) * ues,
                     (uint32_t)(SL * ues), &ufull[buf], pol_stream);
            if (tgt)
              bulk_g2s(tbuf + (size_t)(buf * NB + b) * SLM,
                       p.target + ((size_t)b * G + ks) * V + v0, (uint32_t)(SL * 4), &ufull[buf],
                       pol_stream);
          }
          u_issued = ks + 1;
        }
        const int slot = g % NS;
        if (g >= NS &&
            !mbar_wait_or_abort(&empty[slot], (uint32_t)(((g - NS) / NS) & 1), &ms->abort)) {
          stop = true;
          break;
        }
        const int rows = min(R, SL - s * R);
        const uint32_t bytes = (uint32_t)(rows * row_bytes);
        mbar_expect_tx(&full[slot], bytes);
        bulk_g2s(ring + (size_t)slot * p.stage_bytes,
                 (const uint8_t*)p.W2 + (size_t)(v0 + s * R) * row_bytes, bytes, &full[slot], pol_w);
        issued = g + 1;
      }
      if (stop) atomicMax(&hdr->status, kErrTimeout);
      // every copy this warp started must land before the block may exit
      for (int g = max(0, issued - NS); g < issued; ++g)
        mbar_wait(&full[g % NS], (uint32_t)((g / NS) & 1));
      for (int k = max(0, u_issued - 2); k < u_issued; ++k)
        mbar_wait(&ufull[k & 1], (uint32_t)((k >> 1) & 1));
    }
    return;
  }

  // =========================================================== consumer warps
  // Eq 7 inputs of the owned request (request b is owned by block b): the hidden half
  // w[0:d].h[b][k] for every k, and w[d:d+r] kept in shared memory for the per-step half.
  if (conf && cta < B) {
    for (int j = tid; j < r; j += kCThreads) wsm[j] = to_f<WT>(((const WT*)p.w)[p.d + j]);
    for (int k = warp; k < G; k += kCWarps) {
      const size_t base = ((size_t)cta * G + k) * p.d;
      float acc = 0.f;
#pragma unroll 4
      for (int j = lane; j < p.d; j += 32)
        acc += to_f<WT>(((const WT*)p.w)[j]) * ld_act(p.h, base + j, p.u_bf16);
      acc = warp_sum(acc);
      if (lane == 0) ms->hdot[k] = acc;
    }
  }
  fill_noise<NB>(gbuf, SLM, SL, v0, B, 0, p.seed_lo, p.seed_hi, tid, kCThreads);

  bool failed = false;
  const int jrow = lane / NB, bq = lane % NB;  // this lane's (row, request) in a super-group

  for (int ks = 0; ks < G; ++ks) {
    const int buf = ks & 1;
    // (a) conditioning vectors e_b = W1[x_{k-1}] (Eq 5 lookup), fp32 in shared memory
    for (int i = tid; i < NB * r; i += kCThreads) {
      const int b = i / r, j = i - b * r;
      float val = 0.f;
      if (b < B && ms->valid[b]) val = to_f<WT>(((const WT*)p.W1)[(size_t)ms->cond[b] * r + j]);
      ebuf[i] = val;
    }
    csync();
    // (b) Eq 7 and the prefix survival for the owned request (shared memory only)
    if (conf && cta < B && warp == 0) {
      float acc = 0.f;
      for (int j = lane; j < r; j += 32) acc += wsm[j] * ebuf[cta * r + j];
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
    // (c) this lane's K-chunks of every e_b in registers
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
    if (ubulk) {
      const bool ok = mbar_wait(&ufull[buf], (uint32_t)((ks >> 1) & 1));
      if (csync_or(!ok)) {
        failed = true;
        break;
      }
    } else if (SL > 0) {
      for (int i = tid; i < B * SL; i += kCThreads) {
        const int b = i / SL, vl = i - b * SL;
        const size_t src = ((size_t)b * G + ks) * V + v0 + vl;
        if (p.u_bf16)
          ((uint16_t*)ubuf)[(size_t)(buf * NB + b) * SLM + vl] = ((const uint16_t*)p.U)[src];
        else
          ((float*)ubuf)[(size_t)(buf * NB + b) * SLM + vl] = ((const float*)p.U)[src];
        if (tgt) tbuf[(size_t)(buf * NB + b) * SLM + vl] = p.target[src];
      }
      csync();
    }

    // (e) this warp's stages: bias dot products, logits, sampling, normalisers
    Slot st;
    slot_init(st);
    const uint8_t* ub = ubuf + (size_t)(buf * NB + bq) * SLM * ues;
    const float* tb = tbuf + (size_t)(buf * NB + bq) * SLM;
    const float* gb = gbuf + (size_t)bq * SLM;
    bool wfail = false;
    for (int s = warp; s < nst; s += kCWarps) {
      const int g = ks * nst + s;
      const int slot = g % NS;
      if (!mbar_wait(&full[slot], (uint32_t)((g / NS) & 1))) {
        wfail = true;
        break;
      }
      const int rows = min(R, SL - s * R);
      const uint8_t* stg = ring + (size_t)slot * p.stage_bytes;
      for (int r0 = 0; r0 < rows; r0 += SR) {
        float part[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) part[i] = 0.f;
#pragma unroll
        for (int t = 0; t < NCV; ++t) {
          const int cv = lane + 32 * t;
          if (cv < VR) {
#pragma unroll
            for (int j = 0; j < SR; ++j) {
              if (r0 + j < rows) {
                const uint4 q = *(const uint4*)(stg + (size_t)(r0 + j) * row_bytes + cv * 16);
                float wv[VEC];
                Vec<WT>::unpack(q, wv);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                  float a0 = part[j * NB + b], a1 = 0.f;
#pragma unroll
                  for (int i = 0; i < VEC; i += 2) {
                    a0 = fmaf(wv[i], ereg[b][t][i], a0);
                    a1 = fmaf(wv[i + 1], ereg[b][t][i + 1], a1);
                  }
                  part[j * NB + b] = a0 + a1;
                }
              }
            }
          }
        }
        const float bias = transpose_reduce32(part, lane);
        const int row = r0 + jrow;
        if (bq < B && row < rows) {
          const int vl = s * R + row;
          const int v = v0 + vl;
          const float uval = p.u_bf16 ? __uint_as_float((uint32_t)((const uint16_t*)ub)[vl] << 16)
                                      : ((const float*)ub)[vl];
          const float z = uval + bias;
          if (p.logits) p.logits[((size_t)bq * G + ks) * V + v] = z;
          const float y = z * p.invT;
          lse_push(st.m, st.l, y);
          const float sc = y + gb[vl];
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
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (csync_or(wfail)) {
      failed = true;
      break;
    }

    // (f) merge lanes of the same request (fixed butterfly), then warps in a fixed order
#pragma unroll
    for (int o = NB; o < 32; o <<= 1) {
      const Slot q = slot_shfl(st, o);
      slot_merge(st, q);
    }
    if (lane < NB) slots[warp * 4 + lane] = st;
    csync();
    if (tid < B) {
      const int b = tid;
      Slot a;
      slot_init(a);
      for (int w = 0; w < kCWarps; ++w) slot_merge(a, slots[w * 4 + b]);
      if (SL > 0 && ms->valid[b]) {
        atomicMax(&p.keys[(size_t)ks * B + b], make_key(a.best, a.tok));
        // if this block's candidate wins, every block gathers its W1 row next: warm L2 now
        prefetch_l2((const uint8_t*)p.W1 + (size_t)a.tok * row_bytes, (uint32_t)row_bytes);
      }
      p.ml[((size_t)ks * B + b) * nCTA + cta] = make_float2(a.m, a.l);
      if (tgt) p.mlt[((size_t)ks * B + b) * nCTA + cta] = make_float2(a.mt, a.lt);
    }

    // (g) every block has published step ks; the next step's noise is made while waiting
    c_grid_arrive(hdr);
    if (ks + 1 < G) fill_noise<NB>(gbuf, SLM, SL, v0, B, ks + 1, p.seed_lo, p.seed_hi, tid, kCThreads);
    if (!c_grid_wait(hdr, (unsigned)(ks + 1), &ms->flag)) {
      failed = true;
      break;
    }

    // (h) x_k and the next conditioning token
    if (tid < B) {
      const int b = tid;
      const bool was_valid = ms->valid[b];
      const int xk = was_valid ? (int)key_token(ld_acquire64(&p.keys[(size_t)ks * B + b])) : -1;
      int nxt = p.forced ? p.forced[(size_t)b * G + ks] : xk;
      const bool ok = was_valid && nxt >= 0 && nxt < V;
      if (was_valid && !ok && cta == 0) atomicMax(&hdr->status, kErrInvalid);
      ms->cond[b] = ok ? nxt : 0;
      ms->valid[b] = ok;
      if (cta == b) p.tokens[(size_t)b * G + ks] = was_valid ? xk : -1;
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
      csync();
      for (int b = 0; b < B; ++b) {
        const float Ld = ms->Ld[b], Lt = ms->Lt[b];
        float acc = 0.f;
        for (int vl = tid; vl < SL; vl += kCThreads)
          acc += fabsf(__expf(ybuf[(size_t)b * SLM + vl] - Ld) -
                       __expf(tbuf[(size_t)(buf * NB + b) * SLM + vl] * p.invT - Lt));
        acc = warp_sum(acc);
        if (lane == 0) ms->red[warp] = acc;
        csync();
        if (tid == 0) {
          float s = 0.f;
          for (int w = 0; w < kCWarps; ++w) s += ms->red[w];
          p.l1p[((size_t)ks * B + b) * nCTA + cta] = s;
        }
        csync();
      }
    }
    csync();
    // (i) U/target buffer `buf` is free again for step ks + 2
    if (ubulk && tid == 0) mbar_arrive(&uempty[buf]);
  }

  if (failed) {
    // unwind: stop the producer (it drains its own copies), record the timeout
    ms->abort = 1;
    if (tid == 0) atomicMax(&hdr->status, kErrTimeout);
    return;
  }

  // the owned request's log-normalisers, and Eq 8 of every step but the last (whose partial
  // sums are complete only once every block is done): one warp per step
  if (cta < B) {
    const int b = cta;
    for (int k = warp; k < G; k += kCWarps) {
      const float2 ml = warp_merge_ml(p.ml + ((size_t)k * B + b) * nCTA, nCTA, lane);
      const bool vb = p.tokens[(size_t)b * G + k] >= 0;
      if (lane == 0) p.lse[(size_t)b * G + k] = vb ? ml.x + logf(ml.y) : NAN;
      if (tgt && k + 1 < G) {
        const float s = warp_sum_strided(p.l1p + ((size_t)k * B + b) * nCTA, nCTA, lane);
        if (lane == 0) {
          const size_t o = (size_t)b * G + k;
          p.l1[o] = vb ? s : NAN;
          p.cstar[o] = vb ? fminf(1.f, fmaxf(0.f, 1.f - 0.5f * s)) : NAN;
        }
      }
    }
  }

  // last block out: Eq 8 of the final step, then leave the workspace ready for the next call
  csync();
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&hdr->exit_count, 1u);
    ms->last = (old == (unsigned)nCTA - 1u);
  }
  csync();
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
    for (int i = tid; i < G * B; i += kCThreads) p.keys[i] = 0ull;
    csync();
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

// Ring geometry: stages of at least 16 KB holding a multiple of 32 W2 rows, as many stages as
// the shared memory left after the per-step buffers allows (at most 16).
bool draft_cc_configure(DraftParams& p, size_t smem_optin) {
  const int row_bytes = p.r * (p.w_bf16 ? 2 : 4);
  int rows = 16384 / row_bytes;
  rows = rows < 32 ? 32 : rows / 32 * 32;
  p.stage_bytes = rows * row_bytes;
  p.nstages = 0;
  const size_t base = cc_layout(p, nb_of(p.B)).total;
  const size_t avail = smem_optin > base + 64 ? smem_optin - base - 64 : 0;
  p.nstages = (int)(avail / ((size_t)p.stage_bytes + 16));
  if (p.nstages > 16) p.nstages = 16;
  if (p.nstages < 2) return false;
  p.smem_bytes = cc_layout(p, nb_of(p.B)).total;
  return p.smem_bytes <= smem_optin;
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
