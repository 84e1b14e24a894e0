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
//   * with 512-byte W2 rows the first 16 stages of the slice are copied into TMEM during the
//     first step and read back from there afterwards, so the producer streams only the rest;
//   * stages go round-robin to the consumer warps (24 for one request, 16 for two, 8 for four).
//     A warp takes 32/NB rows at a time, every lane accumulating a 16-byte K-chunk of each row
//     for each request (bf16 operands go straight into mixed-precision FMAs), then one
//     transposing shuffle reduction leaves lane l with the full dot product of (row l/NB,
//     request l%NB), and the lanes fuse +U_k, /T, the online (max, sum-exp), the Gumbel-max
//     update and, with a target, the target's (max, sum-exp);
//   * the Gumbel noise of step k+1 is computed while the block waits at the grid barrier of
//     step k (it does not depend on the tokens);
//   * grid barrier and argmax in one: each block merges its warps' results (warp reductions)
//     and publishes a step-tagged 64-bit key in its own slot; every block polls all slots, so
//     the barrier completes when the last key lands and its maximum is the drawn token.  Each
//     block also prefetches its candidate's W1 row into L2 so the winner's row is warm when
//     every block gathers it after the barrier.  (Opt-in: clusters of blocks first merge in
//     distributed shared memory and publish one slot per cluster.)
//   * the Eq 8 label needs both normalisers, so its L1 sum runs right after the barrier from y
//     and target values kept in shared memory;
//   * the tensor-core variant (TCV, bf16, B = 3-4) computes the bias with tcgen05 MMAs, the
//     vocabulary rows on M and the B conditioning vectors on N, from an MMA warp.
#include <type_traits>

#include <cstring>

#include "draft.cuh"
#include "rnn.cuh"
#include "tc.cuh"

namespace dspark {
namespace {

constexpr int kMaxCW = 24;  // most consumer warps of any variant

struct Slot {  // running state of one (request, vocab subset)
  float best;
  uint32_t tok;
  float m, l, mt, lt;
};

struct Misc {
  int cond[4];        // conditioning token of the next step per request
  int valid[4];       // request still valid
  float S_run;        // running prefix survival of the owned request
  float Ld[4], Lt[4];
  float red[kMaxCW];
  int flag;
  int last;
  volatile int abort;
  volatile int stage_tag[16];  // which global stage each ring slot currently holds
  uint32_t tmem_base;          // TMEM columns caching the first stages of the slice
  float cbuf[64];              // last block: Eq 7 of every (request, step)
  bool cvalid[64];             // last block: the step's token is valid
  // cluster leader (rank 0): each block's key and (max, sum-exp) partials of p^d and p^t for
  // the current step, per request, written by the blocks of the cluster (the key last, with
  // release semantics; its step tag tells the leader it is there)
  unsigned long long ckey[4][8];
  float2 cml[4][8], cmlt[4][8];
};

struct CCLayout {
  size_t ring, res, ebf, ubuf, tbuf, ybuf, gbuf, ebuf, wsm, rbuf, sbuf, u3, slots, misc, bars, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline CCLayout cc_layout(const DraftParams& p, int NB) {
  CCLayout L;
  const size_t ues = p.u_bf16 ? 2 : 4;
  const bool tgt = p.target != nullptr;
  size_t off = 0;
  L.ring = off;
  off += (size_t)p.nstages * p.stage_bytes;
  // tensor-core variant: resident slabs, then the MMA's B operand (16 rows x r bf16 in the
  // 128-byte swizzle, one 2 KB block per 64 K); all 1024-byte aligned
  L.res = off;
  off += p.tcv ? (size_t)p.nres_s * p.stage_bytes : 0;
  L.ebf = off;
  off += p.tcv ? (size_t)(p.r / 64) * 2048 : 0;
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
  const bool rnn = p.head == 1;
  L.rbuf = off;  // RNN: a_k of every request
  off = align_up(off + (rnn ? (size_t)NB * p.r * 4 : 0), 128);
  L.sbuf = off;  // RNN: the owned request's state s_k
  off = align_up(off + (rnn ? (size_t)p.r * 4 : 0), 128);
  L.u3 = off;    // RNN: the owned request's projection Wj z_k
  off = align_up(off + (rnn ? (size_t)3 * p.r * 4 : 0), 128);
  L.slots = off;
  off = align_up(off + kMaxCW * 4 * sizeof(Slot), 128);
  L.misc = off;
  off = align_up(off + sizeof(Misc), 128);
  L.bars = off;
  // ring full/empty, U full/empty; tensor-core variant: efull, mdone, accfull[32], tready[16],
  // rfull[16]
  off += (size_t)(2 * p.nstages + 4 + (p.tcv ? 2 + 32 + 16 + 16 : 0) + 1) * 8;  // + never
  L.total = align_up(off, 128) + (p.tcv ? 1024 : 0);  // slack to align the base to 1024
  return L;
}

// ------------------------------------------------------------------ consumer-only barriers
template <int NT>
__device__ __forceinline__ void csync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}
template <int NT>
__device__ __forceinline__ int csync_or(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "n"(NT)
      : "memory");
  return r;
}
// barrier of the four warps of consumer group g (named barrier 2 + g, 128 threads), returning
// whether any of them passed a true predicate
__device__ __forceinline__ int gsync_or(int g, int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "r"(2 + g)
      : "memory");
  return r;
}
// grid barrier among the consumer threads of every block (the producer warp never takes part)
template <int NT>
__device__ __forceinline__ void c_grid_arrive(WsHeader* hdr) {
  csync<NT>();
  if (threadIdx.x == 0) {
    __threadfence();
    red_release_add(&hdr->arrive, 1u);
  }
}
template <int NT>
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
  csync<NT>();
  return *s_flag != 0;
}

// bounded mbarrier wait that also gives up when the consumers abort
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity,
                                                   volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) {
    if (*abort || globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// Wait until ring slot `slot` holds stage g and its bytes have landed.  A warp consumes every
// CW-th stage, so it may reach a slot before the slot's previous use has completed; the phase
// parity alone would then be ambiguous, so the producer tags the slot with the stage it holds
// before arming it, and the parity is only read once the tag matches.
__device__ __forceinline__ bool wait_stage(volatile int* tag, uint64_t* full, int slot, int g,
                                           int NS) {
  if (tag[slot] != g) {
    const unsigned long long t0 = globaltimer();
    while (tag[slot] != g) {
      if (globaltimer() - t0 > kWaitLimitNs) return false;
      __nanosleep(32);
    }
  }
  return mbar_wait(full + slot, (uint32_t)((g / NS) & 1));
}

__device__ __forceinline__ float ld_act(const void* p, size_t i, int bf16) {
  return bf16 ? __bfloat162float(((const __nv_bfloat16*)p)[i]) : ((const float*)p)[i];
}

// TCV tile processing order of a step: tiles tr0 .. nt-1, then 0 .. tr0-1.
__device__ __forceinline__ int tile_at(int n, int tr0, int nt) {
  const int t = n + tr0;
  return t < nt ? t : t - nt;
}

// TCV slab order: tile by tile, K block by K block; position i is (tile i / nsk, K block i % nsk).
// The first positions are the TMEM-cached slabs, then the resident ones, then the streamed ones.
__device__ __forceinline__ void slab_at(int i, int nsk, int& t, int& sk) {
  t = i / nsk;
  sk = i - t * nsk;
}

// Global index of stage s of step ks in the producer's issue order: every stage on the first
// step, then only the stages that are not cached in TMEM.
__device__ __forceinline__ int stage_index(int ks, int s, int nst, int nres) {
  return ks == 0 ? s : nst + (ks - 1) * (nst - nres) + (s - nres);
}

// Tagged argmax key of one block for one (step, request):
//   bits 63..32  orderable fp32 perturbed score (larger is better),
//   bits 31..24  step tag k+1 (the key's slot is zero until this launch publishes it),
//   bits 23..0   0xFFFFFF - v (so equal scores prefer the smaller v; V <= 2^24).
// A block with nothing to offer publishes score bits 0, below every finite score.
__device__ __forceinline__ unsigned long long tagged_key(float score, uint32_t v, int ks) {
  return ((unsigned long long)orderable(score) << 32) | ((unsigned long long)(ks + 1) << 24) |
         (unsigned long long)(0xFFFFFFu - v);
}
__device__ __forceinline__ unsigned long long tagged_key_empty(int ks) {
  return (unsigned long long)(ks + 1) << 24;
}
__device__ __forceinline__ uint32_t tagged_token(unsigned long long key) {
  return 0xFFFFFFu - (uint32_t)(key & 0xFFFFFFull);
}
__device__ __forceinline__ void st_release64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ float ld_acquire_f32(const float* p) {
  float v;
  asm volatile("ld.acquire.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Whole-warp merges of the per-step results, each a short dependency chain: the largest 64-bit
// key by two warp reductions (the high words; then the low words of the lanes holding that high
// word), and (max, sum-exp) by one reduction of the maxima, one exponential per lane and a
// butterfly sum (fixed order, so the result does not depend on timing).
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long k) {
  const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(k >> 32));
  const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(k >> 32) == hi ? (uint32_t)k : 0u);
  return ((unsigned long long)hi << 32) | lo;
}
__device__ __forceinline__ float from_orderable(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}
__device__ __forceinline__ void warp_lse(float& m, float& l) {
  const float M = from_orderable(__reduce_max_sync(0xffffffffu, orderable(m)));
  float s = l != 0.f ? l * __expf(m - M) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  m = s != 0.f ? M : -INFINITY;
  l = s;
}

// Grid barrier and argmax in one: wait (bounded) until every block has published its tagged
// key for step ks, then return the largest.  One warp; each lane covers every 32nd block.
// (The failure-path test hook polls for a tag no block writes, with a short limit.)
__device__ __forceinline__ bool poll_keys(const unsigned long long* keys, int n, int ks, int lane,
                                          bool acquire, unsigned long long* best, bool stuck,
                                          unsigned long long limit_ns) {
  const unsigned long long tag = (unsigned long long)(ks + 1) + (stuck ? 0x40ull : 0ull);
  unsigned long long t0 = 0;
  for (;;) {
    unsigned long long m = 0;
    bool mine = true;
    for (int i = lane; i < n; i += 32) {
      const unsigned long long k = ld_relaxed64(keys + i);
      mine = mine && ((k >> 24) & 0xFF) == tag;
      m = k > m ? k : m;
    }
    if (__all_sync(0xffffffffu, mine)) {
      // with release stores behind the keys, one fence turns the relaxed loads into an
      // acquire of everything those blocks wrote before publishing
      if (acquire) fence_acq_rel_gpu();
      *best = warp_max_key(m);
      return true;
    }
    if (t0 == 0) t0 = globaltimer();
    else if (globaltimer() - t0 > limit_ns) return false;
    __nanosleep(32);
  }
}

// Eq 7 hidden halves w[0:d] . h[b][k], one (b, k) pair per block in turn, block-wide dot
// products with 16-byte loads, written to the workspace for the owner of request b.
template <typename WT, int NT>
__device__ void hidden_dots(const DraftParams& p, Misc* ms, int tid, int cta, int nCTA) {
  const int npairs = p.B * p.gamma;
  for (int i = cta; i < npairs; i += nCTA) {
    float acc = 0.f;
    const size_t base = (size_t)i * p.d;
    if (p.u_bf16 && sizeof(WT) == 2) {
      for (int j = tid * 8; j < p.d; j += NT * 8) {
        const uint4 hq = *(const uint4*)((const __nv_bfloat16*)p.h + base + j);
        const uint4 wq = *(const uint4*)((const WT*)p.w + j);
        float hv[8], wv[8];
        Vec<__nv_bfloat16>::unpack(hq, hv);
        Vec<__nv_bfloat16>::unpack(wq, wv);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(hv[e], wv[e], acc);
      }
    } else {
      for (int j = tid; j < p.d; j += NT)
        acc += to_f<WT>(((const WT*)p.w)[j]) * ld_act(p.h, base + j, p.u_bf16);
    }
    acc = warp_sum(acc);
    if ((tid & 31) == 0) ms->red[tid >> 5] = acc;
    csync<NT>();
    if (tid == 0) {
      float s = 0.f;
      for (int w = 0; w < NT / 32; ++w) s += ms->red[w];
      p.hdot[i] = s;
    }
    csync<NT>();
  }
}

template <int N>
struct Log2 {
  static constexpr int v = 1 + Log2<N / 2>::v;
};
template <>
struct Log2<1> {
  static constexpr int v = 0;
};

// Sum N values per lane (N a power of two <= 32) across the warp: lane l ends with the total
// of value index l >> (5 - log2 N); each index is held by 32/N neighbouring lanes.
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

// (max, sum-exp) of all blocks' partials for one (step, request), merged by one warp in a
// fixed order (deterministic): lane-strided merge, then a butterfly.
// (max, sum-exp) of all blocks' partials, merged by one warp in a fixed order: each lane issues
// the loads of up to 8 partials, the warp takes their maximum M, then sums l_i exp(m_i - M)
// (empty partials are (-inf, 0) and add nothing)
__device__ __forceinline__ float2 warp_merge_ml(const float2* part, int n, int lane) {
  float M = -INFINITY, L = 0.f;
  for (int i0 = 0; i0 < n; i0 += 256) {
    float2 q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + lane + 32 * j;
      q[j] = i < n ? part[i] : make_float2(-INFINITY, 0.f);
    }
    float mb = fmaxf(fmaxf(fmaxf(q[0].x, q[1].x), fmaxf(q[2].x, q[3].x)),
                     fmaxf(fmaxf(q[4].x, q[5].x), fmaxf(q[6].x, q[7].x)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    const float Mn = fmaxf(M, mb);  // the same in every lane
    if (Mn == -INFINITY) continue;
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) sum += q[j].y * __expf(q[j].x - Mn);
    L = L * __expf(M - Mn) + sum;
    M = Mn;
  }
  return make_float2(M, warp_sum(L));
}

// sum of n floats by one warp, up to 8 loads in flight per lane (fixed order)
__device__ __forceinline__ float warp_sum_strided(const float* part, int n, int lane) {
  float s = 0.f;
  for (int i0 = 0; i0 < n; i0 += 256) {
    float q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + lane + 32 * j;
      q[j] = i < n ? part[i] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) s += q[j];
  }
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
// Row dot-product accumulation for one 16-byte W2 chunk against this lane's K-chunk of e.
// bf16: the packed mixed-precision FMA reads both bf16 operands from register halves and
// accumulates in fp32 (bf16 -> fp32 is exact, so this equals converting first).
template <typename WT>
struct Dot;
template <>
struct Dot<__nv_bfloat16> {
  using E = uint32_t;  // e kept as packed bf16 pairs
  static constexpr int NE = 4;
  __device__ __forceinline__ static E load_e(const float* ebuf, int idx2) {
    // ebuf holds fp32 copies of bf16 values: repack two of them exactly
    return (__float_as_uint(ebuf[2 * idx2]) >> 16) | (__float_as_uint(ebuf[2 * idx2 + 1]) & 0xFFFF0000u);
  }
  __device__ __forceinline__ static float run(const uint4& q, const E (&e)[NE], float acc) {
    float a0 = acc, a1 = 0.f;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      asm("{\n\t.reg .b16 wl, wh, el, eh;\n\t"
          "mov.b32 {wl, wh}, %2;\n\t"
          "mov.b32 {el, eh}, %3;\n\t"
          "fma.rn.f32.bf16 %0, wl, el, %0;\n\t"
          "fma.rn.f32.bf16 %1, wh, eh, %1;\n\t}"
          : "+f"(a0), "+f"(a1)
          : "r"(w[i]), "r"(e[i]));
    return a0 + a1;
  }
};
template <>
struct Dot<float> {
  using E = float;
  static constexpr int NE = 4;
  __device__ __forceinline__ static E load_e(const float* ebuf, int idx) { return ebuf[idx]; }
  __device__ __forceinline__ static float run(const uint4& q, const E (&e)[NE], float acc) {
    float a0 = fmaf(__uint_as_float(q.x), e[0], acc), a1 = __uint_as_float(q.y) * e[1];
    a0 = fmaf(__uint_as_float(q.z), e[2], a0);
    a1 = fmaf(__uint_as_float(q.w), e[3], a1);
    return a0 + a1;
  }
};

// RNN head: the conditioning vector a_k is fp32, so W2 is widened and multiplied in fp32.
template <typename WT>
struct DotF {
  using E = float;
  static constexpr int NE = Vec<WT>::N;
  __device__ __forceinline__ static E load_e(const float* ebuf, int idx) { return ebuf[idx]; }
  __device__ __forceinline__ static float run(const uint4& q, const E (&e)[NE], float acc) {
    float w[NE];
    Vec<WT>::unpack(q, w);
    float a0 = acc, a1 = 0.f;
#pragma unroll
    for (int i = 0; i < NE; i += 2) {
      a0 = fmaf(w[i], e[i], a0);
      a1 = fmaf(w[i + 1], e[i + 1], a1);
    }
    return a0 + a1;
  }
};

// TCV: the bias product on the tensor cores.  W2 is tiled as 128 vocabulary rows x 64 K (one
// "slab", 16 KB, 128-byte swizzle, loaded by 2-D TMA); an MMA warp issues kind::f16 MMAs with
// M = 128 vocabulary rows, N = 16 columns holding the B conditioning vectors in bf16 (RNN: a_k
// split into bf16 hi and lo parts, rows b and 8 + b), K = r, into one TMEM accumulator per
// tile, so each consumer thread reads the bias of one vocabulary row for every request.  The
// first slabs of the slice move into TMEM after the first step and feed the MMA as its A
// operand from there; the next ones stay resident in shared memory; the rest stream through
// the ring every step.
template <typename WT, int NB, int NCV, int CW, bool RNN, bool TCV>
__global__ void __launch_bounds__(CW * 32 + 32 + (TCV ? 32 : 0), 1)
    draft_cc_kernel(const DraftParams p, const __grid_constant__ CUtensorMap tmW2) {
  constexpr int kCWarps = CW;
  constexpr int kCThreads = CW * 32;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = TCV ? (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023) : smem_raw;
  const CCLayout Lay = cc_layout(p, NB);
  uint8_t* ring = smem + Lay.ring;
  uint8_t* ubuf = smem + Lay.ubuf;
  float* tbuf = (float*)(smem + Lay.tbuf);
  float* ybuf = (float*)(smem + Lay.ybuf);
  float* gbuf = (float*)(smem + Lay.gbuf);
  float* ebuf = (float*)(smem + Lay.ebuf);
  float* wsm = (float*)(smem + Lay.wsm);
  float* rbuf = (float*)(smem + Lay.rbuf);
  float* sbuf = (float*)(smem + Lay.sbuf);
  float* u3 = (float*)(smem + Lay.u3);
  Slot* slots = (Slot*)(smem + Lay.slots);
  Misc* ms = (Misc*)(smem + Lay.misc);
  uint64_t* full = (uint64_t*)(smem + Lay.bars);
  uint64_t* empty = full + p.nstages;
  uint64_t* ufull = empty + p.nstages;
  uint64_t* uempty = ufull + 2;
  uint64_t* efull = uempty + 2;   // TCV: the B operand of step ks is in shared memory
  uint64_t* mdone = efull + 1;    // TCV: every MMA the MMA warp issued has completed
  uint64_t* accfull = mdone + 1;  // TCV: [32] tile t's accumulator holds step ks's bias
  uint64_t* tready = accfull + 32;  // TCV: [16] slab j has been copied into TMEM
  uint64_t* rfull = tready + 16;    // TCV: [16] resident slab i has landed
  // no thread arrives on it (failure-path test hook); the last barrier of the region
  uint64_t* never = full + 2 * p.nstages + 4 + (TCV ? 2 + 32 + 16 + 16 : 0);
  uint8_t* res = smem + Lay.res;
  uint8_t* ebf = smem + Lay.ebf;

  constexpr int VEC = Vec<WT>::N;
  constexpr int SR = 8 / NB;  // rows per sub-group: SR rows x NB requests = 8 sums per lane
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nCTA = gridDim.x, cta = blockIdx.x;
  // clusters of C consecutive blocks (C = 1: none); cluster cid publishes slot cid of nCL
  const int C = p.cl;
  const int crk = C > 1 ? (int)cluster_rank() : 0, cid = cta / C, nCL = nCTA / C;
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
  const bool ubulk = p.u_bulk && SL > 0;
  // TCV geometry: tiles of 128 rows, r / 64 slabs each, in the order slab_at gives
  const int nsk = r / 64;
  const int nt = TCV ? (SL + 127) / 128 : 0;
  const int nall = nt * nsk;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], TCV ? 1 : 4);  // the MMA (or a copying group) / the four warps
    }
    if (TCV) {
      mbar_init(efull, 1);
      mbar_init(mdone, 1);
      for (int i = 0; i < 32; ++i) mbar_init(&accfull[i], 1);
      for (int i = 0; i < 16; ++i) {
        mbar_init(&tready[i], 1);
        mbar_init(&rfull[i], 1);
      }
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ufull[i], 1);
      mbar_init(&uempty[i], 1);
    }
    mbar_init(never, 1);
    for (int i = 0; i < 4 * 8; ++i) ms->ckey[i / 8][i % 8] = 0ull;  // no step's tag
    fence_mbar_init();
    ms->S_run = 1.f;
    ms->abort = 0;
    for (int i = 0; i < 16; ++i) ms->stage_tag[i] = -1;
  }
  if (tid < 4) {
    const int b = tid;
    const int x = b < B ? p.x0[b] : 0;
    const bool ok = b < B && x >= 0 && x < V;
    ms->cond[b] = ok ? x : 0;
    ms->valid[b] = ok;
    if (b < B && !ok) atomicMax(&hdr->status, kErrInvalid);
  }
  // stages (CUDA cores) or slabs (tensor cores) of the slice cached in TMEM after the first step
  const int nres = TCV ? min(p.nres, nall) : min(p.nres, nst);
  const int nres_s = TCV ? min(p.nres_s, nall - nres) : 0;  // slabs resident in shared memory
  const bool use_tmem = TCV || nres > 0;
  if (use_tmem && warp == 0) {
    tc::tmem_alloc(&ms->tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();  // the last block-wide barrier: from here the producer warp runs on its own
  if (C > 1) cluster_sync_all();  // every leader's barriers are initialised before any arrival
  tc::fence_after_sync();

  // =========================================================== producer warp
  if (warp == kCWarps) {
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_w = policy_evict_last();  // W2 is re-read every step: keep it in L2
      int issued = 0, u_issued = 0;
      bool stop = false;
      int g = 0;
      for (int ks = 0; ks < G && !stop; ++ks) {
        if (ubulk) {  // U_k (and target) rows of step ks
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
        if constexpr (TCV) {
          if (ks == 0)  // resident slabs: straight to their own buffers, once
            for (int i = 0; i < nres_s; ++i) {
              int t, sk;
              slab_at(nres + i, nsk, t, sk);
              mbar_expect_tx(&rfull[i], 16384u);
              tc::tma_load_2d(res + (size_t)i * 16384, &tmW2, 64 * sk, v0 + 128 * t, &rfull[i],
                              pol_w);
            }
          // ring slabs in the MMA's order: on the first step every slab but the resident ones
          // (those bound for TMEM first), later only the streamed ones
          for (int j = ks == 0 ? 0 : nres + nres_s; j < nall; ++j) {
            if (ks == 0 && j >= nres && j < nres + nres_s) continue;
            const int slot = g % NS;
            if (g >= NS &&
                !mbar_wait_or_abort(&empty[slot], (uint32_t)(((g - NS) / NS) & 1), &ms->abort)) {
              stop = true;
              break;
            }
            int t, sk;
            slab_at(j, nsk, t, sk);
            ms->stage_tag[slot] = g;
            mbar_expect_tx(&full[slot], 16384u);
            tc::tma_load_2d(ring + (size_t)slot * 16384, &tmW2, 64 * sk, v0 + 128 * t, &full[slot],
                            pol_w);
            issued = ++g;
          }
        } else {
          for (int s = (ks == 0 ? 0 : nres); s < nst; ++s, ++g) {
            const int slot = g % NS;
            if (g >= NS &&
                !mbar_wait_or_abort(&empty[slot], (uint32_t)(((g - NS) / NS) & 1), &ms->abort)) {
              stop = true;
              break;
            }
            const int rows = min(R, SL - s * R);
            const uint32_t bytes = (uint32_t)(rows * row_bytes);
            ms->stage_tag[slot] = g;
            mbar_expect_tx(&full[slot], bytes);
            bulk_g2s(ring + (size_t)slot * p.stage_bytes,
                     (const uint8_t*)p.W2 + (size_t)(v0 + s * R) * row_bytes, bytes, &full[slot],
                     pol_w);
            issued = g + 1;
          }
        }
      }
      if (stop) atomicMax(&hdr->status, kErrTimeout);
      // every copy this warp started must land before the block may exit
      for (int g = max(0, issued - NS); g < issued; ++g)
        mbar_wait(&full[g % NS], (uint32_t)((g / NS) & 1));
      for (int k = max(0, u_issued - 2); k < u_issued; ++k)
        mbar_wait(&ufull[k & 1], (uint32_t)((k >> 1) & 1));
      if (TCV)
        for (int i = 0; i < nres_s; ++i) mbar_wait(&rfull[i], 0);
    }
    if (C > 1) cluster_sync_all();  // no block leaves while a peer may still write to it
    return;
  }

  // =========================================================== MMA warp (TCV)
  if (TCV && warp == kCWarps + 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(128, 16);
      const uint32_t tmem = ms->tmem_base;
      const uint32_t acc0 = tmem + 32 * p.nres;  // accumulators follow the largest TMEM cache
      // operand descriptors, built once: B (K block sk, K step kk) and the bases of the ring
      // and the resident slabs
      uint64_t bdesc[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        bdesc[q] = tc::sdesc_sw128(smem_u32(ebf) + (q >> 2) * 2048 + (q & 3) * 32);
      const uint64_t ring_desc = tc::sdesc_sw128(smem_u32(ring));
      const uint64_t res_desc = tc::sdesc_sw128(smem_u32(res));
      bool stop = false;
      int g = nres;  // ring uses 0 .. nres-1 carry the first step's TMEM-bound slabs
      for (int ks = 0; ks < G && !stop; ++ks) {
        if (!mbar_wait_or_abort(efull, (uint32_t)(ks & 1), &ms->abort)) {
          stop = true;
          break;
        }
        tc::fence_after_sync();
        // after the first step the tiles that stream through the ring go first, so the ring
        // refills while the MMAs read the resident tiles
        const int tr0 = ks == 0 ? 0 : min(nt, (nres + nres_s) / nsk);
        for (int n = 0; n < nt && !stop; ++n) {
          const int t = tile_at(n, tr0, nt);
          const uint32_t d = acc0 + 16 * t;
#pragma unroll
          for (int sk = 0; sk < 4; ++sk) {  // nsk <= 4 K blocks; unrolled so bdesc stays in registers
            if (sk >= nsk) break;
            const int i = t * nsk + sk;  // position in the slab order (tile by tile)
            const uint64_t* bd = bdesc + 4 * sk;
            if (i < nres) {  // A from TMEM (copied there during the first step)
              if (ks == 0) {
                if (!mbar_wait_or_abort(&tready[i], 0, &ms->abort)) {
                  stop = true;
                  break;
                }
                tc::fence_after_sync();
              }
              const uint32_t a = tmem + 32 * i;
              if (sk == 0) tc::mma_bf16_ts_c<false>(d, a, bd[0], idesc);
              else tc::mma_bf16_ts_c<true>(d, a, bd[0], idesc);
              tc::mma_bf16_ts_c<true>(d, a + 8, bd[1], idesc);
              tc::mma_bf16_ts_c<true>(d, a + 16, bd[2], idesc);
              tc::mma_bf16_ts_c<true>(d, a + 24, bd[3], idesc);
            } else {
              int slot = -1;
              uint64_t ad;
              if (i < nres + nres_s) {  // A resident in shared memory
                if (ks == 0 && !mbar_wait_or_abort(&rfull[i - nres], 0, &ms->abort)) {
                  stop = true;
                  break;
                }
                ad = res_desc + (uint64_t)((i - nres) * 1024);  // 16 KB per slab, in 16 B units
              } else {  // A streamed through the ring
                slot = g % NS;
                if (!mbar_wait_or_abort(&full[slot], (uint32_t)((g / NS) & 1), &ms->abort)) {
                  stop = true;
                  break;
                }
                tc::fence_after_sync();
                ad = ring_desc + (uint64_t)(slot * 1024);
                ++g;
              }
              // a K step of 16 elements is 32 bytes further along the swizzled rows: +2 in the
              // descriptor's address field
              if (sk == 0) tc::mma_bf16_c<false>(d, ad, bd[0], idesc);
              else tc::mma_bf16_c<true>(d, ad, bd[0], idesc);
              tc::mma_bf16_c<true>(d, ad + 2, bd[1], idesc);
              tc::mma_bf16_c<true>(d, ad + 4, bd[2], idesc);
              tc::mma_bf16_c<true>(d, ad + 6, bd[3], idesc);
              if (slot >= 0) tc::mma_commit(&empty[slot]);  // free once these MMAs have read it
            }
          }
          if (!stop) tc::mma_commit(&accfull[t]);
        }
      }
      if (stop) atomicMax(&hdr->status, kErrTimeout);
      tc::mma_commit(mdone);  // lets the TMEM owner free the columns once these MMAs are done
    }
    if (C > 1) cluster_sync_all();
    return;
  }

  // =========================================================== consumer warps
  if (conf && cta < B)
    for (int j = tid; j < r; j += kCThreads) wsm[j] = to_f<WT>(((const WT*)p.w)[p.d + j]);
  if (RNN && cta < B)
    for (int j = tid; j < r; j += kCThreads) sbuf[j] = p.s0 ? p.s0[(size_t)cta * r + j] : 0.f;
  if (conf && G == 1) hidden_dots<WT, kCThreads>(p, ms, tid, cta, nCTA);
  fill_noise<NB>(gbuf, SLM, SL, v0, B, 0, p.seed_lo, p.seed_hi, tid, kCThreads);

  if (TCV) {  // the B operand's padding rows stay zero
    for (int i = tid; i < nsk * 512; i += kCThreads) ((uint32_t*)ebf)[i] = 0u;
  }

  bool failed = false;
  // after the 8-value reduction lane l holds value (l >> 2) = (row, request) = (idx/NB, idx%NB);
  // lanes 4 idx own it
  const int idx8 = lane >> 2, jrow = idx8 / NB, bq = idx8 % NB;
  const bool owner = (lane & 3) == 0;
  constexpr int kGroups = kCWarps / 4;
  const int grp = warp / 4, qw = warp % 4;

  for (int ks = 0; ks < G; ++ks) {
    const int buf = ks & 1;
    // (a) conditioning vectors e_b = W1[x_{k-1}] (Eq 5 lookup), fp32 in shared memory
    for (int i = tid; i < NB * r; i += kCThreads) {
      const int b = i / r, j = i - b * r;
      float val = 0.f;
      if (b < B && ms->valid[b]) val = to_f<WT>(((const WT*)p.W1)[(size_t)ms->cond[b] * r + j]);
      ebuf[i] = val;
    }
    csync<kCThreads>();
    if (RNN) {
      // (a') Eq 6 for the owned request, published for every block; then collect a_k of all
      if (cta < B) {
        rnn_row_update<kCThreads>(p, cta, ks, sbuf, ebuf + cta * r, u3,
                                  p.rnn_a + ((size_t)ks * B + cta) * r, tid);
        if (tid == 0) st_release_u32(&p.rnn_flag[(size_t)ks * B + cta], (unsigned)(ks + 1));
      }
      bool okf = true;
      if (warp < B && lane == 0) okf = wait_flag(&p.rnn_flag[(size_t)ks * B + warp], (unsigned)(ks + 1));
      if (csync_or<kCThreads>(!okf)) {
        failed = true;
        break;
      }
      for (int i = tid; i < NB * r; i += kCThreads) {
        const int b = i / r;
        rbuf[i] = b < B ? ld_acquire_f32(&p.rnn_a[((size_t)ks * B + b) * r + (i - b * r)]) : 0.f;
      }
      csync<kCThreads>();
    }
    // (b) this lane's K-chunks of every e_b (RNN: a_k) in registers; TCV: the MMA's B operand
    using DT = typename std::conditional<RNN, DotF<WT>, Dot<WT>>::type;
    const float* cvec = RNN ? rbuf : ebuf;
    typename DT::E ereg[NB][NCV][DT::NE];
    if constexpr (TCV) {
      // row b = bf16(e_b) (exact: e_b is a bf16 row of W1); RNN: row b = bf16(a_b) and row
      // 8 + b = bf16(a_b - that), so the two columns add up to a_b within 2^-16 relative.
      // 16-byte chunk c of row n sits in K block c / 8 at chunk position (c % 8) ^ (n % 8).
      const int nch = r / 8;
      for (int i = tid; i < NB * nch; i += kCThreads) {
        const int b = i / nch, c = i - b * nch;
        const float* src = cvec + b * r + 8 * c;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(src[2 * q], src[2 * q + 1]);
          hi[q] = *(const uint32_t*)&h2;
          if (RNN) {
            const float2 hf = __bfloat1622float2(h2);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(src[2 * q] - hf.x, src[2 * q + 1] - hf.y);
            lo[q] = *(const uint32_t*)&l2;
          }
        }
        const int blk = (c >> 3) * 2048, cc = c & 7;
        *(uint4*)(ebf + blk + b * 128 + ((cc ^ (b & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if (RNN) {
          const int n = 8 + b;
          *(uint4*)(ebf + blk + n * 128 + ((cc ^ (n & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      fence_proxy_async_smem();  // generic-proxy writes, read by the tensor cores
      csync<kCThreads>();
      if (tid == 0) mbar_arrive(efull);
    } else {
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int t = 0; t < NCV; ++t) {
          const int cv = lane + 32 * t;
#pragma unroll
          for (int i = 0; i < DT::NE; ++i)
            ereg[b][t][i] = cv < VR ? DT::load_e(cvec + b * r + cv * VEC, i) : typename DT::E(0);
        }
    }
    // (c) U_k (and target) rows of the slice
    if (ubulk) {
      const bool ok = mbar_wait(&ufull[buf], (uint32_t)((ks >> 1) & 1));
      if (csync_or<kCThreads>(!ok)) {
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
      csync<kCThreads>();
    }

    // (d) this warp's stages: bias dot products, logits, sampling, normalisers
    Slot st;
    slot_init(st);
    const uint8_t* ub = ubuf + (size_t)(buf * NB + bq) * SLM * ues;
    const float* tb = tbuf + (size_t)(buf * NB + bq) * SLM;
    const float* gb = gbuf + (size_t)bq * SLM;
    bool wfail = false;
    if (p.test_stuck == 2 && ks == 0)  // failure-path test hook: a wait nothing will end
      wfail = !mbar_wait_warp_lim(never, 0, p.test_wait_ns);
    // +U_k, /T, online (max, sum-exp), Gumbel-max update for slice entry vl of request bq
    auto epilogue = [&](int vl, float bias) {
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
    };
    // TCV: one thread per vocabulary row and all requests; slot sb[b] per request
    Slot sb[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) slot_init(sb[b]);
    if constexpr (TCV) {
      const uint32_t tmem = ms->tmem_base;
      const uint32_t lq = (uint32_t)(32 * qw) << 16;  // this warp's TMEM lane quarter
      if (ks == 0) {
        // slabs bound for TMEM: the group's four warps copy rows 32 qw + lane of each (one
        // 16-byte chunk at a time out of the swizzled slab) into TMEM columns [32 j, 32 j + 32)
        for (int j = grp; j < nres && !wfail; j += kGroups) {
          const int slot = j % NS;  // ring use j
          const bool okw = __all_sync(0xffffffffu, wait_stage(ms->stage_tag, full, slot, j, NS));
          if (gsync_or(grp, !okw)) {
            wfail = true;
            break;
          }
          const uint8_t* sp = ring + (size_t)slot * 16384;
          const int m = 32 * qw + lane;
          uint32_t wv[32];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *(uint4*)&wv[4 * c] = *(const uint4*)(sp + m * 128 + ((c ^ (m & 7)) << 4));
          tc::tmem_st32(tmem + lq + 32 * j, wv);
          tc::tmem_st_wait();
          tc::fence_before_sync();
          gsync_or(grp, 0);
          if (qw == 0 && lane == 0) {
            mbar_arrive(&tready[j]);
            mbar_arrive(&empty[slot]);
          }
        }
      }
      const uint32_t acc0 = tmem + 32 * p.nres;
      const int tr0 = ks == 0 ? 0 : min(nt, (nres + nres_s) / nsk);  // the MMA warp's order
      for (int n = grp; n < nt && !wfail; n += kGroups) {
        const int t = tile_at(n, tr0, nt);
        const bool oka = mbar_wait_warp(&accfull[t], (uint32_t)(ks & 1));
        if (!oka) {
          wfail = true;
          break;
        }
        tc::fence_after_sync();
        uint32_t acc[16];
        tc::tmem_ld16(acc0 + lq + 16 * t, acc);
        tc::tmem_ld_wait();
        const int vl = 128 * t + 32 * qw + lane;
        if (vl < SL) {
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            if (b >= B) break;
            float bias = __uint_as_float(acc[b]);
            if (RNN) bias += __uint_as_float(acc[8 + b]);
            const int v = v0 + vl;
            const float uval =
                p.u_bf16 ? __uint_as_float((uint32_t)((const uint16_t*)ubuf)[(size_t)(buf * NB + b) * SLM + vl] << 16)
                         : ((const float*)ubuf)[(size_t)(buf * NB + b) * SLM + vl];
            const float z = uval + bias;
            if (p.logits) p.logits[((size_t)b * G + ks) * V + v] = z;
            const float y = z * p.invT;
            lse_push(sb[b].m, sb[b].l, y);
            const float sc = y + gbuf[(size_t)b * SLM + vl];
            if (sc > sb[b].best) {  // v grows along this thread's rows: ties keep the smaller v
              sb[b].best = sc;
              sb[b].tok = (uint32_t)v;
            }
            if (tgt) {
              lse_push(sb[b].mt, sb[b].lt, tbuf[(size_t)(buf * NB + b) * SLM + vl] * p.invT);
              ybuf[(size_t)b * SLM + vl] = y;
            }
          }
        }
      }
      tc::fence_before_sync();  // the accumulators are read: the next step may overwrite them
    }
    float bb = 0.f;       // NB == 1: the row sum this lane holds for the batched epilogue
    int vlb = -1, nb = 0;  // its slice entry (-1: none) and the stages batched so far
    // Four warps share each stage: warp q of a group takes rows [q R/4, (q+1) R/4) in
    // sub-groups of SR rows, so a slot is handed back a quarter of a stage's work after its
    // bytes land.  Stages go round-robin to the groups.
    for (int s = grp; s < (TCV ? 0 : nst) && !wfail; s += kGroups) {
      const int rows = min(R, SL - s * R);
      const int rq0 = qw * (R / 4), rq1 = min(rows, rq0 + R / 4);
      if (R == 32 && NCV == 1) {
        // This warp's 8 rows of the stage, one 16-byte K-chunk per lane, staged in registers:
        // from TMEM for a cached stage after the first step, else from the ring (and, on the
        // first step, copied into TMEM for the later steps).
        uint32_t wv[32];
        const uint32_t taddr = ms->tmem_base + ((uint32_t)(32 * qw) << 16) + 32 * s;
        if (ks > 0 && s < nres) {
          tc::tmem_ld32(taddr, wv);
          tc::tmem_ld_wait();
        } else {
          const int g = stage_index(ks, s, nst, nres);
          const int slot = g % NS;
          // warp-uniform verdict: the TMEM store below needs the whole warp
          if (!__all_sync(0xffffffffu, wait_stage(ms->stage_tag, full, slot, g, NS))) {
            wfail = true;
            break;
          }
          const uint8_t* stg = ring + (size_t)slot * p.stage_bytes;
          const int cv = min(lane, VR - 1);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *(uint4*)&wv[4 * j] = *(const uint4*)(stg + (size_t)(rq0 + j) * row_bytes + cv * 16);
          if (ks == 0 && s < nres) {
            tc::tmem_st32(taddr, wv);
            tc::tmem_st_wait();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
        }
#pragma unroll
        for (int sg = 0; sg < 8 / SR; ++sg) {
          float part[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) part[i] = 0.f;
#pragma unroll
          for (int j = 0; j < SR; ++j) {
            const uint4 q = *(const uint4*)&wv[4 * (sg * SR + j)];
#pragma unroll
            for (int b = 0; b < NB; ++b) part[j * NB + b] = DT::run(q, ereg[b][0], part[j * NB + b]);
          }
          const float bias = transpose_reduce<8>(part, lane);
          if (NB == 1) {
            // one request: gather the 8 row sums of this stage into lanes 8 nb .. 8 nb + 7 and
            // run the epilogue once per 4 stages, on all 32 lanes (rows still reach each lane
            // in increasing v)
            const float mine = __shfl_sync(0xffffffffu, bias, (lane & 7) << 2);
            if ((lane >> 3) == nb) {
              bb = mine;
              vlb = rq0 + (lane & 7) < rq1 ? s * R + rq0 + (lane & 7) : -1;
            }
            if (++nb == 4) {
              if (vlb >= 0) epilogue(vlb, bb);
              vlb = -1;
              nb = 0;
            }
          } else {
            const int row = rq0 + sg * SR + jrow;
            if (owner && bq < B && row < rq1) epilogue(s * R + row, bias);
          }
        }
        continue;
      }
      const int g = stage_index(ks, s, nst, nres);
      const int slot = g % NS;
      if (!wait_stage(ms->stage_tag, full, slot, g, NS)) {
        wfail = true;
        break;
      }
      const uint8_t* stg = ring + (size_t)slot * p.stage_bytes;
      if (rq1 <= rq0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
      for (int r0 = rq0; r0 < rq1; r0 += SR) {
        float part[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) part[i] = 0.f;
        // No per-row guard here (a data-dependent guard serialises the loads): rows past the
        // end of a short stage read in-bounds stale ring bytes and are masked in the epilogue;
        // lanes past the row width read a chunk of the same row against zero e values.
#pragma unroll
        for (int t = 0; t < NCV; ++t) {
          const int cv = min(lane + 32 * t, VR - 1);
#pragma unroll
          for (int j = 0; j < SR; ++j) {
            const uint4 q = *(const uint4*)(stg + (size_t)(r0 + j) * row_bytes + cv * 16);
#pragma unroll
            for (int b = 0; b < NB; ++b) part[j * NB + b] = DT::run(q, ereg[b][t], part[j * NB + b]);
          }
        }
        if (r0 + SR >= rq1) {  // this warp's bytes of the stage are in registers: hand it back
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
        }
        const float bias = transpose_reduce<8>(part, lane);
        const int row = r0 + jrow;
        if (owner && bq < B && row < rq1) epilogue(s * R + row, bias);
      }
    }
    if (NB == 1 && nb > 0 && vlb >= 0) epilogue(vlb, bb);  // a partial batch of stages
    if (csync_or<kCThreads>(wfail)) {
      failed = true;
      break;
    }

    // (e) merge lanes of the same request, then warps (fixed butterflies), and publish this
    // block's candidate for step ks as a tagged argmax key with release semantics: the key is
    // the grid barrier's arrival too.  With a target the second pass right after the barrier
    // needs the global normalisers, so the (max, sum-exp) partials go out before the key;
    // without one only the argmax is on the critical path and the partials follow the key.
    if constexpr (TCV) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        Slot& a = sb[b];
        const unsigned long long key =
            warp_max_key(a.tok != 0xFFFFFFFFu ? tagged_key(a.best, a.tok, ks) : 0ull);
        warp_lse(a.m, a.l);
        if (tgt) warp_lse(a.mt, a.lt);
        if (lane == 0) {
          Slot& o = slots[warp * 4 + b];
          o.best = __uint_as_float((uint32_t)(key >> 32));
          o.tok = (uint32_t)key;
          o.m = a.m;
          o.l = a.l;
          o.mt = a.mt;
          o.lt = a.lt;
        }
      }
    } else {
      unsigned long long key = st.tok != 0xFFFFFFFFu ? tagged_key(st.best, st.tok, ks) : 0ull;
      // lanes of the same request: those 4 NB apart hold the owner results; with one request
      // the batched epilogue leaves results on every lane, so all 32 are merged
      if (NB == 1) {
        key = warp_max_key(key);
        warp_lse(st.m, st.l);
        if (tgt) warp_lse(st.mt, st.lt);
      }
#pragma unroll
      for (int o = 4 * NB; NB > 1 && o < 32; o <<= 1) {
        const unsigned long long q = __shfl_xor_sync(0xffffffffu, key, o);
        key = q > key ? q : key;
        lse_merge(st.m, st.l, __shfl_xor_sync(0xffffffffu, st.m, o), __shfl_xor_sync(0xffffffffu, st.l, o));
        if (tgt)
          lse_merge(st.mt, st.lt, __shfl_xor_sync(0xffffffffu, st.mt, o),
                    __shfl_xor_sync(0xffffffffu, st.lt, o));
      }
      if (lane < 4 * NB && owner) {
        Slot& o = slots[warp * 4 + (lane >> 2)];
        o.best = __uint_as_float((uint32_t)(key >> 32));
        o.tok = (uint32_t)key;
        o.m = st.m;
        o.l = st.l;
        o.mt = st.mt;
        o.lt = st.lt;
      }
    }
    csync<kCThreads>();
    bool ok = true;
    if (warp < B) {
      const int b = warp;
      const size_t o = ((size_t)ks * B + b) * nCL + cid;  // the block's (C = 1) or cluster's slot
      const bool has = SL > 0 && ms->valid[b];
      unsigned long long kb = 0;
      if (lane < kCWarps) {
        const Slot& q = slots[lane * 4 + b];
        kb = ((unsigned long long)__float_as_uint(q.best) << 32) | q.tok;
      }
      kb = warp_max_key(kb);
      const unsigned long long pub = has && kb ? kb : tagged_key_empty(ks);
      if (C == 1 && !tgt && lane == 0) st_relaxed64(&p.keys[o], pub);
      float m = -INFINITY, l = 0.f, mt = -INFINITY, lt = 0.f;
      if (lane < kCWarps) {
        const Slot& q = slots[lane * 4 + b];
        m = q.m;
        l = q.l;
        mt = q.mt;
        lt = q.lt;
      }
      warp_lse(m, l);
      if (tgt) warp_lse(mt, lt);
      if (lane == 0) {
        if (C == 1) {
          p.ml[o] = make_float2(m, l);
          if (tgt) {
            p.mlt[o] = make_float2(mt, lt);
            st_release64(&p.keys[o], pub);
          }
        } else {  // to the cluster's leader, in its shared memory
          st_cluster_f2(cluster_addr(&ms->cml[b][crk], 0), make_float2(m, l));
          if (tgt) st_cluster_f2(cluster_addr(&ms->cmlt[b][crk], 0), make_float2(mt, lt));
          st_release_cluster_u64(cluster_addr(&ms->ckey[b][crk], 0), pub);
        }
        // if this block's candidate wins, every block gathers its W1 row next: warm L2 now
        if (has && kb)
          prefetch_l2((const uint8_t*)p.W1 + (size_t)tagged_token(kb) * row_bytes, (uint32_t)row_bytes);
      }
      if (C > 1 && crk == 0) {
        // leader: once every block of the cluster has written, merge the C results in a fixed
        // order (largest key; (max, sum-exp) by a butterfly) and publish the cluster's slot
        unsigned long long kc = 0ull;
        {
          bool seen = lane >= C;
          unsigned long long t0 = 0;
          for (;;) {  // bounded: until every slot carries step ks's tag
            if (!seen) {
              kc = ld_acquire_cluster_u64(&ms->ckey[b][lane]);
              seen = ((kc >> 24) & 0xFF) == (unsigned long long)(ks + 1);
            }
            if (__all_sync(0xffffffffu, seen)) break;
            if (t0 == 0) t0 = globaltimer();
            else if (globaltimer() - t0 > kWaitLimitNs) {
              ok = false;
              break;
            }
          }
        }
        if (ok) {
          kc = warp_max_key(kc);
          if (!tgt && lane == 0) st_relaxed64(&p.keys[o], kc);
          float2 a = lane < C ? ms->cml[b][lane] : make_float2(-INFINITY, 0.f);
          float2 t = tgt && lane < C ? ms->cmlt[b][lane] : make_float2(-INFINITY, 0.f);
          warp_lse(a.x, a.y);
          if (tgt) warp_lse(t.x, t.y);
          if (lane == 0) {
            p.ml[o] = a;
            if (tgt) {
              p.mlt[o] = t;
              st_release64(&p.keys[o], kc);
            }
          }
        }
      }
    }

    // (f) while the other blocks finish: next step's noise, Eq 7's embedding half of this step
    // (owned request), the hidden halves (first step); then every block's key for step ks
    // (the polling warps b < B skip the noise so that they start polling at once)
    if (ks + 1 < G && warp >= B)
      fill_noise<NB>(gbuf, SLM, SL, v0, B, ks + 1, p.seed_lo, p.seed_hi, tid - 32 * B,
                     kCThreads - 32 * B);
    if (conf && cta < B && warp == kCWarps - 1) {
      float acc = 0.f;
      for (int j = lane; j < r; j += 32) acc += wsm[j] * ebuf[cta * r + j];
      acc = warp_sum(acc);
      if (lane == 0) p.hdot[(size_t)(B + cta) * G + ks] = acc;  // embedding half
    }
    if (conf && ks == 0 && G > 1) hidden_dots<WT, kCThreads>(p, ms, tid, cta, nCTA);
    if (warp < B && ok) {
      const int b = warp;
      unsigned long long best = 0;
      ok = poll_keys(p.keys + ((size_t)ks * B + b) * nCL, nCL, ks, lane, tgt, &best,
                     p.test_stuck == 1, p.test_stuck == 1 ? p.test_wait_ns : kWaitLimitNs);
      if (lane == 0 && ok) {
        const bool was_valid = ms->valid[b];
        const int xk = was_valid ? (int)tagged_token(best) : -1;
        const int nxt = p.forced ? p.forced[(size_t)b * G + ks] : xk;
        const bool nv = was_valid && nxt >= 0 && nxt < V;
        if (was_valid && !nv && cta == 0) atomicMax(&hdr->status, kErrInvalid);
        ms->cond[b] = nv ? nxt : 0;
        ms->valid[b] = nv;
        if (cta == b) p.tokens[(size_t)b * G + ks] = was_valid ? xk : -1;
      }
    }
    if (csync_or<kCThreads>(!ok)) {
      failed = true;
      break;
    }

    if (tgt) {
      // Eq 8 second pass over the slice: needs the global normalisers of p^d and p^t
      if (warp < B) {
        const float2 a = warp_merge_ml(p.ml + ((size_t)ks * B + warp) * nCL, nCL, lane);
        const float2 t = warp_merge_ml(p.mlt + ((size_t)ks * B + warp) * nCL, nCL, lane);
        if (lane == 0) {
          ms->Ld[warp] = a.x + logf(a.y);
          ms->Lt[warp] = t.x + logf(t.y);
        }
      }
      csync<kCThreads>();
      for (int b = 0; b < B; ++b) {
        const float Ld = ms->Ld[b], Lt = ms->Lt[b];
        float acc = 0.f;
        for (int vl = tid; vl < SL; vl += kCThreads)
          acc += fabsf(__expf(ybuf[(size_t)b * SLM + vl] - Ld) -
                       __expf(tbuf[(size_t)(buf * NB + b) * SLM + vl] * p.invT - Lt));
        acc = warp_sum(acc);
        if (lane == 0) ms->red[warp] = acc;
        csync<kCThreads>();
        if (tid == 0) {
          float s = 0.f;
          for (int w = 0; w < kCWarps; ++w) s += ms->red[w];
          p.l1p[((size_t)ks * B + b) * nCTA + cta] = s;
        }
        csync<kCThreads>();
      }
    }
    // (g) U/target buffer `buf` is free again for step ks + 2
    if (ubulk && tid == 0) mbar_arrive(&uempty[buf]);
  }

  // TMEM is no longer read: hand it back (every consumer warp has waited for its own loads;
  // with the tensor cores, the MMA warp's last commit says its MMAs are done too)
  if (failed) ms->abort = 1;  // a waiting producer or MMA warp gives up at once
  if (use_tmem) {
    if (TCV && warp == 0) mbar_wait(mdone, 0);
    tc::fence_before_sync();
    csync<kCThreads>();
    if (warp == 0) {
      tc::fence_after_sync();
      tc::tmem_dealloc(ms->tmem_base, 512);
    }
  }

  if (failed) {
    // unwind: stop the producer (it drains its own copies), record the timeout
    ms->abort = 1;
    if (tid == 0) atomicMax(&hdr->status, kErrTimeout);
    if (C > 1) cluster_sync_all();
    return;
  }

  if (RNN && cta < B && p.s_out)
    for (int j = tid; j < r; j += kCThreads) p.s_out[(size_t)cta * r + j] = sbuf[j];

  // with a target the owned request's normalisers and Eq 8 of every step but the last are
  // complete here (their partials went out before each key); the rest waits for the last block
  if (tgt && cta < B) {
    const int b = cta;
    for (int k = warp; k < G; k += kCWarps) {
      const bool vb = p.tokens[(size_t)b * G + k] >= 0;
      const float2 ml = warp_merge_ml(p.ml + ((size_t)k * B + b) * nCL, nCL, lane);
      if (lane == 0) p.lse[(size_t)b * G + k] = vb ? ml.x + logf(ml.y) : NAN;
      if (k + 1 < G) {
        const float s = warp_sum_strided(p.l1p + ((size_t)k * B + b) * nCTA, nCTA, lane);
        if (lane == 0) {
          const size_t o = (size_t)b * G + k;
          p.l1[o] = vb ? s : NAN;
          p.cstar[o] = vb ? fminf(1.f, fmaxf(0.f, 1.f - 0.5f * s)) : NAN;
        }
      }
    }
  }

  // last block out: what needs every block's writes -- Eq 7 and S_k of every request (the
  // hidden and embedding halves come from several blocks), the log-normalisers without a
  // target, Eq 8 of the final step -- then leave the workspace ready for the next call
  __threadfence();  // this thread's global writes are visible before the block counts itself out
  csync<kCThreads>();
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&hdr->exit_count, 1u);
    ms->last = (old == (unsigned)nCTA - 1u);
  }
  csync<kCThreads>();
  if (ms->last) {
    __threadfence();
    const volatile int32_t* vtok = p.tokens;
    if (conf) {
      // one thread per (b, k) loads and squashes, then one per request runs the product
      float* cbuf = ms->cbuf;
      for (int i = tid; i < B * G; i += kCThreads) {
        ms->cvalid[i] = vtok[i] >= 0;
        cbuf[i] = sigmoidf_acc(p.hdot[i] + p.hdot[(size_t)B * G + i]);
      }
      csync<kCThreads>();
      if (tid < B) {
        float surv = 1.f;
        bool vb = true;
        for (int k = 0; k < G; ++k) {
          const int o = tid * G + k;
          vb = vb && ms->cvalid[o];
          const float cv = vb ? cbuf[o] : NAN;
          surv = vb ? surv * cv : NAN;
          p.c[o] = cv;
          p.S[o] = surv;
        }
      }
    }
    if (!tgt)
      for (int i = warp; i < B * G; i += kCWarps) {
        const int b = i / G, k = i - b * G;
        const float2 ml = warp_merge_ml(p.ml + ((size_t)k * B + b) * nCL, nCL, lane);
        if (lane == 0) p.lse[i] = vtok[i] >= 0 ? ml.x + logf(ml.y) : NAN;
      }
    if (tgt && warp < B) {
      const int b = warp;
      const float s = warp_sum_strided(p.l1p + ((size_t)(G - 1) * B + b) * nCTA, nCTA, lane);
      if (lane == 0) {
        const size_t o = (size_t)b * G + G - 1;
        const bool vb = vtok[o] >= 0;
        p.l1[o] = vb ? s : NAN;
        p.cstar[o] = vb ? fminf(1.f, fmaxf(0.f, 1.f - 0.5f * s)) : NAN;
      }
    }
    for (int i = tid; i < G * B * nCL; i += kCThreads) p.keys[i] = 0ull;
    if (RNN)
      for (int i = tid; i < G * B; i += kCThreads) p.rnn_flag[i] = 0u;
    csync<kCThreads>();
    if (tid == 0) {
      hdr->exit_count = 0;
      __threadfence();
    }
  }
  if (C > 1) cluster_sync_all();
}

template <typename WT, int NB, int NCV, bool TCV>
cudaError_t launch_k(DraftParams& p, const CUtensorMap& tm, int nblocks, cudaStream_t stream) {
  // consumer warps: 24 for one request on the CUDA cores (the stage loop is latency-bound and
  // the variant fits 80 registers), 16 for two, 8 for four
  constexpr int CW = (NB <= 1 && !TCV) ? 24 : NB <= 2 ? 16 : 8;
  constexpr int kThreads = CW * 32 + 32 + (TCV ? 32 : 0);
  auto kern = p.head == 1 ? draft_cc_kernel<WT, NB, NCV, CW, true, TCV>
                          : draft_cc_kernel<WT, NB, NCV, CW, false, TCV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)p.smem_bytes);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&p, (void*)&tm};
  if (p.cl <= 1)
    return cudaLaunchCooperativeKernel((const void*)kern, dim3(nblocks), dim3(kThreads), args,
                                       p.smem_bytes, stream);
  // cooperative (every block resident at once: the per-step merge waits on all of them) and in
  // clusters of p.cl consecutive blocks
  if (nblocks % p.cl != 0) return cudaErrorInvalidValue;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = (unsigned)p.cl;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(nblocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelExC(&cfg, (const void*)kern, args);
}

template <typename WT, int NB, int NCV>
cudaError_t launch_t(DraftParams& p, int nblocks, cudaStream_t stream) {
  CUtensorMap tm;
  std::memset(&tm, 0, sizeof tm);
  if constexpr (std::is_same<WT, __nv_bfloat16>::value && NCV == 1) {
    if (p.tcv) {
      // W2 [V][r] as 128-row x 64-column tiles in the 128-byte swizzle
      if (!encode_bf16_2d(&tm, p.W2, p.V, p.r, p.r, 128)) return cudaErrorInvalidValue;
      return launch_k<WT, NB, NCV, true>(p, tm, nblocks, stream);
    }
  }
  if (p.tcv) return cudaErrorNotSupported;
  return launch_k<WT, NB, NCV, false>(p, tm, nblocks, stream);
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

// Tensor-core variant: bf16, B <= 4, K = r in whole 64-element blocks with one 128-row tile of A
// in at most 128 TMEM columns, and at most 32 tiles (16 accumulator columns each) per slice.
int draft_tcv_supported(int B, int r, int w_bf16, int slice_max) {
  return w_bf16 && B >= 1 && B <= 4 && r % 64 == 0 && r <= 256 && slice_max >= 1 &&
         (slice_max + 127) / 128 <= 32;
}

// Ring geometry: stages of at least 16 KB holding a multiple of 32 W2 rows, as many stages as
// the shared memory left after the per-step buffers allows (at most 16).
bool draft_cc_configure(DraftParams& p, size_t smem_optin) {
  if (p.tcv) {
    // 16 KB slabs; TMEM holds the accumulators (16 columns per tile) and as many 32-column
    // slabs as fit beside them (at most 16); shared memory holds a ring of up to 6 slabs and,
    // from what is left, up to 16 resident slabs
    const int nsk = p.r / 64, ntmax = (p.slice_max + 127) / 128;
    const int nall = ntmax * nsk;
    p.stage_bytes = 16384;
    int nres = (512 - 16 * ntmax) / 32;
    nres = nres < 0 ? 0 : nres > 16 ? 16 : nres;
    p.nres = nres < nall ? nres : nall;
    p.nstages = 0;
    p.nres_s = 0;
    const size_t base = cc_layout(p, nb_of(p.B)).total;
    const size_t avail = smem_optin > base + 64 ? smem_optin - base - 64 : 0;
    int slabs = (int)(avail / (16384 + 16));
    const int rest = nall - p.nres;
    if (slabs < 2) return false;
    p.nstages = slabs < 6 ? slabs : 6;
    if (p.nstages > rest) p.nstages = rest < 1 ? 1 : rest;
    int nres_s = slabs - p.nstages;
    if (nres_s > rest - p.nstages) nres_s = rest - p.nstages;
    p.nres_s = nres_s < 0 ? 0 : nres_s > 16 ? 16 : nres_s;
    p.smem_bytes = cc_layout(p, nb_of(p.B)).total;
    return p.smem_bytes <= smem_optin;
  }
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
  // 512-byte rows give every consumer warp 8 rows x one 16-byte chunk per lane of a stage, which
  // is one 32-column TMEM block of its lane quarter: the 512 columns hold 16 stages
  p.nres = row_bytes == 512 && p.stage_bytes == 32 * 512 ? 16 : 0;
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
