// draft_tc.cu -- persistent tensor-core draft kernel for larger batches (bf16 weights, B > 4).
//
// Same block of the DSpark sequential head as draft_cc.cu ("DSpark -- paper verification",
// section 1, Eqs 4, 5, 7, 8), but once B is large the bias product e W2^T (e = the gathered
// W1 rows, [B x r]) is a real dense contraction, so it runs on the 5th-generation tensor cores:
//   * MMA tile: M = 128 requests (one batch chunk), N = 128 vocab entries, K = r in 64-wide
//     slabs; A (the gathered W1 rows) is written into shared memory in the 128-byte-swizzled
//     K-major layout by the epilogue warps, B (W2, stored [V][r] or as the pages write it,
//     [r][V]) arrives by 2-D TMA; the fp32 accumulator lives in TMEM (4 buffers of 128
//     columns); with at most 64 requests two vocabulary tiles share one accumulator;
//   * the blocks form one group per 128-request chunk and the blocks of a group split the
//     vocabulary, walking their tiles in a serpentine order so that W2 is re-read from L2;
//   * warp 0 produces W2 slabs and, when U is bf16 with 16-byte rows, U tiles by 3-D TMA (it
//     runs ahead across tiles, chunks and steps), warp 1 issues the MMAs from one thread and
//     owns TMEM, warps 4..19 are the epilogue: four warps per TMEM lane quarter, each taking 32
//     of a tile's 128 columns for its 32 requests;
//   * the epilogue fuses +U_k, /T, the online (max, sum-exp), and Gumbel-max sampling with an
//     exact skip, in log2 units (y2 = y log2 e, exponentials by ex2): with w = 1 - u (exact
//     from the Philox bits) and q = exp(y - best), an entry with w >= 1.001 q cannot beat the
//     running best (-ln u >= w, so its score is below best - 0.0009), so the two logarithms
//     run only for the rare entries that might; the test is one FMA and one compare per entry,
//     and the Philox rounds that do not depend on the vocabulary index are computed once;
//   * per step, each block publishes one candidate per request with a 64-bit atomicMax on an
//     order-independent key, then a bounded grid barrier; the Eq 8 label runs its second pass
//     over the block's slice from y saved in the workspace, after the barrier and while the
//     next step's first MMAs run; the target's normalisers, which do not depend on the drafted
//     tokens, come from a streaming launch before the draft (target_part_kernel), so the
//     epilogue never reads the target;
//   * the two spare warps compute Eq 7's w[:d] . h_k for the block's own requests up front (it
//     does not depend on the drafted tokens); after the last step one warp per owned (request,
//     position) finishes the token, the log-normaliser, c_k and Eq 8, then S_k.
#include <cuda.h>

#include <cstring>
#include <type_traits>

#include "draft.cuh"
#include "rnn.cuh"
#include "tc.cuh"

namespace dspark {
namespace {

constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 4 * 32 + kEpiThreads;  // producer, MMA, two spare warps, epilogue
constexpr int kM = 128;                          // requests per chunk
constexpr int kNT = 128;                         // vocab entries per tile
constexpr int kSlab = 16384;                     // bytes of one 128 x 64 bf16 swizzled slab
constexpr int kAcc = 4;                          // TMEM accumulators of kNT columns
constexpr int kTmemCols = kAcc * kNT;            // 512

struct TSlot {
  float best;
  uint32_t tok;
  float m, l, mt, lt;
};

struct TMisc {
  uint32_t tmem_base;
  int flag;
  int last;
  volatile int abort;
  float red[kEpiWarps];
};

struct TCLayout {
  size_t a, ring, ubuf, scratch, sbest, rnnbuf, misc, bars, total;
  int nslab, na, nstage, aslabs, nu;
  int abytes;  // bytes of one A slab: 128 rows, or 192 when two vocabulary tiles share a tile
};

constexpr int kUTile = 2 * kSlab;  // U of one tile: 128 requests x 128 entries bf16, two boxes

__host__ __device__ inline size_t align_up_t(size_t x, size_t a) { return (x + a - 1) / a * a; }

// RNN head: each A buffer holds the bf16 high halves of a_k, then the low halves.
// Packed mode (one chunk of at most 64 requests): each A slab holds 192 rows, [0; e; 0], so
// that rows 64..191 ([e; 0]) and rows 0..127 ([0; e]) are the A operands of two MMAs that put
// vocabulary tile t in TMEM lanes 0-63 and tile t + 1 in lanes 64-127 of one accumulator.
__host__ __device__ inline TCLayout tc_layout(int r, int na, int nstage, bool rnn, int nu,
                                              bool packed) {
  TCLayout L;
  L.nslab = (r + 63) / 64;
  L.aslabs = L.nslab * (rnn ? 2 : 1);
  L.na = na;
  L.nstage = nstage;
  L.nu = nu;
  L.abytes = packed ? kSlab * 3 / 2 : kSlab;
  size_t off = 0;
  L.a = off;
  off += (size_t)na * L.aslabs * L.abytes;
  L.ring = off;
  off += (size_t)nstage * kSlab;
  L.ubuf = off;  // U tiles staged by TMA (two 16 KB swizzled boxes of 64 entries each)
  off += (size_t)nu * kUTile;
  L.scratch = off;
  off = align_up_t(off + 4 * kM * sizeof(TSlot), 128);  // partial states of the merge
  L.sbest = off;  // running best of every (part, request row) during the tiles, [8][kM] floats
  off = align_up_t(off + 8 * kM * sizeof(float), 128);
  L.rnnbuf = off;  // RNN: e (r), s (r), Wj z (3r) of the request being updated
  off = align_up_t(off + (rnn ? (size_t)5 * r * 4 : 0), 128);
  L.misc = off;
  off = align_up_t(off + sizeof(TMisc), 128);
  L.bars = off;
  off += (size_t)(2 * nstage + 2 * kAcc + 2 * na + 3 + 2 * nu + 1) * 8;
  L.total = align_up_t(off, 1024) + 1024;  // + slack to align the dynamic base to 1024
  return L;
}

template <int NT>
__device__ __forceinline__ void esync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}
template <int NT>
__device__ __forceinline__ int esync_or(int pred) {
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

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) {
    if (*abort || globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return true;
}


__device__ __forceinline__ float ld_u(const void* p, size_t i, int bf16) {
  return bf16 ? __bfloat162float(((const __nv_bfloat16*)p)[i]) : ((const float*)p)[i];
}

__device__ __forceinline__ void tslot_init(TSlot& s) {
  s.best = -INFINITY;
  s.tok = 0xFFFFFFFFu;
  s.m = -INFINITY;
  s.l = 0.f;
  s.mt = -INFINITY;
  s.lt = 0.f;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// log2(-ln u) for the Philox word `bits`, u = (2 (bits >> 9) + 1) 2^-24: the Gumbel noise in
// log2 units is minus this.  t = -ln u = -ln(1 - w), w = 1 - u (exact): the series
// w + w^2/2 + ... + w^5/5 for w <= 1/16 (truncation below w^5/6 = 1.6e-7 relative), else
// -log2(u) ln 2 with lg2.approx (|log2 u| >= 0.093 there, so the relative error stays below
// 3e-6); both are computed and one is selected, so the lanes of a warp do not diverge.  The
// outer logarithm is lg2.approx too.  The score's error is then below 5e-6 (log2 units), far
// inside the 1e-4 band the sampler's parity treats as a near-tie.
__device__ __forceinline__ float gumbel_log2(uint32_t bits) {
  const float u = __uint_as_float(0x3F800000u | (bits >> 9)) - 0.99999994f;  // exact
  const float w = 1.f - u;                                                    // exact
  const float ts = w * fmaf(w, fmaf(w, fmaf(w, fmaf(w, 0.2f, 0.25f), 0.33333334f), 0.5f), 1.f);
  float lu, l2;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lu) : "f"(u));
  const float t = w <= 0.0625f ? ts : -lu * 0.6931471805599453f;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(t));
  return l2;
}

// 2^x on the special-function unit (relative error about 2^-22; 0 for x = -inf)
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (max, sum-exp) of all blocks' partials, merged by one warp in a fixed order: each lane issues
// the loads of up to 8 partials, the warp takes their maximum M, then sums l_i exp(m_i - M)
// (empty partials are (-inf, 0) and add nothing)
__device__ __forceinline__ float2 merge_ml(const float2* part, int n, int lane) {
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

// Sum of n floats, one warp, up to 8 loads in flight per lane (fixed order)
__device__ __forceinline__ float warp_sum_n(const float* a, int n, int lane) {
  float s = 0.f;
  for (int i0 = 0; i0 < n; i0 += 256) {
    float q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + lane + 32 * j;
      q[j] = i < n ? a[i] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) s += q[j];
  }
  return warp_sum(s);
}

// 8 bf16 (one 16-byte chunk) -> floats
__device__ __forceinline__ void bf16x8(const uint4& q, float* f) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Eq 7's two dot products for one warp (w and W1 bf16; h bf16 or fp32).  16-byte loads, four
// chunks in flight per lane, when w is 16-byte aligned; h and W1 always are (the ABI requires
// it, and d, r are multiples of 8).
// w[:d] . h[o] for the (request, position) row o
__device__ __forceinline__ float eq7_hdot(const DraftParams& p, size_t o, int lane) {
  const __nv_bfloat16* w = (const __nv_bfloat16*)p.w;
  float acc = 0.f;
  if (((uintptr_t)w & 15) == 0) {
    const int nd = p.d / 8;
    const uint4* w4 = (const uint4*)w;
    for (int j0 = 0; j0 < nd; j0 += 128) {
      uint4 wq[4];
      float hv[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + lane + 32 * u;
        wq[u] = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) hv[u][i] = 0.f;
        if (j < nd) {
          wq[u] = w4[j];
          if (p.u_bf16) {
            bf16x8(((const uint4*)((const __nv_bfloat16*)p.h + o * p.d))[j], hv[u]);
          } else {
            const float4* hp = (const float4*)((const float*)p.h + o * p.d) + 2 * j;
            *(float4*)&hv[u][0] = hp[0];
            *(float4*)&hv[u][4] = hp[1];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float wf[8];
        bf16x8(wq[u], wf);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = fmaf(wf[i], hv[u][i], acc);
      }
    }
  } else {
    for (int j = lane; j < p.d; j += 32) acc += ld_u(p.w, j, 1) * ld_u(p.h, o * p.d + j, p.u_bf16);
  }
  return warp_sum(acc);
}
// w[d:] . W1[x]
__device__ __forceinline__ float eq7_edot(const DraftParams& p, int x, int lane) {
  const __nv_bfloat16* w = (const __nv_bfloat16*)p.w;
  const __nv_bfloat16* e = (const __nv_bfloat16*)p.W1 + (size_t)x * p.r;
  float acc = 0.f;
  if (((uintptr_t)w & 15) == 0) {
    const uint4* w4 = (const uint4*)w + p.d / 8;
    for (int j = lane; j < p.r / 8; j += 32) {
      float wf[8], ef[8];
      bf16x8(w4[j], wf);
      bf16x8(((const uint4*)e)[j], ef);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(wf[i], ef[i], acc);
    }
  } else {
    for (int j = lane; j < p.r; j += 32) acc += ld_u(p.w, (size_t)p.d + j, 1) * __bfloat162float(e[j]);
  }
  return warp_sum(acc);
}

// Conditioning token of step ks for request b and whether the request is still valid.
__device__ __forceinline__ int cond_token(const DraftParams& p, int b, int ks, bool* valid) {
  const int V = p.V, G = p.gamma;
  int x = p.x0[b];
  bool ok = x >= 0 && x < V;
  if (p.forced) {
    for (int j = 0; j < ks && ok; ++j) {
      const int f = p.forced[(size_t)b * G + j];
      ok = f >= 0 && f < V;
    }
    if (ks > 0 && ok) x = p.forced[(size_t)b * G + ks - 1];
  } else if (ks > 0 && ok) {
    x = (int)key_token(ld_acquire64(&p.keys[(size_t)(ks - 1) * p.B + b]));
    ok = x >= 0 && x < V;
  }
  *valid = ok;
  return ok ? x : 0;
}

// ------------------------------------------------------------------ target normalisers
// The target's log-normaliser of every (request, position) row does not depend on the drafted
// tokens, so it is formed before the draft, at streaming speed, instead of inside the latency-
// bound epilogue: (max, sum exp) of t / T over each 16384-entry chunk, natural units, in
// mlt[(k B + b) ntp + chunk]; the Eq 8 second pass merges a row's ntp partials.
constexpr int kTChunk = 16384;
constexpr int kTThr = 256;
__host__ __device__ inline int target_chunks(int V) { return (V + kTChunk - 1) / kTChunk; }

__global__ void __launch_bounds__(kTThr) target_part_kernel(const float* __restrict__ tgt, int B, int G,
                                                            int V, float s2, float2* __restrict__ mlt) {
  __shared__ float2 red[kTThr / 32];
  const int ntp = target_chunks(V);
  const long long blk = blockIdx.x, row = blk / ntp;  // row = b G + k
  const int ch = (int)(blk % ntp);
  const int b = (int)(row / G), k = (int)(row % G);
  const float* t = tgt + row * V;
  const int v0 = ch * kTChunk, v1 = min(V, v0 + kTChunk);
  float m = -INFINITY, l = 0.f;  // log2 units here
  if ((V & 3) == 0) {  // 16-byte aligned rows: all sixteen loads of a thread at once
    const float4* t4 = (const float4*)(t + v0);
    const int n4 = (v1 - v0) >> 2;
    float4 q[kTChunk / 4 / kTThr];
#pragma unroll
    for (int u = 0; u < kTChunk / 4 / kTThr; ++u) {
      const int i = (int)threadIdx.x + u * kTThr;
      q[u] = i < n4 ? __ldcs(t4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < kTChunk / 4 / kTThr; ++u) mx = fmaxf(mx, fmaxf(fmaxf(q[u].x, q[u].y), fmaxf(q[u].z, q[u].w)));
    if (mx != -INFINITY) {
      m = mx * s2;
#pragma unroll
      for (int u = 0; u < kTChunk / 4 / kTThr; ++u)
        l += ex2f(fmaf(q[u].x, s2, -m)) + ex2f(fmaf(q[u].y, s2, -m)) + ex2f(fmaf(q[u].z, s2, -m)) +
             ex2f(fmaf(q[u].w, s2, -m));
    }
  } else {
    for (int v = v0 + (int)threadIdx.x; v < v1; v += kTThr) {
      const float y = t[v] * s2;
      if (y > m) {
        l = l * ex2f(m - y) + 1.f;
        m = y;
      } else {
        l += ex2f(y - m);
      }
    }
  }
  auto merge2 = [](float& a, float& c, float a2, float c2) {
    if (c2 == 0.f) return;
    if (c == 0.f) {
      a = a2;
      c = c2;
      return;
    }
    const float mm = fmaxf(a, a2);
    c = c * ex2f(a - mm) + c2 * ex2f(a2 - mm);
    a = mm;
  };
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) merge2(m, l, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, l, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float2(m, l);
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = -INFINITY, c = 0.f;
    for (int w = 0; w < kTThr / 32; ++w) merge2(a, c, red[w].x, red[w].y);
    mlt[((size_t)k * B + b) * ntp + ch] = make_float2(a * kLn2, c);  // natural units
  }
}

// Vocabulary tile visited at position t of unit u (one request chunk of one step): the units
// alternate direction over the block's tiles, so the W2 tiles a unit reads first are the ones
// the unit before it read last, still in L2 (W2 is loaded evict-last, U evict-first).  With
// several 128-request chunks W2 is then re-read mostly from L2 instead of once per chunk from
// DRAM, and from one step to the next the same holds.
__device__ __forceinline__ int tile_at(int t, int u, int ntile) { return (u & 1) ? ntile - 1 - t : t; }

template <bool RNN, bool TGT>
__global__ void __launch_bounds__(kThreads, 1)
    draft_tc_kernel(const DraftParams p, const __grid_constant__ CUtensorMap tmap_w2,
                    const __grid_constant__ CUtensorMap tmap_u, int na, int nstage, int nu) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const bool pk = p.tc_pk != 0;  // packed: one chunk of at most 64 requests, tiles in pairs
  const TCLayout Lay = tc_layout(p.r, na, nstage, RNN, nu, pk);
  const int ab_bytes = Lay.abytes;
  float* r_e = (float*)(smem + Lay.rnnbuf);
  float* r_s = r_e + p.r;
  float* r_u = r_s + p.r;
  uint8_t* abuf = smem + Lay.a;
  uint8_t* ring = smem + Lay.ring;
  TSlot* scratch = (TSlot*)(smem + Lay.scratch);
  volatile float* sbest = (volatile float*)(smem + Lay.sbest);
  TMisc* ms = (TMisc*)(smem + Lay.misc);
  uint64_t* full = (uint64_t*)(smem + Lay.bars);
  uint64_t* empty = full + nstage;
  uint64_t* acc_full = empty + nstage;
  uint64_t* acc_empty = acc_full + kAcc;
  uint64_t* a_full = acc_empty + kAcc;
  uint64_t* a_empty = a_full + na;
  uint64_t* tmem_done = a_empty + na;
  uint64_t* mma_done = tmem_done + 1;
  uint64_t* hdot_ready = mma_done + 1;  // the spare warps have written w[:d] . h_k (Eq 7)
  uint64_t* u_full = hdot_ready + 1;  // [nu] a U tile has landed
  uint64_t* u_empty = u_full + nu;   // [nu] every epilogue warp has read it
  uint64_t* never = u_empty + nu;    // no thread arrives on it (failure-path test hook)
  uint8_t* ubuf = smem + Lay.ubuf;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nCTA = gridDim.x, cta = blockIdx.x;
  const int B = p.B, G = p.gamma, V = p.V, r = p.r;
  const int nslab = Lay.nslab;
  const int nchunk = (B + kM - 1) / kM;
  constexpr bool tgt = TGT;  // a target is given (Eq 8): fixed per instantiation
  WsHeader* hdr = p.hdr;

  // Work split.  The blocks form ngrp groups, one per 128-request chunk (while there are no
  // more chunks than blocks); group g takes chunks g, g + ngrp, ... and its nslice blocks split
  // the vocabulary.  So a block gathers its chunk's conditioning rows once per step and walks a
  // wide vocabulary slice with one running best per request, instead of walking a narrow slice
  // once per chunk; the ngrp blocks that share a slice have adjacent ids and read the same W2
  // tiles at about the same time, so L2 serves the repeats.  Blocks past ngrp * nslice have no
  // tiles (they still take part in the barriers).
  const int ngrp = min(nchunk, nCTA);
  const int nslice = nCTA / ngrp;
  const int grp = cta % ngrp, slc = cta / ngrp;
  const int nck = grp < nchunk ? (nchunk - 1 - grp) / ngrp + 1 : 0;  // chunks of this block

  // vocab tiles of this block
  const int ntile_all = (V + kNT - 1) / kNT;
  const int t0 = slc < nslice ? (int)(((long long)ntile_all * slc) / nslice) : 0;
  const int t1 = slc < nslice ? (int)(((long long)ntile_all * (slc + 1)) / nslice) : 0;
  const int ntile = t1 - t0;
  const int nround = pk ? (ntile + 1) / 2 : ntile;  // accumulator rounds per chunk
  const int sl0 = t0 * kNT, sl1 = min(V, t1 * kNT);  // vocab slice [sl0, sl1)
  const int ntp = target_chunks(V);  // target normaliser partials per row (target_part_kernel)

  if (tid == 0) {
    for (int i = 0; i < nstage; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
    }
    for (int i = 0; i < na; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    mbar_init(tmem_done, kEpiWarps);
    mbar_init(mma_done, 1);
    mbar_init(hdot_ready, 2);
    for (int i = 0; i < nu; ++i) {
      mbar_init(&u_full[i], 1);
      mbar_init(&u_empty[i], kEpiWarps);
    }
    mbar_init(never, 1);
    fence_mbar_init();
    ms->abort = 0;
  }
  if (warp == 1) {
    tc::tmem_alloc(&ms->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();  // last block-wide barrier: roles split from here
  tc::fence_after_sync();
  const uint32_t tmem = ms->tmem_base;

  // =========================================================== producer: W2 slabs
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      const uint64_t pol_u = policy_evict_first();  // U is read once
      int g = 0, ui = 0;
      bool stop = false;
      for (int ks = 0; ks < G && !stop; ++ks)
        for (int ci = 0; ci < nck && !stop; ++ci)
          for (int t = 0; t < ntile && !stop; ++t) {
            const int c = grp + ci * ngrp;  // the chunk
            // U of the round that starts with tile t (packed: tiles t and t + 1, 64 rows each,
            // into rows 0-63 and 64-127 of the two 64-entry boxes), ahead of use
            const int u = ks * nck + ci;  // this block's unit (step, chunk)
            if (nu > 0 && (!pk || (t & 1) == 0)) {
              const int us = ui % nu;
              if (ui >= nu &&
                  !wait_or_abort(&u_empty[us], (uint32_t)(((ui / nu) - 1) & 1), &ms->abort)) {
                stop = true;
                break;
              }
              uint8_t* dst = ubuf + (size_t)us * kUTile;
              const int x = (t0 + tile_at(t, u, ntile)) * kNT;
              if (!pk) {
                mbar_expect_tx(&u_full[us], kUTile);
                tc::tma_load_3d(dst, &tmap_u, x, ks, c * kM, &u_full[us], pol_u);
                tc::tma_load_3d(dst + kSlab, &tmap_u, x + 64, ks, c * kM, &u_full[us], pol_u);
              } else {
                const bool two = t + 1 < ntile;
                mbar_expect_tx(&u_full[us], two ? kUTile : kUTile / 2);
                tc::tma_load_3d(dst, &tmap_u, x, ks, 0, &u_full[us], pol_u);
                tc::tma_load_3d(dst + kSlab, &tmap_u, x + 64, ks, 0, &u_full[us], pol_u);
                if (two) {
                  const int x2 = (t0 + tile_at(t + 1, u, ntile)) * kNT;
                  tc::tma_load_3d(dst + kSlab / 2, &tmap_u, x2, ks, 0, &u_full[us], pol_u);
                  tc::tma_load_3d(dst + kSlab + kSlab / 2, &tmap_u, x2 + 64, ks, 0,
                                  &u_full[us], pol_u);
                }
              }
              ++ui;
            }
            const int yt = (t0 + tile_at(t, u, ntile)) * kNT;
            for (int s = 0; s < nslab; ++s, ++g) {
              const int slot = g % nstage;
              if (g >= nstage &&
                  !wait_or_abort(&empty[slot], (uint32_t)(((g / nstage) - 1) & 1), &ms->abort)) {
                stop = true;
                break;
              }
              mbar_expect_tx(&full[slot], kSlab);
              if (!p.w2_rv) {  // [V][r]: 128 vocabulary rows x 64 K (K-major)
                tc::tma_load_2d(ring + (size_t)slot * kSlab, &tmap_w2, s * 64, yt, &full[slot], pol);
              } else {  // [r][V]: two boxes of 64 vocabulary entries x 64 K rows (MN-major)
                tc::tma_load_2d(ring + (size_t)slot * kSlab, &tmap_w2, yt, s * 64, &full[slot], pol);
                tc::tma_load_2d(ring + (size_t)slot * kSlab + kSlab / 2, &tmap_w2, yt + 64, s * 64,
                                &full[slot], pol);
              }
            }
          }
      if (stop) atomicMax(&hdr->status, kErrTimeout);
      for (int k = max(0, g - nstage); k < g; ++k)  // every copy must land before exit
        mbar_wait(&full[k % nstage], (uint32_t)((k / nstage) & 1));
      for (int k = max(0, ui - nu); k < ui; ++k)
        mbar_wait(&u_full[k % nu], (uint32_t)((k / nu) & 1));
    }
    return;
  }

  // =========================================================== MMA issuer + TMEM owner
  if (warp == 1) {
    if (lane == 0) {
      // W2 as [r][V] is an MN-major B operand: 64-entry blocks 8 KB apart, K steps of 16 rows
      // 2 KB apart; as [V][r] it is K-major, K steps 32 bytes apart along the swizzled rows
      // (descriptors are built once per slab; a K step adds to the 16-byte-unit address field,
      // which cannot carry: every address stays inside its slab, below the 256 KB window)
      const bool bmn = p.w2_rv != 0;
      const uint32_t idesc = tc::idesc_bf16_f32(kM, kNT) | (bmn ? tc::kIdescBMajorMN : 0u);
      const uint64_t bstep = bmn ? 2048 >> 4 : 32 >> 4;
      int g = 0, acc_i = 0;
      bool stop = false;
      for (int ks = 0; ks < G && !stop; ++ks)
        for (int ci = 0; ci < nck && !stop; ++ci) {
          const int u = ks * nck + ci, ab = u % na;
          if (!wait_or_abort(&a_full[ab], (uint32_t)((u / na) & 1), &ms->abort)) {
            stop = true;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a_base = smem_u32(abuf + (size_t)ab * Lay.aslabs * ab_bytes);
          for (int rd = 0; rd < nround && !stop; ++rd, ++acc_i) {
            const int acc = acc_i % kAcc;
            if (acc_i >= kAcc &&
                !wait_or_abort(&acc_empty[acc], (uint32_t)(((acc_i / kAcc) - 1) & 1), &ms->abort)) {
              stop = true;
              break;
            }
            tc::fence_after_sync();
            // packed: tile 2 rd against A rows 64..191 ([e; 0]), tile 2 rd + 1 against rows
            // 0..127 ([0; e]); otherwise tile rd against the 128 rows
            const int nt_rd = pk ? min(2, ntile - 2 * rd) : 1;
            for (int h = 0; h < nt_rd && !stop; ++h) {
              const uint32_t a_row = pk ? (h == 0 ? 64u * 128u : 0u) : 0u;
              for (int s = 0; s < nslab; ++s, ++g) {
                const int slot = g % nstage;
                if (!wait_or_abort(&full[slot], (uint32_t)((g / nstage) & 1), &ms->abort)) {
                  stop = true;
                  break;
                }
                tc::fence_after_sync();
                const uint32_t b_base = smem_u32(ring + (size_t)slot * kSlab);
                const uint32_t a_s = a_base + s * ab_bytes + a_row;
                const uint64_t bd = bmn ? tc::sdesc_sw128_mn(b_base, kSlab / 2) : tc::sdesc_sw128(b_base);
                const uint64_t ad = tc::sdesc_sw128(a_s);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  tc::mma_bf16(tmem + acc * kNT, ad + 2 * kk, bd + bstep * kk, idesc, (h | s | kk) != 0);
                if (RNN) {  // a_k = hi + lo: the low halves against the same W2 slab
                  const uint64_t alo = tc::sdesc_sw128(a_s + nslab * ab_bytes);
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    tc::mma_bf16(tmem + acc * kNT, alo + 2 * kk, bd + bstep * kk, idesc, 1u);
                }
                tc::mma_commit(&empty[slot]);
              }
            }
            if (!stop) tc::mma_commit(&acc_full[acc]);
          }
          if (!stop) tc::mma_commit(&a_empty[ab]);
        }
      if (stop) atomicMax(&hdr->status, kErrTimeout);
      tc::mma_commit(mma_done);  // arrives once every MMA issued above has completed
      mbar_wait(mma_done, 0);
    }
    __syncwarp();
    // TMEM is freed only after the epilogue is done reading it
    if (lane == 0) wait_or_abort(tmem_done, 0, &ms->abort);
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
    return;
  }
  // owned requests: b = cta + i nCTA (Eq 7 / S_k, tokens and normalisers are finished by them)
  const int nown = cta < B ? (B - 1 - cta) / nCTA + 1 : 0;

  // =========================================================== spare warps: w[:d] . h_k (Eq 7)
  // for every owned (request, position); these do not depend on the drafted tokens
  if (warp == 2 || warp == 3) {
    if (p.h && p.w)
      for (int pi = warp - 2; pi < nown * G; pi += 2) {
        const size_t o = (size_t)(cta + (pi / G) * nCTA) * G + pi % G;
        const float hd = eq7_hdot(p, o, lane);
        if (lane == 0) p.hdot[o] = hd;
      }
    __syncwarp();
    if (lane == 0) mbar_arrive(hdot_ready);
    return;
  }

  // =========================================================== epilogue warps
  const int et = tid - 128;          // 0..511
  const int ew = warp - 4;           // 0..15
  const int q = warp & 3;            // TMEM lane quarter
  const int cq = ew >> 2;            // 32-column quarter of each tile
  const int lrow = 32 * q + lane;    // this thread's TMEM lane (accumulator row)
  // request within the chunk: the lane, or in packed mode lane mod 64 (lanes 64-127 hold the
  // same requests for the round's second vocabulary tile)
  const int m = pk ? (lrow & 63) : lrow;
  const int half = pk ? (q >> 1) : 0;  // packed: which tile of the round
  // part of the request's row this thread holds: column quarter, and in packed mode the tile
  const int kpart = half * 4 + cq, npart = pk ? 8 : 4;
  // gather role: row and the share of the row's 16-byte chunks (packed: 64 rows, 8 shares)
  const int gm = pk ? (et & 63) : (et & (kM - 1)), gh = pk ? (et >> 6) : (et >> 7);
  const int gstep = pk ? 8 : 4;
  const int nchk = r / 8;            // 16-byte chunks of a W1 row
  // 16-byte vector loads of U (bf16) and the target need 16-byte aligned rows
  const bool vec_u = p.u_bf16 && (V % 8) == 0;
  const bool vec_t = (V % 4) == 0;
  int acc_i = 0, ui = 0;
  bool failed = false;
  if (pk) {  // rows 0-63 and 128-191 of every A slab stay zero
    for (size_t i = et; i < (size_t)na * Lay.aslabs * ab_bytes / 16; i += kEpiThreads) {
      const int row = (int)((i * 16 % ab_bytes) / 128);
      if (row < 64 || row >= 128) ((uint4*)abuf)[i] = make_uint4(0, 0, 0, 0);
    }
  }

  // y and the target in log2 units: y2 = z log2(e) / T, so that 2^(y2 - m2) = exp(y - m)
  const float s2 = p.invT * kLog2e;
  const void* const Up = p.U;
  const float* const tgp = p.target;
  float* const lgp = p.logits;
  float* const ybp = p.ybuf;

  // One group of 8 consecutive vocabulary entries v..v+7 of this thread's row: logits (Eq 4),
  // the online normaliser, Philox Gumbel-max with the exact skip; with a target, y saved for the
  // Eq 8 second pass.  st.m, st.best and tb are in log2 units here (y2 = z s2), and pairs of
  // entries go through the packed fp32 instructions (add, fma on float2).
  //
  // Normaliser: st.m is a reference point, not the running maximum.  The row's first group sets
  // it to that group's maximum; lsum accumulates 2^(y2 - st.m) over the row.  Later groups skip
  // the maximum and are rescaled only when their sum passes 2^64 (an entry more than 64
  // octaves above the reference; inf included), which routes them to the rare path below.
  //
  // Skip test: with w = 1 - u (u the entry's uniform) and q = exp(y - best), an entry with
  // w >= 1.001 q cannot win (-ln u >= w, so its score is below best - 0.0009 in natural units).
  // f = 0x3F800000 | (bits >> 9) (one funnel shift) is the float 1 + u - 2^-24 = 2 - 2^-24 - w,
  // on the 2^-23 grid of [1, 2).  P = pe Cp is the computed 1.002 q (within 1e-5 of it), and
  // X = fl(2 - P) (one fma).  An entry is a candidate iff f >= X; a skipped one has
  // f <= X - 2^-23 <= 2 - P - 2^-24, i.e. w >= P >= 1.001 q, so it is one the exact fp32
  // comparison would also reject.  (P = 0 x inf gives X = NaN: not a candidate, and such an
  // entry, y = -inf or 126 octaves below the first group's maximum, cannot win.)
  // FAST (a compile-time constant at each call): all 8 entries exist, U is staged, no debug
  // output, and the target (if any) has 16-byte aligned rows.
  auto group = [&](auto fast_tag, int gi, int vb, const uint32_t* bs, const uint8_t* ub,
                   size_t urow, int b, TSlot& st, float2& lsum, float& tb, float& Cp,
                   const PhiloxFixed& pfx, volatile float* sb_own) {
    constexpr bool FAST = decltype(fast_tag)::value;
    const int v = vb + 8 * gi;
    if (!FAST && v >= V) return;
    const bool full = FAST || v + 8 <= V;
    float z[8];
    uint4 uq = make_uint4(0, 0, 0, 0);
    bool vq = false;
    if (FAST || nu > 0) {  // staged: 16-byte chunk (cq % 2) * 4 + gi of the row sits at chunk ^ (row % 8)
      uq = *(const uint4*)(ub + (((((cq & 1) << 2) + gi) ^ (lrow & 7)) << 4));
      vq = true;
    } else if (vec_u && full) {
      uq = __ldcs((const uint4*)((const __nv_bfloat16*)Up + urow + v));
      vq = true;
    }
    if (FAST || (vq && full)) {
      const uint32_t uw[4] = {uq.x, uq.y, uq.z, uq.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 zz = __fadd2_rn(
            make_float2(__uint_as_float(uw[i] << 16), __uint_as_float(uw[i] & 0xFFFF0000u)),
            make_float2(__uint_as_float(bs[2 * i]), __uint_as_float(bs[2 * i + 1])));
        z[2 * i] = zz.x;
        z[2 * i + 1] = zz.y;
      }
    } else {  // the slice's ragged end, or U rows without 16-byte alignment
      float uf[8];
      bf16x8(uq, uf);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int vv = v + e;
        const float uval = vq ? uf[e] : (vv < V ? ld_u(Up, urow + vv, p.u_bf16) : 0.f);
        z[e] = vv < V ? uval + __uint_as_float(bs[e]) : -INFINITY;
      }
    }
    if (!FAST && lgp)  // debug output: z
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (v + e < V) lgp[urow + v + e] = z[e];
    uint32_t wd[8];
    {
      const U4 r0 = philox_var((uint32_t)(v >> 2), pfx, p.rk0, p.rk1);
      const U4 r1 = philox_var((uint32_t)(v >> 2) + 1u, pfx, p.rk0, p.rk1);
      wd[0] = r0.x; wd[1] = r0.y; wd[2] = r0.z; wd[3] = r0.w;
      wd[4] = r1.x; wd[5] = r1.y; wd[6] = r1.z; wd[7] = r1.w;
    }
    if (st.m == -INFINITY) {  // the row's first group: the normaliser's reference point, and
      // the running best seeded with the exact score of the group's largest entry (a real
      // score, so a lower bound of the row's best: without it every entry of the group would be
      // a candidate).  That entry is tested again below and changes nothing.
      int es = 0;
      float zs = z[0];
#pragma unroll
      for (int e = 1; e < 8; ++e)
        if (z[e] > zs) {
          zs = z[e];
          es = e;
        }
      st.m = zs * s2;
      if (zs != -INFINITY) {
        uint32_t ws = wd[0];
#pragma unroll
        for (int e = 1; e < 8; ++e)
          if (es == e) ws = wd[e];
        const float sc = zs * s2 - gumbel_log2(ws);
        if (sc > st.best || (sc == st.best && (uint32_t)(v + es) < st.tok)) {
          st.best = sc;
          st.tok = (uint32_t)(v + es);
        }
        *sb_own = st.best;
        tb = fmaxf(tb, st.best);
      }
      Cp = 1.002f * ex2f(st.m - tb);
    }
    const float2 s22 = make_float2(s2, s2);
    float2 nm2 = make_float2(-st.m, -st.m);
    float2 pe[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t2 = __ffma2_rn(make_float2(z[2 * i], z[2 * i + 1]), s22, nm2);
      pe[i] = make_float2(ex2f(t2.x), ex2f(t2.y));
    }
    float2 gs = __fadd2_rn(__fadd2_rn(pe[0], pe[1]), __fadd2_rn(pe[2], pe[3]));
    bool any = gs.x > 0x1p64f || gs.y > 0x1p64f;
    const float2 ncp2 = make_float2(-Cp, -Cp), two2 = make_float2(2.f, 2.f);
    float X[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x2 = __ffma2_rn(pe[i], ncp2, two2);
      X[2 * i] = x2.x;
      X[2 * i + 1] = x2.y;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) any = any || __uint_as_float(__funnelshift_r(wd[e], 0x7Fu, 9)) >= X[e];
    if (any) {  // rare: a rescale of the reference, or entries that might beat the running best
      if (gs.x + gs.y > 0x1p64f) {
        const float gmax = fmaxf(fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3])),
                                 fmaxf(fmaxf(z[4], z[5]), fmaxf(z[6], z[7]))) * s2;
        const float sc = ex2f(st.m - gmax);
        lsum = make_float2(lsum.x * sc, lsum.y * sc);
        st.m = gmax;
        Cp = 1.002f * ex2f(st.m - tb);
        nm2 = make_float2(-st.m, -st.m);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 t2 = __ffma2_rn(make_float2(z[2 * i], z[2 * i + 1]), s22, nm2);
          pe[i] = make_float2(ex2f(t2.x), ex2f(t2.y));
          X[2 * i] = fmaf(pe[i].x, -Cp, 2.f);
          X[2 * i + 1] = fmaf(pe[i].y, -Cp, 2.f);
        }
        gs = __fadd2_rn(__fadd2_rn(pe[0], pe[1]), __fadd2_rn(pe[2], pe[3]));
      }
      uint32_t mask = 0;  // entries that might beat the running best
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (__uint_as_float(__funnelshift_r(wd[e], 0x7Fu, 9)) >= X[e]) mask |= 1u << e;
      if (mask) {  // the candidates in order; the lanes of a warp hold different requests, so
                   // this runs whenever any lane has one
        while (mask) {
          const int e = __ffs(mask) - 1;
          mask &= mask - 1;
          // z[e], wd[e] by a three-level select on the bits of e (registers cannot be indexed)
          const bool b0 = e & 1, b1 = e & 2, b2 = e & 4;
          const float z01 = b0 ? z[1] : z[0], z23 = b0 ? z[3] : z[2];
          const float z45 = b0 ? z[5] : z[4], z67 = b0 ? z[7] : z[6];
          const uint32_t w01 = b0 ? wd[1] : wd[0], w23 = b0 ? wd[3] : wd[2];
          const uint32_t w45 = b0 ? wd[5] : wd[4], w67 = b0 ? wd[7] : wd[6];
          const float ze = b2 ? (b1 ? z67 : z45) : (b1 ? z23 : z01);
          const uint32_t we = b2 ? (b1 ? w67 : w45) : (b1 ? w23 : w01);
          const float sc = ze * s2 - gumbel_log2(we);
          // ties go to the smaller entry whatever order the tiles are visited in
          if (sc > st.best || (sc == st.best && (uint32_t)(v + e) < st.tok)) {
            st.best = sc;
            st.tok = (uint32_t)(v + e);
          }
        }
        *sb_own = st.best;
        tb = fmaxf(tb, st.best);
        Cp = 1.002f * ex2f(st.m - tb);
      }
    }
    lsum = __fadd2_rn(lsum, gs);
    if (TGT) {  // the target's normalisers come from target_part_kernel
      float* yo = ybp + (size_t)b * V + v;  // y2 = z s2, read back by the second pass
      if (FAST || (vec_t && full)) {
        *(float4*)yo = make_float4(z[0] * s2, z[1] * s2, z[2] * s2, z[3] * s2);
        *(float4*)(yo + 4) = make_float4(z[4] * s2, z[5] * s2, z[6] * s2, z[7] * s2);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (v + e < V) yo[e] = z[e] * s2;
      }
    }
  };

  // Eq 8 of step kp over this block's slice, once every block has published step kp.
  // (1) The global normalisers of p^d and p^t of each request of a chunk: eight threads per
  //     request merge the slices' partials in a fixed order, every load of a batch in flight at
  //     once, then three shuffles; the results go to shared memory (the merge scratch, idle
  //     until the tiles end).
  // (2) One warp per request: the slice's sum of |p^d - p^t| from y2 (the workspace, still in
  //     L2 from the first pass) and the target, eight 16-byte loads of each in flight per lane.
  //     (Prefetching the target slice into L2 when the block publishes a step, or the
  //     candidates' W1 rows, measured slower: both evict data the step reads again.)
  auto second_pass = [&](int kp) {
    float2* const LdLt = (float2*)scratch;  // [kM]: (Ld2, Lt2) of the requests of one chunk
    for (int ci2 = 0; ci2 < nck; ++ci2) {
      const int cb = (grp + ci2 * ngrp) * kM;  // the chunk's first request
      const int nr = min(kM, B - cb);
      for (int r0 = 0; r0 < nr; r0 += kEpiThreads / 8) {
        const int i = r0 + et / 8, sub = et & 7;
        float M = -INFINITY, L = 0.f, Mt = -INFINITY, Lt = 0.f;
        if (i < nr) {
          // up to 20 slices and 2 target chunks per thread in one round of loads (152 slices
          // and 16 chunks at most on GB300); more take further rounds
          const float2* pd = p.ml + ((size_t)kp * B + cb + i) * nCTA;
          const float2* pt = p.mlt + ((size_t)kp * B + cb + i) * ntp;
          for (int j0 = sub, t0 = sub; j0 < nslice || t0 < ntp; j0 += 160, t0 += 16) {
            float2 q[20], qt[2];
#pragma unroll
            for (int j = 0; j < 20; ++j)
              q[j] = j0 + 8 * j < nslice ? pd[j0 + 8 * j] : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int j = 0; j < 2; ++j)
              qt[j] = t0 + 8 * j < ntp ? pt[t0 + 8 * j] : make_float2(-INFINITY, 0.f);
            float mb = M;
#pragma unroll
            for (int j = 0; j < 20; ++j) mb = fmaxf(mb, q[j].x);
            if (mb > -INFINITY) {
              float sum = L * __expf(M - mb);
#pragma unroll
              for (int j = 0; j < 20; ++j) sum += q[j].y * __expf(q[j].x - mb);
              M = mb;
              L = sum;
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) lse_merge(Mt, Lt, qt[j].x, qt[j].y);
          }
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {  // the request's eight threads are adjacent lanes
          lse_merge(M, L, __shfl_xor_sync(0xffffffffu, M, o), __shfl_xor_sync(0xffffffffu, L, o));
          lse_merge(Mt, Lt, __shfl_xor_sync(0xffffffffu, Mt, o), __shfl_xor_sync(0xffffffffu, Lt, o));
        }
        if (i < nr && sub == 0)
          LdLt[i] = make_float2((M + logf(L)) * kLog2e, (Mt + logf(Lt)) * kLog2e);
      }
      esync<kEpiThreads>();
      for (int i = ew; i < nr; i += kEpiWarps) {
        const int b = cb + i;
        const float Ld2 = LdLt[i].x, Lt2 = LdLt[i].y;
        const float* yr = ybp + (size_t)b * V;
        const float* tr = tgp + ((size_t)b * G + kp) * V;
        float acc = 0.f;
        int vt = sl0;  // first entry left for the scalar tail
        if (vec_t) {   // sl0 is a multiple of 128
          const int n4 = (sl1 - sl0) >> 2;
          const float4* y4 = (const float4*)(yr + sl0);
          const float4* t4 = (const float4*)(tr + sl0);
          for (int i0 = 0; i0 < n4; i0 += 256) {
            float4 yv[8], tq[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int q = i0 + lane + 32 * j;
              yv[j] = q < n4 ? __ldcs(y4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
              tq[j] = q < n4 ? __ldcs(t4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (i0 + lane + 32 * j < n4)
                acc += fabsf(ex2f(yv[j].x - Ld2) - ex2f(tq[j].x * s2 - Lt2)) +
                       fabsf(ex2f(yv[j].y - Ld2) - ex2f(tq[j].y * s2 - Lt2)) +
                       fabsf(ex2f(yv[j].z - Ld2) - ex2f(tq[j].z * s2 - Lt2)) +
                       fabsf(ex2f(yv[j].w - Ld2) - ex2f(tq[j].w * s2 - Lt2));
          }
          vt = sl0 + 4 * n4;
        }
        for (int v = vt + lane; v < sl1; v += 32)
          acc += fabsf(ex2f(yr[v] - Ld2) - ex2f(tr[v] * s2 - Lt2));
        acc = warp_sum(acc);
        if (lane == 0) p.l1p[((size_t)kp * B + b) * nCTA + slc] = acc;
      }
      esync<kEpiThreads>();  // LdLt is rewritten for the next chunk
    }
  };

  for (int ks = 0; ks < G && !failed; ++ks) {
    if (RNN) {
      // Eq 6 for the requests this block owns (b = cta mod grid), published for every block
      for (int b = cta; b < B; b += nCTA) {
        bool valid = false;
        const int x = cond_token(p, b, ks, &valid);
        for (int j = et; j < r; j += kEpiThreads) {
          r_e[j] = __bfloat162float(((const __nv_bfloat16*)p.W1)[(size_t)x * r + j]);
          r_s[j] = ks == 0 ? (p.s0 ? p.s0[(size_t)b * r + j] : 0.f) : p.rnn_s[(size_t)b * r + j];
        }
        esync<kEpiThreads>();
        rnn_row_update<kEpiThreads>(p, b, ks, r_s, r_e, r_u, p.rnn_a + ((size_t)ks * B + b) * r, et);
        for (int j = et; j < r; j += kEpiThreads) p.rnn_s[(size_t)b * r + j] = r_s[j];
        esync<kEpiThreads>();
        if (et == 0) st_release_u32(&p.rnn_flag[(size_t)ks * B + b], (unsigned)(ks + 1));
      }
    }
    for (int ci = 0; ci < nck && !failed; ++ci) {
      const int c = grp + ci * ngrp;  // the chunk
      const int u = ks * nck + ci, ab = u % na;
      // ---- A operand: the chunk's conditioning rows W1[x_{k-1}], swizzled K-major bf16
      if (u >= na) {
        const bool ok = wait_or_abort(&a_empty[ab], (uint32_t)(((u / na) - 1) & 1), &ms->abort);
        if (esync_or<kEpiThreads>(!ok)) {
          failed = true;
          break;
        }
      }
      bool gok = true;
      {
        const int b = c * kM + gm;
        bool valid = false;
        const int x = b < B ? cond_token(p, b, ks, &valid) : 0;
        const int arow = pk ? 64 + gm : gm;  // packed: the e rows are rows 64..127
        uint8_t* dst = abuf + (size_t)ab * Lay.aslabs * ab_bytes + (arow >> 3) * 1024 + (arow & 7) * 128;
        if (!RNN) {
          const uint4* src = (const uint4*)((const __nv_bfloat16*)p.W1 + (size_t)x * r);
          for (int j = gh; j < nslab * 8; j += gstep) {
            const uint4 val = (valid && j < nchk) ? src[j] : make_uint4(0, 0, 0, 0);
            *(uint4*)(dst + (j >> 3) * ab_bytes + (((j & 7) ^ (arow & 7)) << 4)) = val;
          }
        } else {
          // the flag is read with acquire semantics by this thread, so plain loads of the a_k
          // it publishes see the owner's stores
          if (b < B) gok = wait_flag(&p.rnn_flag[(size_t)ks * B + b], (unsigned)(ks + 1));
          const float* src = p.rnn_a + ((size_t)ks * B + b) * r;
          for (int j = gh; j < nslab * 8; j += gstep) {
            uint32_t hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
            if (gok && valid && j < nchk) {
              float av[8];
              *(float4*)&av[0] = *(const float4*)(src + 8 * j);
              *(float4*)&av[4] = *(const float4*)(src + 8 * j + 4);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float a0 = av[2 * e];
                const float a1 = av[2 * e + 1];
                const __nv_bfloat16 h0 = __float2bfloat16_rn(a0), h1 = __float2bfloat16_rn(a1);
                const __nv_bfloat16 l0 = __float2bfloat16_rn(a0 - __bfloat162float(h0));
                const __nv_bfloat16 l1 = __float2bfloat16_rn(a1 - __bfloat162float(h1));
                hi[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                lo[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
              }
            }
            const int off = (j >> 3) * ab_bytes + (((j & 7) ^ (arow & 7)) << 4);
            *(uint4*)(dst + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *(uint4*)(dst + nslab * ab_bytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
      }
      if (esync_or<kEpiThreads>(!gok)) {
        failed = true;
        break;
      }
      sbest[kpart * kM + m] = -INFINITY;  // no best known yet for this chunk and step
      fence_proxy_async_smem();
      esync<kEpiThreads>();
      if (et == 0) mbar_arrive(&a_full[ab]);

      // Eq 8 of the previous step, while the MMAs of this step's first rounds run
      if (tgt && ci == 0 && ks > 0) {
        second_pass(ks - 1);
        esync<kEpiThreads>();
      }

      // ---- tiles: bias from TMEM, logits, sampling, normalisers
      const int b = c * kM + m;
      const bool row_ok = b < B;
      const size_t urow = ((size_t)b * G + ks) * V;
      const PhiloxFixed pfx = philox_fix((uint32_t)ks, (uint32_t)b, kNoiseTag, p.seed_lo, p.seed_hi);
      TSlot st;
      tslot_init(st);
      float2 lsum = make_float2(0.f, 0.f);  // sum of 2^(y2 - st.m) over the row so far, in two halves
      // The skip threshold uses tb, the best score known for this request in the block: this
      // thread's own and the other parts' (the 4 column quarters, and in packed mode the two
      // tiles of a round, hold the same requests), published in shared memory.  An entry
      // skipped against another part's score is below a score that part has evaluated, so it
      // cannot win; a stale (smaller) value only skips less.
      float tb = -INFINITY;
      float Cp = INFINITY;           // 1.002 exp(m - tb)
      volatile float* const sb_own = sbest + kpart * kM + m;
      for (int rd = 0; rd < nround; ++rd, ++acc_i) {
        const int acc = acc_i % kAcc;
        const int t = pk ? 2 * rd + half : rd;  // this warp's tile position of the round
        const bool tile_ok = t < ntile;          // (packed, odd count: the last round has one)
        const int vb = (t0 + tile_at(t, u, ntile)) * kNT + cq * 32;  // first entry of this thread's 32
        // the tile's U: staged by TMA, kept until the tile is done; else read from global
        int us = -1;
        if (nu > 0) {
          us = ui % nu;
          const bool oku = mbar_wait_warp(&u_full[us], (uint32_t)((ui / nu) & 1));
          ++ui;
          if (!oku) {
            failed = true;
            break;
          }
        }
        const uint8_t* ub = nu > 0 ? ubuf + (size_t)us * kUTile + (cq >> 1) * kSlab + lrow * 128 : nullptr;
        const bool ok = p.test_stuck == 2 ? mbar_wait_warp_lim(never, 0, p.test_wait_ns)
                                          : mbar_wait_warp(&acc_full[acc], (uint32_t)((acc_i / kAcc) & 1));
        if (!ok) {
          failed = true;
          break;
        }
        tc::fence_after_sync();
        const uint32_t tcol = tmem + ((uint32_t)(32 * q) << 16) + acc * kNT + cq * 32;
        if (row_ok) {  // the other parts' bests for this request
          float ob = -INFINITY;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < npart && i != kpart) ob = fmaxf(ob, sbest[i * kM + m]);
          if (ob > tb) {
            tb = ob;
            Cp = 1.002f * ex2f(st.m - tb);
          }
        }
        // one 8-column TMEM load (the whole warp) per 8-entry group; the loops stay rolled to
        // keep the code small.  Whole staged tiles without debug output take the fast group
        // (the condition is the same for every lane of the warp).
        if (tile_ok && nu > 0 && lgp == nullptr && vb + 32 <= V && (!TGT || vec_t)) {
#pragma unroll 1
          for (int gi = 0; gi < 4; ++gi) {
            uint32_t bias[8];
            __syncwarp();
            tc::tmem_ld8_wait(tcol + 8 * gi, bias);
            if (row_ok) group(std::true_type{}, gi, vb, bias, ub, urow, b, st, lsum, tb, Cp, pfx, sb_own);
          }
        } else {
#pragma unroll 1
          for (int gi = 0; gi < 4; ++gi) {
            uint32_t bias[8];
            __syncwarp();
            tc::tmem_ld8_wait(tcol + 8 * gi, bias);
            if (row_ok && tile_ok) group(std::false_type{}, gi, vb, bias, ub, urow, b, st, lsum, tb, Cp, pfx, sb_own);
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&acc_empty[acc]);
          if (nu > 0) mbar_arrive(&u_empty[us]);
        }
      }
      if (esync_or<kEpiThreads>(failed)) {
        failed = true;
        break;
      }
      // back to natural units for the normalisers (the published best stays in log2 units: it
      // is only compared with other blocks' log2 scores)
      st.l = lsum.x + lsum.y;
      st.m *= kLn2;
      st.mt *= kLn2;
      // ---- merge each request's partial states (column quarters; packed: also the two tiles
      // of each round) in a fixed order, publish the candidate
      const int pstride = pk ? 64 : kM;
      if (kpart > 0) scratch[(kpart - 1) * pstride + m] = st;
      esync<kEpiThreads>();
      if (kpart == 0 && row_ok) {
        for (int i = 0; i < npart - 1; ++i) {
          const TSlot& o = scratch[i * pstride + m];
          best_merge(st.best, st.tok, o.best, o.tok);
          lse_merge(st.m, st.l, o.m, o.l);
          lse_merge(st.mt, st.lt, o.mt, o.lt);
        }
        bool valid = false;
        cond_token(p, b, ks, &valid);
        if (valid && ntile > 0 && sl1 > sl0) atomicMax(&p.keys[(size_t)ks * B + b], make_key(st.best, st.tok));
        p.ml[((size_t)ks * B + b) * nCTA + slc] = make_float2(st.m, st.l);
      }
      esync<kEpiThreads>();
    }
    if (failed) break;

    // ---- every block has published step ks
    esync<kEpiThreads>();
    if (et == 0) {
      int ok = 1;
      __threadfence();
      red_release_add(&hdr->arrive, 1u);
      // (the test hook waits for one arrival more than there are blocks, with a short limit)
      const unsigned target = (unsigned)(ks + 1) * gridDim.x + (p.test_stuck == 1 ? 1u : 0u);
      const unsigned long long lim = p.test_stuck == 1 ? p.test_wait_ns : kWaitLimitNs;
      if (ld_acquire(&hdr->arrive) < target) {
        const unsigned long long tw = globaltimer();
        while (ld_acquire(&hdr->arrive) < target) {
          if (globaltimer() - tw > lim) {
            ok = 0;
            break;
          }
          __nanosleep(32);
        }
      }
      __threadfence();
      ms->flag = ok;
    }
    esync<kEpiThreads>();
    if (!ms->flag) {
      failed = true;
      break;
    }
  }

  // release TMEM to its owner (also on the failure path)
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(tmem_done);
  if (failed) {
    ms->abort = 1;
    if (et == 0) atomicMax(&hdr->status, kErrTimeout);
    return;
  }
  if (tgt) {  // Eq 8 of the last step
    second_pass(G - 1);
    esync<kEpiThreads>();
  }

  // ---- owned requests, one warp per (request, position): token, log-normaliser, Eq 7, and
  // Eq 8 for all but the last position (the last block out finishes that one)
  const bool conf = p.h && p.w;
  if (conf && !mbar_wait_warp(hdot_ready, 0) && lane == 0) atomicMax(&hdr->status, kErrTimeout);
  for (int pi = ew; pi < nown * G; pi += kEpiWarps) {
    const int b = cta + (pi / G) * nCTA, k = pi % G;
    const size_t o = (size_t)b * G + k;
    bool valid = false;  // once false, false for every later position of the request
    const int x = cond_token(p, b, k, &valid);
    if (!valid && lane == 0) atomicMax(&hdr->status, kErrInvalid);
    const int tok = valid ? (int)key_token(ld_acquire64(&p.keys[(size_t)k * B + b])) : -1;
    const float2 ml = merge_ml(p.ml + ((size_t)k * B + b) * nCTA, nslice, lane);
    if (conf) {
      const float z7 = ((volatile float*)p.hdot)[o] + eq7_edot(p, x, lane);
      if (lane == 0) p.c[o] = valid ? sigmoidf_acc(z7) : NAN;
    }
    if (lane == 0) {
      p.tokens[o] = tok;
      p.lse[o] = valid ? ml.x + logf(ml.y) : NAN;
    }
    if (tgt && k + 1 < G) {
      const float s = warp_sum_n(p.l1p + ((size_t)k * B + b) * nCTA, nslice, lane);
      if (lane == 0) {
        p.l1[o] = valid ? s : NAN;
        p.cstar[o] = valid ? fminf(1.f, fmaxf(0.f, 1.f - 0.5f * s)) : NAN;
      }
    }
  }
  if (conf) {  // S_k = prod_{i <= k} c_i, from the c this block's warps just wrote
    esync<kEpiThreads>();
    for (int i = et; i < nown; i += kEpiThreads) {
      const size_t o = (size_t)(cta + i * nCTA) * G;
      float surv = 1.f;
      for (int k = 0; k < G; ++k) {
        surv *= ((volatile float*)p.c)[o + k];
        p.S[o + k] = surv;
      }
    }
  }

  if (RNN && p.s_out)
    for (int b = cta; b < B; b += nCTA)
      for (int j = et; j < r; j += kEpiThreads) p.s_out[(size_t)b * r + j] = p.rnn_s[(size_t)b * r + j];

  // last block out: Eq 8 of the final step; leave the workspace ready for the next call
  esync<kEpiThreads>();
  if (et == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&hdr->exit_count, 1u);
    ms->last = (old == (unsigned)nCTA - 1u);
  }
  esync<kEpiThreads>();
  if (ms->last) {
    __threadfence();
    if (tgt)
      for (int b = ew; b < B; b += kEpiWarps) {
        const float s = warp_sum_n(p.l1p + ((size_t)(G - 1) * B + b) * nCTA, nslice, lane);
        if (lane == 0) {
          const size_t o = (size_t)b * G + G - 1;
          const bool vb = ((volatile int32_t*)p.tokens)[o] >= 0;
          p.l1[o] = vb ? s : NAN;
          p.cstar[o] = vb ? fminf(1.f, fmaxf(0.f, 1.f - 0.5f * s)) : NAN;
        }
      }
    for (int i = et; i < G * B; i += kEpiThreads) p.keys[i] = 0ull;
    if (RNN)
      for (int i = et; i < G * B; i += kEpiThreads) p.rnn_flag[i] = 0u;
    esync<kEpiThreads>();
    if (et == 0) {
      hdr->arrive = 0;
      hdr->exit_count = 0;
      __threadfence();
    }
  }
}

}  // namespace

int draft_tc_supported(int B, int r, int w_bf16) { return w_bf16 && B >= 1 && r % 8 == 0 && r <= 512; }

bool draft_tc_configure(DraftParams& p, size_t smem_optin) {
  // U tiles are staged by TMA when U is bf16 with 16-byte aligned rows; prefer (at most 64
  // requests) vocabulary tiles in pairs so that all 128 TMEM lanes and epilogue warps work, then
  // the most staged U tiles (up to 3: measured at B = 512, one staged tile costs 1.5x, a third
  // one saves 3% over two), then two A buffers, then the deepest W2 ring (at least 3 stages;
  // 3 and 5 measured the same)
  const int nu_max = p.u_bf16 && p.V % 8 == 0 ? 3 : 0;
  for (int pk = p.B <= 64 ? 1 : 0; pk >= 0; --pk)
    for (int nu = nu_max; nu >= 0; --nu)
      for (int na = 2; na >= 1; --na)
        for (int ns = 8; ns >= 3; --ns) {
          const TCLayout L = tc_layout(p.r, na, ns, p.head == 1, nu, pk != 0);
          if (L.total <= smem_optin && (nu > 0 || nu_max == 0 || pk == 0)) {
            p.tc_pk = pk;
            p.tc_na = na;
            p.tc_nu = nu;
            p.nstages = ns;
            p.smem_bytes = L.total;
            return true;
          }
        }
  return false;
}

cudaError_t launch_draft_tc(DraftParams& p, int nblocks, cudaStream_t stream) {
  CUtensorMap tmap;  // W2 tiles: [V][r] in boxes of 128 rows x 64 K, [r][V] in 64 x 64 boxes
  if (!(p.w2_rv ? encode_bf16_2d(&tmap, p.W2, p.r, p.V, p.V, 64)
                : encode_bf16_2d(&tmap, p.W2, p.V, p.r, p.r, kNT)))
    return cudaErrorInvalidValue;
  const bool tg = p.target != nullptr;
  const void* kern = p.head == 1 ? (tg ? (const void*)draft_tc_kernel<true, true>
                                       : (const void*)draft_tc_kernel<true, false>)
                                 : (tg ? (const void*)draft_tc_kernel<false, true>
                                       : (const void*)draft_tc_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)p.smem_bytes);
  if (e != cudaSuccess) return e;
  CUtensorMap tmap_u;
  std::memset(&tmap_u, 0, sizeof tmap_u);
  if (p.tc_nu > 0 && !encode_u_bf16_3d(&tmap_u, p.U, p.B, p.gamma, p.V, p.tc_pk ? 64 : 128))
    return cudaErrorInvalidValue;
  if (tg) {  // the target's normalisers first, on the same stream
    const int ntp = target_chunks(p.V);
    target_part_kernel<<<(unsigned)((long long)p.B * p.gamma * ntp), kTThr, 0, stream>>>(
        p.target, p.B, p.gamma, p.V, p.invT * kLog2e, p.mlt);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  int na = p.tc_na, ns = p.nstages, nu = p.tc_nu;
  void* args[] = {(void*)&p, (void*)&tmap, (void*)&tmap_u, (void*)&na, (void*)&ns, (void*)&nu};
  return cudaLaunchCooperativeKernel(kern, dim3(nblocks), dim3(kThreads), args, p.smem_bytes, stream);
}

}  // namespace dspark
