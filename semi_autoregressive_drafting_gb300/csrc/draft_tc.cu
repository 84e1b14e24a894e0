// draft_tc.cu -- persistent tensor-core draft kernel for larger batches (bf16 weights, B > 4).
//
// Same block of the DSpark sequential head as draft_cc.cu ("DSpark -- paper verification",
// section 1, Eqs 4, 5, 7, 8), but once B is large the bias product e W2^T (e = the gathered
// W1 rows, [B x r]) is a real dense contraction, so it runs on the 5th-generation tensor cores:
//   * MMA tile: M = 128 requests (one batch chunk), N = 128 vocab entries, K = r in 64-wide
//     slabs; A (the gathered W1 rows) is written into shared memory in the 128-byte-swizzled
//     K-major layout by the epilogue warps, B (W2 rows, stored [V][r]) arrives by 2-D TMA;
//     the fp32 accumulator lives in TMEM (4 buffers of 128 columns);
//   * warp 0 produces W2 slabs (runs ahead across tiles, chunks and steps), warp 1 issues the
//     MMAs from one thread and owns TMEM, warps 4..19 are the epilogue: four warps per TMEM
//     lane quarter, each taking 32 of a tile's 128 columns for its 32 requests, with U and the
//     target fetched as 16-byte vectors issued before the accumulator wait;
//   * the epilogue fuses +U_k, /T, the online (max, sum-exp), and Gumbel-max sampling with an
//     exact skip: with w = 1 - u (exact from the Philox bits) and q = exp(y - best), an entry
//     with w >= 1.001 q cannot beat the running best (-ln u >= w, so its score is below
//     best - 0.0009), so the two logarithms run only for the rare entries that might;
//   * per step, each block publishes one candidate per request with a 64-bit atomicMax on an
//     order-independent key, then a bounded grid barrier; the Eq 8 label runs its second pass
//     over the block's slice after the barrier from y saved in the workspace.
#include <cuda.h>

#include <cstring>

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
  size_t a, ring, ubuf, scratch, rnnbuf, misc, bars, total;
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
  L.rnnbuf = off;  // RNN: e (r), s (r), Wj z (3r) of the request being updated
  off = align_up_t(off + (rnn ? (size_t)5 * r * 4 : 0), 128);
  L.misc = off;
  off = align_up_t(off + sizeof(TMisc), 128);
  L.bars = off;
  off += (size_t)(2 * nstage + 2 * kAcc + 2 * na + 2 + 2 * nu) * 8;
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
  while (!mbar_try_wait(bar, parity)) {
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

// (max, sum-exp) of all blocks' partials, merged by one warp in a fixed order
__device__ __forceinline__ float2 merge_ml(const float2* part, int n, int lane) {
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
  TMisc* ms = (TMisc*)(smem + Lay.misc);
  uint64_t* full = (uint64_t*)(smem + Lay.bars);
  uint64_t* empty = full + nstage;
  uint64_t* acc_full = empty + nstage;
  uint64_t* acc_empty = acc_full + kAcc;
  uint64_t* a_full = acc_empty + kAcc;
  uint64_t* a_empty = a_full + na;
  uint64_t* tmem_done = a_empty + na;
  uint64_t* mma_done = tmem_done + 1;
  uint64_t* u_full = mma_done + 1;   // [nu] a U tile has landed
  uint64_t* u_empty = u_full + nu;   // [nu] every epilogue warp has read it
  uint8_t* ubuf = smem + Lay.ubuf;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nCTA = gridDim.x, cta = blockIdx.x;
  const int B = p.B, G = p.gamma, V = p.V, r = p.r;
  const int nslab = Lay.nslab;
  const int nchunk = (B + kM - 1) / kM;
  constexpr bool tgt = TGT;  // a target is given (Eq 8): fixed per instantiation
  WsHeader* hdr = p.hdr;

  // vocab tiles of this block
  const int ntile_all = (V + kNT - 1) / kNT;
  const int t0 = (int)(((long long)ntile_all * cta) / nCTA);
  const int t1 = (int)(((long long)ntile_all * (cta + 1)) / nCTA);
  const int ntile = t1 - t0;
  const int nround = pk ? (ntile + 1) / 2 : ntile;  // accumulator rounds per chunk
  const int sl0 = t0 * kNT, sl1 = min(V, t1 * kNT);  // vocab slice [sl0, sl1)

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
    for (int i = 0; i < nu; ++i) {
      mbar_init(&u_full[i], 1);
      mbar_init(&u_empty[i], kEpiWarps);
    }
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
        for (int c = 0; c < nchunk && !stop; ++c)
          for (int t = 0; t < ntile && !stop; ++t) {
            // U of the round that starts with tile t (packed: tiles t and t + 1, 64 rows each,
            // into rows 0-63 and 64-127 of the two 64-entry boxes), ahead of use
            if (nu > 0 && (!pk || (t & 1) == 0)) {
              const int us = ui % nu;
              if (ui >= nu &&
                  !wait_or_abort(&u_empty[us], (uint32_t)(((ui / nu) - 1) & 1), &ms->abort)) {
                stop = true;
                break;
              }
              uint8_t* dst = ubuf + (size_t)us * kUTile;
              const int x = (t0 + t) * kNT;
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
                  tc::tma_load_3d(dst + kSlab / 2, &tmap_u, x + kNT, ks, 0, &u_full[us], pol_u);
                  tc::tma_load_3d(dst + kSlab + kSlab / 2, &tmap_u, x + kNT + 64, ks, 0,
                                  &u_full[us], pol_u);
                }
              }
              ++ui;
            }
            for (int s = 0; s < nslab; ++s, ++g) {
              const int slot = g % nstage;
              if (g >= nstage &&
                  !wait_or_abort(&empty[slot], (uint32_t)(((g / nstage) - 1) & 1), &ms->abort)) {
                stop = true;
                break;
              }
              mbar_expect_tx(&full[slot], kSlab);
              tc::tma_load_2d(ring + (size_t)slot * kSlab, &tmap_w2, s * 64, (t0 + t) * kNT,
                              &full[slot], pol);
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
      const uint32_t idesc = tc::idesc_bf16_f32(kM, kNT);
      int g = 0, acc_i = 0;
      bool stop = false;
      for (int ks = 0; ks < G && !stop; ++ks)
        for (int c = 0; c < nchunk && !stop; ++c) {
          const int u = ks * nchunk + c, ab = u % na;
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
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  tc::mma_bf16(tmem + acc * kNT, tc::sdesc_sw128(a_s + kk * 32),
                               tc::sdesc_sw128(b_base + kk * 32), idesc, (h | s | kk) != 0);
                if (RNN) {  // a_k = hi + lo: the low halves against the same W2 slab
                  const uint32_t a_lo = a_s + nslab * ab_bytes;
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    tc::mma_bf16(tmem + acc * kNT, tc::sdesc_sw128(a_lo + kk * 32),
                                 tc::sdesc_sw128(b_base + kk * 32), idesc, 1u);
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
  if (warp < 4) return;

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
    for (int c = 0; c < nchunk && !failed; ++c) {
      const int u = ks * nchunk + c, ab = u % na;
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
      fence_proxy_async_smem();
      esync<kEpiThreads>();
      if (et == 0) mbar_arrive(&a_full[ab]);

      // ---- tiles: bias from TMEM, logits, sampling, normalisers
      const int b = c * kM + m;
      const bool row_ok = b < B;
      const size_t urow = ((size_t)b * G + ks) * V;
      TSlot st;
      tslot_init(st);
      float C = INFINITY;  // exp(m - best) of this thread's running state
      for (int rd = 0; rd < nround; ++rd, ++acc_i) {
        const int acc = acc_i % kAcc;
        const int t = pk ? 2 * rd + half : rd;  // this warp's vocabulary tile of the round
        const bool tile_ok = t < ntile;          // (packed, odd count: the last round has one)
        const int vb = (t0 + t) * kNT + cq * 32;  // first vocab entry of this thread's 32
        // the tile's U: staged by TMA (row m; 16-byte chunk (cq % 2) * 4 + g of box cq / 2 sits at
        // chunk position ^ (m % 8)), kept until the tile is done; else read from global
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
        const bool ok = mbar_wait_warp(&acc_full[acc], (uint32_t)((acc_i / kAcc) & 1));
        if (!ok) {
          failed = true;
          break;
        }
        tc::fence_after_sync();
        const uint32_t tcol = tmem + ((uint32_t)(32 * q) << 16) + acc * kNT + cq * 32;
        // groups of GE entries, rolled to keep the code small: bias from TMEM, U, GE / 4
        // independent Philox calls; the running max moves at most once per group.  (16-entry
        // groups measured slower on GB300: 3.32 against 2.97 ms per block at B = 512.)
        constexpr int GE = 8;
#pragma unroll 1
        for (int gi = 0; gi < 32 / GE; ++gi) {
          uint32_t bias[GE];
          __syncwarp();
#pragma unroll
          for (int h8 = 0; h8 < GE / 8; ++h8)  // the whole warp, every group
            tc::tmem_ld8(tcol + GE * gi + 8 * h8, *(uint32_t(*)[8])&bias[8 * h8]);
          tc::tmem_ld_wait();
          const int v = vb + GE * gi;
          if (!row_ok || !tile_ok || v >= V) continue;  // (no further warp-collective work)
          const bool full = v + GE <= V;  // every entry exists (all groups but the slice's last)
          uint4 uq[GE / 8];
#pragma unroll
          for (int h8 = 0; h8 < GE / 8; ++h8) {
            const int c8 = GE / 8 * gi + h8;  // 16-byte chunk of this thread's 32 entries
            if (nu > 0) uq[h8] = *(const uint4*)(ub + (((((cq & 1) << 2) + c8) ^ (lrow & 7)) << 4));
            else if (vec_u && full)
              uq[h8] = __ldcs((const uint4*)((const __nv_bfloat16*)p.U + urow + v + 8 * h8));
          }
          const bool vq = nu > 0 || (vec_u && full);
          float y[GE], tv[GE];
          float gmax = -INFINITY, tmax = -INFINITY;
          if (vq && full) {
#pragma unroll
            for (int e = 0; e < GE; ++e) {
              const uint32_t wd = ((const uint32_t*)&uq[e >> 3])[(e & 7) >> 1];
              const float uval = __uint_as_float((e & 1) ? (wd & 0xFFFF0000u) : (wd << 16));
              y[e] = uval + __uint_as_float(bias[e]);  // z for now
            }
            if (TGT) {
              if (vec_t) {
#pragma unroll
                for (int e = 0; e < GE; e += 4) {
                  const float4 t4 = __ldcs((const float4*)(p.target + urow + v + e));
                  tv[e] = t4.x; tv[e + 1] = t4.y; tv[e + 2] = t4.z; tv[e + 3] = t4.w;
                }
              } else {
#pragma unroll
                for (int e = 0; e < GE; ++e) tv[e] = p.target[urow + v + e];
              }
#pragma unroll
              for (int e = 0; e < GE; ++e) {
                tv[e] *= p.invT;
                tmax = fmaxf(tmax, tv[e]);
              }
            }
          } else {  // the slice's ragged end, or U rows without 16-byte alignment
#pragma unroll
            for (int e = 0; e < GE; ++e) {
              const int vv = v + e;
              float uval;
              if (vq) {
                const uint32_t wd = ((const uint32_t*)&uq[e >> 3])[(e & 7) >> 1];
                uval = __uint_as_float((e & 1) ? (wd & 0xFFFF0000u) : (wd << 16));
              } else {
                uval = vv < V ? ld_u(p.U, urow + vv, p.u_bf16) : 0.f;
              }
              y[e] = vv < V ? uval + __uint_as_float(bias[e]) : -INFINITY;  // z for now
              if (TGT) {
                tv[e] = vv < V ? p.target[urow + vv] * p.invT : -INFINITY;
                tmax = fmaxf(tmax, tv[e]);
              }
            }
          }
          if (p.logits)  // debug output: z
#pragma unroll
            for (int e = 0; e < GE; ++e)
              if (v + e < V) p.logits[urow + v + e] = y[e];
#pragma unroll
          for (int e = 0; e < GE; ++e) {  // y = z / T
            y[e] *= p.invT;
            gmax = fmaxf(gmax, y[e]);
          }
          if (gmax > st.m) {  // rescale the running sum to the new max, once per group
            st.l *= __expf(st.m - gmax);
            st.m = gmax;
            C = __expf(st.m - st.best);
          }
          uint32_t words[GE];
#pragma unroll
          for (int q4 = 0; q4 < GE / 4; ++q4) {  // independent Philox calls, one per 4 entries
            const U4 rq = philox4x32_10((uint32_t)(v >> 2) + q4, (uint32_t)ks, (uint32_t)b,
                                        kNoiseTag, p.seed_lo, p.seed_hi);
            words[4 * q4] = rq.x;
            words[4 * q4 + 1] = rq.y;
            words[4 * q4 + 2] = rq.z;
            words[4 * q4 + 3] = rq.w;
          }
          float ls[2] = {0.f, 0.f};  // two partial sums: a shorter dependency chain
#pragma unroll
          for (int e = 0; e < GE; ++e) {
            const float pe = __expf(y[e] - st.m);
            ls[e & 1] += pe;
            // exact skip: w = 1 - u; -ln u >= w, so w >= 1.001 exp(y - best) rules it out
            const float w = bits_to_uniform(~words[e]);
            if (!(w >= 1.001f * (pe * C))) {
              const float sc = y[e] + gumbel_from_uniform(bits_to_uniform(words[e]));
              if (sc > st.best) {  // entries grow along this thread's sequence: ties keep the smaller
                st.best = sc;
                st.tok = (uint32_t)(v + e);
                C = __expf(st.m - st.best);
              }
            }
          }
          st.l += ls[0] + ls[1];
          if (TGT) {
            if (tmax > st.mt) {
              st.lt *= __expf(st.mt - tmax);
              st.mt = tmax;
            }
#pragma unroll
            for (int e = 0; e < GE; ++e) st.lt += __expf(tv[e] - st.mt);
            float* yo = p.ybuf + (size_t)b * V + v;
            if (vec_t && full) {
#pragma unroll
              for (int e = 0; e < GE; e += 4) *(float4*)(yo + e) = make_float4(y[e], y[e + 1], y[e + 2], y[e + 3]);
            } else {
#pragma unroll
              for (int e = 0; e < GE; ++e)
                if (v + e < V) yo[e] = y[e];
            }
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
      // ---- merge each request's partial states (column quarters; packed: also the two tiles
      // of each round) in a fixed order, publish the candidate
      const int kpart = half * 4 + cq, npart = pk ? 8 : 4, pstride = pk ? 64 : kM;
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
        p.ml[((size_t)ks * B + b) * nCTA + cta] = make_float2(st.m, st.l);
        if (tgt) p.mlt[((size_t)ks * B + b) * nCTA + cta] = make_float2(st.mt, st.lt);
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
      const unsigned target = (unsigned)(ks + 1) * gridDim.x;
      if (ld_acquire(&hdr->arrive) < target) {
        const unsigned long long tw = globaltimer();
        while (ld_acquire(&hdr->arrive) < target) {
          if (globaltimer() - tw > kWaitLimitNs) {
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

    if (tgt) {
      // ---- Eq 8 second pass over this block's slice, all requests: normalisers of p^d, p^t
      for (int b = 0; b < B; ++b) {
        if (ew == (b % kEpiWarps)) {
          const float2 a = merge_ml(p.ml + ((size_t)ks * B + b) * nCTA, nCTA, lane);
          const float2 tt = merge_ml(p.mlt + ((size_t)ks * B + b) * nCTA, nCTA, lane);
          const float Ld = a.x + logf(a.y), Lt = tt.x + logf(tt.y);
          const float* yr = p.ybuf + (size_t)b * V;
          const float* tr = p.target + ((size_t)b * G + ks) * V;
          float acc = 0.f, acc2 = 0.f;
          int vt = sl0;  // first entry left for the scalar tail
          if (vec_t) {   // 16-byte loads (sl0 is a multiple of 128), several in flight per lane
            const int n4 = (sl1 - sl0) >> 2;
#pragma unroll 4
            for (int i = lane; i < n4; i += 32) {
              const float4 yv = __ldcs((const float4*)(yr + sl0) + i);
              const float4 tv = __ldcs((const float4*)(tr + sl0) + i);
              acc += fabsf(__expf(yv.x - Ld) - __expf(tv.x * p.invT - Lt)) +
                     fabsf(__expf(yv.y - Ld) - __expf(tv.y * p.invT - Lt));
              acc2 += fabsf(__expf(yv.z - Ld) - __expf(tv.z * p.invT - Lt)) +
                      fabsf(__expf(yv.w - Ld) - __expf(tv.w * p.invT - Lt));
            }
            vt = sl0 + 4 * n4;
          }
          for (int v = vt + lane; v < sl1; v += 32)
            acc += fabsf(__expf(yr[v] - Ld) - __expf(tr[v] * p.invT - Lt));
          acc = warp_sum(acc + acc2);
          if (lane == 0) p.l1p[((size_t)ks * B + b) * nCTA + cta] = acc;
        }
      }
      esync<kEpiThreads>();
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

  // ---- owned requests (b % nCTA == cta): tokens, log-normalisers, Eq 7 / S_k, Eq 8
  for (int b = cta + ew * nCTA; b < B; b += kEpiWarps * nCTA) {
    float surv = 1.f;
    bool alive = true;
    for (int k = 0; k < G; ++k) {
      const size_t o = (size_t)b * G + k;
      bool valid = false;
      const int x = cond_token(p, b, k, &valid);
      if (alive && !valid && lane == 0) atomicMax(&hdr->status, kErrInvalid);
      alive = alive && valid;
      const int tok = alive ? (int)key_token(ld_acquire64(&p.keys[(size_t)k * B + b])) : -1;
      const float2 ml = merge_ml(p.ml + ((size_t)k * B + b) * nCTA, nCTA, lane);
      if (p.h && p.w) {
        float acc = 0.f;
        for (int j = lane; j < p.d; j += 32)
          acc += ld_u(p.w, j, 1) * ld_u(p.h, o * p.d + j, p.u_bf16);
        for (int j = lane; j < r; j += 32)
          acc += ld_u(p.w, (size_t)p.d + j, 1) * ld_u(p.W1, (size_t)x * r + j, 1);
        acc = warp_sum(acc);
        const float cv = alive ? sigmoidf_acc(acc) : NAN;
        surv = alive ? surv * cv : NAN;
        if (lane == 0) {
          p.c[o] = cv;
          p.S[o] = surv;
        }
      }
      if (lane == 0) {
        p.tokens[o] = tok;
        p.lse[o] = alive ? ml.x + logf(ml.y) : NAN;
      }
      if (tgt && k + 1 < G) {
        float s = 0.f;
        for (int i = lane; i < nCTA; i += 32) s += p.l1p[((size_t)k * B + b) * nCTA + i];
        s = warp_sum(s);
        if (lane == 0) {
          p.l1[o] = alive ? s : NAN;
          p.cstar[o] = alive ? fminf(1.f, fmaxf(0.f, 1.f - 0.5f * s)) : NAN;
        }
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
        float s = 0.f;
        for (int i = lane; i < nCTA; i += 32) s += p.l1p[((size_t)(G - 1) * B + b) * nCTA + i];
        s = warp_sum(s);
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
  // two staged U tiles, then two A buffers, then the deepest W2 ring (at least 3 stages)
  const int nu_max = p.u_bf16 && p.V % 8 == 0 ? 2 : 0;
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
  CUtensorMap tmap;
  if (!encode_bf16_2d(&tmap, p.W2, p.V, p.r, p.r, kNT)) return cudaErrorInvalidValue;
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
  int na = p.tc_na, ns = p.nstages, nu = p.tc_nu;
  void* args[] = {(void*)&p, (void*)&tmap, (void*)&tmap_u, (void*)&na, (void*)&ns, (void*)&nu};
  return cudaLaunchCooperativeKernel(kern, dim3(nblocks), dim3(kThreads), args, p.smem_bytes, stream);
}

}  // namespace dspark
