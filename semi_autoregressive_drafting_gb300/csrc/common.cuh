// common.cuh -- device helpers shared by the libdspark kernels (sm_103a only).
//
// Philox4x32-10 here is written from the round function published by Salmon, Moraes, Dror and
// Shaw ("Parallel Random Numbers: As Easy as 1, 2, 3", SC'11).  Every wait between thread
// blocks and every mbarrier wait is bounded by %globaltimer; when a bound runs out the kernel
// records DSPARK_ERR_TIMEOUT in the workspace status word and unwinds instead of hanging.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dspark {

// status codes (same values as dspark_status in include/dspark.h)
constexpr unsigned kOk = 0, kErrInvalid = 1, kErrTimeout = 4;

constexpr uint32_t kNoiseTag = 0x44535052u;  // "DSPR": 4th counter word of the sampling noise
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // one second per wait
// Longest a thread stays suspended inside one mbarrier try_wait before it re-checks its abort
// flag and time bound; it resumes as soon as the phase completes, so waiting threads take no
// issue slots from the warps doing the work.
constexpr uint32_t kSuspendHintNs = 20000;

// Workspace header (first 256 bytes of every draft workspace).
struct WsHeader {
  unsigned status;      // most severe device error since the last dspark_get_status()
  unsigned arrive;      // grid-barrier arrivals during the current launch
  unsigned exit_count;  // thread blocks that have finished the current launch
  unsigned pad[61];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

// ------------------------------------------------------------------ Philox4x32-10 and noise

struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                            uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return U4{c0, c1, c2, c3};
}

// The same generator when counter words 1-3 are fixed and only word 0 varies (one request and
// position, many vocabulary quads).  The parts of rounds 1 and 2 that do not depend on word 0
// are computed once by philox_fix; philox_var then costs 18 of the 20 multiplies.  Round 1 maps
// (c0, c1, c2, c3) to (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); its
// word 0 is fixed, so round 2's M0 product is fixed too.
struct PhiloxFixed {
  uint32_t x2;  // round 1: word 2 = hi(M0 c0) ^ x2
  uint32_t y0;  // round 2: word 0 = hi(M1 w2) ^ y0
  uint32_t y2;  // round 2: word 2 = lo(M0 c0) ^ y2
  uint32_t l2;  // round 2: word 3
};
__host__ __device__ __forceinline__ PhiloxFixed philox_fix(uint32_t c1, uint32_t c2, uint32_t c3,
                                                         uint32_t k0, uint32_t k1) {
  const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
  const uint32_t a0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;  // round 1, word 0
  const uint32_t a1 = (uint32_t)p1;                     // round 1, word 1
  const uint64_t p0 = (uint64_t)0xD2511F53u * a0;       // round 2's M0 product
  PhiloxFixed f;
  f.x2 = c3 ^ k1;
  f.y0 = a1 ^ (k0 + 0x9E3779B9u);
  f.y2 = (uint32_t)(p0 >> 32) ^ (k1 + 0xBB67AE85u);
  f.l2 = (uint32_t)p0;
  return f;
}
// The varying part, with the round keys given (rk0[i] = k0 + i * 0x9E3779B9, rk1[i] = k1 +
// i * 0xBB67AE85; e.g. from kernel parameters, so that no key arithmetic runs per call).
__host__ __device__ __forceinline__ U4 philox_var(uint32_t c0, const PhiloxFixed& f,
                                                     const uint32_t (&rk0)[10],
                                                     const uint32_t (&rk1)[10]) {
  const uint64_t p0 = (uint64_t)0xD2511F53u * c0;  // round 1
  const uint32_t w2 = (uint32_t)(p0 >> 32) ^ f.x2;
  const uint64_t p1 = (uint64_t)0xCD9E8D57u * w2;  // round 2
  uint32_t x0 = (uint32_t)(p1 >> 32) ^ f.y0, x1 = (uint32_t)p1;
  uint32_t x2 = (uint32_t)p0 ^ f.y2, x3 = f.l2;
#pragma unroll
  for (int round = 2; round < 10; ++round) {
    const uint64_t q0 = (uint64_t)0xD2511F53u * x0;
    const uint64_t q1 = (uint64_t)0xCD9E8D57u * x2;
    x0 = (uint32_t)(q1 >> 32) ^ x1 ^ rk0[round];
    x1 = (uint32_t)q1;
    x2 = (uint32_t)(q0 >> 32) ^ x3 ^ rk1[round];
    x3 = (uint32_t)q0;
  }
  return U4{x0, x1, x2, x3};
}

__device__ __forceinline__ uint32_t pick(const U4& q, int lane) {
  return lane == 0 ? q.x : lane == 1 ? q.y : lane == 2 ? q.z : q.w;
}

// u = (2 * (bits >> 9) + 1) * 2^-24: the odd multiples of 2^-24 inside (0, 1), exact in fp32.
__device__ __forceinline__ float bits_to_uniform(uint32_t bits) {
  return __uint2float_rn(((bits >> 9) << 1) | 1u) * 5.9604644775390625e-08f;
}

// Gumbel noise g = -ln(-ln u), with the accurate logf (u close to 1 needs it: -ln u ~ 6e-8).
__device__ __forceinline__ float gumbel_from_uniform(float u) { return -logf(-logf(u)); }

// ------------------------------------------------------------------ argmax keys
// key = (orderable fp32 score << 32) | (0xFFFFFFFF - v): the u64 maximum is the largest score,
// and among equal scores the smallest v.  Order-independent, so atomicMax is deterministic.
__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ unsigned long long make_key(float score, uint32_t v) {
  return ((unsigned long long)orderable(score) << 32) | (unsigned long long)(0xFFFFFFFFu - v);
}
__device__ __forceinline__ uint32_t key_token(unsigned long long key) {
  return 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
}
__device__ __forceinline__ float key_score(unsigned long long key) {
  const uint32_t o = (uint32_t)(key >> 32);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// Running state of one (request, vocab subset): Gumbel-max winner and online log-sum-exp.
struct RowState {
  float best;     // winning perturbed score
  uint32_t tok;   // its vocab id
  float m, l;     // running max of y and sum exp(y - m)
};
__device__ __forceinline__ void rs_init(RowState& s) {
  s.best = -INFINITY;
  s.tok = 0xFFFFFFFFu;
  s.m = -INFINITY;
  s.l = 0.f;
}
__device__ __forceinline__ void lse_push(float& m, float& l, float y) {
  if (y > m) {
    l = l * __expf(m - y) + 1.f;
    m = y;
  } else {
    l += __expf(y - m);
  }
}
__device__ __forceinline__ void lse_merge(float& m, float& l, float m2, float l2) {
  if (l2 == 0.f) return;
  if (l == 0.f) {
    m = m2;
    l = l2;
    return;
  }
  const float mm = fmaxf(m, m2);
  l = l * __expf(m - mm) + l2 * __expf(m2 - mm);
  m = mm;
}
__device__ __forceinline__ void best_merge(float& best, uint32_t& tok, float b2, uint32_t t2) {
  if (b2 > best || (b2 == best && t2 < tok)) {
    best = b2;
    tok = t2;
  }
}

// ------------------------------------------------------------------ loads
template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

// 16 bytes -> VEC floats (VEC = 4 for fp32, 8 for bf16)
template <typename T>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& q, float* f) {
    f[0] = __uint_as_float(q.x);
    f[1] = __uint_as_float(q.y);
    f[2] = __uint_as_float(q.z);
    f[3] = __uint_as_float(q.w);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4& q, float* f) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

// ------------------------------------------------------------------ timers, fences, barriers
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid-wide barrier of a co-resident (cooperative) grid, split in two so a block can do
// independent work between arriving and waiting.  Barrier number `n` (1-based within the
// launch) completes when every block has arrived n times.  grid_arrive: every thread calls it
// (it starts with __syncthreads); thread 0 publishes the block's writes and arrives.
// grid_wait: every thread calls it; thread 0 spins with a time bound; returns false (and records
// DSPARK_ERR_TIMEOUT) if the bound ran out.
__device__ __forceinline__ void grid_arrive(WsHeader* hdr) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    red_release_add(&hdr->arrive, 1u);
  }
}
__device__ __forceinline__ bool grid_wait(WsHeader* hdr, unsigned n, int* s_flag) {
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned target = n * gridDim.x;
    if (ld_acquire(&hdr->arrive) < target) {
      const unsigned long long t0 = globaltimer();
      while (ld_acquire(&hdr->arrive) < target) {
        if (globaltimer() - t0 > kWaitLimitNs) {
          atomicMax(&hdr->status, kErrTimeout);
          ok = 0;
          break;
        }
        __nanosleep(20);
      }
    }
    __threadfence();
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}
__device__ __forceinline__ bool grid_barrier(WsHeader* hdr, unsigned n, int* s_flag) {
  grid_arrive(hdr);
  return grid_wait(hdr, n, s_flag);
}

// L2 prefetch of `bytes` (multiple of 16) starting at a 16-byte aligned global address.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ mbarrier + bulk copies
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait with a suspend-time hint: the thread may sleep up to hint_ns inside the instruction
// until the phase completes, instead of spinning on the issue slots other warps need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Bounded wait of one lane, sleeping between polls, with the verdict given to the whole warp.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0 && !mbar_try_wait(bar, parity)) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) {
      if (globaltimer() - t0 > kWaitLimitNs) {
        ok = false;
        break;
      }
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0);
}
// The same with the time bound given (the draft kernels' failure-path test hook).
__device__ __forceinline__ bool mbar_wait_warp_lim(uint64_t* bar, uint32_t parity,
                                                   unsigned long long limit_ns) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0 && !mbar_try_wait(bar, parity)) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait_sleep(bar, parity, 1000)) {
      if (globaltimer() - t0 > limit_ns) {
        ok = false;
        break;
      }
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0);
}
// Bounded wait for the phase with the given parity; false when the time bound ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) {
    if (globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// ------------------------------------------------------------------ thread-block clusters
// (distributed shared memory: a block addresses a peer's shared memory through mapa)
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the variable at `p` (this block's shared memory) in block `rank`
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f2(uint32_t addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y)
               : "memory");
}
// store with release semantics at cluster scope: this thread's earlier writes (local or remote)
// are visible to any thread of the cluster that reads the value with acquire semantics
__device__ __forceinline__ void st_release_cluster_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.release.cluster.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_cluster_u64(const void* p) {
  unsigned long long v;
  asm volatile("ld.acquire.cluster.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
// Every thread of every block of the cluster: release what this thread wrote, wait for all
// (hardware cluster barrier; each thread reaches it after bounded waits only)
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// L2 policy: stream once (weights re-read next step may still hit L2, but do not displace
// the data that is read twice within a step).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction count on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float sigmoidf_acc(float x) { return 1.f / (1.f + expf(-x)); }

}  // namespace dspark
