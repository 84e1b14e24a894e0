// gemm_tc.cu -- split-K tensor-core GEMM for the RNN head's parallel pre-pass.
//
// Eq 6 ("DSpark -- paper verification", section 1) projects z_k = [s_{k-1}; W1[x_{k-1}]; h_k]
// with one joint matrix Wj = [W_g; W_c; W_o].  The h_k columns do not depend on the sampled
// tokens, so their product G_h = h Wj[:, 2r:]^T is computed for every (request, position) at
// once before the sequential loop: a plain dense GEMM of [B*gamma x d] by [d x 3r].
//
//   part[ks][m][n] = sum over k in split ks of A[m][k] * Bm[n][k]     (fp32 partials)
//
// A and Bm are bf16, K-major (row stride lda / ldb elements), loaded by 2-D TMA into the
// 128-byte-swizzled layout; one thread issues kind::f16 MMAs (M = 128, N = 256) into TMEM;
// four warps read TMEM and store the fp32 partial tile.  The consumer adds the splits in a fixed
// order, so the result does not depend on scheduling.
#include <cuda.h>

#include "draft.cuh"
#include "tc.cuh"

namespace dspark {
namespace {

constexpr int kGM = 128, kGN = 256;
constexpr int kGA = kGM * 128;         // A slab bytes (128 rows x 64 bf16)
constexpr int kGB = kGN * 128;         // B slab bytes (256 rows x 64 bf16)
constexpr int kGStage = kGA + kGB;     // 48 KB
constexpr int kGStages = 4;
constexpr int kGThreads = 256;

struct GemmArgs {
  int M, N, nslab, per_split;
  float* part;       // [ksplit][M][N]
  unsigned* status;  // workspace status word (a timed-out wait records DSPARK_ERR_TIMEOUT)
};

__global__ void __launch_bounds__(kGThreads, 1)
    gemm_tc_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(smem + kGStages * kGStage);
  uint64_t* empty = full + kGStages;
  uint64_t* done = empty + kGStages;
  uint32_t* tbase = (uint32_t*)(done + 1);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m0 = blockIdx.x * kGM, n0 = blockIdx.y * kGN;
  const int s0 = blockIdx.z * a.per_split, s1 = min(a.nslab, s0 + a.per_split);
  const int ns = max(0, s1 - s0);

  if (tid == 0) {
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tbase, kGN);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tbase;

  if (warp == 0 && lane == 0) {
    const uint64_t pol = policy_evict_first();
    for (int i = 0; i < ns; ++i) {
      const int slot = i % kGStages;
      if (i >= kGStages && !mbar_wait(&empty[slot], (uint32_t)(((i / kGStages) - 1) & 1))) {
        atomicMax(a.status, kErrTimeout);
        break;
      }
      uint8_t* st = smem + slot * kGStage;
      mbar_expect_tx(&full[slot], kGStage);
      tc::tma_load_2d(st, &tmA, (s0 + i) * 64, m0, &full[slot], pol);
      tc::tma_load_2d(st + kGA, &tmB, (s0 + i) * 64, n0, &full[slot], pol);
    }
    for (int i = max(0, ns - kGStages); i < ns; ++i)  // every copy lands before exit
      mbar_wait(&full[i % kGStages], (uint32_t)((i / kGStages) & 1));
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(kGM, kGN);
      for (int i = 0; i < ns; ++i) {
        const int slot = i % kGStages;
        if (!mbar_wait(&full[slot], (uint32_t)((i / kGStages) & 1))) {
          atomicMax(a.status, kErrTimeout);
          break;
        }
        tc::fence_after_sync();
        const uint32_t sa = smem_u32(smem + slot * kGStage), sb = sa + kGA;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tmem, tc::sdesc_sw128(sa + kk * 32), tc::sdesc_sw128(sb + kk * 32), idesc,
                       (i | kk) != 0);
        tc::mma_commit(&empty[slot]);
      }
      tc::mma_commit(done);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int q = warp & 3, m = m0 + 32 * q + lane;
    const bool ok = mbar_wait(done, 0);
    if (!ok && lane == 0) atomicMax(a.status, kErrTimeout);
    tc::fence_after_sync();
    float* out = a.part + ((size_t)blockIdx.z * a.M + m) * a.N;
    for (int g = 0; g < kGN / 32; ++g) {
      uint32_t v[32];
      tc::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + g * 32, v);
      tc::tmem_ld_wait();
      if (m >= a.M) continue;
      const int n = n0 + g * 32;
      const bool live = ok && ns > 0;
      if (n + 32 <= a.N && (a.N & 3) == 0) {  // 16-byte stores of this row's 32 columns
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *(float4*)(out + n + j) =
              live ? make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                 __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        for (int j = 0; j < 32; ++j)
          if (n + j < a.N) out[n + j] = live ? __uint_as_float(v[j]) : 0.f;
      }
    }
    tc::fence_before_sync();
  }
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kGN);
  }
}

}  // namespace

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against the driver
// library), looked up once.
static EncodeTiled tmap_encoder() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiled)f;
  }
  return fn;
}

bool encode_bf16_2d(CUtensorMap* m, const void* base, int rows, int cols, int ld, int box_rows) {
  EncodeTiled enc = tmap_encoder();
  if (!enc) return false;
  const cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_u_bf16_3d(CUtensorMap* m, const void* U, int B, int G, int V, int box_rows) {
  EncodeTiled enc = tmap_encoder();
  if (!enc) return false;
  const cuuint64_t gdim[3] = {(cuuint64_t)V, (cuuint64_t)G, (cuuint64_t)B};
  const cuuint64_t gstride[2] = {(cuuint64_t)V * 2, (cuuint64_t)G * V * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(U), gdim, gstride, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t gemm_tc_smem_bytes() { return (size_t)kGStages * kGStage + 1024 + 256; }

// part[ks][M][N] = A[M][K] Bm[N][K]^T over split ks; A row stride lda, Bm row stride ldb
// (elements, multiples of 8; base pointers 16-byte aligned).  Returns the number of K splits
// written through *ksplit_out (the consumer sums that many partial planes).
cudaError_t launch_gemm_tc(const void* A, int lda, const void* Bm, int ldb, int M, int N, int K,
                           float* part, int max_split, int nsm, int* ksplit_out, unsigned* status,
                           cudaStream_t stream) {
  CUtensorMap ta, tb;
  if (!encode_bf16_2d(&ta, A, M, K, lda, kGM) || !encode_bf16_2d(&tb, Bm, N, K, ldb, kGN))
    return cudaErrorInvalidValue;
  const int nslab = (K + 63) / 64;
  const int tiles = ((M + kGM - 1) / kGM) * ((N + kGN - 1) / kGN);
  int ks = (nsm + tiles - 1) / tiles;  // fill the machine with K splits
  ks = ks < 1 ? 1 : ks > max_split ? max_split : ks;
  ks = ks > nslab ? nslab : ks;
  const int per = (nslab + ks - 1) / ks;
  ks = (nslab + per - 1) / per;
  GemmArgs ga{M, N, nslab, per, part, status};
  const size_t smem = gemm_tc_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((M + kGM - 1) / kGM, (N + kGN - 1) / kGN, ks);
  gemm_tc_kernel<<<grid, kGThreads, smem, stream>>>(ga, ta, tb);
  *ksplit_out = ks;
  return cudaGetLastError();
}

}  // namespace dspark
