// noalloc.cu -- the Markov draft for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory at the point where they draft: code that
// runs inside another framework's memory pool or a serving engine that forbids allocation on
// its decode path, plugins handed only pre-allocated input and output buffers, and processes
// whose allocator must not be touched while requests are in flight.  For them this file keeps
// the draft's scratch (the status word, per-block argmax slots and normaliser partials) in one
// file-scope device array that exists for as long as the library is loaded on a GPU, and calls
// the ordinary Markov draft with that array as its workspace.  Nothing here allocates: the
// array's device address is looked up once per device, and each call only clears and copies.
#include <cstdio>
#include <mutex>

#include "dspark.h"
#include "draft.cuh"

namespace dspark {
void set_last_error(const char* msg);  // defined in api.cu
}

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)1 << 20;  // 1 MiB on every GPU that loads us

// The scratch itself.  Shared by every call on a device; holds the previous call's contents.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64];  // device address of the array, per device ordinal

// Device address of the array on the current device.  The host-side symbol is only a stand-in:
// the address the kernels need comes from cudaGetSymbolAddress, asked once per device with that
// device current.
dspark_status scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    dspark::set_last_error("dspark_markov_draft_noalloc: no usable current device");
    return DSPARK_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      char buf[256];
      snprintf(buf, sizeof buf, "dspark_markov_draft_noalloc: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(e));
      dspark::set_last_error(buf);
      return DSPARK_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return DSPARK_OK;
}

}  // namespace

extern "C" dspark_status dspark_markov_draft_noalloc(
    int B, int gamma, int V, int r, int d, float T, uint64_t seed, dspark_dtype wdt,
    const void* W1, const void* W2, const void* w, dspark_dtype udt, const void* U, const void* h,
    const int32_t* x0, const int32_t* forced, const float* target, int32_t* tokens, float* lse,
    float* c, float* S, float* cstar, float* l1, float* logits, int32_t* status, void* stream) {
  const size_t need = dspark_workspace_bytes(0, B, gamma, V, r, d, target ? DSPARK_WS_TARGET : 0);
  if (need > kNoAllocScratchBytes) {
    char buf[256];
    snprintf(buf, sizeof buf,
             "dspark_markov_draft_noalloc: this problem needs %zu bytes of scratch, the built-in "
             "array holds %zu; use dspark_markov_draft with a workspace",
             need, kNoAllocScratchBytes);
    dspark::set_last_error(buf);
    return DSPARK_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  dspark_status st = scratch_on_current_device(&ws);
  if (st != DSPARK_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  // The draft expects its status word and argmax slots to start at zero, and the array still
  // holds whatever the previous call (possibly a failed one) left: clear the part this call uses.
  if (need > 0) {
    const cudaError_t e = cudaMemsetAsync(ws, 0, need, s);
    if (e != cudaSuccess) {
      dspark::set_last_error("dspark_markov_draft_noalloc: clearing the scratch failed");
      return DSPARK_ERR_CUDA;
    }
  }
  st = dspark_markov_draft(B, gamma, V, r, d, T, seed, wdt, W1, W2, DSPARK_W2_VR, w, udt, U, h, x0, forced,
                           target, tokens, lse, c, S, cstar, l1, logits, ws, kNoAllocScratchBytes,
                           stream);
  if (st != DSPARK_OK) return st;
  if (status) {  // the device status of this call, for a caller that cannot read the array
    const cudaError_t e =
        cudaMemcpyAsync(status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) {
      dspark::set_last_error("dspark_markov_draft_noalloc: copying the status failed");
      return DSPARK_ERR_CUDA;
    }
  }
  return DSPARK_OK;
}
