// kernels.h -- host launchers of the libdspark kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dspark {

// dst[c][r] = src[r][c] for a rows x cols matrix of 2- or 4-byte elements (es), both row-major.
cudaError_t launch_transpose(const void* src, void* dst, int rows, int cols, int es, cudaStream_t stream);
cudaError_t launch_confidence(int B, int G, int V, int r, int d, int w_bf16, const void* W1,
                              const void* w, int u_bf16, const void* h, const int32_t* x0,
                              const int32_t* tokens, float* c, float* S, cudaStream_t stream);
cudaError_t launch_tv_label(int N, int V, float T, const float* d, const float* t, float* cstar,
                            float* l1, cudaStream_t stream);
size_t verify_workspace_bytes(int B, int G, int V);
cudaError_t launch_verify(int B, int G, int V, float T, uint64_t seed, const float* zd,
                          const float* zt, const int32_t* tok, int32_t* n_acc, int32_t* out,
                          void* workspace, cudaStream_t stream);
size_t loss_workspace_bytes(int B, int G, int V);
cudaError_t launch_loss(int B, int G, int V, float T, const float* zd, const float* zt,
                        const int32_t* lab, const float* conf, float a_ce, float a_tv, float a_conf,
                        float* loss, float* parts, float* grad_z, float* grad_c, void* workspace,
                        cudaStream_t stream);
size_t sts_workspace_bytes(int N, int G, int ng, int bins);
cudaError_t launch_sts(int N, int G, const float* conf, const int32_t* acc, int ng, const float* grid,
                       int bins, float* tau, float* ece, float* ece_grid, void* workspace,
                       cudaStream_t stream);
cudaError_t launch_prefix_schedule(int B, int G, const float* S, const double* sps, int32_t* len,
                                   double* theta, cudaStream_t stream);

}  // namespace dspark
