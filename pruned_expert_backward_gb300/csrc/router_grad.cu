// Routing-weight gradient of the retained pairs.
//
// The layer output is out_t = sum_j alpha_{t,j} y_{t,j} with y = W_down[e] phi, so the loss
// gradient with respect to a routing weight is g_t . y_{t,j}.  The retained rows already pass
// through dphi = (alpha_u g_t) W_down[e] in the grouped backward, and
//   dphi . phi_u = alpha_u * (g_t . W_down[e] phi_u) = alpha_u * (g_t . y_u),
// so the var-M epilogue that applies the SwiGLU backward also forms dphi . phi (with phi
// recomputed from the gate and up rows it already holds) in parts of 64 or 128 columns.
// row_dot sums the parts of a row in index order (deterministic); router_grad divides by
// alpha_u and returns the result to pair order.  A dropped pair has no row and gets 0 ("LRMoE:
// Trimming Backward Work in Memory-Bound MoE Training", section "The part that is easy to get
// wrong": only the retained rows are packed and computed).
#include "common.cuh"
#include "kernels.h"

namespace lrm {

namespace {

__global__ void __launch_bounds__(256) row_dot_kernel(const float* __restrict__ part, int n_part,
                                                      const int32_t* __restrict__ seg, int E, int64_t cap,
                                                      float* __restrict__ row_dot) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t rows = __ldg(seg + E);
  if (rows > cap) rows = cap;
  if (r >= rows) return;
  const float* pr = part + r * n_part;
  float acc = 0.f;
  for (int i = 0; i < n_part; ++i) acc += pr[i];
  row_dot[r] = acc;
}

__global__ void __launch_bounds__(256) router_grad_kernel(const int32_t* __restrict__ row_of_pair,
                                                          const float* __restrict__ alpha,
                                                          const float* __restrict__ row_dot, int64_t P, int64_t cap,
                                                          float* __restrict__ dalpha) {
  const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= P) return;
  const int32_t r = row_of_pair[u];
  float d = 0.f;
  if (r >= 0 && (int64_t)r < cap) {
    const float a = alpha[u];
    if (a != 0.f) d = row_dot[r] / a;
  }
  dalpha[u] = d;
}

}  // namespace

void launch_row_dot(const float* part, int n_part, const int32_t* seg_offsets, int32_t E, int64_t cap,
                    float* row_dot, cudaStream_t s) {
  if (cap <= 0) return;
  row_dot_kernel<<<(unsigned)((cap + 255) / 256), 256, 0, s>>>(part, n_part, seg_offsets, E, cap, row_dot);
}

void launch_router_grad(const int32_t* row_of_pair, const float* alpha, const float* row_dot, int64_t P,
                        int64_t cap, float* dalpha, cudaStream_t s) {
  if (P <= 0) return;
  router_grad_kernel<<<(unsigned)((P + 255) / 256), 256, 0, s>>>(row_of_pair, alpha, row_dot, P, cap, dalpha);
}

}  // namespace lrm
