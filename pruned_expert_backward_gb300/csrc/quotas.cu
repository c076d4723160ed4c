// Per-expert loads and backward retention quotas.
//
// "LRMoE: Trimming Backward Work in Memory-Bound MoE Training", section "Backward demand is
// not a constant": before the expert forward the controller observes each expert's routed
// demand and fixes a retention quota that holds for the whole layer call.  The controller's
// memory/network model is outside this library; the quota follows one fixed rule.
#include "common.cuh"
#include "kernels.h"

namespace lrm {

namespace {

__global__ void __launch_bounds__(256) load_hist_kernel(const int32_t* __restrict__ idx, int64_t P, int E,
                                                        int32_t* __restrict__ loads, int32_t* status) {
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < P; u += (int64_t)gridDim.x * blockDim.x) {
    const int e = idx[u];
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else
      set_status(status, LRM_ERR_BAD_INDEX);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (hist[e]) atomicAdd(&loads[e], hist[e]);
}

__global__ void quota_rule_kernel(const int32_t* __restrict__ loads, int E, int kind, int32_t num, int32_t den,
                                  int32_t cap, const int32_t* __restrict__ explicit_q, int32_t* __restrict__ quotas) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) quotas[e] = quota_rule(loads[e], kind, num, den, cap, explicit_q, e);
}

}  // namespace

void launch_plan_quotas(const int32_t* topk_idx, int64_t P, int32_t E, int kind, int32_t num, int32_t den,
                        int32_t cap, const int32_t* explicit_q, int32_t* loads, int32_t* quotas, int32_t* status,
                        cudaStream_t s) {
  cudaMemsetAsync(loads, 0, sizeof(int32_t) * E, s);
  if (P > 0) {
    int64_t blocks = (P + 255) / 256;
    if (blocks > 152 * 4) blocks = 152 * 4;
    load_hist_kernel<<<(unsigned)blocks, 256, E * sizeof(int), s>>>(topk_idx, P, E, loads, status);
  }
  quota_rule_kernel<<<1, 1024, 0, s>>>(loads, E, kind, num, den, cap, explicit_q, quotas);
}

}  // namespace lrm
