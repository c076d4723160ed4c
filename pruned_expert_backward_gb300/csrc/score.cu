// LRM score of every token-expert pair.
//
// "LRMoE: Trimming Backward Work in Memory-Bound MoE Training", section "LRM: a decomposable
// contribution score": pair u = (t, e) adds the rank-one term G_u = (alpha_u g_t) phi_u^T to
// the down projection's weight gradient, so ||G_u||_F^2 = alpha_u^2 * ||g_t||^2 * ||phi_u||^2
// and no gradient matrix has to be formed.
//
// One warp per pair row; the k warps of a token each reduce g_t (one DRAM read, the rest L2
// hits) and their own phi_u row.  All loads are 16-byte and coalesced; phi is streamed past L1.
// No block-wide barrier, so warps retire as soon as their loads return.  HBM-bound.
#include "common.cuh"
#include "kernels.h"

namespace lrm {

template <typename T>
__global__ void __launch_bounds__(256) score_kernel(const float* __restrict__ alpha, const T* __restrict__ g,
                                                   const T* __restrict__ phi, int64_t n_pairs, int k, int H, int I,
                                                   float* __restrict__ scores, int32_t* status) {
  // One warp per pair row u = (t, j): it reduces phi_u and, on its own, the token's g_t row (the
  // token's other k-1 warps read g_t too, from L2).  No block-wide barrier: a warp issues all its
  // loads, reduces, writes its score and retires.
  constexpr int VN = VecTraits<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (u >= n_pairs) return;
  const int64_t t = u / k;
  const float a = alpha[u];
  const T* gt = g + t * H;
  const T* pu = phi + u * (int64_t)I;
  const int nvg = H / VN, nvp = I / VN;
  float gs = 0.f, ps = 0.f;
#pragma unroll 4
  for (int v = lane; v < nvp; v += 32) {
    float f[VN];
    unpack(ld_stream16(pu + (int64_t)v * VN), f);
#pragma unroll
    for (int q = 0; q < VN; ++q) ps = fmaf(f[q], f[q], ps);
  }
#pragma unroll 8
  for (int v = lane; v < nvg; v += 32) {
    float f[VN];
    unpack(ldg16(gt + (int64_t)v * VN), f);
#pragma unroll
    for (int q = 0; q < VN; ++q) gs = fmaf(f[q], f[q], gs);
  }
  gs = warp_sum(gs);
  ps = warp_sum(ps);
  if (lane == 0) {
    const float r = (a * a) * gs * ps;
    scores[u] = r;
    if (!isfinite(r)) set_status(status, LRM_ERR_NONFINITE);
  }
}

void launch_score(const float* alpha, const void* g, const void* phi, int64_t T, int32_t k, int32_t H, int32_t I,
                  lrm_dtype dt, float* scores, int32_t* status, cudaStream_t s) {
  if (T == 0) return;
  const int64_t P = T * k;
  const int64_t blocks = (P + 7) / 8;  // 8 warps (pair rows) per CTA
  if (dt == LRM_BF16)
    score_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
        alpha, (const __nv_bfloat16*)g, (const __nv_bfloat16*)phi, P, k, H, I, scores, status);
  else
    score_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(alpha, (const float*)g, (const float*)phi, P, k, H, I,
                                                         scores, status);
}

}  // namespace lrm
