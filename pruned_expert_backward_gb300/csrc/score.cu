// LRM score of every token-expert pair.
//
// "LRMoE: Trimming Backward Work in Memory-Bound MoE Training", section "LRM: a decomposable
// contribution score": pair u = (t, e) adds the rank-one term G_u = (alpha_u g_t) phi_u^T to
// the down projection's weight gradient, so ||G_u||_F^2 = alpha_u^2 * ||g_t||^2 * ||phi_u||^2
// and no gradient matrix has to be formed.
//
// One group of k warps per token, several tokens per CTA (up to 1024 threads).  The token's
// g_t row is split over its k warps (each row of g is read once), warp j reduces phi_u for
// u = t*k + j; the k phi rows of consecutive tokens are contiguous, so a CTA streams one
// contiguous span of memory.  All loads are 16-byte, coalesced, not allocated in L1 (nothing
// here is re-read).  HBM-bound.
#include "common.cuh"
#include "kernels.h"

namespace lrm {

template <typename T>
__global__ void __launch_bounds__(1024) score_kernel(const float* __restrict__ alpha, const T* __restrict__ g,
                                                    const T* __restrict__ phi, int64_t n_tok, int k, int H, int I,
                                                    float* __restrict__ scores, int32_t* status) {
  constexpr int VN = VecTraits<T>::N;
  __shared__ float g_part[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tok_per_blk = blockDim.x / (32 * k);
  const int tok_in_blk = warp / k, j = warp - tok_in_blk * k;
  const int64_t t = (int64_t)blockIdx.x * tok_per_blk + tok_in_blk;
  const int nvg = H / VN, nvp = I / VN;

  float gs = 0.f, ps = 0.f;
  if (t < n_tok) {
    const T* gt = g + t * H;
    for (int v = j * 32 + lane; v < nvg; v += 32 * k) {
      float f[VN];
      unpack(ld_stream16(gt + (int64_t)v * VN), f);
#pragma unroll
      for (int q = 0; q < VN; ++q) gs = fmaf(f[q], f[q], gs);
    }
    const T* pu = phi + (t * k + j) * (int64_t)I;
#pragma unroll 4
    for (int v = lane; v < nvp; v += 32) {
      float f[VN];
      unpack(ld_stream16(pu + (int64_t)v * VN), f);
#pragma unroll
      for (int q = 0; q < VN; ++q) ps = fmaf(f[q], f[q], ps);
    }
  }
  gs = warp_sum(gs);
  ps = warp_sum(ps);
  if (lane == 0) g_part[warp] = gs;
  __syncthreads();
  if (t < n_tok && lane == 0) {
    float gn = 0.f;
    for (int w = 0; w < k; ++w) gn += g_part[tok_in_blk * k + w];
    const int64_t u = t * k + j;
    const float a = alpha[u];
    const float r = (a * a) * gn * ps;
    scores[u] = r;
    if (!isfinite(r)) set_status(status, LRM_ERR_NONFINITE);
  }
}

void launch_score(const float* alpha, const void* g, const void* phi, int64_t T, int32_t k, int32_t H, int32_t I,
                  lrm_dtype dt, float* scores, int32_t* status, cudaStream_t s) {
  if (T == 0) return;
  const int tok_per_blk = k >= 32 ? 1 : 32 / k;  // up to 32 warps: several tokens per CTA
  const int threads = 32 * k * tok_per_blk;
  const int64_t blocks = (T + tok_per_blk - 1) / tok_per_blk;
  if (dt == LRM_BF16)
    score_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, s>>>(
        alpha, (const __nv_bfloat16*)g, (const __nv_bfloat16*)phi, T, k, H, I, scores, status);
  else
    score_kernel<float><<<(unsigned)blocks, threads, 0, s>>>(alpha, (const float*)g, (const float*)phi, T, k, H, I,
                                                             scores, status);
}

}  // namespace lrm
