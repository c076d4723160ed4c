// LRM score of every token-expert pair.
//
// "LRMoE: Trimming Backward Work in Memory-Bound MoE Training", section "LRM: a decomposable
// contribution score": pair u = (t, e) adds the rank-one term G_u = (alpha_u g_t) phi_u^T to
// the down projection's weight gradient, so ||G_u||_F^2 = alpha_u^2 * ||g_t||^2 * ||phi_u||^2
// and no gradient matrix has to be formed.
//
// One warp per token: g_t is read once, then the token's k phi rows (contiguous) two rows at a
// time.  All loads are 16-byte, coalesced and streamed past L1; no block-wide barrier, so warps
// retire as soon as their loads return.  HBM-bound.
#include "common.cuh"
#include "kernels.h"

namespace lrm {

// Per-lane partial sum of squares (ABS: of magnitudes) of one row of nv 16-byte vectors
// (v = lane, lane+32, ...): all of the lane's loads are issued before any is used (at most MAXV).
template <typename T, int MAXV, bool ABS = false>
__device__ __forceinline__ float lane_sumsq(const T* row, int nv, int lane) {
  constexpr int VN = VecTraits<T>::N;
  uint4 buf[MAXV];
#pragma unroll
  for (int m = 0; m < MAXV; ++m) {
    const int v = lane + 32 * m;
    buf[m] = v < nv ? ld_stream16(row + (int64_t)v * VN) : make_uint4(0, 0, 0, 0);
  }
  float acc = 0.f;
#pragma unroll
  for (int m = 0; m < MAXV; ++m) {
    float f[VN];
    unpack(buf[m], f);
#pragma unroll
    for (int q = 0; q < VN; ++q) acc = ABS ? acc + fabsf(f[q]) : fmaf(f[q], f[q], acc);
  }
  return acc;
}
// Same, for rows of any length (a loop; used when a row exceeds MAXV vectors per lane).
template <typename T, bool ABS = false>
__device__ __forceinline__ float lane_sumsq_any(const T* row, int nv, int lane) {
  constexpr int VN = VecTraits<T>::N;
  float acc = 0.f;
  for (int v = lane; v < nv; v += 32) {
    float f[VN];
    unpack(ld_stream16(row + (int64_t)v * VN), f);
#pragma unroll
    for (int q = 0; q < VN; ++q) acc = ABS ? acc + fabsf(f[q]) : fmaf(f[q], f[q], acc);
  }
  return acc;
}

template <typename T, int GV, int PV>
__global__ void __launch_bounds__(256) score_kernel(const float* __restrict__ alpha, const T* __restrict__ g,
                                                   const T* __restrict__ phi, int64_t n_tok, int k, int H, int I,
                                                   float* __restrict__ scores, int32_t* status) {
  // One warp per token: ||g_t||^2 once, then the token's k contiguous phi rows two at a time.
  // GV / PV bound the 16-byte vectors per lane of a g row / phi row (0 = unbounded, looped).
  chain_wait();
  constexpr int VN = VecTraits<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= n_tok) return;
  const int nvg = H / VN, nvp = I / VN;
  const T* pt = phi + t * k * (int64_t)I;
  const float my_alpha = lane < k ? alpha[t * k + lane] : 0.f;
  float gs = GV ? lane_sumsq<T, (GV ? GV : 1)>(g + t * H, nvg, lane) : lane_sumsq_any<T>(g + t * H, nvg, lane);
  gs = warp_sum(gs);
  for (int j = 0; j < k; j += 2) {
    const bool two = j + 1 < k;
    const T* r0 = pt + (int64_t)j * I;
    float p0, p1 = 0.f;
    if (PV) {
      p0 = lane_sumsq<T, (PV ? PV : 1)>(r0, nvp, lane);
      if (two) p1 = lane_sumsq<T, (PV ? PV : 1)>(r0 + I, nvp, lane);
    } else {
      p0 = lane_sumsq_any<T>(r0, nvp, lane);
      if (two) p1 = lane_sumsq_any<T>(r0 + I, nvp, lane);
    }
    p0 = warp_sum(p0);
    p1 = warp_sum(p1);
    const float a0 = __shfl_sync(0xffffffffu, my_alpha, j);
    const float a1 = __shfl_sync(0xffffffffu, my_alpha, two ? j + 1 : j);
    if (lane == 0) {
      const float s0 = (a0 * a0) * gs * p0;
      scores[t * k + j] = s0;
      if (!isfinite(s0)) set_status(status, LRM_ERR_NONFINITE);
      if (two) {
        const float s1 = (a1 * a1) * gs * p1;
        scores[t * k + j + 1] = s1;
        if (!isfinite(s1)) set_status(status, LRM_ERR_NONFINITE);
      }
    }
  }
}

// One round trip per token: a lane issues all of its g and phi loads (GV + MAXK * PV 16-byte
// vectors) before it uses any, so a warp waits for memory once instead of once per row group.
// Used when that fits in registers (the 8k-token Qwen3 shape: 8 + 8 * 3 vectors per lane).
template <typename T, int GV, int PV, int MAXK>
__global__ void __launch_bounds__(128) score_onepass_kernel(const float* __restrict__ alpha, const T* __restrict__ g,
                                                           const T* __restrict__ phi, int64_t n_tok, int k, int H,
                                                           int I, float* __restrict__ scores, int32_t* status) {
  chain_wait();
  constexpr int VN = VecTraits<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= n_tok) return;
  const int nvg = H / VN, nvp = I / VN;
  const T* gt = g + t * H;
  const T* pt = phi + t * k * (int64_t)I;
  const float my_alpha = lane < k ? alpha[t * k + lane] : 0.f;
  uint4 gb[GV], pb[MAXK][PV];
#pragma unroll
  for (int m = 0; m < GV; ++m) {
    const int v = lane + 32 * m;
    gb[m] = v < nvg ? ld_stream16(gt + (int64_t)v * VN) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int j = 0; j < MAXK; ++j)
#pragma unroll
    for (int m = 0; m < PV; ++m) {
      const int v = lane + 32 * m;
      pb[j][m] = (j < k && v < nvp) ? ld_stream16(pt + (int64_t)j * I + (int64_t)v * VN) : make_uint4(0, 0, 0, 0);
    }
  float gs = 0.f;
#pragma unroll
  for (int m = 0; m < GV; ++m) {
    float f[VN];
    unpack(gb[m], f);
#pragma unroll
    for (int q = 0; q < VN; ++q) gs = fmaf(f[q], f[q], gs);
  }
  gs = warp_sum(gs);
  float mine = 0.f;  // lane j ends up with row j's ||phi||^2
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    if (j >= k) break;
    float ps = 0.f;
#pragma unroll
    for (int m = 0; m < PV; ++m) {
      float f[VN];
      unpack(pb[j][m], f);
#pragma unroll
      for (int q = 0; q < VN; ++q) ps = fmaf(f[q], f[q], ps);
    }
    ps = warp_sum(ps);
    if (lane == j) mine = ps;
  }
  if (lane < k) {
    const float sc = (my_alpha * my_alpha) * gs * mine;
    scores[t * k + lane] = sc;
    if (!isfinite(sc)) set_status(status, LRM_ERR_NONFINITE);
  }
}

// The same score with ||phi_u||^2 handed in (from a forward that emits it, see forward.cu): one
// warp per token reads g_t once and writes its k scores; phi itself is not read.
template <typename T, int GV>
__global__ void __launch_bounds__(256) score_norms_kernel(const float* __restrict__ alpha, const T* __restrict__ g,
                                                         const float* __restrict__ phi_sq, int64_t n_tok, int k,
                                                         int H, float* __restrict__ scores, int32_t* status) {
  constexpr int VN = VecTraits<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= n_tok) return;
  float a = 0.f, p = 0.f;
  if (lane < k) {  // issued before the g loads complete
    a = alpha[t * k + lane];
    p = phi_sq[t * k + lane];
  }
  float gs = GV ? lane_sumsq<T, (GV ? GV : 1)>(g + t * H, H / VN, lane) : lane_sumsq_any<T>(g + t * H, H / VN, lane);
  gs = warp_sum(gs);
  if (lane < k) {
    const float sc = (a * a) * gs * p;
    scores[t * k + lane] = sc;
    if (!isfinite(sc)) set_status(status, LRM_ERR_NONFINITE);
  }
}

void launch_score_norms(const float* alpha, const void* g, const float* phi_sq, int64_t T, int32_t k, int32_t H,
                        lrm_dtype dt, float* scores, int32_t* status, cudaStream_t s) {
  if (T == 0) return;
  const unsigned blocks = (unsigned)((T + 7) / 8);
  const int gv = (H / (dt == LRM_BF16 ? 8 : 4) + 31) / 32;
  using B = __nv_bfloat16;
  if (dt == LRM_BF16) {
    if (gv <= 16) score_norms_kernel<B, 16><<<blocks, 256, 0, s>>>(alpha, (const B*)g, phi_sq, T, k, H, scores, status);
    else score_norms_kernel<B, 0><<<blocks, 256, 0, s>>>(alpha, (const B*)g, phi_sq, T, k, H, scores, status);
  } else {
    if (gv <= 16)
      score_norms_kernel<float, 16><<<blocks, 256, 0, s>>>(alpha, (const float*)g, phi_sq, T, k, H, scores, status);
    else
      score_norms_kernel<float, 0><<<blocks, 256, 0, s>>>(alpha, (const float*)g, phi_sq, T, k, H, scores, status);
  }
}

// Gradient-only ablation scores ("LRMoE: Trimming Backward Work in Memory-Bound MoE Training",
// section "What the measurements show": squared gradient norm and absolute gradient magnitude):
// one warp per token computes ||g_t||_2^2 (ABS = false) or ||g_t||_1 (ABS = true) and writes it
// to the token's k pairs.
template <typename T, bool ABS, int GV>
__global__ void __launch_bounds__(256) grad_score_kernel(const T* __restrict__ g, int64_t n_tok, int k, int H,
                                                         float* __restrict__ scores, int32_t* status) {
  constexpr int VN = VecTraits<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= n_tok) return;
  const T* gt = g + t * H;
  float acc = GV ? lane_sumsq<T, (GV ? GV : 1), ABS>(gt, H / VN, lane) : lane_sumsq_any<T, ABS>(gt, H / VN, lane);
  acc = warp_sum(acc);
  if (lane < k) scores[t * k + lane] = acc;
  if (lane == 0 && !isfinite(acc)) set_status(status, LRM_ERR_NONFINITE);
}

void launch_grad_score(const void* g, int64_t T, int32_t k, int32_t H, lrm_dtype dt, bool abs_mode, float* scores,
                       int32_t* status, cudaStream_t s) {
  if (T == 0) return;
  const unsigned blocks = (unsigned)((T + 7) / 8);
  const int gv = (H / (dt == LRM_BF16 ? 8 : 4) + 31) / 32;  // vectors per lane of a g row
  using B = __nv_bfloat16;
#define LRM_GRAD_LAUNCH(TYPE, ABS)                                                                      \
  do {                                                                                                  \
    if (gv <= 16)                                                                                       \
      grad_score_kernel<TYPE, ABS, 16><<<blocks, 256, 0, s>>>((const TYPE*)g, T, k, H, scores, status); \
    else                                                                                                \
      grad_score_kernel<TYPE, ABS, 0><<<blocks, 256, 0, s>>>((const TYPE*)g, T, k, H, scores, status);  \
  } while (0)
  if (dt == LRM_BF16 && abs_mode) LRM_GRAD_LAUNCH(B, true);
  else if (dt == LRM_BF16) LRM_GRAD_LAUNCH(B, false);
  else if (abs_mode) LRM_GRAD_LAUNCH(float, true);
  else LRM_GRAD_LAUNCH(float, false);
#undef LRM_GRAD_LAUNCH
}

void launch_score(const float* alpha, const void* g, const void* phi, int64_t T, int32_t k, int32_t H, int32_t I,
                  lrm_dtype dt, float* scores, int32_t* status, cudaStream_t s) {
  if (T == 0) return;
  const int64_t blocks = (T + 7) / 8;  // 8 warps (tokens) per CTA
  const int vn = dt == LRM_BF16 ? 8 : 4;
  const int gv = (H / vn + 31) / 32, pv = (I / vn + 31) / 32;  // vectors per lane of a g / phi row
  if (dt == LRM_BF16 && gv <= 8 && pv <= 3 && k <= 8) {
    using B = __nv_bfloat16;
    launch_chained(score_onepass_kernel<B, 8, 3, 8>, dim3((unsigned)((T + 3) / 4)), dim3(128), 0, s, alpha,
                   (const B*)g, (const B*)phi, T, k, H, I, scores, status);
    return;
  }
  const bool fits = gv <= 16 && pv <= 6;
#define LRM_SCORE_LAUNCH(TYPE, GV, PV)                                                                 \
  launch_chained(score_kernel<TYPE, GV, PV>, dim3((unsigned)blocks), dim3(256), 0, s, alpha, (const TYPE*)g, \
                 (const TYPE*)phi, T, k, H, I, scores, status)
  if (dt == LRM_BF16) {
    if (fits) LRM_SCORE_LAUNCH(__nv_bfloat16, 16, 6); else LRM_SCORE_LAUNCH(__nv_bfloat16, 0, 0);
  } else {
    if (fits) LRM_SCORE_LAUNCH(float, 16, 6); else LRM_SCORE_LAUNCH(float, 0, 0);
  }
#undef LRM_SCORE_LAUNCH
}

}  // namespace lrm
