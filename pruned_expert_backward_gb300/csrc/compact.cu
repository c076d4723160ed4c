// Physical compaction and the return to token layout.
//
// "LRMoE: Trimming Backward Work in Memory-Bound MoE Training", section "The part that is
// easy to get wrong": zero-masking dropped rows saves nothing; the retained gradient rows
// and their saved activations are repacked into contiguous, unpadded, expert-segmented
// buffers.  "LRMoE poda a passagem reversa do MoE..." (news.hamidun.com), compaction step:
// afterwards the result returns to the original layout.
//
// compact: one CTA per token.  The compacted row of every pair is already known
// (row_of_pair), so the kernel walks tokens, reads g_t and x_t once, and writes them (g_t
// scaled by alpha_u) into each kept pair's row; the token's k rows of h and phi are one
// contiguous span, read only where the pair is kept.  16-byte coalesced loads and stores.
//
// scatter_dx: a CTA covers several tokens (up to 512 threads); each thread owns one 16-byte
// column slice of one token, issues the k row loads together and adds them in j order in
// fp32 (deterministic, no atomics).
#include "common.cuh"
#include "kernels.h"

namespace lrm {

namespace {

template <typename T>
__global__ void __launch_bounds__(256) compact_kernel(const int32_t* __restrict__ row_of_pair,
                                                      const float* __restrict__ alpha, const T* __restrict__ g,
                                                      const T* __restrict__ x, const T* __restrict__ h,
                                                      const T* __restrict__ phi, int k, int H, int I, int64_t cap,
                                                      T* __restrict__ dy_c, T* __restrict__ x_c, T* __restrict__ h_c,
                                                      T* __restrict__ phi_c) {
  constexpr int VN = VecTraits<T>::N;
  __shared__ int64_t s_row[LRM_MAX_TOPK];
  __shared__ float s_alpha[LRM_MAX_TOPK];
  __shared__ int s_any;
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x, nt = blockDim.x;
  if (tid == 0) s_any = 0;
  __syncthreads();
  if (tid < k) {
    const int r = row_of_pair[t * k + tid];
    const bool kept = r >= 0 && (int64_t)r < cap;
    s_row[tid] = kept ? (int64_t)r : -1;
    s_alpha[tid] = alpha[t * k + tid];
    if (kept) s_any = 1;
  }
  __syncthreads();
  if (!s_any) return;

  const int nvH = H / VN;
  const T* gt = g + t * H;
  const T* xt = x + t * H;
  for (int v = tid; v < nvH; v += nt) {
    const uint4 gv = ld_stream16(gt + v * VN);
    const uint4 xv = x_c != nullptr ? ld_stream16(xt + v * VN) : make_uint4(0, 0, 0, 0);
    float f[VN];
    unpack(gv, f);
    for (int j = 0; j < k; ++j) {
      const int64_t r = s_row[j];
      if (r < 0) continue;
      const float a = s_alpha[j];
      float o[VN];
#pragma unroll
      for (int q = 0; q < VN; ++q) o[q] = a * f[q];
      st16(dy_c + r * H + v * VN, pack(o));
      if (x_c != nullptr) st16(x_c + r * H + v * VN, xv);
    }
  }
  if (h_c == nullptr) return;  // compaction-free variant: only the scaled gradient rows

  const int nv2 = 2 * I / VN;
  const T* ht = h + t * k * (int64_t)(2 * I);
  for (int v = tid; v < k * nv2; v += nt) {
    const int j = v / nv2;
    const int64_t r = s_row[j];
    if (r < 0) continue;
    st16(h_c + r * (2 * I) + (v - j * nv2) * VN, ld_stream16(ht + (int64_t)v * VN));
  }
  const int nv1 = I / VN;
  const T* pt = phi + t * k * (int64_t)I;
  for (int v = tid; v < k * nv1; v += nt) {
    const int j = v / nv1;
    const int64_t r = s_row[j];
    if (r < 0) continue;
    st16(phi_c + r * I + (v - j * nv1) * VN, ld_stream16(pt + (int64_t)v * VN));
  }
}

template <typename T, int MAXK>
__global__ void __launch_bounds__(512, MAXK <= 8 ? 2 : 1) scatter_dx_kernel(const int32_t* __restrict__ row_of_pair,
                                                          const T* __restrict__ dx_c, int64_t n_tok, int k, int H,
                                                          int tok_per_blk, T* __restrict__ dx) {
  constexpr int VN = VecTraits<T>::N;
  extern __shared__ int32_t s_rows[];  // [tok_per_blk][k]
  const int64_t t0 = (int64_t)blockIdx.x * tok_per_blk;
  for (int i = threadIdx.x; i < tok_per_blk * k; i += blockDim.x) {
    const int64_t u = t0 * k + i;
    s_rows[i] = u < n_tok * k ? row_of_pair[u] : -1;
  }
  __syncthreads();
  const int nvH = H / VN;
  for (int w = threadIdx.x; w < tok_per_blk * nvH; w += blockDim.x) {
    const int tt = w / nvH, v = w - tt * nvH;
    const int64_t t = t0 + tt;
    if (t >= n_tok) break;
    const int32_t* srow = s_rows + tt * k;
    int32_t rows[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) rows[j] = j < k ? srow[j] : -1;
    uint4 vals[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      if (rows[j] >= 0) vals[j] = ld_stream16(dx_c + (int64_t)rows[j] * H + v * VN);
    }
    float acc[VN];
#pragma unroll
    for (int q = 0; q < VN; ++q) acc[q] = 0.f;
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      if (rows[j] >= 0) {
        float f[VN];
        unpack(vals[j], f);
#pragma unroll
        for (int q = 0; q < VN; ++q) acc[q] += f[q];
      }
    }
    st16(dx + t * H + v * VN, pack(acc));
  }
}

int threads_for(int n_vec) {
  int t = n_vec < 512 ? n_vec : 512;
  t = (t + 31) / 32 * 32;
  return t < 32 ? 32 : t;
}

}  // namespace

void launch_compact(const int32_t* row_of_pair, const float* alpha, const void* g, const void* x, const void* h,
                    const void* phi, int64_t T, int32_t k, int32_t H, int32_t I, lrm_dtype dt, int64_t cap,
                    void* dy_c, void* x_c, void* h_c, void* phi_c, cudaStream_t s) {
  if (T == 0) return;
  if (dt == LRM_BF16) {
    using B = __nv_bfloat16;
    compact_kernel<B><<<(unsigned)T, 256, 0, s>>>(row_of_pair, alpha, (const B*)g, (const B*)x, (const B*)h,
                                                  (const B*)phi, k, H, I, cap, (B*)dy_c, (B*)x_c, (B*)h_c,
                                                  (B*)phi_c);
  } else {
    compact_kernel<float><<<(unsigned)T, 256, 0, s>>>(row_of_pair, alpha, (const float*)g, (const float*)x,
                                                      (const float*)h, (const float*)phi, k, H, I, cap,
                                                      (float*)dy_c, (float*)x_c, (float*)h_c, (float*)phi_c);
  }
}

void launch_scatter_dx(const int32_t* row_of_pair, const void* dx_c, int64_t T, int32_t k, int32_t H, lrm_dtype dt,
                       void* dx, cudaStream_t s) {
  if (T == 0) return;
  const int nvH = H / (dt == LRM_BF16 ? 8 : 4);
  int tok = nvH >= 512 ? 1 : 512 / nvH;  // one thread per 16-byte column slice, up to 512 threads
  if (tok > 64) tok = 64;
  const int threads = threads_for(nvH * tok);
  const unsigned blocks = (unsigned)((T + tok - 1) / tok);
  const size_t smem = sizeof(int32_t) * tok * k;
  using B = __nv_bfloat16;
  if (dt == LRM_BF16 && k <= 8)
    scatter_dx_kernel<B, 8><<<blocks, threads, smem, s>>>(row_of_pair, (const B*)dx_c, T, k, H, tok, (B*)dx);
  else if (dt == LRM_BF16)
    scatter_dx_kernel<B, LRM_MAX_TOPK><<<blocks, threads, smem, s>>>(row_of_pair, (const B*)dx_c, T, k, H, tok,
                                                                     (B*)dx);
  else if (k <= 8)
    scatter_dx_kernel<float, 8><<<blocks, threads, smem, s>>>(row_of_pair, (const float*)dx_c, T, k, H, tok,
                                                              (float*)dx);
  else
    scatter_dx_kernel<float, LRM_MAX_TOPK><<<blocks, threads, smem, s>>>(row_of_pair, (const float*)dx_c, T, k, H,
                                                                         tok, (float*)dx);
}

}  // namespace lrm
