// Physical compaction and the return to token layout.
//
// "LRMoE: Trimming Backward Work in Memory-Bound MoE Training", section "The part that is
// easy to get wrong": zero-masking dropped rows saves nothing; the retained gradient rows
// and their saved activations are repacked into contiguous, unpadded, expert-segmented
// buffers.  "LRMoE poda a passagem reversa do MoE..." (news.hamidun.com), compaction step:
// afterwards the result returns to the original layout.
//
// compact: one CTA per token (two 16-byte vectors of a g row per thread, 64-256 threads).  The compacted row of every pair is already known
// (row_of_pair), so the kernel walks tokens, reads g_t and x_t once, and writes them (g_t
// scaled by alpha_u) into each kept pair's row; the token's k rows of h and phi are one
// contiguous span, read only where the pair is kept.  16-byte coalesced loads and stores.
//
// scatter_dx: a CTA covers 8 tokens; each thread owns one 16-byte column slice, walks the
// CTA's kept rows with 8 loads in flight and adds each token's rows in j order in fp32
// (deterministic, no atomics).
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
                                                      T* __restrict__ phi_c, int32_t* __restrict__ status) {
  chain_wait();
  constexpr int VN = VecTraits<T>::N;
  __shared__ int64_t s_row[LRM_MAX_TOPK];
  __shared__ float s_alpha[LRM_MAX_TOPK];
  __shared__ int s_kept[LRM_MAX_TOPK];  // the token's kept choices j, ascending
  __shared__ int s_nk;
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x, nt = blockDim.x;
  if (tid < 32) {
    int64_t r = -1;
    if (tid < k) {
      r = checked_row(row_of_pair[t * k + tid], cap, status);  // outside [-1, cap): flagged, dropped
      s_row[tid] = r;
      s_alpha[tid] = alpha[t * k + tid];
    }
    const unsigned m = __ballot_sync(0xffffffffu, r >= 0);
    if (r >= 0) s_kept[__popc(m & ((1u << tid) - 1u))] = tid;
    if (tid == 0) s_nk = __popc(m);
  }
  __syncthreads();
  const int nk = s_nk;
  if (nk == 0) return;

  const int nvH = H / VN;
  const T* gt = g + t * H;
  const T* xt = x + t * H;
  for (int v = tid; v < nvH; v += nt) {
    const uint4 gv = ld_stream16(gt + v * VN);
    const uint4 xv = x_c != nullptr ? ld_stream16(xt + v * VN) : make_uint4(0, 0, 0, 0);
    float f[VN];
    unpack(gv, f);
    for (int jj = 0; jj < nk; ++jj) {
      const int j = s_kept[jj];
      const int64_t r = s_row[j];
      const float a = s_alpha[j];
      float o[VN];
#pragma unroll
      for (int q = 0; q < VN; ++q) o[q] = a * f[q];
      st16(dy_c + r * H + v * VN, pack(o));
      if (x_c != nullptr) st16(x_c + r * H + v * VN, xv);
    }
  }
  if (h_c == nullptr) return;  // compaction-free variant: only the scaled gradient rows

  // the kept pairs' h and phi rows only (v runs over kept rows x vectors)
  const int nv2 = 2 * I / VN;
  const T* ht = h + t * k * (int64_t)(2 * I);
  for (int v = tid; v < nk * nv2; v += nt) {
    const int jj = v / nv2, c = v - jj * nv2;
    const int j = s_kept[jj];
    st16(h_c + s_row[j] * (2 * I) + c * VN, ld_stream16(ht + ((int64_t)j * nv2 + c) * VN));
  }
  const int nv1 = I / VN;
  const T* pt = phi + t * k * (int64_t)I;
  for (int v = tid; v < nk * nv1; v += nt) {
    const int jj = v / nv1, c = v - jj * nv1;
    const int j = s_kept[jj];
    st16(phi_c + s_row[j] * I + c * VN, ld_stream16(pt + ((int64_t)j * nv1 + c) * VN));
  }
}

// A CTA takes kScatterTok consecutive tokens.  Warp 0 lists their kept rows in (token, j) order
// in shared memory; then every thread walks that list for one 16-byte column slice, keeping
// kScatterLoads row loads in flight however few rows each token kept, and adds each token's rows
// in j order in fp32 (deterministic: the same sum in the same order as one row at a time).
constexpr int kScatterTok = 8;  // 16: 5 % slower at T = 32768 (fewer CTAs, longer lists), 32: slower still
constexpr int kScatterLoads = 8;

template <typename T>
__global__ void __launch_bounds__(256) scatter_dx_kernel(const int32_t* __restrict__ row_of_pair,
                                                         const T* __restrict__ dx_c, int64_t n_tok, int k, int H,
                                                         int64_t cap, T* __restrict__ dx, int32_t* __restrict__ status) {
  chain_wait();
  constexpr int VN = VecTraits<T>::N;
  constexpr int B = kScatterLoads;
  __shared__ int2 s_item[kScatterTok * LRM_MAX_TOPK];  // (token within the CTA, compacted row)
  __shared__ int s_n;
  const int64_t t0 = (int64_t)blockIdx.x * kScatterTok;
  const int ntok = (int)min((int64_t)kScatterTok, n_tok - t0);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int base = 0;
    for (int q0 = 0; q0 < ntok * k; q0 += 32) {
      const int q = q0 + lane;
      // a row outside [-1, cap) is flagged and not followed
      const int r = q < ntok * k ? (int)checked_row(row_of_pair[t0 * k + q], cap, status) : -1;
      const unsigned m = __ballot_sync(0xffffffffu, r >= 0);
      if (r >= 0) s_item[base + __popc(m & ((1u << lane) - 1u))] = make_int2(q / k, r);
      base += __popc(m);
    }
    if (lane == 0) s_n = base;
  }
  __syncthreads();
  const int n = s_n;
  const int nvH = H / VN;
  for (int v = threadIdx.x; v < nvH; v += blockDim.x) {
    float acc[VN];
#pragma unroll
    for (int q = 0; q < VN; ++q) acc[q] = 0.f;
    int cur = 0;  // the token acc belongs to; tokens before it are written
    for (int b0 = 0; b0 < n; b0 += B) {
      uint4 vals[B];
#pragma unroll
      for (int m = 0; m < B; ++m)
        if (b0 + m < n) vals[m] = ld_stream16(dx_c + (int64_t)s_item[b0 + m].y * H + (int64_t)v * VN);
#pragma unroll
      for (int m = 0; m < B; ++m) {
        if (b0 + m >= n) break;
        const int tok = s_item[b0 + m].x;
        while (cur < tok) {  // cur is complete (tokens with nothing kept get 0)
          st16(dx + (t0 + cur) * H + (int64_t)v * VN, pack(acc));
#pragma unroll
          for (int q = 0; q < VN; ++q) acc[q] = 0.f;
          ++cur;
        }
        float f[VN];
        unpack(vals[m], f);
#pragma unroll
        for (int q = 0; q < VN; ++q) acc[q] += f[q];
      }
    }
    while (cur < ntok) {
      st16(dx + (t0 + cur) * H + (int64_t)v * VN, pack(acc));
#pragma unroll
      for (int q = 0; q < VN; ++q) acc[q] = 0.f;
      ++cur;
    }
  }
}


}  // namespace

void launch_compact(const int32_t* row_of_pair, const float* alpha, const void* g, const void* x, const void* h,
                    const void* phi, int64_t T, int32_t k, int32_t H, int32_t I, lrm_dtype dt, int64_t cap,
                    void* dy_c, void* x_c, void* h_c, void* phi_c, int32_t* status, cudaStream_t s) {
  if (T == 0) return;
  // two 16-byte vectors of g_t / x_t per thread, 64 to 256 threads: a token that keeps few pairs
  // then holds fewer threads, and more tokens are in flight per SM (on GB300, Qwen3-shaped rows
  // (H = 2048, 128 threads): the Zipf-1.5 stress layer 368 -> 310 us, the others 1-2 % faster;
  // GLM4.5-shaped rows (H = 4096) keep 256)
  const int nvH = H / (dt == LRM_BF16 ? 8 : 4);
  int threads = (nvH / 2 + 31) / 32 * 32;
  threads = threads < 64 ? 64 : (threads > 256 ? 256 : threads);
  if (dt == LRM_BF16) {
    using B = __nv_bfloat16;
    launch_chained(compact_kernel<B>, dim3((unsigned)T), dim3(threads), 0, s, row_of_pair, alpha, (const B*)g,
                   (const B*)x, (const B*)h, (const B*)phi, k, H, I, cap, (B*)dy_c, (B*)x_c, (B*)h_c, (B*)phi_c, status);
  } else {
    launch_chained(compact_kernel<float>, dim3((unsigned)T), dim3(threads), 0, s, row_of_pair, alpha, (const float*)g,
                   (const float*)x, (const float*)h, (const float*)phi, k, H, I, cap, (float*)dy_c, (float*)x_c,
                   (float*)h_c, (float*)phi_c, status);
  }
}

void launch_scatter_dx(const int32_t* row_of_pair, const void* dx_c, int64_t T, int32_t k, int32_t H, lrm_dtype dt,
                       int64_t cap, void* dx, int32_t* status, cudaStream_t s) {
  if (T == 0) return;
  const int nvH = H / (dt == LRM_BF16 ? 8 : 4);
  int threads = (nvH + 31) / 32 * 32;  // one thread per 16-byte column slice (warp 0 also builds the list)
  if (threads > 256) threads = 256;
  const unsigned blocks = (unsigned)((T + kScatterTok - 1) / kScatterTok);
  if (dt == LRM_BF16)
    launch_chained(scatter_dx_kernel<__nv_bfloat16>, dim3(blocks), dim3(threads), 0, s, row_of_pair,
                   (const __nv_bfloat16*)dx_c, T, k, H, cap, (__nv_bfloat16*)dx, status);
  else
    launch_chained(scatter_dx_kernel<float>, dim3(blocks), dim3(threads), 0, s, row_of_pair, (const float*)dx_c, T,
                   k, H, cap, (float*)dx, status);
}

}  // namespace lrm
