// Forward-side steps beside the pruned backward, each fused with the work next to it.
//
// route: the router's top-k and routing weights, with the per-expert loads and the backward
//   retention quotas computed in the same launch.  "LRMoE: Trimming Backward Work in
//   Memory-Bound MoE Training", section "Backward demand is not a constant": each expert's quota
//   is fixed from its routed demand before the expert forward, so it can be set where the routing
//   is decided.  One warp per token keeps the token's logits in registers (lane l holds experts
//   l, l+32, ...), picks the k largest by repeated warp arg-max (ties to the lower expert id) and
//   takes the softmax over them; a CTA counts its tokens' experts in shared memory and adds the
//   counts to accumulators in the workspace; the CTA that finishes last copies them to `loads`
//   and applies the quota rule.  A few CTAs per SM walk the tokens, so few counts are flushed.
//
// swiglu_forward: phi = SiLU(gate) * up for every pair row, stored in the input dtype, and
//   ||phi_u||^2 of the stored row.  Section "LRM: a decomposable contribution score": the score
//   needs only that norm of the saved projection input, so a forward that emits it spares the
//   backward a second read of phi.  One warp per row, 16-byte loads and stores, all of a lane's
//   loads issued before any is used.
#include "common.cuh"
#include "kernels.h"

namespace lrm {

namespace {

constexpr int kRouteWarps = 16;  // 512-thread CTAs, two per SM: few count flushes

template <int MAXM>  // E <= 32 * MAXM
__global__ void __launch_bounds__(32 * kRouteWarps) route_kernel(
    const float* __restrict__ logits, int64_t n_tok, int E, int k, int kind, int32_t num, int32_t den, int32_t cap,
    const int32_t* __restrict__ explicit_q, int32_t* __restrict__ topk_idx, float* __restrict__ alpha,
    int32_t* __restrict__ loads, int32_t* __restrict__ quotas, uint32_t* __restrict__ done,
    int32_t* __restrict__ acc, int32_t* status) {
  extern __shared__ int hist[];  // [E]
  __shared__ bool s_last;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kRouteWarps;
  // the next token's logits are loaded while this token's experts are picked
  float nxt[MAXM];
  auto load_row = [&](int64_t tt) {
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
      const int e = lane + 32 * m;
      nxt[m] = (tt < n_tok && e < E) ? __ldg(logits + tt * E + e) : -INFINITY;
    }
  };
  int64_t t = (int64_t)blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  load_row(t);
  for (; t < n_tok; t += stride) {
    float v[MAXM];
    bool bad = false;
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
      const int e = lane + 32 * m;
      float x = nxt[m];
      if (e < E && !isfinite(x)) {
        bad = true;
        x = -INFINITY;  // a non-finite logit is never preferred, and is reported
      }
      v[m] = x;
    }
    load_row(t + stride);
    if (bad) set_status(status, LRM_ERR_NONFINITE);
    uint32_t taken = 0;  // bit m: expert lane + 32m already chosen
    int my_e = 0;
    float my_v = -INFINITY;
    for (int j = 0; j < k; ++j) {
      // this lane's best remaining expert: larger logit, then smaller id (m ascending = id ascending)
      float bv = -INFINITY;
      int be = INT32_MAX;
#pragma unroll
      for (int m = 0; m < MAXM; ++m) {
        const int e = lane + 32 * m;
        if (e < E && !((taken >> m) & 1u) && (v[m] > bv || be == INT32_MAX)) {
          bv = v[m];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == j) {
        my_e = be;
        my_v = bv;
      }
    }
    const float top = __shfl_sync(0xffffffffu, my_v, 0);
    const float w = lane < k ? expf(my_v - top) : 0.f;
    const float sum = warp_sum(w);
    if (lane < k) {
      topk_idx[t * k + lane] = my_e;
      alpha[t * k + lane] = w / sum;
      atomicAdd(&hist[my_e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (hist[e]) atomicAdd(&acc[e], hist[e]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int32_t l = *reinterpret_cast<volatile int32_t*>(acc + e);
    loads[e] = l;
    quotas[e] = quota_rule(l, kind, num, den, cap, explicit_q, e);
  }
}

template <typename T, int PV>  // PV: bound on the 16-byte vectors per lane of a phi row (0 = looped)
__global__ void __launch_bounds__(256) swiglu_fwd_kernel(const T* __restrict__ h, int64_t n_rows, int I,
                                                         T* __restrict__ phi, float* __restrict__ phi_sq) {
  constexpr int VN = VecTraits<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (u >= n_rows) return;
  const int nv = I / VN;
  const T* hg = h + u * 2 * (int64_t)I;
  const T* hu = hg + I;
  T* out = phi + u * (int64_t)I;
  float acc = 0.f;
  auto one = [&](uint4 gv, uint4 uv, int v) {
    float gate[VN], up[VN], f[VN];
    unpack(gv, gate);
    unpack(uv, up);
#pragma unroll
    for (int q = 0; q < VN; ++q) f[q] = gate[q] / (1.f + expf(-gate[q])) * up[q];
    const uint4 pv = pack(f);
    st16(out + (int64_t)v * VN, pv);
    float r[VN];
    unpack(pv, r);  // the norm of the stored (rounded) row
#pragma unroll
    for (int q = 0; q < VN; ++q) acc = fmaf(r[q], r[q], acc);
  };
  if (PV > 0) {
    constexpr int M = PV > 0 ? PV : 1;
    uint4 gb[M], ub[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int v = lane + 32 * m;
      if (v < nv) {
        gb[m] = ld_stream16(hg + (int64_t)v * VN);
        ub[m] = ld_stream16(hu + (int64_t)v * VN);
      }
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int v = lane + 32 * m;
      if (v < nv) one(gb[m], ub[m], v);
    }
  } else {
    for (int v = lane; v < nv; v += 32) one(ld_stream16(hg + (int64_t)v * VN), ld_stream16(hu + (int64_t)v * VN), v);
  }
  acc = warp_sum(acc);
  if (lane == 0 && phi_sq != nullptr) phi_sq[u] = acc;
}

}  // namespace

lrm_status launch_route(const float* logits, int64_t T, int32_t E, int32_t k, int kind, int32_t num, int32_t den,
                        int32_t cap, const int32_t* explicit_q, int32_t* topk_idx, float* alpha, int32_t* loads,
                        int32_t* quotas, uint32_t* ws, int32_t* status, cudaStream_t s) {
  // ws: [0] the finished-CTA counter, [1 .. E] the load accumulators; one memset clears both
  uint32_t* done = ws;
  int32_t* acc = reinterpret_cast<int32_t*>(ws + 1);
  if (cudaMemsetAsync(ws, 0, sizeof(uint32_t) * (E + 1), s) != cudaSuccess) return LRM_ERR_CUDA;
  int64_t blocks = (T + kRouteWarps - 1) / kRouteWarps;
  if (blocks > 152 * 2) blocks = 152 * 2;  // grid-stride beyond two CTAs per SM: fewer count flushes
  if (blocks < 1) blocks = 1;              // T = 0 still applies the rule (all loads 0)
  const size_t smem = sizeof(int) * E;
#define LRM_ROUTE(MAXM)                                                                                   \
  route_kernel<MAXM><<<(unsigned)blocks, 32 * kRouteWarps, smem, s>>>(logits, T, E, k, kind, num, den, cap, \
                                                                      explicit_q, topk_idx, alpha, loads,   \
                                                                      quotas, done, acc, status)
  if (E <= 128) LRM_ROUTE(4);
  else if (E <= 256) LRM_ROUTE(8);
  else if (E <= 512) LRM_ROUTE(16);
  else LRM_ROUTE(32);
#undef LRM_ROUTE
  return cudaGetLastError() == cudaSuccess ? LRM_OK : LRM_ERR_CUDA;
}

void launch_swiglu_forward(const void* h, int64_t P, int32_t I, lrm_dtype dt, void* phi, float* phi_sq,
                           cudaStream_t s) {
  if (P == 0) return;
  const unsigned blocks = (unsigned)((P + 7) / 8);
  const int pv = (I / (dt == LRM_BF16 ? 8 : 4) + 31) / 32;
  using B = __nv_bfloat16;
  if (dt == LRM_BF16) {
    if (pv <= 6) swiglu_fwd_kernel<B, 6><<<blocks, 256, 0, s>>>((const B*)h, P, I, (B*)phi, phi_sq);
    else swiglu_fwd_kernel<B, 0><<<blocks, 256, 0, s>>>((const B*)h, P, I, (B*)phi, phi_sq);
  } else {
    if (pv <= 6) swiglu_fwd_kernel<float, 6><<<blocks, 256, 0, s>>>((const float*)h, P, I, (float*)phi, phi_sq);
    else swiglu_fwd_kernel<float, 0><<<blocks, 256, 0, s>>>((const float*)h, P, I, (float*)phi, phi_sq);
  }
}

}  // namespace lrm
