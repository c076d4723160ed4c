// CUDA-core grouped GEMMs of the SwiGLU expert backward (fp32 accumulation).
//
// Used for fp32 inputs, where tensor-core formats (TF32/BF16) would not reach fp32
// accuracy, and on request for bf16.  Segment sizes are read on the device from
// seg_offsets, so nothing waits on the host ("LRMoE: Trimming Backward Work in
// Memory-Bound MoE Training", section "The part that is easy to get wrong": the actual
// retained row counts drive variable-size grouped GEMMs, with no padding).
//
//  var-M (rows of a segment are the M dimension):
//    dphi = dy_c[e] W_down[e]  with the SwiGLU backward fused into the epilogue -> dh_c
//    dx_c = dh_c[e] W_gate_up[e]
//  var-K (rows of a segment are the reduction dimension):
//    dW_down[e] = dy_c[e]^T phi_c[e],  dW_gate_up[e] = dh_c[e]^T x_c[e]
// 64 x 64 output tiles, 16-deep K slices in shared memory, 256 threads x 4 x 4 outputs.
#include "common.cuh"
#include "kernels.h"

namespace lrm {

namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

enum { EPI_SWIGLU = 0, EPI_STORE = 1 };

// seg_offsets must be a segmentation of [0, seg[E]] within [0, cap]: seg[0] = 0, no decreasing
// step, seg[E] <= cap.  Checked by every block before it reads a row (block-wide vote); a block
// that finds it broken records LRM_ERR_BAD_SEGMENTS and computes nothing.
__device__ bool segments_valid(const int32_t* seg, int E, int64_t cap, int32_t* status) {
  int ok = 1;
  for (int e = threadIdx.x; e < E; e += blockDim.x) ok &= seg[e] <= seg[e + 1] ? 1 : 0;
  if (threadIdx.x == 0) ok &= (seg[0] == 0 && (int64_t)seg[E] <= cap) ? 1 : 0;
  const bool valid = __syncthreads_and(ok) != 0;
  if (!valid && threadIdx.x == 0) set_status(status, LRM_ERR_BAD_SEGMENTS);
  return valid;
}

// Row of h / phi (pair) or x (token, when div > 0) named by a kept_pair entry u, or -1 when u is
// outside [0, n_pairs) (recorded as LRM_ERR_BAD_INDEX; the row then reads as zeros).
__device__ __forceinline__ int64_t gathered_row(int32_t u, int64_t n_pairs, int div, int32_t* status) {
  if (u < 0 || (int64_t)u >= n_pairs) {
    set_status(status, LRM_ERR_BAD_INDEX);
    return -1;
  }
  return div > 0 ? u / div : u;
}

// Map a virtual M-tile id to (expert, first row, end row) from the per-expert tile prefix.
__device__ __forceinline__ bool find_mtile(const int32_t* seg, int E, int vt, int* s_prefix, int* e_out,
                                           int* r0_out, int* r1_out) {
  // s_prefix[e] = number of M tiles of experts < e (computed by the caller's block).
  int lo = 0, hi = E;  // find largest e with s_prefix[e] <= vt
  if (vt >= s_prefix[E]) return false;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_prefix[mid] <= vt) lo = mid; else hi = mid;
  }
  const int e = lo;
  const int r0 = seg[e] + (vt - s_prefix[e]) * BM;
  *e_out = e;
  *r0_out = r0;
  *r1_out = min(seg[e + 1], r0 + BM);
  return true;
}

__device__ void mtile_prefix(const int32_t* seg, int E, int* s_prefix) {
  // serial prefix by thread 0 is fine: E <= 1024 and this kernel is the fallback path
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      s_prefix[e] = acc;
      acc += (seg[e + 1] - seg[e] + BM - 1) / BM;
    }
    s_prefix[E] = acc;
  }
  __syncthreads();
}

// C[r, n] = sum_k A[r, k] * B_e[k, n]; A [rows, K] row-major, B_e [K, N] row-major (BT: B_e is
// stored as [N, K], i.e. C = A B_e^T, as for the rows of W_gate_up).
template <typename T, int EPI, bool BT = false>
__global__ void __launch_bounds__(NT) varm_kernel(const int32_t* __restrict__ seg, int E,
                                                  const T* __restrict__ A, const T* __restrict__ B, int K, int N,
                                                  const T* __restrict__ h_c, T* __restrict__ out,
                                                  float* __restrict__ dot_part, int n_part,
                                                  const int32_t* __restrict__ h_rows, int64_t n_pairs, int64_t cap,
                                                  int32_t* __restrict__ status) {
  // h_rows (compaction-free variant): the gate/up row of output row r is h_c[h_rows[r]]
  __shared__ int s_prefix[LRM_MAX_EXPERTS + 1];
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  if (!segments_valid(seg, E, cap, status)) return;
  mtile_prefix(seg, E, s_prefix);
  int e, r0, r1;
  if (!find_mtile(seg, E, blockIdx.x, s_prefix, &e, &r0, &r1)) return;
  const int n0 = blockIdx.y * BN;
  const T* Be = B + (int64_t)e * K * N;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    // A tile: 64 rows x 16 k; thread loads 4 consecutive k of one row
    {
      const int m = threadIdx.x / 4, kq = (threadIdx.x % 4) * 4;
      const int r = r0 + m;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kk = k0 + kq + q;
        As[kq + q][m] = (r < r1 && kk < K) ? to_f(A[(int64_t)r * K + kk]) : 0.f;
      }
    }
    // B tile: 16 k x 64 n
    {
      const int kk = threadIdx.x / 16, nq = (threadIdx.x % 16) * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int n = n0 + nq + q;
        const int64_t bi = BT ? (int64_t)n * K + (k0 + kk) : (int64_t)(k0 + kk) * N + n;
        Bs[kk][nq + q] = (k0 + kk < K && n < N) ? to_f(Be[bi]) : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float rdot[4] = {0.f, 0.f, 0.f, 0.f};  // EPI_SWIGLU: dphi . phi over this thread's columns
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty * 4 + i;
    if (r >= r1) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      if (EPI == EPI_SWIGLU) {
        // N = I here; h_c row is [gate (I) ; up (I)]
        const int64_t hr = h_rows ? gathered_row(h_rows[r], n_pairs, 0, status) : (int64_t)r;
        const float gate = hr >= 0 ? to_f(h_c[hr * 2 * N + n]) : 0.f;
        const float up = hr >= 0 ? to_f(h_c[hr * 2 * N + N + n]) : 0.f;
        const float sg = 1.f / (1.f + expf(-gate));
        const float dphi = acc[i][j];
        const float du = dphi * gate * sg;
        out[(int64_t)r * 2 * N + n] = from_f<T>(dphi * up * sg * (1.f + gate * (1.f - sg)));
        out[(int64_t)r * 2 * N + N + n] = from_f<T>(du);
        rdot[i] = fmaf(du, up, rdot[i]);  // dphi * phi, phi = gate * s * up
      } else {
        out[(int64_t)r * N + n] = from_f<T>(acc[i][j]);
      }
    }
  }
  if (EPI == EPI_SWIGLU && dot_part != nullptr) {
    // the 16 threads of a row group (tx = lane & 15) add their parts in a fixed order
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) rdot[i] += __shfl_xor_sync(0xffffffffu, rdot[i], o);
      const int r = r0 + ty * 4 + i;
      if (tx == 0 && r < r1) dot_part[(int64_t)r * n_part + blockIdx.y] = rdot[i];
    }
  }
}

// C_e[m, n] = sum_{r in segment e} A[r, m] * B[r', n]; A [rows, M], B [*, N] row-major, where
// r' = r, or (compaction-free variant) r' = b_rows[r] / b_div (b_div > 0) or b_rows[r].
template <typename T>
__global__ void __launch_bounds__(NT) vark_kernel(const int32_t* __restrict__ seg, int E, const T* __restrict__ A,
                                                  const T* __restrict__ B, int M, int N, float* __restrict__ C,
                                                  const int32_t* __restrict__ b_rows, int b_div, int64_t n_pairs,
                                                  int64_t cap, int32_t* __restrict__ status) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  if (!segments_valid(seg, E, cap, status)) return;
  const int e = blockIdx.z;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int r0 = seg[e], r1 = seg[e + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = r0; k0 < r1; k0 += BK) {
    {
      const int kk = threadIdx.x / 16, q4 = (threadIdx.x % 16) * 4;
      const int r = k0 + kk;
      int64_t rb = r;
      if (b_rows != nullptr && r < r1) rb = gathered_row(b_rows[r], n_pairs, b_div, status);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int m = m0 + q4 + q, n = n0 + q4 + q;
        As[kk][q4 + q] = (r < r1 && m < M) ? to_f(A[(int64_t)r * M + m]) : 0.f;
        Bs[kk][q4 + q] = (r < r1 && n < N && rb >= 0) ? to_f(B[rb * N + n]) : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* Ce = C + (int64_t)e * M * N;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) Ce[(int64_t)m * N + n] = acc[i][j];
    }
  }
}

// phi_c[r] = SiLU(gate) * up from the row h_c[r] = [gate ; up] (as stored), rows r < seg_offsets[E].
template <typename T>
__global__ void __launch_bounds__(256) phi_rows_kernel(const int32_t* __restrict__ seg, int E, int64_t cap, int I,
                                                       const T* __restrict__ h_c, T* __restrict__ phi_c,
                                                       int32_t* __restrict__ status) {
  if (!segments_valid(seg, E, cap, status)) return;
  int64_t rows = seg[E];
  if (rows > cap) rows = cap;
  const int64_t n = rows * I;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / I;
    const int c = (int)(i - r * I);
    const float g = to_f(h_c[r * 2 * I + c]), u = to_f(h_c[r * 2 * I + I + c]);
    phi_c[i] = from_f<T>(g / (1.f + expf(-g)) * u);
  }
}

template <typename T>
void recompute_all(const RecomputeArgs& a, cudaStream_t s) {
  const int64_t mtiles = (a.cap + BM - 1) / BM + a.E;
  // h_c = x_c W_gate_up[e]^T over the 2I columns, then phi_c from the stored h_c rows
  varm_kernel<T, EPI_STORE, true><<<dim3((unsigned)mtiles, (2 * a.I + BN - 1) / BN), NT, 0, s>>>(
      a.seg_offsets, a.E, (const T*)a.x_c, (const T*)a.w_gate_up, a.H, 2 * a.I, nullptr, (T*)a.h_c, nullptr, 0,
      nullptr, 0, a.cap, a.status);
  phi_rows_kernel<T><<<1216, 256, 0, s>>>(a.seg_offsets, a.E, a.cap, a.I, (const T*)a.h_c, (T*)a.phi_c, a.status);
}

template <typename T>
void run_all(const GroupedArgs& a, cudaStream_t s) {
  const int E = a.E, H = a.H, I = a.I;
  // Upper bound on M tiles: every expert adds at most one partial tile.
  const int64_t mtiles = (a.cap + BM - 1) / BM + E;
  const T* dy = (const T*)a.dy_c;
  const bool gather = a.kept_pair != nullptr;  // compaction-free: x / h / phi rows read by index
  const T* xc = (const T*)(gather ? a.x : a.x_c);
  const T* hc = (const T*)(gather ? a.h : a.h_c);
  const T* pc = (const T*)(gather ? a.phi : a.phi_c);
  T* dh = (T*)a.dh_c;
  T* dx = (T*)a.dx_c;
  if (mtiles > 0) {
    // dphi + SwiGLU backward: [R_e, H] x [H, I]
    const int n_part = (I + BN - 1) / BN;
    varm_kernel<T, EPI_SWIGLU><<<dim3((unsigned)mtiles, n_part), NT, 0, s>>>(
        a.seg_offsets, E, dy, (const T*)a.w_down, H, I, hc, dh, a.row_dot ? a.dot_part : nullptr, n_part,
        a.kept_pair, a.n_pairs, a.cap, a.status);
    if (a.row_dot != nullptr) launch_row_dot(a.dot_part, n_part, a.seg_offsets, E, a.cap, a.row_dot, s);
  }
  // dW_down[e] = dy_c^T phi_c : [H, I]
  vark_kernel<T><<<dim3((I + BN - 1) / BN, (H + BM - 1) / BM, E), NT, 0, s>>>(
      a.seg_offsets, E, dy, pc, H, I, a.dw_down, a.kept_pair, 0, a.n_pairs, a.cap, a.status);
  // dW_gate_up[e] = dh_c^T x_c : [2I, H]
  vark_kernel<T><<<dim3((H + BN - 1) / BN, (2 * I + BM - 1) / BM, E), NT, 0, s>>>(
      a.seg_offsets, E, (const T*)dh, xc, 2 * I, H, a.dw_gate_up, a.kept_pair, a.k, a.n_pairs, a.cap, a.status);
  if (mtiles > 0) {
    // dx_c = dh_c W_gate_up[e] : [R_e, 2I] x [2I, H]
    varm_kernel<T, EPI_STORE><<<dim3((unsigned)mtiles, (H + BN - 1) / BN), NT, 0, s>>>(
        a.seg_offsets, E, (const T*)dh, (const T*)a.w_gate_up, 2 * I, H, nullptr, dx, nullptr, 0, nullptr, 0, a.cap,
        a.status);
  }
}

}  // namespace

void launch_recompute_simt(const RecomputeArgs& a, lrm_dtype dt, cudaStream_t s) {
  if (dt == LRM_BF16)
    recompute_all<__nv_bfloat16>(a, s);
  else
    recompute_all<float>(a, s);
}

void launch_grouped_simt(const GroupedArgs& a, lrm_dtype dt, cudaStream_t s) {
  if (dt == LRM_BF16)
    run_all<__nv_bfloat16>(a, s);
  else
    run_all<float>(a, s);
}

}  // namespace lrm
