// C ABI of the LRM-pruned expert backward: argument validation, workspace layout, dispatch.
// Every entry point only queues work on the caller's stream; nothing here allocates or
// synchronises.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "kernels.h"

namespace lrm {

namespace {

constexpr size_t kAlign = 256;
size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

lrm_status check_dims(int64_t T, int32_t k, int32_t E, int32_t H, int32_t I) {
  if (T < 0 || k < 1 || E < 1 || H < 1 || I < 1) return LRM_ERR_INVALID_ARG;
  if (k > LRM_MAX_TOPK || E > LRM_MAX_EXPERTS) return LRM_ERR_SHAPE;
  if (H % 8 != 0 || I % 8 != 0) return LRM_ERR_SHAPE;
  if (T > INT32_MAX / k) return LRM_ERR_SHAPE;  // P = T*k <= INT32_MAX, tested before multiplying
  return LRM_OK;
}
lrm_status check_dt(lrm_dtype dt) { return (dt == LRM_BF16 || dt == LRM_F32) ? LRM_OK : LRM_ERR_DTYPE; }

lrm_status after_launch() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? LRM_OK : LRM_ERR_CUDA;
}

}  // namespace

bool nvtx_enabled() {
  static const bool on = [] {
    const char* v = getenv("LRM_NVTX");
    return v != nullptr && v[0] == '1' && v[1] == 0;
  }();
  return on;
}
void nvtx_push(const char* name) { nvtxRangePushA(name); }
void nvtx_pop() { nvtxRangePop(); }

size_t gemm_plan_bytes(int32_t E) { return up(sizeof(int32_t) * (2 * (size_t)E + 3 + kTileCounters)); }
size_t gemm_ws_bytes(int32_t E) { return gemm_plan_bytes(E) + 128 * 6 * (size_t)E; }

// lrm_grouped_backward's scratch: tile tables and tensor maps, then (only when row_dot is
// requested) the dphi . phi parts of every row.
size_t grouped_ws_bytes(int64_t cap, int32_t E, int32_t I, bool row_dot) {
  size_t b = up(gemm_ws_bytes(E));
  if (row_dot) b += up(sizeof(float) * (size_t)(cap > 0 ? cap : 1) * dot_parts_max(I));
  return b;
}

WsLayout workspace_layout(int64_t P, int32_t E) {
  WsLayout w{};
  const int64_t nc = (P + kSelChunk - 1) / kSelChunk;
  size_t off = 0;
  w.counts = off;       off += up(sizeof(int32_t) * (size_t)(nc > 0 ? nc : 1) * E);
  w.bucket_start = off; off += up(sizeof(int32_t) * (size_t)(E + 1));
  w.keep = off;         off += up(sizeof(int32_t) * (size_t)E);
  w.loads = off;        off += up(sizeof(int32_t) * (size_t)E);
  w.sorted_u = off;     off += up(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
  w.sorted_key = off;   off += up(sizeof(uint32_t) * (size_t)(P > 0 ? P : 1));
  w.gemm = off;         off += up(gemm_ws_bytes(E));
  w.total = off;
  return w;
}

}  // namespace lrm

using namespace lrm;

extern "C" {

const char* lrm_status_string(lrm_status s) {
  switch (s) {
    case LRM_OK: return "ok";
    case LRM_ERR_INVALID_ARG: return "invalid argument (null/misaligned pointer, negative size or bad enum)";
    case LRM_ERR_SHAPE: return "size outside the supported limits";
    case LRM_ERR_DTYPE: return "unknown dtype";
    case LRM_ERR_WORKSPACE: return "workspace missing or too small";
    case LRM_ERR_CUDA: return "CUDA launch or runtime error";
    case LRM_ERR_CAPACITY: return "kept rows exceed the capacity";
    case LRM_ERR_NONFINITE: return "non-finite score";
    case LRM_ERR_TIMEOUT: return "a bounded device wait gave up";
    case LRM_ERR_BAD_INDEX: return "index out of range (expert id outside [0, E) or compacted row outside [-1, cap))";
    case LRM_ERR_UNSUPPORTED: return "unsupported device or configuration";
    case LRM_ERR_BAD_SEGMENTS: return "seg_offsets not a valid segmentation of [0, cap)";
  }
  return "unknown status";
}

lrm_status lrm_workspace_size(int64_t T, int32_t k, int32_t E, int32_t H, int32_t I, lrm_dtype dt, size_t* bytes) {
  LRM_NVTX_RANGE();
  if (!bytes) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(T, k, E, H, I);
  if (st) return st;
  if ((st = check_dt(dt))) return st;
  const size_t sel = workspace_layout(T * k, E).total, grp = grouped_ws_bytes(T * k, E, I, true);
  *bytes = sel > grp ? sel : grp;
  return LRM_OK;
}

lrm_status lrm_plan_quotas(const int32_t* topk_idx, int64_t T, int32_t k, int32_t E, lrm_quota_kind kind,
                           int32_t num, int32_t den, int32_t cap, const int32_t* explicit_quotas, int32_t* loads,
                           int32_t* quotas, int32_t* dev_status, cudaStream_t stream) {
  LRM_NVTX_RANGE();
  lrm_status st = check_dims(T, k, E, 8, 8);
  if (st) return st;
  if ((T > 0 && !topk_idx) || !loads || !quotas) return LRM_ERR_INVALID_ARG;
  if (kind == LRM_QUOTA_RATIO) {
    if (num <= 0 || den <= 0) return LRM_ERR_INVALID_ARG;
  } else if (kind == LRM_QUOTA_CAP) {
    if (cap < 0) return LRM_ERR_INVALID_ARG;
  } else if (kind == LRM_QUOTA_EXPLICIT) {
    if (!explicit_quotas) return LRM_ERR_INVALID_ARG;
  } else {
    return LRM_ERR_INVALID_ARG;
  }
  launch_plan_quotas(topk_idx, T * k, E, (int)kind, num, den, cap, explicit_quotas, loads, quotas, dev_status, stream);
  return after_launch();
}

lrm_status lrm_score(const float* alpha, const void* g, const void* phi, int64_t T, int32_t k, int32_t H, int32_t I,
                     lrm_dtype dt, float* scores, int32_t* dev_status, cudaStream_t stream) {
  LRM_NVTX_RANGE();
  lrm_status st = check_dims(T, k, 1, H, I);
  if (st) return st;
  if ((st = check_dt(dt))) return st;
  if (T > 0 && (!alpha || !g || !phi || !scores)) return LRM_ERR_INVALID_ARG;
  if (!al16(g) || !al16(phi)) return LRM_ERR_INVALID_ARG;
  launch_score(alpha, g, phi, T, k, H, I, dt, scores, dev_status, stream);
  return after_launch();
}

lrm_status lrm_score_norms(const float* alpha, const void* g, const float* phi_sq, int64_t T, int32_t k, int32_t H,
                           lrm_dtype dt, float* scores, int32_t* dev_status, cudaStream_t stream) {
  LRM_NVTX_RANGE();
  lrm_status st = check_dims(T, k, 1, H, 8);
  if (st) return st;
  if ((st = check_dt(dt))) return st;
  if (T > 0 && (!alpha || !g || !phi_sq || !scores)) return LRM_ERR_INVALID_ARG;
  if (!al16(g)) return LRM_ERR_INVALID_ARG;
  launch_score_norms(alpha, g, phi_sq, T, k, H, dt, scores, dev_status, stream);
  return after_launch();
}

lrm_status lrm_route(const float* logits, int64_t T, int32_t E, int32_t k, lrm_quota_kind kind, int32_t num,
                     int32_t den, int32_t cap, const int32_t* explicit_quotas, int32_t* topk_idx, float* alpha,
                     int32_t* loads, int32_t* quotas, void* ws, size_t ws_bytes, int32_t* dev_status,
                     cudaStream_t stream) {
  LRM_NVTX_RANGE();
  lrm_status st = check_dims(T, k, E, 8, 8);
  if (st) return st;
  if (k > E) return LRM_ERR_SHAPE;
  if (!loads || !quotas) return LRM_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !topk_idx || !alpha)) return LRM_ERR_INVALID_ARG;
  if (kind == LRM_QUOTA_RATIO) {
    if (num <= 0 || den <= 0) return LRM_ERR_INVALID_ARG;
  } else if (kind == LRM_QUOTA_CAP) {
    if (cap < 0) return LRM_ERR_INVALID_ARG;
  } else if (kind == LRM_QUOTA_EXPLICIT) {
    if (!explicit_quotas) return LRM_ERR_INVALID_ARG;
  } else {
    return LRM_ERR_INVALID_ARG;
  }
  if (!ws || ws_bytes < sizeof(uint32_t) * (E + 1) || (reinterpret_cast<uintptr_t>(ws) & 3u)) return LRM_ERR_WORKSPACE;
  return launch_route(logits, T, E, k, (int)kind, num, den, cap, explicit_quotas, topk_idx, alpha, loads, quotas,
                      static_cast<uint32_t*>(ws), dev_status, stream);
}

lrm_status lrm_swiglu_forward(const void* h, int64_t P, int32_t I, lrm_dtype dt, void* phi, float* phi_sq,
                              cudaStream_t stream) {
  LRM_NVTX_RANGE();
  lrm_status st = check_dims(P, 1, 1, 8, I);
  if (st) return st;
  if ((st = check_dt(dt))) return st;
  if (P > 0 && (!h || !phi)) return LRM_ERR_INVALID_ARG;
  if (!al16(h) || !al16(phi)) return LRM_ERR_INVALID_ARG;
  launch_swiglu_forward(h, P, I, dt, phi, phi_sq, stream);
  return after_launch();
}

lrm_status lrm_score_mode(const float* alpha, const void* g, const void* phi, int64_t T, int32_t k, int32_t H,
                          int32_t I, lrm_dtype dt, lrm_score_kind mode, float* scores, int32_t* dev_status,
                          cudaStream_t stream) {
  LRM_NVTX_RANGE();
  if (mode == LRM_SCORE_LRM) return lrm_score(alpha, g, phi, T, k, H, I, dt, scores, dev_status, stream);
  if (mode != LRM_SCORE_GRAD_SQ && mode != LRM_SCORE_GRAD_ABS) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(T, k, 1, H, 8);
  if (st) return st;
  if ((st = check_dt(dt))) return st;
  if (T > 0 && (!g || !scores)) return LRM_ERR_INVALID_ARG;
  if (!al16(g)) return LRM_ERR_INVALID_ARG;
  launch_grad_score(g, T, k, H, dt, mode == LRM_SCORE_GRAD_ABS, scores, dev_status, stream);
  return after_launch();
}

lrm_status lrm_select(const int32_t* topk_idx, const float* scores, const int32_t* quotas, int64_t T, int32_t k,
                      int32_t E, int64_t cap, int32_t* seg_offsets, int32_t* kept_pair, int32_t* row_of_pair,
                      void* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  LRM_NVTX_RANGE();
  lrm_status st = check_dims(T, k, E, 8, 8);
  if (st) return st;
  const int64_t P = T * k;
  if (cap < 0 || cap > INT32_MAX) return LRM_ERR_INVALID_ARG;
  if (!quotas || !seg_offsets) return LRM_ERR_INVALID_ARG;
  if (P > 0 && (!topk_idx || !scores || !row_of_pair)) return LRM_ERR_INVALID_ARG;
  if (cap > 0 && !kept_pair) return LRM_ERR_INVALID_ARG;
  const WsLayout w = workspace_layout(P, E);
  if (!ws || ws_bytes < w.total) return LRM_ERR_WORKSPACE;
  char* b = static_cast<char*>(ws);
  SelectWs sw;
  sw.counts = reinterpret_cast<int32_t*>(b + w.counts);
  sw.bucket_start = reinterpret_cast<int32_t*>(b + w.bucket_start);
  sw.keep = reinterpret_cast<int32_t*>(b + w.keep);
  sw.loads = reinterpret_cast<int32_t*>(b + w.loads);
  sw.sorted_u = reinterpret_cast<int32_t*>(b + w.sorted_u);
  sw.sorted_key = reinterpret_cast<uint32_t*>(b + w.sorted_key);
  sw.n_chunks = (P + kSelChunk - 1) / kSelChunk;
  launch_select(topk_idx, scores, quotas, P, E, cap, seg_offsets, kept_pair, row_of_pair, sw, dev_status, stream);
  return after_launch();
}

lrm_status lrm_compact(const int32_t* row_of_pair, const float* alpha, const void* g, const void* x, const void* h,
                       const void* phi, int64_t T, int32_t k, int32_t H, int32_t I, lrm_dtype dt, int64_t cap,
                       void* dy_c, void* x_c, void* h_c, void* phi_c, int32_t* dev_status, cudaStream_t stream) {
  LRM_NVTX_RANGE();
  lrm_status st = check_dims(T, k, 1, H, I);
  if (st) return st;
  if ((st = check_dt(dt))) return st;
  if (cap < 0 || cap > INT32_MAX) return LRM_ERR_INVALID_ARG;
  // x_c, h_c, phi_c all NULL: the compaction-free variant (only dy_c is written); h_c and phi_c
  // NULL with x_c given: the variant that recomputes h and phi from x_c (dy_c and x_c written)
  const bool want_x = x_c != nullptr, want_h = h_c != nullptr || phi_c != nullptr;
  if (want_h && (!want_x || !h_c || !phi_c)) return LRM_ERR_INVALID_ARG;
  if (T > 0 && (!row_of_pair || !alpha || !g)) return LRM_ERR_INVALID_ARG;
  if (T > 0 && want_x && !x) return LRM_ERR_INVALID_ARG;
  if (T > 0 && want_h && (!h || !phi)) return LRM_ERR_INVALID_ARG;
  if (cap > 0 && !dy_c) return LRM_ERR_INVALID_ARG;
  const void* ptrs[] = {g, x, h, phi, dy_c, x_c, h_c, phi_c};
  for (const void* p : ptrs)
    if (!al16(p)) return LRM_ERR_INVALID_ARG;
  launch_compact(row_of_pair, alpha, g, x, h, phi, T, k, H, I, dt, cap, dy_c, x_c, h_c, phi_c, dev_status, stream);
  return after_launch();
}

}  // extern "C"

namespace {

// Shared by both grouped-backward entry points: validation, workspace carving, dispatch.
lrm_status grouped_impl(GroupedArgs a, lrm_dtype dt, void* ws, size_t ws_bytes, int32_t flags,
                        cudaStream_t stream) {
  const int32_t E = a.E, H = a.H, I = a.I;
  const int64_t cap = a.cap;
  lrm_status st = check_dims(0, 1, E, H, I);
  if (st) return st;
  if ((st = check_dt(dt))) return st;
  if (cap < 0 || cap > INT32_MAX) return LRM_ERR_INVALID_ARG;
  if (flags != LRM_GEMM_DEFAULT && flags != LRM_GEMM_FORCE_SIMT) return LRM_ERR_INVALID_ARG;
  if (!a.seg_offsets || !a.w_gate_up || !a.w_down || !a.dw_gate_up || !a.dw_down) return LRM_ERR_INVALID_ARG;
  const bool gather = a.kept_pair != nullptr;
  if (cap > 0 && (!a.dy_c || !a.dh_c || !a.dx_c)) return LRM_ERR_INVALID_ARG;
  if (cap > 0 && !gather && (!a.x_c || !a.h_c || !a.phi_c)) return LRM_ERR_INVALID_ARG;
  if (cap > 0 && gather && (!a.x || !a.h || !a.phi || a.k < 1 || a.k > LRM_MAX_TOPK)) return LRM_ERR_INVALID_ARG;
  const void* ptrs[] = {a.dy_c, a.x_c, a.h_c, a.phi_c, a.w_gate_up, a.w_down, a.dw_gate_up, a.dw_down, a.dh_c,
                        a.dx_c, a.x, a.h, a.phi};
  for (const void* p : ptrs)
    if (!al16(p)) return LRM_ERR_INVALID_ARG;
  if (a.row_dot && (reinterpret_cast<uintptr_t>(a.row_dot) & 3u)) return LRM_ERR_INVALID_ARG;
  if (!ws || ws_bytes < grouped_ws_bytes(cap, E, I, a.row_dot != nullptr)) return LRM_ERR_WORKSPACE;
  if (cap == 0) {  // no rows anywhere (seg_offsets[E] <= cap): every dW is exactly zero
    if (cudaMemsetAsync(a.dw_gate_up, 0, sizeof(float) * (size_t)E * 2 * I * H, stream) != cudaSuccess ||
        cudaMemsetAsync(a.dw_down, 0, sizeof(float) * (size_t)E * H * I, stream) != cudaSuccess)
      return LRM_ERR_CUDA;
    return LRM_OK;
  }
  a.dot_part = a.row_dot ? reinterpret_cast<float*>(static_cast<char*>(ws) + up(gemm_ws_bytes(E))) : nullptr;
  if (dt == LRM_BF16 && flags == LRM_GEMM_DEFAULT) {
    // workspace: tile tables and per-expert tensor maps at the start of ws
    GemmWs gw;
    gw.plan = static_cast<int32_t*>(ws);
    gw.maps = static_cast<char*>(ws) + gemm_plan_bytes(E);
    return launch_grouped_tc(a, gw, stream);
  }
  launch_grouped_simt(a, dt, stream);
  return after_launch();
}

}  // namespace

extern "C" {

lrm_status lrm_grouped_backward(const int32_t* seg_offsets, const void* dy_c, const void* x_c, const void* h_c,
                                const void* phi_c, const void* w_gate_up, const void* w_down, int32_t E, int32_t H,
                                int32_t I, lrm_dtype dt, int64_t cap, float* dw_gate_up, float* dw_down, void* dh_c,
                                void* dx_c, float* row_dot, void* ws, size_t ws_bytes, int32_t flags,
                                int32_t* dev_status, cudaStream_t stream) {
  LRM_NVTX_RANGE();
  GroupedArgs a{seg_offsets, dy_c, x_c, h_c, phi_c, w_gate_up, w_down, E, H, I, cap, dw_gate_up, dw_down,
                dh_c, dx_c, dev_status, row_dot, nullptr, nullptr, 0, nullptr, nullptr, nullptr, 0};
  return grouped_impl(a, dt, ws, ws_bytes, flags, stream);
}

lrm_status lrm_grouped_backward_gather(const int32_t* seg_offsets, const int32_t* kept_pair, int64_t T, int32_t k,
                                       const void* dy_c, const void* x, const void* h, const void* phi,
                                       const void* w_gate_up, const void* w_down, int32_t E, int32_t H, int32_t I,
                                       lrm_dtype dt, int64_t cap, float* dw_gate_up, float* dw_down, void* dh_c,
                                       void* dx_c, float* row_dot, void* ws, size_t ws_bytes, int32_t flags,
                                       int32_t* dev_status, cudaStream_t stream) {
  LRM_NVTX_RANGE();
  if (cap > 0 && !kept_pair) return LRM_ERR_INVALID_ARG;
  if (T < 0 || k < 1 || k > LRM_MAX_TOPK) return LRM_ERR_INVALID_ARG;
  if (T > INT32_MAX / k) return LRM_ERR_SHAPE;
  GroupedArgs a{seg_offsets, dy_c, nullptr, nullptr, nullptr, w_gate_up, w_down, E, H, I, cap, dw_gate_up,
                dw_down, dh_c, dx_c, dev_status, row_dot, nullptr, kept_pair, k, x, h, phi, T * k};
  return grouped_impl(a, dt, ws, ws_bytes, flags, stream);
}

lrm_status lrm_recompute_forward(const int32_t* seg_offsets, const void* x_c, const void* w_gate_up, int32_t E,
                                 int32_t H, int32_t I, lrm_dtype dt, int64_t cap, void* h_c, void* phi_c, void* ws,
                                 size_t ws_bytes, int32_t flags, int32_t* dev_status, cudaStream_t stream) {
  LRM_NVTX_RANGE();
  lrm_status st = check_dims(0, 1, E, H, I);
  if (st) return st;
  if ((st = check_dt(dt))) return st;
  if (cap < 0 || cap > INT32_MAX) return LRM_ERR_INVALID_ARG;
  if (flags != LRM_GEMM_DEFAULT && flags != LRM_GEMM_FORCE_SIMT) return LRM_ERR_INVALID_ARG;
  if (!seg_offsets || !w_gate_up) return LRM_ERR_INVALID_ARG;
  if (cap > 0 && (!x_c || !h_c || !phi_c)) return LRM_ERR_INVALID_ARG;
  const void* ptrs[] = {x_c, w_gate_up, h_c, phi_c};
  for (const void* p : ptrs)
    if (!al16(p)) return LRM_ERR_INVALID_ARG;
  if (!ws || ws_bytes < up(gemm_ws_bytes(E))) return LRM_ERR_WORKSPACE;
  if (cap == 0) return LRM_OK;  // no rows to recompute
  RecomputeArgs a{seg_offsets, x_c, w_gate_up, E, H, I, cap, h_c, phi_c, dev_status};
  if (dt == LRM_BF16 && flags == LRM_GEMM_DEFAULT) {
    GemmWs gw;
    gw.plan = static_cast<int32_t*>(ws);
    gw.maps = static_cast<char*>(ws) + gemm_plan_bytes(E);
    return launch_recompute_tc(a, gw, stream);
  }
  launch_recompute_simt(a, dt, stream);
  return after_launch();
}

lrm_status lrm_scatter_dx(const int32_t* row_of_pair, const void* dx_c, int64_t T, int32_t k, int32_t H,
                          lrm_dtype dt, int64_t cap, void* dx, int32_t* dev_status, cudaStream_t stream) {
  LRM_NVTX_RANGE();
  lrm_status st = check_dims(T, k, 1, H, 8);
  if (st) return st;
  if ((st = check_dt(dt))) return st;
  if (cap < 0 || cap > INT32_MAX) return LRM_ERR_INVALID_ARG;
  if (T > 0 && (!row_of_pair || !dx)) return LRM_ERR_INVALID_ARG;
  if (T > 0 && cap > 0 && !dx_c) return LRM_ERR_INVALID_ARG;
  if (!al16(dx_c) || !al16(dx)) return LRM_ERR_INVALID_ARG;
  launch_scatter_dx(row_of_pair, dx_c, T, k, H, dt, cap, dx, dev_status, stream);
  return after_launch();
}

lrm_status lrm_router_grad(const int32_t* row_of_pair, const float* alpha, const float* row_dot, int64_t T,
                           int32_t k, int64_t cap, float* dalpha, cudaStream_t stream) {
  LRM_NVTX_RANGE();
  lrm_status st = check_dims(T, k, 1, 8, 8);
  if (st) return st;
  if (cap < 0 || cap > INT32_MAX) return LRM_ERR_INVALID_ARG;
  if (T > 0 && (!row_of_pair || !alpha || !dalpha)) return LRM_ERR_INVALID_ARG;
  if (T > 0 && cap > 0 && !row_dot) return LRM_ERR_INVALID_ARG;
  launch_router_grad(row_of_pair, alpha, row_dot, T * k, cap, dalpha, stream);
  return after_launch();
}

lrm_status lrm_selftest_wait_timeout(int32_t* dev_status, int64_t limit_ns, cudaStream_t stream) {
  LRM_NVTX_RANGE();
  if (!dev_status || limit_ns <= 0 || limit_ns > 10000000000ll) return LRM_ERR_INVALID_ARG;
  return launch_wait_selftest(dev_status, limit_ns, stream);
}

}  // extern "C"
