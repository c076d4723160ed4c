// Internal launchers of the LRM-pruned expert backward kernels.  abi.cu validates the
// arguments of the public entry points and calls these; they only launch.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "lrm.h"

namespace lrm {

// Selection works on chunks of this many consecutive pairs (one CTA, one pair per thread).
constexpr int kSelChunk = 256;

struct SelectWs {
  int32_t* counts;        // [n_chunks][E]  per-chunk expert counts, then exclusive bases
  int32_t* bucket_start;  // [E+1]          start of each expert's bucket in sorted_u
  int32_t* keep;          // [E]            min(max(quota,0), load), or 0 on capacity overflow
  int32_t* loads;         // [E]            pairs routed to each expert
  int32_t* sorted_u;      // [P]            pairs grouped by expert, u ascending
  uint32_t* sorted_key;   // [P]            score bits in the same order
  int64_t n_chunks;
};

// Scratch of the tensor-core grouped GEMMs: tile tables, then 6*E per-expert TMA tensor maps
// (128 bytes each, 128-byte aligned) built on the device from seg_offsets.
struct GemmWs {
  int32_t* plan;  // [2E+3+kTileCounters]
  void* maps;     // [6][E] CUtensorMap
};
// var-K launches of one grouped call whose tile counters sit in the plan region
constexpr int kTileCounters = 2;
size_t gemm_plan_bytes(int32_t E);  // plan[2E+3+kTileCounters]: tile tables, checks, tile counters
size_t gemm_ws_bytes(int32_t E);

struct WsLayout {
  size_t counts, bucket_start, keep, loads, sorted_u, sorted_key, gemm, total;
};
WsLayout workspace_layout(int64_t P, int32_t E);

void launch_plan_quotas(const int32_t* topk_idx, int64_t P, int32_t E, int kind, int32_t num, int32_t den,
                        int32_t cap, const int32_t* explicit_q, int32_t* loads, int32_t* quotas, int32_t* status,
                        cudaStream_t s);

void launch_score(const float* alpha, const void* g, const void* phi, int64_t T, int32_t k, int32_t H, int32_t I,
                  lrm_dtype dt, float* scores, int32_t* status, cudaStream_t s);

void launch_score_norms(const float* alpha, const void* g, const float* phi_sq, int64_t T, int32_t k, int32_t H,
                        lrm_dtype dt, float* scores, int32_t* status, cudaStream_t s);

lrm_status launch_route(const float* logits, int64_t T, int32_t E, int32_t k, int kind, int32_t num, int32_t den,
                        int32_t cap, const int32_t* explicit_q, int32_t* topk_idx, float* alpha, int32_t* loads,
                        int32_t* quotas, uint32_t* done, int32_t* status, cudaStream_t s);

void launch_swiglu_forward(const void* h, int64_t P, int32_t I, lrm_dtype dt, void* phi, float* phi_sq,
                           cudaStream_t s);

void launch_grad_score(const void* g, int64_t T, int32_t k, int32_t H, lrm_dtype dt, bool abs_mode, float* scores,
                       int32_t* status, cudaStream_t s);

void launch_select(const int32_t* topk_idx, const float* scores, const int32_t* quotas, int64_t P, int32_t E,
                   int64_t cap, int32_t* seg_offsets, int32_t* kept_pair, int32_t* row_of_pair, const SelectWs& ws,
                   int32_t* status, cudaStream_t s);

void launch_compact(const int32_t* row_of_pair, const float* alpha, const void* g, const void* x, const void* h,
                    const void* phi, int64_t T, int32_t k, int32_t H, int32_t I, lrm_dtype dt, int64_t cap,
                    void* dy_c, void* x_c, void* h_c, void* phi_c, int32_t* status, cudaStream_t s);

void launch_scatter_dx(const int32_t* row_of_pair, const void* dx_c, int64_t T, int32_t k, int32_t H, lrm_dtype dt,
                       int64_t cap, void* dx, int32_t* status, cudaStream_t s);

struct GroupedArgs {
  const int32_t* seg_offsets;
  const void *dy_c, *x_c, *h_c, *phi_c, *w_gate_up, *w_down;
  int32_t E, H, I;
  int64_t cap;
  float *dw_gate_up, *dw_down;
  void *dh_c, *dx_c;
  int32_t* status;
  float* row_dot;   // optional [cap]: dphi . phi per retained row
  float* dot_part;  // scratch for row_dot: [cap][dot_parts_max(I)]
  // Compaction-free variant (kept_pair non-null): x_c, h_c, phi_c are not used; their rows are
  // read from x [T,H] (token u / k), h [P,2I] and phi [P,I] (pair u = kept_pair[r]).
  const int32_t* kept_pair;
  int32_t k;
  const void *x, *h, *phi;
  int64_t n_pairs;  // T*k: rows of h and phi; a kept_pair entry outside [0, n_pairs) is not followed
};

// Parts of the dphi . phi row sums: one per 128 output columns (tensor-core path) or per 64
// (CUDA-core path); scratch is sized for the larger count.
inline int dot_parts_max(int32_t I) { return (I + 63) / 64; }
void launch_row_dot(const float* part, int n_part, const int32_t* seg_offsets, int32_t E, int64_t cap,
                    float* row_dot, cudaStream_t s);
void launch_router_grad(const int32_t* row_of_pair, const float* alpha, const float* row_dot, int64_t P,
                        int64_t cap, float* dalpha, cudaStream_t s);

void launch_grouped_simt(const GroupedArgs& a, lrm_dtype dt, cudaStream_t s);

// The saved forward state of the retained rows, recomputed from x_c (lrm_recompute_forward).
struct RecomputeArgs {
  const int32_t* seg_offsets;
  const void *x_c, *w_gate_up;
  int32_t E, H, I;
  int64_t cap;
  void *h_c, *phi_c;
  int32_t* status;
};
lrm_status launch_recompute_tc(const RecomputeArgs& a, const GemmWs& ws, cudaStream_t s);
void launch_recompute_simt(const RecomputeArgs& a, lrm_dtype dt, cudaStream_t s);
// Returns LRM_OK, or LRM_ERR_UNSUPPORTED / LRM_ERR_CUDA when the tensor-core path cannot run.
lrm_status launch_grouped_tc(const GroupedArgs& a, const GemmWs& ws, cudaStream_t s);
lrm_status launch_wait_selftest(int32_t* status, int64_t limit_ns, cudaStream_t s);

}  // namespace lrm
