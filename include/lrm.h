/*
 * lrm.h — C ABI of the LRM-pruned MoE expert backward on one GPU (sm_103a).
 *
 * The operation is the expert-layer backward of LRMoE, as described in
 *   "LRMoE: Trimming Backward Work in Memory-Bound MoE Training" (aimodeling.com), sections
 *   "Backward demand is not a constant", "LRM: a decomposable contribution score" and
 *   "The part that is easy to get wrong", and in the five-step list of
 *   "LRMoE poda a passagem reversa do MoE e acelera o treinamento em 21–45%" (news.hamidun.com),
 *   section "O que o LRMoE faz: forward completo, backward podado":
 *     quotas -> LRM score -> keep each expert's top-quota pairs -> physical compaction ->
 *     variable-size grouped GEMMs -> result back to the original layout.
 *
 * Notation.  T tokens, k routed experts per token, P = T*k pairs, pair u = t*k + j
 * (token-major), E experts, H hidden, I expert intermediate, R_e retained rows of expert e,
 * R = sum_e R_e.  The expert is a SwiGLU MLP: h_u = W_gate_up[e] x_t = [gate_u; up_u] (2I),
 * phi_u = SiLU(gate_u) * up_u (I), output alpha_u W_down[e] phi_u; g_t (H) is the upstream
 * gradient of the layer output.
 *
 * Conventions shared by every entry point.
 *  - Every call is asynchronous on the caller's stream (NULL = legacy default stream). The
 *    library never allocates, frees or synchronises; a call returns after its launches are
 *    queued.
 *  - Every pointer argument is caller-owned DEVICE memory unless stated otherwise, aligned
 *    to 16 bytes, and must stay valid until the stream work completes.  The library keeps
 *    no pointer after a call returns.
 *  - Row-major, densely packed tensors.  lrm_dtype fixes the element type of g, x, h, phi,
 *    the weights, the compacted buffers and dX; alpha and scores are always fp32, indices
 *    are int32, weight gradients are always fp32.
 *  - Host-detected errors are returned (nothing is launched, outputs are untouched).
 *    Device-detected errors are written to the optional `dev_status` word (int32, device
 *    memory, caller zeroes it): the first error code wins (atomic compare-and-swap from 0).
 *    The caller reads it whenever it chooses; the library never does.
 *  - Limits: 1 <= E <= LRM_MAX_EXPERTS, 1 <= k <= LRM_MAX_TOPK, P <= INT32_MAX (checked
 *    without forming an overflowing product), H and I positive multiples of 8.
 *  - Index arrays handed from one call to the next (row_of_pair, seg_offsets) are checked
 *    where they are used: an index outside its range is never followed; the pair (or the
 *    whole grouped backward) is skipped and the status word records why.  A build with
 *    -DLRM_DEBUG (liblrm_debug.so) adds the same kind of check to every index the kernels
 *    form themselves (bucket slots, compacted rows of a tile, gathered pair rows); a failed
 *    check records LRM_ERR_BAD_INDEX and skips the access, it never traps.
 *  - Each entry point opens an NVTX range of its own name around its host work when the
 *    environment variable LRM_NVTX is 1 at the library's first call (off otherwise).
 *  - The kernels of lrm_score, lrm_select, lrm_select_static, lrm_compact,
 *    lrm_grouped_backward (tensor-core path) and lrm_scatter_dx use programmatic dependent launch: each waits (griddepcontrol.wait) for the
 *    work queued before it on the stream to complete before it touches memory, and lets the
 *    next launch on the stream start early.  Ordinary stream order therefore holds for every
 *    caller; a caller kernel that is itself launched with programmatic stream serialization
 *    right after one of these calls must execute griddepcontrol.wait (or
 *    cudaGridDependencySynchronize) before it reads their outputs.
 */
#ifndef LRM_H
#define LRM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LRM_MAX_EXPERTS 1024
#define LRM_MAX_TOPK 16

typedef enum lrm_status {
  LRM_OK = 0,
  LRM_ERR_INVALID_ARG = 1, /* null pointer, misaligned pointer, negative size, bad enum   */
  LRM_ERR_SHAPE = 2,       /* a size outside the limits above                           */
  LRM_ERR_DTYPE = 3,       /* unknown lrm_dtype                                         */
  LRM_ERR_WORKSPACE = 4,   /* workspace null or smaller than lrm_workspace_size         */
  LRM_ERR_CUDA = 5,        /* a CUDA launch/runtime call failed                         */
  LRM_ERR_CAPACITY = 6,    /* device: sum of kept rows exceeds `cap` (nothing is kept)  */
  LRM_ERR_NONFINITE = 7,   /* device: a score is NaN or infinite                        */
  LRM_ERR_TIMEOUT = 8,     /* device: a bounded wait gave up                            */
  LRM_ERR_BAD_INDEX = 9,   /* device: an expert id outside [0, E), or a compacted row
                              outside [-1, cap) (the pair is treated as dropped)        */
  LRM_ERR_UNSUPPORTED = 10, /* no kernel for this device / configuration                */
  LRM_ERR_BAD_SEGMENTS = 11 /* device: seg_offsets[0] != 0, a decreasing step, or
                              seg_offsets[E] > cap (the grouped backward computes nothing) */
} lrm_status;

typedef enum lrm_dtype { LRM_BF16 = 0, LRM_F32 = 1 } lrm_dtype;

typedef enum lrm_quota_kind {
  LRM_QUOTA_RATIO = 0,    /* quota_e = ceil(num/den * load_e), exact integer arithmetic   */
  LRM_QUOTA_CAP = 1,      /* quota_e = min(load_e, cap)                                   */
  LRM_QUOTA_EXPLICIT = 2  /* quota_e = explicit_quotas[e] (copied)                        */
} lrm_quota_kind;

/* Flags of lrm_grouped_backward. */
#define LRM_GEMM_DEFAULT 0     /* tcgen05 tensor-core kernels for bf16, SIMT fp32 kernels for fp32 */
#define LRM_GEMM_FORCE_SIMT 1  /* CUDA-core kernels for bf16 too (fp32 accumulation)               */

/* Text for a status code (static storage, never NULL). */
const char* lrm_status_string(lrm_status s);

/*
 * Bytes of scratch `ws` that lrm_select and lrm_grouped_backward need for these sizes (one
 * buffer serves both; calls on one stream may share it).  Writes *bytes.  Host-only, no GPU
 * work.  Errors: LRM_ERR_INVALID_ARG (bytes NULL, negative size), LRM_ERR_SHAPE, LRM_ERR_DTYPE.
 */
lrm_status lrm_workspace_size(int64_t T, int32_t k, int32_t E, int32_t H, int32_t I, lrm_dtype dt,
                              size_t* bytes);

/*
 * Per-expert loads and backward retention quotas, fixed before the expert forward and
 * constant for the layer call ("Backward demand is not a constant"; the Portuguese list's
 * second step).  The articles' controller derives them from memory and network state; this
 * entry point applies one of the fixed rules of lrm_quota_kind.
 *   topk_idx [T*k] int32    expert id of each pair (ids outside [0,E) are counted nowhere and
 *                           set LRM_ERR_BAD_INDEX in dev_status)
 *   explicit_quotas [E]     int32, read only for LRM_QUOTA_EXPLICIT (may be NULL otherwise)
 *   loads [E], quotas [E]   int32 outputs
 * num > 0, den > 0 for RATIO; cap >= 0 for CAP.  Launches a memset and two small kernels.
 */
lrm_status lrm_plan_quotas(const int32_t* topk_idx, int64_t T, int32_t k, int32_t E, lrm_quota_kind kind,
                           int32_t num, int32_t den, int32_t cap, const int32_t* explicit_quotas,
                           int32_t* loads, int32_t* quotas, int32_t* dev_status, cudaStream_t stream);

/*
 * LRM score of every pair ("LRM: a decomposable contribution score"):
 *   R_u = alpha_u^2 * ||g_t||_2^2 * ||phi_u||_2^2  (= ||(alpha_u g_t) phi_u^T||_F^2),
 * accumulated and returned in fp32.
 *   alpha [T*k] fp32, g [T,H] dt, phi [T*k, I] dt  ->  scores [T*k] fp32.
 * A non-finite score sets LRM_ERR_NONFINITE in dev_status (the score is still written).
 */
lrm_status lrm_score(const float* alpha, const void* g, const void* phi, int64_t T, int32_t k, int32_t H,
                     int32_t I, lrm_dtype dt, float* scores, int32_t* dev_status, cudaStream_t stream);

/* Scores for the selection ablations of "LRMoE: Trimming Backward Work in Memory-Bound MoE
 * Training", section "What the measurements show". */
typedef enum lrm_score_kind {
  LRM_SCORE_LRM = 0,      /* alpha_u^2 * ||g_t||_2^2 * ||phi_u||_2^2 (lrm_score)                  */
  LRM_SCORE_GRAD_SQ = 1,  /* squared gradient norm ||g_t||_2^2 (every pair of token t alike)     */
  LRM_SCORE_GRAD_ABS = 2  /* absolute gradient magnitude ||g_t||_1 = sum_h |g_t[h]|              */
} lrm_score_kind;

/*
 * Score of every pair under one of the lrm_score_kind rules, fp32 accumulation.  The gradient-
 * only rules read g alone (alpha and phi may be NULL) and give the k pairs of a token the same
 * score, so lrm_select falls back to its pair-index tie-break inside a token.  Random dropping,
 * the pages' third ablation, is lrm_select on caller-drawn uniform scores.  Layouts, errors and
 * the non-finite flag as for lrm_score.
 */
lrm_status lrm_score_mode(const float* alpha, const void* g, const void* phi, int64_t T, int32_t k, int32_t H,
                          int32_t I, lrm_dtype dt, lrm_score_kind mode, float* scores, int32_t* dev_status,
                          cudaStream_t stream);

/*
 * Keep each expert's top-quota pairs (Portuguese list, step "Seleção pela métrica LRM": inside
 * the quota the highest-scoring pairs stay).  Expert e keeps min(max(quota_e,0), load_e) pairs:
 * largest score first, equal scores to the smaller pair index u.
 *   topk_idx [T*k] int32, scores [T*k] fp32 (finite, >= 0), quotas [E] int32
 *   seg_offsets [E+1] int32   out: exclusive prefix sum of kept counts (segment e = rows
 *                             seg_offsets[e] .. seg_offsets[e+1]-1)
 *   kept_pair [cap] int32     out: kept pair indices, expert-major, u ascending in a segment
 *   row_of_pair [T*k] int32   out: compacted row of each pair, -1 if dropped
 *   cap                       rows available in kept_pair (and in the compacted buffers later);
 *                             if the kept total exceeds it, LRM_ERR_CAPACITY is set and nothing
 *                             is kept (seg_offsets all 0, row_of_pair all -1).  cap = T*k
 *                             always suffices.
 *   ws, ws_bytes              scratch of at least lrm_workspace_size bytes
 * Deterministic: the output does not depend on scheduling.
 */
lrm_status lrm_select(const int32_t* topk_idx, const float* scores, const int32_t* quotas, int64_t T,
                      int32_t k, int32_t E, int64_t cap, int32_t* seg_offsets, int32_t* kept_pair,
                      int32_t* row_of_pair, void* ws, size_t ws_bytes, int32_t* dev_status,
                      cudaStream_t stream);

/*
 * Physical compaction ("The part that is easy to get wrong": retained gradient rows and their
 * saved activations repacked into contiguous expert-specific buffers, no padding).  For every
 * kept pair u = t*k + j with r = row_of_pair[u] >= 0:
 *   dy_c[r] = round_dt(alpha_u * g_t)   (fp32 product, round to nearest even)
 *   x_c[r] = x_t,   h_c[r] = h_u,   phi_c[r] = phi_u
 *   row_of_pair [T*k] int32 (from lrm_select), alpha [T*k] fp32, g [T,H], x [T,H],
 *   h [T*k, 2I], phi [T*k, I]  ->  dy_c [cap,H], x_c [cap,H], h_c [cap,2I], phi_c [cap,I] (dt).
 * Rows are visited token by token, so g_t and x_t are read once per token.  A row_of_pair
 * entry outside [-1, cap) is not followed: the pair is skipped and LRM_ERR_BAD_INDEX is set in
 * dev_status.  With x_c, h_c and phi_c all NULL only dy_c is written (x, h, phi may then be
 * NULL): the compaction-free variant, whose grouped backward reads those rows in place
 * (lrm_grouped_backward_gather).  With h_c and phi_c NULL and x_c given, dy_c and x_c are
 * written (h and phi may be NULL): the variant whose forward did not keep h and phi, which
 * lrm_recompute_forward then rebuilds for the retained rows.
 */
lrm_status lrm_compact(const int32_t* row_of_pair, const float* alpha, const void* g, const void* x,
                       const void* h, const void* phi, int64_t T, int32_t k, int32_t H, int32_t I,
                       lrm_dtype dt, int64_t cap, void* dy_c, void* x_c, void* h_c, void* phi_c,
                       int32_t* dev_status, cudaStream_t stream);

/*
 * SwiGLU expert backward as variable-size grouped GEMMs driven by the retained row counts
 * ("The part that is easy to get wrong"; the Portuguese list's compaction step).  For each
 * expert e over its segment (R_e rows, read on the device from seg_offsets; no host sync):
 *   dw_down[e]    = dy_c[e]^T phi_c[e]                               [E,H,I]  fp32, overwritten
 *   dphi          = dy_c[e] w_down[e]; s = sigmoid(gate)
 *   dh_c[e]       = [dphi*up*s*(1+gate*(1-s)) ; dphi*gate*s]         [cap,2I] dt
 *   dw_gate_up[e] = dh_c[e]^T x_c[e]                                 [E,2I,H] fp32, overwritten
 *   dx_c[e]       = dh_c[e] w_gate_up[e]                             [cap,H]  dt
 * An expert with R_e = 0 gets dw = 0 exactly.  w_gate_up [E,2I,H] (gate rows first),
 * w_down [E,H,I].  Accumulation is fp32.  `flags` is LRM_GEMM_DEFAULT or LRM_GEMM_FORCE_SIMT.
 * seg_offsets must start at 0, be non-decreasing and end at seg_offsets[E] <= cap (as lrm_select
 * writes them).  The kernels check this on the device before any tile runs: otherwise they set
 * LRM_ERR_BAD_SEGMENTS in dev_status and compute nothing (every output keeps its old contents).
 * Optional row_dot [cap] fp32 (NULL skips it; 4-byte aligned): for every retained row
 * r < seg_offsets[E], row_dot[r] = sum_i dphi[r,i] * phi~[r,i], where phi~ = SiLU(gate)*up is
 * recomputed in fp32 from h_c inside the same epilogue; for the pair u = (t, e) of row r that is
 * alpha_u * (g_t . W_down[e] phi_u), the input of lrm_router_grad.  Its parts are summed in a
 * fixed order (deterministic).  Rows >= seg_offsets[E] are not written.
 * ws, ws_bytes: scratch of at least lrm_workspace_size bytes (with row_dot it must cover `cap`
 * rows: lrm_workspace_size for T*k >= cap does).
 * Errors: host as usual; LRM_ERR_UNSUPPORTED when the tensor-core kernels are requested on a
 * device that is not sm_103; device LRM_ERR_TIMEOUT if a pipeline wait gives up (the kernel
 * then returns early and its outputs are incomplete).
 */
lrm_status lrm_grouped_backward(const int32_t* seg_offsets, const void* dy_c, const void* x_c, const void* h_c,
                                const void* phi_c, const void* w_gate_up, const void* w_down, int32_t E,
                                int32_t H, int32_t I, lrm_dtype dt, int64_t cap, float* dw_gate_up,
                                float* dw_down, void* dh_c, void* dx_c, float* row_dot, void* ws,
                                size_t ws_bytes, int32_t flags, int32_t* dev_status, cudaStream_t stream);

/*
 * Compaction-free variant of lrm_grouped_backward (measured against the materialised compaction
 * the pages insist on, "The part that is easy to get wrong"): the same products and outputs,
 * with only dy_c compacted.  The rows of x, h and phi are read where they are, through the
 * compacted-row -> pair map kept_pair from lrm_select: row r stands for pair u = kept_pair[r]
 * of token u / k.  The dW GEMMs copy their x / phi operand rows by index straight into the
 * operand tiles; the SwiGLU epilogue reads h by index.  Results are bit-identical to
 * lrm_grouped_backward on the materialised buffers (same values, same order of arithmetic).
 *   kept_pair [cap] int32, x [T,H], h [T*k,2I], phi [T*k,I] (dt); the rest as in
 *   lrm_grouped_backward.  Errors as there; a kept_pair entry outside [0, T*k) is not followed
 *   (its row reads as zeros) and sets LRM_ERR_BAD_INDEX in dev_status.
 */
lrm_status lrm_grouped_backward_gather(const int32_t* seg_offsets, const int32_t* kept_pair, int64_t T, int32_t k,
                                       const void* dy_c, const void* x, const void* h, const void* phi,
                                       const void* w_gate_up, const void* w_down, int32_t E, int32_t H, int32_t I,
                                       lrm_dtype dt, int64_t cap, float* dw_gate_up, float* dw_down, void* dh_c,
                                       void* dx_c, float* row_dot, void* ws, size_t ws_bytes, int32_t flags,
                                       int32_t* dev_status, cudaStream_t stream);

/*
 * The saved forward state of the retained rows, recomputed from their x rows (the variant of
 * "The part that is easy to get wrong" whose forward keeps x and the score's ||phi_u||^2 instead of
 * h and phi; lrm_swiglu_forward emits the norms).  For each expert e over its segment (R_e rows,
 * read on the device from seg_offsets):
 *   h_c[r]   = round_dt(W_gate_up[e] x_c[r])                     [cap,2I] dt (gate first), fp32 sums
 *   phi_c[r] = round_dt(SiLU(gate) * up), gate / up taken from the stored h_c[r]   [cap,I] dt
 * i.e. what the forward's expert projection and lrm_swiglu_forward would have stored for those
 * pairs.  x_c [cap,H], w_gate_up [E,2I,H].  Rows >= seg_offsets[E] are not written.  ws: scratch of
 * at least lrm_workspace_size bytes (shared with the other calls on the stream).  The same
 * segment check as lrm_grouped_backward (LRM_ERR_BAD_SEGMENTS: nothing computed).  flags as
 * there (fp32 inputs, or LRM_GEMM_FORCE_SIMT, run on the CUDA cores).
 */
lrm_status lrm_recompute_forward(const int32_t* seg_offsets, const void* x_c, const void* w_gate_up, int32_t E,
                                 int32_t H, int32_t I, lrm_dtype dt, int64_t cap, void* h_c, void* phi_c, void* ws,
                                 size_t ws_bytes, int32_t flags, int32_t* dev_status, cudaStream_t stream);

/*
 * Routing-weight gradient of the pairs.  The layer output is out_t = sum_j alpha_{t,j} y_{t,j}
 * with y_u = W_down[e_u] phi_u (the expert output), so dL/dalpha_u = g_t . y_u.  The LRMoE
 * pages say nothing about it under pruning; here a dropped pair, removed from the whole expert
 * backward ("The part that is easy to get wrong": only retained rows are packed and computed),
 * gets 0, and a retained pair the exact value:
 *   r = row_of_pair[u];  dalpha[u] = (0 <= r < cap) ? row_dot[r] / alpha_u : 0
 * with row_dot from lrm_grouped_backward.  Where alpha_u == 0 the alpha-scaled rows carry no
 * trace of g_t . y_u and dalpha[u] = 0.
 *   row_of_pair [T*k] int32, alpha [T*k] fp32, row_dot [cap] fp32  ->  dalpha [T*k] fp32.
 * Errors: LRM_ERR_INVALID_ARG (NULL pointer, cap outside [0, INT32_MAX]), LRM_ERR_SHAPE,
 * LRM_ERR_CUDA.
 */
lrm_status lrm_router_grad(const int32_t* row_of_pair, const float* alpha, const float* row_dot, int64_t T,
                           int32_t k, int64_t cap, float* dalpha, cudaStream_t stream);

/*
 * Back to the original token layout (Portuguese list: "the result returns to the original
 * layout"):  dx[t] = sum over j = 0..k-1, in that order, of dx_c[row_of_pair[t*k+j]] for kept
 * pairs, summed in fp32 and rounded once to dt; a token with no kept pair gets 0.  No atomics:
 * the result is deterministic.
 *   row_of_pair [T*k] int32, dx_c [cap,H] dt  ->  dx [T,H] dt.
 * cap is the row count of dx_c: an entry of row_of_pair outside [-1, cap) is not followed (the
 * pair adds nothing) and sets LRM_ERR_BAD_INDEX in the optional dev_status.
 */
lrm_status lrm_scatter_dx(const int32_t* row_of_pair, const void* dx_c, int64_t T, int32_t k, int32_t H,
                          lrm_dtype dt, int64_t cap, void* dx, int32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Forward-side steps beside the path, each fused with the work next to it.
 * ------------------------------------------------------------------------------------------- */

/*
 * Router top-k with the loads and quotas in the same launch ("Backward demand is not a constant":
 * each expert's quota is fixed from its routed demand before the expert forward; here it is
 * computed where the routing is decided, replacing a separate lrm_plan_quotas pass).
 *   logits [T,E] fp32 (row-major)  ->  topk_idx [T*k] int32: the k largest logits of each token in
 *   descending order, ties to the lower expert id; alpha [T*k] fp32: softmax over those k logits;
 *   loads [E], quotas [E] int32 exactly as lrm_plan_quotas writes them for this routing.
 *   kind/num/den/cap/explicit_quotas as in lrm_plan_quotas.
 *   ws: 4-byte-aligned device scratch of >= 4 * (E + 1) bytes (a buffer of lrm_workspace_size bytes does).
 * A non-finite logit is never chosen ahead of a finite one and sets LRM_ERR_NONFINITE in
 * dev_status.  Integer results are deterministic.  Errors: LRM_ERR_INVALID_ARG, LRM_ERR_SHAPE
 * (also k > E), LRM_ERR_WORKSPACE, LRM_ERR_CUDA.
 */
lrm_status lrm_route(const float* logits, int64_t T, int32_t E, int32_t k, lrm_quota_kind kind, int32_t num,
                     int32_t den, int32_t cap, const int32_t* explicit_quotas, int32_t* topk_idx, float* alpha,
                     int32_t* loads, int32_t* quotas, void* ws, size_t ws_bytes, int32_t* dev_status,
                     cudaStream_t stream);

/*
 * SwiGLU activation of the expert forward, also emitting the row norms the LRM score needs
 * ("LRM: a decomposable contribution score": only ||phi_u||^2 of the saved projection input
 * enters the score, so the forward can hand it over and the backward need not re-read phi).
 *   h [P, 2I] dt (gate first)  ->  phi [P, I] dt = round_dt(SiLU(gate) * up) (fp32 arithmetic),
 *   phi_sq [P] fp32 = ||phi_u||^2 of the stored (rounded) row, or NULL to skip it.
 * Errors: LRM_ERR_INVALID_ARG (NULL or misaligned h/phi), LRM_ERR_SHAPE, LRM_ERR_DTYPE, LRM_ERR_CUDA.
 */
lrm_status lrm_swiglu_forward(const void* h, int64_t P, int32_t I, lrm_dtype dt, void* phi, float* phi_sq,
                              cudaStream_t stream);

/*
 * LRM score from the forward's row norms: scores[u] = alpha_u^2 * ||g_t||^2 * phi_sq[u], the value
 * lrm_score computes, with phi_sq [T*k] fp32 in place of phi.  Reads g once per token and never
 * reads phi.  Same errors and non-finite flag as lrm_score.
 */
lrm_status lrm_score_norms(const float* alpha, const void* g, const float* phi_sq, int64_t T, int32_t k,
                           int32_t H, lrm_dtype dt, float* scores, int32_t* dev_status, cudaStream_t stream);

/*
 * Self-test of failure detection (no counterpart in the pages; part of this library's fault
 * handling).  The tensor-core kernels bound every wait on an mbarrier (about one second of
 * %globaltimer): on expiry they record LRM_ERR_TIMEOUT, drain their in-flight copies and MMAs,
 * free TMEM and return, so a stalled pipeline never hangs the GPU.  This entry point runs that
 * same wait routine on an mbarrier that nothing ever arrives on, with the limit `limit_ns`
 * (0 < limit_ns <= 1e10): the kernel returns after about limit_ns and writes LRM_ERR_TIMEOUT to
 * *dev_status (device memory, caller zeroes it).  Errors: LRM_ERR_INVALID_ARG, LRM_ERR_CUDA.
 */
lrm_status lrm_selftest_wait_timeout(int32_t* dev_status, int64_t limit_ns, cudaStream_t stream);

/*
 * lrm_select_static — lrm_select for callers that cannot allocate device memory.
 * The LRMoE pages have no counterpart: this is a deployment convenience of this library.
 *
 * Some callers cannot give the library a workspace: a plugin inside a host framework that owns
 * every device buffer and passes its plugins only their inputs and outputs, or a process whose
 * device memory is reserved up front by a pool allocator, where a cudaMalloc would fail or break
 * the pool's accounting.  This entry point takes the same arguments as lrm_select minus ws and
 * ws_bytes, gives the same results, and allocates nothing: its scratch is a fixed array inside the
 * library (about 12 MB on every GPU that loads it, held until the process exits).
 *   - Limit: T*k <= LRM_SELECT_STATIC_MAX_PAIRS (and the usual E, k limits); larger problems
 *     return LRM_ERR_SHAPE before any GPU work — use lrm_select with a workspace for them.
 *   - The first call on a device, with that device current, looks up the array's device address
 *     (cudaGetSymbolAddress) and remembers it; make that first call before any stream capture.
 *     The address is kept together with the identity of the CUDA context it belongs to: after a
 *     cudaDeviceReset (a new primary context) the next call looks it up again, so that call too
 *     should come before any stream capture.  A failed look-up returns LRM_ERR_CUDA.
 *   - All calls share the one array and leave their data in it.  Nothing in it needs to start
 *     at zero, but calls that overlap on the GPU (different streams, or threads without ordering
 *     between their streams) race on it: serialise them.
 */
#define LRM_SELECT_STATIC_MAX_PAIRS 524288
lrm_status lrm_select_static(const int32_t* topk_idx, const float* scores, const int32_t* quotas, int64_t T,
                             int32_t k, int32_t E, int64_t cap, int32_t* seg_offsets, int32_t* kept_pair,
                             int32_t* row_of_pair, int32_t* dev_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LRM_H */
