// lrm_select_static: the per-expert top-quota selection for callers that cannot allocate.
//
// Some callers of this library cannot hand it scratch memory: a plugin inside a host
// framework that owns every device buffer and passes its plugins only their inputs and
// outputs, or a process whose device memory is reserved up front by a pool allocator, where
// a cudaMalloc would fail or break the pool's accounting.  For them this entry point runs
// the same selection kernels as lrm_select, with their scratch in a fixed array that
// is part of the library image on every GPU that loads it (about 12 MB, held until exit).
//
// Set-up: the first call on a device (with that device current) looks up the array's
// device address with cudaGetSymbolAddress and keeps it, together with the unique id of the
// CUDA context it belongs to; later calls on that device reuse it while the context is the
// same.  A cudaDeviceReset destroys the primary context (and the array's address with it):
// the next call sees a new context id and looks the address up again.  Make the first call
// on each device, and the first call after a reset, before any stream capture.
// Sharing: every call uses the same array and leaves its contents behind.  No word of it has
// to start at zero (each call writes everything it reads first), but two calls that overlap
// on the GPU (different streams or threads without ordering between them) race on it.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace lrm {

namespace {

constexpr int64_t kStaticMaxPairs = LRM_SELECT_STATIC_MAX_PAIRS;

constexpr size_t round256(size_t v) { return (v + 255) / 256 * 256; }
// The selection regions of workspace_layout(kStaticMaxPairs, LRM_MAX_EXPERTS), sized at compile time
// (the grouped-GEMM region that follows them in a workspace is not needed here).
constexpr size_t kStaticBytes =
    round256(sizeof(int32_t) * (size_t)((kStaticMaxPairs + kSelChunk - 1) / kSelChunk) * LRM_MAX_EXPERTS) +
    round256(sizeof(int32_t) * (LRM_MAX_EXPERTS + 1)) + 2 * round256(sizeof(int32_t) * LRM_MAX_EXPERTS) +
    round256(sizeof(int32_t) * kStaticMaxPairs) + round256(sizeof(uint32_t) * kStaticMaxPairs);

static __device__ __align__(256) unsigned char g_select_scratch[kStaticBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the current CUDA context (0 if the driver cannot say), through driver entry
// points fetched by the runtime.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the array on the current device, looked up on the first call in each CUDA
// context of that device (0: the context id is unknown, so it is looked up on every call), or
// nullptr.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned long long ctx = current_context_id();  // 0 before the runtime has made a context current
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = current_context_id();  // the look-up has made the primary context current
  }
  return g_scratch_ptr[dev];
}

}  // namespace

}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_select_static(const int32_t* topk_idx, const float* scores, const int32_t* quotas,
                                        int64_t T, int32_t k, int32_t E, int64_t cap, int32_t* seg_offsets,
                                        int32_t* kept_pair, int32_t* row_of_pair, int32_t* dev_status,
                                        cudaStream_t stream) {
  LRM_NVTX_RANGE();
  if (T < 0 || k < 1 || E < 1) return LRM_ERR_INVALID_ARG;
  if (k > LRM_MAX_TOPK || E > LRM_MAX_EXPERTS) return LRM_ERR_SHAPE;
  if (T > kStaticMaxPairs / k) return LRM_ERR_SHAPE;  // tested before forming T*k
  const int64_t P = T * (int64_t)k;
  if (P > kStaticMaxPairs) return LRM_ERR_SHAPE;  // beyond the fixed scratch: use lrm_select
  if (cap < 0 || cap > INT32_MAX) return LRM_ERR_INVALID_ARG;
  if (!quotas || !seg_offsets) return LRM_ERR_INVALID_ARG;
  if (P > 0 && (!topk_idx || !scores || !row_of_pair)) return LRM_ERR_INVALID_ARG;
  if (cap > 0 && !kept_pair) return LRM_ERR_INVALID_ARG;
  const WsLayout w = workspace_layout(P, E);
  if (w.gemm > kStaticBytes) return LRM_ERR_SHAPE;
  char* b = static_cast<char*>(scratch_for_current_device());
  if (b == nullptr) return LRM_ERR_CUDA;
  SelectWs sw;
  sw.counts = reinterpret_cast<int32_t*>(b + w.counts);
  sw.bucket_start = reinterpret_cast<int32_t*>(b + w.bucket_start);
  sw.keep = reinterpret_cast<int32_t*>(b + w.keep);
  sw.loads = reinterpret_cast<int32_t*>(b + w.loads);
  sw.sorted_u = reinterpret_cast<int32_t*>(b + w.sorted_u);
  sw.sorted_key = reinterpret_cast<uint32_t*>(b + w.sorted_key);
  sw.n_chunks = (P + kSelChunk - 1) / kSelChunk;
  launch_select(topk_idx, scores, quotas, P, E, cap, seg_offsets, kept_pair, row_of_pair, sw, dev_status, stream);
  return cudaGetLastError() == cudaSuccess ? LRM_OK : LRM_ERR_CUDA;
}
