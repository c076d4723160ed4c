// Shared device helpers of the LRM-pruned expert backward kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "lrm.h"

namespace lrm {

// First device error wins: a later error never overwrites an earlier one.
__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (st != nullptr) atomicCAS(st, 0, code);
}

// Index check of the LRM_DEBUG build: true when `cond` holds; otherwise records `code` in the
// status word and yields false, so that the caller skips the access.  In the ordinary build it
// is `true` and costs nothing.  Checks of indices that a caller hands in (row_of_pair,
// seg_offsets, expert ids) are not made with it: those are always on.
#ifdef LRM_DEBUG
#define LRM_DCHECK(cond, st, code) ((cond) ? true : (::lrm::set_status((st), (code)), false))
#else
#define LRM_DCHECK(cond, st, code) true
#endif

// A compacted row index taken from row_of_pair: -1 (dropped) or a row in [0, cap).  Anything
// else is recorded as LRM_ERR_BAD_INDEX and the pair is treated as dropped.
__device__ __forceinline__ int64_t checked_row(int32_t r, int64_t cap, int32_t* st) {
  if (r == -1) return -1;
  if (r < 0 || (int64_t)r >= cap) {
    set_status(st, LRM_ERR_BAD_INDEX);
    return -1;
  }
  return r;
}

// 16-byte vector helpers.  A "vec" is 16 bytes: 8 bf16 or 4 fp32 elements.
template <typename T> struct VecTraits;
template <> struct VecTraits<__nv_bfloat16> { static constexpr int N = 8; };
template <> struct VecTraits<float> { static constexpr int N = 4; };

__device__ __forceinline__ uint4 ldg16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
// Streamed once: do not allocate it in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// Unpack a 16-byte vector into fp32 values.
__device__ __forceinline__ void unpack(uint4 v, float (&f)[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 p = __bfloat1622float2(b[i]);
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}
__device__ __forceinline__ void unpack(uint4 v, float (&f)[4]) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ uint4 pack(const float (&f)[8]) {
  uint4 v;
  __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) b[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}
__device__ __forceinline__ uint4 pack(const float (&f)[4]) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The fixed quota rules of lrm_quota_kind for one expert with load l (exact integer arithmetic).
__device__ __forceinline__ int32_t quota_rule(int64_t l, int kind, int32_t num, int32_t den, int32_t cap,
                                              const int32_t* explicit_q, int e) {
  int64_t q;
  if (kind == LRM_QUOTA_RATIO)
    q = ((int64_t)num * l + den - 1) / den;  // ceil(num/den * load)
  else if (kind == LRM_QUOTA_CAP)
    q = l < cap ? l : cap;
  else
    q = explicit_q[e];
  return (int32_t)(q > INT32_MAX ? INT32_MAX : q);
}

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Kernels of the backward chain (score, selection, compaction, tile plan, grouped GEMMs, scatter)
// are launched with programmatic stream serialization: such a kernel may start while the kernel
// before it on the stream is finishing.  Each of them calls chain_wait() before its first global
// memory access: it waits until the previous grid has completed and its writes are visible (so,
// since every kernel of the chain does the same, until every earlier kernel has), then lets the
// next kernel of the chain launch.  Launched without the attribute, the wait returns at once.
__device__ __forceinline__ void chain_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One-time set-up that belongs to a device (kernel attributes, occupancy, SM counts) is kept
// per device: a process may drive several GPUs.
constexpr int kDeviceSlots = 64;
inline int current_device_slot() {
  int d = -1;
  return cudaGetDevice(&d) == cudaSuccess && d >= 0 && d < kDeviceSlots ? d : -1;
}
// Allows `Kernel` `bytes` of dynamic shared memory on the current device (once per device).
template <auto Kernel>
inline cudaError_t ensure_max_smem(int bytes) {
  static bool done[kDeviceSlots] = {};
  const int d = current_device_slot();
  if (d < 0) return cudaErrorInvalidDevice;
  if (done[d]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[d] = true;
  return e;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                  Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace lrm

// NVTX range of an entry point (host side): pushed only when LRM_NVTX=1 at the first call.
namespace lrm {
bool nvtx_enabled();
void nvtx_push(const char* name);
void nvtx_pop();
struct NvtxRange {
  bool on;
  explicit NvtxRange(const char* name) : on(nvtx_enabled()) {
    if (on) nvtx_push(name);
  }
  ~NvtxRange() {
    if (on) nvtx_pop();
  }
};
}  // namespace lrm
#define LRM_NVTX_RANGE() ::lrm::NvtxRange lrm_nvtx_range_(__func__)
