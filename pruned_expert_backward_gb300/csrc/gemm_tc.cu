// Tensor-core grouped GEMMs of the SwiGLU expert backward on sm_103a: tcgen05.mma with
// TMEM accumulators, operands staged by TMA, one persistent CTA per SM.
//
// "LRMoE: Trimming Backward Work in Memory-Bound MoE Training", section "The part that is
// easy to get wrong": after physical compaction the actual retained row counts drive
// variable-size grouped GEMMs with no padding.  The segment sizes live on the device
// (seg_offsets); a one-block plan kernel turns them into tile tables, and every CTA walks
// its share of the tiles without any host round trip.
//
// Problems (one launch each):
//   VM_SWIGLU  dphi = dy_c[e] W_down[e]            (M = R_e rows, K = H, N = I), epilogue
//              fuses the SwiGLU backward and writes dh_c = [dgate ; dup]
//   VM_STORE   dx_c = dh_c[e] W_gate_up[e]         (M = R_e rows, K = 2I, N = H)
//   VK         dW[e] = A[e]^T B[e] over the segment rows (K = R_e):
//              dW_down = dy_c^T phi_c, dW_gate_up = dh_c^T x_c; fp32 out
//
// CTA layout (320 threads): warp 0 issues TMA loads, warp 1 owns TMEM and issues the MMAs
// (one thread), warps 2-9 drain the accumulators (tcgen05.ld; two warps per 32-row TMEM
// quarter, each taking half of the columns).  Tiles are 128 x 256 with 64-deep K slices;
// 4 smem stages of 48 KB; two 256-column fp32 accumulators in TMEM so the epilogue of one
// tile overlaps the MMAs of the next.
//
// Shared-memory operand layouts are the 128-byte-swizzled canonical forms:
//   K-major  (rows of 64 K-elements = 128 B): SBO = 1024 B between 8-row groups;
//   MN-major (lines of 64 MN-elements = 128 B, one line per K index): LBO = 8192 B between
//            64-wide MN blocks (one TMA box each), SBO = 1024 B between 8-line K groups.
// In the var-K problems a K slice that runs past the end of a segment would pick up the
// next expert's rows.  The plan kernel therefore writes, per expert, copies of the operand
// tensor maps whose row extent ends at that expert's segment end (tensormap.replace on a
// template encoded by the host); TMA then fills the rows beyond it with zeros.
//
// Every wait is bounded (about one second of %globaltimer); on expiry the CTA records
// LRM_ERR_TIMEOUT, raises a CTA-wide abort flag, drains its outstanding TMA loads and
// MMAs, frees TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace lrm {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kMaxStages = 4;
constexpr int kVmStages = 4;
constexpr int kVkStages = 4;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kBBytes = kBN * kBK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each taking half of the columns
constexpr int kThreads = 64 + 32 * kEpiWarps;
// Epilogue staging per epilogue warp: a 32 x 32 fp32 block with rows padded to 33 floats
// (scalar shared accesses are conflict-free both row-per-thread and row-contiguous).
constexpr int kVmLd = 33;
constexpr int kEpiBytes = 32 * kVmLd * 4;
constexpr int kTmemCols = 512;
constexpr uint64_t kWaitNs = 1000000000ull;

enum Kind { VM_SWIGLU = 0, VM_STORE = 1, VK = 2 };

struct TcParams {
  int kind;
  int stages;
  int E;
  int M, N, K;         // VM: N, K fixed (M per expert); VK: M, N fixed (K per expert)
  int nM, nN;          // tile counts along the fixed dims (VK: nM and nN; VM: nN)
  const int32_t* seg;  // [E+1]
  const int32_t* plan; // [E+1] m-tile prefix (VM), then [E] experts by R_e descending (VK)
  void* out;           // VM_SWIGLU: dh_c [rows, 2N]; VM_STORE: dx_c [rows, N]; VK: fp32 [E, M, N]
  const __nv_bfloat16* h_c;  // VM_SWIGLU: [rows, 2N]
  int32_t* status;
  const CUtensorMap* maps_a;  // VK: per-expert maps of A and B whose row extent ends at the
  const CUtensorMap* maps_b;  //     expert's segment end (TMA zero-fills the rows beyond it)
};

// ---------------------------------------------------------------- PTX wrappers -------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait.  Returns false (and raises the abort flag) when the barrier does not
// complete within kWaitNs, or when another role of the CTA has already aborted.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* status,
                                       bool honour_abort = true) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (globaltimer() - t0 > kWaitNs) break;
    }
  }
  *abort_flag = 1;
  set_status(status, LRM_ERR_TIMEOUT);
  return false;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
// A tensor map written by another kernel (generic proxy) must be acquired by the tensormap
// proxy before a TMA instruction uses it.
__device__ __forceinline__ void tensormap_acquire(const CUtensorMap* m) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(m))
               : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: D fp32, A and B bf16, dense, M = 128, N = 256.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t a_mn_major, uint32_t b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn_major << 15) | (b_mn_major << 16) |
         ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

// ---------------------------------------------------------------- tile decode --------
struct Tile {
  int e;
  int row0, row_end;  // VM: output rows; VK: reduction rows
  int m0, n0;         // VK: output tile origin; VM: n0 only
  int k_iters;
};

// The tile tables (seg_offsets and the plan) are tiny and read through the read-only cache.
__device__ __forceinline__ int total_tiles(const TcParams& p) {
  return p.kind == VK ? p.E * p.nM * p.nN : __ldg(p.plan + p.E) * p.nN;
}

__device__ __forceinline__ Tile decode(const TcParams& p, int t) {
  Tile d;
  if (p.kind == VK) {
    const int per = p.nM * p.nN;
    const int ei = t / per, r = t - ei * per;
    d.e = __ldg(p.plan + p.E + 1 + ei);
    const int mt = r / p.nN, nt = r - mt * p.nN;
    d.m0 = mt * kBM;
    d.n0 = nt * kBN;
    d.row0 = __ldg(p.seg + d.e);
    d.row_end = __ldg(p.seg + d.e + 1);
    d.k_iters = (d.row_end - d.row0 + kBK - 1) / kBK;
  } else {
    const int mg = t / p.nN, nt = t - mg * p.nN;
    int lo = 0, hi = p.E;  // largest e with prefix[e] <= mg
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.plan + mid) <= mg) lo = mid; else hi = mid;
    }
    d.e = lo;
    d.row0 = __ldg(p.seg + lo) + (mg - __ldg(p.plan + lo)) * kBM;
    d.row_end = min(__ldg(p.seg + lo + 1), d.row0 + kBM);
    d.m0 = 0;
    d.n0 = nt * kBN;
    d.k_iters = (p.K + kBK - 1) / kBK;
  }
  return d;
}

__host__ __device__ constexpr uint32_t epi_offset(int stages) { return (uint32_t)stages * kStageBytes; }
__host__ __device__ constexpr uint32_t bar_offset(int stages) { return epi_offset(stages) + kEpiWarps * kEpiBytes; }

// ---------------------------------------------------------------- the kernel ---------
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  uint8_t* epi = smem + epi_offset(S);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + bar_offset(S));
  // bars: full[kMaxStages], empty[kMaxStages], acc_full[2], acc_empty[2], drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 5);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);
  const uint32_t accf0 = smem_u32(bars + 2 * kMaxStages), acce0 = smem_u32(bars + 2 * kMaxStages + 2);
  const uint32_t drain = smem_u32(bars + 2 * kMaxStages + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accf0, 1);
    mbar_init(accf0 + 8, 1);
    mbar_init(acce0, kEpiWarps);
    mbar_init(acce0 + 8, kEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int n_tiles = total_tiles(p);
  volatile int* abortv = abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer -------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      int last_e = -1;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        const Tile d = decode(p, t);
        const CUtensorMap* ma = &tmA;
        const CUtensorMap* mb = &tmB;
        if (p.kind == VK) {
          ma = p.maps_a + d.e;
          mb = p.maps_b + d.e;
          if (d.e != last_e && d.k_iters > 0) {
            tensormap_acquire(ma);
            tensormap_acquire(mb);
            last_e = d.e;
          }
        }
        for (int kb = 0; kb < d.k_iters; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1u;
          if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abortv, p.status)) { ok = false; break; }
          const uint32_t a_dst = smem_u32(smem + s * kStageBytes), b_dst = a_dst + kABytes;
          const uint32_t fb = full0 + 8 * s;
          mbar_expect_tx(fb, kStageBytes);
          if (p.kind == VK) {
            const int r = d.row0 + kb * kBK;
            tma_load_2d(a_dst, ma, d.m0, r, fb);
            tma_load_2d(a_dst + 8192, ma, d.m0 + 64, r, fb);
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_2d(b_dst + 8192 * j, mb, d.n0 + 64 * j, r, fb);
          } else {
            tma_load_2d(a_dst, &tmA, kb * kBK, d.row0, fb);
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_3d(b_dst + 8192 * j, &tmB, d.n0 + 64 * j, kb * kBK, d.e, fb);
          }
        }
      }
      // drain: every load this thread issued must have landed before the CTA exits
      const uint32_t first = it > (uint32_t)S ? it - S : 0u;
      for (uint32_t i = first; i < it; ++i) mbar_wait(full0 + 8 * (i % S), (i / S) & 1u, abortv, p.status, false);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer ---------
    const bool a_mn = p.kind == VK;
    const uint32_t idesc = instr_desc(a_mn ? 1u : 0u, 1u);
    uint32_t it = 0;
    int lt = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++lt) {
      const Tile d = decode(p, t);
      const uint32_t acc = lt & 1, acc_ph = (lt >> 1) & 1;
      if (!mbar_wait(acce0 + 8 * acc, acc_ph ^ 1u, abortv, p.status)) break;
      tc_fence_after();
      const uint32_t tmem_d = tmem_base + acc * kBN;
      for (int kb = 0; kb < d.k_iters; ++kb, ++it) {
        const uint32_t s = it % S, ph = (it / S) & 1u;
        if (!mbar_wait(full0 + 8 * s, ph, abortv, p.status)) { ok = false; break; }
        tc_fence_after();
        uint8_t* a_st = smem + s * kStageBytes;
        uint8_t* b_st = a_st + kABytes;
        if (lane == 0) {
          const uint32_t a_addr = smem_u32(a_st), b_addr = smem_u32(b_st);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t adesc = a_mn ? smem_desc(a_addr + kk * 2048, 8192, 1024)
                                        : smem_desc(a_addr + kk * 32, 16, 1024);
            const uint64_t bdesc = smem_desc(b_addr + kk * 2048, 8192, 1024);
            mma_bf16(tmem_d, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(empty0 + 8 * s);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma_commit(accf0 + 8 * acc);
      __syncwarp();
    }
    // drain: all MMAs issued by this CTA complete before TMEM is released
    if (lane == 0) mma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, abortv, p.status, false);
  } else {
    // ------------------------------------------------------------ epilogue -----------
    // Warp w may read TMEM lanes 32*(w%4) .. +31 (tile rows q*32 .. q*32+31); the two warps
    // of a quarter split the eight 32-column chunks.  Each chunk is read row-per-thread
    // (tcgen05.ld 32x32b), staged in shared memory and written back row-contiguous, so global
    // stores (and the SwiGLU h_c loads) are coalesced; var-M rows are masked at the segment end.
    const int ew = warp - 2, q = warp & 3, half = ew >> 2;
    float* stg = reinterpret_cast<float*>(epi + ew * kEpiBytes);
    int lt = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++lt) {
      const Tile d = decode(p, t);
      const uint32_t acc = lt & 1, acc_ph = (lt >> 1) & 1;
      if (!mbar_wait(accf0 + 8 * acc, acc_ph, abortv, p.status)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * kBN + ((uint32_t)(q * 32) << 16);
      const bool have_acc = d.k_iters > 0;
      const int row_base = p.kind == VK ? d.m0 + q * 32 : d.row0 + q * 32;
      const int row_lim = p.kind == VK ? p.M : d.row_end;
      const int nrows = min(32, row_lim - row_base);
      for (int c = half * 4; c < half * 4 + 4; ++c) {
        const int n = d.n0 + c * 32;
        if (n >= p.N) break;  // warp-uniform
        uint32_t v[32];
        if (have_acc) tmem_ld32(tbase + c * 32, v);
        else
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        if (nrows <= 0) continue;
#pragma unroll
        for (int i = 0; i < 32; ++i) stg[lane * kVmLd + i] = __uint_as_float(v[i]);
        __syncwarp();
        if (p.kind == VK) {
          // fp32 dW: 4 rows x 128 B per instruction
          const int sub = lane >> 3, piece = lane & 7;
          const int col = n + piece * 4;
          float* out = reinterpret_cast<float*>(p.out) + (int64_t)d.e * p.M * p.N;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = i * 4 + sub;
            if (rr < nrows && col < p.N) {
              const float* sv = stg + rr * kVmLd + piece * 4;
              *reinterpret_cast<float4*>(out + (int64_t)(row_base + rr) * p.N + col) =
                  make_float4(sv[0], sv[1], sv[2], sv[3]);
            }
          }
        } else {
          // bf16 rows: 8 rows x 64 B per instruction; lane owns 8 columns of one row
          const int sub = lane >> 2, piece = lane & 3;
          const int col = n + piece * 8;
          if (p.kind == VM_SWIGLU) {
            const int I = p.N;
            uint4 gv[4], uv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = i * 8 + sub;
              if (rr < nrows && col < I) {
                const __nv_bfloat16* hrow = p.h_c + (int64_t)(row_base + rr) * 2 * I;
                gv[i] = ldg16(hrow + col);
                uv[i] = ldg16(hrow + I + col);
              }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = i * 8 + sub;
              if (rr < nrows && col < I) {
                const float* sv = stg + rr * kVmLd + piece * 8;
                float gate[8], up[8], dg[8], du[8];
                unpack(gv[i], gate);
                unpack(uv[i], up);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float dphi = sv[j];
                  const float sg = 1.f / (1.f + __expf(-gate[j]));
                  dg[j] = dphi * up[j] * sg * (1.f + gate[j] * (1.f - sg));
                  du[j] = dphi * gate[j] * sg;
                }
                __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + (int64_t)(row_base + rr) * 2 * I;
                st16(orow + col, pack(dg));
                st16(orow + I + col, pack(du));
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = i * 8 + sub;
              if (rr < nrows && col < p.N) {
                const float* sv = stg + rr * kVmLd + piece * 8;
                float f[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] = sv[j];
                __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + (int64_t)(row_base + rr) * p.N;
                st16(orow + col, pack(f));
              }
            }
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * acc);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Tile tables from seg_offsets: plan[0..E] = exclusive prefix of ceil(R_e / kBM) (var-M tiles),
// plan[E+1 .. 2E] = experts ordered by R_e descending, ties by expert id (var-K, longest first).
// maps[j][e] = template j with its row extent cut at seg_offsets[e+1] (var-K operands).
struct MapTemplates {
  CUtensorMap t[4];
};
__global__ void __launch_bounds__(1024) tc_plan_kernel(const int32_t* __restrict__ seg, int E,
                                                       int32_t* __restrict__ plan, CUtensorMap* __restrict__ maps,
                                                       const __grid_constant__ MapTemplates tpl) {
  __shared__ int s_r[LRM_MAX_EXPERTS];
  __shared__ int warp_tot[32];
  const int e = threadIdx.x;
  const int r = e < E ? seg[e + 1] - seg[e] : 0;
  if (e < E) s_r[e] = r;
  const int mt = (r + kBM - 1) / kBM;
  // exclusive block scan of mt
  const int lane = e & 31, w = e >> 5;
  int incl = mt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int v = warp_tot[lane];
    int wi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - v;
  }
  __syncthreads();
  const int excl = warp_tot[w] + incl - mt;
  if (e < E) plan[e] = excl;
  if (e == E - 1) plan[E] = excl + mt;
  if (e < E) {
    int rank = 0;
    for (int j = 0; j < E; ++j) {
      const int rj = s_r[j];
      rank += (rj > r) || (rj == r && j < e);
    }
    plan[E + 1 + rank] = e;
    const uint32_t rows_end = (uint32_t)max(1, seg[e + 1]);
    for (int j = 0; j < 4; ++j) {
      CUtensorMap* dst = maps + j * E + e;
      const uint4* src = reinterpret_cast<const uint4*>(&tpl.t[j]);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int w = 0; w < 8; ++w) d4[w] = src[w];
      asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(
                       reinterpret_cast<uint64_t>(dst)),
                   "r"(rows_end)
                   : "memory");
    }
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  }
}

// ---------------------------------------------------------------- host side ----------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 row-major [rows, cols] with a {64, box_rows} box, 128-byte swizzle.
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// bf16 [E, K, N] (N contiguous) with a {64, 64, 1} box, 128-byte swizzle.
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t E, uint64_t K, uint64_t N) {
  const cuuint64_t dims[3] = {N, K, E};
  const cuuint64_t strides[2] = {N * 2, K * N * 2};
  const cuuint32_t box[3] = {64, 64, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t smem_bytes(int stages) { return 1024 + bar_offset(stages) + (2 * kMaxStages + 5) * 8 + 8; }

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

bool device_ok() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3;
}

lrm_status launch_one(const CUtensorMap& a, const CUtensorMap& b, const TcParams& p, int64_t tiles_bound,
                      cudaStream_t s) {
  if (tiles_bound <= 0) return LRM_OK;
  const size_t smem = smem_bytes(p.stages);
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(tc_grouped_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_bytes(kMaxStages)) != cudaSuccess)
      return LRM_ERR_CUDA;
    attr_set = true;
  }
  const int grid = (int)(tiles_bound < sm_count() ? tiles_bound : sm_count());
  tc_grouped_kernel<<<grid, kThreads, smem, s>>>(a, b, p);
  return cudaGetLastError() == cudaSuccess ? LRM_OK : LRM_ERR_CUDA;
}

}  // namespace

lrm_status launch_grouped_tc(const GroupedArgs& g, const GemmWs& ws, cudaStream_t s) {
  if (!device_ok() || encode_fn() == nullptr) return LRM_ERR_UNSUPPORTED;
  const int E = g.E, H = g.H, I = g.I;
  const uint64_t rows = g.cap > 0 ? (uint64_t)g.cap : 1;
  int32_t* plan = ws.plan;  // [2E+1] tile tables
  CUtensorMap* maps = static_cast<CUtensorMap*>(ws.maps);
  MapTemplates tpl;
  if (!make_map_2d(&tpl.t[0], g.dy_c, rows, H, 64) || !make_map_2d(&tpl.t[1], g.phi_c, rows, I, 64) ||
      !make_map_2d(&tpl.t[2], g.dh_c, rows, 2 * I, 64) || !make_map_2d(&tpl.t[3], g.x_c, rows, H, 64))
    return LRM_ERR_CUDA;
  tc_plan_kernel<<<1, 1024, 0, s>>>(g.seg_offsets, E, plan, maps, tpl);
  if (cudaGetLastError() != cudaSuccess) return LRM_ERR_CUDA;

  CUtensorMap mA, mB;
  const int64_t vm_bound = ((int64_t)g.cap + kBM - 1) / kBM + E;
  lrm_status st;
  // dphi = dy_c W_down[e], SwiGLU backward fused -> dh_c
  if (!make_map_2d(&mA, g.dy_c, rows, H, kBM) || !make_map_3d(&mB, g.w_down, E, H, I)) return LRM_ERR_CUDA;
  TcParams p{VM_SWIGLU, kVmStages, E, 0, I, H, 0, (I + kBN - 1) / kBN, g.seg_offsets, plan, g.dh_c,
             (const __nv_bfloat16*)g.h_c, g.status, nullptr, nullptr};
  if ((st = launch_one(mA, mB, p, vm_bound * p.nN, s))) return st;
  // dW_down[e] = dy_c^T phi_c  (M = H, N = I)
  p = TcParams{VK, kVkStages, E, H, I, 0, (H + kBM - 1) / kBM, (I + kBN - 1) / kBN, g.seg_offsets, plan, g.dw_down,
               nullptr, g.status, maps + 0 * E, maps + 1 * E};
  mA = tpl.t[0];
  mB = tpl.t[1];
  if ((st = launch_one(mA, mB, p, (int64_t)E * p.nM * p.nN, s))) return st;
  // dW_gate_up[e] = dh_c^T x_c  (M = 2I, N = H)
  p = TcParams{VK, kVkStages, E, 2 * I, H, 0, (2 * I + kBM - 1) / kBM, (H + kBN - 1) / kBN, g.seg_offsets, plan,
               g.dw_gate_up, nullptr, g.status, maps + 2 * E, maps + 3 * E};
  mA = tpl.t[2];
  mB = tpl.t[3];
  if ((st = launch_one(mA, mB, p, (int64_t)E * p.nM * p.nN, s))) return st;
  // dx_c = dh_c W_gate_up[e]  (K = 2I, N = H)
  if (!make_map_2d(&mA, g.dh_c, rows, 2 * I, kBM) || !make_map_3d(&mB, g.w_gate_up, E, 2 * I, H))
    return LRM_ERR_CUDA;
  p = TcParams{VM_STORE, kVmStages, E, 0, H, 2 * I, 0, (H + kBN - 1) / kBN, g.seg_offsets, plan, g.dx_c, nullptr,
               g.status, nullptr, nullptr};
  if ((st = launch_one(mA, mB, p, vm_bound * p.nN, s))) return st;
  return LRM_OK;
}

}  // namespace lrm
