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
//   VM_FWD     h_c = x_c[e] W_gate_up[e]^T         (M = R_e rows, K = H, N = 2I), the saved forward
//              state recomputed for the retained rows: B is K-major (W_gate_up's rows), a pair tile
//              holds 128 gate columns and the matching 128 up columns, and the epilogue writes h_c
//              and phi_c = SiLU(gate) * up
//
// CTAs run in pairs (a cluster of two) and use the 2-SM MMA: the leader (even) CTA issues
// tcgen05.mma.cta_group::2, which computes a 256 x 256 tile from both CTAs' shared memory
// (each CTA stages its own 128 rows of A and its own 128 columns of B) into both CTAs' TMEM
// (128 rows each).  Per SM that is 32 KB of operands per 64-deep K slice instead of 48 KB
// for a 128 x 256 single-SM tile, and 6 stages fit in shared memory (5 for the dphi launch,
// whose epilogue needs room for its gate/up tiles).
// CTA layout (320 threads): warp 0 issues TMA loads (both CTAs; they complete on the
// leader's full barrier), warp 1 owns TMEM (allocated collectively by the pair) and, in the
// leader, issues the MMAs from one thread; warps 2-9 drain this CTA's accumulator rows
// (tcgen05.ld; two warps per 32-row TMEM quarter, each taking half of the columns) and write
// them out through TMA stores.  Two 256-column fp32 accumulators in TMEM let the epilogue of
// one tile overlap the MMAs of the next; both CTAs' epilogues release an accumulator on the
// leader's barrier.
// Tiles go to the CTA pairs round robin, except in the var-K launches of a call with long tiles
// (mean retained rows per expert >= kDynMinRowsPerExpert, decided on the device by the plan
// kernel), where each pair takes its next tile from a global counter as it becomes free (TileSeq).
//
// Shared-memory operand layouts are the 128-byte-swizzled canonical forms:
//   K-major  (rows of 64 K-elements = 128 B): SBO = 1024 B between 8-row groups;
//   MN-major (lines of 64 MN-elements = 128 B, one line per K index): LBO = 8192 B between
//            64-wide MN blocks, SBO = 1024 B between 8-line K groups; both blocks of a CTA's
//            128 columns come in one TMA box where the column count allows (see merged_a).
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

constexpr int kBM = 128;  // output rows per CTA; a CTA pair computes 256-row tiles
constexpr int kBN = 256;  // output columns of a pair tile; each CTA stages half of B
constexpr int kBK = 64;
// Operand pipeline depth (32 KB stages).  The dphi + SwiGLU launch runs one stage shallower:
// its epilogue also reads the gate/up rows, and fewer operand loads in flight leave those
// reads less queueing (measured on GB300: 223 -> 211 us on the Qwen3 T=8192 layer, while the
// other three problems are 2-4 % slower with 5 stages than with 6).
constexpr int kStages = 6;
constexpr int kSwigluStages = 5;
constexpr int kABytes = kBM * kBK * 2;            // 16 KB: this CTA's 128 rows of A
constexpr int kBHalfBytes = (kBN / 2) * kBK * 2;  // 16 KB: this CTA's 128 columns of B
constexpr int kStageBytes = kABytes + kBHalfBytes;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each taking half of the columns
// Gathering B rows (compaction-free variant), warp 0 and these extra warps copy them: one warp
// alone cannot keep enough copies in flight.  Other launches leave the extra warps idle.
constexpr int kGatherExtraWarps = 2;
constexpr int kGatherWarps = 1 + kGatherExtraWarps;
constexpr int kThreads = 64 + 32 * kEpiWarps + 32 * kGatherExtraWarps;
// Epilogue staging per epilogue warp: a 32 x 32 fp32 block with rows padded to 33 floats
// (scalar shared accesses are conflict-free both row-per-thread and row-contiguous).
constexpr int kVmLd = 33;
constexpr int kEpiBytes = 32 * kVmLd * 4;
// var-K: the same region holds two 2 KB staging boxes per warp for TMA stores, used in turn
// (4 KB, 1024-byte-aligned)
constexpr int kBoxBytes = 4096;
static_assert(kBoxBytes <= kEpiBytes, "staging box must fit in the per-warp epilogue region");
// var-M epilogue through TMA (compacted rows): results leave by TMA stores of 32-row x 32-column
// bf16 boxes (64-byte swizzle) through per-expert maps whose row extent ends at the segment end,
// so rows past it are clipped by the hardware; the SwiGLU gate/up tiles arrive by TMA one chunk
// ahead, into two 4 KB buffers per warp (the launches with a shallower operand pipeline have the
// room: 8 KB per epilogue warp).
constexpr int kEpiBytesWide = 8192;
template <int S>
__host__ __device__ constexpr int epi_bytes() { return S < kStages ? kEpiBytesWide : kEpiBytes; }
constexpr int kVmBoxBytes = 2048;  // 32 rows x 64 bytes
static_assert(kSwigluStages < kStages, "the dphi launch's epilogue needs the wide per-warp buffers");
constexpr int kTmemCols = 512;
constexpr uint64_t kWaitNs = 1000000000ull;

enum Kind { VM_SWIGLU = 0, VM_STORE = 1, VK = 2, VM_FWD = 3 };

template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};

struct TcParams {
  int kind;
  int E;
  int M, N, K;         // VM: N, K fixed (M per expert); VK: M, N fixed (K per expert)
  int nM, nN;          // tile counts along the fixed dims (VK: nM and nN; VM: nN)
  const int32_t* seg;  // [E+1]
  const int32_t* plan; // [E+1] m-tile prefix (VM), then [E] experts by R_e descending (VK), then
                       // the segment check word (1: seg_offsets valid; 0: run no tile)
  void* out;           // VM_SWIGLU: dh_c [rows, 2N]; VM_STORE: dx_c [rows, N]; VK: fp32 [E, M, N]
  const __nv_bfloat16* h_c;  // VM_SWIGLU: [rows, 2N]
  int32_t* status;
  const CUtensorMap* maps_a;  // VK: per-expert maps of A and B whose row extent ends at the
  const CUtensorMap* maps_b;  //     expert's segment end (TMA zero-fills the rows beyond it)
  float* dot_part;            // VM_SWIGLU, optional: [rows][n_part] parts of dphi . phi (one per
  int n_part;                 //     128 output columns), summed in order by the reduce kernel
  // Gather mode (kept_pair non-null; the compaction-free variant): compacted row r stands for
  // pair u = kept_pair[r].  VM_SWIGLU reads gate/up from gsrc = h [P, 2I] at row u; VK gathers
  // its B operand rows from gsrc (phi at row u, or x at row u / gk when gk > 0) with cp.async.
  const int32_t* kept_pair;
  const __nv_bfloat16* gsrc;
  int gk;   // VK: > 0 when the gathered rows are tokens (u / gk)
  int gld;  // elements per row of gsrc
  // MN-major operands whose 64-column blocks come in one TMA box: the map views the operand as
  // [column block][K line][64 columns], so one {64, 64, 2} box fills both 8 KB blocks of a CTA's
  // 128 columns (the same shared-memory layout as two {64, 64} boxes, in one instruction).
  // Only where the column count is a multiple of 64 (a partial block would wrap into the next
  // line instead of being zero-filled).
  int merged_a;  // VK: A
  int merged_b;  // VK and VM: B
  // VM, compacted rows: epilogue through TMA.  maps_a then holds the per-expert output maps
  // (dh_c viewed as [rows][2][I], dx_c as [rows][H]), and tmC the gate/up map of h_c ([rows][2][I]).
  int tma_epi;
  int gP;  // gather mode: pairs in h / phi (T*k); a kept_pair entry outside [0, gP) is not followed
  // var-K launches: counter of the dynamic tile order (see TileSeq), used when the plan kernel
  // switched it on for this call (plan[2E+2] = 1)
  int32_t* tile_counter;
};

// Pair named by kept_pair for a gathered row: in [0, gP), or -1 (flagged; the row reads as zeros).
__device__ __forceinline__ int gather_pair(const TcParams& p, int r) {
  const int u = __ldg(p.kept_pair + r);
  if (u < 0 || u >= p.gP) {
    set_status(p.status, LRM_ERR_BAD_INDEX);
    return -1;
  }
  return u;
}

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
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait.  Returns false (and raises the abort flag) when the barrier does not
// complete within kWaitNs, or when another role of the CTA has already aborted.  The common
// case (already complete) stays inline; the polling loop is out of line.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            int32_t* status, bool honour_abort, uint64_t limit_ns = kWaitNs,
                                            bool cluster_acquire = false) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (cluster_acquire ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) break;
    }
  }
  *abort_flag = 1;
  set_status(status, LRM_ERR_TIMEOUT);
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* status,
                                          bool honour_abort = true) {
  if (mbar_try(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, status, honour_abort);
}
// The same with cluster-scope acquire: the waiter then sees what the other CTA of the pair wrote
// before its release-arrive (shared-memory operands copied by threads, not by TMA).
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             int32_t* status) {
  if (mbar_try_cluster(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, status, true, kWaitNs, true);
}
// Cluster helpers.  CTAs run in pairs (a cluster of two); the even CTA is the MMA leader.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// Address, in the cluster shared window, of the same shared offset in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx_cluster(uint32_t cbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(cbar), "r"(bytes) : "memory");
}
// TMA load into this CTA's shared memory that completes on an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t cbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(cbar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                 uint32_t cbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(cbar)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                                 uint32_t cbar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(cbar)
      : "memory");
}
// TMA load into this CTA's shared memory, completing on this CTA's mbarrier.
__device__ __forceinline__ void tma_load_3d_cta(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
// 16-byte cp.async into shared memory; src_bytes < 16 zero-fills the rest (0: nothing is read).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// The mbarrier receives one arrival once all of this thread's earlier cp.async have completed
// (the barrier's expected count includes it; the thread does not wait).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Generic-proxy writes to shared memory become visible to the async proxy (tensor core reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Arrive on an mbarrier of either CTA of the pair, ordering this thread's earlier writes before it
// for a waiter anywhere in the cluster.
__device__ __forceinline__ void mbar_arrive_release_cluster(uint32_t cbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}
// TMA tensor store from this CTA's shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_le1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// A tensor map written by another kernel (generic proxy) must be acquired by the tensormap
// proxy before a TMA instruction uses it.
__device__ __forceinline__ void tensormap_acquire(const CUtensorMap* m) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(m))
               : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
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
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Completion of this CTA pair's MMAs arrives on the mbarrier at the same offset in both CTAs.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)0x3)
      : "memory");
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
// Instruction descriptor of kind::f16: D fp32, A and B bf16, dense, M = 256 (the CTA pair),
// N = 256.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t a_mn_major, uint32_t b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn_major << 15) | (b_mn_major << 16) |
         ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)((2 * kBM) >> 4) << 24);
}

// ---------------------------------------------------------------- tile decode --------
// Work is handed out in pair tiles: a cluster of two CTAs computes two vertically adjacent
// 128-row tiles (rank 0 the upper, rank 1 the lower) that share the same 256 B columns.
struct Tile {
  int e;
  int row0, row_end;  // VM: this CTA's output rows; VK: the expert's reduction rows
  int m0, n0;         // VK: output tile origin of this CTA; VM: n0 only
  int k_iters;
  bool has_rows;      // this CTA's half of the pair tile holds output rows
};

// The tile tables (seg_offsets and the plan) are tiny and read through the read-only cache.
// Segments that failed the plan kernel's check give no tile at all.
__device__ __forceinline__ int total_tiles(const TcParams& p) {
  if (__ldg(p.plan + 2 * p.E + 1) != 1) return 0;
  return p.kind == VK ? p.E * ((p.nM + 1) / 2) * p.nN : __ldg(p.plan + p.E) * p.nN;
}

__device__ __forceinline__ Tile decode(const TcParams& p, int t, int rank) {
  Tile d;
  if (p.kind == VK) {
    const int nMp = (p.nM + 1) / 2;
    const int per = nMp * p.nN;
    const int ei = t / per, r = t - ei * per;
    d.e = __ldg(p.plan + p.E + 1 + ei);
    const int mp = r / p.nN, nt = r - mp * p.nN;
    d.m0 = (2 * mp + rank) * kBM;
    d.n0 = nt * kBN;
    d.row0 = __ldg(p.seg + d.e);
    d.row_end = __ldg(p.seg + d.e + 1);
    d.k_iters = (d.row_end - d.row0 + kBK - 1) / kBK;
    d.has_rows = d.m0 < p.M;
  } else {
    const int mg = t / p.nN, nt = t - mg * p.nN;
    int lo = 0, hi = p.E;  // largest e with prefix[e] <= mg
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.plan + mid) <= mg) lo = mid; else hi = mid;
    }
    d.e = lo;
    const int seg_end = __ldg(p.seg + lo + 1);
    d.row0 = __ldg(p.seg + lo) + (mg - __ldg(p.plan + lo)) * (2 * kBM) + rank * kBM;
    d.row_end = min(seg_end, d.row0 + kBM);
    d.m0 = 0;
    d.n0 = nt * (p.kind == VM_FWD ? kBN / 2 : kBN);  // VM_FWD: 128 gate (and 128 up) columns
    d.k_iters = (p.K + kBK - 1) / kBK;
    d.has_rows = d.row0 < seg_end;
  }
  return d;
}

template <int S>
__host__ __device__ constexpr uint32_t epi_offset() { return (uint32_t)S * kStageBytes; }
template <int S>
__host__ __device__ constexpr uint32_t bar_offset() { return epi_offset<S>() + kEpiWarps * epi_bytes<S>(); }
// Tile ring of the dynamic tile order: the leader's producer publishes each tile index it takes
// into kRing slots in both CTAs; every other role of the pair reads it there and frees the slot on
// the leader's tile_empty barrier (kRingReaders arrivals: the MMA issuer, the other CTA's producer
// and the epilogue warps of both CTAs).
constexpr int kRing = 16;
constexpr int kRingReaders = 2 + 2 * kEpiWarps;
// barriers: full[S], empty[S], acc_full[2], acc_empty[2], drain, gathered[S], two per epilogue
// warp for its gate/up buffers, then tile_full[kRing], tile_empty[kRing]
template <int S>
__host__ __device__ constexpr int n_barriers() { return 3 * S + 5 + 2 * kEpiWarps + 2 * kRing; }
template <int S>
__host__ __device__ constexpr int ring_bar_index() { return 3 * S + 5 + 2 * kEpiWarps; }

// The tile sequence of one role of a CTA pair.  Static order: pair, pair + n_pairs, ...  Dynamic
// order (var-K launches with long tiles): the leader's producer takes tiles from a global counter
// in plan order as its pair becomes free and publishes them (take / publish), one tile ahead of its
// own loads; the other roles read them from their CTA's ring (next).  The tiles running at any moment
// are then consecutive in the plan whatever their lengths, so the tiles of one expert stay together
// in time and share its operand rows through L2; with the fixed round robin the pairs drift apart
// once experts of different lengths mix, and an expert's rows are fetched from DRAM again and again.
// A value >= n_tiles ends the sequence; -1 means a wait gave up.
struct TileSeq {
  bool dyn;
  int t, n_tiles, n_pairs;
  uint32_t full0, empty0, empty_lead;  // this CTA's tile_full / tile_empty, the leader's tile_empty
  volatile int* slots;                 // this CTA's ring
  uint32_t slot, ph;
  volatile int* abort;
  int32_t* status;
  bool local;  // a reader in the leader CTA (releases its slot on its own CTA's barrier)

  __device__ __forceinline__ int first(int pair) {
    if (!dyn) return t = pair;
    return t = read();
  }
  __device__ __forceinline__ int next() {
    if (!dyn) return t += n_pairs;
    return t = read();
  }
  // reader side (one thread)
  __device__ __forceinline__ int read() {
    if (!mbar_wait_cl(full0 + 8 * slot, ph, abort, status)) return -1;
    const int v = slots[slot];
    if (local)
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty0 + 8 * slot) : "memory");
    else
      mbar_arrive_release_cluster(empty_lead + 8 * slot);
    if (++slot == (uint32_t)kRing) { slot = 0; ph ^= 1u; }
    return v;
  }
  // taker side (the leader's producer thread)
  __device__ __forceinline__ int take(int32_t* counter) {
    const int v = atomicAdd(counter, 1);
    return v < n_tiles ? v : n_tiles;
  }
  __device__ __forceinline__ bool publish(int v, uint32_t remote_slots, uint32_t remote_full0) {
    if (!mbar_wait_cl(empty0 + 8 * slot, ph ^ 1u, abort, status)) return false;  // all readers freed it
    slots[slot] = v;
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote_slots + 4 * slot), "r"(v) : "memory");
    mbar_arrive_release_cluster(cluster_addr(full0 + 8 * slot, 0));
    mbar_arrive_release_cluster(remote_full0 + 8 * slot);
    if (++slot == (uint32_t)kRing) { slot = 0; ph ^= 1u; }
    t = v;
    return true;
  }
};


// ---------------------------------------------------------------- the kernel ---------
// S: operand pipeline depth.  RING: the kernel can follow the dynamic tile order (the var-K
// launches); the others are compiled without it.
template <int S, bool RING>
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi = smem + epi_offset<S>();
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + bar_offset<S>());
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + n_barriers<S>());
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  int* ring_slots = abort_flag + 1;  // [kRing]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
  const uint32_t accf0 = smem_u32(bars + 2 * S), acce0 = smem_u32(bars + 2 * S + 2);
  const uint32_t drain = smem_u32(bars + 2 * S + 4);
  const uint32_t gath0 = smem_u32(bars + 2 * S + 5);  // this CTA's gathered B rows of a stage landed

  const bool gather_b = p.kind == VK && p.kept_pair != nullptr;  // B rows gathered by threads
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // leader's: both producers arrive with their byte counts (and, gathering, the other CTA
      // once more when its copies of the stage have landed)
      mbar_init(full0 + 8 * s, gather_b ? 3 : 2);
      mbar_init(gath0 + 8 * s, 32 * kGatherWarps);  // gathering: every copying lane's copies
      mbar_init(empty0 + 8 * s, 1);  // the leader's MMA commit, multicast to the pair
    }
    mbar_init(accf0, 1);
    mbar_init(accf0 + 8, 1);
    mbar_init(acce0, 2 * kEpiWarps);  // leader's: the epilogue warps of both CTAs
    mbar_init(acce0 + 8, 2 * kEpiWarps);
    mbar_init(drain, 1);
    for (int i = 0; i < 2 * kEpiWarps; ++i) mbar_init(smem_u32(bars + 3 * S + 5 + i), 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(smem_u32(bars + ring_bar_index<S>() + i), 1);                     // tile_full: the taker
      mbar_init(smem_u32(bars + ring_bar_index<S>() + kRing + i), kRingReaders);  // tile_empty (leader's)
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), kTmemCols);  // collective over the pair
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote operation targets them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // the set-up above touches no global memory, so it overlaps the end of the previous kernel
  chain_wait();
  const int n_tiles = total_tiles(p);
  volatile int* abortv = abort_flag;
  const uint32_t full_lead = cluster_addr(full0, 0), acce_lead = cluster_addr(acce0, 0);
  const uint32_t tfull0 = smem_u32(bars + ring_bar_index<S>()), tempty0 = tfull0 + 8 * kRing;
  // this role's tile sequence (TileSeq): dynamic for the var-K launches when the plan kernel chose it
  const bool dyn_order =
      RING && p.kind == VK && p.tile_counter != nullptr && !gather_b && __ldg(p.plan + 2 * p.E + 2) == 1;
  TileSeq seq{dyn_order, 0, n_tiles, n_pairs, tfull0, tempty0, cluster_addr(tempty0, 0), ring_slots, 0u, 0u,
              abort_flag, p.status, leader};

  const int first_extra = 2 + kEpiWarps;  // warps first_extra.. are the extra gather warps
  if (gather_b && (warp == 0 || warp >= first_extra)) {
    // ------------------------------------------------ producer, B rows gathered --------
    // A (the compacted rows) still comes by TMA from warp 0's lane 0.  The B rows of a K slice
    // are pairs (or their tokens) named by kept_pair: the gather warps copy this CTA's 128
    // columns of the slice's 64 rows (row pairs split round-robin between them) with 16-byte
    // cp.async straight into the 128-byte-swizzled MN-major layout a TMA box would produce
    // (rows past the segment and columns past N are zero-filled).
    // Each lane's copies of a stage arrive on gathered[s] when they land; the lanes never wait.
    // The walk over (tile, K slice) is flat, and the next slice's row indices are loaded one
    // step ahead (across tiles too), so the copies never wait on an index load.
    const int gw = warp == 0 ? 0 : warp - first_extra + 1;  // this warp's share of the rows
    uint32_t it = 0, st = 0, sph = 0;
    bool ok = true;
    int last_e = -1;
    // pairs named by kept_pair for K rows r0 + lane and r0 + 32 + lane of a slice (-1 past the segment)
    auto load_idx = [&](const Tile& dd, int kbb, int& u0, int& u1) {
      const int r0 = dd.row0 + kbb * kBK;
      u0 = r0 + lane < dd.row_end ? gather_pair(p, r0 + lane) : -1;
      u1 = r0 + 32 + lane < dd.row_end ? gather_pair(p, r0 + 32 + lane) : -1;
    };
    int t = pair, kb = 0;
    Tile d{};
    bool have = false;
    for (; t < n_tiles; t += n_pairs) {
      d = decode(p, t, rank);
      if (d.k_iters > 0) { have = true; break; }
    }
    int cu0 = -1, cu1 = -1;
    if (have) load_idx(d, 0, cu0, cu1);
    while (have) {
      // the slice after this one, and its indices (used next step)
      int tn = t, kbn = kb + 1;
      Tile dn = d;
      bool haven = true;
      if (kbn >= d.k_iters) {
        kbn = 0;
        haven = false;
        for (tn = t + n_pairs; tn < n_tiles; tn += n_pairs) {
          dn = decode(p, tn, rank);
          if (dn.k_iters > 0) { haven = true; break; }
        }
      }
      int nu0 = -1, nu1 = -1;
      if (haven) load_idx(dn, kbn, nu0, nu1);

      const CUtensorMap* ma = p.maps_a + d.e;
      if (gw == 0 && lane == 0 && d.e != last_e) tensormap_acquire(ma);
      last_e = d.e;
      const uint32_t s = st, ph = sph;
      if (++st == (uint32_t)S) { st = 0; sph ^= 1u; }
      bool w = true;
      if (lane == 0) w = mbar_wait(empty0 + 8 * s, ph ^ 1u, abortv, p.status);
      if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) { ok = false; break; }
      const uint32_t a_dst = smem_u32(smem + s * kStageBytes), b_dst = a_dst + kABytes;
      const uint32_t fb = full_lead + 8 * s;
      const int r0 = d.row0 + kb * kBK;
      if (gw == 0 && lane == 0) {
        mbar_expect_tx_cluster(fb, d.has_rows ? kABytes : 0);
        if (d.has_rows) {
          if (p.merged_a) {
            tma_load_3d_pair(a_dst, ma, 0, r0, d.m0 / 64, fb);
          } else {
            tma_load_2d_pair(a_dst, ma, d.m0, r0, fb);
            tma_load_2d_pair(a_dst + 8192, ma, d.m0 + 64, r0, fb);
          }
        }
      }
      // source rows (pairs, or their tokens) of K rows lane and lane + 32
      const int sr0 = cu0 < 0 ? -1 : (p.gk > 0 ? cu0 / p.gk : cu0);
      const int sr1 = cu1 < 0 ? -1 : (p.gk > 0 ? cu1 / p.gk : cu1);
      // each instruction copies two rows' 256 contiguous bytes: half-warp hi = lane >> 4 takes
      // row 2j + hi, its lanes the 16 chunks (MN block b = chunk >> 3, 16-byte chunk c = chunk & 7)
      const int nb = d.n0 + rank * (kBN / 2);
      const int hi = lane >> 4, b = (lane >> 3) & 1, c = lane & 7;
      const int col = nb + b * 64 + c * 8;
      const bool col_live = col < p.N;
      for (int j = gw; j < 32; j += kGatherWarps) {
        const int l = 2 * j + hi;  // K row of the slice
        const int sr = __shfl_sync(0xffffffffu, l < 32 ? sr0 : sr1, l & 31);
        const bool live = col_live && sr >= 0;
        cp_async16(b_dst + b * 8192 + l * 128 + ((c ^ (l & 7)) << 4),
                   live ? p.gsrc + (int64_t)sr * p.gld + col : p.gsrc, live ? 16u : 0u);
      }
      cp_async_arrive_noinc(gath0 + 8 * s);
      ++it;
      t = tn;
      kb = kbn;
      d = dn;
      have = haven;
      cu0 = nu0;
      cu1 = nu1;
    }
    cp_async_wait_all();  // no copy may outlive the CTA (after an abort too)
    if (gw == 0 && lane == 0) {
      // drain: every stage this warp filled has been consumed
      const uint32_t first = it > (uint32_t)S ? it - S : 0u;
      for (uint32_t i = first; i < it; ++i) mbar_wait(empty0 + 8 * (i % S), (i / S) & 1u, abortv, p.status, false);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer -------
    // Both CTAs load their own 128 rows of A and their own 128 columns of B; the loads
    // complete on the leader's full barrier, which the leader's MMA waits on.
    if (lane == 0) {
      uint32_t it = 0, st = 0, sph = 0;  // iteration count, its stage and phase
      bool ok = true;
      int last_e = -1;
      // dynamic order: the leader's producer is the taker and publishes into both CTAs' rings
      const bool taker = seq.dyn && leader;
      const uint32_t rslots = cluster_addr(smem_u32(ring_slots), 1), rfull0 = cluster_addr(tfull0, 1);
      // The taker keeps the ring one tile ahead of its own loads: when it starts tile t, tile t's
      // successor is already published, and the tile after that is taken from the counter (the
      // atomic's round trip overlaps t's loads) and published once t's loads are queued.
      int t, t_next = n_tiles;
      if (taker) {
        t = seq.take(p.tile_counter);
        if (!seq.publish(t, rslots, rfull0)) t = -1;
        if (t >= 0 && t < n_tiles) {
          t_next = seq.take(p.tile_counter);
          if (!seq.publish(t_next, rslots, rfull0)) t = -1;
        }
      } else {
        t = seq.first(pair);
      }
      while (t >= 0 && t < n_tiles && ok) {
        const int t_after = taker && t_next < n_tiles ? seq.take(p.tile_counter) : n_tiles;
        const Tile d = decode(p, t, rank);
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
        const int nb = d.n0 + rank * (kBN / 2);  // this CTA's half of the B columns
        for (int kb = 0; kb < d.k_iters; ++kb, ++it) {
          const uint32_t s = st, ph = sph;
          if (++st == (uint32_t)S) { st = 0; sph ^= 1u; }
          if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abortv, p.status)) { ok = false; break; }
          const uint32_t a_dst = smem_u32(smem + s * kStageBytes), b_dst = a_dst + kABytes;
          const uint32_t fb = full_lead + 8 * s;
          mbar_expect_tx_cluster(fb, kBHalfBytes + (d.has_rows ? kABytes : 0));
          if (p.kind == VK) {
            const int r = d.row0 + kb * kBK;
            if (d.has_rows) {
              if (p.merged_a) {
                tma_load_3d_pair(a_dst, ma, 0, r, d.m0 / 64, fb);
              } else {
                tma_load_2d_pair(a_dst, ma, d.m0, r, fb);
                tma_load_2d_pair(a_dst + 8192, ma, d.m0 + 64, r, fb);
              }
            }
            if (p.merged_b) {
              tma_load_3d_pair(b_dst, mb, 0, r, nb / 64, fb);
            } else {
              tma_load_2d_pair(b_dst, mb, nb, r, fb);
              tma_load_2d_pair(b_dst + 8192, mb, nb + 64, r, fb);
            }
          } else if (p.kind == VM_FWD) {
            if (d.has_rows) tma_load_2d_pair(a_dst, &tmA, kb * kBK, d.row0, fb);
            // this CTA's 128 B rows (K-major): the expert's gate rows n0.. (leader) or its up rows
            // I + n0.. (the other CTA), so that the pair tile's columns are gate then matching up
            tma_load_3d_pair(b_dst, &tmB, kb * kBK, (rank == 0 ? 0 : p.N) + d.n0, d.e, fb);
          } else {
            if (d.has_rows) tma_load_2d_pair(a_dst, &tmA, kb * kBK, d.row0, fb);
            if (p.merged_b) {
              tma_load_4d_pair(b_dst, &tmB, 0, kb * kBK, nb / 64, d.e, fb);
            } else {
              tma_load_3d_pair(b_dst, &tmB, nb, kb * kBK, d.e, fb);
              tma_load_3d_pair(b_dst + 8192, &tmB, nb + 64, kb * kBK, d.e, fb);
            }
          }
        }
        if (!ok) break;
        if (taker) {
          if (t_next < n_tiles && !seq.publish(t_after, rslots, rfull0)) break;
          t = t_next;
          t_next = t_after;
        } else {
          t = seq.next();
        }
      }
      // drain: every stage this thread filled has been consumed (so its data landed)
      const uint32_t first = it > (uint32_t)S ? it - S : 0u;
      for (uint32_t i = first; i < it; ++i) mbar_wait(empty0 + 8 * (i % S), (i / S) & 1u, abortv, p.status, false);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer ---------
    // Only the leader issues: tcgen05.mma.cta_group::2 computes the 256 x 256 pair tile from
    // both CTAs' shared memory into both CTAs' TMEM (128 rows each).
    if (leader && lane == 0) {
      const bool b_kmajor = p.kind == VM_FWD;  // W_gate_up's rows, K contiguous
      const uint32_t idesc = instr_desc(p.kind == VK ? 1u : 0u, b_kmajor ? 0u : 1u);
      // descriptors of stage 0; a stage or a 16-deep K step is a constant offset in the address
      // field (addresses stay below 256 KB, so the 14-bit field never carries)
      const uint32_t a0 = smem_u32(smem), b0 = a0 + kABytes;
      const uint64_t adesc0 = p.kind == VK ? smem_desc(a0, 8192, 1024) : smem_desc(a0, 16, 1024);
      const uint64_t bdesc0 = b_kmajor ? smem_desc(b0, 16, 1024) : smem_desc(b0, 8192, 1024);
      const uint64_t a_kstep = p.kind == VK ? (2048 >> 4) : (32 >> 4);
      const uint64_t b_kstep = b_kmajor ? (32 >> 4) : (2048 >> 4);
      // the issue loop, compiled once per kind of B delivery (the loop is on the critical path)
      auto issue = [&](auto gather_tag) {
        constexpr bool G = decltype(gather_tag)::value;
        uint32_t st = 0, sph = 0;
        int lt = 0;
        bool ok = true;
        // the next tile is read before this one's MMAs are issued (it is published a tile ahead), so
        // no ring access sits between two tiles' MMAs
        int t = seq.first(pair);
        for (int tn; t >= 0 && t < n_tiles && ok; t = tn, ++lt) {
          tn = seq.next();
          const Tile d = decode(p, t, 0);
          const uint32_t acc = lt & 1, acc_ph = (lt >> 1) & 1;
          if (!mbar_wait(acce0 + 8 * acc, acc_ph ^ 1u, abortv, p.status)) break;
          tc_fence_after();
          const uint32_t tmem_d = tmem_base + acc * kBN;
          for (int kb = 0; kb < d.k_iters; ++kb) {
            const uint32_t s = st, ph = sph;
            if (++st == (uint32_t)S) { st = 0; sph ^= 1u; }
            if (!(G ? mbar_wait_cl(full0 + 8 * s, ph, abortv, p.status)
                    : mbar_wait(full0 + 8 * s, ph, abortv, p.status))) {
              ok = false;
              break;
            }
            if (G) {
              // this CTA's copied B rows have landed; make them visible to the tensor core (the
              // other CTA's were fenced by its relay before it arrived on full)
              if (!mbar_wait(gath0 + 8 * s, ph, abortv, p.status)) {
                ok = false;
                break;
              }
              fence_proxy_async_smem();
            }
            tc_fence_after();
            const uint64_t soff = (uint64_t)((s * kStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_bf16(tmem_d, adesc0 + soff + kk * a_kstep, bdesc0 + soff + kk * b_kstep, idesc,
                       (kb | kk) != 0 ? 1u : 0u);
            mma_commit_pair(empty0 + 8 * s);
          }
          if (!ok) break;
          mma_commit_pair(accf0 + 8 * acc);
        }
      };
      if (gather_b) issue(BoolTag<true>{});
      else issue(BoolTag<false>{});
      mma_commit_pair(drain);
    }
    if (!leader && gather_b && lane == 0) {
      // relay: once this CTA's copies of a stage have landed, fence them for the async proxy and
      // release them to the leader's MMA through its full barrier
      uint32_t st = 0, sph = 0;
      bool ok = true;
      for (int t = pair; t < n_tiles && ok; t += n_pairs) {
        const Tile d = decode(p, t, rank);
        for (int kb = 0; kb < d.k_iters; ++kb) {
          const uint32_t s = st, ph = sph;
          if (++st == (uint32_t)S) { st = 0; sph ^= 1u; }
          if (!mbar_wait(gath0 + 8 * s, ph, abortv, p.status)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
          mbar_arrive_release_cluster(full_lead + 8 * s);
        }
      }
    }
    __syncwarp();
    // drain: all MMAs writing this CTA's TMEM complete before it is released
    mbar_wait(drain, 0, abortv, p.status, false);
  } else if (warp >= 2 && warp < first_extra && p.kind == VM_FWD) {
    // ---------------------------------------------- epilogue, recomputed forward state ------
    // The pair tile's 256 accumulator columns are 128 gate columns (the leader's B rows) and then
    // the 128 matching up columns (the other CTA's).  Warp w reads TMEM lanes 32*(w%4) .. +31 (one
    // row per lane) and takes 64 of the gate columns with their up columns, 32 at a time: gate and
    // up are rounded to bf16 (the h row the forward stores), phi = SiLU(gate) * up is formed from
    // the rounded values as the forward's SwiGLU does, and the three 32 x 32 bf16 boxes (64-byte
    // swizzle) leave by TMA stores through the expert's maps (h_c as [rows][2][I], phi_c as
    // [rows][I]), whose row extent ends at the segment end.
    const int ew = warp - 2, q = warp & 3, half = ew >> 2;
    uint8_t* wbuf = epi + ew * epi_bytes<S>();
    const uint32_t wbuf_s = smem_u32(wbuf);
    const int swz = (lane >> 1) & 3;
    int last_e = -1;
    bool ok = true;
    int lt = 0;
    auto tile_at = [&](bool first) {  // lane 0 follows the pair's tile sequence for the warp
      int v = 0;
      if (lane == 0) v = first ? seq.first(pair) : seq.next();
      return __shfl_sync(0xffffffffu, v, 0);
    };
    for (int t = tile_at(true); t >= 0 && t < n_tiles && ok; t = tile_at(false), ++lt) {
      const Tile d = decode(p, t, rank);
      const uint32_t acc = lt & 1, acc_ph = (lt >> 1) & 1;
      const int row_base = d.row0 + q * 32;
      const int nrows = d.has_rows ? min(32, d.row_end - row_base) : 0;
      const CUtensorMap* hmap = p.maps_a + d.e;
      const CUtensorMap* fmap = p.maps_b + d.e;
      if (lane == 0 && nrows > 0 && d.e != last_e) {
        tensormap_acquire(hmap);
        tensormap_acquire(fmap);
        last_e = d.e;
      }
      if (!mbar_wait(accf0 + 8 * acc, acc_ph, abortv, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * kBN + ((uint32_t)(q * 32) << 16);
      for (int c2 = 0; c2 < 2 && nrows > 0; ++c2) {
        const int cc = half * 64 + c2 * 32;  // gate column within the tile
        const int col = d.n0 + cc;           // column of h's gate half and of phi
        if (col >= p.N) break;               // warp-uniform
        uint32_t vg[32], vu[32];
        tmem_ld32(tbase + cc, vg);
        tmem_ld32(tbase + kBN / 2 + cc, vu);
        if (lane == 0) bulk_wait_read_all();  // the previous chunk's stores have read the boxes
        __syncwarp();
        uint8_t* grow = wbuf + lane * 64;
        uint8_t* urow = grow + kVmBoxBytes;
        uint8_t* frow = grow + 2 * kVmBoxBytes;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          float gf[8], uf[8], fo[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            gf[i] = __uint_as_float(vg[8 * jj + i]);
            uf[i] = __uint_as_float(vu[8 * jj + i]);
          }
          const uint4 gq = pack(gf), uq = pack(uf);  // the stored gate / up values
          unpack(gq, gf);
          unpack(uq, uf);
#pragma unroll
          for (int i = 0; i < 8; ++i) fo[i] = gf[i] / (1.f + expf(-gf[i])) * uf[i];
          *reinterpret_cast<uint4*>(grow + ((jj ^ swz) << 4)) = gq;
          *reinterpret_cast<uint4*>(urow + ((jj ^ swz) << 4)) = uq;
          *reinterpret_cast<uint4*>(frow + ((jj ^ swz) << 4)) = pack(fo);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(hmap, wbuf_s, col, 0, row_base);
          tma_store_3d(hmap, wbuf_s + kVmBoxBytes, col, 1, row_base);
          tma_store_2d(fmap, wbuf_s + 2 * kVmBoxBytes, col, row_base);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce_lead + 8 * acc);
    }
    if (lane == 0) bulk_wait_all();  // stores complete before the CTA exits
  } else if (warp >= 2 && warp < first_extra && p.kind != VK && p.tma_epi) {
    // ---------------------------------------------------- epilogue, var-M through TMA -------
    // Warp w reads TMEM lanes 32*(w%4) .. +31 (tile rows q*32 .. +31) and half of the 256 columns,
    // 32 at a time, one row per lane.  A chunk's 32 x 32 results are packed to bf16 into a
    // 64-byte-swizzled box (16-byte piece j of row r at j ^ ((r >> 1) & 3)) and leave by one TMA
    // store per box through the expert's output map, which clips the rows past the segment end.
    // dphi + SwiGLU: the chunk's gate and up tiles arrive by TMA (issued one chunk ahead, the first
    // before the accumulator is ready) into the buffer the results then overwrite.
    const int ew = warp - 2, q = warp & 3, half = ew >> 2;
    const bool swiglu = p.kind == VM_SWIGLU;
    uint8_t* wbuf = epi + ew * (swiglu ? epi_bytes<S>() : kBoxBytes);
    const uint32_t wbuf_s = smem_u32(wbuf);
    const uint32_t hb0 = smem_u32(bars + 3 * S + 5 + 2 * ew);  // this warp's two gate/up buffer barriers
    const int swz = (lane >> 1) & 3;
    uint32_t h_next = 0, h_use = 0, n_st = 0;  // gate/up loads issued / consumed, dx stores issued
    int last_e = -1;
    bool ok = true;
    int lt = 0;
    auto tile_at = [&](bool first) {  // lane 0 follows the pair's tile sequence for the warp
      int v = 0;
      if (lane == 0) v = first ? seq.first(pair) : seq.next();
      return __shfl_sync(0xffffffffu, v, 0);
    };
    for (int t = tile_at(true); t >= 0 && t < n_tiles && ok; t = tile_at(false), ++lt) {
      const Tile d = decode(p, t, rank);
      const uint32_t acc = lt & 1, acc_ph = (lt >> 1) & 1;
      const int row_base = d.row0 + q * 32;
      const int nrows = d.has_rows ? min(32, d.row_end - row_base) : 0;
      int nch = 0;  // live 32-column chunks of this warp
      if (nrows > 0)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (d.n0 + (half * 4 + j) * 32 < p.N) nch = j + 1;
      const CUtensorMap* omap = p.maps_a + d.e;
      if (lane == 0 && nch > 0 && d.e != last_e) {
        tensormap_acquire(omap);
        last_e = d.e;
      }
      // lane 0: the gate and up boxes of chunk c into buffer h_next & 1 (whose previous contents
      // were last read by a TMA store, so that read completes first)
      auto issue_h = [&](int c) {
        const uint32_t b = h_next & 1u, buf = wbuf_s + b * 4096, bar = hb0 + 8 * b;
        bulk_wait_read_all();
        mbar_expect_tx(bar, 2 * kVmBoxBytes);
        tma_load_3d_cta(buf, &tmC, d.n0 + c * 32, 0, row_base, bar);
        tma_load_3d_cta(buf + kVmBoxBytes, &tmC, d.n0 + c * 32, 1, row_base, bar);
      };
      if (swiglu && nch > 0) {
        if (lane == 0) issue_h(half * 4);
        ++h_next;
      }
      if (!mbar_wait(accf0 + 8 * acc, acc_ph, abortv, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * kBN + ((uint32_t)(q * 32) << 16);
      // dphi . phi over this lane's row and the warp's columns, in four parts (one per 8-column
      // group of a chunk) added as (p0 + p1) + (p2 + p3): the same order as the other epilogue,
      // so that both row deliveries give bit-identical results
      float rp[4] = {0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < nch; ++j) {
        const int c = half * 4 + j, n = d.n0 + c * 32;
        if (swiglu && j + 1 < nch) {
          if (lane == 0) issue_h(c + 1);
          ++h_next;
        }
        uint32_t v[32];
        tmem_ld32(tbase + c * 32, v);
        if (swiglu) {
          const uint32_t g = h_use++;
          if (!__all_sync(0xffffffffu, mbar_wait(hb0 + 8 * (g & 1u), (g >> 1) & 1u, abortv, p.status))) {
            ok = false;
            break;
          }
          uint8_t* hbuf = wbuf + (g & 1u) * 4096;
          uint8_t* grow = hbuf + lane * 64;
          uint8_t* urow = grow + kVmBoxBytes;
          uint4 gq[4], uq[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            gq[jj] = *reinterpret_cast<const uint4*>(grow + ((jj ^ swz) << 4));
            uq[jj] = *reinterpret_cast<const uint4*>(urow + ((jj ^ swz) << 4));
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            float gate[8], up[8], dg[8], du[8];
            unpack(gq[jj], gate);
            unpack(uq[jj], up);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float dphi = __uint_as_float(v[8 * jj + i]);
              const float sg = 1.f / (1.f + __expf(-gate[i]));
              dg[i] = dphi * up[i] * sg * (1.f + gate[i] * (1.f - sg));
              du[i] = dphi * gate[i] * sg;
              if (n + 8 * jj + i < p.N) rp[jj] = fmaf(du[i], up[i], rp[jj]);
            }
            *reinterpret_cast<uint4*>(grow + ((jj ^ swz) << 4)) = pack(dg);
            *reinterpret_cast<uint4*>(urow + ((jj ^ swz) << 4)) = pack(du);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(omap, smem_u32(hbuf), n, 0, row_base);
            tma_store_3d(omap, smem_u32(hbuf) + kVmBoxBytes, n, 1, row_base);
          }
        } else {
          uint8_t* box = wbuf + (n_st & 1u) * kVmBoxBytes;
          ++n_st;
          if (lane == 0) bulk_wait_read_le1();  // the store before last (this box's) has read it
          __syncwarp();
          uint8_t* row = box + lane * 64;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(v[8 * jj + i]);
            *reinterpret_cast<uint4*>(row + ((jj ^ swz) << 4)) = pack(f);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) tma_store_2d(omap, smem_u32(box), n, row_base);
        }
      }
      if (!ok) break;
      if (swiglu && p.dot_part != nullptr && nch > 0 && lane < nrows)
        p.dot_part[(int64_t)(row_base + lane) * p.n_part + d.n0 / 128 + half] = (rp[0] + rp[1]) + (rp[2] + rp[3]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce_lead + 8 * acc);
    }
    // no gate/up load may land, and no store may read, after the CTA has exited
    for (uint32_t g = h_use; g < h_next; ++g)
      mbar_wait(hb0 + 8 * (g & 1u), (g >> 1) & 1u, abortv, p.status, false);
    if (lane == 0) bulk_wait_all();
  } else if (warp >= 2 && warp < first_extra) {
    // ------------------------------------------------------------ epilogue -----------
    // var-K (fp32 dW through TMA stores) and var-M of the compaction-free variant, whose gate/up
    // rows are named by kept_pair and so cannot come as TMA tiles.
    // Warp w may read TMEM lanes 32*(w%4) .. +31 (tile rows q*32 .. q*32+31); the two warps
    // of a quarter split the eight 32-column chunks.  Each chunk is read row-per-thread
    // (tcgen05.ld 32x32b); var-M chunks are staged in shared memory and written back
    // row-contiguous, so global stores (and the SwiGLU gate/up loads) are coalesced, masked at
    // the segment end.
    const int ew = warp - 2, q = warp & 3, half = ew >> 2;
    const int sub = lane >> 2, piece = lane & 3;  // var-M stores: lane owns 8 columns of one row
    float* stg = reinterpret_cast<float*>(epi + ew * (p.kind == VK ? kBoxBytes : epi_bytes<S>()));
    int lt = 0;
    auto tile_at = [&](bool first) {  // lane 0 follows the pair's tile sequence for the warp
      int v = 0;
      if (lane == 0) v = first ? seq.first(pair) : seq.next();
      return __shfl_sync(0xffffffffu, v, 0);
    };
    for (int t = tile_at(true); t >= 0 && t < n_tiles; t = tile_at(false), ++lt) {
      const Tile d = decode(p, t, rank);
      const uint32_t acc = lt & 1, acc_ph = (lt >> 1) & 1;
      const int row_base = p.kind == VK ? d.m0 + q * 32 : d.row0 + q * 32;
      const int row_lim = p.kind == VK ? p.M : d.row_end;
      const int nrows = d.has_rows ? min(32, row_lim - row_base) : 0;
      if (p.kind == VM_SWIGLU && lane < nrows) {
        // while the tile's MMAs run, pull this warp's gate and up rows (its 128 columns of
        // each) into L2, so that the SwiGLU epilogue below reads them from L2
        const int I = p.N, col = d.n0 + half * 128;
        const int64_t hr = p.kept_pair ? (int64_t)gather_pair(p, row_base + lane) : (int64_t)(row_base + lane);
        const __nv_bfloat16* hrow = (p.kept_pair ? p.gsrc : p.h_c) + hr * 2 * I;
        if (col < I && hr >= 0) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            if (col + b * 64 >= I) break;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(hrow + col + b * 64));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(hrow + I + col + b * 64));
          }
        }
      }
      if (!mbar_wait(accf0 + 8 * acc, acc_ph, abortv, p.status)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * kBN + ((uint32_t)(q * 32) << 16);
      const bool have_acc = d.k_iters > 0;
      // VM_SWIGLU: this lane's part of dphi . phi for rows i*8 + sub over its columns, where
      // dphi . phi = sum of dup * up (dup = dphi * gate * s, phi = gate * s * up)
      float rdot[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = half * 4; c < half * 4 + 4 && nrows > 0; ++c) {
        const int n = d.n0 + c * 32;
        if (n >= p.N) break;  // warp-uniform
        uint32_t v[32];
        if (have_acc) tmem_ld32(tbase + c * 32, v);
        else
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        if (p.kind == VK) {
          // fp32 dW: the warp's 32 x 32 block leaves as two 32-row x 16-column TMA tensor stores
          // from two 2 KB, 64-byte-swizzled staging boxes used in turn, so that a warp always has
          // one store in flight while it fills the other box (the map clips rows >= M, columns >= N)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint8_t* box = reinterpret_cast<uint8_t*>(stg) + hh * 2048;
            if (lane == 0) bulk_wait_read_le1();  // the store before last (this box's) has read it
            __syncwarp();
            uint8_t* line = box + lane * 64;
            const int sw = (lane >> 1) & 3;  // 64-byte swizzle: 16-byte chunk j of row r -> j ^ ((r >> 1) & 3)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              *reinterpret_cast<uint4*>(line + ((jj ^ sw) << 4)) =
                  make_uint4(v[16 * hh + 4 * jj], v[16 * hh + 4 * jj + 1], v[16 * hh + 4 * jj + 2],
                             v[16 * hh + 4 * jj + 3]);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tma_store_3d(&tmC, smem_u32(box), n + 16 * hh, row_base, d.e);
          }
          continue;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) stg[lane * kVmLd + i] = __uint_as_float(v[i]);
        __syncwarp();
        {
          // bf16 rows: 8 rows x 64 B per instruction; lane owns 8 columns of one row
          const int col = n + piece * 8;
          if (p.kind == VM_SWIGLU) {
            const int I = p.N;
            uint4 gv[4], uv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = i * 8 + sub;
              if (rr < nrows && col < I) {
                // gate/up row: the compacted row, or (compaction-free) the pair's row of h
                const int64_t hr =
                    p.kept_pair ? (int64_t)gather_pair(p, row_base + rr) : (int64_t)(row_base + rr);
                const __nv_bfloat16* hrow = (p.kept_pair ? p.gsrc : p.h_c) + hr * 2 * I;
                gv[i] = hr >= 0 ? ldg16(hrow + col) : make_uint4(0, 0, 0, 0);
                uv[i] = hr >= 0 ? ldg16(hrow + I + col) : make_uint4(0, 0, 0, 0);
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
                  rdot[i] = fmaf(du[j], up[j], rdot[i]);
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
      if (p.kind == VM_SWIGLU && p.dot_part != nullptr && nrows > 0 && d.n0 + half * 128 < p.N) {
        // warp-uniform; the four lanes of a row add their parts in a fixed order
        const int part = d.n0 / 128 + half;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          rdot[i] += __shfl_xor_sync(0xffffffffu, rdot[i], 1);
          rdot[i] += __shfl_xor_sync(0xffffffffu, rdot[i], 2);
          const int rr = i * 8 + sub;
          if (piece == 0 && rr < nrows) p.dot_part[(int64_t)(row_base + rr) * p.n_part + part] = rdot[i];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce_lead + 8 * acc);
    }
    if (p.kind == VK && lane == 0) bulk_wait_all();  // stores complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no multicast or remote arrive may target a CTA that has exited
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Tile tables from seg_offsets: plan[0..E] = exclusive prefix of ceil(R_e / 256) (var-M pair tiles),
// plan[E+1 .. 2E] = experts ordered by R_e descending, ties by expert id (var-K, longest first),
// plan[2E+2] = 1 for the dynamic tile order of the var-K launches (mean rows per expert at least
// kDynMinRowsPerExpert), plan[2E+3 ..] = their tile counters (zeroed here),
// plan[2E+1] = 1 if seg_offsets is a segmentation of [0, seg_offsets[E]] within [0, cap]
// (seg_offsets[0] = 0, no decreasing step, seg_offsets[E] <= cap), else 0: then
// LRM_ERR_BAD_SEGMENTS is recorded and the GEMM launches run no tile (total_tiles), so no map
// built from the bad offsets is ever used.
// maps[j][e] = template j with its row extent cut at seg_offsets[e+1] (var-K operands, var-M outputs).
// Templates 0-3: var-K operands (row extent is dimension 1); 4: dh_c as [rows][2][I] (rows are
// dimension 2); 5: dx_c as [rows][H] (dimension 1).
constexpr int kMapSets = 6;
constexpr int kDynMinRowsPerExpert = 1024;
struct MapTemplates {
  CUtensorMap t[kMapSets];
};
__global__ void __launch_bounds__(1024) tc_plan_kernel(const int32_t* __restrict__ seg, int E, int64_t cap,
                                                       int32_t* __restrict__ plan, CUtensorMap* __restrict__ maps,
                                                       const __grid_constant__ MapTemplates tpl,
                                                       int32_t* __restrict__ status) {
  chain_wait();
  __shared__ int s_r[LRM_MAX_EXPERTS];
  __shared__ int warp_tot[32];
  const int e = threadIdx.x;
  bool good = true;
  if (e < E) good = seg[e] <= seg[e + 1];
  if (e == 0) good = good && seg[0] == 0;
  if (e == E - 1) good = good && (int64_t)seg[E] <= cap;
  const bool valid = __syncthreads_and(good ? 1 : 0) != 0;
  if (e == 0) {
    plan[2 * E + 1] = valid ? 1 : 0;
    if (!valid) set_status(status, LRM_ERR_BAD_SEGMENTS);
    // dynamic tile order for the var-K launches when their tiles are long (TileSeq): below this
    // mean the ring's round trip per tile costs more than the L2 reuse it buys
    plan[2 * E + 2] = valid && (int64_t)seg[E] >= (int64_t)kDynMinRowsPerExpert * E ? 1 : 0;
  }
  if (e < kTileCounters) plan[2 * E + 3 + e] = 0;  // the var-K launches' tile counters
  const int r = e < E && valid ? seg[e + 1] - seg[e] : 0;
  if (e < E) s_r[e] = r;
  const int mt = (r + 2 * kBM - 1) / (2 * kBM);
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
  }
  // one (template, expert) map per thread
  for (int i = threadIdx.x; i < kMapSets * E; i += blockDim.x) {
    const int j = i / E, ee = i - j * E;
    const uint32_t rows_end = valid ? (uint32_t)max(1, seg[ee + 1]) : 1u;
    {
      CUtensorMap* dst = maps + j * E + ee;
      const uint4* src = reinterpret_cast<const uint4*>(&tpl.t[j]);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int w = 0; w < 8; ++w) d4[w] = src[w];
      if (j == 4)
        asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 2, %1;" ::"l"(
                         reinterpret_cast<uint64_t>(dst)),
                     "r"(rows_end)
                     : "memory");
      else
        asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(
                         reinterpret_cast<uint64_t>(dst)),
                     "r"(rows_end)
                     : "memory");
    }
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing will ever arrive
// on.  The wait must give up after `limit_ns`, record LRM_ERR_TIMEOUT and return normally.
__global__ void wait_selftest_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  mbar_wait_slow(b, 0, &abort_flag, status, true, limit_ns);  // phase 0 never completes
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

// bf16 row-major [rows, cols] viewed as [cols / 64 blocks][rows][64] with a {64, 64, 2} box: one box
// fills a CTA's two 64-column blocks of a 64-line K slice (cols a multiple of 64).
bool make_map_blocks_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  const cuuint64_t dims[3] = {64, rows, cols / 64};
  const cuuint64_t strides[2] = {cols * 2, 128};
  const cuuint32_t box[3] = {64, 64, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// bf16 [E, K, N] viewed as [E][N / 64 blocks][K][64] with a {64, 64, 2, 1} box (N a multiple of 64).
bool make_map_blocks_3d(CUtensorMap* m, const void* base, uint64_t E, uint64_t K, uint64_t N) {
  const cuuint64_t dims[4] = {64, K, N / 64, E};
  const cuuint64_t strides[3] = {N * 2, 128, K * N * 2};
  const cuuint32_t box[4] = {64, 64, 2, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// bf16 [E, rows, K] (K contiguous: the rows of W_gate_up) with a {64, 128, 1} box, 128-byte swizzle.
bool make_map_kmajor_3d(CUtensorMap* m, const void* base, uint64_t E, uint64_t rows, uint64_t K) {
  const cuuint64_t dims[3] = {K, rows, E};
  const cuuint64_t strides[2] = {K * 2, rows * K * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// bf16 [rows][2][I] (gate / up halves of a row, e.g. h_c or dh_c) with a {32, 1, 32} box,
// 64-byte swizzle: one box is 32 columns of one half for 32 rows.
bool make_map_halves(CUtensorMap* m, const void* base, uint64_t rows, uint64_t I) {
  const cuuint64_t dims[3] = {I, 2, rows};
  const cuuint64_t strides[2] = {I * 2, I * 4};
  const cuuint32_t box[3] = {32, 1, 32};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// bf16 [rows][cols] with a {32, 32} box, 64-byte swizzle.
bool make_map_rows32(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// Column counts whose 64-column blocks may share one box (see TcParams::merged_a).
bool mergeable(uint64_t cols) { return cols % 64 == 0 && cols >= 128; }

// fp32 [E, M, N] output with a {16, 32, 1} box and 64-byte swizzle (the epilogue's 2 KB staging boxes).
bool make_map_out3d(CUtensorMap* m, void* base, uint64_t E, uint64_t M, uint64_t N) {
  const cuuint64_t dims[3] = {N, M, E};
  const cuuint64_t strides[2] = {N * 4, M * N * 4};
  const cuuint32_t box[3] = {16, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int S>
size_t smem_bytes() { return 1024 + bar_offset<S>() + n_barriers<S>() * 8 + 8 + 4 * kRing; }

int sm_count() {
  static int count[kDeviceSlots] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int d = current_device_slot();
  int n = d >= 0 ? count[d] : 0;
  if (n == 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
    if (d >= 0) count[d] = n;
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

template <int S, bool RING>
lrm_status launch_stages(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c, const TcParams& p,
                         int64_t tiles_bound, cudaStream_t s) {
  const size_t smem = smem_bytes<S>();
  if (ensure_max_smem<tc_grouped_kernel<S, RING>>((int)smem) != cudaSuccess) return LRM_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see chain_wait()
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the extra gather warps are launched only where B rows are gathered
  cfg.blockDim = dim3(p.kind == VK && p.kept_pair != nullptr ? kThreads : kThreads - 32 * kGatherExtraWarps);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // the occupancy query sees the cluster shape only
  static int max_pairs_dev[kDeviceSlots] = {};  // resident CTA pairs, per device
  const int dslot = current_device_slot();
  int max_pairs = dslot >= 0 ? max_pairs_dev[dslot] : 0;
  if (max_pairs == 0) {
    cfg.gridDim = dim3(2 * sm_count() / 2);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_grouped_kernel<S, RING>, &cfg) != cudaSuccess || n <= 0) n = sm_count() / 2;
    max_pairs = n;
    if (dslot >= 0) max_pairs_dev[dslot] = n;
  }
  cfg.numAttrs = 2;
  const int64_t pairs = tiles_bound < max_pairs ? tiles_bound : max_pairs;
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  if (cudaLaunchKernelEx(&cfg, tc_grouped_kernel<S, RING>, a, b, c, p) != cudaSuccess) return LRM_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? LRM_OK : LRM_ERR_CUDA;
}

lrm_status launch_one(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c, const TcParams& p,
                      int64_t tiles_bound, cudaStream_t s) {
  if (tiles_bound <= 0) return LRM_OK;
  // dphi + SwiGLU and the recomputed forward state need the wide per-warp epilogue buffers
  if (p.kind == VK) return launch_stages<kStages, true>(a, b, c, p, tiles_bound, s);
  return p.kind == VM_SWIGLU || p.kind == VM_FWD ? launch_stages<kSwigluStages, false>(a, b, c, p, tiles_bound, s)
                                                 : launch_stages<kStages, false>(a, b, c, p, tiles_bound, s);
}

}  // namespace

lrm_status launch_recompute_tc(const RecomputeArgs& g, const GemmWs& ws, cudaStream_t s) {
  if (!device_ok() || encode_fn() == nullptr) return LRM_ERR_UNSUPPORTED;
  const int E = g.E, H = g.H, I = g.I;
  const uint64_t rows = g.cap > 0 ? (uint64_t)g.cap : 1;
  int32_t* plan = ws.plan;
  CUtensorMap* maps = static_cast<CUtensorMap*>(ws.maps);
  // per-expert output maps: set 4 = h_c as [rows][2][I], set 5 = phi_c as [rows][I] (the plan
  // kernel cuts both at the segment end); sets 0-3 are not used here and only need to be valid
  MapTemplates tpl;
  if (!make_map_halves(&tpl.t[4], g.h_c, rows, I) || !make_map_rows32(&tpl.t[5], g.phi_c, rows, I))
    return LRM_ERR_CUDA;
  for (int j = 0; j < 4; ++j) tpl.t[j] = tpl.t[5];
  launch_chained(tc_plan_kernel, dim3(1), dim3(1024), 0, s, g.seg_offsets, E, g.cap, plan, maps, tpl, g.status);
  if (cudaGetLastError() != cudaSuccess) return LRM_ERR_CUDA;
  CUtensorMap mA, mB;
  if (!make_map_2d(&mA, g.x_c, rows, H, kBM) || !make_map_kmajor_3d(&mB, g.w_gate_up, E, 2 * (uint64_t)I, H))
    return LRM_ERR_CUDA;
  TcParams p{VM_FWD, E, 0, I, H, 0, (I + kBN / 2 - 1) / (kBN / 2), g.seg_offsets, plan, nullptr, nullptr, g.status,
             maps + 4 * E, maps + 5 * E};
  p.tma_epi = 1;
  const int64_t vm_bound = ((int64_t)g.cap + 2 * kBM - 1) / (2 * kBM) + E;
  return launch_one(mA, mB, mA, p, vm_bound * p.nN, s);
}

lrm_status launch_wait_selftest(int32_t* status, int64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, (uint64_t)limit_ns);
  return cudaGetLastError() == cudaSuccess ? LRM_OK : LRM_ERR_CUDA;
}

lrm_status launch_grouped_tc(const GroupedArgs& g, const GemmWs& ws, cudaStream_t s) {
  if (!device_ok() || encode_fn() == nullptr) return LRM_ERR_UNSUPPORTED;
  const int E = g.E, H = g.H, I = g.I;
  const uint64_t rows = g.cap > 0 ? (uint64_t)g.cap : 1;
  int32_t* plan = ws.plan;  // [2E+2] tile tables and the segment check word
  CUtensorMap* maps = static_cast<CUtensorMap*>(ws.maps);
  MapTemplates tpl;
  const bool gather = g.kept_pair != nullptr;  // compaction-free: phi / x rows gathered by index
  // (gathering, the B templates are never used; they are encoded over dy_c only to stay valid)
  // var-K operand maps (MN-major): one box per CTA and K slice where the column count allows (the
  // two-box form otherwise, or if the driver declines the blocked view)
  bool merged[4];
  auto vk_map = [&](int j, const void* base, uint64_t cols) {
    merged[j] = mergeable(cols) && make_map_blocks_2d(&tpl.t[j], base, rows, cols);
    return merged[j] || make_map_2d(&tpl.t[j], base, rows, cols, 64);
  };
  if (!vk_map(0, g.dy_c, H) || !vk_map(1, gather ? g.dy_c : g.phi_c, I) || !vk_map(2, g.dh_c, 2 * I) ||
      !vk_map(3, gather ? g.dy_c : g.x_c, H))
    return LRM_ERR_CUDA;
  // var-M outputs (per-expert copies clip the rows past the segment end)
  if (!make_map_halves(&tpl.t[4], g.dh_c, rows, I) || !make_map_rows32(&tpl.t[5], g.dx_c, rows, H))
    return LRM_ERR_CUDA;
  const int tma_epi = gather ? 0 : 1;  // compacted rows: var-M epilogue through TMA
  // var-M weight maps: [E, K, N], blocked the same way where N allows
  auto vm_map = [&](CUtensorMap* m, const void* base, uint64_t K, uint64_t N, int* merged_b) {
    *merged_b = mergeable(N) && make_map_blocks_3d(m, base, E, K, N);
    return *merged_b || make_map_3d(m, base, E, K, N);
  };
  launch_chained(tc_plan_kernel, dim3(1), dim3(1024), 0, s, g.seg_offsets, E, g.cap, plan, maps, tpl, g.status);
  if (cudaGetLastError() != cudaSuccess) return LRM_ERR_CUDA;

  CUtensorMap mA, mB;
  const int64_t vm_bound = ((int64_t)g.cap + 2 * kBM - 1) / (2 * kBM) + E;  // pair tiles along M
  lrm_status st;
  // dphi = dy_c W_down[e], SwiGLU backward fused -> dh_c
  int vm_merged = 0;
  if (!make_map_2d(&mA, g.dy_c, rows, H, kBM) || !vm_map(&mB, g.w_down, H, I, &vm_merged)) return LRM_ERR_CUDA;
  using B16 = const __nv_bfloat16*;
  TcParams p{VM_SWIGLU, E, 0, I, H, 0, (I + kBN - 1) / kBN, g.seg_offsets, plan, g.dh_c,
             (B16)g.h_c, g.status, maps + 4 * E, nullptr, g.dot_part, (I + 127) / 128,
             g.kept_pair, gather ? (B16)g.h : nullptr, 0, 2 * I, 0, vm_merged, tma_epi, (int)g.n_pairs};
  CUtensorMap mH = mA;  // gate/up tiles of h_c for the TMA epilogue
  if (tma_epi && !make_map_halves(&mH, g.h_c, rows, I)) return LRM_ERR_CUDA;
  if ((st = launch_one(mA, mB, mH, p, vm_bound * p.nN, s))) return st;
  if (g.row_dot != nullptr) launch_row_dot(g.dot_part, p.n_part, g.seg_offsets, E, g.cap, g.row_dot, s);
  // dW_down[e] = dy_c^T phi_c  (M = H, N = I)
  p = TcParams{VK, E, H, I, 0, (H + kBM - 1) / kBM, (I + kBN - 1) / kBN, g.seg_offsets, plan, g.dw_down,
               nullptr, g.status, maps + 0 * E, maps + 1 * E, nullptr, 0,
               g.kept_pair, gather ? (B16)g.phi : nullptr, 0, I, merged[0], merged[1], 0, (int)g.n_pairs};
  mA = tpl.t[0];
  mB = tpl.t[1];
  CUtensorMap mC;
  if (!make_map_out3d(&mC, g.dw_down, E, H, I)) return LRM_ERR_CUDA;
  int32_t* counters = plan + 2 * E + 3;  // zeroed by the plan kernel
  p.tile_counter = counters + 0;
  if ((st = launch_one(mA, mB, mC, p, (int64_t)E * ((p.nM + 1) / 2) * p.nN, s))) return st;
  // dW_gate_up[e] = dh_c^T x_c  (M = 2I, N = H)
  p = TcParams{VK, E, 2 * I, H, 0, (2 * I + kBM - 1) / kBM, (H + kBN - 1) / kBN, g.seg_offsets, plan,
               g.dw_gate_up, nullptr, g.status, maps + 2 * E, maps + 3 * E, nullptr, 0,
               g.kept_pair, gather ? (B16)g.x : nullptr, g.k, H, merged[2], merged[3], 0, (int)g.n_pairs};
  mA = tpl.t[2];
  mB = tpl.t[3];
  if (!make_map_out3d(&mC, g.dw_gate_up, E, 2 * I, H)) return LRM_ERR_CUDA;
  p.tile_counter = counters + 1;
  if ((st = launch_one(mA, mB, mC, p, (int64_t)E * ((p.nM + 1) / 2) * p.nN, s))) return st;
  // dx_c = dh_c W_gate_up[e]  (K = 2I, N = H)
  if (!make_map_2d(&mA, g.dh_c, rows, 2 * I, kBM) || !vm_map(&mB, g.w_gate_up, 2 * I, H, &vm_merged))
    return LRM_ERR_CUDA;
  p = TcParams{VM_STORE, E, 0, H, 2 * I, 0, (H + kBN - 1) / kBN, g.seg_offsets, plan, g.dx_c, nullptr,
               g.status, maps + 5 * E, nullptr};
  p.merged_b = vm_merged;
  p.tma_epi = tma_epi;
  if ((st = launch_one(mA, mB, mA, p, vm_bound * p.nN, s))) return st;
  return LRM_OK;
}

}  // namespace lrm
