// Per-expert top-quota selection.
//
// "LRMoE poda a passagem reversa do MoE..." (news.hamidun.com), step "Seleção pela métrica
// LRM": inside each expert's quota the highest-scoring pairs are kept.  Equal scores go to
// the smaller pair index u; inside a segment the kept pairs are listed in u order.
//
// Four launches, all deterministic:
//  1. count:   one CTA per chunk of kSelChunk consecutive pairs counts the chunk's experts.
//  2. scan:    one CTA per expert: exclusive scan of that expert's chunk counts (bucket
//              bases inside the expert's bucket) and its load.
//  3. bucket:  one CTA per chunk derives the expert-level prefixes (bucket starts, kept counts
//              min(quota, load), segment offsets, capacity check; CTA 0 publishes them),
//              then scatters its pairs stably into the expert buckets (u ascending) with
//              their score bits: ranks within a warp from __match_any_sync, across warps from
//              per-warp expert counts.
//  4. expert:  one CTA per expert (1024 threads, the bucket's keys held in shared memory
//              when they fit): MSD radix select (up to 4 x 8 bits, stopping early once the
//              bin of the quota-th largest score is kept whole) of that score, then one
//              ordered pass that keeps everything above the threshold plus the first `need`
//              pairs equal to it, and writes kept_pair and row_of_pair through a block-wide
//              prefix sum.
// Scores are finite and >= 0, so their IEEE bit patterns order like their values.
#include "common.cuh"
#include "kernels.h"

namespace lrm {

namespace {

// Exclusive block-wide prefix sum of one int per thread (blockDim.x a multiple of 32, <= 1024).
// `sm` needs 33 ints.  Returns the exclusive prefix; *total receives the block total.
__device__ __forceinline__ int block_excl_scan(int v, int* total, int* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? sm[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) sm[lane] = wi - w;
    if (lane == 31) sm[32] = wi;
  }
  __syncthreads();
  const int res = sm[warp] + incl - v;
  *total = sm[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kSelChunk) sel_count_kernel(const int32_t* __restrict__ idx, int64_t P, int E,
                                                              int32_t* __restrict__ counts, int32_t* status) {
  extern __shared__ int hist[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t c = blockIdx.x;
  const int64_t u = c * kSelChunk + threadIdx.x;
  const int e = u < P ? idx[u] : -1;
  const bool good = u < P && e >= 0 && e < E;
  if (u < P && !good) set_status(status, LRM_ERR_BAD_INDEX);
  // warp-aggregated: one shared atomic per distinct expert in the warp
  const unsigned peers = __match_any_sync(0xffffffffu, good ? e : -1);
  if (good && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[e], __popc(peers));
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[c * E + e] = hist[e];
}

// One CTA per expert: exclusive scan down the expert's column of chunk counts.
__global__ void __launch_bounds__(1024) sel_colscan_kernel(int32_t* __restrict__ counts, int64_t n_chunks, int E,
                                                           int32_t* __restrict__ loads) {
  __shared__ int sm[33];
  __shared__ int s_run;
  const int e = blockIdx.x;
  if (threadIdx.x == 0) s_run = 0;
  __syncthreads();
  for (int64_t c0 = 0; c0 < n_chunks; c0 += blockDim.x) {
    const int64_t c = c0 + threadIdx.x;
    const int v = c < n_chunks ? counts[c * E + e] : 0;
    int tot;
    const int ex = block_excl_scan(v, &tot, sm);
    if (c < n_chunks) counts[c * E + e] = s_run + ex;
    __syncthreads();
    if (threadIdx.x == 0) s_run += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) loads[e] = s_run;
}

__global__ void __launch_bounds__(kSelChunk) sel_bucket_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ scores, int64_t P, int E, int64_t n_chunks,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ loads, const int32_t* __restrict__ quotas,
    int64_t cap, int32_t* __restrict__ bucket_start, int32_t* __restrict__ keep, int32_t* __restrict__ seg_offsets,
    int32_t* __restrict__ sorted_u, uint32_t* __restrict__ sorted_key, int32_t* __restrict__ row_of_pair,
    int32_t* status) {
  constexpr int kWarps = kSelChunk / 32;
  extern __shared__ int sh[];
  int* s_base = sh;              // [E]  this chunk's first slot of each expert
  int* s_wcnt = sh + E;          // [kWarps][E] per-warp counts, then per-warp exclusive offsets
  int* s_seg = sh + E + kWarps * E;  // [E] segment starts (block 0 publishes)
  __shared__ int sm[33];
  __shared__ int s_base_l, s_base_k, s_overflow;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t c = blockIdx.x;

  // this thread's pair (issued first so its latency overlaps the prefix work below)
  const int64_t u = c * kSelChunk + tid;
  const bool valid = u < P;
  const int e_raw = valid ? idx[u] : -1;
  const bool good = valid && e_raw >= 0 && e_raw < E;
  const uint32_t key = good ? __float_as_uint(scores[u]) : 0u;

  // expert-level prefixes: bucket starts, kept counts, segment offsets (E <= 1024)
  if (tid == 0) { s_base_l = 0; s_base_k = 0; }
  for (int i = tid; i < kWarps * E; i += kSelChunk) s_wcnt[i] = 0;
  __syncthreads();
  int kp_mine[4];
  for (int r = 0; r < (E + kSelChunk - 1) / kSelChunk; ++r) {
    const int e = r * kSelChunk + tid;
    const int l = e < E ? loads[e] : 0;
    int kp = 0;
    if (e < E) {
      const int q = quotas[e];
      kp = q < 0 ? 0 : (q > l ? l : q);
    }
    kp_mine[r] = kp;
    int tl, tk;
    const int xl = block_excl_scan(l, &tl, sm);
    const int xk = block_excl_scan(kp, &tk, sm);
    if (e < E) {
      s_base[e] = s_base_l + xl + (c < n_chunks ? counts[c * E + e] : 0);
      s_seg[e] = s_base_k + xk;
    }
    __syncthreads();
    if (tid == 0) { s_base_l += tl; s_base_k += tk; }
    __syncthreads();
  }
  if (tid == 0) s_overflow = (int64_t)s_base_k > cap;
  __syncthreads();
  const bool overflow = s_overflow;
  if (blockIdx.x == 0) {
    for (int r = 0; r < (E + kSelChunk - 1) / kSelChunk; ++r) {
      const int e = r * kSelChunk + tid;
      if (e < E) {
        bucket_start[e] = s_base[e];  // block 0 is chunk 0, whose offset inside every bucket is 0
        keep[e] = overflow ? 0 : kp_mine[r];
        seg_offsets[e] = overflow ? 0 : s_seg[e];
      }
    }
    if (tid == 0) {
      bucket_start[E] = s_base_l;
      seg_offsets[E] = overflow ? 0 : s_base_k;
      if (overflow) set_status(status, LRM_ERR_CAPACITY);
    }
  }

  // stable rank of this pair among the chunk's pairs of the same expert (u order)
  const unsigned peers = __match_any_sync(0xffffffffu, good ? e_raw : -1);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  if (good && rank_w == 0) s_wcnt[warp * E + e_raw] = __popc(peers);
  __syncthreads();
  for (int e = tid; e < E; e += kSelChunk) {  // per expert: exclusive offsets over the warps
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int v = s_wcnt[w * E + e];
      s_wcnt[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  if (valid && !good) row_of_pair[u] = -1;
  if (good) {
    const int pos = s_base[e_raw] + s_wcnt[warp * E + e_raw] + rank_w;
    sorted_u[pos] = (int32_t)u;
    sorted_key[pos] = key;
  }
}

constexpr int kExpThreads = 1024;
constexpr int kExpIPT = 8;  // bucket elements per thread per round
// A bucket of up to this many keys is copied into shared memory once and every pass reads it
// there (192 KB); a larger one is read from global memory on every pass.
constexpr int kExpSmemKeys = 49152;

__global__ void __launch_bounds__(kExpThreads) sel_expert_kernel(
    const int32_t* __restrict__ bucket_start, const int32_t* __restrict__ keep_arr,
    const int32_t* __restrict__ seg_offsets, const int32_t* __restrict__ sorted_u,
    const uint32_t* __restrict__ sorted_key, int32_t* __restrict__ kept_pair, int32_t* __restrict__ row_of_pair) {
  extern __shared__ uint32_t s_keys[];  // [kExpSmemKeys]
  __shared__ int sm[33];
  __shared__ int hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need, s_whole;
  const int e = blockIdx.x, tid = threadIdx.x;
  const int b0 = bucket_start[e];
  const int load = bucket_start[e + 1] - b0;
  const int keep = keep_arr[e];
  const int base = seg_offsets[e];
  const int32_t* bu = sorted_u + b0;
  const uint32_t* bk = sorted_key + b0;

  if (keep >= load) {
    for (int i = tid; i < load; i += kExpThreads) {
      const int u = bu[i];
      kept_pair[base + i] = u;
      row_of_pair[u] = base + i;
    }
    return;
  }
  if (keep <= 0) {
    for (int i = tid; i < load; i += kExpThreads) row_of_pair[bu[i]] = -1;
    return;
  }

  // the keys every pass reads: a shared-memory copy when the bucket fits
  const uint32_t* ks = bk;
  if (load <= kExpSmemKeys) {
    for (int i0 = 0; i0 < load; i0 += kExpThreads * 8) {
      uint32_t v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {  // all eight loads in flight before any store
        const int i = i0 + q * kExpThreads + tid;
        v[q] = i < load ? bk[i] : 0u;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * kExpThreads + tid;
        if (i < load) s_keys[i] = v[q];
      }
    }
    ks = s_keys;
    __syncthreads();
  }

  // MSD radix select, 8 bits a pass: find the key value `thr` of the keep-th largest key and
  // how many of the keys equal to it are kept (`need`).  When the bin that holds the keep-th
  // largest key is kept whole, no finer pass is needed: every key >= the bin's lowest value
  // is kept, which is the rule key > thr with thr = that value - 1 and need = 0 (the value is
  // > 0 there, because keep < load).
  uint32_t prefix = 0, thr = 0;
  int need = keep;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const uint32_t hi_mask = pass == 0 ? 0u : (0xffffffffu << (32 - 8 * pass));
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < load; i0 += kExpThreads * 8) {  // warp-uniform trip count
      uint32_t keys[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * kExpThreads + tid;
        keys[q] = i < load ? ks[i] : 0u;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * kExpThreads + tid;
        const bool in = i < load && (keys[q] & hi_mask) == prefix;
        const int bin = in ? (int)((keys[q] >> shift) & 255u) : -1;
        // scores cluster in a few bins: aggregate per warp before touching shared memory
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (in && (tid & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
      }
    }
    __syncthreads();
    // suffix counts over bins, highest bin first: thread b' handles bin 255 - b'
    const int bin = 255 - tid;
    const int cnt = tid < 256 ? hist[bin] : 0;
    int tot;
    const int above = block_excl_scan(cnt, &tot, sm);  // keys in bins > bin
    if (tid < 256 && above < need && above + cnt >= need) {
      s_prefix = prefix | ((uint32_t)bin << shift);
      s_need = need - above;
      s_whole = above + cnt == need;
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    const bool whole = s_whole;
    __syncthreads();
    if (whole) {
      thr = prefix - 1u;
      need = 0;
      break;
    }
    thr = prefix;
  }

  // Ordered keep pass.
  int run_eq = 0, run_kept = 0;
  for (int r0 = 0; r0 < load; r0 += kExpThreads * kExpIPT) {
    const int i0 = r0 + tid * kExpIPT;
    uint32_t keys[kExpIPT];
    int n_eq = 0;
#pragma unroll
    for (int q = 0; q < kExpIPT; ++q) {
      const int i = i0 + q;
      keys[q] = i < load ? ks[i] : 0u;
      n_eq += (i < load && keys[q] == thr);
    }
    int tot_eq;
    int eq_rank = run_eq + block_excl_scan(n_eq, &tot_eq, sm);
    bool kf[kExpIPT];
    int n_kept = 0;
#pragma unroll
    for (int q = 0; q < kExpIPT; ++q) {
      const int i = i0 + q;
      const bool in = i < load;
      const bool is_eq = in && keys[q] == thr;
      kf[q] = in && (keys[q] > thr || (is_eq && eq_rank < need));
      eq_rank += is_eq;
      n_kept += kf[q];
    }
    int tot_kept;
    int pos = run_kept + block_excl_scan(n_kept, &tot_kept, sm);
#pragma unroll
    for (int q = 0; q < kExpIPT; ++q) {
      const int i = i0 + q;
      if (i < load) {
        const int u = bu[i];
        if (kf[q]) {
          kept_pair[base + pos] = u;
          row_of_pair[u] = base + pos;
          ++pos;
        } else {
          row_of_pair[u] = -1;
        }
      }
    }
    run_eq += tot_eq;
    run_kept += tot_kept;
  }
}

}  // namespace

void launch_select(const int32_t* topk_idx, const float* scores, const int32_t* quotas, int64_t P, int32_t E,
                   int64_t cap, int32_t* seg_offsets, int32_t* kept_pair, int32_t* row_of_pair, const SelectWs& ws,
                   int32_t* status, cudaStream_t s) {
  const int64_t nc = ws.n_chunks;
  if (nc > 0)
    sel_count_kernel<<<(unsigned)nc, kSelChunk, E * sizeof(int), s>>>(topk_idx, P, E, ws.counts, status);
  sel_colscan_kernel<<<E, 1024, 0, s>>>(ws.counts, nc, E, ws.loads);
  const size_t bsmem = (size_t)(2 + kSelChunk / 32) * E * sizeof(int);
  sel_bucket_kernel<<<nc > 0 ? (unsigned)nc : 1u, kSelChunk, bsmem, s>>>(
      topk_idx, scores, P, E, nc, ws.counts, ws.loads, quotas, cap, ws.bucket_start, ws.keep, seg_offsets,
      ws.sorted_u, ws.sorted_key, row_of_pair, status);
  if (P > 0) {
    static bool attr_set = false;
    const int smem = kExpSmemKeys * (int)sizeof(uint32_t);
    if (!attr_set) {
      cudaFuncSetAttribute(sel_expert_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      attr_set = true;
    }
    sel_expert_kernel<<<E, kExpThreads, smem, s>>>(ws.bucket_start, ws.keep, seg_offsets, ws.sorted_u,
                                                  ws.sorted_key, kept_pair, row_of_pair);
  }
}

}  // namespace lrm
