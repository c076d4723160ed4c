// Per-expert top-quota selection.
//
// "LRMoE poda a passagem reversa do MoE..." (news.hamidun.com), step "Seleção pela métrica
// LRM": inside each expert's quota the highest-scoring pairs are kept.  Equal scores go to
// the smaller pair index u; inside a segment the kept pairs are listed in u order.
//
// Four launches (five from 131072 pairs on), all deterministic:
//  1. count:   one CTA per chunk of kSelChunk consecutive pairs counts the chunk's experts.
//  2. scan:    one CTA per expert: exclusive scan of that expert's chunk counts (bucket
//              bases inside the expert's bucket) and its load.
//  3. bucket:  one CTA per chunk derives the expert-level prefixes (bucket starts, kept counts
//              min(quota, load), segment offsets, capacity check; CTA 0 publishes them),
//              then scatters its pairs stably into the expert buckets (u ascending) with
//              their score bits: ranks within a warp from __match_any_sync, across warps from
//              per-warp expert counts.
//  4. expert:  one CTA per expert (1024 threads, the bucket's keys held in shared memory
//              when they fit): MSD radix select of the quota-th largest score over 11 + 11 +
//              10 bits, each pass after the first reading only the keys left in the chosen
//              bin (stopping early once that bin is kept whole), then one ordered pass that
//              keeps everything above the threshold plus the first `need` pairs equal to it,
//              and writes kept_pair and row_of_pair through ballots and a prefix over warps.
//  5. rows:    (from 131072 pairs on) scatters row_of_pair from the rows step 4 left in bucket
//              order, on the whole GPU.
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
  chain_wait();
  extern __shared__ int hist[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t c = blockIdx.x;
  const int64_t u = c * kSelChunk + threadIdx.x;
  const int e = u < P ? idx[u] : -1;
  const bool good = u < P && e >= 0 && e < E;
  if (u < P && !good) set_status(status, LRM_ERR_BAD_INDEX);
  if (good) atomicAdd(&hist[e], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[c * E + e] = hist[e];
}

// One CTA per expert: exclusive scan down the expert's column of chunk counts.
__global__ void __launch_bounds__(1024) sel_colscan_kernel(int32_t* __restrict__ counts, int64_t n_chunks, int E,
                                                           int32_t* __restrict__ loads) {
  chain_wait();
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
  chain_wait();
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
    if (LRM_DCHECK(pos >= 0 && pos < P, status, LRM_ERR_BAD_INDEX)) {
      sorted_u[pos] = (int32_t)u;
      sorted_key[pos] = key;
    }
  }
}

constexpr int kExpThreads = 1024;
constexpr int kExpWarps = kExpThreads / 32;
constexpr int kExpBins = 2048;  // radix digits of 11, 11 and 10 bits
// Shared memory of the per-expert kernel: the digit histogram, the bucket's keys when they fit
// (read once from global memory instead of on every pass) and the candidate keys left after a
// pass (those in the bin of the quota-th largest key), which the next pass reads instead of
// the whole bucket.
constexpr int kExpKeysCap = 36864;  // 144 KB
constexpr int kExpCandCap = 18432;  // 72 KB
constexpr size_t kExpSmemBytes = sizeof(int) * kExpBins + sizeof(uint32_t) * (kExpKeysCap + kExpCandCap);

// Exclusive prefix over the block's warps of one int per warp (lane 0's value counts); every
// thread gets its warp's prefix and the block total.  `sm` needs 33 ints.
__device__ __forceinline__ int warp_excl_scan(int v, int* total, int* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < kExpWarps ? sm[lane] : 0;
    int incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    sm[lane] = incl - w;
    if (lane == 31) sm[32] = incl;
  }
  __syncthreads();
  const int res = sm[warp];
  *total = sm[32];
  __syncthreads();
  return res;
}

// `direct`: write row_of_pair[u] here.  Otherwise each bucket slot's row (or -1) is written in
// bucket order over the key it replaces (the slot's key has been read by then, by the same
// thread) and sel_rows_kernel scatters them: the scattered stores then run on the whole GPU
// instead of on the CTA of the largest bucket.
__global__ void __launch_bounds__(kExpThreads) sel_expert_kernel(
    const int32_t* __restrict__ bucket_start, const int32_t* __restrict__ keep_arr,
    const int32_t* __restrict__ seg_offsets, const int32_t* __restrict__ sorted_u, uint32_t* sorted_key,
    int32_t* __restrict__ kept_pair, int32_t* __restrict__ row_of_pair, int direct, int64_t P, int64_t cap,
    int32_t* __restrict__ status) {
  chain_wait();
  extern __shared__ uint32_t s_dyn[];
  int* hist = reinterpret_cast<int*>(s_dyn);  // [kExpBins]
  uint32_t* s_keys = s_dyn + kExpBins;        // [kExpKeysCap]
  uint32_t* s_cand = s_keys + kExpKeysCap;    // [kExpCandCap]
  __shared__ int sm[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need, s_whole, s_cnt, s_fill;
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b0 = bucket_start[e];
  const int load = bucket_start[e + 1] - b0;
  const int keep = keep_arr[e];
  const int base = seg_offsets[e];
  const int32_t* bu = sorted_u + b0;
  uint32_t* bk = sorted_key + b0;

  if (keep >= load) {
    for (int i = tid; i < load; i += kExpThreads) {
      const int u = bu[i];
      if (!LRM_DCHECK(u >= 0 && u < P && base + i < cap, status, LRM_ERR_BAD_INDEX)) continue;
      kept_pair[base + i] = u;
      if (direct) row_of_pair[u] = base + i;
      else bk[i] = (uint32_t)(base + i);
    }
    return;
  }
  if (keep <= 0) {
    for (int i = tid; i < load; i += kExpThreads) {
      if (direct) {
        if (LRM_DCHECK(bu[i] >= 0 && bu[i] < P, status, LRM_ERR_BAD_INDEX)) row_of_pair[bu[i]] = -1;
      } else {
        bk[i] = 0xffffffffu;
      }
    }
    return;
  }

  // the bucket's keys: a shared-memory copy when they fit
  const uint32_t* ks = bk;
  if (load <= kExpKeysCap) {
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
  }

  // MSD radix select over 11 + 11 + 10 bits: find the value `thr` of the keep-th largest key and
  // how many of the keys equal to it are kept (`need`).  A pass looks only at the keys whose
  // higher digits equal `prefix`: after the first pass those are copied into s_cand (when they
  // fit), so that later passes read only them.  When the bin holding the keep-th largest key is
  // kept whole, no finer pass is needed: every key >= the bin's lowest value is kept, which is
  // the rule key > thr with thr = that value - 1 and need = 0 (the value is > 0 there, because
  // keep < load).
  uint32_t prefix = 0, thr = 0;
  int need = keep;
  const uint32_t* src = ks;  // what the current pass reads
  int n_src = load;
  bool src_filtered = false;  // src holds only keys that match prefix
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t digit_mask = pass == 2 ? 1023u : 2047u;
    const uint32_t hi_mask = pass == 0 ? 0u : (pass == 1 ? 0xffe00000u : 0xfffffc00u);
    for (int b = tid; b < kExpBins; b += kExpThreads) hist[b] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n_src; i0 += kExpThreads * 8) {  // warp-uniform trip count
      uint32_t keys[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * kExpThreads + tid;
        keys[q] = i < n_src ? src[i] : 0u;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * kExpThreads + tid;
        const bool in = i < n_src && (src_filtered || (keys[q] & hi_mask) == prefix);
        // one shared atomic per key: on this GPU that beats aggregating equal bins across the
        // warp first (__match_any_sync), even though the scores cluster in a few bins
        if (in) atomicAdd(&hist[(keys[q] >> shift) & digit_mask], 1);
      }
    }
    __syncthreads();
    // suffix counts over bins, highest first: thread i takes bins 2047 - 2i and 2046 - 2i
    const int bhi = kExpBins - 1 - 2 * tid, blo = bhi - 1;
    const int chi = hist[bhi], clo = hist[blo];
    int tot;
    const int above = block_excl_scan(chi + clo, &tot, sm);  // keys in bins > bhi
    if (above < need && above + chi >= need) {
      s_prefix = prefix | ((uint32_t)bhi << shift);
      s_need = need - above;
      s_whole = above + chi == need;
      s_cnt = chi;
    } else if (above + chi < need && above + chi + clo >= need) {
      s_prefix = prefix | ((uint32_t)blo << shift);
      s_need = need - above - chi;
      s_whole = above + chi + clo == need;
      s_cnt = clo;
    }
    if (tid == 0) s_fill = 0;
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    const bool whole = s_whole;
    const int cnt = s_cnt;
    if (whole) {
      thr = prefix - 1u;
      need = 0;
      break;
    }
    thr = prefix;
    if (pass == 2) break;
    // keep only the keys of the chosen bin for the next pass (in place when src is s_cand: a
    // batch is read into registers before any of it is overwritten, and the write position never
    // passes the read position)
    if (cnt <= kExpCandCap) {
      const uint32_t sel_mask = pass == 0 ? 0xffe00000u : 0xfffffc00u;
      for (int i0 = 0; i0 < n_src; i0 += kExpThreads * 8) {
        uint32_t keys[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = i0 + q * kExpThreads + tid;
          keys[q] = i < n_src ? src[i] : 0u;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = i0 + q * kExpThreads + tid;
          const bool m = i < n_src && (keys[q] & sel_mask) == prefix;
          const unsigned bal = __ballot_sync(0xffffffffu, m);
          int off = 0;
          if (lane == 0 && bal) off = atomicAdd(&s_fill, __popc(bal));
          off = __shfl_sync(0xffffffffu, off, 0);
          const int slot = off + __popc(bal & ((1u << lane) - 1u));
          if (m && LRM_DCHECK(slot < kExpCandCap, status, LRM_ERR_BAD_INDEX)) s_cand[slot] = keys[q];
        }
        __syncthreads();
      }
      src = s_cand;
      n_src = cnt;
      src_filtered = true;
    } else {
      src_filtered = false;  // too many to copy: the next pass reads all keys and matches prefix
      src = ks;
      n_src = load;
    }
    __syncthreads();
  }

  // Ordered keep pass.  A round covers kExpThreads * 8 keys; warp w takes 256 consecutive keys,
  // lane l the keys w * 256 + q * 32 + l (q = 0..7), so reads are coalesced and conflict-free and
  // the bucket order is kept through ballots.
  const unsigned lt_mask = (1u << lane) - 1u;
  int run_eq = 0, run_kept = 0;
  for (int r0 = 0; r0 < load; r0 += kExpThreads * 8) {
    const int wb = r0 + warp * 256;
    uint32_t keys[8];
    unsigned eqm[8];
    int w_eq = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = wb + q * 32 + lane;
      keys[q] = i < load ? ks[i] : 0u;
      eqm[q] = __ballot_sync(0xffffffffu, i < load && keys[q] == thr);
      w_eq += __popc(eqm[q]);
    }
    int tot_eq;
    int eq_before = run_eq + warp_excl_scan(w_eq, &tot_eq, sm);
    unsigned kfm[8];
    int w_kept = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = wb + q * 32 + lane;
      const bool is_eq = (eqm[q] >> lane) & 1u;
      const int eq_rank = eq_before + __popc(eqm[q] & lt_mask);
      const bool kf = i < load && (keys[q] > thr || (is_eq && eq_rank < need));
      eq_before += __popc(eqm[q]);
      kfm[q] = __ballot_sync(0xffffffffu, kf);
      w_kept += __popc(kfm[q]);
    }
    int tot_kept;
    int pos = run_kept + warp_excl_scan(w_kept, &tot_kept, sm);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = wb + q * 32 + lane;
      if (i < load) {
        const bool kept = (kfm[q] >> lane) & 1u;
        const int r = kept ? base + pos + __popc(kfm[q] & lt_mask) : -1;
        if (LRM_DCHECK(bu[i] >= 0 && bu[i] < P && r < cap, status, LRM_ERR_BAD_INDEX)) {
          if (kept) kept_pair[r] = bu[i];
          if (direct) row_of_pair[bu[i]] = r;
          else bk[i] = (uint32_t)r;
        }
      }
      pos += __popc(kfm[q]);
    }
    run_eq += tot_eq;
    run_kept += tot_kept;
  }
}

// row_of_pair[sorted_u[i]] = the row that sel_expert_kernel left in slot i (deferred mode).
__global__ void __launch_bounds__(256) sel_rows_kernel(const int32_t* __restrict__ bucket_start, int E,
                                                       const int32_t* __restrict__ sorted_u,
                                                       const uint32_t* __restrict__ slot_row,
                                                       int32_t* __restrict__ row_of_pair, int64_t P,
                                                       int32_t* __restrict__ status) {
  chain_wait();
  const int64_t n = bucket_start[E];
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t u = sorted_u[i];
    if (LRM_DCHECK(u >= 0 && u < P, status, LRM_ERR_BAD_INDEX)) row_of_pair[u] = (int32_t)slot_row[i];
  }
}

// From this many pairs on, the rows are scattered by sel_rows_kernel (one launch more; the
// largest bucket's CTA no longer issues its scattered stores alone).
constexpr int64_t kDeferRowsMinPairs = 131072;

}  // namespace

void launch_select(const int32_t* topk_idx, const float* scores, const int32_t* quotas, int64_t P, int32_t E,
                   int64_t cap, int32_t* seg_offsets, int32_t* kept_pair, int32_t* row_of_pair, const SelectWs& ws,
                   int32_t* status, cudaStream_t s) {
  const int64_t nc = ws.n_chunks;
  if (nc > 0)
    launch_chained(sel_count_kernel, dim3((unsigned)nc), dim3(kSelChunk), E * sizeof(int), s, topk_idx, P, E,
                   ws.counts, status);
  launch_chained(sel_colscan_kernel, dim3(E), dim3(1024), 0, s, ws.counts, nc, E, ws.loads);
  const size_t bsmem = (size_t)(2 + kSelChunk / 32) * E * sizeof(int);
  launch_chained(sel_bucket_kernel, dim3(nc > 0 ? (unsigned)nc : 1u), dim3(kSelChunk), bsmem, s, topk_idx, scores, P,
                 E, nc, (const int32_t*)ws.counts, (const int32_t*)ws.loads, quotas, cap, ws.bucket_start, ws.keep,
                 seg_offsets, ws.sorted_u, ws.sorted_key, row_of_pair, status);
  if (P > 0) {
    const int smem = (int)kExpSmemBytes;
    ensure_max_smem<sel_expert_kernel>(smem);  // a failure surfaces as the launch's error
    const bool direct = P < kDeferRowsMinPairs;
    launch_chained(sel_expert_kernel, dim3(E), dim3(kExpThreads), (size_t)smem, s, (const int32_t*)ws.bucket_start,
                   (const int32_t*)ws.keep, (const int32_t*)seg_offsets, (const int32_t*)ws.sorted_u, ws.sorted_key,
                   kept_pair, row_of_pair, direct ? 1 : 0, P, cap, status);
    if (!direct) {
      const int64_t blocks = (P + 255) / 256;
      launch_chained(sel_rows_kernel, dim3((unsigned)(blocks < 1216 ? blocks : 1216)), dim3(256), 0, s,
                     (const int32_t*)ws.bucket_start, E, (const int32_t*)ws.sorted_u, (const uint32_t*)ws.sorted_key,
                     row_of_pair, P, status);
    }
  }
}

}  // namespace lrm
