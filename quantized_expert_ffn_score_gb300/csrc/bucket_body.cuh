// bucket_body.cuh -- the bucketing of (token, slot) pairs by expert as a
// device function of one CTA: used by the bucket kernel and, for a single
// token, by the top-k kernel right after it has chosen the experts.
//
// A stable counting sort of pair ids p = t*k + j by topk_idx[p] (the grouping
// step that precedes the expert FFN; "Running a 2.78-Trillion-Parameter Model
// Across Two Desks", Act II computes each selected expert once per layer for
// the tokens routed to it).  Warp w of the first nw owns the contiguous pair
// range [w*P/nw, (w+1)*P/nw):
//   1. per-warp histograms hist[w][e] with warp-aggregated shared atomics
//      (__match_any_sync groups lanes holding the same expert; the group's
//      leader adds the group size);
//   2. per expert, an exclusive scan over warps gives each warp's base inside
//      the expert's bucket; a block scan over experts gives offsets;
//   3. each warp re-walks its range in order and writes pair ids: the rank of a
//      lane inside its match group plus the running per-(warp, expert) count.
// Ascending p within every bucket, independent of timing.
#pragma once

#include "moe_internal.cuh"

namespace moe {
namespace bucket_detail {

// Exclusive scan of v over the block (all threads participate); returns the
// prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) scratch[lane] = s;  // inclusive per-warp totals
  }
  __syncthreads();
  int base = warp > 0 ? scratch[warp - 1] : 0;
  *total = scratch[nw - 1];
  __syncthreads();
  return base + x - v;
}

// One chunk of experts (one per thread, cnt = bucket size, 0 past E): appends
// the experts with a non-empty bucket to active[] in ascending order; `carry`
// holds the running count across chunks.  Every thread of the block calls it.
__device__ __forceinline__ void active_step(int e, int cnt, int32_t* active, int* scratch, int& carry) {
  const int f = cnt > 0 ? 1 : 0;
  int total;
  const int pos = block_exclusive_scan(f, scratch, &total) + carry;
  if (f) active[1 + pos] = e;
  carry += total;
}

}  // namespace bucket_detail

// The first nw warps own the pairs; all blockDim threads take part in the
// per-expert scans.  bsm: nw * E + 32 ints of shared memory.
__device__ __forceinline__ void bucket_block(const BucketArgs& a, int nw, int* bsm) {
  const int E = a.E, P = a.T * a.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* hist = bsm;                    // [nw][E]: counts, then running slot positions
  int* scan_scratch = hist + nw * E;  // [32]
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int per = (P + nw - 1) / nw;
  const int p_begin = warp < nw ? min(P, warp * per) : P;
  const int p_end = warp < nw ? min(P, p_begin + per) : P;
  // 1. histograms
  for (int base = p_begin; base < p_end; base += 32) {
    const int p = base + lane;
    int e = p < p_end ? a.topk_idx[p] : -1;
    if (p < p_end && (e < 0 || e >= E)) {
      dev_error(a.err, MOE_ERR_BAD_EXPERT_INDEX, e);
      e = -1;
    }
    const unsigned act = __ballot_sync(0xffffffffu, e >= 0);
    if (e >= 0) {
      const unsigned grp = __match_any_sync(act, e);
      if (lane == __ffs(grp) - 1) atomicAdd(&hist[warp * E + e], __popc(grp));
    }
  }
  __syncthreads();
  // 2. per expert: counts and per-warp bases; block scans over experts give
  //    the offsets and the list of experts with tokens
  int carry = 0, n_active = 0;
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    int cnt = 0;
    if (e < E) {
      for (int w = 0; w < nw; ++w) {
        const int c = hist[w * E + e];
        hist[w * E + e] = cnt;  // exclusive base of warp w inside expert e's bucket
        cnt += c;
      }
    }
    int total;
    const int off = bucket_detail::block_exclusive_scan(cnt, scan_scratch, &total) + carry;
    bucket_detail::active_step(e, e < E ? cnt : 0, a.active, scan_scratch, n_active);
    if (e < E) {
      a.counts[e] = cnt;
      a.offsets[e] = off;
      for (int w = 0; w < nw; ++w) hist[w * E + e] += off;  // absolute running position
    }
    carry += total;
  }
  if (threadIdx.x == 0) {
    a.offsets[E] = carry;
    a.active[0] = n_active;
  }
  __syncthreads();
  // 3. stable scatter, walking each warp's range in ascending p
  for (int base = p_begin; base < p_end; base += 32) {
    const int p = base + lane;
    int e = p < p_end ? a.topk_idx[p] : -1;
    if (e >= E) e = -1;
    const unsigned act = __ballot_sync(0xffffffffu, e >= 0);
    if (e >= 0) {
      const unsigned grp = __match_any_sync(act, e);
      const int rank = __popc(grp & ((1u << lane) - 1u));
      const int pos = hist[warp * E + e] + rank;
      a.pair_ids[pos] = p;
      __syncwarp(grp);
      if (lane == __ffs(grp) - 1) hist[warp * E + e] += __popc(grp);
    }
    __syncwarp();
  }
}


// The same result for a single token (T = 1, k <= 32 distinct experts): no
// histogram or scan.  With the k selected ids sel[j], an expert's offset is the
// number of selected ids below it, pair j lands at the rank of sel[j], and
// every selected expert has one token.  The offsets come from a bit mask of
// the selected ids and its per-word population-count prefix.  a.counts may be
// null (not wanted).  Every thread of the block calls it.
__device__ __forceinline__ void bucket_one_token(const BucketArgs& a, int* sel_smem, bool preloaded = false) {
  __shared__ uint32_t sel_mask[kMaxE / 32 + 1];
  __shared__ int mask_prefix[kMaxE / 32 + 1];
  const int E = a.E, k = a.k, nw = (E >> 5) + 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < k) {
    int e = preloaded ? sel_smem[threadIdx.x] : a.topk_idx[threadIdx.x];
    if (e < 0 || e >= E) {
      dev_error(a.err, MOE_ERR_BAD_EXPERT_INDEX, e);
      e = E;  // sorts last, never counted
    }
    sel_smem[threadIdx.x] = e;
  }
  for (int w = threadIdx.x; w < nw; w += blockDim.x) sel_mask[w] = 0u;
  __syncthreads();
  if (threadIdx.x < k && sel_smem[threadIdx.x] < E)
    atomicOr(&sel_mask[sel_smem[threadIdx.x] >> 5], 1u << (sel_smem[threadIdx.x] & 31));
  __syncthreads();
  if (warp == 0) {
    const int e = lane < k ? sel_smem[lane] : 0x7fffffff;
    int rank = 0, nvalid = 0;
    for (int j = 0; j < k; ++j) {
      const int o = sel_smem[j];
      rank += (o < e) ? 1 : 0;
      nvalid += (o < E) ? 1 : 0;
    }
    if (lane < k && e < E) {
      a.pair_ids[rank] = lane;
      a.active[1 + rank] = e;
    }
    if (lane == 0) a.active[0] = nvalid;
    // exclusive prefix of the words' population counts, 32 words at a time
    int carry = 0;
    for (int w0 = 0; w0 < nw; w0 += 32) {
      const int w = w0 + lane;
      const int c = w < nw ? __popc(sel_mask[w]) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (w < nw) mask_prefix[w] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    const int w = e >> 5, b = e & 31;
    const uint32_t m = sel_mask[w];
    a.offsets[e] = mask_prefix[w] + __popc(m & ((1u << b) - 1u));
    if (e < E && a.counts) a.counts[e] = (int)((m >> b) & 1u);
  }
}

}  // namespace moe
