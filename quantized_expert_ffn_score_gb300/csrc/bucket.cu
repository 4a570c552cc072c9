// bucket.cu -- group the (token, slot) pairs by expert: a stable counting sort
// of pair ids p = t*k + j by topk_idx[p] (the grouping step that precedes the
// expert FFN; "Running a 2.78-Trillion-Parameter Model Across Two Desks", Act II
// computes each selected expert once per layer for the tokens routed to it).
//
// One CTA.  Warp w owns the contiguous pair range [w*P/W, (w+1)*P/W).
//   1. per-warp histograms hist[w][e] with warp-aggregated shared atomics
//      (__match_any_sync groups lanes holding the same expert; the group's
//      leader adds the group size);
//   2. per expert, an exclusive scan over warps gives each warp's base inside
//      the expert's bucket; a block scan over experts gives offsets;
//   3. each warp re-walks its range in order and writes pair ids: the rank of a
//      lane inside its match group plus the running per-(warp, expert) count.
// Ascending p within every bucket, independent of timing.
#include <utility>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBucketMaxWarps = 32;

// Exclusive scan of v over the block (all threads participate); returns the
// prefix and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* scratch, int* total) {
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

// Running totals of the expert lists across chunks of the expert range.
struct SplitCarry {
  int cold = 0, hot = 0, blk = 0;
};

// One chunk of experts (one per thread, cnt = bucket size, 0 past E): appends
// the GEMV-path experts to active[] and the GEMM-path experts to hot[] with
// their token-block prefix.  Every thread of the block calls it.
__device__ void split_step(int e, int cnt, int32_t* active, const HotSplit& sp, int* scratch, SplitCarry& c) {
  const bool is_hot = sp.hot != nullptr && sp.gemm_min > 0 && cnt >= sp.gemm_min;
  const int f_cold = (cnt > 0 && !is_hot) ? 1 : 0;
  int t_cold, t_hot, t_blk;
  const int pos_cold = block_exclusive_scan(f_cold, scratch, &t_cold) + c.cold;
  if (f_cold) active[1 + pos_cold] = e;
  if (sp.hot != nullptr) {
    const int nblk = is_hot ? (cnt + 127) / 128 : 0;
    const int pos_hot = block_exclusive_scan(is_hot ? 1 : 0, scratch, &t_hot) + c.hot;
    const int pos_blk = block_exclusive_scan(nblk, scratch, &t_blk) + c.blk;
    if (is_hot) {
      sp.hot[1 + pos_hot] = e;
      sp.hot_blk[pos_hot] = pos_blk;
    }
    c.hot += t_hot;
    c.blk += t_blk;
  }
  c.cold += t_cold;
}

__device__ void split_finish(int32_t* active, const HotSplit& sp, const SplitCarry& c) {
  active[0] = c.cold;
  if (sp.hot != nullptr) {
    sp.hot[0] = c.hot;
    sp.hot_blk[c.hot] = c.blk;
  }
}

// The first nw warps own the pairs; all blockDim threads take part in the
// per-expert scans (blockDim is sized from E, nw from T*k).
__global__ void bucket_kernel(BucketArgs a, int nw) {
  extern __shared__ int bsm[];
  const int E = a.E, P = a.T * a.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* hist = bsm;                    // [nw][E]: counts, then running slot positions
  int* scan_scratch = hist + nw * E;  // [32]
  pdl_wait();
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  pdl_launch_dependents();
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
  //    the offsets and the expert lists (GEMV-path and GEMM-path experts)
  int carry = 0;
  SplitCarry sc;
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
    const int off = block_exclusive_scan(cnt, scan_scratch, &total) + carry;
    split_step(e, e < E ? cnt : 0, a.active, a.split, scan_scratch, sc);
    if (e < E) {
      a.counts[e] = cnt;
      a.offsets[e] = off;
      for (int w = 0; w < nw; ++w) hist[w * E + e] += off;  // absolute running position
    }
    carry += total;
  }
  if (threadIdx.x == 0) {
    a.offsets[E] = carry;
    split_finish(a.active, a.split, sc);
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

// Expert lists from offsets alone (used when the expert FFN is called on its
// own): active[0] = count, active[1..] = GEMV-path experts with a non-empty
// bucket; the GEMM-path experts go to split.hot.
__global__ void active_kernel(const int32_t* offsets, int E, int32_t* active, HotSplit split) {
  __shared__ int scratch[32];
  pdl_wait();
  SplitCarry sc;
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    const int cnt = e < E ? offsets[e + 1] - offsets[e] : 0;
    split_step(e, cnt, active, split, scratch, sc);
  }
  if (threadIdx.x == 0) split_finish(active, split, sc);
}

}  // namespace

cudaError_t launch_bucket(const BucketArgs& a, bool pdl, cudaStream_t s) {
  const int P = a.T * a.k;
  int nw = (P + 255) / 256;  // pair warps: ~8 rounds of 32 pairs each
  nw = nw < 1 ? 1 : (nw > kBucketMaxWarps ? kBucketMaxWarps : nw);
  const int nw_smem = (200 * 1024 / 4 - 32) / a.E;  // per-warp histograms must fit in shared memory
  if (nw > nw_smem) nw = nw_smem;
  int nthreads = 32 * ((a.E + 31) / 32);  // one scan element per thread where possible
  if (nthreads > 1024) nthreads = 1024;
  if (nthreads < 32 * nw) nthreads = 32 * nw;
  const size_t smem = ((size_t)nw * a.E + 32) * sizeof(int);
  ensure_smem(bucket_kernel, smem);
  return launch("bucket", bucket_kernel, dim3(1), dim3(nthreads), smem, s, pdl, a, nw);
}

cudaError_t launch_active_from_offsets(const int32_t* offsets, int E, int32_t* active, const HotSplit& split, bool pdl,
                                       cudaStream_t s) {
  return launch("active_list", active_kernel, dim3(1), dim3(256), 0, s, pdl, offsets, E, active, split);
}

}  // namespace moe
