// bucket.cu -- launchers of the bucketing step (bucket_body.cuh): the bucket
// kernel after the top-k, and the expert lists from offsets alone for the
// standalone expert call.
#include <utility>

#include "bucket_body.cuh"

namespace moe {
namespace {

constexpr int kBucketMaxWarps = 32;

// One CTA.
__global__ void bucket_kernel(BucketArgs a, int nw) {
  extern __shared__ int bsm[];
  pdl_wait();
  pdl_launch_dependents();
  bucket_block(a, nw, bsm);
}

// Expert list from offsets alone (used when the expert FFN is called on its
// own): active[0] = count, active[1..] = the experts with a non-empty bucket.
__global__ void active_kernel(const int32_t* offsets, int E, int32_t* active) {
  __shared__ int scratch[32];
  pdl_wait();
  int n_active = 0;
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    const int cnt = e < E ? offsets[e + 1] - offsets[e] : 0;
    bucket_detail::active_step(e, cnt, active, scratch, n_active);
  }
  if (threadIdx.x == 0) active[0] = n_active;
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

cudaError_t launch_active_from_offsets(const int32_t* offsets, int E, int32_t* active, bool pdl, cudaStream_t s) {
  return launch("active_list", active_kernel, dim3(1), dim3(256), 0, s, pdl, offsets, E, active);
}

}  // namespace moe
