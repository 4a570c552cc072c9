// rvq3_repack.cu -- converts RVQ3 expert records from the stage-planar,
// row-major code layout to the stage-planar, position-major one the RVQ3
// kernels read (WASTE README, "3 bits per expert weight": one 8-bit code per
// stage for every 8 consecutive weights of a row).
//
// Row-major ("canonical") record:
//   gate [3][ff][d/8] | up [3][ff][d/8] | down [3][d][ff/8]
// Position-major record:
//   gate [3][d/8][ff] | up [3][d/8][ff] | down [3][ff/8][d]
// Every one of the 9 planes (matrix, stage) is a byte matrix [rows][nv]
// transposed to [nv][rows]; the record size is unchanged.  One 32 x 32 tile of
// a plane per step: the 32 x 32 bytes are read row by row (32 contiguous
// bytes per warp), stored in shared memory and written out column by column.
#include "moe_internal.cuh"

namespace moe {
namespace {

struct PlaneGeom {
  int rows, nv;     // plane shape in the row-major record
  int tiles_r, tiles_v;
};

__global__ void __launch_bounds__(256) rvq3_repack_kernel(const uint8_t* const* src, uint8_t* const* dst, int n,
                                                          int d, int ff, int* err) {
  __shared__ uint8_t tile[32][33];
  const PlaneGeom pg[2] = {{ff, d / 8, ff / 32, (d / 8 + 31) / 32}, {d, ff / 8, d / 32, (ff / 8 + 31) / 32}};
  const long long per_gu = (long long)pg[0].tiles_r * pg[0].tiles_v;  // tiles of one gate or up plane
  const long long per_dn = (long long)pg[1].tiles_r * pg[1].tiles_v;  // tiles of one down plane
  const long long per_rec = 6 * per_gu + 3 * per_dn;
  const size_t plane_gu = (size_t)ff * (d / 8), plane_dn = (size_t)d * (ff / 8);
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (long long w = blockIdx.x; w < (long long)n * per_rec; w += gridDim.x) {
    const int rec = (int)(w / per_rec);
    long long t = w % per_rec;
    const uint8_t* s = src[rec];
    uint8_t* o = dst[rec];
    if (s == nullptr || o == nullptr || s == o) {  // one report per record: its first tile
      if (t == 0 && threadIdx.x == 0) dev_error(err, s == o && s != nullptr ? MOE_ERR_INVALID_ARG : MOE_ERR_MISSING_EXPERT, rec);
      continue;
    }
    int kind;  // 0: a gate or up plane, 1: a down plane
    size_t off;
    if (t < 6 * per_gu) {
      kind = 0;
      off = (size_t)(t / per_gu) * plane_gu;
      t %= per_gu;
    } else {
      t -= 6 * per_gu;
      kind = 1;
      off = 6 * plane_gu + (size_t)(t / per_dn) * plane_dn;
      t %= per_dn;
    }
    const PlaneGeom g = pg[kind];
    const int r0 = (int)(t / g.tiles_v) * 32, v0 = (int)(t % g.tiles_v) * 32;
    __syncthreads();  // the previous tile's reads of `tile` are done
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = ty + 8 * i;  // rows are a multiple of 32: always in range
      if (v0 + tx < g.nv) tile[r][tx] = s[off + (size_t)(r0 + r) * g.nv + v0 + tx];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int v = ty + 8 * i;
      if (v0 + v < g.nv) o[off + (size_t)(v0 + v) * g.rows + r0 + tx] = tile[tx][v];
    }
  }
}

}  // namespace

cudaError_t launch_rvq3_repack(const uint8_t* const* src, uint8_t* const* dst, int n, int d, int ff, int* err,
                               int num_sms, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  return launch("rvq3_repack", rvq3_repack_kernel, dim3(8 * num_sms), dim3(256), 0, s, false, src, dst, n, d, ff, err);
}

}  // namespace moe
