// fill.cu -- the stand-alone bias fill, for a transposed conv whose engine
// grid has no tiles (every output is the bias).  Otherwise the engine's own
// fill warp does this work beside the convolution.
#include "fill.cuh"

#include <algorithm>
#include <cstdint>

namespace tc3d {

namespace {

// Work unit: one plane of one slice, one warp (fill_plane).
constexpr int kFillWarps = 4;

__global__ void __launch_bounds__(32 * kFillWarps) fill_slab_kernel(const __grid_constant__ FillParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long u = (long long)blockIdx.x * kFillWarps + warp;
  if (u >= (long long)p.NC * p.O[0]) return;
  const int nc = (int)(u / p.O[0]), z = (int)(u - (long long)nc * p.O[0]);
  const float b = p.bias ? __ldg(p.bias + nc % p.Cout) : 0.f;
  fill_plane(p, nc, z, b, lane);
}

}  // namespace

cudaError_t fill_slab_launch(const FillParams& p, cudaStream_t st) {
  // a warp per (slice, plane)
  const long long units = (long long)p.NC * p.O[0];
  const long long grid = (units + kFillWarps - 1) / kFillWarps;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  fill_slab_kernel<<<(unsigned)grid, 32 * kFillWarps, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace tc3d
