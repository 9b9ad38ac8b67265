// fill.cu -- the bias fill of a transposed conv's outputs that the engine
// does not write (tap-less parity classes), run beside the engine.
#include "engine.cuh"
#include "ptx.cuh"

#include <algorithm>
#include <cstdint>

namespace tc3d {

namespace {

// Bias fill of the outputs the engine does not write.  Per (n, c) slice,
// with zl = s_out * M clipped to O (rows m >= M of the transposed-conv row
// grid hold only tap-less classes):
//   planes z >= zl0, rows y >= zl1: the whole x range;
//   in row mode (s0 > 0: the engine writes only the rows of the class pair
//   (r0, r1) of its one class with taps): planes with z % s0 != r0 and rows
//   with y % s1 != r1, the whole x range;
//   the engine's rows: x in [zl2, O2).
// Work unit: one plane of one slice, one warp.  Spans go out
// as bulk copies (TMA engine) from a per-warp shared buffer holding the
// bias, with scalar stores for the ends off the 16-byte grid; scattered rows
// take one lane each.  Blocks are small (4 warps of 32 registers, 8 KB of
// shared memory) so that one fits on an SM beside an engine CTA: the fill
// runs concurrently with the engine, and costs it few issue slots.
constexpr int kFillWarps = 4;
constexpr int kFillBuf = 512;  // floats of a warp's bias buffer

// [p, p + n) from buffer src (a bulk copy per kFillBuf floats, issued by
// lanes in turn; scalar ends)
__device__ __forceinline__ void fill_span(float* p, long long n, float b, uint32_t src, int lane) {
  const int to16 = (int)((4 - ((reinterpret_cast<uintptr_t>(p) >> 2) & 3)) & 3);
  const int head = n < to16 ? (int)n : to16;
  if (lane < head) p[lane] = b;
  p += head;
  n -= head;
  const long long mid = n & ~3LL;
  if (lane < (int)(n - mid)) p[mid + lane] = b;
  const long long chunks = (mid + kFillBuf - 1) / kFillBuf;
  for (long long c = lane; c < chunks; c += 32) {
    const long long o = c * kFillBuf;
    const long long len = mid - o < kFillBuf ? mid - o : kFillBuf;
    bulk_s2g(p + o, src, (uint32_t)(len * 4));
  }
}

// rows y_j = s j + r (j < nrows) of a plane, x in [x0, O2): lane per row
__device__ __forceinline__ void fill_rows_run(float* plane, int nrows, int s, int r, int x0, int O2,
                                              float b, uint32_t src, int lane) {
  for (int j = lane; j < nrows; j += 32) {
    float* row = plane + (long long)(s * j + r) * O2 + x0;
    const int n = O2 - x0;
    const int to16 = (int)((4 - ((reinterpret_cast<uintptr_t>(row) >> 2) & 3)) & 3);
    const int head = n < to16 ? n : to16;
    for (int i = 0; i < head; ++i) row[i] = b;
    const int rest = n - head, mid = rest & ~3;
    for (int i = head + mid; i < n; ++i) row[i] = b;
    for (int o = 0; o < mid; o += kFillBuf) {
      const int len = mid - o < kFillBuf ? mid - o : kFillBuf;
      bulk_s2g(row + head + o, src, (uint32_t)(len * 4));
    }
  }
}

__global__ void __launch_bounds__(32 * kFillWarps, 16) fill_slab_kernel(const __grid_constant__ FillParams p) {
  __shared__ __align__(128) float buf[kFillWarps][kFillBuf];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long u = (long long)blockIdx.x * kFillWarps + warp;
  if (u >= (long long)p.NC * p.O[0]) return;
  const int nc = (int)(u / p.O[0]), z = (int)(u - (long long)nc * p.O[0]);
  const float b = p.bias ? __ldg(p.bias + nc % p.Cout) : 0.f;
  for (int i = lane; i < kFillBuf; i += 32) buf[warp][i] = b;
  fence_proxy_async_smem();
  __syncwarp();
  const uint32_t src = smem_u32(&buf[warp][0]);
  const int O1 = p.O[1], O2 = p.O[2];
  float* plane = p.y + ((long long)nc * p.O[0] + z) * ((long long)O1 * O2);
  if (z >= p.zl[0] || (p.s0 > 0 && z % p.s0 != p.r0)) {
    fill_span(plane, (long long)O1 * O2, b, src, lane);
  } else {
    const int zl1 = p.zl[1];
    // the rows y < zl1 of the fill (y % s1 != r1): for each of the s1 - 1
    // residues a run of rows with stride s1
    if (p.s0 > 0)
      for (int rr = 0; rr < p.s1; ++rr)
        if (rr != p.r1 && rr < zl1)
          fill_rows_run(plane, (zl1 - rr + p.s1 - 1) / p.s1, p.s1, rr, 0, O2, b, src, lane);
    // the engine's rows past x = zl2
    if (p.zl[2] < O2) {
      const int s = p.s0 > 0 ? p.s1 : 1, r = p.s0 > 0 ? p.r1 : 0;
      if (r < zl1) fill_rows_run(plane, (zl1 - r + s - 1) / s, s, r, p.zl[2], O2, b, src, lane);
    }
    if (zl1 < O1) fill_span(plane + (long long)zl1 * O2, (long long)(O1 - zl1) * O2, b, src, lane);
  }
  // the copies have read the buffer before the warp leaves (their writes
  // complete with the grid)
  bulk_commit();
  bulk_wait_read();
}

}  // namespace

cudaError_t fill_slab_launch(const FillParams& p, cudaStream_t st) {
  // a warp per (slice, plane)
  const long long units = (long long)p.NC * p.O[0];
  const long long grid = (units + kFillWarps - 1) / kFillWarps;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  // the largest shared-memory carveout, the engine's: an SM holds CTAs of
  // one carveout at a time, so only then can a fill CTA join an engine CTA
  const cudaError_t e = cudaFuncSetAttribute(fill_slab_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  fill_slab_kernel<<<(unsigned)grid, 32 * kFillWarps, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace tc3d
