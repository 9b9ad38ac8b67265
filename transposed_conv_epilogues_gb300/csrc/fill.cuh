// fill.cuh -- the bias fill of a transposed conv's outputs that the engine
// does not write (tap-less parity classes): one plane of one (n, c) slice per
// call, by one warp, with streaming vector stores.  Used by the engine's
// epilogue warps and by the stand-alone fill kernel (grids without engine
// tiles).  Plain stores, not bulk copies: inside the engine the
// SM's TMA unit is busy with the input boxes and weight stages, and a queue
// of fill copies ahead of them would hold the MMAs up.
#pragma once
#include "engine.cuh"

namespace tc3d {

// [p, p + n) = b: 16-byte streaming stores by the warp's lanes, scalar
// stores for the ends off the 16-byte grid
__device__ __forceinline__ void fill_span(float* p, long long n, float b, int lane) {
  const int to16 = (int)((4 - ((reinterpret_cast<uintptr_t>(p) >> 2) & 3)) & 3);
  const int head = n < to16 ? (int)n : to16;
  if (lane < head) __stcs(p + lane, b);
  p += head;
  n -= head;
  const long long nvec = n >> 2;
  if (lane < (int)(n & 3)) __stcs(p + 4 * nvec + lane, b);
  float4* q = reinterpret_cast<float4*>(p);
  const float4 b4 = make_float4(b, b, b, b);
  for (long long i = lane; i < nvec; i += 32) __stcs(q + i, b4);
}

// rows y_j = s j + r (j < nrows) of a plane, x in [x0, O2): the warp per row
// for long rows, a lane per row for short ones
__device__ __forceinline__ void fill_rows_run(float* plane, int nrows, int s, int r, int x0, int O2,
                                              float b, int lane) {
  const int n = O2 - x0;
  if (n >= 32) {
    for (int j = 0; j < nrows; ++j) fill_span(plane + (long long)(s * j + r) * O2 + x0, n, b, lane);
    return;
  }
  for (int j = lane; j < nrows; j += 32) {
    float* row = plane + (long long)(s * j + r) * O2 + x0;
    for (int i = 0; i < n; ++i) __stcs(row + i, b);
  }
}

// The fill of plane z of slice nc.  With zl = s_out * M clipped to O (rows m
// >= M of the transposed-conv row grid hold only tap-less classes):
//   planes z >= zl0, rows y >= zl1: the whole x range;
//   in row mode (s0 > 0: the engine writes only the rows of the class pair
//   (r0, r1) of its one class with taps): planes with z % s0 != r0 and rows
//   with y % s1 != r1, the whole x range;
//   the engine's rows: x in [zl2, O2).
__device__ __forceinline__ void fill_plane(const FillParams& p, int nc, int z, float b, int lane) {
  const int O1 = p.O[1], O2 = p.O[2];
  float* plane = p.y + ((long long)nc * p.O[0] + z) * ((long long)O1 * O2);
  if (z >= p.zl[0] || (p.s0 > 0 && z % p.s0 != p.r0)) {
    fill_span(plane, (long long)O1 * O2, b, lane);
    return;
  }
  const int zl1 = p.zl[1];
  // the rows y < zl1 of the fill (y % s1 != r1): for each of the s1 - 1
  // residues a run of rows with stride s1
  if (p.s0 > 0)
    for (int rr = 0; rr < p.s1; ++rr)
      if (rr != p.r1 && rr < zl1)
        fill_rows_run(plane, (zl1 - rr + p.s1 - 1) / p.s1, p.s1, rr, 0, O2, b, lane);
  // the engine's rows past x = zl2
  if (p.zl[2] < O2) {
    const int s = p.s0 > 0 ? p.s1 : 1, r = p.s0 > 0 ? p.r1 : 0;
    if (r < zl1) fill_rows_run(plane, (zl1 - r + s - 1) / s, s, r, p.zl[2], O2, b, lane);
  }
  if (zl1 < O1) fill_span(plane + (long long)zl1 * O2, (long long)(O1 - zl1) * O2, b, lane);
}

}  // namespace tc3d
