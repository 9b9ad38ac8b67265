// lag.cu -- batch statistics of the algebraic BN-pool path in lag form (see
// lag_slot in plan.h): per region of x, the sums of x[c, z] and of the
// products x[c, z] x[c', z + delta], delta in {-1, 0, 1}^3, on CUDA cores,
// then their reduction over the grid.
//
// Why not the tensor core.  The same statistics as patch Gram matrices are a
// GEMM with M = N = D <= 24 and K = rows; a tcgen05 MMA has 128 rows (64 at
// half width), so at least 5x of its work would be padding, and its A operand
// (the patches, with their low parts) would have to be written to shared
// memory first, 2 x 24 floats per row.  The lag form needs 126 multiply-adds
// per input position and no staging beyond the input itself; on CUDA cores it
// is the cheaper of the two.
//
// Work: a CTA (8 warps) takes one job, (segment s0 of axis 0, 8 rows of axis
// 1, 32 columns of axis 2), and a share of its (sample, plane) steps.  Warp w
// owns row 8 b1 + w, lane l column 32 b2 + l; the thread walks its column
// along axis 0 with the 3 x 3 (row, column) window of the planes z0 and z0 + 1
// in registers (the products with plane z0 - 1 are taken one step earlier,
// as those of z0 + 1 with z0).  Each warp brings its window planes in by TMA
// (box: 40 columns x 3 rows x 4 planes x Cin channels, zero outside x) into a
// ring of its own in shared memory; every step reads one new plane.  A
// thread's positions all lie in one region (its row and column fix two
// segments, the job the third), so it keeps one set of sums, reduced per
// region at the end and written as its share of every box sum (a box: one
// segment range per axis, the z range of a class entry's first factor).
#include <type_traits>

#include "pool.cuh"
#include "ptx.cuh"

namespace tc3d {

namespace {

constexpr int kLagThreads = kLagRows * 32;
// registers a thread: the finalize kernels launched while this one runs
// need 4096 of the SM's 65536 beside its 256 threads
constexpr int kLagMaxRegs = 232;
constexpr int kLagRing = 3;                   // chunk slots per warp
constexpr int kLagPlane = kLagBoxRows * kLagBoxCols;  // floats of one channel's window plane
// a chunk slot holds one box: [Cin][kLagChunk planes][3 rows][40 columns];
// tensor copies write to 128-byte aligned shared memory, so slots are
// 128-byte multiples
constexpr int kLagChunkFloats = (kLagMaxCin * kLagChunk * kLagPlane + 31) / 32 * 32;
constexpr int kLagRedStride = kLagSlots + 1;  // per-thread row of the end reduction
constexpr int kLagMaxReg2 = kLagMaxSeg * kLagMaxSeg;

// dynamic shared memory (float indices from a 128-byte aligned base): [per-warp
// rings | end-reduction rows (aliases the rings)] [per-region sums, two
// halves] [per-warp barriers]
constexpr int kLagRingFloats = kLagRows * kLagRing * kLagChunkFloats;
constexpr int kLagRedFloats = kLagThreads * kLagRedStride;
constexpr int kLagBufFloats =
    ((kLagRedFloats > kLagRingFloats ? kLagRedFloats : kLagRingFloats) + 31) / 32 * 32;
constexpr int kLagOutFloats = 2 * kLagMaxReg2 * kLagSlots;
constexpr int kLagBarFloat = kLagBufFloats + kLagOutFloats;
constexpr size_t kLagSmem = ((size_t)kLagBarFloat + 2 * kLagRows * kLagRing) * 4 + 128;

extern __shared__ __align__(128) float lag_dsm[];

// next chunk (sample n, first plane z) of the stream a CTA reads: its steps
// are items [it, i1) of (sample, plane in the segment); a run of consecutive
// planes za .. zb - 1 of one sample reads the planes za - 1 .. zb, in chunks
// of kLagChunk consecutive planes from za - 1
struct ChunkCursor {
  long long it, i1;
  int len, z0a;
  int n, z, zend;
};

__device__ __forceinline__ bool next_chunk(ChunkCursor& c, int& n, int& z) {
  if (c.z > c.zend) {
    if (c.it >= c.i1) return false;
    c.n = (int)(c.it / c.len);
    const int za = c.z0a + (int)(c.it - (long long)c.n * c.len);
    const long long rend = min(c.i1, (long long)(c.n + 1) * c.len);
    c.zend = c.z0a + (int)(rend - (long long)c.n * c.len);
    c.z = za - 1;
    c.it = rend;
  }
  n = c.n;
  z = c.z;
  c.z += kLagChunk;
  return true;
}

// One warp's walk: its row of the job, its own ring of chunks (TMA box of
// 40 columns x 3 rows x 4 planes x Cin channels; lane 0 keeps up to
// kLagRing - 1 chunks in flight ahead of the warp's reads), so warps never
// wait for one another.
template <int CIN>
struct LagWarp {
  static constexpr int NS = lag_nslots(CIN);
  const CUtensorMap* map;
  int ring;        // float index of this warp's slot 0
  uint32_t full0;  // barrier of slot 0 (slot i: full0 + 8 i)
  unsigned long long tmo;
  int* err;
  volatile int* abortf;
  int lane, z1, c2x;  // c2x: column of the box's first element
  int qc = 0, qi = 0; // chunk being read, chunks issued
  int cslot = 0;      // slot of chunk qc
  uint32_t cpar = 0;  // parity of chunk qc's barrier phase
  int k = 0;          // plane of the run being read next (0 = za - 1)
  int b = 0;          // float index of this lane's window corner in the last plane read
  ChunkCursor cc;
  bool ok = true;

  // lane 0: issue the chunks of stream index < limit (a slot is refilled
  // only after the warp moved on from it)
  __device__ __forceinline__ void produce(int limit) {
    int n, z;
    while (qi < limit && next_chunk(cc, n, z)) {
      const int slot = qi % kLagRing;
      const uint32_t bar = full0 + 8u * (uint32_t)slot;
      mbar_arrive_expect_tx(bar, (uint32_t)(CIN * kLagChunk * kLagPlane * 4));
      tma_load_5d(smem_u32(lag_dsm + ring + slot * kLagChunkFloats), map, c2x, z1 - 1, z, 0, n,
                  bar);
      ++qi;
    }
  }

  // wait for chunk qc (lane 0 first tops up the chunks in flight)
  __device__ __forceinline__ void wait_chunk() {
    if (lane == 0) produce(qc + kLagRing);
    if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8u * (uint32_t)cslot, cpar, tmo, abortf))) {
      ok = false;
      if (lane == 0) {
        *abortf = 1;
        atomicExch(err, 1);
      }
    }
  }
  __device__ __forceinline__ void next_chunk_slot() {
    ++qc;
    if (++cslot == kLagRing) {
      cslot = 0;
      cpar ^= 1u;
    }
  }

  // the warp's 3 x 3 window of plane k of the run into dst (plane k lies in
  // chunk qc at index k % 4; entering a chunk waits for it).  With live
  // false the run has no plane k: nothing advances, the loads repeat the
  // last plane read (their values are not used), so the step stays free of
  // branches around its loads.
  __device__ __forceinline__ void read_plane(float (&dst)[CIN][9], bool live = true) {
    if (live) {
      const int idx = k & (kLagChunk - 1);
      if (idx == 0) {
        if (k > 0) next_chunk_slot();
        wait_chunk();
      }
      b = ring + cslot * kLagChunkFloats + idx * kLagPlane + 3 + lane;
      ++k;
    }
#pragma unroll
    for (int c = 0; c < CIN; ++c)
#pragma unroll
      for (int dr = 0; dr < 3; ++dr)
#pragma unroll
        for (int dc = 0; dc < 3; ++dc)
          dst[c][dr * 3 + dc] = lag_dsm[b + c * kLagChunk * kLagPlane + dr * kLagBoxCols + dc];
  }
  // a new run starts with a new chunk
  __device__ __forceinline__ void end_run() {
    next_chunk_slot();
    k = 0;
  }

  // products x[c, z'] x[c2, z0, z1 + d1, z2 + d2] of the position z' = (z0 +
  // 1, z1, z2) with the plane before it (delta0 = -1; distinct channels only),
  // from the center of buffer NB (plane z0 + 1) and the window of buffer CB
  // (plane z0).  They belong to z', which lies in the same region as z0
  // whenever both are steps of one run.
  template <int CB, int NB>
  __device__ __forceinline__ void back_products(const float (&win)[2][CIN][9], float (&acc)[NS],
                                                float weight = 1.f) {
#pragma unroll
    for (int c = 0; c < CIN; ++c) {
      const float xn = win[NB][c][4] * weight;  // weight 0: z0 + 1 is not a step of the run
#pragma unroll
      for (int c2 = c + 1; c2 < CIN; ++c2)
#pragma unroll
        for (int qq = 0; qq < 9; ++qq) {
          const int s = lag_slot(CIN, c, c2, qq);
          acc[s] = fmaf(xn, win[CB][c2][qq], acc[s]);
        }
    }
  }

  // one step at plane z0 in buffer PH, plane z0 + 1 in the other.  back:
  // z0 + 1 is a step of this run (take its products with z0); more: read the
  // plane z0 + 2 into buffer PH once z0's window is no longer needed.
  template <int PH>
  __device__ __forceinline__ void step(float (&win)[2][CIN][9], float (&acc)[NS], bool back,
                                       bool more) {
    constexpr int C = PH, NX = 1 - PH;
    float xc[CIN];
#pragma unroll
    for (int c = 0; c < CIN; ++c) {
      xc[c] = win[C][c][4];
      acc[c] += xc[c];
    }
    // delta0 = 0 (j = 9 + qq): for one channel only the lags after 0, and 0
#pragma unroll
    for (int c = 0; c < CIN; ++c)
#pragma unroll
      for (int c2 = c; c2 < CIN; ++c2)
#pragma unroll
        for (int qq = 0; qq < 9; ++qq) {
          if (c2 == c && qq < 4) continue;
          const int s = lag_slot(CIN, c, c2, 9 + qq);
          acc[s] = fmaf(xc[c], win[C][c2][qq], acc[s]);
        }
    back_products<C, NX>(win, acc, back ? 1.f : 0.f);
    read_plane(win[C], more);
    // delta0 = +1 (j = 18 + qq)
#pragma unroll
    for (int c = 0; c < CIN; ++c)
#pragma unroll
      for (int c2 = c; c2 < CIN; ++c2)
#pragma unroll
        for (int qq = 0; qq < 9; ++qq) {
          const int s = lag_slot(CIN, c, c2, 18 + qq);
          acc[s] = fmaf(xc[c], win[NX][c2][qq], acc[s]);
        }
  }
};

// Three channels: the sums of one thread, with the second-factor channels 1
// and 2 paired in float2 lanes so that one packed multiply-add (f32x2)
// updates both.  Window planes are kept the same way: w0 = channel 0, w12 =
// (channel 1, channel 2), each 3 x 3 (row, column) positions q.
struct Win3 {
  float w0[9];
  float2 w12[9];
};
struct Acc3 {
  float s[3];      // sums of x[c, z]
  float2 p0[27];   // c = 0, c2 = (1, 2), lags j = 0..26
  float2 p1[14];   // c = 1, c2 = (1, 2), j = 13..26
  float s00[14];   // c = 0, c2 = 0, j = 13..26
  float s12[13];   // c = 1, c2 = 2, j = 0..12
  float s22[14];   // c = 2, c2 = 2, j = 13..26
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < 3; ++i) s[i] = 0.f;
#pragma unroll
    for (int i = 0; i < 27; ++i) p0[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 14; ++i) {
      p1[i] = make_float2(0.f, 0.f);
      s00[i] = 0.f;
      s22[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < 13; ++i) s12[i] = 0.f;
  }
  // every sum to its slot (lag_slot order) in a row of the end reduction
  __device__ __forceinline__ void store(float* row) const {
#pragma unroll
    for (int c = 0; c < 3; ++c) row[c] = s[c];
#pragma unroll
    for (int j = 0; j < 27; ++j) {
      row[lag_slot(3, 0, 1, j)] = p0[j].x;
      row[lag_slot(3, 0, 2, j)] = p0[j].y;
    }
#pragma unroll
    for (int j = 13; j < 27; ++j) {
      row[lag_slot(3, 1, 1, j)] = p1[j - 13].x;
      row[lag_slot(3, 1, 2, j)] = p1[j - 13].y;
      row[lag_slot(3, 0, 0, j)] = s00[j - 13];
      row[lag_slot(3, 2, 2, j)] = s22[j - 13];
    }
#pragma unroll
    for (int j = 0; j < 13; ++j) row[lag_slot(3, 1, 2, j)] = s12[j];
  }
};

// the paired form of LagWarp's window read and step (three channels)
struct LagWarp3 : LagWarp<3> {
  __device__ __forceinline__ void read_plane3(Win3& dst, bool live = true) {
    if (live) {
      const int idx = k & (kLagChunk - 1);
      if (idx == 0) {
        if (k > 0) next_chunk_slot();
        wait_chunk();
      }
      b = ring + cslot * kLagChunkFloats + idx * kLagPlane + 3 + lane;
      ++k;
    }
    constexpr int cs = kLagChunk * kLagPlane;  // channel stride in a chunk
#pragma unroll
    for (int dr = 0; dr < 3; ++dr)
#pragma unroll
      for (int dc = 0; dc < 3; ++dc) {
        const int o = b + dr * kLagBoxCols + dc;
        dst.w0[dr * 3 + dc] = lag_dsm[o];
        dst.w12[dr * 3 + dc] = make_float2(lag_dsm[o + cs], lag_dsm[o + 2 * cs]);
      }
  }
  // products of z' = (z0 + 1, z1, z2) with plane z0 (delta0 = -1, j = q;
  // distinct channels only), weighted 0 when z' is not a step of the run
  __device__ __forceinline__ void back3(const Win3& cw, const Win3& nw, Acc3& a, float weight) {
    const float xn0 = nw.w0[4] * weight, xn1 = nw.w12[4].x * weight;
    const float2 d0 = make_float2(xn0, xn0);
#pragma unroll
    for (int q = 0; q < 9; ++q) {
      a.p0[q] = __ffma2_rn(d0, cw.w12[q], a.p0[q]);
      a.s12[q] = fmaf(xn1, cw.w12[q].y, a.s12[q]);
    }
  }
  // one step at plane z0 (cw), plane z0 + 1 (nw); reads plane z0 + 2 into
  // cw once z0's window is no longer needed
  __device__ __forceinline__ void step3(Win3& cw, Win3& nw, Acc3& a, bool back, bool more) {
    const float x0 = cw.w0[4], x1 = cw.w12[4].x, x2 = cw.w12[4].y;
    a.s[0] += x0;
    a.s[1] += x1;
    a.s[2] += x2;
    const float2 d0 = make_float2(x0, x0), d1 = make_float2(x1, x1);
    // delta0 = 0: j = 9 + q
#pragma unroll
    for (int q = 0; q < 9; ++q) {
      a.p0[9 + q] = __ffma2_rn(d0, cw.w12[q], a.p0[9 + q]);
      if (q >= 4) {
        a.s00[q - 4] = fmaf(x0, cw.w0[q], a.s00[q - 4]);
        a.p1[q - 4] = __ffma2_rn(d1, cw.w12[q], a.p1[q - 4]);
        a.s22[q - 4] = fmaf(x2, cw.w12[q].y, a.s22[q - 4]);
      } else {
        a.s12[9 + q] = fmaf(x1, cw.w12[q].y, a.s12[9 + q]);
      }
    }
    back3(cw, nw, a, back ? 1.f : 0.f);
    read_plane3(cw, more);
    // delta0 = +1: j = 18 + q
#pragma unroll
    for (int q = 0; q < 9; ++q) {
      a.p0[18 + q] = __ffma2_rn(d0, nw.w12[q], a.p0[18 + q]);
      a.s00[5 + q] = fmaf(x0, nw.w0[q], a.s00[5 + q]);
      a.p1[5 + q] = __ffma2_rn(d1, nw.w12[q], a.p1[5 + q]);
      a.s22[5 + q] = fmaf(x2, nw.w12[q].y, a.s22[5 + q]);
    }
  }
};

// segment of position z along axis a (positions past x: the wide segment;
// their values are zero)
__device__ __forceinline__ int seg_of(const LagParams& p, int a, int z) {
  if (z >= p.L[a]) return p.bulk[a];
  int s = 0;
  while (s + 1 < p.nseg[a] && z >= p.seg[a][s + 1]) ++s;
  return s;
}

template <int CIN>
__global__ void __maxnreg__(kLagMaxRegs) lag_stats_kernel(const __grid_constant__ LagParams p) {
  constexpr int NS = lag_nslots(CIN);
  // float index of the 128-byte aligned base
  const int a0 = (int)(((128u - (smem_u32(lag_dsm) & 127u)) & 127u) >> 2);
  float* buf = lag_dsm + a0;
  float* outa = buf + kLagBufFloats;
  __shared__ int segw[kLagRows], segl[32];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // the job of this CTA
  int s0 = 0;
  while (s0 + 1 < p.nseg[0] && (int)blockIdx.x >= p.cta0[s0 + 1]) ++s0;
  const int local = (int)blockIdx.x - p.cta0[s0];
  const int nc = p.nc[s0];
  const int job = local / nc, kc = local - job * nc;
  const int b1 = job / p.nb2, b2 = job - b1 * p.nb2;
  const int z0a = p.seg[0][s0], len = p.seg[0][s0 + 1] - z0a;
  const long long items = (long long)p.N * len;
  const long long i0 = items * kc / nc, i1 = items * (kc + 1) / nc;

  typename std::conditional<CIN == 3, LagWarp3, LagWarp<CIN>>::type lw;
  lw.map = &p.xmap;
  lw.ring = a0 + warp * kLagRing * kLagChunkFloats;
  lw.full0 = smem_u32(buf + kLagBarFloat) + 8u * (uint32_t)(warp * kLagRing);
  lw.tmo = p.timeout_cycles;
  lw.err = p.err;
  lw.abortf = &abort_flag;
  lw.lane = lane;
  lw.z1 = kLagRows * b1 + warp;
  lw.c2x = kLagCols * b2 - 4;
  lw.cc.it = i0;
  lw.cc.i1 = i1;
  lw.cc.len = len;
  lw.cc.z0a = z0a;
  lw.cc.z = 1;
  lw.cc.zend = 0;

  if (lane == 0) {
    for (int i = 0; i < kLagRing; ++i) mbar_init(lw.full0 + 8u * i, 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    prefetch_tensormap(&p.xmap);
  }
  // The finalize kernels that follow may be launched now: this kernel is
  // launched normally (all work queued before it has finished), and what
  // they do before their own wait reads only the call's inputs and writes
  // only buffers no kernel of the call before them touches.  Small enough
  // to share an SM with this kernel, they stage their tables meanwhile.
  grid_launch_dependents();
  if (threadIdx.x < kLagRows) segw[threadIdx.x] = seg_of(p, 1, kLagRows * b1 + threadIdx.x);
  if (threadIdx.x < 32) segl[threadIdx.x] = seg_of(p, 2, kLagCols * b2 + threadIdx.x);
  __syncthreads();

  // runs of consecutive planes za .. zb - 1 of one sample; a run reads the
  // planes za - 1 .. zb.  Two steps per iteration: plane z0 in window
  // buffer 1, then z0 + 1 in buffer 0.
  float acc[CIN == 3 ? 1 : NS];
  Acc3 acc3;
  if constexpr (CIN == 3) {
    acc3.zero();
    Win3 wa, wb;  // buffers 0 and 1
    bool first = true;
    for (long long it = i0; it < i1 && lw.ok;) {
      const int n = (int)(it / len);
      const int za = z0a + (int)(it - (long long)n * len);
      const long long rend = min(i1, (long long)(n + 1) * len);
      const int zb = z0a + (int)(rend - (long long)n * len);
      it = rend;
      if (!first) lw.end_run();
      first = false;
      lw.read_plane3(wa);  // za - 1
      lw.read_plane3(wb);  // za
      if (!lw.ok) break;
      lw.back3(wa, wb, acc3, 1.f);  // za with za - 1
      lw.read_plane3(wa);           // za + 1
      int z0 = za;
      for (; z0 + 1 < zb && lw.ok; z0 += 2) {
        lw.step3(wb, wa, acc3, true, z0 + 2 <= zb);
        lw.step3(wa, wb, acc3, z0 + 2 < zb, z0 + 3 <= zb);
      }
      if (z0 < zb && lw.ok) lw.step3(wb, wa, acc3, false, false);
    }
  } else {
#pragma unroll
    for (int s = 0; s < NS; ++s) acc[s] = 0.f;
    float win[2][CIN][9];
    bool first = true;
    for (long long it = i0; it < i1 && lw.ok;) {
      const int n = (int)(it / len);
      const int za = z0a + (int)(it - (long long)n * len);
      const long long rend = min(i1, (long long)(n + 1) * len);
      const int zb = z0a + (int)(rend - (long long)n * len);
      it = rend;
      if (!first) lw.end_run();
      first = false;
      lw.read_plane(win[0]);  // za - 1
      lw.read_plane(win[1]);  // za
      if (!lw.ok) break;
      lw.template back_products<0, 1>(win, acc);  // za with za - 1
      lw.read_plane(win[0]);                      // za + 1
      int z0 = za;
      for (; z0 + 1 < zb && lw.ok; z0 += 2) {
        lw.template step<1>(win, acc, true, z0 + 2 <= zb);
        lw.template step<0>(win, acc, z0 + 2 < zb, z0 + 3 <= zb);
      }
      if (z0 < zb && lw.ok) lw.template step<1>(win, acc, false, false);
    }
  }
  // on a time-out, the chunks still in flight land before the warp leaves
  if (lane == 0 && !lw.ok) {
    for (int q = lw.qc; q < lw.qi; ++q)
      mbar_wait(lw.full0 + 8u * (uint32_t)(q % kLagRing), (uint32_t)((q / kLagRing) & 1), lw.tmo,
                nullptr);
  }
  __syncthreads();
  if (abort_flag) return;

  // per-region sums: every thread's sums into a row of the (former) rings,
  // then thread (h, k) adds slot k over the lanes of warps 4h .. 4h + 3
  float* red = buf;
  if constexpr (CIN == 3) {
    acc3.store(red + threadIdx.x * kLagRedStride);
  } else {
#pragma unroll
    for (int s = 0; s < NS; ++s) red[threadIdx.x * kLagRedStride + s] = acc[s];
  }
  for (int e = threadIdx.x; e < kLagOutFloats; e += kLagThreads) outa[e] = 0.f;
  // runs of lanes (columns) of one segment: run i is lanes [lrun[i], lrun[i +
  // 1]) of segment lseg[i] (a segment may recur: columns past x take the
  // wide one)
  __shared__ int lrun[33], lseg[32], nlrun;
  if (warp == 0) {
    const bool start = lane == 0 || segl[lane] != segl[lane - 1];
    const unsigned m = __ballot_sync(0xffffffffu, start);
    if (start) {
      const int i = __popc(m & ((1u << lane) - 1u));
      lrun[i] = lane;
      lseg[i] = segl[lane];
    }
    if (lane == 0) {
      lrun[__popc(m)] = 32;
      nlrun = __popc(m);
    }
  }
  __syncthreads();
  {
    // thread (h, k) adds slot k over the lanes of warps 4h .. 4h + 3, run by
    // run, 8 loads in flight (each (region, slot) cell of a half has one
    // writer)
    const int h = threadIdx.x >> 7, k = threadIdx.x & 127;
    if (k < NS) {
      float* oh = outa + (size_t)h * kLagMaxReg2 * kLagSlots + k;
      for (int wv = 4 * h; wv < 4 * h + 4; ++wv) {
        const int base = segw[wv] * kLagMaxSeg;  // region (s1, s2) at s1 kLagMaxSeg + s2
        const float* col = red + (size_t)wv * 32 * kLagRedStride + k;
        for (int i = 0; i < nlrun; ++i) {
          const int l1 = lrun[i + 1];
          int l = lrun[i];
          float a[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) a[u] = 0.f;
          for (; l + 8 <= l1; l += 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u) a[u] += col[(l + u) * kLagRedStride];
          }
#pragma unroll
          for (int u = 0; u < 7; ++u)
            if (l + u < l1) a[u] += col[(l + u) * kLagRedStride];
          oh[(base + lseg[i]) * kLagSlots] += ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
        }
      }
    }
  }
  __syncthreads();
  // this CTA's share of every box sum (the boxes whose axis-0 range holds
  // its segment s0): the sum of its regions inside the box.  Per slot k:
  // R[s1][s2] = both halves; T[s1][b2] = sum of R over range b2 of axis 2;
  // box (b0, b1, b2) = [s0 in range b0] * sum of T over range b1 of axis 1.
  // The ranges as bit masks of segments, the sums unrolled over the maxima.
  if (threadIdx.x < 128) {
    const int k = threadIdx.x;
    const int nr0 = p.nrange[0], nr1 = p.nrange[1], nr2 = p.nrange[2];
    unsigned m1[4], m2[4];
    bool in0[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      m1[b] = b < nr1 ? (1u << p.range[1][b][1]) - (1u << p.range[1][b][0]) : 0u;
      m2[b] = b < nr2 ? (1u << p.range[2][b][1]) - (1u << p.range[2][b][0]) : 0u;
      in0[b] = b < nr0 && s0 >= p.range[0][b][0] && s0 < p.range[0][b][1];
    }
    // the region sums, loaded unconditionally (the region table has room
    // for kLagMaxSeg^2 regions; cells past (ns1, ns2) are zero)
    float R[kLagMaxSeg][kLagMaxSeg];
#pragma unroll
    for (int s1 = 0; s1 < kLagMaxSeg; ++s1)
#pragma unroll
      for (int s2 = 0; s2 < kLagMaxSeg; ++s2) {
        const int r = s1 * kLagMaxSeg + s2;
        R[s1][s2] = outa[r * kLagSlots + k] + outa[(kLagMaxReg2 + r) * kLagSlots + k];
      }
    float* dst = p.part + (size_t)blockIdx.x * p.nbox * kLagSlots + k;
#pragma unroll
    for (int b2 = 0; b2 < 4; ++b2) {
      if (b2 >= nr2) break;
      float T[kLagMaxSeg];
#pragma unroll
      for (int s1 = 0; s1 < kLagMaxSeg; ++s1) {
        float t = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < kLagMaxSeg; ++s2) t += ((m2[b2] >> s2) & 1u) ? R[s1][s2] : 0.f;
        T[s1] = t;
      }
#pragma unroll
      for (int b1 = 0; b1 < 4; ++b1) {
        if (b1 >= nr1) break;
        float v = 0.f;
#pragma unroll
        for (int s1 = 0; s1 < kLagMaxSeg; ++s1) v += ((m1[b1] >> s1) & 1u) ? T[s1] : 0.f;
#pragma unroll
        for (int b0 = 0; b0 < 4; ++b0) {
          if (b0 >= nr0) break;
          dst[((b0 * nr1 + b1) * nr2 + b2) * kLagSlots] = in0[b0] ? v : 0.f;
        }
      }
    }
  }
}

}  // namespace

size_t lag_smem_bytes() { return kLagSmem; }

cudaError_t lag_set_smem() {
  cudaError_t e = cudaSuccess;
  // the largest shared-memory carveout: the finalize kernels launched while
  // this one runs take the SMs' leftover shared memory, and an SM holds CTAs
  // of one carveout at a time
  for (const void* f : {(const void*)lag_stats_kernel<1>, (const void*)lag_stats_kernel<2>,
                        (const void*)lag_stats_kernel<3>}) {
    const cudaError_t ec = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                (int)cudaSharedmemCarveoutMaxShared);
    if (ec != cudaSuccess) e = ec;
  }
  const cudaError_t e1 = cudaFuncSetAttribute(lag_stats_kernel<1>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLagSmem);
  const cudaError_t e2 = cudaFuncSetAttribute(lag_stats_kernel<2>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLagSmem);
  const cudaError_t e3 = cudaFuncSetAttribute(lag_stats_kernel<3>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLagSmem);
  if (e1 != cudaSuccess) e = e1;
  if (e2 != cudaSuccess) e = e2;
  if (e3 != cudaSuccess) e = e3;
  return e;
}

cudaError_t lag_launch(const LagParams& p, int cin, cudaStream_t st) {
  switch (cin) {
    case 1: lag_stats_kernel<1><<<p.grid, kLagThreads, kLagSmem, st>>>(p); break;
    case 2: lag_stats_kernel<2><<<p.grid, kLagThreads, kLagSmem, st>>>(p); break;
    case 3: lag_stats_kernel<3><<<p.grid, kLagThreads, kLagSmem, st>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace tc3d
