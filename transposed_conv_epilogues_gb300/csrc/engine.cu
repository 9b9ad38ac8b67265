// engine.cu -- the implicit-GEMM convolution engine for sm_103a.
//
// One persistent CTA per SM walks its share of tiles.  A tile is n_acc
// accumulators of 128 rows (see plan.cpp for what a row is); every
// accumulator is a 128 x n_tile fp32 block in tensor memory (TMEM).  Per
// tile, per column block and per channel chunk:
//
//   warp 0  (raw producer)   one TMA box load of the raw fp32 input region
//                            the tile's rows read (zero fill = padding)
//   warp 1  (B producer)     bulk copies of pre-packed weight K-steps
//                            (resident in shared memory when they fit)
//   last 8 warps (conversion) gather, for each K-step of 8 (channel, tap)
//                            pairs and each row, x and x - trunc_tf32(x) from
//                            the raw box and store them to TMEM (A operand)
//   warps 2, 3 (MMA)         tcgen05.mma kind::tf32, A from TMEM, B from
//                            shared memory: D += A.Bw + A.Blo + Alo.Bw
//                            (3xTF32: the tensor core reads the top 19 bits
//                            of each fp32 operand, so x itself is the "hi"
//                            part and only the low parts are formed).  Warp
//                            2 issues for the even accumulators, warp 3 for
//                            the odd ones, so that one issuer's barrier wait
//                            and commit overlap the other's queued MMAs.
//   warps 4.. (epilogue)     tcgen05.ld of D and the fused epilogue
//   The store epilogue's warps also do the bias fill of a transposed conv's
//   outputs that no tile writes: a part of it per tile iteration, and what
//   is left after their last tile.
//
// Every mbarrier wait is bounded; on time-out the CTA sets an error word and
// all roles return, TMEM is freed, the kernel exits.
#include "engine.cuh"
#include "fill.cuh"
#include "ptx.cuh"

namespace tc3d {

// Set to 1 by any CTA whose bounded wait ran out; read and cleared by the host.
__device__ int g_tc3d_error = 0;

cudaError_t error_flag_address(int** addr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(addr), g_tc3d_error);
}

namespace {

struct Bars {
  uint32_t base;
  __device__ __forceinline__ uint32_t raw_full(int i) const { return base + 8u * i; }
  __device__ __forceinline__ uint32_t raw_empty(int i) const { return base + 24u + 8u * i; }
  __device__ __forceinline__ uint32_t b_full(int i) const { return base + 48u + 8u * i; }
  __device__ __forceinline__ uint32_t b_empty(int i) const { return base + 176u + 8u * i; }
  __device__ __forceinline__ uint32_t a_full(int i) const { return base + 304u + 8u * i; }
  __device__ __forceinline__ uint32_t a_empty(int i) const { return base + 432u + 8u * i; }
  __device__ __forceinline__ uint32_t d_full(int i) const { return base + 560u + 8u * i; }
  __device__ __forceinline__ uint32_t d_empty(int i) const { return base + 576u + 8u * i; }
  __device__ __forceinline__ uint32_t epi(int i) const { return base + 592u + 8u * i; }
};
constexpr unsigned kBarTmemSlot = 608;
constexpr unsigned kBarAbort = 612;

struct TileCoord {
  int n;
  int o[3];
};

__device__ __forceinline__ TileCoord decode_tile(const EngineParams& p, int t) {
  TileCoord c;
  const int t1 = fast_div(p.ntile_div[2], t);
  const int b2 = t - t1 * p.ntile[2];
  const int t2 = fast_div(p.ntile_div[1], t1);
  const int b1 = t1 - t2 * p.ntile[1];
  c.n = fast_div(p.ntile_div[0], t2);
  const int b0 = t2 - c.n * p.ntile[0];
  c.o[0] = b0 * p.T[0];
  c.o[1] = b1 * p.T[1];
  c.o[2] = b2 * p.T[2];
  return c;
}

// local row coordinates of (accumulator a, lane quarter q, lane l); the
// quarter box Q and the quarter arrangement Pq are powers of two
__device__ __forceinline__ void row_local(const EngineParams& p, int a, int q, int l, int (&t)[3]) {
  const int j = a * 4 + q;
  const int p0 = j >> (p.lPq[1] + p.lPq[2]);
  const int p1 = (j >> p.lPq[2]) & (p.Pq[1] - 1);
  const int p2 = j & (p.Pq[2] - 1);
  const int l0 = l >> (p.lQ[1] + p.lQ[2]);
  const int l1 = (l >> p.lQ[2]) & (p.Q[1] - 1);
  const int l2 = l & (p.Q[2] - 1);
  t[0] = (p0 << p.lQ[0]) + l0;
  t[1] = (p1 << p.lQ[1]) + l1;
  t[2] = (p2 << p.lQ[2]) + l2;
}

// global row coordinates of (accumulator a, lane quarter q, lane l) in the
// tile at origin o, and whether the row lies inside M
__device__ __forceinline__ bool row_global(const EngineParams& p, const int (&o)[3], int a, int q,
                                           int l, int (&m)[3]) {
  int t[3];
  row_local(p, a, q, l, t);
  bool rv = true;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    m[i] = o[i] + t[i];
    rv = rv && m[i] < p.M[i];
  }
  return rv;
}

__device__ __forceinline__ void raise_abort(const EngineParams& p, volatile int* abortf) {
  *abortf = 1;
  atomicExch(p.err, 1);
}

__device__ __forceinline__ float tf32_trunc(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// Sum 8 values over all 32 lanes; lane ends with the total of value index
// 4*b4 + 2*b3 + b2 (b = lane bits).
__device__ __forceinline__ float reduce_scatter8_sum(const float (&v)[8], int lane) {
  float w4[4], w2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b4 ? v[i] : v[i + 4];
    const float keep = b4 ? v[i + 4] : v[i];
    w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b3 ? w4[i] : w4[i + 2];
    const float keep = b3 ? w4[i + 2] : w4[i];
    w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  const float send = b2 ? w2[0] : w2[1];
  const float keep = b2 ? w2[1] : w2[0];
  float w1 = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  w1 += __shfl_xor_sync(0xffffffffu, w1, 2);
  return w1 + __shfl_xor_sync(0xffffffffu, w1, 1);
}
__device__ __forceinline__ int scatter8_index(int lane) {
  return 4 * ((lane >> 4) & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
}

// Sum 8 values over the 8 lanes of a 2x2x2 pool window (lane bits 0, 3, 4);
// lane ends with the total of value index 4*b0 + 2*b3 + b4.
// BN-pool class sums of one row for 8 channels.  u holds, per channel h,
// the 8 parity classes r = 4 r0 + 2 r1 + r2 of the row.  Class r lies inside
// the output iff 2m + r < O on every axis; a row inside M has 2m < O, so
// class r is in iff f_i = [2 m_i + 1 < O_i] holds on every axis with r_i = 1.
// Its weight is f0^r0 f1^r1 f2^r2, and the sums nest as a tree of FMAs over
// those 0/1 weights.  ps[h]: the row's sum (a row whose 4x4x4 window is
// stored has every class inside, so this is then the plain sum of the 8);
// with STATS, the sums and sums of squares also run into s1/s2 with the
// row's weight fr (0 for rows past M).
template <bool STATS>
__device__ __forceinline__ void bn_class_sums(const uint32_t (&u)[64], int nch, float f0, float f1,
                                              float f2, float fr, float (&ps)[8], float (&s1)[8],
                                              float (&s2)[8]) {
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    ps[h] = 0.f;
    if (h >= 4 && nch <= 4) continue;
    float a[4], c[4];  // per (r0, r1): classes r2 = 0, 1 combined
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float ve = __uint_as_float(u[h * 8 + 2 * k]);
      const float vo = __uint_as_float(u[h * 8 + 2 * k + 1]);
      const float w = f2 * vo;
      a[k] = ve + w;
      if (STATS) c[k] = fmaf(w, vo, ve * ve);
    }
    const float sum = fmaf(f0, fmaf(f1, a[3], a[2]), fmaf(f1, a[1], a[0]));
    ps[h] = sum;
    if (STATS) {
      const float sq = fmaf(f0, fmaf(f1, c[3], c[2]), fmaf(f1, c[1], c[0]));
      s1[h] = fmaf(fr, sum, s1[h]);
      s2[h] = fmaf(fr, sq, s2[h]);
    }
  }
}

__device__ __forceinline__ float reduce_scatter8_window_sum(const float (&v)[8], int lane) {
  float w4[4], w2[2];
  const bool b0 = lane & 1, b3 = lane & 8, b4 = lane & 16;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b0 ? v[i] : v[i + 4];
    const float keep = b0 ? v[i + 4] : v[i];
    w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b3 ? w4[i] : w4[i + 2];
    const float keep = b3 ? w4[i + 2] : w4[i];
    w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  const float send = b4 ? w2[0] : w2[1];
  const float keep = b4 ? w2[1] : w2[0];
  return keep + __shfl_xor_sync(0xffffffffu, send, 16);
}
__device__ __forceinline__ int window8_index(int lane) {
  return 4 * (lane & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 4) & 1);
}

// Reduce 16 values over the 8 lanes of a 2x2x2 pool window (lane bits 0, 3,
// 4) with op; lane ends with 2 values of index 8*b0 + 4*b3 + 2*b4 + {0,1}.
template <bool MAX>
__device__ __forceinline__ void reduce_scatter16_window(const float (&v)[16], int lane,
                                                        float (&out)[2]) {
  float w8[8], w4[4];
  const bool b0 = lane & 1, b3 = lane & 8, b4 = lane & 16;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = b0 ? v[i] : v[i + 8];
    const float keep = b0 ? v[i + 8] : v[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 1);
    w8[i] = MAX ? fmaxf(keep, r) : keep + r;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b3 ? w8[i] : w8[i + 4];
    const float keep = b3 ? w8[i + 4] : w8[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 8);
    w4[i] = MAX ? fmaxf(keep, r) : keep + r;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b4 ? w4[i] : w4[i + 2];
    const float keep = b4 ? w4[i + 2] : w4[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 16);
    out[i] = MAX ? fmaxf(keep, r) : keep + r;
  }
}



// Read 32 (16) accumulator columns of this thread's row; with the fused
// [w | w_lo] MMA the accumulator has a second half lo_off columns to the right
// whose values are added.
__device__ __forceinline__ void load_acc32(uint32_t taddr, uint32_t lo_off, uint32_t (&v)[32]) {
  tmem_ld32(taddr, v);
  if (lo_off) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t u[16];
      tmem_ld16(taddr + lo_off + 16 * h, u);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i)
        v[16 * h + i] = __float_as_uint(__uint_as_float(v[16 * h + i]) + __uint_as_float(u[i]));
    }
  } else {
    tmem_wait_ld();
  }
}
__device__ __forceinline__ void load_acc16(uint32_t taddr, uint32_t lo_off, uint32_t (&v)[16]) {
  tmem_ld16(taddr, v);
  if (lo_off) {
    uint32_t u[16];
    tmem_ld16(taddr + lo_off, u);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(u[i]));
  } else {
    tmem_wait_ld();
  }
}

// An MMA issuer.  The whole warp runs this loop (warp-uniform control flow)
// and one elected lane issues each tcgen05 instruction; the loop over this
// warp's NACC accumulators (a = a_first, a_first + a_stride, ...) is unrolled
// at compile time, ring positions advance incrementally and descriptors are
// formed by adds.  Every barrier this warp commits to counts one arrival per
// issuer.  Per (accumulator, K-step):
//   WIDE:  D[0:2n] (+)= x . [w | w_lo]   (one N = 2n MMA over the adjacent
//                                          weight halves) and D[0:n] += x_lo . w
//   else:  D (+)= x . w,  D += x . w_lo,  D += x_lo . w
template <int NACC, bool WIDE>
__device__ __forceinline__ void mma_role(const EngineParams& p, const Bars& bars, uint32_t sbase,
                                         uint32_t tmem_base, uint32_t a_col0, int dcols,
                                         int a_first, int a_stride, volatile int* abortf,
                                         unsigned long long tmo, int lane) {
  const uint32_t idesc_n = idesc_tf32(128, (uint32_t)p.n_tile);
  const uint32_t idesc_2n = idesc_tf32(128, (uint32_t)(2 * p.n_tile));
  const uint64_t bdesc0 = smem_desc_noswz(sbase + p.sm_b, 128, 256);
  const uint64_t lo_step = (uint64_t)(p.n_tile * 32) >> 4;     // w_lo follows w in a K-step
  const uint64_t stage_step = (uint64_t)p.b_stage_bytes >> 4;  // one streamed stage
  const uint64_t kstep_step = (uint64_t)(64 * p.n_tile) >> 4;  // one K-step of weights
  const uint32_t acc_cols = (uint32_t)p.acc_cols;
  const uint32_t kstep_cols = 16u * (uint32_t)p.n_acc;  // A columns of one K-step
  bool ok = true;
  if (p.b_resident) {
    ok = __all_sync(0xffffffffu, mbar_wait(bars.b_full(0), 0, tmo, abortf));
    if (!ok && lane == 0) raise_abort(p, abortf);
  }
  int bstage = 0, as = 0, dslot = 0;
  uint32_t bphase = 0, aphase = 0, dphase = 0;
  for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
    for (int cb = 0; cb < p.n_colblocks && ok; ++cb) {
      ok = __all_sync(0xffffffffu, mbar_wait(bars.d_empty(dslot), dphase ^ 1, tmo, abortf));
      if (!ok) {
        if (lane == 0) raise_abort(p, abortf);
        break;
      }
      tc_fence_after();
      const uint32_t d_base = tmem_base + (uint32_t)(dslot * dcols);
      uint32_t accumulate = 0;
      int kres = 0;  // K-step index within the resident weight block
      for (int c = 0; c < p.n_chunks && ok; ++c) {
        for (int j0 = 0; j0 < p.ksteps_chunk; j0 += p.ks_stage) {
          ok = __all_sync(0xffffffffu, mbar_wait(bars.a_full(as), aphase, tmo, abortf));
          if (!ok) {
            if (lane == 0) raise_abort(p, abortf);
            break;
          }
          tc_fence_after();
          const uint32_t a_stage = tmem_base + a_col0 + (uint32_t)as * kstep_cols * p.ks_stage;
          uint64_t bstage_desc;
          if (p.b_resident) {
            bstage_desc = bdesc0 + (uint64_t)kres * kstep_step;
          } else {
            ok = __all_sync(0xffffffffu, mbar_wait(bars.b_full(bstage), bphase, tmo, abortf));
            if (!ok) {
              if (lane == 0) raise_abort(p, abortf);
              break;
            }
            bstage_desc = bdesc0 + (uint64_t)bstage * stage_step;
          }
          const int kcount = min(p.ks_stage, p.ksteps_chunk - j0);
          for (int kk = 0; kk < kcount; ++kk) {
            const uint64_t bw = bstage_desc + (uint64_t)kk * kstep_step;
            const uint32_t a_tm = a_stage + (uint32_t)kk * kstep_cols;
#pragma unroll
            for (int i = 0; i < NACC; ++i) {
              const int a = a_first + i * a_stride;
              const uint32_t d_tm = d_base + (uint32_t)a * acc_cols;
              const uint32_t x_tm = a_tm + 16u * (uint32_t)a;
              if (WIDE) {
                mma_tf32_ts_elect(d_tm, x_tm, bw, idesc_2n, accumulate);          // x.[w|w_lo]
                mma_tf32_ts_elect(d_tm, x_tm + 8, bw, idesc_n, 1u);               // x_lo . w
              } else {
                mma_tf32_ts_elect(d_tm, x_tm, bw, idesc_n, accumulate);           // x . w
                mma_tf32_ts_elect(d_tm, x_tm, bw + lo_step, idesc_n, 1u);         // x . w_lo
                mma_tf32_ts_elect(d_tm, x_tm + 8, bw, idesc_n, 1u);               // x_lo . w
              }
            }
            accumulate = 1;
          }
          kres += kcount;
          if (!p.b_resident) {
            mma_commit_elect(bars.b_empty(bstage));
            if (++bstage == p.b_stages) {
              bstage = 0;
              bphase ^= 1;
            }
          }
          mma_commit_elect(bars.a_empty(as));
          if (++as == p.a_stages) {
            as = 0;
            aphase ^= 1;
          }
        }
      }
      if (!ok) break;
      mma_commit_elect(bars.d_full(dslot));
      if (++dslot == p.dbuf) {
        dslot = 0;
        dphase ^= 1;
      }
    }
  }
}

// View mode (plain stride-1 conv, no x halo, x lines filling 128-row
// accumulators): row r of accumulator a is raw-box position a*B1*B2 + r, so
// for tap t the A operand of an octet of channels is the 128 x 8 window at
// position a*B1*B2 + toff[t] of a channels-last copy of the box.  A slot
// holds one octet: x as [2][box volume][4] floats (4-channel groups, each
// position 16 bytes), then x_lo in the same layout.  In the no-swizzle
// K-major layout a core matrix is 8 positions x 4 channels (128 contiguous
// bytes): SBO = 128 B between 8-position groups, LBO = box volume x 16 B
// between the two 4-channel groups.
//
// The MMA issuer of accumulator a: per octet slot, the taps' MMAs
// back-to-back (x.[w|w_lo] and x_lo.w when wide, else 3 per tap), one
// commit per slot.  Weights are resident in K-step order (octet-major,
// tap-minor).
template <bool WIDE>
__device__ __forceinline__ void mma_view_role(const EngineParams& p, const Bars& bars,
                                              uint32_t sbase, const int* ktab, uint32_t tmem_base,
                                              int dcols, int a, volatile int* abortf,
                                              unsigned long long tmo, int lane) {
  const uint32_t idesc_n = idesc_tf32(128, (uint32_t)p.n_tile);
  const uint32_t idesc_2n = idesc_tf32(128, (uint32_t)(2 * p.n_tile));
  const uint64_t bdesc0 = smem_desc_noswz(sbase + p.sm_b, 128, 256);
  const uint64_t lo_step = (uint64_t)(p.n_tile * 32) >> 4;   // w_lo follows w in a K-step
  const uint64_t kstep_step = (uint64_t)(64 * p.n_tile) >> 4;  // one K-step of weights
  const uint32_t bvol = (uint32_t)(p.box[0] * p.box[1] * p.box[2]);
  const uint32_t gstride = bvol * 16u;                  // bytes between 4-channel groups
  const uint32_t lo_off = (uint32_t)p.slot_bytes / 2u;  // x_lo follows x in a slot
  const uint32_t row0 = (uint32_t)(a * p.box[1] * p.box[2]) * 16u;
  const int noct = p.cin_chunk / 8;
  bool ok = __all_sync(0xffffffffu, mbar_wait(bars.b_full(0), 0, tmo, abortf));
  if (!ok && lane == 0) raise_abort(p, abortf);
  int slot = 0, dslot = 0;
  uint32_t sphase = 0, dphase = 0;
  for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
    for (int cb = 0; cb < p.n_colblocks && ok; ++cb) {
      ok = __all_sync(0xffffffffu, mbar_wait(bars.d_empty(dslot), dphase ^ 1, tmo, abortf));
      if (!ok) {
        if (lane == 0) raise_abort(p, abortf);
        break;
      }
      tc_fence_after();
      const uint32_t d_tm = tmem_base + (uint32_t)(dslot * dcols + a * p.acc_cols);
      uint32_t accumulate = 0;
      int kres = 0;  // K-step index within the resident weights
      for (int c = 0; c < p.n_chunks && ok; ++c) {
        for (int o = 0; o < noct; ++o) {
          ok = __all_sync(0xffffffffu, mbar_wait(bars.a_full(slot), sphase, tmo, abortf));
          if (!ok) {
            if (lane == 0) raise_abort(p, abortf);
            break;
          }
          tc_fence_after();
          const uint32_t xaddr = sbase + p.sm_xs + (uint32_t)slot * (uint32_t)p.slot_bytes + row0;
          for (int t = 0; t < p.nUtot; ++t, ++kres) {
            const uint32_t aaddr = xaddr + (uint32_t)ktab[t] * 16u;
            const uint64_t ahi = smem_desc_noswz(aaddr, gstride, 128);
            const uint64_t alo = smem_desc_noswz(aaddr + lo_off, gstride, 128);
            const uint64_t bw = bdesc0 + (uint64_t)kres * kstep_step;
            if (WIDE) {
              mma_tf32_ss_elect(d_tm, ahi, bw, idesc_2n, accumulate);  // x.[w|w_lo]
              mma_tf32_ss_elect(d_tm, alo, bw, idesc_n, 1u);           // x_lo . w
            } else {
              mma_tf32_ss_elect(d_tm, ahi, bw, idesc_n, accumulate);   // x . w
              mma_tf32_ss_elect(d_tm, ahi, bw + lo_step, idesc_n, 1u); // x . w_lo
              mma_tf32_ss_elect(d_tm, alo, bw, idesc_n, 1u);           // x_lo . w
            }
            accumulate = 1;
          }
          mma_commit_elect(bars.a_empty(slot));
          if (++slot == p.nslots) {
            slot = 0;
            sphase ^= 1;
          }
        }
      }
      if (!ok) break;
      mma_commit_elect(bars.d_full(dslot));
      if (++dslot == p.dbuf) {
        dslot = 0;
        dphase ^= 1;
      }
    }
  }
}

// View-mode conversion: per raw stage (a channel chunk in TMA's [c][position]
// layout) and per channel octet, write the slot's channels-last x and x_lo.
// Thread i takes positions i, i + 256, ...; a lane reads 4 channels of its
// position and stores them as one 16-byte vector, so both sides are
// conflict-free.  Channels past the chunk's valid ones are written as 0.
__device__ __forceinline__ void view_conversion_role(const EngineParams& p, const Bars& bars,
                                                     uint8_t* gbase, int cw, int lane,
                                                     volatile int* abortf,
                                                     unsigned long long tmo) {
  const int bvol = p.box[0] * p.box[1] * p.box[2];
  const int noct = p.cin_chunk / 8;
  const int tid = cw * 32 + lane;
  int rstage = 0, slot = 0;
  uint32_t rphase = 0, sphase = 0;
  bool ok = true;
  for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
    for (int cb = 0; cb < p.n_colblocks && ok; ++cb) {
      for (int c = 0; c < p.n_chunks && ok; ++c) {
        ok = __all_sync(0xffffffffu, mbar_wait(bars.raw_full(rstage), rphase, tmo, abortf));
        if (!ok) {
          if (lane == 0) raise_abort(p, abortf);
          break;
        }
        const float* raw =
            reinterpret_cast<const float*>(gbase + p.sm_raw + rstage * p.raw_stage_bytes);
        const int cin_valid = min(p.cin_chunk, p.cin_g - c * p.cin_chunk);
        for (int o = 0; o < noct; ++o) {
          ok = __all_sync(0xffffffffu, mbar_wait(bars.a_empty(slot), sphase ^ 1, tmo, abortf));
          if (!ok) {
            if (lane == 0) raise_abort(p, abortf);
            break;
          }
          float4* xs = reinterpret_cast<float4*>(gbase + p.sm_xs + slot * p.slot_bytes);
          float4* xl = xs + 2 * bvol;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const int c0 = 8 * o + 4 * g;
            for (int pos = tid; pos < bvol; pos += 8 * 32) {
              float v[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                v[i] = c0 + i < cin_valid ? raw[(size_t)(c0 + i) * bvol + pos] : 0.f;
              float lo[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                lo[i] = v[i] - __uint_as_float(__float_as_uint(v[i]) & 0xFFFFE000u);
              xs[g * bvol + pos] = make_float4(v[0], v[1], v[2], v[3]);
              xl[g * bvol + pos] = make_float4(lo[0], lo[1], lo[2], lo[3]);
            }
          }
          // the tensor core reads the slot through the async proxy
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.a_full(slot));
          if (++slot == p.nslots) {
            slot = 0;
            sphase ^= 1;
          }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(bars.raw_empty(rstage));
        if (++rstage == p.raw_stages) {
          rstage = 0;
          rphase ^= 1;
        }
      }
    }
  }
}

// The bias fill inside the engine.  The epilogue warps of all CTAs take the
// fill's (slice, plane) units one at a time from a shared counter.  During
// the tile loop a warp does a paced quota, its even share of the units
// spread over the CTA's tile iterations (a burst of fill stores at the start
// would hold up the engine's own loads and evict its input from L2); after
// its last tile it takes units until none are left, so CTAs that finish
// their tiles early do more of the fill.
struct EngineFill {
  const FillParams* f;
  long long units, share, done;
  bool left;  // units may remain

  __device__ __forceinline__ void init(const EngineParams& p, int nparts) {
    f = &p.fill;
    units = p.fill_on ? (long long)f->NC * f->O[0] : 0;
    share = units / ((long long)gridDim.x * nparts);
    done = 0;
    left = units > 0;
  }
  // take a unit and fill it (whole warp); false when none was left
  __device__ __forceinline__ bool step(int lane) {
    unsigned long long idx = 0;
    if (lane == 0) idx = atomicAdd(f->ctr, 1ull);
    idx = __shfl_sync(0xffffffffu, idx, 0);
    if (idx >= (unsigned long long)units) {
      left = false;
      return false;
    }
    const int nc = (int)(idx / (unsigned long long)f->O[0]);
    const int z = (int)(idx - (unsigned long long)nc * f->O[0]);
    const float b = f->bias ? __ldg(f->bias + nc % f->Cout) : 0.f;
    fill_plane(*f, nc, z, b, lane);
    ++done;
    return true;
  }
  // the quota up to fraction k / n of the share
  __device__ __forceinline__ void upto(long long k, long long n, int lane,
                                       const volatile int* abortf) {
    const long long target = share * k / n;
    while (left && done < target && !*abortf) step(lane);
  }
  // every unit still left
  __device__ __forceinline__ void drain(int lane, const volatile int* abortf) {
    while (left && !*abortf) step(lane);
  }
};

}  // namespace

// CL: the channels-last mode (store epilogue only), a template parameter so
// that the NCDHW kernels compile without its branches
template <int EPI, bool VIEW, bool CL>
__global__ void __launch_bounds__(WarpCfg<EPI>::kThreads, 1)
    engine_kernel(const __grid_constant__ EngineParams p) {
  constexpr int kWarpConv0 = WarpCfg<EPI>::kConv0;
  constexpr int kThreads = WarpCfg<EPI>::kThreads;
  extern __shared__ uint8_t smem_dyn[];
  const uint32_t s_unaligned = smem_u32(smem_dyn);
  const uint32_t sbase = (s_unaligned + 1023u) & ~1023u;
  uint8_t* gbase = smem_dyn + (sbase - s_unaligned);
  const Bars bars{sbase + p.sm_bar};
  volatile int* abortf = reinterpret_cast<volatile int*>(gbase + p.sm_bar + kBarAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + p.sm_bar + kBarTmemSlot);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long tmo = p.timeout_cycles;

  // ---------------- set-up ----------------
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxRawStages; ++i) {
      mbar_init(bars.raw_full(i), 1);
      mbar_init(bars.raw_empty(i), kNumConvWarps);
    }
    // stages and accumulator buffers are released by a commit of every issuer
    const uint32_t issuers = p.n_acc >= 2 ? 2u : 1u;
    for (int i = 0; i < kMaxBStages; ++i) {
      mbar_init(bars.b_full(i), 1);
      mbar_init(bars.b_empty(i), issuers);
    }
    // both conversion groups fill every A-stage (alternate K-steps of it)
    for (int i = 0; i < kMaxAStages; ++i) {
      mbar_init(bars.a_full(i), kNumConvWarps);
      mbar_init(bars.a_empty(i), issuers);
    }
    // BatchNorm pooling: both epilogue groups work on every tile
    const uint32_t epi_arrivals = EPI == EPI_BN_POOL ? 2 * kEpiGroup : kEpiGroup;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.d_full(i), issuers);
      mbar_init(bars.d_empty(i), epi_arrivals);
      mbar_init(bars.epi(i), epi_arrivals);
    }
    *abortf = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(sbase + p.sm_bar + kBarTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpRaw && lane == 0 && p.use_tma) prefetch_tensormap(&p.xmap);
  if constexpr (VIEW) {
    // per tap: raw-box position offset of the tap's window.  A box's x start
    // is rounded down to 16 bytes; tile x origins are multiples of 4, so the
    // shift it leaves is the same for every tile.
    int* ktab = reinterpret_cast<int*>(gbase + p.sm_ktab);
    const int xshift = p.u_min[2] - (p.u_min[2] & ~3);
    for (int t = threadIdx.x; t < p.nUtot; t += kThreads) {
      const int t0 = t / (p.nU[1] * p.nU[2]), t1 = (t / p.nU[2]) % p.nU[1], t2 = t % p.nU[2];
      ktab[t] = (p.u_rel[0][t0] * p.box[1] + p.u_rel[1][t1]) * p.box[2] + p.u_rel[2][t2] + xshift;
    }
  } else if (CL) {
    // channels-last: per K-step j of a chunk (tap j / (cin_chunk / 8), its
    // channels 8 (j % (cin_chunk / 8)) .. + 7), the float offset of its first
    // value from a row's own position in the raw box
    int* ktab = reinterpret_cast<int*>(gbase + p.sm_ktab);
    const int per_tap = p.cin_chunk / 8;
    for (int j = threadIdx.x; j < p.ksteps_chunk; j += kThreads) {
      const int t = j / per_tap, c8 = j - t * per_tap;
      const int t0 = t / (p.nU[1] * p.nU[2]), t1 = (t / p.nU[2]) % p.nU[1], t2 = t % p.nU[2];
      ktab[j] = ((p.u_rel[0][t0] * p.box[1] + p.u_rel[1][t1]) * p.box[2] + p.u_rel[2][t2]) *
                    p.cl_cb +
                8 * c8;
    }
  } else {
    // GEMM-K table of one channel chunk: raw-box offset of (channel, tap) pair k
    int* ktab = reinterpret_cast<int*>(gbase + p.sm_ktab);
    const int bvol = p.box[0] * p.box[1] * p.box[2];
    for (int k = threadIdx.x; k < p.ksteps_chunk * 8; k += kThreads) {
      int off = 0;
      if (k < p.k_chunk) {
        const int c = k / p.nUtot, t = k % p.nUtot;
        const int t0 = t / (p.nU[1] * p.nU[2]), t1 = (t / p.nU[2]) % p.nU[1], t2 = t % p.nU[2];
        off = c * bvol + (p.u_rel[0][t0] * p.box[1] + p.u_rel[1][t1]) * p.box[2] + p.u_rel[2][t2];
      }
      ktab[k] = off;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the set-up above touches no global memory; everything below may read
  // what the previous kernel of the stream (the weight pre-pack) wrote
  grid_dependency_wait();
  const int dcols = p.n_acc * p.acc_cols;  // columns of one D buffer
  const uint32_t a_col0 = (uint32_t)(p.dbuf * dcols);

  // ================= raw-input producer =================
  if (warp == kWarpRaw) {
    const int bvol = p.box[0] * p.box[1] * p.box[2];
    int rs = 0;        // raw ring stage
    uint32_t rph = 0;  // and its phase
    for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x) {
      if (*abortf) break;
      const TileCoord tc = decode_tile(p, tile);
      const int zc = p.s_in[0] * tc.o[0] + p.u_min[0];
      const int yc = p.s_in[1] * tc.o[1] + p.u_min[1];
      // the x start is rounded down to 16 bytes where x is the innermost axis
      const int xc = (p.s_in[2] * tc.o[2] + p.u_min[2]) & (CL ? ~0 : ~3);
      bool ok = true;
      // column block cb belongs to group g (nb_per_group blocks per group)
      for (int cb = 0, g = 0, nb = 0; cb < p.n_colblocks && ok;
           ++cb, nb = (nb + 1 == p.nb_per_group) ? 0 : nb + 1, g += (nb == 0)) {
        for (int c = 0; c < p.n_chunks; ++c) {
          const int stage = rs;
          const uint32_t par = rph ^ 1;
          if (++rs == p.raw_stages) {
            rs = 0;
            rph ^= 1;
          }
          ok = mbar_wait(bars.raw_empty(stage), par, tmo, abortf);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            if (lane == 0) raise_abort(p, abortf);
            break;
          }
          const int ch0 = g * p.cin_g + c * p.cin_chunk;
          const uint32_t dst = sbase + p.sm_raw + stage * p.raw_stage_bytes;
          if (p.use_tma) {
            if (lane == 0) {
              if (CL) {
                mbar_arrive_expect_tx(bars.raw_full(stage), (uint32_t)(p.cl_cb * bvol * 4));
                tma_load_5d(dst, &p.xmap, ch0, xc, yc, zc, tc.n, bars.raw_full(stage));
              } else {
                mbar_arrive_expect_tx(bars.raw_full(stage), (uint32_t)(p.cin_chunk * bvol * 4));
                tma_load_5d(dst, &p.xmap, xc, yc, zc, ch0, tc.n, bars.raw_full(stage));
              }
            }
          } else if (CL) {
            // channels-last box without TMA: element e is channel e % cl_cb
            // of position e / cl_cb, copied by lane e % 32 (zero outside x)
            const uint32_t dst0 = sbase + p.sm_raw + stage * p.raw_stage_bytes;
            const int total = p.cl_cb * bvol;
            for (int e = lane; e < total; e += 32) {
              const int cl = e % p.cl_cb, pos = e / p.cl_cb;
              const int i2 = pos % p.box[2], i1 = (pos / p.box[2]) % p.box[1];
              const int i0 = pos / (p.box[2] * p.box[1]);
              const int gx = xc + i2, gy = yc + i1, gz = zc + i0, ch = ch0 + cl;
              const bool in = ch < p.C && gx >= 0 && gx < p.S[2] && gy >= 0 && gy < p.S[1] &&
                              gz >= 0 && gz < p.S[0];
              const float* src =
                  in ? p.x + ((((long long)tc.n * p.S[0] + gz) * p.S[1] + gy) * p.S[2] + gx) * p.C + ch
                     : p.x;
              cp_async4_zfill(dst0 + 4u * (uint32_t)e, src, in);
            }
            cp_async_wait_all();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.raw_full(stage));
          } else {
            // Element e of the box (channel-major, x fastest) is copied by
            // lane e % 32 with a 4-byte cp.async (zero-filled outside the
            // input), so the copies of the whole box are in flight together.
            // A lane's box coordinates (cl, i0, i1, i2) advance by 32
            // elements at a time with carries, without divisions.
            const uint32_t dst0 = sbase + p.sm_raw + stage * p.raw_stage_bytes;
            const int total = p.cin_chunk * bvol;
            const long long s12 = (long long)p.S[1] * p.S[2];
            int i2 = lane % p.box[2], r = lane / p.box[2];
            int i1 = r % p.box[1], i0 = (r / p.box[1]) % p.box[0];
            int cl = r / (p.box[1] * p.box[0]);
            for (int e = lane; e < total; e += 32) {
              const int gx = xc + i2, gy = yc + i1, gz = zc + i0, ch = ch0 + cl;
              const bool in = ch < p.C && gx >= 0 && gx < p.S[2] && gy >= 0 && gy < p.S[1] &&
                              gz >= 0 && gz < p.S[0];
              const float* src = in ? p.x + (((long long)tc.n * p.C + ch) * p.S[0] + gz) * s12 +
                                          (long long)gy * p.S[2] + gx
                                    : p.x;
              cp_async4_zfill(dst0 + 4u * (uint32_t)e, src, in);
              i2 += 32;
              while (i2 >= p.box[2]) {
                i2 -= p.box[2];
                if (++i1 == p.box[1]) {
                  i1 = 0;
                  if (++i0 == p.box[0]) {
                    i0 = 0;
                    ++cl;
                  }
                }
              }
            }
            cp_async_wait_all();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.raw_full(stage));
          }
        }
      }
      if (!ok) break;
    }
  }
  // ================= weight producer =================
  else if (warp == kWarpB) {
    if (lane == 0) {
      if (p.b_resident) {
        mbar_arrive_expect_tx(bars.b_full(0), p.b_stages * p.b_stage_bytes);
        for (int s = 0; s < p.b_stages; ++s)
          bulk_g2s(sbase + p.sm_b + s * p.b_stage_bytes,
                   p.wpack + (size_t)s * (p.b_stage_bytes / 4), p.b_stage_bytes, bars.b_full(0));
      } else {
        int stage = 0;       // weight ring stage
        uint32_t bph = 0;    // and its phase
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
          for (int cb = 0; cb < p.n_colblocks && ok; ++cb)
            for (int c = 0; c < p.n_chunks && ok; ++c)
              for (int j = 0; j < p.ksteps_chunk;
                   j += p.ks_stage, stage = (stage + 1 == p.b_stages) ? 0 : stage + 1,
                       bph ^= (stage == 0)) {
                const uint32_t bytes =
                    (uint32_t)(min(p.ks_stage, p.ksteps_chunk - j) * 64 * p.n_tile);
                if (!mbar_wait(bars.b_empty(stage), bph ^ 1, tmo, abortf)) {
                  raise_abort(p, abortf);
                  ok = false;
                  break;
                }
                mbar_arrive_expect_tx(bars.b_full(stage), bytes);
                const size_t src =
                    (((size_t)cb * p.n_chunks + c) * p.ksteps_chunk + j) * (16 * (size_t)p.n_tile);
                bulk_g2s(sbase + p.sm_b + stage * p.b_stage_bytes, p.wpack + src, bytes,
                         bars.b_full(stage));
              }
        }
      }
    }
  }
  // ================= MMA issuer =================
  else if (VIEW && (warp == kWarpMMA || warp == kWarpMMA1)) {
    // view mode: two accumulators, warp 2 takes accumulator 0, warp 3 takes 1
    const int a = warp - kWarpMMA;
    const int* ktab = reinterpret_cast<const int*>(gbase + p.sm_ktab);
    if (p.wide)
      mma_view_role<true>(p, bars, sbase, ktab, tmem_base, dcols, a, abortf, tmo, lane);
    else
      mma_view_role<false>(p, bars, sbase, ktab, tmem_base, dcols, a, abortf, tmo, lane);
  } else if (warp == kWarpMMA || warp == kWarpMMA1) {
    // with two or more accumulators warp 2 takes the even ones, warp 3 the
    // odd ones; with one, warp 2 takes it and warp 3 has nothing to do
    const int par = warp - kWarpMMA;
    const int stride = p.n_acc >= 2 ? 2 : 1;
    const int mine = (p.n_acc - par + stride - 1) / stride;
    switch (mine * 2 + p.wide) {
      case 0: case 1: break;
#define TC3D_MMA_ROLE(n, w) \
  mma_role<n, w>(p, bars, sbase, tmem_base, a_col0, dcols, par, stride, abortf, tmo, lane)
      case 2: TC3D_MMA_ROLE(1, false); break;
      case 3: TC3D_MMA_ROLE(1, true); break;
      case 4: TC3D_MMA_ROLE(2, false); break;
      default: TC3D_MMA_ROLE(2, true); break;
#undef TC3D_MMA_ROLE
    }
  }
  // ================= conversion warps =================
  // The first and last four conversion warps are two groups; each covers
  // all four TMEM lane quarters.  An A-stage holds ks_stage K-steps of all
  // accumulators (16 columns each: x then x_lo).  Group g fills the K-steps
  // kk with kk % 2 == g of every stage, for all accumulators, so that a warp
  // has the gathers of n_acc rows in flight at once.
  else if (VIEW && warp >= kWarpConv0) {
    view_conversion_role(p, bars, gbase, warp - kWarpConv0, lane, abortf, tmo);
  } else if (warp >= kWarpConv0) {
    const int cw = warp - kWarpConv0;
    const int half = cw >> 2;
    const int q = warp & 3;
    const int* ktab = reinterpret_cast<const int*>(gbase + p.sm_ktab);
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    int rstage = 0, as = 0;
    uint32_t rphase = 0, aphase = 0;
    bool ok = true;
    // raw-box offset of this lane's row of each accumulator, before the
    // tile's x alignment shift
    int row_base[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      int t[3];
      row_local(p, a < p.n_acc ? a : 0, q, lane, t);
      row_base[a] = ((p.s_in[0] * t[0]) * p.box[1] + p.s_in[1] * t[1]) * p.box[2] +
                    p.s_in[2] * t[2];
      if (CL) row_base[a] *= p.cl_cb;  // channels-last: positions of cl_cb floats
    }
    for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
      // only the x origin of the tile matters here (its alignment shift; none
      // in channels-last mode)
      const int b2 = tile - fast_div(p.ntile_div[2], tile) * p.ntile[2];
      const int xs = p.s_in[2] * (b2 * p.T[2]) + p.u_min[2];
      const int xshift = CL ? 0 : xs - (xs & ~3);
      for (int cb = 0; cb < p.n_colblocks && ok; ++cb) {
        for (int c = 0; c < p.n_chunks && ok; ++c) {
          ok = __all_sync(0xffffffffu, mbar_wait(bars.raw_full(rstage), rphase, tmo, abortf));
          if (!ok) {
            if (lane == 0) raise_abort(p, abortf);
            break;
          }
          // raw box of this chunk, moved by the tile's x alignment shift
          const float* raw =
              reinterpret_cast<const float*>(gbase + p.sm_raw + rstage * p.raw_stage_bytes) +
              xshift;
          const int cin_valid = min(p.cin_chunk, p.cin_g - c * p.cin_chunk);
          const int valid_k = cin_valid * p.nUtot;
          for (int j0 = 0; j0 < p.ksteps_chunk; j0 += p.ks_stage) {
            {  // fill this group's K-steps of A-stage as
              ok = __all_sync(0xffffffffu, mbar_wait(bars.a_empty(as), aphase ^ 1, tmo, abortf));
              if (!ok) {
                if (lane == 0) raise_abort(p, abortf);
                break;
              }
              tc_fence_after();
              const uint32_t stage_col =
                  tmem_base + lane_addr + a_col0 + (uint32_t)(as * 16 * p.n_acc * p.ks_stage);
              const int kcount = min(p.ks_stage, p.ksteps_chunk - j0);
              for (int kk = half; kk < kcount; kk += 2) {
                const int j = j0 + kk;
                const uint32_t kcol = stage_col + (uint32_t)(kk * 16 * p.n_acc);
                // the gathers of all accumulators first (independent loads in
                // flight together), then the splits and TMEM stores
                float xg[4][8];
                if (CL) {
                  // channels-last: the K-step's 8 values of a row are 8
                  // consecutive channels of one position, two 16-byte loads
                  // (channels past the valid ones are zero-filled by the load)
                  const int off = ktab[j];
#pragma unroll
                  for (int a = 0; a < 4; ++a) {
                    if (a >= p.n_acc) break;
                    const float4 v0 = *reinterpret_cast<const float4*>(raw + row_base[a] + off);
                    const float4 v1 = *reinterpret_cast<const float4*>(raw + row_base[a] + off + 4);
                    xg[a][0] = v0.x, xg[a][1] = v0.y, xg[a][2] = v0.z, xg[a][3] = v0.w;
                    xg[a][4] = v1.x, xg[a][5] = v1.y, xg[a][6] = v1.z, xg[a][7] = v1.w;
                  }
                } else {
                  const int4 ka = *reinterpret_cast<const int4*>(ktab + j * 8);
                  const int4 kb = *reinterpret_cast<const int4*>(ktab + j * 8 + 4);
                  // GEMM-K entries past the chunk's valid ones (ragged last
                  // chunk, K padding) have zero weights; they read the row's
                  // own first raw element, which is already a term of the
                  // row's sum
                  const int kbase = j * 8;
                  const int kraw[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
                  int kofs[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) kofs[e] = kbase + e < valid_k ? kraw[e] : 0;
#pragma unroll
                  for (int a = 0; a < 4; ++a) {
                    if (a >= p.n_acc) break;
                    const float* rp = raw + row_base[a];
#pragma unroll
                    for (int e = 0; e < 8; ++e) xg[a][e] = rp[kofs[e]];
                  }
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                  if (a >= p.n_acc) break;
                  uint32_t v[16];
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    v[e] = __float_as_uint(xg[a][e]);
                    v[8 + e] = __float_as_uint(xg[a][e] - tf32_trunc(xg[a][e]));
                  }
                  tmem_st16(kcol + (uint32_t)(a * 16), v);
                }
              }
              tmem_wait_st();
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bars.a_full(as));
            }
            if (++as == p.a_stages) {
              as = 0;
              aphase ^= 1;
            }
          }
          __syncwarp();
          if (ok && lane == 0) mbar_arrive(bars.raw_empty(rstage));
          if (++rstage == p.raw_stages) {
            rstage = 0;
            rphase ^= 1;
          }
        }
      }
    }
  }
  // ================= epilogue warps =================
  else {
    const int q = warp & 3;
    const int egroup = (warp - kWarpEpi0) / kEpiGroup;  // 0 or 1
    const uint32_t lo_off = p.wide ? (uint32_t)p.n_tile : 0u;
    const int ew = (warp - kWarpEpi0) % kEpiGroup;       // 0..3 within the group
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    const long long ovol = (long long)p.O[0] * p.O[1] * p.O[2];
    const long long o12 = (long long)p.O[1] * p.O[2];
    int it_d = 0;
    bool ok = true;
    // BatchNorm partial sums (bias-free values) of the 8 channels this
    // lane's group takes.  With one column block they run over every tile
    // and are written once at the end, to the slot of this CTA and lane
    // quarter; with several they are reduced and written per tile.
    float s1[8], s2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s1[i] = 0.f;
      s2[i] = 0.f;
    }
    // running statistics: the affine map is known, no partial sums
    const bool bn_eval = EPI == EPI_BN_POOL && p.bn_affine != nullptr;
    EngineFill fill;
    fill.init(p, WarpCfg<EPI>::kEpiWarps);
    // tile iterations of this CTA (the fill's pace)
    const long long n_it =
        (long long)((p.tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x) *
        p.n_colblocks;
    for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
      const TileCoord tc = decode_tile(p, tile);
      // pool-LSE running state per accumulator (channels this lane holds)
      float lse_m[4], lse_s[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        lse_m[a] = -INFINITY;
        lse_s[a] = 0.f;
      }
      // column block cb is block nb of group g
      for (int cb = 0, g = 0, nb = 0; cb < p.n_colblocks && ok;
           ++cb, ++it_d, nb = (nb + 1 == p.nb_per_group) ? 0 : nb + 1, g += (nb == 0)) {
        // BatchNorm pooling: both groups take every tile (group g the
        // channels 8g..8g+7).  A single group (pool + logsumexp) takes every
        // tile too.  Otherwise, with two accumulator buffers group g takes
        // buffer g; with one, group 0 takes every tile.
        if constexpr (EPI == EPI_STORE) fill.upto(it_d + 1, n_it + 1, lane, abortf);
        constexpr bool kAllTiles =
            EPI == EPI_BN_POOL || WarpCfg<EPI>::kEpiWarps == kEpiGroup;
        if (!kAllTiles && (p.dbuf == 2 ? ((it_d & 1) != egroup) : (egroup != 0))) continue;
        const int oc0 = g * p.cout_g + nb * p.ocb;
        const int ocb_valid = min(p.ocb, p.cout_g - nb * p.ocb);
        const int dslot = p.dbuf == 2 ? (it_d & 1) : 0;
        const uint32_t dpar = (uint32_t)(p.dbuf == 2 ? (it_d >> 1) : it_d) & 1u;
        ok = mbar_wait(bars.d_full(dslot), dpar, tmo, abortf);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          if (lane == 0) raise_abort(p, abortf);
          break;
        }
        tc_fence_after();
        const uint32_t dbase = tmem_base + lane_addr + (uint32_t)(dslot * dcols);

        if constexpr (EPI == EPI_STORE) {
          const int F = p.s_out[0] * p.s_out[1] * p.s_out[2];
          if (CL) {
            // channels-last y: a row's channels are contiguous, so each lane
            // stores its own row's 32 channels of a chunk, as 16-byte vectors
            // where the row's start allows
            for (int cc = 0; cc < p.n_tile; cc += 32) {
              const int oc_lane = cc + lane;
              const float bl =
                  (p.bias && oc_lane < ocb_valid) ? __ldg(p.bias + oc0 + oc_lane) : 0.f;
              const int nvalid = min(32, ocb_valid - cc);
#pragma unroll 1
              for (int a = 0; a < p.n_acc; ++a) {
                uint32_t v[32];
                load_acc32(dbase + (uint32_t)(a * p.acc_cols + cc), lo_off, v);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                  v[jj] = __float_as_uint(__uint_as_float(v[jj]) + __shfl_sync(0xffffffffu, bl, jj));
                int mm[3];
                const bool rv = row_global(p, tc.o, a, q, lane, mm);
                if (!rv) continue;
                float* yr = p.y +
                            ((((long long)tc.n * p.O[0] + mm[0]) * p.O[1] + mm[1]) * p.O[2] + mm[2]) *
                                p.Cout +
                            oc0 + cc;
                if (nvalid == 32 && (reinterpret_cast<uintptr_t>(yr) & 15) == 0) {
#pragma unroll
                  for (int g = 0; g < 8; ++g)
                    reinterpret_cast<float4*>(yr)[g] =
                        make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                    __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3]));
                } else {
#pragma unroll
                  for (int jj = 0; jj < 32; ++jj)
                    if (jj < nvalid) yr[jj] = __uint_as_float(v[jj]);
                }
              }
            }
          } else if (F == 1) {
            // a convolution (or a stride-1 transposed one): one output per
            // row and channel.  Column chunks outer, so that each chunk's
            // bias is loaded once for all accumulators; a full chunk stores
            // its 32 channels without bound checks.
            for (int cc = 0; cc < p.n_tile; cc += 32) {
              const int oc_lane = cc + lane;
              const float bl =
                  (p.bias && oc_lane < ocb_valid) ? __ldg(p.bias + oc0 + oc_lane) : 0.f;
              const bool full = cc + 32 <= ocb_valid;
#pragma unroll 1
              for (int a = 0; a < p.n_acc; ++a) {
                uint32_t v[32];
                load_acc32(dbase + (uint32_t)(a * p.acc_cols + cc), lo_off, v);
                int mm[3];
                const bool rv = row_global(p, tc.o, a, q, lane, mm);
                float* yo = p.y + ((long long)tc.n * p.Cout + oc0 + cc) * ovol +
                            (long long)mm[0] * o12 + (long long)mm[1] * p.O[2] + mm[2];
                if (full) {
#pragma unroll
                  for (int jj = 0; jj < 32; ++jj) {
                    const float b = __shfl_sync(0xffffffffu, bl, jj);
                    if (rv) *yo = __uint_as_float(v[jj]) + b;
                    yo += ovol;
                  }
                } else {
#pragma unroll
                  for (int jj = 0; jj < 32; ++jj) {
                    if (cc + jj >= ocb_valid) break;
                    const float b = __shfl_sync(0xffffffffu, bl, jj);
                    if (rv) *yo = __uint_as_float(v[jj]) + b;
                    yo += ovol;
                  }
                }
              }
            }
          } else if (p.cls_fast && p.s_out[2] == 2) {
            // one class with taps, stride 2 along x: dense stores of the
            // rows of its class pair (r0, r1) (both x classes: the value and
            // the bias) and, with stride 2 along y, of the other y class's
            // row beside it (the bias); the other rows are the bias fill's.
            // The Q2 lanes of a row group hold consecutive m2 with
            // equal (m0, m1), so the group's outputs at x = 2 m2 + r2 form
            // one run of 2 Q2 floats.  The warp's 64 values are written by 2
            // stores of 32 consecutive floats per run: writer lane l of
            // store k takes flattened position i = 32 k + l, i.e. run g =
            // i / (2 Q2) at x offset i % (2 Q2), whose value sits in source
            // lane g Q2 + (i % (2 Q2)) / 2.
            const int star01 = p.cls_star >> 1, star2 = p.cls_star & 1;
            const int rstar = p.cls_r[2 * star01], offstar = p.cls_off[2 * star01];
            // the other y class of the pair's plane: row offset and class
            const bool ybeside = p.s_out[1] == 2;
            const int ry = (rstar >> 8) & 255, roth = 1 - ry;
            const long long offoth = (long long)(roth - ry) * p.O[2];
            int src[2], xodd[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int i = 32 * k + lane;
              const int xl = i & (2 * p.Q[2] - 1);
              src[k] = (i >> (p.lQ[2] + 1)) * p.Q[2] + (xl >> 1);
              xodd[k] = xl & 1;
            }
#pragma unroll 1
            for (int a = 0; a < p.n_acc; ++a) {
              const uint32_t taddr = dbase + (uint32_t)(a * p.acc_cols);
              float* pk[2];
              bool mk[2], mo[2];  // this writer's output of the pair (of the row beside) lies inside
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                int t[3];
                row_local(p, a, q, src[k], t);
                const int m0 = tc.o[0] + t[0], m1 = tc.o[1] + t[1], m2 = tc.o[2] + t[2];
                const bool rv = m0 < p.M[0] && m1 < p.M[1] && m2 < p.M[2];
                const int zb0 = p.s_out[0] * m0, zb1 = p.s_out[1] * m1, xb = 2 * m2 + xodd[k];
                pk[k] = p.y + ((long long)tc.n * p.Cout + oc0) * ovol + (long long)zb0 * o12 +
                        (long long)zb1 * p.O[2] + xb + offstar;
                const bool in = rv && xb < p.O[2] && zb0 + (rstar & 255) < p.O[0];
                mk[k] = in && zb1 + ry < p.O[1];
                mo[k] = ybeside && in && zb1 + roth < p.O[1];
              }
              for (int cc = 0; cc < p.n_tile; cc += 32) {
                uint32_t v[32];
                load_acc32(taddr + (uint32_t)cc, lo_off, v);
                const int oc_lane = cc + lane;
                const float bl =
                    (p.bias && oc_lane < ocb_valid) ? __ldg(p.bias + oc0 + oc_lane) : 0.f;
                float* y0 = pk[0] + (long long)cc * ovol;
                float* y1 = pk[1] + (long long)cc * ovol;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                  if (cc + jj >= ocb_valid) break;
                  const float b = __shfl_sync(0xffffffffu, bl, jj);
                  const float val = __uint_as_float(v[jj]) + b;
                  const float v0 = __shfl_sync(0xffffffffu, val, src[0]);
                  const float v1 = __shfl_sync(0xffffffffu, val, src[1]);
                  if (mk[0]) *y0 = xodd[0] == star2 ? v0 : b;
                  if (mk[1]) *y1 = xodd[1] == star2 ? v1 : b;
                  if (mo[0]) y0[offoth] = b;
                  if (mo[1]) y1[offoth] = b;
                  y0 += ovol;
                  y1 += ovol;
                }
              }
            }
          } else if (p.cls_fast) {
            // one class with taps (cls_star), the others hold the bias.
            // Class f = (r0, r1, r2) of the s_out grid sits at offset
            // cls_off[f] from the row's first output (tables from the host).
#pragma unroll 1
            for (int a = 0; a < p.n_acc; ++a) {
              const uint32_t taddr = dbase + (uint32_t)(a * p.acc_cols);
              int mm[3];
              const bool rv = row_global(p, tc.o, a, q, lane, mm);
              const int zb0 = p.s_out[0] * mm[0], zb1 = p.s_out[1] * mm[1],
                        zb2 = p.s_out[2] * mm[2];
              uint32_t mask = 0;
#pragma unroll
              for (int f = 0; f < 8; ++f) {
                const int r = p.cls_r[f];
                if (rv && f < F && zb0 + (r & 255) < p.O[0] && zb1 + ((r >> 8) & 255) < p.O[1] &&
                    zb2 + (r >> 16) < p.O[2])
                  mask |= 1u << f;
              }
              float* yrow = p.y + ((long long)tc.n * p.Cout + oc0) * ovol + (long long)zb0 * o12 +
                            (long long)zb1 * p.O[2] + zb2;
              for (int cc = 0; cc < p.n_tile; cc += 32) {
                uint32_t v[32];
                load_acc32(taddr + (uint32_t)cc, lo_off, v);
                const int oc_lane = cc + lane;
                const float bl =
                    (p.bias && oc_lane < ocb_valid) ? __ldg(p.bias + oc0 + oc_lane) : 0.f;
                float* yo = yrow + (long long)cc * ovol;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                  if (cc + jj >= ocb_valid) break;
                  const float b = __shfl_sync(0xffffffffu, bl, jj);
                  const float val = __uint_as_float(v[jj]) + b;
#pragma unroll
                  for (int f = 0; f < 8; ++f)
                    if ((mask >> f) & 1u) yo[p.cls_off[f]] = (f == p.cls_star) ? val : b;
                  yo += ovol;
                }
              }
            }
          } else {
            // general path: several classes with taps (oc-major columns)
#pragma unroll 1
            for (int a = 0; a < p.n_acc; ++a) {
              const uint32_t taddr = dbase + (uint32_t)(a * p.acc_cols);
              int mm[3];
              const bool rv = row_global(p, tc.o, a, q, lane, mm);
              const int zb0 = p.s_out[0] * mm[0], zb1 = p.s_out[1] * mm[1],
                        zb2 = p.s_out[2] * mm[2];
              const long long ybase = (long long)tc.n * p.Cout * ovol + (long long)zb0 * o12 +
                                      (long long)zb1 * p.O[2] + zb2;
              for (int cc = 0; cc < p.n_tile; cc += 16) {
                uint32_t v[16];
                load_acc16(taddr + (uint32_t)cc, lo_off, v);
                if (!rv) continue;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                  const int col = cc + jj;
                  const int oc_l = col / p.nR, ri = col - oc_l * p.nR;
                  if (oc_l < ocb_valid) {
                    const int oc = oc0 + oc_l;
                    const int ri2 = ri % p.nRaxis[2];
                    const int ri1 = (ri / p.nRaxis[2]) % p.nRaxis[1];
                    const int ri0 = ri / (p.nRaxis[1] * p.nRaxis[2]);
                    const int r0 = p.r_axis[0][ri0], r1 = p.r_axis[1][ri1], r2 = p.r_axis[2][ri2];
                    if (zb0 + r0 < p.O[0] && zb1 + r1 < p.O[1] && zb2 + r2 < p.O[2]) {
                      const float b = p.bias ? __ldg(p.bias + oc) : 0.f;
                      p.y[ybase + (long long)oc * ovol + (long long)r0 * o12 +
                          (long long)r1 * p.O[2] + r2] = __uint_as_float(v[jj]) + b;
                    }
                  }
                }
                if (p.nEmpty > 0) {
                  // classes without a tap hold the bias; each channel is written
                  // by the chunk holding its last column
                  for (int oc_l = cc / p.nR; oc_l * p.nR <= cc + 15; ++oc_l) {
                    const int last = oc_l * p.nR + p.nR - 1;
                    if (last < cc || last > cc + 15 || oc_l >= ocb_valid) continue;
                    const int oc = oc0 + oc_l;
                    const float b = p.bias ? __ldg(p.bias + oc) : 0.f;
                    for (int r0 = 0; r0 < p.s_out[0]; ++r0)
                      for (int r1 = 0; r1 < p.s_out[1]; ++r1)
                        for (int r2 = 0; r2 < p.s_out[2]; ++r2) {
                          if (((p.cls_mask[0] >> r0) & 1) && ((p.cls_mask[1] >> r1) & 1) &&
                              ((p.cls_mask[2] >> r2) & 1))
                            continue;
                          if (zb0 + r0 < p.O[0] && zb1 + r1 < p.O[1] && zb2 + r2 < p.O[2])
                            p.y[ybase + (long long)oc * ovol + (long long)r0 * o12 +
                                (long long)r1 * p.O[2] + r2] = b;
                        }
                  }
                }
              }
            }
          }
        } else if constexpr (EPI == EPI_POOL_LSE) {
          // rows of a quarter are a 2x2x8 block of positions: lanes
          // {l, l^1, l^8, l^16} form one MaxPool3d(2) window
          const int bsel = 8 * (lane & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 4) & 1);
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            if (a >= p.n_acc) break;
            const uint32_t taddr = dbase + (uint32_t)(a * p.acc_cols);
            for (int cc = 0; cc < p.n_tile; cc += 32) {
              uint32_t u[32];
              load_acc32(taddr + (uint32_t)cc, lo_off, u);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int c16 = cc + 16 * hh;
                if (c16 >= p.n_tile) break;
                float v[16], mx[2];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) v[jj] = __uint_as_float(u[16 * hh + jj]);
                reduce_scatter16_window<true>(v, lane, mx);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int oc_l = c16 + bsel + h;
                  if (oc_l < ocb_valid) {
                    const float val = mx[h] + (p.bias ? __ldg(p.bias + oc0 + oc_l) : 0.f);
                    const float nm = fmaxf(lse_m[a], val);
                    lse_s[a] = lse_s[a] * expf(lse_m[a] - nm) + expf(val - nm);
                    lse_m[a] = nm;
                  }
                }
              }
            }
          }
          if (cb == p.n_colblocks - 1) {
#pragma unroll
            for (int a = 0; a < 4; ++a) {
              if (a >= p.n_acc) break;
              float mm = lse_m[a], ss = lse_s[a];
#pragma unroll
              for (int sh = 0; sh < 3; ++sh) {
                const int x = sh == 0 ? 1 : (sh == 1 ? 8 : 16);
                const float om = __shfl_xor_sync(0xffffffffu, mm, x);
                const float os = __shfl_xor_sync(0xffffffffu, ss, x);
                const float nm = fmaxf(mm, om);
                ss = (ss > 0.f ? ss * expf(mm - nm) : 0.f) + (os > 0.f ? os * expf(om - nm) : 0.f);
                mm = nm;
              }
              int mm3[3];
              row_global(p, tc.o, a, q, lane, mm3);
              const int w0 = mm3[0] >> 1, w1 = mm3[1] >> 1, w2 = mm3[2] >> 1;
              if ((lane & 0x19) == 0 && w0 < p.P[0] && w1 < p.P[1] && w2 < p.P[2]) {
                const float l = mm + logf(ss);
                p.y[(((long long)tc.n * p.P[0] + w0) * p.P[1] + w1) * p.P[2] + w2] = fmaxf(l, 0.f);
              }
            }
          }
        } else {  // EPI_BN_POOL: stride-2 transposed conv, 8 classes per row (oc-major columns)
          // group g takes the channels 8g .. 8g+7 of the column block: 64
          // columns, two TMEM loads in flight together
          const int ch0 = 8 * egroup;
          const int nch = min(8, ocb_valid - ch0);
#pragma unroll 1
          for (int a = 0; a < p.n_acc && nch > 0; ++a) {
            const uint32_t taddr = dbase + (uint32_t)(a * p.acc_cols + 8 * ch0);
            int mm[3];
            const bool rv = row_global(p, tc.o, a, q, lane, mm);
            // class weights of this row (see bn_class_sums)
            const float f0 = 2 * mm[0] + 1 < p.O[0] ? 1.f : 0.f;
            const float f1 = 2 * mm[1] + 1 < p.O[1] ? 1.f : 0.f;
            const float f2 = 2 * mm[2] + 1 < p.O[2] ? 1.f : 0.f;
            const float fr = rv ? 1.f : 0.f;
            uint32_t u[64];
            tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
            if (nch > 4) tmem_ld32(taddr + 32u, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
            tmem_wait_ld();
            float ps[8];
            if (bn_eval)
              bn_class_sums<false>(u, nch, f0, f1, f2, fr, ps, s1, s2);
            else
              bn_class_sums<true>(u, nch, f0, f1, f2, fr, ps, s1, s2);
            // pooled sums over the 8 rows of each 4x4x4 window
            const float pw = reduce_scatter8_window_sum(ps, lane);
            const int w0 = mm[0] >> 1, w1 = mm[1] >> 1, w2 = mm[2] >> 1;
            const int oc_l = ch0 + window8_index(lane);
            if (w0 < p.P[0] && w1 < p.P[1] && w2 < p.P[2] && oc_l < ocb_valid) {
              const int oc = oc0 + oc_l;
              float v;
              if (bn_eval) {
                const float2 ab = __ldg(p.bn_affine + oc);
                v = fmaf(pw * (1.0f / 64.0f), ab.x, ab.y);
              } else {
                v = pw * (1.0f / 64.0f) + (p.bias ? __ldg(p.bias + oc) : 0.f);
              }
              p.y[(((long long)tc.n * p.Cout + oc) * p.P[0] + w0) * p.P[1] * p.P[2] +
                  (long long)w1 * p.P[2] + w2] = v;
            }
          }
          if (p.n_colblocks > 1 && !bn_eval) {
            // BatchNorm partial sums of this tile: all lanes, then the 4
            // quarters of both groups
            const float t1 = reduce_scatter8_sum(s1, lane);
            const float t2 = reduce_scatter8_sum(s2, lane);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              s1[i] = 0.f;
              s2[i] = 0.f;
            }
            float2* red = reinterpret_cast<float2*>(gbase + p.sm_misc) + (it_d & 1) * 64;
            if ((lane & 3) == 0) red[ew * 16 + ch0 + scatter8_index(lane)] = make_float2(t1, t2);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.epi(it_d & 1));
            if (warp == kWarpEpi0) {
              ok = mbar_wait(bars.epi(it_d & 1), (it_d >> 1) & 1, tmo, abortf);
              if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                if (lane == 0) raise_abort(p, abortf);
                break;
              }
              if (lane < ocb_valid) {
                float2 acc = red[lane];
#pragma unroll
                for (int w = 1; w < kEpiGroup; ++w) {
                  acc.x += red[w * 16 + lane].x;
                  acc.y += red[w * 16 + lane].y;
                }
                p.partials[(size_t)(oc0 + lane) * p.part_slots + tile] = acc;
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.d_empty(dslot));
      }
    }
    if constexpr (EPI == EPI_STORE) fill.drain(lane, abortf);
    if constexpr (EPI == EPI_BN_POOL) {
      if (ok && p.n_colblocks == 1 && !bn_eval) {
        // slot: CTA-major, then lane quarter; each channel's slots are all
        // written by the 4 warps of the group that takes it
        const float t1 = reduce_scatter8_sum(s1, lane);
        const float t2 = reduce_scatter8_sum(s2, lane);
        const int oc = 8 * egroup + scatter8_index(lane);
        const int slot = blockIdx.x * kBnSlotsPerCta + ew;
        if ((lane & 3) == 0 && oc < p.cout_g)
          p.partials[(size_t)oc * p.part_slots + slot] = make_float2(t1, t2);
      }
    }
  }

  // ---------------- tear-down ----------------
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMMA) tmem_dealloc(tmem_base, kTmemCols);
}

static_assert(WarpCfg<EPI_BN_POOL>::kEpiWarps == 2 * kEpiGroup && kBnSlotsPerCta == kEpiGroup,
              "BatchNorm pooling: two groups of 8 channels, one partial slot per lane quarter");

template __global__ void engine_kernel<EPI_STORE, false, false>(const __grid_constant__ EngineParams p);
template __global__ void engine_kernel<EPI_POOL_LSE, false, false>(const __grid_constant__ EngineParams p);
template __global__ void engine_kernel<EPI_BN_POOL, false, false>(const __grid_constant__ EngineParams p);
template __global__ void engine_kernel<EPI_STORE, true, false>(const __grid_constant__ EngineParams p);
template __global__ void engine_kernel<EPI_STORE, false, true>(const __grid_constant__ EngineParams p);

// ---------------------------------------------------------------------------
// weight pre-pack: W -> [colblock][chunk][kstep][w | w_lo][n_tile x 8] in the
// tensor core's K-major, no-swizzle layout (8-row x 16-byte core matrices;
// the two K-halves of a row group 128 bytes apart, row groups 256 apart).
// ---------------------------------------------------------------------------
__global__ void pack_weights_kernel(const __grid_constant__ PackParams p) {
  // the engine that follows may start its set-up now; it waits for this
  // grid's completion before it reads the packed weights or the counter
  grid_launch_dependents();
  if (p.zero_ctr && blockIdx.x == 0 && threadIdx.x == 0) *p.zero_ctr = 0ull;
  const long long per_step = 2LL * p.n_tile * 8;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < p.total;
       i += (long long)gridDim.x * blockDim.x) {
    long long r = i;
    const int e = (int)(r % 8);
    r /= 8;
    const int nrow = (int)(r % p.n_tile);
    r /= p.n_tile;
    const int hl = (int)(r % 2);
    r /= 2;
    const int j = (int)(r % p.ksteps_chunk);
    r /= p.ksteps_chunk;
    const int c = (int)(r % p.n_chunks);
    const int cb = (int)(r / p.n_chunks);
    const int g = cb / p.nb_per_group, nb = cb % p.nb_per_group;
    float w = 0.f;
    const int oc_l = nrow / p.nR, ri = nrow % p.nR;
    const int k = j * 8 + e;
    // GEMM-K index k of the chunk -> (channel, tap): channel-major, or, in
    // view mode, K-step j = (channel octet, tap) with the 8 channels inside
    const int c_l = p.tap_major     ? k % p.cin_chunk
                    : p.octet_major ? (j / p.nUtot) * 8 + e
                                    : k / p.nUtot;
    const int t = p.tap_major ? k / p.cin_chunk : p.octet_major ? j % p.nUtot : k % p.nUtot;
    const int icl = c * p.cin_chunk + c_l;
    const int ocg = nb * p.ocb + oc_l;  // output channel within the group
    if (oc_l < p.ocb && ocg < p.cout_g && k < p.k_chunk && icl < p.cin_g) {
      const int t0 = t / (p.nU[1] * p.nU[2]), t1 = (t / p.nU[2]) % p.nU[1], t2 = t % p.nU[2];
      const int ri0 = ri / (p.nRaxis[1] * p.nRaxis[2]), ri1 = (ri / p.nRaxis[2]) % p.nRaxis[1],
                ri2 = ri % p.nRaxis[2];
      const int k0 = p.kidx[0][ri0][t0], k1 = p.kidx[1][ri1][t1], k2 = p.kidx[2][ri2][t2];
      if (k0 >= 0 && k1 >= 0 && k2 >= 0) {
        const long long tap = ((long long)k0 * p.k[1] + k1) * p.k[2] + k2;
        const long long kvol = (long long)p.k[0] * p.k[1] * p.k[2];
        long long widx;
        if (!p.transposed)  // [Cout, Cin/G, k]
          widx = ((long long)(g * p.cout_g + ocg) * p.cin_g + icl) * kvol + tap;
        else  // [Cin, Cout/G, k]
          widx = ((long long)(g * p.cin_g + icl) * p.cout_g + ocg) * kvol + tap;
        w = __ldg(p.w + widx);
      }
    }
    const float v = hl == 0 ? w : w - __uint_as_float(__float_as_uint(w) & 0xFFFFE000u);
    const long long blk = i / per_step;  // (cb, c, j) block
    const int off = (nrow / 8) * 64 + (e / 4) * 32 + (nrow % 8) * 4 + (e % 4);
    p.out[blk * per_step + (long long)hl * p.n_tile * 8 + off] = v;
  }
}

// ---------------------------------------------------------------------------
// BatchNorm finalize (second pass of the two-pass grid reduction)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void block_sum2(double& a, double& b) {
  __shared__ double sa[256], sb[256];
  sa[threadIdx.x] = a;
  sb[threadIdx.x] = b;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) {
      sa[threadIdx.x] += sa[threadIdx.x + s];
      sb[threadIdx.x] += sb[threadIdx.x + s];
    }
    __syncthreads();
  }
  a = sa[0];
  b = sb[0];
}

// partials of bias-free values per (channel, tile); mean adds the bias back
__global__ void __launch_bounds__(256) bn_stats_f2_kernel(const float2* part, int nparts,
                                                          const float* bias, const float* gamma,
                                                          const float* beta, double count,
                                                          float eps, int Cout, float2* stat) {
  const int c = blockIdx.x;
  double s1 = 0.0, s2 = 0.0;
  for (int i = threadIdx.x; i < nparts; i += 256) {
    const float2 v = part[(size_t)c * nparts + i];
    s1 += v.x;
    s2 += v.y;
  }
  block_sum2(s1, s2);
  if (threadIdx.x == 0) {
    const double mean_a = s1 / count;
    double var = s2 / count - mean_a * mean_a;
    if (var < 0.0) var = 0.0;
    const double mean = mean_a + (bias ? (double)bias[c] : 0.0);
    const double g = gamma ? (double)gamma[c] : 1.0, be = beta ? (double)beta[c] : 0.0;
    const double scale = g / sqrt(var + (double)eps);
    stat[c] = make_float2((float)scale, (float)(be - mean * scale));
  }
}

// unfused path: per (n, c) slice sums of the full transposed-conv output
__global__ void __launch_bounds__(256) bn_slice_sums_kernel(const float* t, long long slice,
                                                            float2* /*unused*/, double* out2) {
  const float* s = t + (long long)blockIdx.x * slice;
  double a = 0.0, b = 0.0;
  for (long long i = threadIdx.x; i < slice; i += 256) {
    const double v = s[i];
    a += v;
    b += v * v;
  }
  block_sum2(a, b);
  if (threadIdx.x == 0) {
    out2[2 * blockIdx.x] = a;
    out2[2 * blockIdx.x + 1] = b;
  }
}

// part2: [N][Cout] double pairs (slice order n-major)
__global__ void __launch_bounds__(256) bn_stats_d2_kernel(const double* part2, int nparts,
                                                          const float* gamma, const float* beta,
                                                          double count, float eps, int Cout,
                                                          float2* stat) {
  const int c = blockIdx.x;
  double s1 = 0.0, s2 = 0.0;
  for (int n = threadIdx.x; n < nparts; n += 256) {
    s1 += part2[2 * ((size_t)n * Cout + c)];
    s2 += part2[2 * ((size_t)n * Cout + c) + 1];
  }
  block_sum2(s1, s2);
  if (threadIdx.x == 0) {
    const double mean = s1 / count;
    double var = s2 / count - mean * mean;
    if (var < 0.0) var = 0.0;
    const double g = gamma ? (double)gamma[c] : 1.0, be = beta ? (double)beta[c] : 0.0;
    const double scale = g / sqrt(var + (double)eps);
    stat[c] = make_float2((float)scale, (float)(be - mean * scale));
  }
}

__global__ void bn_apply_kernel(float* y, long long n, long long inner, int Cout,
                                const float2* stat) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)((i / inner) % Cout);
    const float2 s = stat[c];
    y[i] = fmaf(y[i], s.x, s.y);
  }
}

// running statistics (evaluation mode): per channel scale and shift
__global__ void bn_eval_affine_kernel(const float* rmean, const float* rvar, const float* gamma,
                                      const float* beta, const float* bias, float eps, int Cout,
                                      float2* stat) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= Cout) return;
  const double g = gamma ? (double)gamma[c] : 1.0, be = beta ? (double)beta[c] : 0.0;
  const double b = bias ? (double)bias[c] : 0.0;
  const double scale = g / sqrt((double)rvar[c] + (double)eps);
  stat[c] = make_float2((float)scale, (float)(be + (b - (double)rmean[c]) * scale));
}

// unfused path: y = scale * mean of the 4x4x4 window + shift
__global__ void bn_pool4_kernel(const float* t, float* y, int N, int Cout, int O0, int O1, int O2,
                                int P0, int P1, int P2, const float2* stat) {
  const long long total = (long long)N * Cout * P0 * P1 * P2;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    long long r = i;
    const int q2 = (int)(r % P2);
    r /= P2;
    const int q1 = (int)(r % P1);
    r /= P1;
    const int q0 = (int)(r % P0);
    r /= P0;
    const int c = (int)(r % Cout);
    const float* s = t + r * (long long)O0 * O1 * O2;
    float acc = 0.f;
    for (int a = 0; a < 4; ++a)
      for (int b = 0; b < 4; ++b)
        for (int e = 0; e < 4; ++e)
          acc += s[((long long)(4 * q0 + a) * O1 + (4 * q1 + b)) * O2 + 4 * q2 + e];
    const float2 st = stat[c];
    y[i] = fmaf(acc * (1.0f / 64.0f), st.x, st.y);
  }
}

__global__ void wait_timeout_kernel(int* err, unsigned long long timeout_cycles) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, timeout_cycles, nullptr)) atomicExch(err, 1);
}

// ---------------------------------------------------------------------------
// host-side launch wrappers
// ---------------------------------------------------------------------------
cudaError_t engine_set_smem(int kid, int bytes) {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  switch (kid) {
    case EPI_STORE: return cudaFuncSetAttribute(engine_kernel<EPI_STORE, false, false>, a, bytes);
    case EPI_POOL_LSE:
      return cudaFuncSetAttribute(engine_kernel<EPI_POOL_LSE, false, false>, a, bytes);
    case EPI_BN_POOL:
      return cudaFuncSetAttribute(engine_kernel<EPI_BN_POOL, false, false>, a, bytes);
    case kEngineCl: return cudaFuncSetAttribute(engine_kernel<EPI_STORE, false, true>, a, bytes);
    default: return cudaFuncSetAttribute(engine_kernel<EPI_STORE, true, false>, a, bytes);
  }
}

// The engine is launched as a dependent of the weight pre-pack before it:
// its launch and set-up overlap the pre-pack's tail.
cudaError_t engine_launch(int kid, const EngineParams& p, unsigned grid, size_t smem,
                          cudaStream_t st) {
  switch (kid) {
    case EPI_STORE:
      return launch_dependent(engine_kernel<EPI_STORE, false, false>, dim3(grid),
                              dim3(WarpCfg<EPI_STORE>::kThreads), smem, st, p);
    case EPI_POOL_LSE:
      return launch_dependent(engine_kernel<EPI_POOL_LSE, false, false>, dim3(grid),
                              dim3(WarpCfg<EPI_POOL_LSE>::kThreads), smem, st, p);
    case EPI_BN_POOL:
      return launch_dependent(engine_kernel<EPI_BN_POOL, false, false>, dim3(grid),
                              dim3(WarpCfg<EPI_BN_POOL>::kThreads), smem, st, p);
    case kEngineCl:
      return launch_dependent(engine_kernel<EPI_STORE, false, true>, dim3(grid),
                              dim3(WarpCfg<EPI_STORE>::kThreads), smem, st, p);
    default:
      return launch_dependent(engine_kernel<EPI_STORE, true, false>, dim3(grid),
                              dim3(WarpCfg<EPI_STORE>::kThreads), smem, st, p);
  }
}

cudaError_t pack_launch(const PackParams& pp, unsigned blocks, cudaStream_t st) {
  pack_weights_kernel<<<blocks, 256, 0, st>>>(pp);
  return cudaGetLastError();
}

cudaError_t bn_stats_f2_launch(const float2* part, int nparts, const float* bias,
                               const float* gamma, const float* beta, double count, float eps,
                               int Cout, float2* stat, cudaStream_t st) {
  bn_stats_f2_kernel<<<Cout, 256, 0, st>>>(part, nparts, bias, gamma, beta, count, eps, Cout,
                                           stat);
  return cudaGetLastError();
}

cudaError_t bn_apply_launch(float* y, long long n, long long inner, int Cout, const float2* stat,
                            unsigned blocks, cudaStream_t st) {
  bn_apply_kernel<<<blocks, 256, 0, st>>>(y, n, inner, Cout, stat);
  return cudaGetLastError();
}

cudaError_t bn_eval_affine_launch(const float* rmean, const float* rvar, const float* gamma,
                                  const float* beta, const float* bias, float eps, int Cout,
                                  float2* stat, cudaStream_t st) {
  bn_eval_affine_kernel<<<(unsigned)((Cout + 127) / 128), 128, 0, st>>>(rmean, rvar, gamma, beta,
                                                                        bias, eps, Cout, stat);
  return cudaGetLastError();
}

cudaError_t bn_pool4_launch(const float* full, float* y, int N, int Cout, const int O[3],
                            const int P[3], const float2* stat, unsigned blocks,
                            cudaStream_t st) {
  bn_pool4_kernel<<<blocks, 256, 0, st>>>(full, y, N, Cout, O[0], O[1], O[2], P[0], P[1], P[2],
                                          stat);
  return cudaGetLastError();
}

cudaError_t bn_unfused_launch(const float* full, float* y, double* part2, int N, int Cout,
                              const int O[3], const int P[3], const float* gamma,
                              const float* beta, float eps, float2* stat, unsigned blocks,
                              cudaStream_t st) {
  const long long slice = (long long)O[0] * O[1] * O[2];
  bn_slice_sums_kernel<<<(unsigned)(N * Cout), 256, 0, st>>>(full, slice, nullptr, part2);
  const double count = (double)N * (double)slice;
  bn_stats_d2_kernel<<<Cout, 256, 0, st>>>(part2, N, gamma, beta, count, eps, Cout, stat);
  bn_pool4_kernel<<<blocks, 256, 0, st>>>(full, y, N, Cout, O[0], O[1], O[2], P[0], P[1], P[2],
                                          stat);
  return cudaGetLastError();
}

cudaError_t wait_timeout_launch(int* err, unsigned long long timeout_cycles, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(err, timeout_cycles);
  return cudaGetLastError();
}

}  // namespace tc3d
