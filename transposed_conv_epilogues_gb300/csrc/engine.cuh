// engine.cuh -- launch parameters shared by the host launcher and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"

namespace tc3d {

// Warp roles of the implicit-GEMM kernel (one CTA per SM):
//   warp 0        TMA (or plain-load) producer of raw input boxes
//   warp 1        bulk-copy producer of packed weight K-steps
//   warp 2        TMEM allocator + MMA issuer of the even accumulators
//   warp 3        MMA issuer of the odd accumulators (idle with one)
//   warps 4..     epilogue: one group of 4 warps (TMEM lane quarter = warp % 4),
//                 or two groups that alternate accumulator buffers when the
//                 epilogue uses two buffers (stores, BatchNorm pooling);
//                 the store epilogue also does the bias fill of the outputs
//                 no tile writes (a transposed conv's tap-less classes)
//   last 8 warps  conversion: raw fp32 -> (x, x - trunc(x)) in TMEM
// (20 warps at most: an SM sub-partition's 16K registers hold 5 warps of 96.)
constexpr int kWarpRaw = 0;
constexpr int kWarpB = 1;
constexpr int kWarpMMA = 2;
constexpr int kWarpMMA1 = 3;
constexpr int kWarpEpi0 = 4;
constexpr int kEpiGroup = 4;  // warps per epilogue group
constexpr int kNumConvWarps = 8;

template <int EPI>
struct WarpCfg {
  static constexpr int kEpiWarps = EPI == EPI_POOL_LSE ? 4 : 8;
  static constexpr int kConv0 = kWarpEpi0 + kEpiWarps;
  static constexpr int kWarps = kConv0 + kNumConvWarps;
  static constexpr int kThreads = kWarps * 32;
};

// Division of an int in [0, 2^31) by a fixed divisor d >= 1 as one 64-bit
// multiply and a shift (division by invariant integers, Granlund and
// Montgomery, PLDI 1994): with l = ceil(log2 d), shift = 32 + l and
// mul = ceil(2^shift / d), (n * mul) >> shift = floor(n / d), because
// mul * d - 2^shift < d and n < 2^31 keep the error term below 1 / (2d).
// mul < 2^33, so the product stays below 2^64.
struct FastDiv {
  unsigned long long mul;
  int shift;
  int d;
};

inline FastDiv make_fastdiv(int d) {
  int l = 0;
  while ((1LL << l) < (long long)d) ++l;
  FastDiv f;
  f.shift = 32 + l;
  f.d = d;
  const unsigned long long num = 1ULL << f.shift;  // shift <= 63 for d < 2^31
  f.mul = num / (unsigned long long)d + (num % (unsigned long long)d ? 1 : 0);
  return f;
}

__host__ __device__ __forceinline__ int fast_div(const FastDiv& f, int n) {
  return (int)(((unsigned long long)(unsigned)n * f.mul) >> f.shift);
}

constexpr int kMaxRawStages = 3;
constexpr int kMaxBStages = 16;
constexpr int kMaxAStages = 16;  // TMEM A-stage ring: one K-step of all accumulators per stage

// Bias fill of a transposed conv: bias (or 0) into the outputs at z_a >=
// zl[a] for any axis a (outputs of rows past the GEMM row grid; all of them
// in classes without taps) and, with s0 > 0, into every output row (z, y)
// with z % s0 != r0 or y % s1 != r1 (rows of tap-less class pairs)
struct FillParams {
  float* y;           // [N * Cout][O0][O1][O2]
  const float* bias;  // [Cout] or nullptr (0)
  int NC, Cout, O[3], zl[3];
  int s0, s1, r0, r1;  // s0 == 0: no row mode
  // inside the engine: the next unit to take, shared by all CTAs (zeroed by
  // the weight pre-pack before the engine starts)
  unsigned long long* ctr;
};

struct EngineParams {
  CUtensorMap xmap;  // 5-D map over x (dims S2, S1, S0, C, N), used when use_tma
  const float* x;
  const float* wpack;
  const float* bias;
  float* y;
  float2* partials;  // BN-pool: [Cout][part_slots] (sum, sum of squares) of bias-free values
  int part_slots;    // one per epilogue warp of the grid (one column block), else one per tile
  int* err;
  unsigned long long timeout_cycles;  // bound of every mbarrier wait (SM clock cycles)
  int use_tma;

  int N, C, Cout, G, cin_g, cout_g;
  int S[3];
  int O[3];
  int P[3];
  int M[3], s_in[3], s_out[3], u_min[3];
  int nU[3], nUtot;
  int u_rel[3][kMaxAxisTaps];
  int nR, nRaxis[3], nEmpty;
  int r_axis[3][kMaxClassesAxis];
  int cls_mask[3];  // per axis: bit r set iff class r has a tap
  // one class with taps and at most 8 classes: output offset of class f =
  // (r0, r1, r2) from its row's first output, the class packed as
  // r0 | r1 << 8 | r2 << 16, and the index of the class with taps
  int cls_fast, cls_off[8], cls_r[8], cls_star;

  int ocb, n_tile, nb_per_group, n_colblocks;
  int n_acc, dbuf, a_stages;  // a_stages: ring depth, 16*n_acc*ks_stage TMEM columns each
  int ks_stage;              // K-steps per A-stage
  int wide, acc_cols;        // fused [w | w_lo] MMA; TMEM columns of one accumulator
  int Q[3], Pq[3], T[3], ntile[3];
  int lQ[3], lPq[3];     // log2 of Q and Pq (powers of two)
  FastDiv ntile_div[3];  // tile index -> tile coordinates
  int tiles;

  int cin_chunk, n_chunks, k_chunk, ksteps_chunk;
  int box[3];
  int raw_stages;
  unsigned raw_stage_bytes;
  int b_resident, b_stages;
  unsigned b_stage_bytes;

  // channels-last mode: x [N][S0][S1][S2][C] and y [N][O0][O1][O2][Cout];
  // the raw box is [position][cl_cb] (cl_cb = cin_chunk + 4 channels)
  int cl, cl_cb;

  // view mode: A read by the tensor core from channels-last octet slots
  int view, nslots;
  unsigned slot_bytes;

  // dynamic shared-memory layout (offsets from the 1024-aligned base)
  unsigned sm_raw, sm_b, sm_xs, sm_ktab, sm_misc, sm_bar;

  // BN-pool with running statistics: per channel (scale, shift), the bias
  // folded into shift; the epilogue then stores final values and no partial
  // sums.  nullptr: batch statistics.
  const float2* bn_affine;

  // store epilogue: the bias fill of the outputs no tile writes, done by the
  // epilogue warps (fill_on = 0: none)
  FillParams fill;
  int fill_on;
};

struct PackParams {
  const float* w;
  float* out;
  int transposed;
  int cin_g, cout_g;
  int k[3];
  int nUtot, nU[3];
  int nR, nRaxis[3];
  int kidx[3][kMaxClassesAxis][kMaxAxisTaps];
  int ocb, n_tile, nb_per_group, n_colblocks;
  int cin_chunk, n_chunks, k_chunk, ksteps_chunk;
  int octet_major;  // 1: K-step j of a chunk is channel octet j / nUtot at tap j % nUtot
  int tap_major;    // 1: GEMM-K index k of a chunk is tap k / cin_chunk, channel k % cin_chunk
  long long total;  // floats in the packed buffer
  unsigned long long* zero_ctr;  // set to 0 when non-null (the engine's bias-fill counter)
};

// host-side launch wrappers (engine.cu; kernels are launched from the
// translation unit that defines them)
// kernel id: the epilogue kind, or kEngineView for the view-mode store
// kernel, kEngineCl for the channels-last one
constexpr int kEngineView = 3;
constexpr int kEngineCl = 4;
cudaError_t engine_set_smem(int kid, int bytes);
cudaError_t engine_launch(int kid, const EngineParams& p, unsigned grid, size_t smem,
                          cudaStream_t st);
cudaError_t pack_launch(const PackParams& pp, unsigned blocks, cudaStream_t st);
cudaError_t bn_stats_f2_launch(const float2* part, int nparts, const float* bias,
                               const float* gamma, const float* beta, double count, float eps,
                               int Cout, float2* stat, cudaStream_t st);
cudaError_t bn_apply_launch(float* y, long long n, long long inner, int Cout, const float2* stat,
                            unsigned blocks, cudaStream_t st);
// running statistics: stat[c] = (scale, shift) with scale = gamma/sqrt(var +
// eps), shift = beta + (bias - mean) * scale (bias may be nullptr)
cudaError_t bn_eval_affine_launch(const float* rmean, const float* rvar, const float* gamma,
                                  const float* beta, const float* bias, float eps, int Cout,
                                  float2* stat, cudaStream_t st);
// unfused pooling: y = mean of each 4x4x4 window of full * scale + shift
cudaError_t bn_pool4_launch(const float* full, float* y, int N, int Cout, const int O[3],
                            const int P[3], const float2* stat, unsigned blocks, cudaStream_t st);
cudaError_t bn_unfused_launch(const float* full, float* y, double* part2, int N, int Cout,
                              const int O[3], const int P[3], const float* gamma,
                              const float* beta, float eps, float2* stat, unsigned blocks,
                              cudaStream_t st);
// the stand-alone fill (grids without engine tiles)
cudaError_t fill_slab_launch(const FillParams& p, cudaStream_t st);
cudaError_t wait_timeout_launch(int* err, unsigned long long timeout_cycles, cudaStream_t st);

// device address of the library's error word on the current device
cudaError_t error_flag_address(int** addr);

}  // namespace tc3d
