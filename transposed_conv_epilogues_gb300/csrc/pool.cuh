// pool.cuh -- kernels of the algebraic BN-pool path (see PoolPlan in plan.h):
// the patch Gram matrices of the transposed conv's rows, their reduction, and
// the per-channel finalize that folds the BatchNorm affine map and the 1/64
// of the 4x4x4 pool into the pooled convolution's weights and bias.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"

namespace tc3d {

// Gram CTA: 32q threads per 8x8 Gram block, q = max(1, 8 / blocks), so
// 256 threads for up to 8 blocks and 320 for the 10 blocks of a 32-entry patch
constexpr int kGramMaxThreads = 320;
inline int gram_threads(int nblk) { return nblk * 32 * (nblk >= 8 ? 1 : 8 / nblk); }

// Work unit of box b: Tn samples at one m_a0 and a tile of T1 x T2 rows
// (m_a1, m_a2), with (a0, a1, a2) the box's axis order.  Its input is a slab
// of x: for every sample, channel and offset u of axis a0, the plane
// z_a0 = m_a0 + u over the tile's (z_a1, z_a2) range widened by the offsets,
// stored [sample][channel][u index][W1][W2p] (zero outside x).
struct GramParams {
  const float* x;  // [N, C, L0, L1, L2]
  float* part;     // [slot][kGramEntries]: G (32 x 32, row-major, upper 8x8 blocks) then s
  int N, C, L[3];
  int D, V, nU[3], U[3][kMaxAxisTaps];
  int nb, nblk;    // 8-wide blocks of the D x D Gram; blocks (bi <= bj) computed
  int nbox;
  int box_lo[kGramMaxBoxes][3], box_ext[kGramMaxBoxes][3];
  int box_perm[kGramMaxBoxes][3];
  int box_Tn[kGramMaxBoxes];                          // samples per unit
  int box_T1[kGramMaxBoxes], box_T2[kGramMaxBoxes];
  int box_W1[kGramMaxBoxes], box_W2p[kGramMaxBoxes];  // W2p = 4 x odd
  int vec16;  // x 16-byte aligned and L2 % 4 == 0: rows along axis 2 move as 16-byte copies
  int box_nt1[kGramMaxBoxes], box_nt2[kGramMaxBoxes];  // tiles along a1, a2
  long long box_units[kGramMaxBoxes];
  int box_cta0[kGramMaxBoxes + 1];  // CTAs [box_cta0[b], box_cta0[b+1]) take box b
};

// Lag kernel (lag.cu): region sums of x[c, z] and x[c, z] x[c', z + delta]
// per CTA, then summed over the grid.  Tables as in PoolPlan (lag_*).
struct LagParams {
  CUtensorMap xmap;  // x [N, C, L0, L1, L2] as (L2, L1, L0, C, N); box (40, 3, 4, C, 1)
  float* part;       // [grid][nbox][kLagSlots]
  float* rs;         // [nbox][kLagSlots]: box sums over the grid
  int* err;
  unsigned long long timeout_cycles;
  int N, L[3];
  int nseg[3], seg[3][kLagMaxSeg + 1], bulk[3];
  int nrange[3], range[3][4][2], nbox;  // boxes: a segment range per axis
  int nb1, nb2;
  int nc[kLagMaxSeg], cta0[kLagMaxSeg + 1];
  int grid;
};
size_t lag_smem_bytes();
cudaError_t lag_set_smem();
// the lag kernel (cin channels, 1..3)
cudaError_t lag_launch(const LagParams& p, int cin, cudaStream_t st);

// Pooled convolution on CUDA cores (pool.cu): stride 2, at most 3 taps per
// axis, Cin <= 4, Cout <= 64; y = s2 conv(x, w2) + b2 over P0 x P1 x P2
// outputs, input position 2 q + e - pad.  A CTA takes items (n, q0, 4 rows of
// q1, 16 of q2) with one warp per 16 channels; the input boxes and the weights
// come in by TMA.
constexpr int kPooledMaxCin = 4;
constexpr int kPooledMaxCout = 64;
constexpr int kPooledRows = 4;     // q1 outputs per item (per lane)
constexpr int kPooledQ2 = 16;      // q2 outputs per CTA (one per lane pair)
constexpr int kPooledBoxCols = 36; // columns of the input box (33 used + alignment shift)
constexpr int kPooledBoxRows = 2 * kPooledRows + 1;
struct PooledParams {
  CUtensorMap xmap;  // x as (L2, L1, L0, Cin, N); box (36, 9, 3, Cin, 1)
  const float* w2;   // [ci][e0][e1][e2][coutp], 3 taps per axis (zero past Ke)
  const float* b2;   // [Cout] or nullptr
  const float* s2;   // [Cout] scale of the sums (y = s2 * acc + b2), or nullptr (1)
  unsigned* ctr;     // item counter, zero at launch (CTAs take items from it), or nullptr
                     // (CTA b takes items b, b + grid, ...)
  float* y;          // [N][Cout][P0][P1][P2]
  int* err;
  unsigned long long timeout_cycles;
  int N, Cin, Cout, coutp, P[3], pad[3];
  int nq1b, nq2b;    // q1 blocks of 4, q2 blocks of 16
};
// the kernel takes the problem (sizes, taps, channels); x's tensor map is
// encoded by the caller
bool pooled_ok(int Cin, int Cout, const int Ke[3], const int P[3], int N);
inline int pooled_coutp(int Cout) { return (Cout + 15) / 16 * 16; }
size_t pooled_smem_bytes(int Cin, int coutp);
cudaError_t pooled_launch(const PooledParams& p, int sm_count, cudaStream_t st);

struct PoolFinParams {
  const float* w;  // transposed-conv weights [Cin][Cout][k0][k1][k2]
  const float* bias;
  const float* gamma;
  const float* beta;
  const float* rmean;   // evaluation mode only
  const float* rvar;
  const double* gcls;   // batch statistics: per class combined Gram [ncls][kGramEntries];
                        // nullptr in evaluation mode and in lag form
  const float* lrs;     // batch statistics in lag form: box sums [nbox][kLagSlots]
  unsigned wkmask[3][kMaxAxisTaps];  // per axis and summed tap e: bit k set iff W[k] adds in
  // per class c and entry i of its patch (rows off[c] .. off[c + 1] - 1 of
  // all classes): the patch index d, the index of its weight in a channel's
  // [Cin][k0][k1][k2] block, and in lag form its channel and offset indices
  // (ci | v0 << 4 | v1 << 8 | v2 << 12) and its box as a first factor
  int ent_off[9];
  int ent_d[8 * kGramMaxD], ent_w[8 * kGramMaxD], ent_cv[8 * kGramMaxD], ent_box[8 * kGramMaxD];
  int pooled_layout;    // 1: w2 as [ci][e0][e1][e2][w2_stride] with 3 taps per axis
  int w2_stride;        //    (zero past Ke), the pooled-conv kernel's layout
  float* w2;            // [Cout][Cin][Ke0][Ke1][Ke2]
  float* b2;            // [Cout]
  float* s2;            // lag form with the pooled layout: [Cout] scale / 64, which the
                        // pooled conv applies (w2 then holds unscaled sums); else nullptr
  unsigned* pool_ctr;   // the pooled conv's item counter, zeroed here (or nullptr)
  float eps;
  double count;         // outputs per channel, N * O0 * O1 * O2
  double inv_count;     // 1 / count
  int Cin, Cout, k[3], pad[3], dil[3];
  int V, nU[3];
  int ntap[3][2], tap_k[3][2][kMaxAxisTaps], tap_u[3][2][kMaxAxisTaps];
  int ncls, cls_r[8][3];
  int e_min[3], Ke[3];
};

// raise the Gram kernel's dynamic shared-memory limit (once per device)
cudaError_t gram_set_smem();
// grid: total CTAs over the boxes (box_cta0 filled by the caller)
cudaError_t gram_launch(const GramParams& p, unsigned ctas, cudaStream_t st);

// gcls[c][e] = sum over boxes b of cls_coef[c][b] * (sum over box b's CTA
// slots of part[slot][e]), in double
cudaError_t gram_reduce_launch(const float* part, const int* box_cta0_host, int nbox,
                               const int (*cls_coef)[kGramMaxBoxes], int ncls, double* gcls,
                               cudaStream_t st);
// Lag form, after the lag kernel (dependent launches): the reduction of its
// per-CTA box sums part[ctas][nent] into p.lrs (the entries the statistics
// read), then the finalize of every channel, a CTA each: statistics, b2 and
// s2 (or, without s2, the weights w2 with the scale folded in)
cudaError_t lag_finalize_launch(const PoolFinParams& p, const float* part, int ctas, int nent,
                                cudaStream_t st);
// evaluation mode, or batch statistics from the Gram path's class Grams (a
// normal launch: the first kernel of a call, or after the Gram reduction)
cudaError_t pool_finalize_launch(const PoolFinParams& p, cudaStream_t st);

}  // namespace tc3d
