// pool.cuh -- kernels of the algebraic BN-pool path (see PoolPlan in plan.h):
// the patch Gram matrices of the transposed conv's rows, their reduction, and
// the per-channel finalize that folds the BatchNorm affine map and the 1/64
// of the 4x4x4 pool into the pooled convolution's weights and bias.
#pragma once
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

struct PoolFinParams {
  const float* w;  // transposed-conv weights [Cin][Cout][k0][k1][k2]
  const float* bias;
  const float* gamma;
  const float* beta;
  const float* rmean;   // evaluation mode only
  const float* rvar;
  const double* gcls;   // batch statistics: per class combined Gram [ncls][kGramEntries];
                        // nullptr in evaluation mode
  float* w2;            // [Cout][Cin][Ke0][Ke1][Ke2]
  float* b2;            // [Cout]
  float eps;
  double count;         // outputs per channel, N * O0 * O1 * O2
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
cudaError_t pool_finalize_launch(const PoolFinParams& p, cudaStream_t st);

}  // namespace tc3d
