// plan.h -- host-side planning for the implicit-GEMM engine (pure integer
// code, no CUDA): output sizes, argument validation, the transposed
// convolution's output-parity classes and tap tables, tile shapes and the
// shared/tensor-memory budget of one launch.
#pragma once
#include <algorithm>
#include <cstddef>
#include <cstdint>

// functions shared by the host planner and the kernels
#if defined(__CUDACC__)
#define TC3D_HD __host__ __device__
#else
#define TC3D_HD
#endif

namespace tc3d {

enum OpKind : int {
  OP_CONV = 0,             // conv3d_fwd
  OP_CONVT = 1,            // conv_transpose3d_fwd
  OP_CONV_POOL_LSE = 2,    // conv_maxpool_lse_relu
  OP_CONVT_BN_POOL = 3,    // convT_bn_avgpool (batch statistics)
  OP_CONVT_BN_EVAL = 4,    // convT_bneval_avgpool (running statistics)
  OP_CONV_NDHWC = 5,       // conv3d_fwd_ndhwc (planned as OP_CONV; x and y channels-last)
};

inline bool is_bn_op(int op) { return op == OP_CONVT_BN_POOL || op == OP_CONVT_BN_EVAL; }

enum EpiKind : int {
  EPI_STORE = 0,     // bias add + store every output (all parity classes)
  EPI_POOL_LSE = 1,  // MaxPool3d(2) + channel logsumexp + ReLU
  EPI_BN_POOL = 2,   // 4x4x4 pooled sums + per-tile BatchNorm partial sums, or,
                     // with the BatchNorm affine known up front, the final values
};

constexpr int kMaxAxisTaps = 16;    // per-axis kernel extent limit
constexpr int kMaxClassesAxis = 8;  // per-axis stride limit of a transposed conv
constexpr int kMaxKChunk = 1024;    // GEMM-K values staged per channel chunk
constexpr int kMaxBStagesPlan = 16; // streamed weight stages (mbarrier pairs in the kernel)
constexpr int kTmemCols = 512;
constexpr int kMaxSmem = 227 * 1024;
constexpr int kMaxGrid = 1024;      // CTAs of a persistent engine launch, at most
constexpr int kBnSlotsPerCta = 4;   // BatchNorm partial slots per CTA (one per lane quarter)

struct Problem {
  int op;
  int N, Cin, S[3], Cout, k[3], stride[3], pad[3], dil[3], out_pad[3], groups;
  // internal convolutions only: output extents below the formula's (0: the
  // formula's own); rows past them are not computed
  int out_ext[3];
  // 1: x and y are channels-last (NDHWC); the plan then takes the engine's
  // channels-last mode where it applies (Plan::cl)
  int cl;
};

// Everything a launch needs, derived from a Problem.  Row space: for every
// batch n a grid M0 x M1 x M2 of "rows"; row m reads input positions
// s_in*m + u (u in the per-axis offset lists) and produces outputs
// s_out*m + r for every parity class r (s_out = 1, one class, for a conv).
struct Plan {
  int status;  // 0 or a negative TC3D_ERR_* code
  Problem pb;
  int transposed;
  int64_t O[3];   // conv / transposed-conv output extents
  int64_t P[3];   // pooled extents (pool-LSE: O/2, BN-pool: O/2/2)
  int64_t y_elems;
  int cin_g, cout_g;
  int epi;        // EpiKind of the main launch
  int fused;      // 0: convT_bn_avgpool runs through the unfused fallback

  // rows and taps
  int M[3], s_in[3], s_out[3];
  int nU[3];                  // union of input offsets per axis
  int u_rel[3][kMaxAxisTaps]; // offset - u_min
  int u_min[3], u_max[3];
  // parity classes (transposed conv): per axis the classes with >= 1 tap
  int nRaxis[3];
  int r_axis[3][kMaxClassesAxis];                    // class value r of index ri
  int kidx[3][kMaxClassesAxis][kMaxAxisTaps];        // kernel tap of (ri, offset t), or -1
  int nR;                                            // non-empty classes (product set)
  int nEmpty;                                        // classes with no tap (bias only)
  // outputs at z_a >= s_out*M (all of them in tap-less classes) are written
  // by a separate bias fill; fill_slab says whether any exist
  int fill_slab;
  // one class with taps whose store takes the dense stride-2-along-x path
  // (cls_fast with s_out[2] == 2): the engine writes only the output rows of
  // that class's (r0, r1) pair (and, with stride 2 along y, the rows of the
  // other y class in the same planes), the bias fill all others (fill_rows;
  // then fill_slab is set too)
  int cls_fast;
  int fill_rows;

  // GEMM N: per column block ocb output channels x nR classes, oc-major
  int ocb, n_tile, nb_per_group, n_colblocks;

  // tiles: a tile is n_acc accumulators of 128 rows; each 32-row quarter is a
  // box Q0 x Q1 x Q2, quarters are arranged P0 x P1 x P2 -> tile T = P*Q
  int n_acc, dbuf, a_stages;
  int wide;         // 1: x.[w|w_lo] as one N = 2 n_tile MMA + x_lo.w (accumulator 2 n_tile wide)
  int acc_cols;     // TMEM columns of one accumulator (n_tile, or 2 n_tile when wide)
  int ks_stage;     // K-steps per A-stage (a stage = ks_stage x n_acc x 16 TMEM columns)
  int Q[3], Pq[3], T[3];
  int ntile[3];
  int xslack;       // max misalignment (elements) of a raw box's x start
  int64_t tiles;

  // channel chunks and raw input box
  int cin_chunk, n_chunks, k_chunk, ksteps_chunk;
  int box[3];        // B0, B1, B2 (B2 multiple of 4)
  int raw_stages;
  int64_t raw_stage_bytes;
  int b_resident;    // 1: whole packed weight block stays in smem
  int b_stages;
  int64_t b_stage_bytes;
  int64_t smem_bytes;

  // view mode: every accumulator's 128 rows are 128 consecutive positions of
  // the raw box, so for each tap the A operand is a shifted window of a
  // channels-last copy of the box, read by the tensor core from shared
  // memory.  The copy is kept in slots of one channel octet each ([x | x_lo],
  // each [2][box volume][4] floats); GEMM-K runs octet-major, tap-minor.
  int view;
  int nslots;
  int64_t slot_bytes;
  // channels-last mode (a conv on NDHWC x and y, groups 1): the raw box is
  // [position][cl_cb] with cl_cb = cin_chunk + 4 channels (cl_cb / 4 odd, so
  // 16-byte loads of consecutive positions hit distinct banks), GEMM-K runs
  // tap-major, channel-minor, and a K-step (8 channels of one tap) is two
  // 16-byte loads per row
  int cl;
  int cl_cb;
  // 1: planned in the merged (S1*S2) form of a (k,k,1) conv (see make_plan);
  // O_user are then the caller's output extents, O the merged ones
  int reshaped;
  int64_t O_user[3];

  // workspace (bytes, each region 256-aligned)
  int64_t ws_wpack_off, ws_wpack_bytes;
  int64_t ws_ctr_off;                   // bias fill: the engine's unit counter (8 bytes)
  int64_t ws_part_off, ws_part_bytes;   // BN partials (batch statistics only): fused
                                        // [Cout][slots] float2, else [N][Cout] double2
  int64_t ws_stat_off, ws_stat_bytes;   // BN scale/shift [Cout] float2
  int64_t ws_full_off, ws_full_bytes;   // unfused fallback: full convT output
  int64_t ws_total;
};

// Shared-memory layout of the main kernel (byte offsets from a 1024-aligned
// base): raw input stages, weight stages, GEMM-K offset table, epilogue
// scratch (4 KB), mbarriers (1 KB).  Returns the dynamic smem request.
struct SmemLayout {
  int64_t raw, b, xs, ktab, misc, bar, total;
};
SmemLayout smem_layout(const Plan& pl);

// Fill *plan for problem pb.  Returns plan->status.
// Engine grid: one persistent CTA per SM, never more CTAs than tiles.
inline int64_t engine_grid(const Plan& pl, int sm_count) {
  return std::min<int64_t>(std::min<int64_t>(pl.tiles, sm_count), kMaxGrid);
}

// Slots of the fused BatchNorm partial sums per channel: with one column
// block every CTA keeps running sums per TMEM lane quarter (one slot each),
// otherwise every tile writes one slot.
inline int64_t bn_part_slots(const Plan& pl, int64_t grid) {
  return pl.n_colblocks == 1 ? grid * kBnSlotsPerCta : pl.tiles;
}

int make_plan(const Problem& pb, Plan* plan);

// ---------------------------------------------------------------------------
// Algebraic path of the BN-pool pipelines (transposed conv with stride 2 on
// every axis, groups 1, few input channels).
//
// Pooled output.  A 4x4x4 window q covers z = 4q + j (j = 0..3) per axis.
// Output z takes tap k from input (z + p - d k)/2, so the window's sum reads
// input 2q + e with e = (j + p - d k)/2: the pooled sums are a stride-2
// convolution of x with summed weights W'[e] = sum of W[k] over the (j, k)
// pairs giving e ("Kimi-K2.6 l2_p72", its observation that one pooled output
// depends on a 3x3x3 input footprint).  With the BatchNorm scale folded in,
// that convolution writes final outputs.
//
// Batch statistics.  Row m of the transposed conv holds output 2m + r of
// every class r; class r reads inputs m + u for its offsets u.  Let P(m) be
// the vector of x over (channel, u0, u1, u2) for the union of offsets, D
// entries.  Then the class sum of t is w_r . s_r and the class sum of t^2 is
// w_r^T G_r w_r, with s_r = sum P(m) and G_r = sum P(m) P(m)^T over the rows
// class r has.  The rows of a class are the box [0, M) less, on axes where the
// class ends one row early, the last plane: G_r follows by inclusion-exclusion
// over at most 8 boxes (the full box and its last planes, edges, corner).
constexpr int kGramMaxD = 32;                                   // patch entries
constexpr int kGramEntries = kGramMaxD * kGramMaxD + kGramMaxD; // G then s
constexpr int kGramMaxCtas = 1024;                              // partial slots
constexpr int kGramMaxBoxes = 8;
constexpr int kGramSlabFloats = 12288;                          // one x slab buffer (48 KB)

// Lag form of the batch statistics.  When x has at most 3 channels and every
// axis has one offset or two consecutive ones, an entry of G_r is
//   sum over the rows m of class r of x[c, m + u] x[c', m + u']
//     = sum over z in [u, M_r + u) (per axis) of x[c, z] x[c', z + delta],
// delta = u' - u in {-1, 0, 1}^3 (x zero outside its extent), and an entry
// of s_r is the same kind of sum of x[c, z].  The ends of those z ranges,
// over all classes and offsets, cut each axis into a few segments: one wide
// one and positions of their own at the ends.  The lag kernel sums every
// product x[c, z] x[c', z + delta] (and every x[c, z]) over every region (a
// product of three segments); an entry of G_r or s_r is the sum of the
// regions its range covers.  Per input position that is 126 products for 3
// channels, against the D (D + 1) / 2 = 300 of the 24-entry patch Gram.
constexpr int kLagMaxCin = 3;
constexpr int kLagSlots = 128;    // per region: Cin first-order sums, then the products
constexpr int kLagMaxSeg = 5;     // segments per axis
constexpr int kLagRows = 8;       // axis-1 rows of a CTA (one per warp)
constexpr int kLagCols = 32;      // axis-2 columns of a CTA (one per lane)
constexpr int kLagChunk = 4;      // planes per tensor copy of a warp's window rows
constexpr int kLagBoxCols = kLagCols + 8;  // box columns 32 b2 - 4 .. 32 b2 + 35
constexpr int kLagBoxRows = 3;    // a warp's row and its two neighbours
constexpr int kLagGridTarget = 152;  // CTAs the work is shared among (one per SM)
constexpr int kLagMaxCtas = 1024;

// Slot of the product x[c, z] x[c2, z + delta] among a region's sums, with
// delta = (j / 9 - 1, j / 3 % 3 - 1, j % 3 - 1): channel pairs c <= c2, and for
// c == c2 only the lags delta >= 0 in lexicographic order (j >= 13; the others
// are the same products seen from the other factor).  Slots 0 .. cin-1 hold
// the sums of x[c, z].  Returns -1 for a pair that has no slot.
TC3D_HD constexpr int lag_slot(int cin, int c, int c2, int j) {
  if (c > c2 || (c == c2 && j < 13)) return -1;
  int s = cin;
  for (int cc = 0; cc < c; ++cc) s += 14 + 27 * (cin - 1 - cc);
  return c2 == c ? s + j - 13 : s + 14 + 27 * (c2 - c - 1) + j;
}
// dynamic shared memory (4-byte words) of the lag finalize: the reduction's
// entry flags and list; a channel's weights, and the gather list (the pairs
// i <= j of every class, then the rows) with its coefficients
TC3D_HD constexpr int64_t lag_reduce_smem_ints(int nent) { return 2 * (int64_t)nent; }
TC3D_HD constexpr int64_t lag_channel_smem_floats(int Cin, int kvol, int rows, int pairs) {
  return (int64_t)Cin * kvol + 2 * ((int64_t)pairs + rows);
}
TC3D_HD constexpr int lag_nslots(int cin) { return cin + cin * 14 + 27 * cin * (cin - 1) / 2; }
static_assert(lag_nslots(kLagMaxCin) <= kLagSlots, "lag slots of 3 channels fit a region row");

struct PoolPlan {
  int status;     // 0: the algebraic path applies
  int D;          // patch entries Cin * nU0 * nU1 * nU2 (<= kGramMaxD)
  int nU[3];
  int U[3][kMaxAxisTaps];              // union of input offsets per axis
  // per axis, class r in {0, 1}: taps (kernel index, index into U)
  int ntap[3][2];
  int tap_k[3][2][kMaxAxisTaps], tap_u[3][2][kMaxAxisTaps];
  int M[3];                            // row grid of the transposed conv
  int nbox;
  int box_lo[kGramMaxBoxes][3], box_hi[kGramMaxBoxes][3];
  int64_t box_rows[kGramMaxBoxes];
  int ncls;                            // classes with taps on every axis
  int cls_r[8][3];
  int cls_coef[8][kGramMaxBoxes];      // inclusion-exclusion sign per box
  // Gram work units per box: the box's axes as (a0, a1, a2), a0 its thinnest;
  // a unit is Tn samples n at one m_a0 with a T1 x T2 tile of (m_a1, m_a2),
  // its x slab [Tn][Cin * nU_a0 planes][W1][W2p] floats
  int box_perm[kGramMaxBoxes][3];
  int box_Tn[kGramMaxBoxes];
  int box_T1[kGramMaxBoxes], box_T2[kGramMaxBoxes];
  int box_W1[kGramMaxBoxes], box_W2p[kGramMaxBoxes];
  int e_min[3], Ke[3];                 // pooled conv taps: e in [e_min, e_min + Ke)
  Problem conv;                        // the pooled conv (stride 2, pad -e_min)
  Plan cplan;                          // its engine plan
  int64_t ws_wpack_off;                // = cplan.ws_wpack_off
  int64_t ws_w2_off, ws_w2_bytes;      // summed, scaled weights [Cout][Cin][Ke0][Ke1][Ke2]
  int64_t ws_b2_off;                   // folded bias [Cout], the pooled conv's scale [Cout]
                                       // and its item counter
  int64_t ws_gpart_off, ws_gpart_bytes;// per-CTA Gram partials [kGramMaxCtas][kGramEntries] f32
  int64_t ws_gsum_off;                 // per-class combined Gram [8][kGramEntries] f64

  // lag form of the batch statistics (lag = 1: taken instead of the Gram
  // kernel; see lag_slot)
  int lag;
  int lag_nseg[3];
  int lag_seg[3][kLagMaxSeg + 1];      // segment s of axis a: [lag_seg[a][s], lag_seg[a][s + 1])
  int lag_bulk[3];                     // the wide segment; every other one is one position
  // per axis, class value r and offset index i: the segments [lo, hi) of
  // the z range [U_i, M_r + U_i) clipped to x
  int lag_srange[3][2][kMaxAxisTaps][2];
  // the distinct ranges among them per axis (at most 4), and the range of
  // each (class value, offset index); a class entry is then the sum over one
  // box of ranges
  int lag_nrange[3];
  int lag_range[3][4][2];
  int lag_ridx[3][2][kMaxAxisTaps];
  int lag_nreg;                        // regions, nseg0 * nseg1 * nseg2
  // work: a job is (segment s0 of axis 0, block of 8 rows, block of 32
  // columns); the jobs of segment s0 take lag_nc[s0] CTAs each, which share
  // its N * len(s0) (sample, plane) steps
  int lag_nb1, lag_nb2;
  int lag_nc[kLagMaxSeg];
  int lag_cta0[kLagMaxSeg + 1];        // first CTA of each axis-0 segment
  int lag_grid;
  int lag_nbox;                          // boxes, nrange0 * nrange1 * nrange2
  int64_t ws_lpart_off, ws_lpart_bytes;  // per-CTA box sums [grid][nbox][kLagSlots] f32
  int64_t ws_lrs_off;                    // box sums over the grid [nbox][kLagSlots] f32

  int64_t ws_total;
};

// Fill *pp for a BN-pool plan (op OP_CONVT_BN_POOL / OP_CONVT_BN_EVAL).
// Returns pp->status: 0 when the algebraic path applies.
int make_pool_plan(const Plan& bn, PoolPlan* pp);

// Integer output length of one axis.
int64_t conv_len(int64_t L, int k, int s, int p, int d);
int64_t convT_len(int64_t L, int k, int s, int p, int d, int op);

}  // namespace tc3d
