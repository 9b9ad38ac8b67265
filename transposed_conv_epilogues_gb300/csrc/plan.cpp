// plan.cpp -- host-side planning for the implicit-GEMM engine.
//
// The convolution and the transposed convolution are both cast as one GEMM
// over "rows".  For a convolution a row is an output position o; its GEMM-K
// entries are (input channel, tap) pairs read at input position
// o*stride - pad + dilation*k (direct-convolution formula of the page
// "Kimi-K2.6 l1_p59").  For a transposed convolution a row is a block of
// stride^3 outputs z = stride*m + r, one per output-parity class r.  For a
// fixed class r along an axis, tap k contributes iff (r + p - d*k) is a
// multiple of s, and then reads input m + (r + p - d*k)/s ("Kimi-K2.6
// l1_p77", receive-form derivation; "Kimi-K2.6 l2_p72", per-position tap
// table).  So every class is a dense stride-1 sub-convolution over m, and
// all classes of a row read inputs m + u for u in the union U of their
// offsets.  The GEMM-N axis holds (output channel, non-empty class) pairs;
// the packed weight of pair (class r, offset u) is W[k] with
// k = (r + p - s*u)/d when that is an integer tap, else 0.  No zero-inserted
// input is ever formed.
#include "plan.h"

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "../../include/tc3d.h"

namespace tc3d {

static int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && ((a < 0) != (b < 0))) --q;
  return q;
}
static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
static int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

int64_t conv_len(int64_t L, int k, int s, int p, int d) {
  if (L <= 0 || k <= 0 || s <= 0 || p < 0 || d <= 0) return 0;
  int64_t span = L + 2 * (int64_t)p - (int64_t)d * (k - 1) - 1;
  if (span < 0) return 0;
  return span / s + 1;
}

int64_t convT_len(int64_t L, int k, int s, int p, int d, int op) {
  if (L <= 0 || k <= 0 || s <= 0 || p < 0 || d <= 0 || op < 0) return 0;
  int64_t o = (L - 1) * s - 2 * (int64_t)p + (int64_t)d * (k - 1) + op + 1;
  return o > 0 ? o : 0;
}

static int validate(const Problem& pb, bool transposed) {
  if (pb.N <= 0 || pb.Cin <= 0 || pb.Cout <= 0) return TC3D_ERR_SHAPE;
  for (int a = 0; a < 3; ++a) {
    if (pb.S[a] <= 0 || pb.k[a] <= 0 || pb.stride[a] <= 0 || pb.dil[a] <= 0 || pb.pad[a] < 0)
      return TC3D_ERR_SHAPE;
  }
  if (pb.groups <= 0 || pb.Cin % pb.groups || pb.Cout % pb.groups) return TC3D_ERR_GROUPS;
  for (int a = 0; a < 3; ++a) {
    if (!transposed) {
      if (pb.out_pad[a] != 0) return TC3D_ERR_OUTPUT_PADDING;
    } else {
      if (pb.out_pad[a] < 0 || pb.out_pad[a] >= std::max(pb.stride[a], pb.dil[a]))
        return TC3D_ERR_OUTPUT_PADDING;
    }
  }
  return TC3D_OK;
}

// largest x misalignment (in elements, 0..3) of the raw box start
// s_in2 * T2 * b + u_min2 over tiles b; the start is rounded down to 16 bytes
static int x_slack(const Plan& pl, int t2) {
  int mx = 0;
  for (int b = 0; b < 4; ++b) {
    int64_t v = (int64_t)pl.s_in[2] * t2 * b + pl.u_min[2];
    mx = std::max(mx, (int)(((v % 4) + 4) % 4));
  }
  return mx;
}

// per-axis raw-box extent for a tile extent t (rows)
static int box_extent(const Plan& pl, int a, int t) {
  int64_t e = (int64_t)pl.s_in[a] * (t - 1) + (pl.u_max[a] - pl.u_min[a]) + 1;
  if (a == 2) e = round_up(e + x_slack(pl, t), 4);
  return (int)std::min<int64_t>(e, 1 << 30);
}

static int ilog2(int v) {
  int r = 0;
  while ((1 << (r + 1)) <= v) ++r;
  return r;
}

SmemLayout smem_layout(const Plan& pl) {
  SmemLayout L;
  L.raw = 0;
  L.b = L.raw + (int64_t)pl.raw_stages * pl.raw_stage_bytes;
  L.xs = L.b + (int64_t)pl.b_stages * pl.b_stage_bytes;
  L.ktab = L.xs + (int64_t)pl.nslots * pl.slot_bytes;
  L.misc = L.ktab + round_up((int64_t)pl.ksteps_chunk * 32, 1024);
  L.bar = L.misc + 4096;
  // + 1024 for the barriers and 1024 of slack to align the dynamic base
  L.total = L.bar + 1024 + 1024;
  // one CTA per SM: the kernel owns all 512 TMEM columns
  L.total = std::max<int64_t>(L.total, 120 * 1024);
  return L;
}

static int make_plan_direct(const Problem& pb_in, Plan* out) {
  Plan pl;
  std::memset(&pl, 0, sizeof(pl));
  pl.pb = pb_in;
  const Problem& pb = pl.pb;
  const bool transposed = pb.op == OP_CONVT || is_bn_op(pb.op);
  pl.transposed = transposed;
  pl.status = TC3D_OK;
  auto fail = [&](int st) {
    pl.status = st;
    *out = pl;
    return st;
  };
  if (pb.op < OP_CONV || pb.op > OP_CONVT_BN_EVAL) return fail(TC3D_ERR_UNSUPPORTED);
  int st = validate(pb, transposed);
  if (st) return fail(st);
  pl.cin_g = pb.Cin / pb.groups;
  pl.cout_g = pb.Cout / pb.groups;

  // ---- output and pooled extents
  for (int a = 0; a < 3; ++a) {
    pl.O[a] = transposed ? convT_len(pb.S[a], pb.k[a], pb.stride[a], pb.pad[a], pb.dil[a],
                                     pb.out_pad[a])
                         : conv_len(pb.S[a], pb.k[a], pb.stride[a], pb.pad[a], pb.dil[a]);
    if (pl.O[a] <= 0) return fail(TC3D_ERR_SHAPE);
    if (pl.O[a] > (1 << 30)) return fail(TC3D_ERR_UNSUPPORTED);
  }
  for (int a = 0; a < 3; ++a) {
    if (pb.out_ext[a] < 0 || pb.out_ext[a] > pl.O[a]) return fail(TC3D_ERR_UNSUPPORTED);
    if (pb.out_ext[a] > 0) pl.O[a] = pb.out_ext[a];
  }
  int64_t ovol = pl.O[0] * pl.O[1] * pl.O[2];
  if (pb.op == OP_CONV || pb.op == OP_CONVT) {
    pl.y_elems = (int64_t)pb.N * pb.Cout * ovol;
    pl.epi = EPI_STORE;
  } else if (pb.op == OP_CONV_POOL_LSE) {
    for (int a = 0; a < 3; ++a) {
      pl.P[a] = pl.O[a] / 2;
      if (pl.P[a] <= 0) return fail(TC3D_ERR_SHAPE);
    }
    pl.y_elems = (int64_t)pb.N * pl.P[0] * pl.P[1] * pl.P[2];
    pl.epi = EPI_POOL_LSE;
  } else {
    for (int a = 0; a < 3; ++a) {
      pl.P[a] = pl.O[a] / 2 / 2;
      if (pl.P[a] <= 0) return fail(TC3D_ERR_SHAPE);
    }
    pl.y_elems = (int64_t)pb.N * pb.Cout * pl.P[0] * pl.P[1] * pl.P[2];
    pl.epi = EPI_STORE;  // decided below, once the parity classes are known
  }
  if (pl.y_elems <= 0) return fail(TC3D_ERR_SHAPE);
  for (int a = 0; a < 3; ++a)
    if (pb.k[a] > kMaxAxisTaps) return fail(TC3D_ERR_UNSUPPORTED);
  if ((int64_t)pb.N * pb.Cin * pb.S[0] * pb.S[1] * pb.S[2] >= ((int64_t)1 << 40) ||
      (int64_t)pb.N * pb.Cout * ovol >= ((int64_t)1 << 40))
    return fail(TC3D_ERR_UNSUPPORTED);

  // ---- rows, offsets, classes
  for (int a = 0; a < 3; ++a) {
    const int s = pb.stride[a], p = pb.pad[a], d = pb.dil[a], K = pb.k[a];
    if (!transposed) {
      pl.s_in[a] = s;
      pl.s_out[a] = 1;
      pl.M[a] = (int)pl.O[a];
      pl.nU[a] = K;
      pl.u_min[a] = -p;
      pl.u_max[a] = d * (K - 1) - p;
      for (int t = 0; t < K; ++t) pl.u_rel[a][t] = d * t;
      pl.nRaxis[a] = 1;
      pl.r_axis[a][0] = 0;
      for (int t = 0; t < kMaxAxisTaps; ++t) pl.kidx[a][0][t] = t < K ? t : -1;
    } else {
      if (s > kMaxClassesAxis) return fail(TC3D_ERR_UNSUPPORTED);
      pl.s_in[a] = 1;
      pl.s_out[a] = s;
      // union of offsets u = (r + p - d k)/s over all classes and taps
      int uvals[kMaxClassesAxis * kMaxAxisTaps];
      int nu = 0;
      for (int r = 0; r < s; ++r)
        for (int k = 0; k < K; ++k) {
          int64_t t = (int64_t)r + p - (int64_t)d * k;
          if (((t % s) + s) % s != 0) continue;
          int u = (int)(t / s);
          bool seen = false;
          for (int i = 0; i < nu; ++i) seen |= uvals[i] == u;
          if (!seen) uvals[nu++] = u;
        }
      std::sort(uvals, uvals + nu);
      if (nu > kMaxAxisTaps) return fail(TC3D_ERR_UNSUPPORTED);
      pl.nU[a] = nu;
      pl.u_min[a] = uvals[0];
      pl.u_max[a] = uvals[nu - 1];
      for (int t = 0; t < nu; ++t) pl.u_rel[a][t] = uvals[t] - uvals[0];
      int nr = 0;
      for (int r = 0; r < s; ++r) {
        int row[kMaxAxisTaps];
        bool any = false;
        for (int t = 0; t < kMaxAxisTaps; ++t) row[t] = -1;
        for (int t = 0; t < nu; ++t) {
          int64_t num = (int64_t)r + p - (int64_t)s * uvals[t];
          if (num % d != 0) continue;
          int64_t k = num / d;
          if (k < 0 || k >= K) continue;
          row[t] = (int)k;
          any = true;
        }
        if (!any) continue;
        pl.r_axis[a][nr] = r;
        for (int t = 0; t < kMaxAxisTaps; ++t) pl.kidx[a][nr][t] = row[t];
        ++nr;
      }
      pl.nRaxis[a] = nr;  // >= 1: class (d*k - p) mod s always has tap k
      // rows m whose outputs s*m + r (r a class with taps) lie inside the output
      int64_t mrows = 0;
      for (int i = 0; i < nr; ++i)
        mrows = std::max<int64_t>(mrows, ceil_div(pl.O[a] - pl.r_axis[a][i], s));
      pl.M[a] = (int)mrows;
      if (mrows * s < pl.O[a]) pl.fill_slab = 1;
    }
  }
  pl.nR = pl.nRaxis[0] * pl.nRaxis[1] * pl.nRaxis[2];
  {
    // the one-class store path: at most 8 classes, whose offsets from a
    // row's first output fit in an int; along x with stride 2 it writes only
    // the rows of its class pair, and the bias fill the others
    const int F = pl.s_out[0] * pl.s_out[1] * pl.s_out[2];
    const int64_t maxoff = (int64_t)(pl.s_out[0] - 1) * pl.O[1] * pl.O[2] +
                           (int64_t)(pl.s_out[1] - 1) * pl.O[2] + (pl.s_out[2] - 1);
    pl.cls_fast = pl.nR == 1 && F <= 8 && maxoff <= INT32_MAX;
    pl.fill_rows = pl.cls_fast && pl.s_out[2] == 2 && pl.s_out[0] * pl.s_out[1] > 1;
    if (pl.fill_rows) pl.fill_slab = 1;
  }
  if (is_bn_op(pb.op)) {
    // fused BatchNorm + 4x4x4 pooling: a row is a 2x2x2 output block with all
    // 8 parity classes carrying taps, so a 4^3 window is 2x2x2 rows
    pl.fused = pb.stride[0] == 2 && pb.stride[1] == 2 && pb.stride[2] == 2 && pl.nR == 8;
    pl.epi = pl.fused ? EPI_BN_POOL : EPI_STORE;
  }
  pl.nEmpty = pl.s_out[0] * pl.s_out[1] * pl.s_out[2] - pl.nR;
  if (pl.nR > 128) return fail(TC3D_ERR_UNSUPPORTED);
  const int nUtot = pl.nU[0] * pl.nU[1] * pl.nU[2];

  // ---- GEMM N (column blocks)
  {
    int cap = pl.epi == EPI_POOL_LSE ? 256 : 128;
    pl.ocb = std::max(1, std::min(pl.cout_g, cap / pl.nR));
    pl.n_tile = (int)round_up((int64_t)pl.ocb * pl.nR, 16);
    if (pl.n_tile > 256) return fail(TC3D_ERR_UNSUPPORTED);
    pl.nb_per_group = (int)ceil_div(pl.cout_g, pl.ocb);
    pl.n_colblocks = pb.groups * pl.nb_per_group;
  }

  // ---- accumulators per tile, TMEM budget
  // Accumulators are double-buffered (the epilogue drains one buffer while
  // the MMAs fill the other) whenever two buffers of at least one 128-row
  // accumulator fit in half of TMEM.  Short MMAs (N <= 64) issue about as
  // fast as the tensor core executes them, so when TMEM still allows two
  // accumulators per buffer the x.w and x.w_lo products are fused into one
  // MMA over the adjacent [w | w_lo] weight block (N = 2 n_tile), its two
  // halves summed in the epilogue.
  pl.dbuf = pl.n_tile > 128 ? 1 : 2;
  pl.wide = (pl.epi != EPI_BN_POOL && 2 * pl.n_tile <= 128 &&
             256 / (pl.dbuf * 2 * pl.n_tile) >= 2)
                ? 1
                : 0;
  pl.acc_cols = pl.wide ? 2 * pl.n_tile : pl.n_tile;
  pl.n_acc = std::max(1, std::min(4, 256 / (pl.dbuf * pl.acc_cols)));
  {
    int dcols = pl.n_acc * pl.acc_cols * pl.dbuf;
    // A-stage ring sized below, once the K-steps per channel chunk are known
    pl.a_stages = 0;
  }

  // ---- quarter box Q and quarter arrangement P (search)
  {
    const int nq = 4 * pl.n_acc;
    const int lq = ilog2(nq);
    double best = 1e300;
    int bestQ[3] = {0, 0, 0}, bestP[3] = {0, 0, 0};
    for (int q2 = 0; q2 <= 5; ++q2)
      for (int q1 = 0; q1 + q2 <= 5; ++q1) {
        int q0 = 5 - q1 - q2;
        int Q[3] = {1 << q0, 1 << q1, 1 << q2};
        if (pl.epi != EPI_STORE && !(Q[0] == 2 && Q[1] == 2 && Q[2] == 8)) continue;
        for (int p2 = 0; p2 <= lq; ++p2)
          for (int p1 = 0; p1 + p2 <= lq; ++p1) {
            int p0 = lq - p1 - p2;
            int P[3] = {1 << p0, 1 << p1, 1 << p2};
            int T[3];
            bool ok = true;
            double rows = 1;
            for (int a = 0; a < 3; ++a) {
              T[a] = P[a] * Q[a];
              rows *= (double)round_up(pl.M[a], T[a]);
              int be = box_extent(pl, a, T[a]);
              if (be > 256) ok = false;
            }
            if (!ok) continue;
            double raw = (double)box_extent(pl, 0, T[0]) * box_extent(pl, 1, T[1]) *
                         box_extent(pl, 2, T[2]);
            double per_row = raw / (128.0 * pl.n_acc);
            double cost = rows * (1.0 + 0.04 * per_row);
            if (pl.epi == EPI_STORE) {
              // bytes a warp stores contiguously per (channel, class row)
              int64_t seg = (int64_t)Q[2] * pl.s_out[2];
              if (Q[2] == pl.M[2] && pl.s_out[2] == 1 && pl.M[2] == pl.O[2]) {
                seg *= Q[1];
                if (Q[1] == pl.M[1] && pl.s_out[1] == 1 && pl.M[1] == pl.O[1]) seg *= Q[0];
              }
              const double segb = (double)std::min<int64_t>(seg * 4, 128);
              cost *= 1.0 + 0.25 * (128.0 / segb - 1.0);
            }
            if (cost < best) {
              best = cost;
              for (int a = 0; a < 3; ++a) {
                bestQ[a] = Q[a];
                bestP[a] = P[a];
              }
            }
          }
      }
    if (best >= 1e300) return fail(TC3D_ERR_UNSUPPORTED);
    for (int a = 0; a < 3; ++a) {
      pl.Q[a] = bestQ[a];
      pl.Pq[a] = bestP[a];
      pl.T[a] = bestQ[a] * bestP[a];
      pl.ntile[a] = (int)ceil_div(pl.M[a], pl.T[a]);
      pl.box[a] = box_extent(pl, a, pl.T[a]);
    }
    pl.xslack = x_slack(pl, pl.T[2]);
    pl.tiles = (int64_t)pb.N * pl.ntile[0] * pl.ntile[1] * pl.ntile[2];
    if (pl.tiles >= ((int64_t)1 << 31)) return fail(TC3D_ERR_UNSUPPORTED);
  }

  // ---- channels-last mode: a conv on NDHWC tensors (groups 1, one class)
  // whose box and tap count fit.  The box's x start needs no 16-byte
  // rounding there (channels are the innermost axis), so it has no slack.
  // The tile found above is kept when its box fits the mode's stage budget;
  // else a search of its own picks the tile (no x-store preference: a row's
  // channels are one contiguous run whatever the tile).
  pl.cl = 0;
  if (pb.cl && pb.op == OP_CONV && pb.groups == 1 && pl.nR == 1 && nUtot <= kMaxKChunk / 8) {
    const int64_t bstage = 64LL * pl.n_tile;
    const int64_t fixed = 4096 + 1024 + 1024;
    auto cl_box = [&](int a, int t) {
      return (int)std::min<int64_t>(
          (int64_t)pl.s_in[a] * (t - 1) + (pl.u_max[a] - pl.u_min[a]) + 1, 1 << 30);
    };
    // the chunk of 8, 16, 24 or 32 channels (not past the channel count)
    // whose two raw stages fit beside the weight stages: the fewest K-steps
    // over all chunks (a ragged last chunk is padded), then the widest
    auto fit = [&](Plan& c) {
      for (int a = 0; a < 3; ++a) c.box[a] = cl_box(a, c.T[a]);
      c.xslack = 0;
      const int64_t bvol = (int64_t)c.box[0] * c.box[1] * c.box[2];
      int64_t best_steps = INT64_MAX;
      for (int cc = std::min(32, (int)round_up(c.cin_g, 8)); cc >= 8; cc -= 8) {
        const int64_t raw = round_up(bvol * (cc + 4) * 4, 1024);
        const int64_t ks = (int64_t)(cc / 8) * nUtot;
        if (c.box[0] > 256 || c.box[1] > 256 || c.box[2] > 256 || raw > 96 * 1024 ||
            cc * nUtot > kMaxKChunk)
          continue;
        if (2 * raw + 4 * bstage + fixed + round_up(ks * 32, 1024) > kMaxSmem) continue;
        const int64_t steps = ceil_div(c.cin_g, cc) * ks;
        if (steps >= best_steps) continue;
        best_steps = steps;
        c.cl = 1;
        c.cl_cb = cc + 4;
        c.cin_chunk = cc;
        c.n_chunks = (int)ceil_div(c.cin_g, cc);
        c.k_chunk = cc * nUtot;
        c.ksteps_chunk = (int)ks;
        c.raw_stage_bytes = raw;
      }
      return c.cl == 1;
    };
    Plan c = pl;
    if (!fit(c)) {
      const int lq = ilog2(4 * pl.n_acc);
      double best = 1e300;
      for (int q2 = 0; q2 <= 5; ++q2)
        for (int q1 = 0; q1 + q2 <= 5; ++q1)
          for (int p2 = 0; p2 <= lq; ++p2)
            for (int p1 = 0; p1 + p2 <= lq; ++p1) {
              const int Q[3] = {1 << (5 - q1 - q2), 1 << q1, 1 << q2};
              const int P[3] = {1 << (lq - p1 - p2), 1 << p1, 1 << p2};
              Plan t = pl;
              double rows = 1, bv = 1;
              for (int a = 0; a < 3; ++a) {
                t.Q[a] = Q[a];
                t.Pq[a] = P[a];
                t.T[a] = Q[a] * P[a];
                rows *= (double)round_up(pl.M[a], t.T[a]);
                bv *= cl_box(a, t.T[a]);
              }
              const double cost = rows * (1.0 + 0.04 * bv / (128.0 * pl.n_acc));
              if (cost < best && fit(t)) {
                best = cost;
                c = t;
              }
            }
      if (c.cl) {
        for (int a = 0; a < 3; ++a) c.ntile[a] = (int)ceil_div(c.M[a], c.T[a]);
        c.tiles = (int64_t)pb.N * c.ntile[0] * c.ntile[1] * c.ntile[2];
        if (c.tiles >= ((int64_t)1 << 31)) c.cl = 0;
      }
    }
    if (c.cl) pl = c;
  }

  // ---- channel chunk, smem budget
  {
    const int64_t bvol = (int64_t)pl.box[0] * pl.box[1] * pl.box[2];
    const int64_t raw_ch = bvol * 4;
    const int64_t bstage = 64LL * pl.n_tile;  // w + w_lo, n_tile x 8 tf32 each
    const int64_t fixed = 4096 + 1024 + 1024; // epilogue scratch, barriers, alignment
    if (!pl.cl) {
      int best_cc = 0;
      int64_t best_steps = INT64_MAX;
      int max_cc = std::min(pl.cin_g, kMaxKChunk / nUtot);
      if (max_cc < 1) return fail(TC3D_ERR_UNSUPPORTED);
      for (int cc = 1; cc <= max_cc; ++cc) {
        int64_t need = 2 * round_up(cc * raw_ch, 1024) + 4 * bstage + fixed +
                       round_up(ceil_div((int64_t)cc * nUtot, 8) * 32, 1024);
        if (need > kMaxSmem) break;
        if (cc * raw_ch > 64 * 1024 && cc > 1) break;  // keep one stage modest
        int64_t steps = ceil_div(pl.cin_g, cc) * ceil_div((int64_t)cc * nUtot, 8);
        if (steps <= best_steps) {
          best_steps = steps;
          best_cc = cc;
        }
      }
      if (best_cc == 0) return fail(TC3D_ERR_UNSUPPORTED);
      pl.cin_chunk = best_cc;
      pl.n_chunks = (int)ceil_div(pl.cin_g, best_cc);
      pl.k_chunk = best_cc * nUtot;
      pl.ksteps_chunk = (int)ceil_div(pl.k_chunk, 8);
      pl.raw_stage_bytes = round_up(best_cc * raw_ch, 1024);
    }
    // An A-stage carries up to ks_stage K-steps of all accumulators (up to 24
    // MMAs) so that each stage's barrier wait / commit is amortised; a stage
    // never straddles two channel chunks.  Streamed weight stages match
    // A-stages.
    {
      const int dcols = pl.n_acc * pl.acc_cols * pl.dbuf;
      pl.ks_stage = 1;
      // the last stage of a chunk may hold fewer K-steps; a weight stage
      // stays within 32 KB
      // about 24 MMAs per stage (2 per accumulator and K-step when wide, else 3)
      const int per_ks = pl.n_acc * (pl.wide ? 2 : 3);
      for (int ks = std::min(std::max(1, 24 / per_ks), pl.ksteps_chunk); ks > 1; --ks)
        if (64LL * pl.n_tile * ks <= 32 * 1024 &&
            (kTmemCols - dcols) / (16 * pl.n_acc * ks) >= 2) {
          pl.ks_stage = ks;
          break;
        }
      pl.a_stages = std::min(16, (kTmemCols - dcols) / (16 * pl.n_acc * pl.ks_stage));
      if (pl.a_stages < 2) return fail(TC3D_ERR_UNSUPPORTED);
    }
    const int64_t ktab = round_up((int64_t)pl.ksteps_chunk * 32, 1024);
    const int64_t total_ksteps = (int64_t)pl.n_chunks * pl.ksteps_chunk;
    pl.b_stage_bytes = bstage;
    const int64_t rem = kMaxSmem - fixed - ktab - 2 * pl.raw_stage_bytes;
    if (pl.n_colblocks == 1 && total_ksteps * bstage <= std::min<int64_t>(rem, 112 * 1024)) {
      pl.b_resident = 1;
      pl.b_stages = (int)total_ksteps;
    } else {
      pl.b_resident = 0;
      pl.b_stage_bytes = bstage * pl.ks_stage;
      pl.b_stages = (int)std::min<int64_t>(kMaxBStagesPlan, rem / pl.b_stage_bytes);
      if (pl.b_stages < 2) return fail(TC3D_ERR_UNSUPPORTED);
    }
    const int64_t used = (int64_t)pl.b_stages * pl.b_stage_bytes + ktab + fixed;
    pl.raw_stages = (used + 3 * pl.raw_stage_bytes <= kMaxSmem) ? 3 : 2;
    pl.smem_bytes = smem_layout(pl).total;
    if (pl.smem_bytes > kMaxSmem) return fail(TC3D_ERR_UNSUPPORTED);
  }

  // ---- view mode: a plain stride-1 conv whose accumulators are runs of 128
  // consecutive raw-box positions: row r of accumulator a is position
  // a*B1*B2 + r (+ the tap's offset).  Two geometries qualify:
  //   lines:    one tap along x (no x halo) and x lines filling 128 rows
  //             (x extent 4..32): an accumulator is 128/S2 whole x lines;
  //   segments: a y extent of 1 (the merged form of a (k,k,1) conv, see
  //             make_plan): an accumulator is 128 consecutive x positions,
  //             and an x halo only shifts a tap's window.
  // Channels are padded to octets with zeros.
  {
    const int S2 = pb.S[2];
    const bool base_ok = pb.op == OP_CONV && !pl.cl && !pb.cl && pl.s_in[0] == 1 && pl.s_in[1] == 1 &&
                         pl.s_in[2] == 1 && pl.n_tile <= 128 && pl.nR == 1 &&
                         pl.n_colblocks == 1;
    const bool lines = base_ok && pl.nU[2] == 1 && pl.u_min[2] == 0 && pl.M[2] == S2 &&
                       (S2 == 4 || S2 == 8 || S2 == 16 || S2 == 32);
    const bool segments = base_ok && !lines && pb.S[1] == 1 && pl.nU[1] == 1 &&
                          pl.u_min[1] == 0 && pl.M[1] == 1;
    if (lines || segments) {
      Plan v = pl;
      v.view = 1;
      v.dbuf = 2;
      v.wide = 2 * v.n_tile <= 128 ? 1 : 0;
      v.acc_cols = v.wide ? 2 * v.n_tile : v.n_tile;
      v.n_acc = 2;
      v.ks_stage = 0;
      v.a_stages = 0;
      if (lines) {
        v.Q[0] = 1, v.Q[1] = 32 / S2, v.Q[2] = S2;
        v.Pq[0] = 2, v.Pq[1] = 4, v.Pq[2] = 1;
      } else {
        v.Q[0] = 1, v.Q[1] = 1, v.Q[2] = 32;
        v.Pq[0] = 2, v.Pq[1] = 1, v.Pq[2] = 4;
      }
      for (int a = 0; a < 3; ++a) {
        v.T[a] = v.Q[a] * v.Pq[a];
        v.ntile[a] = (int)ceil_div(v.M[a], v.T[a]);
        v.box[a] = box_extent(v, a, v.T[a]);
      }
      v.xslack = x_slack(v, v.T[2]);
      v.tiles = (int64_t)pb.N * v.ntile[0] * v.ntile[1] * v.ntile[2];
      const int64_t bvol = (int64_t)v.box[0] * v.box[1] * v.box[2];
      const int ntaps = nUtot;
      v.slot_bytes = 2 * bvol * 8 * 4;
      v.nslots = 2;
      const int64_t fixed = 4096 + 1024 + 1024 + 1024 + round_up((int64_t)ntaps * 4, 1024);
      const int cin_pad = (int)round_up(v.cin_g, 8);
      int best = 0;
      int64_t best_w = 0;
      for (int cc = 8; cc <= cin_pad; cc += 8) {
        // weights stay resident: chunks x octets x taps K-steps of 64 * n_tile bytes
        const int64_t wbytes = ceil_div(v.cin_g, cc) * (cc / 8) * ntaps * 64LL * v.n_tile;
        const int64_t raw = round_up(cc * bvol * 4, 1024);
        if (2 * raw + v.nslots * v.slot_bytes + wbytes + fixed <= kMaxSmem) {
          best = cc;
          best_w = wbytes;
        }
      }
      if (best > 0 && bvol <= 16383 && v.box[0] <= 256 && v.box[1] <= 256 &&
          v.box[2] <= 256 && v.tiles < ((int64_t)1 << 31)) {
        v.cin_chunk = best;
        v.n_chunks = (int)ceil_div(v.cin_g, best);
        v.k_chunk = best * ntaps;
        v.ksteps_chunk = (best / 8) * ntaps;
        v.raw_stage_bytes = round_up(best * bvol * 4, 1024);
        v.b_resident = 1;
        v.b_stage_bytes = 64LL * v.n_tile;
        v.b_stages = (int)((int64_t)v.n_chunks * v.ksteps_chunk);
        const int64_t used = 2 * v.raw_stage_bytes + v.nslots * v.slot_bytes + best_w + fixed;
        v.raw_stages = used + v.raw_stage_bytes <= kMaxSmem ? 3 : 2;
        v.smem_bytes = smem_layout(v).total;
        if (v.smem_bytes <= kMaxSmem) pl = v;
      }
    }
  }

  // ---- workspace
  {
    int64_t off = 0;
    pl.ws_wpack_off = off;
    pl.ws_wpack_bytes = (int64_t)pl.n_colblocks * pl.n_chunks * pl.ksteps_chunk * 64 * pl.n_tile;
    off = round_up(off + pl.ws_wpack_bytes, 256);
    if (pl.fill_slab) {
      pl.ws_ctr_off = off;
      off = round_up(off + 8, 256);
    }
    if (is_bn_op(pb.op)) {
      pl.ws_part_off = off;
      // batch statistics: fused, enough slots for any grid; unfused, per
      // (n, c) double sums.  Running statistics need no partial sums.
      const int64_t slots = bn_part_slots(pl, std::min<int64_t>(pl.tiles, kMaxGrid));
      if (pb.op == OP_CONVT_BN_POOL)
        pl.ws_part_bytes = pl.fused ? slots * pb.Cout * 8 : (int64_t)pb.N * pb.Cout * 16;
      off = round_up(off + pl.ws_part_bytes, 256);
      pl.ws_stat_off = off;
      pl.ws_stat_bytes = (int64_t)pb.Cout * 8;
      off = round_up(off + pl.ws_stat_bytes, 256);
      if (!pl.fused) {
        pl.ws_full_off = off;
        pl.ws_full_bytes = (int64_t)pb.N * pb.Cout * ovol * 4;
        off = round_up(off + pl.ws_full_bytes, 256);
      }
    }
    pl.ws_total = std::max<int64_t>(off, 256);
  }
  *out = pl;
  return TC3D_OK;
}

// A conv whose kernel has one tap along the contiguous axis, with no padding
// there, is the same conv over a merged (S1 * S2) axis: x as [N, C, S0, 1,
// S1*S2] with kernel (k0, 1, k1), dilation (d0, 1, d1*S2) and padding
// (p0, 0, p1*S2) -- a tap along S1 shifts the merged index by whole lines
// of S2, and indices outside the merged line are exactly the padded ones.
// The output is y itself, read as [N, Cout, O0, 1, O1*S2].  The merged form
// is used when it runs in view mode; the plan then keeps the caller's
// output extents in O_user.
int make_plan(const Problem& pb, Plan* out) {
  if (pb.op == OP_CONV && pb.k[2] == 1 && pb.pad[2] == 0 && pb.stride[0] == 1 &&
      pb.out_ext[0] == 0 && pb.out_ext[1] == 0 && pb.out_ext[2] == 0 &&
      pb.stride[1] == 1 && pb.stride[2] == 1 && pb.groups == 1 &&
      validate(pb, false) == TC3D_OK && (int64_t)pb.S[1] * pb.S[2] < (1 << 30)) {
    Problem m = pb;
    m.S[1] = 1;
    m.S[2] = pb.S[1] * pb.S[2];
    m.k[1] = 1;
    m.k[2] = pb.k[1];
    m.pad[1] = 0;
    m.pad[2] = pb.pad[1] * pb.S[2];
    m.dil[1] = 1;
    m.dil[2] = pb.dil[1] * pb.S[2];
    Plan pm;
    if (make_plan_direct(m, &pm) == TC3D_OK && pm.view) {
      pm.reshaped = 1;
      pm.O_user[0] = pm.O[0];
      pm.O_user[1] = conv_len(pb.S[1], pb.k[1], 1, pb.pad[1], pb.dil[1]);
      pm.O_user[2] = pb.S[2];
      *out = pm;
      return TC3D_OK;
    }
  }
  const int st = make_plan_direct(pb, out);
  for (int a = 0; a < 3; ++a) out->O_user[a] = out->O[a];
  return st;
}

// Lag form of the batch statistics (see lag_slot in plan.h): segments,
// region count, the per-class segment ranges and the work split.  Leaves
// pp.lag = 0 where it does not apply: more than 3 channels, an axis whose
// offsets are neither one value nor two consecutive ones, rows along axis 2
// that TMA cannot load (extent not a multiple of 4), more than one segment
// wider than one position, or more CTAs than kLagMaxCtas.
static void plan_lag(const Plan& bn, PoolPlan& pp) {
  const Problem& pb = bn.pb;
  pp.lag = 0;
  if (pb.Cin > kLagMaxCin || pb.S[2] % 4 != 0) return;
  for (int a = 0; a < 3; ++a) {
    if (pp.nU[a] > 2) return;
    if (pp.nU[a] == 2 && pp.U[a][1] != pp.U[a][0] + 1) return;
  }
  auto clampi = [](int64_t v, int64_t lo, int64_t hi) {
    return (int)std::min<int64_t>(std::max<int64_t>(v, lo), hi);
  };
  for (int a = 0; a < 3; ++a) {
    const int L = pb.S[a];
    // breakpoints: the ends of the z ranges [u, M_r + u) of every class
    // value r with taps along this axis and every offset u, clipped to x
    int bp[2 + 4 * kMaxAxisTaps], nbp = 0;
    bp[nbp++] = 0;
    bp[nbp++] = L;
    for (int r = 0; r < 2; ++r) {
      if (!pp.ntap[a][r]) continue;
      const int64_t Mr = ceil_div(bn.O[a] - r, 2);
      for (int i = 0; i < pp.nU[a]; ++i) {
        bp[nbp++] = clampi(pp.U[a][i], 0, L);
        bp[nbp++] = clampi(Mr + pp.U[a][i], 0, L);
      }
    }
    std::sort(bp, bp + nbp);
    nbp = (int)(std::unique(bp, bp + nbp) - bp);
    if (nbp - 1 > kLagMaxSeg) return;
    pp.lag_nseg[a] = nbp - 1;
    for (int s = 0; s < nbp; ++s) pp.lag_seg[a][s] = bp[s];
    // one wide segment; every other one a single position
    int bulk = 0;
    for (int s = 1; s < nbp - 1; ++s)
      if (bp[s + 1] - bp[s] > bp[bulk + 1] - bp[bulk]) bulk = s;
    for (int s = 0; s < nbp - 1; ++s)
      if (s != bulk && bp[s + 1] - bp[s] != 1) return;
    pp.lag_bulk[a] = bulk;
    for (int r = 0; r < 2; ++r)
      for (int i = 0; i < kMaxAxisTaps; ++i) pp.lag_srange[a][r][i][0] = pp.lag_srange[a][r][i][1] = 0;
    for (int r = 0; r < 2; ++r) {
      if (!pp.ntap[a][r]) continue;
      const int64_t Mr = ceil_div(bn.O[a] - r, 2);
      for (int i = 0; i < pp.nU[a]; ++i) {
        const int lo = clampi(pp.U[a][i], 0, L), hi = clampi(Mr + pp.U[a][i], 0, L);
        if (lo >= hi) continue;
        const int slo = (int)(std::find(bp, bp + nbp, lo) - bp);
        const int shi = (int)(std::find(bp, bp + nbp, hi) - bp);
        pp.lag_srange[a][r][i][0] = slo;
        pp.lag_srange[a][r][i][1] = shi;
      }
    }
    pp.lag_nrange[a] = 0;
    for (int r = 0; r < 2; ++r)
      for (int i = 0; i < kMaxAxisTaps; ++i) {
        pp.lag_ridx[a][r][i] = 0;
        if (!pp.ntap[a][r] || i >= pp.nU[a]) continue;
        const int lo = pp.lag_srange[a][r][i][0], hi = pp.lag_srange[a][r][i][1];
        int k = 0;
        while (k < pp.lag_nrange[a] && !(pp.lag_range[a][k][0] == lo && pp.lag_range[a][k][1] == hi))
          ++k;
        if (k == pp.lag_nrange[a]) {
          if (k == 4) return;
          pp.lag_range[a][k][0] = lo;
          pp.lag_range[a][k][1] = hi;
          ++pp.lag_nrange[a];
        }
        pp.lag_ridx[a][r][i] = k;
      }
  }
  pp.lag_nreg = pp.lag_nseg[0] * pp.lag_nseg[1] * pp.lag_nseg[2];
  pp.lag_nbox = pp.lag_nrange[0] * pp.lag_nrange[1] * pp.lag_nrange[2];
  // the finalize stages a channel's weights and its gather list in shared
  // memory, the reduction its entry flags (at most 192 KB each)
  int rows = 0, pairs = 0;
  for (int c = 0; c < pp.ncls; ++c) {
    const int ne = pb.Cin * pp.ntap[0][pp.cls_r[c][0]] * pp.ntap[1][pp.cls_r[c][1]] *
                   pp.ntap[2][pp.cls_r[c][2]];
    rows += ne;
    pairs += ne * (ne + 1) / 2;
  }
  if (lag_channel_smem_floats(pb.Cin, pb.k[0] * pb.k[1] * pb.k[2], rows, pairs) * 4 > 192 * 1024 ||
      lag_reduce_smem_ints(pp.lag_nbox * kLagSlots) * 4 > 192 * 1024)
    return;
  // work split: the jobs of axis-0 segment s (one per block of 8 rows and 32
  // columns) cost about N (2 len(s) + 3.5) each, in units of half a step: a
  // step per plane, and per run of consecutive planes (one per sample) the
  // planes it loads first and the wait for its first chunk, which no earlier
  // work hides (measured on GB300: a run costs about 1.7 steps); CTAs in
  // proportion, at least one per job, then spare CTAs to the segment whose
  // CTAs carry most
  pp.lag_nb1 = (int)ceil_div(pb.S[1], kLagRows);
  pp.lag_nb2 = (int)ceil_div(pb.S[2], kLagCols);
  const int64_t jobs_per_seg = (int64_t)pp.lag_nb1 * pp.lag_nb2;
  if (jobs_per_seg * pp.lag_nseg[0] > kLagMaxCtas) return;
  double cost[kLagMaxSeg], total = 0.0;
  for (int s = 0; s < pp.lag_nseg[0]; ++s) {
    const int len = pp.lag_seg[0][s + 1] - pp.lag_seg[0][s];
    cost[s] = (double)pb.N * (2.0 * len + 3.5);
    total += cost[s] * (double)jobs_per_seg;
  }
  int64_t grid = 0;
  for (int s = 0; s < pp.lag_nseg[0]; ++s) {
    const int len = pp.lag_seg[0][s + 1] - pp.lag_seg[0][s];
    const int64_t cap = (int64_t)pb.N * len;
    const int64_t share = (int64_t)((double)kLagGridTarget * cost[s] / total);
    pp.lag_nc[s] = (int)std::max<int64_t>(1, std::min<int64_t>(cap, share));
    grid += jobs_per_seg * pp.lag_nc[s];
  }
  for (;;) {
    int best = -1;
    double worst = 0.0;
    for (int s = 0; s < pp.lag_nseg[0]; ++s) {
      const int len = pp.lag_seg[0][s + 1] - pp.lag_seg[0][s];
      if (pp.lag_nc[s] >= (int64_t)pb.N * len) continue;
      const double per = cost[s] / pp.lag_nc[s];
      if (per > worst) {
        worst = per;
        best = s;
      }
    }
    if (best < 0 || grid + jobs_per_seg > std::max<int64_t>(kLagGridTarget, jobs_per_seg * pp.lag_nseg[0]))
      break;
    ++pp.lag_nc[best];
    grid += jobs_per_seg;
  }
  if (grid > kLagMaxCtas) return;
  pp.lag_cta0[0] = 0;
  for (int s = 0; s < pp.lag_nseg[0]; ++s)
    pp.lag_cta0[s + 1] = pp.lag_cta0[s] + (int)(jobs_per_seg * pp.lag_nc[s]);
  pp.lag_grid = (int)grid;
  pp.lag = 1;
}

int make_pool_plan(const Plan& bn, PoolPlan* out) {
  PoolPlan& pp = *out;
  std::memset(&pp, 0, sizeof(pp));
  pp.status = TC3D_ERR_UNSUPPORTED;
  const Problem& pb = bn.pb;
  if (bn.status != TC3D_OK || !is_bn_op(pb.op) || pb.groups != 1) return pp.status;
  for (int a = 0; a < 3; ++a)
    if (pb.stride[a] != 2) return pp.status;
  // offsets and taps per axis and class: class r, tap k reads m + (r + p - d k)/2
  int V = 1;
  for (int a = 0; a < 3; ++a) {
    const int p = pb.pad[a], d = pb.dil[a];
    int umin = 1 << 30, umax = -(1 << 30);
    for (int r = 0; r < 2; ++r)
      for (int k = 0; k < pb.k[a]; ++k) {
        const int t = r + p - d * k;
        if (t % 2 == 0) {
          umin = std::min(umin, t / 2);
          umax = std::max(umax, t / 2);
        }
      }
    if (umin > umax || umax - umin + 1 > kMaxAxisTaps) return pp.status;
    int used[kMaxAxisTaps] = {0};
    for (int r = 0; r < 2; ++r)
      for (int k = 0; k < pb.k[a]; ++k) {
        const int t = r + p - d * k;
        if (t % 2 == 0) used[t / 2 - umin] = 1;
      }
    int idx[kMaxAxisTaps];
    pp.nU[a] = 0;
    for (int u = umin; u <= umax; ++u)
      if (used[u - umin]) {
        idx[u - umin] = pp.nU[a];
        pp.U[a][pp.nU[a]++] = u;
      }
    for (int r = 0; r < 2; ++r) {
      pp.ntap[a][r] = 0;
      for (int k = 0; k < pb.k[a]; ++k) {
        const int t = r + p - d * k;
        if (t % 2 == 0) {
          const int i = pp.ntap[a][r]++;
          pp.tap_k[a][r][i] = k;
          pp.tap_u[a][r][i] = idx[t / 2 - umin];
        }
      }
    }
    V *= pp.nU[a];
  }
  pp.D = pb.Cin * V;
  if (pp.D > kGramMaxD) return pp.status;

  // rows: class r has rows m < ceil((O - r)/2); the box is the largest of them
  int slab_axis[3], nslab = 0;
  for (int a = 0; a < 3; ++a) {
    int64_t Mr[2];
    for (int r = 0; r < 2; ++r) Mr[r] = pp.ntap[a][r] ? ceil_div(bn.O[a] - r, 2) : 0;
    pp.M[a] = (int)std::max(Mr[0], Mr[1]);
    if (pp.M[a] <= 0) return pp.status;
    for (int r = 0; r < 2; ++r)
      if (pp.ntap[a][r] && Mr[r] < pp.M[a]) {  // at most one row fewer
        slab_axis[nslab++] = a;
        break;
      }
  }
  // boxes: subsets S of the slab axes; on an axis in S only the last row
  pp.nbox = 1 << nslab;
  for (int b = 0; b < pp.nbox; ++b) {
    int64_t rows = pb.N;
    for (int a = 0; a < 3; ++a) {
      pp.box_lo[b][a] = 0;
      pp.box_hi[b][a] = pp.M[a];
    }
    for (int i = 0; i < nslab; ++i)
      if (b >> i & 1) pp.box_lo[b][slab_axis[i]] = pp.M[slab_axis[i]] - 1;
    for (int a = 0; a < 3; ++a) rows *= pp.box_hi[b][a] - pp.box_lo[b][a];
    pp.box_rows[b] = rows;
  }
  // classes with taps on every axis, and their inclusion-exclusion signs
  pp.ncls = 0;
  for (int r0 = 0; r0 < 2; ++r0)
    for (int r1 = 0; r1 < 2; ++r1)
      for (int r2 = 0; r2 < 2; ++r2) {
        const int r[3] = {r0, r1, r2};
        if (!pp.ntap[0][r0] || !pp.ntap[1][r1] || !pp.ntap[2][r2]) continue;
        const int c = pp.ncls++;
        int short_mask = 0;  // slab axes on which this class ends one row early
        for (int i = 0; i < nslab; ++i) {
          const int a = slab_axis[i];
          if (ceil_div(bn.O[a] - r[a], 2) < pp.M[a]) short_mask |= 1 << i;
        }
        for (int a = 0; a < 3; ++a) pp.cls_r[c][a] = r[a];
        for (int b = 0; b < pp.nbox; ++b) {
          int bits = 0;
          for (int i = 0; i < nslab; ++i) bits += b >> i & 1;
          pp.cls_coef[c][b] = (b & ~short_mask) ? 0 : (bits & 1 ? -1 : 1);
        }
      }

  // Gram work units: per box, a0 = its thinnest axis (the first of equals),
  // a2 = the longest of the other two (the later of equals), a1 the third; a
  // unit is Tn samples at one m_a0 and a tile of T1 x T2 rows of
  // (m_a1, m_a2), whose x slabs must fit one buffer
  for (int b = 0; b < pp.nbox; ++b) {
    int ext[3], a0 = 0;
    for (int a = 0; a < 3; ++a) ext[a] = pp.box_hi[b][a] - pp.box_lo[b][a];
    for (int a = 1; a < 3; ++a)
      if (ext[a] < ext[a0]) a0 = a;
    int a1 = a0 == 0 ? 1 : 0, a2 = a0 == 2 ? 1 : 2;
    if (ext[a1] > ext[a2]) std::swap(a1, a2);
    pp.box_perm[b][0] = a0;
    pp.box_perm[b][1] = a1;
    pp.box_perm[b][2] = a2;
    const int span1 = pp.U[a1][pp.nU[a1] - 1] - pp.U[a1][0];
    const int span2 = pp.U[a2][pp.nU[a2] - 1] - pp.U[a2][0];
    const int T2 = std::min(ext[a2], 64);
    // row stride: 4 x an odd number, so that rows are 16-byte copies and the
    // 32 lines a warp reads (each lane at its own rotated start) fall in
    // distinct banks
    int W2p = (T2 + span2 + 3) / 4 * 4;
    if ((W2p / 4) % 2 == 0) W2p += 4;
    const int64_t planes = (int64_t)pb.Cin * pp.nU[a0];
    const int64_t t1 = kGramSlabFloats / (planes * W2p) - span1;
    if (t1 < 1) return pp.status;
    pp.box_T2[b] = T2;
    pp.box_W2p[b] = W2p;
    pp.box_T1[b] = (int)std::min<int64_t>(t1, ext[a1]);
    pp.box_W1[b] = pp.box_T1[b] + span1;
    // thin boxes: several samples per unit, as many slabs as fit, but at
    // least 8 units per box so that several CTAs can share it
    pp.box_Tn[b] = (int)std::max<int64_t>(
        1, std::min<int64_t>({(int64_t)(pb.N + 7) / 8,
                              kGramSlabFloats / (planes * pp.box_W1[b] * W2p)}));
    // the kernel decodes unit indices in 32 bits
    const int64_t units = ceil_div(pb.N, pp.box_Tn[b]) * ext[a0] *
                          ceil_div(ext[a1], pp.box_T1[b]) * ceil_div(ext[a2], T2);
    if (units > INT32_MAX) return pp.status;
  }

  // pooled conv: window z = 4q + j reads input 2q + e, e = (j + p - d k)/2
  for (int a = 0; a < 3; ++a) {
    const int p = pb.pad[a], d = pb.dil[a];
    int emin = 1 << 30, emax = -(1 << 30);
    for (int j = 0; j < 4; ++j)
      for (int k = 0; k < pb.k[a]; ++k) {
        const int t = j + p - d * k;
        if (t % 2 == 0) {
          emin = std::min(emin, t / 2);
          emax = std::max(emax, t / 2);
        }
      }
    if (emin > emax || emin > 0) return pp.status;
    // offsets below e_min have no (j, k) pair: leading taps of weight 0 widen
    // the left padding until the conv formula yields all P windows
    while (conv_len(pb.S[a], emax - emin + 1, 2, -emin, 1) < bn.P[a] &&
           emax - emin + 1 < kMaxAxisTaps)
      --emin;
    if (emax - emin + 1 > kMaxAxisTaps) return pp.status;
    pp.e_min[a] = emin;
    pp.Ke[a] = emax - emin + 1;
  }
  Problem c;
  std::memset(&c, 0, sizeof(c));
  c.op = OP_CONV;
  c.N = pb.N;
  c.Cin = pb.Cin;
  c.Cout = pb.Cout;
  c.groups = 1;
  for (int a = 0; a < 3; ++a) {
    c.S[a] = pb.S[a];
    c.k[a] = pp.Ke[a];
    c.stride[a] = 2;
    c.pad[a] = -pp.e_min[a];
    c.dil[a] = 1;
    c.out_ext[a] = (int)bn.P[a];
  }
  pp.conv = c;
  if (make_plan(c, &pp.cplan) != TC3D_OK) return pp.status;

  if (pb.op == OP_CONVT_BN_POOL) plan_lag(bn, pp);

  // workspace: the pooled conv's packed weights first, then this path's own
  int64_t off = pp.cplan.ws_total;
  pp.ws_wpack_off = pp.cplan.ws_wpack_off;
  pp.ws_w2_off = off;
  // summed weights: [Cout][Cin][Ke] for the engine, or [Cin][3][3][3][Cout
  // padded to 16] for the pooled-conv kernel
  pp.ws_w2_bytes = std::max<int64_t>((int64_t)pb.Cout * pb.Cin * pp.Ke[0] * pp.Ke[1] * pp.Ke[2],
                                     (int64_t)pb.Cin * 27 * ((pb.Cout + 15) / 16 * 16)) *
                   4;
  off = round_up(off + pp.ws_w2_bytes, 256);
  // b2 [Cout], then (lag form) the pooled conv's scale [Cout], then the
  // pooled conv's item counter
  pp.ws_b2_off = off;
  off = round_up(off + (int64_t)pb.Cout * 8 + 16, 256);
  if (pb.op == OP_CONVT_BN_POOL) {
    pp.ws_gpart_off = off;
    pp.ws_gpart_bytes = (int64_t)kGramMaxCtas * kGramEntries * 4;
    off = round_up(off + pp.ws_gpart_bytes, 256);
    pp.ws_gsum_off = off;
    off = round_up(off + (int64_t)kGramMaxBoxes * kGramEntries * 8, 256);
    if (pp.lag) {
      pp.ws_lpart_off = off;
      pp.ws_lpart_bytes = (int64_t)pp.lag_grid * pp.lag_nbox * kLagSlots * 4;
      off = round_up(off + pp.ws_lpart_bytes, 256);
      pp.ws_lrs_off = off;
      off = round_up(off + (int64_t)pp.lag_nbox * kLagSlots * 4, 256);
    }
  }
  pp.ws_total = off;
  pp.status = TC3D_OK;
  return pp.status;
}

}  // namespace tc3d
