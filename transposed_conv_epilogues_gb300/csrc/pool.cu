// pool.cu -- the algebraic BN-pool path: patch Gram matrices, their
// reduction, and the per-channel finalize (see PoolPlan in plan.h).
#include "pool.cuh"

#include <algorithm>
#include <climits>
#include <cstring>

#include "ptx.cuh"

namespace tc3d {

// ---------------------------------------------------------------------------
// Gram matrices.  Every CTA takes work units of one box (see GramParams): it
// stages the unit's slab of x in shared memory with 4-byte asynchronous
// copies (zero outside x), the next unit's slab in flight while the current
// one is used, and accumulates sum P P^T and sum P over the unit's rows.
// Entry d of P(m) is slab[base_d + t1 * W2p + t2] for the row's place (t1,
// t2) in the unit; W2p is 4 x an odd number.  Threads are block-major: the nthr = 32q threads of block
// blk own the 8x8 block blk of the Gram (upper triangle of 8-wide blocks),
// thread j of them the rows j, j + nthr, ... of every unit, so the lanes of
// a warp read one entry of 32 consecutive rows (distinct banks).  The CTA
// then adds its threads' sums in a fixed order and writes one partial slot.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp4_zfill(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
// 16-byte copy, the first `bytes` (0..16) from src and zeros after
__device__ __forceinline__ void cp16_zfill(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_prev() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}
// d = a * b + c on a pair of floats (packed f32x2 multiply-add, round to nearest)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

struct UnitGeo {
  int n, tn, m0, a1, a2, t1u, t2u;  // samples [n, n + tn); m0 along axis a0; tile starts a1, a2
};

// unit u of box b (units < 2^31: 32-bit arithmetic)
__device__ __forceinline__ UnitGeo unit_geo(const GramParams& p, int b, int A0, int A1, int A2,
                                            int u) {
  UnitGeo g;
  const int nt1 = p.box_nt1[b], nt2 = p.box_nt2[b];
  const int i2 = u % nt2;
  u /= nt2;
  const int i1 = u % nt1;
  u /= nt1;
  const int e0 = p.box_ext[b][A0];
  g.m0 = p.box_lo[b][A0] + u % e0;
  g.n = (u / e0) * p.box_Tn[b];
  g.tn = min(p.box_Tn[b], p.N - g.n);
  g.a1 = p.box_lo[b][A1] + i1 * p.box_T1[b];
  g.a2 = p.box_lo[b][A2] + i2 * p.box_T2[b];
  g.t1u = min(p.box_T1[b], p.box_lo[b][A1] + p.box_ext[b][A1] - g.a1);
  g.t2u = min(p.box_T2[b], p.box_lo[b][A2] + p.box_ext[b][A2] - g.a2);
  return g;
}

__global__ void __launch_bounds__(kGramMaxThreads, 1) gram_kernel(const __grid_constant__ GramParams p) {
  extern __shared__ __align__(16) float slab[];  // [2][kGramSlabFloats]
  __shared__ float red[kGramEntries];

  int b = 0;
  while (b + 1 < p.nbox && (int)blockIdx.x >= p.box_cta0[b + 1]) ++b;
  const int cta = (int)blockIdx.x - p.box_cta0[b];
  const int ncta = p.box_cta0[b + 1] - p.box_cta0[b];
  const int t = threadIdx.x, nthreads = blockDim.x;
  for (int e = t; e < kGramEntries; e += nthreads) red[e] = 0.f;

  const int A0 = p.box_perm[b][0], A1 = p.box_perm[b][1], A2 = p.box_perm[b][2];
  const int W1 = p.box_W1[b], W2p = p.box_W2p[b];
  const int nblk = p.nblk, nthr = nthreads / nblk;
  const int blk = t / nthr, j0 = t % nthr;
  int bi = 0, bj = 0;
  {
    int k = blk;
    for (bi = 0; bi < p.nb; ++bi) {
      const int cnt = p.nb - bi;
      if (k < cnt) {
        bj = bi + k;
        break;
      }
      k -= cnt;
    }
  }
  // slab offsets of this thread's 16 patch entries (entries >= D read word
  // 0 of the row: what they accumulate lands in Gram entries never read)
  const int Umin1 = p.U[A1][0], Umin2 = p.U[A2][0];
  auto slab_off = [&](int dd) {
    const int ci = dd / p.V, vi = dd % p.V;
    int ii[3];
    ii[2] = vi % p.nU[2];
    ii[1] = (vi / p.nU[2]) % p.nU[1];
    ii[0] = vi / (p.nU[1] * p.nU[2]);
    return ((ci * p.nU[A0] + ii[A0]) * W1 + p.U[A1][ii[A1]] - Umin1) * W2p + p.U[A2][ii[A2]] -
           Umin2;
  };
  // Carry along the slab's fast axis a2: when a2 has two consecutive offsets
  // and an entry's partner (the same entry one offset further along a2, d + sA2
  // in patch order) lies in the same 8-block, the entry at row t2 + 1 equals
  // its partner at row t2.  A thread then walks slab lines row by row and
  // loads only the partners.  Local order: pairs (entry, partner) at local
  // indices (2k, 2k + 1).
  const int sA2 = A2 == 2 ? 1 : A2 == 1 ? p.nU[2] : p.nU[1] * p.nU[2];
  const bool carry = p.nU[A2] == 2 && p.U[A2][1] == p.U[A2][0] + 1 && 8 % (2 * sA2) == 0;
  int la[8], lc[8];  // local index -> entry within the 8-block
  {
    int k = 0;
    for (int i = 0; i < 8; ++i) la[i] = i;
    if (carry)
      for (int i = 0; i < 8; ++i)
        if ((i % (2 * sA2)) < sA2) {
          la[2 * k] = i;
          la[2 * k + 1] = i + sA2;
          ++k;
        }
    for (int i = 0; i < 8; ++i) lc[i] = la[i];
  }
  int oa[8], oc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int da = 8 * bi + la[i], dc = 8 * bj + lc[i];
    oa[i] = da < p.D ? slab_off(da) : 0;
    oc[i] = dc < p.D ? slab_off(dc) : 0;
  }
  float2 acc[8][4];
  float sacc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    sacc[i] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[i][k] = make_float2(0.f, 0.f);
  }

  const int units = (int)p.box_units[b];
  const long long cstride = (long long)p.L[0] * p.L[1] * p.L[2];
  const long long xs0 = A0 == 0 ? (long long)p.L[1] * p.L[2] : A0 == 1 ? p.L[2] : 1;
  const long long xs1 = A1 == 0 ? (long long)p.L[1] * p.L[2] : A1 == 1 ? p.L[2] : 1;
  const long long xs2 = A2 == 0 ? (long long)p.L[1] * p.L[2] : A2 == 1 ? p.L[2] : 1;
  const int L0 = p.L[A0], L1 = p.L[A1], L2 = p.L[A2];
  const int nU0 = p.nU[A0];
  const int planes = p.C * nU0;
  const int SN = planes * W1 * W2p;  // slab floats per sample
  const int span1 = p.U[A1][p.nU[A1] - 1] - Umin1, span2 = p.U[A2][p.nU[A2] - 1] - Umin2;
  // stage the slab of unit u into buffer h: for every (sample, plane), the
  // warps take its rows y in turn, the lanes the z range
  const int warp = t >> 5, lane = t & 31, nwarps = nthreads >> 5;
  auto issue = [&](int h, int u) {
    const UnitGeo g = unit_geo(p, b, A0, A1, A2, u);
    const int w1 = g.t1u + span1, w2 = g.t2u + span2;
    const int z2s = g.a2 + Umin2;  // global start of every slab row along a2
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(slab + h * kGramSlabFloats);
    // 16-byte rows: lanes take (row rr of R, chunk c of nch)
    const bool v16 = p.vec16 && A2 == 2 && z2s >= 0 && (z2s & 3) == 0;
    const int nch = (w2 + 3) >> 2, R = v16 ? 32 / nch : 1;
    const int rr = lane / nch, cc = lane - rr * nch;
    int ci = 0, v0 = 0;
    for (int sp = 0; sp < g.tn * planes; ++sp) {
      const int nl = sp / planes;  // sample of this plane
      const int z0 = g.m0 + p.U[A0][v0];
      const bool pok = (unsigned)z0 < (unsigned)L0;
      const float* src_pl = p.x + ((long long)(g.n + nl) * p.C + ci) * cstride + z0 * xs0;
      const uint32_t dst_pl = base + 4u * (uint32_t)(nl * SN + (ci * nU0 + v0) * W1 * W2p);
      if (v16) {
        for (int y0 = warp * R; y0 < w1; y0 += nwarps * R) {
          const int y = y0 + rr;
          if (rr < R && y < w1) {
            const int z1 = g.a1 + Umin1 + y;
            const int z2 = z2s + 4 * cc;
            const int nval = (pok && (unsigned)z1 < (unsigned)L1) ? min(max(L2 - z2, 0), 4) : 0;
            cp16_zfill(dst_pl + 4u * (uint32_t)(y * W2p + 4 * cc),
                       nval ? (const void*)(src_pl + z1 * xs1 + z2) : (const void*)p.x, 4 * nval);
          }
        }
      } else {
        for (int y = warp; y < w1; y += nwarps) {
          const int z1 = g.a1 + Umin1 + y;
          const bool rok = pok && (unsigned)z1 < (unsigned)L1;
          const float* src_row = src_pl + z1 * xs1;
          const uint32_t dst_row = dst_pl + 4u * (uint32_t)(y * W2p);
          for (int z = lane; z < w2; z += 32) {
            const int z2 = z2s + z;
            const bool ok = rok && (unsigned)z2 < (unsigned)L2;
            cp4_zfill(dst_row + 4u * z, ok ? src_row + z2 * xs2 : p.x, ok);
          }
        }
      }
      if (++v0 == nU0) {
        v0 = 0;
        if (++ci == p.C) ci = 0;
      }
    }
  };

  int u = cta;
  if (u < units) issue(0, u);
  cp_commit();
  for (int it = 0; u < units; u += ncta, ++it) {
    const int cur = it & 1;
    const int nx = u + ncta;
    __syncthreads();  // the buffer of unit it-1 is consumed
    if (nx < units) issue(cur ^ 1, nx);
    cp_commit();
    cp_wait_prev();   // this thread's copies of unit it have landed
    __syncthreads();  // and everyone's
    {
      const UnitGeo g = unit_geo(p, b, A0, A1, A2, u);
      const float* sb = slab + cur * kGramSlabFloats;
      const bool diag = bi == bj;
      if (carry) {
        // lines (sample nl, t1): thread j0 takes lines j0, j0 + nthr, ...;
        // a line is walked from a rotated start t2s = (line / 8) % 4 to its
        // end and then from 0 to t2s, so that with the row stride 4 x odd the
        // 32 lanes of a warp read distinct banks
        for (int line = j0; line < g.tn * g.t1u; line += nthr) {
          const int nl = line / g.t1u, t1 = line - nl * g.t1u;
          const float* lb = sb + nl * SN + t1 * W2p;
          const int t2s = ((line >> 3) & 3) % g.t2u;
          for (int seg = 0; seg < 2; ++seg) {
            const int lo = seg ? 0 : t2s, hi = seg ? t2s : g.t2u;
            if (lo >= hi) continue;
            float a[8], c[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              a[i] = lb[oa[i] + lo];
              c[i] = diag ? a[i] : lb[oc[i] + lo];
            }
            for (int t2 = lo;;) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                if (diag) sacc[i] += a[i];
                const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  acc[i][k] = ffma2(ai, make_float2(c[2 * k], c[2 * k + 1]), acc[i][k]);
              }
              if (++t2 == hi) break;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                a[2 * k] = a[2 * k + 1];
                a[2 * k + 1] = lb[oa[2 * k + 1] + t2];
                c[2 * k] = c[2 * k + 1];
                c[2 * k + 1] = diag ? a[2 * k + 1] : lb[oc[2 * k + 1] + t2];
              }
            }
          }
        }
      } else {
        const int tt = g.t1u * g.t2u, nr = g.tn * tt;
        // row r = (sample nl, t1, t2), stepped by nthr with carries
        int nl = j0 / tt, t1 = (j0 % tt) / g.t2u, t2 = j0 % g.t2u;
        const int sn = nthr / tt, s1 = (nthr % tt) / g.t2u, s2 = nthr % g.t2u;
        for (int r = j0; r < nr; r += nthr) {
          const int ro = nl * SN + t1 * W2p + t2;
          float a[8], c[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            a[i] = sb[oa[i] + ro];
            c[i] = diag ? a[i] : sb[oc[i] + ro];
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (diag) sacc[i] += a[i];
            const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              acc[i][k] = ffma2(ai, make_float2(c[2 * k], c[2 * k + 1]), acc[i][k]);
          }
          t2 += s2;
          if (t2 >= g.t2u) {
            t2 -= g.t2u;
            ++t1;
          }
          t1 += s1;
          if (t1 >= g.t1u) {
            t1 -= g.t1u;
            ++nl;
          }
          nl += sn;
        }
      }
    }
  }
  // CTA sum in a fixed order: thread rows one after another
  for (int rs = 0; rs < nthr; ++rs) {
    __syncthreads();
    if (j0 == rs) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float* rrow = red + (8 * bi + la[i]) * kGramMaxD + 8 * bj;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          rrow[lc[2 * k]] += acc[i][k].x;
          rrow[lc[2 * k + 1]] += acc[i][k].y;
        }
        if (bi == bj) red[kGramMaxD * kGramMaxD + 8 * bi + la[i]] += sacc[i];
      }
    }
  }
  __syncthreads();
  for (int e = t; e < kGramEntries; e += nthreads)
    p.part[(size_t)blockIdx.x * kGramEntries + e] = red[e];
}

struct GramReduceParams {
  const float* part;
  double* gcls;  // [class][kGramEntries]
  int nbox, ncls;
  int box_cta0[kGramMaxBoxes + 1];
  int cls_coef[8][kGramMaxBoxes];
};

// grid ceil(kGramEntries / 8): 8 entries per CTA.  Thread (g, el) sums, per
// box, the slots i = g mod 32 of that box for entry el; the 32 group sums
// are then added in order, and every class takes its inclusion-exclusion
// combination of the boxes.
__global__ void __launch_bounds__(256) gram_reduce_kernel(const __grid_constant__ GramReduceParams p) {
  __shared__ double sh[32][kGramMaxBoxes][8];
  const int el = threadIdx.x & 7, g = threadIdx.x >> 3;
  const int e = blockIdx.x * 8 + el;
  for (int b = 0; b < p.nbox; ++b) {
    double s = 0.0;
    if (e < kGramEntries)
      for (int i = p.box_cta0[b] + g; i < p.box_cta0[b + 1]; i += 32)
        s += (double)p.part[(size_t)i * kGramEntries + e];
    sh[g][b][el] = s;
  }
  __syncthreads();
  if (g == 0 && e < kGramEntries) {
    double box[kGramMaxBoxes];
    for (int b = 0; b < p.nbox; ++b) {
      double tot = 0.0;
      for (int k = 0; k < 32; ++k) tot += sh[k][b][el];
      box[b] = tot;
    }
    for (int c = 0; c < p.ncls; ++c) {
      double v = 0.0;
      for (int b = 0; b < p.nbox; ++b)
        if (p.cls_coef[c][b]) v += p.cls_coef[c][b] * box[b];
      p.gcls[(size_t)c * kGramEntries + e] = v;
    }
  }
}

// ---------------------------------------------------------------------------
// Finalize: one CTA per output channel.
// ---------------------------------------------------------------------------
// Copies n ints of a table held in the kernel parameters into shared memory.
// Every lane of a warp reads the same element (one broadcast from the
// constant bank); reads whose index differs across a warp would be
// serialised, one constant-cache access per distinct address.
__device__ __forceinline__ void stage_param_ints(int* dst, const int* src, int n) {
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const bool lead = (threadIdx.x & 31) == 0;
#pragma unroll 4
  for (int r = warp; r < n; r += nw) {
    const int v = src[r];
    if (lead) dst[r] = v;
  }
}

__device__ __forceinline__ void block_sum2_pool(double& a, double& b) {
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

__global__ void __launch_bounds__(256) pool_finalize_kernel(const __grid_constant__ PoolFinParams p) {
  const int co = blockIdx.x;
  extern __shared__ float fin_smem[];  // this channel's weights [Cin][k0][k1][k2]
  __shared__ float s_scale;
  double s1 = 0.0, s2 = 0.0;
  const bool batch = p.gcls != nullptr;
  float* wsh = fin_smem;
  const int kvol = p.k[0] * p.k[1] * p.k[2];
  for (int e = threadIdx.x; e < p.Cin * kvol; e += 256) {
    const int ci = e / kvol, kk = e - ci * kvol;
    wsh[e] = __ldg(p.w + ((long long)ci * p.Cout + co) * kvol + kk);
  }
  // (a dependent is signalled only after this wait, so no later kernel of
  // the call runs ahead of work queued before the call)
  grid_dependency_wait();  // the statistics of the kernels before
  grid_launch_dependents();
  // the pooled conv reads its counter only after its wait on this kernel
  if (co == 0 && threadIdx.x == 0 && p.pool_ctr) *p.pool_ctr = 0u;
  __syncthreads();
  if (batch) {
    // class sums of the bias-free transposed conv: w_r . s_r and w_r^T G_r w_r
    // (G_r, s_r: the class's combined Gram).  Thread t takes row t of the
    // entries of all classes (entry i of class c) and its pairs (i, j).  The
    // entry tables are read from shared memory: indexing kernel parameters
    // with values that differ across a warp would serialise the reads.
    __shared__ int e_d[8 * kGramMaxD], e_w[8 * kGramMaxD], e_off[9];
    const int nrows = p.ent_off[p.ncls];
    stage_param_ints(e_d, p.ent_d, nrows);
    stage_param_ints(e_w, p.ent_w, nrows);
    stage_param_ints(e_off, p.ent_off, 9);
    __syncthreads();
    for (int row = threadIdx.x; row < nrows; row += 256) {
      int c = 0;
      while (row >= e_off[c + 1]) ++c;
      const int r0 = e_off[c], ne = e_off[c + 1] - r0;
      const int di = e_d[row];
      const float wi = wsh[e_w[row]];
      const double* G = p.gcls + (size_t)c * kGramEntries;
      s1 += (double)wi * G[kGramMaxD * kGramMaxD + di];
      for (int j = 0; j < ne; ++j) {
        const int dj = e_d[r0 + j];
        const int lo = (di >> 3) <= (dj >> 3) ? di : dj, hi = lo == di ? dj : di;
        s2 += (double)wi * (double)wsh[e_w[r0 + j]] * G[lo * kGramMaxD + hi];
      }
    }
  }
  block_sum2_pool(s1, s2);
  if (threadIdx.x == 0) {
    // the square root in float (fp64 square roots and divisions are slow on
    // this part); mean and variance in double
    const float g = p.gamma ? p.gamma[co] : 1.f, be = p.beta ? p.beta[co] : 0.f;
    float scale, shift;
    if (batch) {
      // y = (pooled mean of t0 - mean of t0) * scale + beta  (the bias cancels)
      const double mean = s1 * p.inv_count;
      double var = s2 * p.inv_count - mean * mean;
      if (var < 0.0) var = 0.0;
      scale = g * rsqrtf((float)var + p.eps);
      shift = be - (float)mean * scale;
    } else {
      const float bv = p.bias ? p.bias[co] : 0.f;
      scale = g * rsqrtf(p.rvar[co] + p.eps);
      shift = be + (bv - p.rmean[co]) * scale;
    }
    s_scale = scale * (1.0f / 64.0f);
    p.b2[co] = shift;
  }
  __syncthreads();
  // summed weights: W'[e] = sum of W[k] over taps k with 2(e_min + e) - p + d k
  // in [0, 3]; in the pooled-conv kernel's layout every axis has 3 taps (zero
  // past Ke) and channels are innermost
  const int K0 = p.pooled_layout ? 3 : p.Ke[0], K1 = p.pooled_layout ? 3 : p.Ke[1],
            K2 = p.pooled_layout ? 3 : p.Ke[2];
  const int kv = K0 * K1 * K2;
  __shared__ unsigned wkm[3 * kMaxAxisTaps];
  stage_param_ints(reinterpret_cast<int*>(wkm), reinterpret_cast<const int*>(&p.wkmask[0][0]),
                   3 * kMaxAxisTaps);
  __syncthreads();
  for (int q = threadIdx.x; q < p.Cin * kv; q += 256) {
    const int ci = q / kv, e = q % kv;
    const int ee[3] = {e / (K1 * K2), (e / K2) % K1, e % K2};
    float acc = 0.f;
    if (ee[0] < p.Ke[0] && ee[1] < p.Ke[1] && ee[2] < p.Ke[2]) {
      // taps k of each axis with 2 (e_min + e) - p + d k in [0, 3]
      const unsigned m0 = wkm[ee[0]], m1 = wkm[kMaxAxisTaps + ee[1]], m2 = wkm[2 * kMaxAxisTaps + ee[2]];
      for (unsigned a = m0; a; a &= a - 1)
        for (unsigned b = m1; b; b &= b - 1)
          for (unsigned c = m2; c; c &= c - 1)
            acc += wsh[ci * kvol + ((__ffs(a) - 1) * p.k[1] + (__ffs(b) - 1)) * p.k[2] + (__ffs(c) - 1)];
    }
    if (p.pooled_layout)
      p.w2[(long long)q * p.w2_stride + co] = acc * s_scale;
    else
      p.w2[((long long)co * p.Cin + ci) * kv + e] = acc * s_scale;
  }
}

// ---------------------------------------------------------------------------
// Lag form, batch statistics: the reduction of the lag kernel's per-CTA box
// sums and the finalize of each channel.
//   Per class c with entries i, j (rows r0 + i of the entry tables), the
//   statistics need G_c[i, j] for i <= j (G_c is symmetric: the box sum of
//   the factor earlier in patch order at lag v_later - v_earlier) and s_c[i],
//   the first-order sums: the "gather list", ntri pairs then the rows.
//   w^T G w = sum over i <= j of (i == j ? 1 : 2) w_i w_j G_ij, so a channel's
//   statistics are two dot products of the gathered values with per-channel
//   coefficients.
// Both kernels are small (128 threads, at most 32 registers) so that they
// share the SMs with the lag kernel, launched while it runs: everything that
// does not need the box sums (the tables from the kernel parameters, the
// gather list, the coefficients, the summed weights) is done then.  After
// their waits, on the call's critical path, each reaches L2 once with all of
// its loads in flight.
// ---------------------------------------------------------------------------
constexpr int kLfThreads = 128;
constexpr int kLfMaxRows = 8 * kGramMaxD;
constexpr int kLrEnt = 8;              // reduction: entries per step of a CTA
constexpr int kLrGroups = kLfThreads / kLrEnt;
constexpr int kLrBatch = 10;           // reduction loads in flight per thread
constexpr int kLcBatch = 8;            // channel: gather loads in flight per thread

// the entry tables in shared memory and the per-class offsets (pairs i <= j)
struct LagTabs {
  int e_d[kLfMaxRows], e_w[kLfMaxRows], e_cv[kLfMaxRows], e_box[kLfMaxRows];
  int e_off[9], toff[9];
};

__device__ void lag_stage_tabs(const PoolFinParams& p, LagTabs& t) {
  const int nrows = p.ent_off[p.ncls];
  stage_param_ints(t.e_d, p.ent_d, nrows);
  stage_param_ints(t.e_w, p.ent_w, nrows);
  stage_param_ints(t.e_cv, p.ent_cv, nrows);
  stage_param_ints(t.e_box, p.ent_box, nrows);
  stage_param_ints(t.e_off, p.ent_off, 9);
  if (threadIdx.x == 0) {
    t.toff[0] = 0;
    for (int c = 0; c < p.ncls; ++c) {
      const int ne = p.ent_off[c + 1] - p.ent_off[c];
      t.toff[c + 1] = t.toff[c] + ne * (ne + 1) / 2;
    }
  }
}

// item q of the gather list: its index into the box sums, and its class
// rows (i, j; i == j == -1 - row for a first-order sum)
__device__ __forceinline__ int lag_gather_item(const PoolFinParams& p, const LagTabs& t, int ntri,
                                               int q, int& ri, int& rj) {
  if (q >= ntri) {
    const int row = q - ntri;
    ri = rj = -1 - row;
    return t.e_box[row] * kLagSlots + (t.e_cv[row] & 15);
  }
  int c = 0;
  while (q >= t.toff[c + 1]) ++c;
  const int r0 = t.e_off[c], ne = t.e_off[c + 1] - r0;
  int l = q - t.toff[c], i = 0;
  while (l >= ne - i) {  // row i of the upper triangle holds ne - i pairs
    l -= ne - i;
    ++i;
  }
  const int j = i + l;
  ri = r0 + i;
  rj = r0 + j;
  const int first = t.e_d[ri] <= t.e_d[rj] ? ri : rj, second = first == ri ? rj : ri;
  const int ca = t.e_cv[first], cb = t.e_cv[second];
  const int jl = 9 * (((cb >> 4) & 15) - ((ca >> 4) & 15) + 1) +
                 3 * (((cb >> 8) & 15) - ((ca >> 8) & 15) + 1) +
                 (((cb >> 12) & 15) - ((ca >> 12) & 15) + 1);
  return t.e_box[first] * kLagSlots + lag_slot(p.Cin, ca & 15, cb & 15, jl);
}

// summed weights (ci, e) of channel co, times sc; wc: the channel's weights
// [Cin][k0][k1][k2]
__device__ __forceinline__ void lag_fold_channel(const PoolFinParams& p, const float* wc,
                                                 const unsigned* wkm, int co, float sc) {
  const int kvol = p.k[0] * p.k[1] * p.k[2];
  const int K0 = p.pooled_layout ? 3 : p.Ke[0], K1 = p.pooled_layout ? 3 : p.Ke[1],
            K2 = p.pooled_layout ? 3 : p.Ke[2];
  const int kv = K0 * K1 * K2;
  for (int q = threadIdx.x; q < p.Cin * kv; q += kLfThreads) {
    const int ci = q / kv, e = q - ci * kv;
    const int ee[3] = {e / (K1 * K2), (e / K2) % K1, e % K2};
    float acc = 0.f;
    if (ee[0] < p.Ke[0] && ee[1] < p.Ke[1] && ee[2] < p.Ke[2]) {
      // taps k of each axis with 2 (e_min + e) - p + d k in [0, 3]
      const unsigned m0 = wkm[ee[0]], m1 = wkm[kMaxAxisTaps + ee[1]], m2 = wkm[2 * kMaxAxisTaps + ee[2]];
      const float* w = wc + ci * kvol;
      for (unsigned a = m0; a; a &= a - 1)
        for (unsigned b = m1; b; b &= b - 1)
          for (unsigned cc = m2; cc; cc &= cc - 1)
            acc += w[((__ffs(a) - 1) * p.k[1] + (__ffs(b) - 1)) * p.k[2] + (__ffs(cc) - 1)];
    }
    if (p.pooled_layout)
      p.w2[(long long)q * p.w2_stride + co] = acc * sc;
    else
      p.w2[((long long)co * p.Cin + ci) * kv + e] = acc * sc;
  }
}

// Reduction: rs[e] = sum over the lag kernel's CTAs of part[cta][e] for the
// entries e the gather list reads.  Before the wait every CTA builds the
// list of those entries (flags, then a block scan), in ascending order; after
// it, a CTA takes 8 entries per step, thread (g, k) adding the CTAs g, g + 16,
// ... of entry k in fp32 and the 16 slice sums added in a fixed pairwise
// order (the partial sums are box sums of one CTA each; the total stays
// within a few units of the fp32 rounding).
__global__ void __launch_bounds__(kLfThreads, 16) lag_reduce_kernel(const __grid_constant__ PoolFinParams p,
                                                                   const float* __restrict__ part,
                                                                   int ctas, int nent) {
  extern __shared__ int lr_smem[];  // [nent] flags, then the list of needed entries
  __shared__ LagTabs t;
  __shared__ int wsum[kLfThreads / 32], nneed;
  __shared__ float sh[kLrGroups][kLrEnt];
  int* flag = lr_smem;
  int* list = lr_smem + nent;
  // the kernels of the call before this one do not write p.lrs, and the
  // following one reads it only after its own wait
  grid_launch_dependents();
  lag_stage_tabs(p, t);
  for (int e = threadIdx.x; e < nent; e += kLfThreads) flag[e] = 0;
  __syncthreads();
  const int nrows = t.e_off[p.ncls], ntri = t.toff[p.ncls];
  for (int q = threadIdx.x; q < ntri + nrows; q += kLfThreads) {
    int ri, rj;
    flag[lag_gather_item(p, t, ntri, q, ri, rj)] = 1;
  }
  __syncthreads();
  // block scan of the flags over contiguous chunks of the entries
  const int per = (nent + kLfThreads - 1) / kLfThreads;
  const int e0 = threadIdx.x * per, e1 = min(nent, e0 + per);
  int cnt = 0;
  for (int e = e0; e < e1; ++e) cnt += flag[e];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int base = incl - cnt;
  for (int w = 0; w < warp; ++w) base += wsum[w];
  if (threadIdx.x == kLfThreads - 1) nneed = base + cnt;
  for (int e = e0; e < e1; ++e)
    if (flag[e]) list[base++] = e;
  __syncthreads();

  grid_dependency_wait();  // the lag kernel's partial sums
  const int k = threadIdx.x % kLrEnt, g = threadIdx.x / kLrEnt;
  for (int s0 = blockIdx.x * kLrEnt; s0 < nneed; s0 += gridDim.x * kLrEnt) {
    const int s = s0 + k;
    const int e = s < nneed ? list[s] : 0;
    float v = 0.f;
    if (s < nneed) {
      for (int i0 = g; i0 < ctas; i0 += kLrGroups * kLrBatch) {
        float r[kLrBatch];
#pragma unroll
        for (int u = 0; u < kLrBatch; ++u) {
          const int i = i0 + kLrGroups * u;
          r[u] = i < ctas ? part[(size_t)i * nent + e] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kLrBatch; ++u) v += r[u];
      }
    }
    sh[g][k] = v;
    __syncthreads();
    if (g == 0 && s < nneed) {
      float a[kLrGroups];
#pragma unroll
      for (int u = 0; u < kLrGroups; ++u) a[u] = sh[u][k];
#pragma unroll
      for (int w = kLrGroups / 2; w > 0; w >>= 1)
#pragma unroll
        for (int u = 0; u < w; ++u) a[u] += a[u + w];
      const_cast<float*>(p.lrs)[e] = a[0];
    }
    __syncthreads();
  }
}

// Finalize of channel co = blockIdx.x: before the wait, the gather list and
// the channel's coefficients (and, with the pooled layout, its unscaled
// summed weights: the pooled conv applies scale / 64 in its epilogue);
// after it, the gather and the two dot products, mean and biased variance,
// the BatchNorm affine; for the engine's layout also the summed weights with
// scale / 64 folded in.
__global__ void __launch_bounds__(kLfThreads, 16) lag_channel_kernel(const __grid_constant__ PoolFinParams p) {
  extern __shared__ float lc_smem[];
  __shared__ LagTabs t;
  __shared__ unsigned wkm[3 * kMaxAxisTaps];
  __shared__ float red[2][kLfThreads / 32];
  __shared__ float s_sc;
  const int co = blockIdx.x;
  const int kvol = p.k[0] * p.k[1] * p.k[2];
  const int wpc = p.Cin * kvol;  // weights of the channel
  float* wc = lc_smem;           // [Cin][kvol]
  // the pooled conv reads w2, s2, b2 and its counter only after its wait on
  // this kernel
  grid_launch_dependents();
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.pool_ctr) *p.pool_ctr = 0u;
  for (int e = threadIdx.x; e < wpc; e += kLfThreads) {
    const int ci = e / kvol, kk = e - ci * kvol;
    wc[e] = __ldg(p.w + ((long long)ci * p.Cout + co) * kvol + kk);
  }
  lag_stage_tabs(p, t);
  stage_param_ints(reinterpret_cast<int*>(wkm), reinterpret_cast<const int*>(&p.wkmask[0][0]),
                   3 * kMaxAxisTaps);
  __syncthreads();
  const int nrows = t.e_off[p.ncls], ntri = t.toff[p.ncls], ngat = ntri + nrows;
  int* gidx = reinterpret_cast<int*>(wc + wpc);      // [ngat]
  float* coef = reinterpret_cast<float*>(gidx + ngat);  // [ngat]
  for (int q = threadIdx.x; q < ngat; q += kLfThreads) {
    int ri, rj;
    gidx[q] = lag_gather_item(p, t, ntri, q, ri, rj);
    if (ri < 0)
      coef[q] = wc[t.e_w[-1 - ri]];
    else
      coef[q] = wc[t.e_w[ri]] * wc[t.e_w[rj]] * (ri == rj ? 1.f : 2.f);
  }
  const bool unscaled = p.s2 != nullptr;
  if (unscaled) lag_fold_channel(p, wc, wkm, co, 1.f);
  __syncthreads();

  grid_dependency_wait();  // the box sums
  float f1 = 0.f, f2 = 0.f;
  for (int q0 = threadIdx.x; q0 < ngat; q0 += kLfThreads * kLcBatch) {
    float v[kLcBatch];
#pragma unroll
    for (int u = 0; u < kLcBatch; ++u) {
      const int q = q0 + kLfThreads * u;
      v[u] = q < ngat ? __ldcg(p.lrs + gidx[q]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kLcBatch; ++u) {
      const int q = q0 + kLfThreads * u;
      if (q < ntri)
        f2 = fmaf(coef[q], v[u], f2);
      else if (q < ngat)
        f1 = fmaf(coef[q], v[u], f1);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    f1 += __shfl_xor_sync(0xffffffffu, f1, o);
    f2 += __shfl_xor_sync(0xffffffffu, f2, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = f1;
    red[1][threadIdx.x >> 5] = f2;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const float t1 = (red[0][0] + red[0][1]) + (red[0][2] + red[0][3]);
    const float t2 = (red[1][0] + red[1][1]) + (red[1][2] + red[1][3]);
    // y = (pooled mean of t0 - mean of t0) * scale + beta (the bias
    // cancels); the square root in float
    const double mean = (double)t1 * p.inv_count;
    double var = (double)t2 * p.inv_count - mean * mean;
    if (var < 0.0) var = 0.0;
    const float scale = (p.gamma ? p.gamma[co] : 1.f) * rsqrtf((float)var + p.eps);
    s_sc = scale * (1.0f / 64.0f);
    if (unscaled) p.s2[co] = scale * (1.0f / 64.0f);
    p.b2[co] = (p.beta ? p.beta[co] : 0.f) - (float)mean * scale;
  }
  if (!unscaled) {
    __syncthreads();
    lag_fold_channel(p, wc, wkm, co, s_sc);
  }
}

cudaError_t lag_finalize_launch(const PoolFinParams& p, const float* part, int ctas, int nent,
                                cudaStream_t st) {
  const int nrows = p.ent_off[p.ncls];
  int ntri = 0;
  for (int c = 0; c < p.ncls; ++c) {
    const int ne = p.ent_off[c + 1] - p.ent_off[c];
    ntri += ne * (ne + 1) / 2;
  }
  const size_t smem_r = (size_t)lag_reduce_smem_ints(nent) * 4;
  const size_t smem_c =
      (size_t)lag_channel_smem_floats(p.Cin, p.k[0] * p.k[1] * p.k[2], nrows, ntri) * 4;
  // both kernels share SMs with the lag kernel, whose shared-memory carveout
  // is the largest: an SM holds CTAs of one carveout at a time
  for (const void* f : {(const void*)lag_reduce_kernel, (const void*)lag_channel_kernel}) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                               (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  if (smem_r > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(lag_reduce_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_r);
    if (e != cudaSuccess) return e;
  }
  if (smem_c > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(lag_channel_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_c);
    if (e != cudaSuccess) return e;
  }
  // reduction CTAs: a step of 8 entries each for at most every gathered value
  // (the needed entries are at most that many)
  const int steps = (ntri + nrows + kLrEnt - 1) / kLrEnt;
  const cudaError_t e = launch_dependent(lag_reduce_kernel, dim3(std::min(steps, 96)),
                                         dim3(kLfThreads), smem_r, st, p, part, ctas, nent);
  if (e != cudaSuccess) return e;
  return launch_dependent(lag_channel_kernel, dim3(p.Cout), dim3(kLfThreads), smem_c, st, p);
}

// ---------------------------------------------------------------------------
// Pooled convolution on CUDA cores: y[n, co, q] = s2[co] (sum over ci and e
// of w2[ci, e, co] x[n, ci, 2 q + e - pad]) + b2[co] (stride 2, 3 taps per
// axis with zero weights past Ke, at most 4 input channels).  An item is
// (sample n, q0, 4 rows of q1, 16 of q2) for all channels, one warp per 16
// channels.  CTAs are persistent: the weights come in once by a bulk copy,
// the items' input boxes (36 columns x 9 rows x 3 planes x Cin, zero outside
// x; the x start rounded down to 16 bytes, so each row starts `shift`
// columns in) by TMA into two buffers, the next item's box landing while the
// current one is used.  A CTA's first two items are blockIdx.x and
// blockIdx.x + gridDim.x; the later ones come from a counter (zeroed by the
// finalize before this kernel), so CTAs that finish early take more.
// Lane (g, q2) computes the 4 rows of its q2 for 8 channels: per (ci, e0,
// e2) it reads the 9 inputs of its column (lanes read consecutive even
// columns: distinct banks; both halves of the warp read the same ones) and,
// per e1, 8 weights (two 16-byte broadcasts), 32 multiply-adds as 16 packed
// f32x2 ones (channel pairs).
// ---------------------------------------------------------------------------
constexpr int kPooledKe = 3;
constexpr int kPooledBoxFloats = kPooledBoxCols * kPooledBoxRows * kPooledKe;  // per channel

size_t pooled_smem_bytes(int Cin, int coutp) {
  const size_t box = ((size_t)Cin * kPooledBoxFloats * 4 + 127) / 128 * 128;
  const size_t wb = (size_t)Cin * 27 * coutp * 4;
  return 128 + 2 * box + wb + 64;
}

__device__ __forceinline__ void pooled_issue(const PooledParams& p, uint32_t dst, uint32_t bar,
                                             int item, uint32_t box_bytes) {
  const int per = p.nq1b * p.nq2b;
  const int s = item / per, r = item - s * per;
  const int n = s / p.P[0], q0 = s - n * p.P[0];
  const int q1b = r / p.nq2b, q2b = r - q1b * p.nq2b;
  mbar_arrive_expect_tx(bar, box_bytes);
  tma_load_5d(dst, &p.xmap, (2 * q2b * kPooledQ2 - p.pad[2]) & ~3, 2 * q1b * kPooledRows - p.pad[1],
              2 * q0 - p.pad[0], 0, n, bar);
}

__global__ void __launch_bounds__(128) pooled_conv_kernel(const __grid_constant__ PooledParams p) {
  extern __shared__ __align__(128) uint8_t pooled_raw[];
  __shared__ int s_item[2];  // the item of each box buffer (>= items: none)
  __shared__ float s_sc[kPooledMaxCout], s_bb[kPooledMaxCout];
  uint8_t* base = pooled_raw + ((128u - (smem_u32(pooled_raw) & 127u)) & 127u);
  const uint32_t box_bytes = (uint32_t)(p.Cin * kPooledBoxFloats * 4);
  const uint32_t box_stride = (box_bytes + 127u) / 128u * 128u;
  const float* xsb = reinterpret_cast<const float*>(base);
  const float* ws = reinterpret_cast<const float*>(base + 2 * box_stride);
  const uint32_t wbytes = (uint32_t)(p.Cin * 27 * p.coutp * 4);
  const uint32_t bar0 = smem_u32(base + 2 * box_stride + wbytes);  // boxes: bar0, bar0 + 8; weights: + 16
  const int items = p.nq1b * p.nq2b * p.N * p.P[0];
  if (threadIdx.x == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    mbar_init(bar0 + 16, 1);
    fence_barrier_init();
    for (int t = 0; t < 2; ++t) {
      const int it = (int)blockIdx.x + t * (int)gridDim.x;
      s_item[t] = it;
      if (it < items) pooled_issue(p, smem_u32(base) + t * box_stride, bar0 + 8u * t, it, box_bytes);
    }
    grid_dependency_wait();  // the summed weights, scales and bias of the finalize
    mbar_arrive_expect_tx(bar0 + 16, wbytes);
    bulk_g2s(smem_u32(ws), p.w2, wbytes, bar0 + 16);
  }
  grid_dependency_wait();
  for (int c = threadIdx.x; c < p.Cout; c += blockDim.x) {
    s_sc[c] = p.s2 ? p.s2[c] : 1.f;
    s_bb[c] = p.b2 ? p.b2[c] : 0.f;
  }
  __syncthreads();
  // every thread takes the same branch on a wait's outcome (the loop holds a
  // CTA barrier)
  bool ok = __syncthreads_and(mbar_wait(bar0 + 16, 0, p.timeout_cycles, nullptr));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q2l = lane & 15, g = lane >> 4;
  const int co0 = 16 * warp + 8 * g;
  const long long pv = (long long)p.P[0] * p.P[1] * p.P[2];
  const int per = p.nq1b * p.nq2b;
  uint32_t ph = 0;  // bit k: phase of box buffer k
  for (int t = 0; ok; ++t) {
    const int buf = t & 1;
    const int item = s_item[buf];
    if (item >= items) break;
    ok = __syncthreads_and(mbar_wait(bar0 + 8u * buf, (ph >> buf) & 1u, p.timeout_cycles, nullptr));
    if (!ok) break;
    ph ^= 1u << buf;
    const int s = item / per, r = item - s * per;
    const int n = s / p.P[0], q0 = s - n * p.P[0];
    const int q1b = r / p.nq2b, q2b = r - q1b * p.nq2b;
    const int q1a = q1b * kPooledRows, q2a = q2b * kPooledQ2;
    const int xc = 2 * q2a - p.pad[2];
    const int shift = xc - (xc & ~3);
    const float* xs = xsb + buf * (box_stride / 4);
    // channel pairs (2 h, 2 h + 1) in one packed f32x2 accumulator
    float2 acc[kPooledRows][4];
#pragma unroll
    for (int i = 0; i < kPooledRows; ++i)
#pragma unroll
      for (int h = 0; h < 4; ++h) acc[i][h] = make_float2(0.f, 0.f);
    for (int ci = 0; ci < p.Cin; ++ci) {
#pragma unroll
      for (int e0 = 0; e0 < kPooledKe; ++e0)
#pragma unroll
        for (int e2 = 0; e2 < kPooledKe; ++e2) {
          const float* col =
              xs + ((ci * kPooledKe + e0) * kPooledBoxRows) * kPooledBoxCols + shift + 2 * q2l + e2;
          float v[kPooledBoxRows];
#pragma unroll
          for (int j = 0; j < kPooledBoxRows; ++j) v[j] = col[j * kPooledBoxCols];
#pragma unroll
          for (int e1 = 0; e1 < kPooledKe; ++e1) {
            const float* wr =
                ws + (((ci * kPooledKe + e0) * kPooledKe + e1) * kPooledKe + e2) * p.coutp + co0;
            const float4 wa = *reinterpret_cast<const float4*>(wr);
            const float4 wb = *reinterpret_cast<const float4*>(wr + 4);
            const float2 w4[4] = {make_float2(wa.x, wa.y), make_float2(wa.z, wa.w),
                                  make_float2(wb.x, wb.y), make_float2(wb.z, wb.w)};
#pragma unroll
            for (int i = 0; i < kPooledRows; ++i) {
              const float2 xv = make_float2(v[2 * i + e1], v[2 * i + e1]);
#pragma unroll
              for (int h = 0; h < 4; ++h) acc[i][h] = __ffma2_rn(xv, w4[h], acc[i][h]);
            }
          }
        }
    }
    // this item's box is read: the CTA's next item may land in it
    __syncthreads();
    if (threadIdx.x == 0) {
      const int nx = p.ctr ? 2 * (int)gridDim.x + (int)atomicAdd(p.ctr, 1u) : item + 2 * (int)gridDim.x;
      s_item[buf] = nx;
      if (nx < items) pooled_issue(p, smem_u32(base) + buf * box_stride, bar0 + 8u * buf, nx, box_bytes);
    }
    const int q2 = q2a + q2l;
    if (q2 < p.P[2]) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int co = co0 + c;
        if (co >= p.Cout) break;
        const float bb = s_bb[co], sc = s_sc[co];
        float* yo = p.y + ((long long)n * p.Cout + co) * pv + (long long)q0 * p.P[1] * p.P[2] + q2;
#pragma unroll
        for (int i = 0; i < kPooledRows; ++i)
          if (q1a + i < p.P[1])
            yo[(long long)(q1a + i) * p.P[2]] = fmaf(c & 1 ? acc[i][c >> 1].y : acc[i][c >> 1].x, sc, bb);
      }
    }
  }
  if (!ok && threadIdx.x == 0) {
    // a wait ran out: flag it; the boxes still in flight land before the CTA
    // leaves (buffer k holds one iff its item is valid: a box is issued for
    // every valid item and not yet waited for)
    atomicExch(p.err, 1);
    for (int k = 0; k < 2; ++k)
      if (s_item[k] < items) mbar_wait(bar0 + 8u * k, (ph >> k) & 1u, p.timeout_cycles, nullptr);
  }
}

bool pooled_ok(int Cin, int Cout, const int Ke[3], const int P[3], int N) {
  if (Cin < 1 || Cin > kPooledMaxCin || Cout < 1 || Cout > kPooledMaxCout) return false;
  for (int a = 0; a < 3; ++a)
    if (Ke[a] < 1 || Ke[a] > kPooledKe || P[a] < 1) return false;
  const long long nq1b = (P[1] + kPooledRows - 1) / kPooledRows;
  const long long nq2b = (P[2] + kPooledQ2 - 1) / kPooledQ2;
  // (item numbers, the counter's included, stay far below 2^31)
  return nq1b * nq2b * N * P[0] <= INT32_MAX / 2 &&
         pooled_smem_bytes(Cin, pooled_coutp(Cout)) <= 100 * 1024;
}

cudaError_t pooled_launch(const PooledParams& p, int sm_count, cudaStream_t st) {
  const long long items = (long long)p.nq1b * p.nq2b * p.N * p.P[0];
  const size_t smem = pooled_smem_bytes(p.Cin, p.coutp);
  const int threads = 32 * (p.coutp / 16);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(pooled_conv_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // the largest carveout, as the finalize CTAs it joins on the SMs
  {
    const cudaError_t e = cudaFuncSetAttribute(pooled_conv_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                               (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  // persistent CTAs: as many as fit on the SMs at once
  int per_sm = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pooled_conv_kernel,
                                                                      threads, smem);
  if (e != cudaSuccess) return e;
  const long long want = items;
  const unsigned grid = (unsigned)std::max<long long>(
      1, std::min<long long>(want, (long long)std::max(per_sm, 1) * sm_count));
  return launch_dependent(pooled_conv_kernel, dim3(grid), dim3(threads), smem, st, p);
}

constexpr size_t kGramSmem = 2 * kGramSlabFloats * sizeof(float);

cudaError_t gram_set_smem() {
  return cudaFuncSetAttribute(gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kGramSmem);
}

cudaError_t gram_launch(const GramParams& p, unsigned ctas, cudaStream_t st) {
  gram_kernel<<<ctas, gram_threads(p.nblk), kGramSmem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t gram_reduce_launch(const float* part, const int* box_cta0_host, int nbox,
                               const int (*cls_coef)[kGramMaxBoxes], int ncls, double* gcls,
                               cudaStream_t st) {
  GramReduceParams rp;
  std::memset(&rp, 0, sizeof(rp));
  rp.part = part;
  rp.gcls = gcls;
  rp.nbox = nbox;
  rp.ncls = ncls;
  for (int i = 0; i <= nbox; ++i) rp.box_cta0[i] = box_cta0_host[i];
  for (int c = 0; c < ncls; ++c)
    for (int b = 0; b < nbox; ++b) rp.cls_coef[c][b] = cls_coef[c][b];
  gram_reduce_kernel<<<(kGramEntries + 7) / 8, 256, 0, st>>>(rp);
  return cudaGetLastError();
}

cudaError_t pool_finalize_launch(const PoolFinParams& p, cudaStream_t st) {
  const size_t smem = (((size_t)p.Cin * p.k[0] * p.k[1] * p.k[2] + 3) & ~(size_t)3) * 4;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(pool_finalize_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  pool_finalize_kernel<<<p.Cout, 256, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace tc3d
