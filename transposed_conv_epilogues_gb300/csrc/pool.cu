// pool.cu -- the algebraic BN-pool path: patch Gram matrices, their
// reduction, and the per-channel finalize (see PoolPlan in plan.h).
#include "pool.cuh"

#include <cstring>

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

// entry i of class c's patch: (ci, tap t0, t1, t2) -> patch index d and weight
__device__ __forceinline__ void class_entry(const PoolFinParams& p, int c, int co, int i, int& d,
                                            float& wv) {
  const int r0 = p.cls_r[c][0], r1 = p.cls_r[c][1], r2 = p.cls_r[c][2];
  const int n0 = p.ntap[0][r0], n1 = p.ntap[1][r1], n2 = p.ntap[2][r2];
  const int t2 = i % n2, t1 = (i / n2) % n1, t0 = (i / (n1 * n2)) % n0, ci = i / (n0 * n1 * n2);
  d = ci * p.V + (p.tap_u[0][r0][t0] * p.nU[1] + p.tap_u[1][r1][t1]) * p.nU[2] +
      p.tap_u[2][r2][t2];
  const int k0 = p.tap_k[0][r0][t0], k1 = p.tap_k[1][r1][t1], k2 = p.tap_k[2][r2][t2];
  wv = __ldg(p.w + (((long long)ci * p.Cout + co) * p.k[0] + k0) * p.k[1] * p.k[2] +
             (long long)k1 * p.k[2] + k2);
}

__global__ void __launch_bounds__(256) pool_finalize_kernel(const __grid_constant__ PoolFinParams p) {
  const int co = blockIdx.x;
  __shared__ float s_scale;
  __shared__ int sd[8][kGramMaxD];
  __shared__ float sw[8][kGramMaxD];
  __shared__ int sne[8], soff[9];
  double s1 = 0.0, s2 = 0.0;
  if (p.gcls) {
    // class sums of the bias-free transposed conv: w_r . s_r and w_r^T G_r w_r
    // (G_r, s_r: the class's combined Gram); first every class's patch
    // entries (index, weight), then all (class, i, j) pairs in one loop
    if (threadIdx.x < 8) {
      const int c = threadIdx.x;
      sne[c] = c < p.ncls ? p.Cin * p.ntap[0][p.cls_r[c][0]] * p.ntap[1][p.cls_r[c][1]] *
                                p.ntap[2][p.cls_r[c][2]]
                          : 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      soff[0] = 0;
      for (int c = 0; c < 8; ++c) soff[c + 1] = soff[c] + sne[c] * sne[c];
    }
    for (int q = threadIdx.x; q < 8 * kGramMaxD; q += 256) {
      const int c = q / kGramMaxD, i = q % kGramMaxD;
      if (i < sne[c]) class_entry(p, c, co, i, sd[c][i], sw[c][i]);
    }
    __syncthreads();
    for (int q = threadIdx.x; q < soff[8]; q += 256) {
      int c = 0;
      while (q >= soff[c + 1]) ++c;
      const int ne = sne[c], i = (q - soff[c]) / ne, j = (q - soff[c]) % ne;
      const int di = sd[c][i], dj = sd[c][j];
      const int lo = (di >> 3) <= (dj >> 3) ? di : dj, hi = lo == di ? dj : di;
      const double* G = p.gcls + (size_t)c * kGramEntries;
      s2 += (double)sw[c][i] * (double)sw[c][j] * G[lo * kGramMaxD + hi];
      if (j == 0) s1 += (double)sw[c][i] * G[kGramMaxD * kGramMaxD + di];
    }
  }
  block_sum2_pool(s1, s2);
  if (threadIdx.x == 0) {
    const double g = p.gamma ? (double)p.gamma[co] : 1.0, be = p.beta ? (double)p.beta[co] : 0.0;
    double scale, shift;
    if (p.gcls) {
      // y = (pooled mean of t0 - mean of t0) * scale + beta  (the bias cancels)
      const double mean = s1 / p.count;
      double var = s2 / p.count - mean * mean;
      if (var < 0.0) var = 0.0;
      scale = g / sqrt(var + (double)p.eps);
      shift = be - mean * scale;
    } else {
      const double bv = p.bias ? (double)p.bias[co] : 0.0;
      scale = g / sqrt((double)p.rvar[co] + (double)p.eps);
      shift = be + (bv - (double)p.rmean[co]) * scale;
    }
    s_scale = (float)(scale / 64.0);
    p.b2[co] = (float)shift;
  }
  __syncthreads();
  // summed weights: W'[e] = sum of W[k] over taps k with 2(e_min + e) - p + d k in [0, 3]
  const int kv = p.Ke[0] * p.Ke[1] * p.Ke[2];
  for (int q = threadIdx.x; q < p.Cin * kv; q += 256) {
    const int ci = q / kv, e = q % kv;
    const int ee[3] = {e / (p.Ke[1] * p.Ke[2]), (e / p.Ke[2]) % p.Ke[1], e % p.Ke[2]};
    float acc = 0.f;
    for (int k0 = 0; k0 < p.k[0]; ++k0) {
      const int j0 = 2 * (p.e_min[0] + ee[0]) - p.pad[0] + p.dil[0] * k0;
      if (j0 < 0 || j0 > 3) continue;
      for (int k1 = 0; k1 < p.k[1]; ++k1) {
        const int j1 = 2 * (p.e_min[1] + ee[1]) - p.pad[1] + p.dil[1] * k1;
        if (j1 < 0 || j1 > 3) continue;
        for (int k2 = 0; k2 < p.k[2]; ++k2) {
          const int j2 = 2 * (p.e_min[2] + ee[2]) - p.pad[2] + p.dil[2] * k2;
          if (j2 < 0 || j2 > 3) continue;
          acc += __ldg(p.w + (((long long)ci * p.Cout + co) * p.k[0] + k0) * p.k[1] * p.k[2] +
                       (long long)k1 * p.k[2] + k2);
        }
      }
    }
    p.w2[((long long)co * p.Cin + ci) * kv + e] = acc * s_scale;
  }
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
  pool_finalize_kernel<<<p.Cout, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace tc3d
