// direct.cu -- direct fp32 convolution for grouped / depthwise convs with few
// channels per group, in NCDHW or NDHWC, and the layout transpose used around
// the engine for channels-last input.
//
// The sum is the direct-convolution formula of the page "Kimi-K2.6 l1_p59"
// with its group rule (output channel oc reads the input channels of group
// oc / (Cout/G)): y[n,oc,o] = bias[oc] + sum_{ci,k} w[oc,ci,k] *
// x[n, g*cin_g + ci, o*s - p + d*k], zero outside x.
#include "direct.cuh"

#include <algorithm>
#include <cstdint>

namespace tc3d {

// One work item = (n, oc, o0, o1, run of kDirectRun outputs along axis 2).
// Items are ordered so that consecutive threads touch consecutive memory:
// NCDHW runs along axis 2 fastest, NDHWC output channels fastest.
template <bool NDHWC, int S2, int D2>
__global__ void __launch_bounds__(256) direct_conv_kernel(const __grid_constant__ DirectParams p) {
  constexpr int R = kDirectRun;
  constexpr int SEG = (R - 1) * S2 + (kDirectMaxK2 - 1) * D2 + 1;  // input row segment
  const long long plane = (long long)p.S[1] * p.S[2];
  const long long xvol = (long long)p.S[0] * plane;
  const long long ovol = (long long)p.O[0] * p.O[1] * p.O[2];
  const int kv = p.k[0] * p.k[1] * p.k[2];
  const int k2n = p.k[2];
  const int seglen = (R - 1) * S2 + (k2n - 1) * D2 + 1;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < p.items;
       it += (long long)gridDim.x * blockDim.x) {
    long long q = it;
    int oc, r2, o1, o0, n;
    if (NDHWC) {
      oc = (int)(q % p.Cout);
      q /= p.Cout;
      r2 = (int)(q % p.nrun2);
      q /= p.nrun2;
      o1 = (int)(q % p.O[1]);
      q /= p.O[1];
      o0 = (int)(q % p.O[0]);
      n = (int)(q / p.O[0]);
    } else {
      r2 = (int)(q % p.nrun2);
      q /= p.nrun2;
      o1 = (int)(q % p.O[1]);
      q /= p.O[1];
      o0 = (int)(q % p.O[0]);
      q /= p.O[0];
      oc = (int)(q % p.Cout);
      n = (int)(q / p.Cout);
    }
    const int ic0 = (oc / p.cout_g) * p.cin_g;
    const int o2s = r2 * R;
    const float bv = p.bias ? __ldg(p.bias + oc) : 0.f;
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = bv;
    const int x2s = o2s * S2 - p.p[2];  // input index of segment element 0
    const float* wo = p.w + (long long)oc * p.cin_g * kv;
    for (int ci = 0; ci < p.cin_g; ++ci) {
      const int ic = ic0 + ci;
      for (int k0 = 0; k0 < p.k[0]; ++k0) {
        const int z = o0 * p.s[0] - p.p[0] + k0 * p.d[0];
        if ((unsigned)z >= (unsigned)p.S[0]) continue;
        for (int k1 = 0; k1 < p.k[1]; ++k1) {
          const int yy = o1 * p.s[1] - p.p[1] + k1 * p.d[1];
          if ((unsigned)yy >= (unsigned)p.S[1]) continue;
          // the input row segment this run needs, zero outside x
          float seg[SEG];
          if (NDHWC) {
            const float* row = p.x + (((long long)n * p.S[0] + z) * p.S[1] + yy) * p.S[2] * p.C + ic;
#pragma unroll
            for (int j = 0; j < SEG; ++j) {
              const int xi = x2s + j;
              seg[j] = (j < seglen && (unsigned)xi < (unsigned)p.S[2])
                           ? __ldg(row + (long long)xi * p.C)
                           : 0.f;
            }
          } else {
            const float* row =
                p.x + ((long long)n * p.C + ic) * xvol + (long long)z * plane + (long long)yy * p.S[2];
#pragma unroll
            for (int j = 0; j < SEG; ++j) {
              const int xi = x2s + j;
              seg[j] = (j < seglen && (unsigned)xi < (unsigned)p.S[2]) ? __ldg(row + xi) : 0.f;
            }
          }
          const float* wk = wo + ((long long)ci * p.k[0] + k0) * p.k[1] * p.k[2] + k1 * p.k[2];
#pragma unroll
          for (int k2 = 0; k2 < kDirectMaxK2; ++k2) {
            if (k2 < k2n) {
              const float wv = __ldg(wk + k2);
#pragma unroll
              for (int r = 0; r < R; ++r) acc[r] = fmaf(wv, seg[r * S2 + k2 * D2], acc[r]);
            }
          }
        }
      }
    }
    if (NDHWC) {
      float* yo = p.y + (((long long)n * p.O[0] + o0) * p.O[1] + o1) * p.O[2] * p.Cout + oc;
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (o2s + r < p.O[2]) yo[(long long)(o2s + r) * p.Cout] = acc[r];
    } else {
      float* yo = p.y + ((long long)n * p.Cout + oc) * ovol + ((long long)o0 * p.O[1] + o1) * p.O[2];
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (o2s + r < p.O[2]) yo[o2s + r] = acc[r];
    }
  }
}

__device__ __forceinline__ void cp4z(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp16z(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ void cp_commit_direct() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_wait_prev_direct() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// Tiled NCDHW form for one input channel per group (depthwise convs and
// channel multipliers), stride and dilation 1 along axis 0.  CTA = (y tile,
// x tile) x (chunk of output planes o0) x (n, group); thread (tx, ty) owns
// outputs x in [x0 + 4 tx, +4), y in [y0 + 4 ty, +4).  The CTA walks its
// output planes keeping a ring of k0 + 1 input planes (W1 rows x W2p
// columns each) in shared memory: the plane the next output plane adds is
// copied while the current one is computed.  Per input plane row a thread
// loads one register segment (16-byte loads) that feeds all 4 x outputs of
// every output row reading it (rows are shared across the 4 y outputs when
// stride and dilation along y are 1).
// K3: 0 for any kernel extent (runtime bounds), or 3 for a 3 x 3 (y, x)
// filter with stride and dilation 1 along y, fully unrolled: the tap
// weights of a plane in registers, taps outermost so that the 16
// accumulators of a thread interleave.
template <int S2, int D2, int K3>
__global__ void __launch_bounds__(128) direct_tiled_kernel(const __grid_constant__ DirectParams p,
                                                           int W1, int W2p, int chunk) {
  constexpr int R = kDirectRun, RY = 4;
  constexpr int TX = 16 * R;  // outputs along x per CTA (16 threads)
  constexpr int SEG = (R - 1) * S2 + (kDirectMaxK2 - 1) * D2 + 1;
  constexpr int SEG4 = (SEG + 3) / 4;  // 16-byte loads per row segment
  extern __shared__ __align__(16) float slab[];          // ring: (k0 + 1) x W1 x W2p
  __shared__ float wsm[16 * 8 * 8 * kDirectMaxK2 / 8];  // the group's filters: cout_g x kv <= 16 x 56
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int ntx = (p.O[2] + TX - 1) / TX;
  const int xt = blockIdx.x % ntx, yt = blockIdx.x / ntx;
  const int G = p.Cout / p.cout_g;
  const int n = blockIdx.z / G, g = blockIdx.z % G;
  const int ob = blockIdx.y * chunk, oe = min(p.O[0], ob + chunk);
  const int x0 = xt * TX, y0 = yt * kTileY;
  const int xi0 = x0 * S2 - p.p[2], yi0 = y0 * p.s[1] - p.p[1];
  const int k0n = p.k[0], k1n = p.k[1], k2n = p.k[2];
  const int kv = k0n * k1n * k2n;
  const int nslot = k0n + 1;
  const int W2 = (TX - 1) * S2 + (k2n - 1) * D2 + 1;
  const int plane = W1 * W2p;
  const bool yreuse = p.s[1] == 1 && p.d[1] == 1;
  const long long xplane = (long long)p.S[1] * p.S[2];
  const long long ovol = (long long)p.O[0] * p.O[1] * p.O[2];
  const float* xc = p.x + ((long long)n * p.C + g) * p.S[0] * xplane;  // cin_g == 1: channel g
  // 16-byte output rows: y 16-byte aligned and rows a multiple of 4 floats
  const bool vec_store = (reinterpret_cast<uintptr_t>(p.y) & 15) == 0 && (p.O[2] & 3) == 0;
  for (int i = threadIdx.x; i < p.cout_g * kv; i += 128)
    wsm[i] = __ldg(p.w + (long long)g * p.cout_g * kv + i);
  // copy input plane zi (zero outside x) into its ring slot: rows over the
  // warps, columns over the lanes
  auto issue = [&](int zi) {
    const int slot = ((zi % nslot) + nslot) % nslot;
    const bool zok = (unsigned)zi < (unsigned)p.S[0];
    const float* src = xc + (long long)(zok ? zi : 0) * xplane;
    for (int row = threadIdx.x >> 5; row < W1; row += 4) {
      const int yi = yi0 + row;
      const bool rok = zok && (unsigned)yi < (unsigned)p.S[1];
      const float* srow = src + (long long)yi * p.S[2];
      const uint32_t dst =
          (uint32_t)__cvta_generic_to_shared(slab + slot * plane + row * W2p);
      for (int c = threadIdx.x & 31; c < W2; c += 32) {
        const int xi = xi0 + c;
        const bool ok = rok && (unsigned)xi < (unsigned)p.S[2];
        cp4z(dst + 4u * c, ok ? srow + xi : p.x, ok);
      }
    }
  };
  // the first output plane's k0 input planes
  for (int k0 = 0; k0 < k0n; ++k0) issue(ob - p.p[0] + k0);
  cp_commit_direct();
  for (int o0 = ob; o0 < oe; ++o0) {
    __syncthreads();  // the previous output plane is done with its slots
    if (o0 + 1 < oe) issue(o0 + 1 - p.p[0] + k0n - 1);
    cp_commit_direct();
    cp_wait_prev_direct();
    __syncthreads();
    for (int co = 0; co < p.cout_g; ++co) {
      const int oc = g * p.cout_g + co;
      const float bv = p.bias ? __ldg(p.bias + oc) : 0.f;
      float acc[RY][R];
#pragma unroll
      for (int a = 0; a < RY; ++a)
#pragma unroll
        for (int r = 0; r < R; ++r) acc[a][r] = bv;
      for (int k0 = 0; k0 < k0n; ++k0) {
        const int zi = o0 - p.p[0] + k0;
        const float* pl = slab + (((zi % nslot) + nslot) % nslot) * plane;
        const float* wk0 = wsm + co * kv + k0 * k1n * k2n;
        if (K3 == 3) {
          // the plane's 9 weights and all RY + 2 row segments first (every
          // shared load in flight together), then the multiply-adds
          constexpr int NS = (R - 1) * S2 + 2 * D2 + 1;  // segment words used
          float wr[9];
#pragma unroll
          for (int i = 0; i < 9; ++i) wr[i] = wk0[i];
          float seg[RY + 2][4 * ((NS + 3) / 4)];
#pragma unroll
          for (int r = 0; r < RY + 2; ++r) {
            const float4* rowp =
                reinterpret_cast<const float4*>(pl + (ty * RY + r) * W2p + tx * R * S2);
#pragma unroll
            for (int j = 0; j < (NS + 3) / 4; ++j) {
              const float4 v = rowp[j];
              seg[r][4 * j] = v.x;
              seg[r][4 * j + 1] = v.y;
              seg[r][4 * j + 2] = v.z;
              seg[r][4 * j + 3] = v.w;
            }
          }
#pragma unroll
          for (int k1 = 0; k1 < 3; ++k1)
#pragma unroll
            for (int k2 = 0; k2 < 3; ++k2) {
              const float wv = wr[k1 * 3 + k2];
#pragma unroll
              for (int a = 0; a < RY; ++a)
#pragma unroll
                for (int rx = 0; rx < R; ++rx)
                  acc[a][rx] = fmaf(wv, seg[a + k1][rx * S2 + k2 * D2], acc[a][rx]);
            }
        } else if (yreuse) {
          // input row r (relative to the thread's first) feeds output row a
          // through tap k1 = r - a
          for (int r = 0; r < RY + k1n - 1; ++r) {
            const float4* rowp =
                reinterpret_cast<const float4*>(pl + (ty * RY + r) * W2p + tx * R * S2);
            float seg[4 * SEG4];
#pragma unroll
            for (int j = 0; j < SEG4; ++j) {
              const float4 v = rowp[j];
              seg[4 * j] = v.x;
              seg[4 * j + 1] = v.y;
              seg[4 * j + 2] = v.z;
              seg[4 * j + 3] = v.w;
            }
#pragma unroll
            for (int a = 0; a < RY; ++a) {
              const int k1 = r - a;
              if (k1 < 0 || k1 >= k1n) continue;
              const float* wk = wk0 + k1 * k2n;
#pragma unroll
              for (int k2 = 0; k2 < kDirectMaxK2; ++k2) {
                if (k2 < k2n) {
                  const float wv = wk[k2];
#pragma unroll
                  for (int rx = 0; rx < R; ++rx)
                    acc[a][rx] = fmaf(wv, seg[rx * S2 + k2 * D2], acc[a][rx]);
                }
              }
            }
          }
        } else {
#pragma unroll
          for (int a = 0; a < RY; ++a) {
            for (int k1 = 0; k1 < k1n; ++k1) {
              const float4* rowp = reinterpret_cast<const float4*>(
                  pl + ((ty * RY + a) * p.s[1] + k1 * p.d[1]) * W2p + tx * R * S2);
              float seg[4 * SEG4];
#pragma unroll
              for (int j = 0; j < SEG4; ++j) {
                const float4 v = rowp[j];
                seg[4 * j] = v.x;
                seg[4 * j + 1] = v.y;
                seg[4 * j + 2] = v.z;
                seg[4 * j + 3] = v.w;
              }
              const float* wk = wk0 + k1 * k2n;
#pragma unroll
              for (int k2 = 0; k2 < kDirectMaxK2; ++k2) {
                if (k2 < k2n) {
                  const float wv = wk[k2];
#pragma unroll
                  for (int rx = 0; rx < R; ++rx)
                    acc[a][rx] = fmaf(wv, seg[rx * S2 + k2 * D2], acc[a][rx]);
                }
              }
            }
          }
        }
      }
      float* yo = p.y + ((long long)n * p.Cout + oc) * ovol + (long long)o0 * p.O[1] * p.O[2];
      const int xo0 = x0 + tx * R;
#pragma unroll
      for (int a = 0; a < RY; ++a) {
        const int yo1 = y0 + ty * RY + a;
        if (yo1 >= p.O[1]) break;
        float* yrow = yo + (long long)yo1 * p.O[2] + xo0;
        if (vec_store && xo0 + R <= p.O[2]) {
          *reinterpret_cast<float4*>(yrow) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        } else {
#pragma unroll
          for (int rx = 0; rx < R; ++rx)
            if (xo0 + rx < p.O[2]) yrow[rx] = acc[a][rx];
        }
      }
    }
  }
}

// NCDHW streaming form for one input channel per group and a 3 x 3 x 3
// filter with stride and dilation 1 along axes 0 and 1 and dilation 1 along
// x: a CTA of 128 threads owns one output channel (n, oc), a kTileY x 64
// output tile (a 4 x 4 (y, x) block per thread) and a run of `chunk` output
// planes.  It walks the input planes under that run once, each plane's
// window copied to a ring of NBUF shared-memory planes (16-byte cp.async
// pieces from a 16-byte-aligned column when V16, the window then starting SH
// columns into the row; 4-byte pieces otherwise) while the ones before it are
// computed; a plane is read once (16-byte shared loads) and added into the
// three output planes it feeds, whose accumulators rotate through three
// register slots, with the channel's 27 weights in registers.  An output
// plane is complete after its last tap, then stored and its slot restarted.
template <int S2>
struct PlaneTile {
  static constexpr int R = kDirectRun, RY = 4, K0 = 3;
  static constexpr int TX = 16 * R, TY = kTileY;             // output tile
  static constexpr int WR = TY + 2;                          // window rows
  static constexpr int WCOPY = (TX - 1) * S2 + 3;            // window columns
  static constexpr int NS = (R - 1) * S2 + 3;                // a thread's columns
  static constexpr int NBUF = S2 == 1 ? 3 : 2;               // ring depth
  // row pitch: the copied window (up to 3 columns of shift, whole 16-byte
  // pieces) and every thread's 16-byte reads fit
  static constexpr int RD = (3 + NS + 3) / 4 * 4;            // read extent, SH = 3
  static constexpr int A = (3 + WCOPY + 3) / 4 * 4;
  static constexpr int B = 15 * R * S2 + RD;
  static constexpr int W2P = A > B ? A : B;
  static constexpr int PLANE = WR * W2P;
};

template <int S2, int SH, bool V16>
__global__ void __launch_bounds__(128, 4) direct_tiled_stream_kernel(
    const __grid_constant__ DirectParams p, int ntx, int chunk) {
  using T = PlaneTile<S2>;
  constexpr int R = T::R, RY = T::RY, K0 = T::K0, NR = RY + 2, NS = T::NS;
  constexpr int NB = (SH + NS + 3) / 4;  // 16-byte loads per window row
  extern __shared__ __align__(16) float ring[];  // NBUF x WR x W2P
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int xt = blockIdx.x % ntx, yt = blockIdx.x / ntx;
  const int oc = blockIdx.z % p.Cout, n = blockIdx.z / p.Cout;
  const int ic = oc / p.cout_g;  // one input channel per group
  const int o0s = blockIdx.y * chunk;
  const int cnt = min(chunk, p.O[0] - o0s);
  const int x0 = xt * T::TX, y0 = yt * T::TY;
  // smem column 0 holds input column xs (16-byte aligned when V16)
  const int xs = x0 * S2 - p.p[2] - SH, ys = y0 - p.p[1];
  const long long xplane = (long long)p.S[1] * p.S[2];
  const float* xc = p.x + ((long long)n * p.C + ic) * p.S[0] * xplane;
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
  const int zb = o0s - p.p[0];
  const int nsteps = cnt + K0 - 1;

  auto issue = [&](int t) {
    const int z = zb + t;
    if (t < nsteps && (unsigned)z < (unsigned)p.S[0]) {
      const float* xz = xc + (long long)z * xplane;
      const uint32_t dst0 = ring_s + (uint32_t)((t % T::NBUF) * T::PLANE) * 4u;
      if (V16) {
        constexpr int PR = T::W2P / 4;  // 16-byte pieces per row
        for (int i = threadIdx.x; i < T::WR * PR; i += 128) {
          const int r = i / PR, c = (i - r * PR) * 4;
          const int yy = ys + r, xx = xs + c;
          // rows hold a multiple of 4 floats: a piece is wholly in or out
          const bool ok = (unsigned)yy < (unsigned)p.S[1] && (unsigned)xx < (unsigned)p.S[2];
          cp16z(dst0 + (uint32_t)(r * T::W2P + c) * 4u, ok ? xz + (long long)yy * p.S[2] + xx : p.x,
                ok);
        }
      } else {
        for (int i = threadIdx.x; i < T::WR * T::WCOPY; i += 128) {
          const int r = i / T::WCOPY, c = i - r * T::WCOPY;
          const int yy = ys + r, xx = xs + c;
          const bool ok = (unsigned)yy < (unsigned)p.S[1] && (unsigned)xx < (unsigned)p.S[2];
          cp4z(dst0 + (uint32_t)(r * T::W2P + c) * 4u, ok ? xz + (long long)yy * p.S[2] + xx : p.x,
               ok);
        }
      }
    }
    cp_commit_direct();
  };

  float wr[K0][9];
  const float* wk = p.w + (long long)oc * (K0 * 9);
#pragma unroll
  for (int k0 = 0; k0 < K0; ++k0)
#pragma unroll
    for (int i = 0; i < 9; ++i) wr[k0][i] = __ldg(wk + k0 * 9 + i);
  const float bv = p.bias ? __ldg(p.bias + oc) : 0.f;
  float acc[K0][RY][R];
#pragma unroll
  for (int s = 0; s < K0; ++s)
#pragma unroll
    for (int a = 0; a < RY; ++a)
#pragma unroll
      for (int r = 0; r < R; ++r) acc[s][a][r] = bv;
  const int o1s = y0 + ty * RY, o2s = x0 + tx * R;
  const long long ovol = (long long)p.O[0] * p.O[1] * p.O[2];
  float* yc = p.y + ((long long)n * p.Cout + oc) * ovol + (long long)o1s * p.O[2] + o2s;
  const bool vec = (reinterpret_cast<uintptr_t>(p.y) & 15) == 0 && (p.O[2] & 3) == 0 &&
                   o2s + R <= p.O[2];
  const int wbase = (ty * RY) * T::W2P + tx * R * S2;  // 16-byte aligned

#pragma unroll
  for (int t = 0; t < T::NBUF - 1; ++t) issue(t);
  for (int t0 = 0; t0 < nsteps; t0 += K0) {
#pragma unroll
    for (int u = 0; u < K0; ++u) {
      const int t = t0 + u;
      if (t < nsteps) {
        if (T::NBUF == 3) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        issue(t + T::NBUF - 1);
        const int z = zb + t;
        if ((unsigned)z < (unsigned)p.S[0]) {
          const float* wp = ring + (t % T::NBUF) * T::PLANE + wbase;
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            float b[4 * NB];
#pragma unroll
            for (int j = 0; j < NB; ++j) {
              const float4 v = reinterpret_cast<const float4*>(wp + r * T::W2P)[j];
              b[4 * j] = v.x;
              b[4 * j + 1] = v.y;
              b[4 * j + 2] = v.z;
              b[4 * j + 3] = v.w;
            }
#pragma unroll
            for (int k0 = 0; k0 < K0; ++k0) {
              const int sl = (u - k0 + K0) % K0;
#pragma unroll
              for (int k1 = 0; k1 < 3; ++k1) {
                const int a = r - k1;
                if (a < 0 || a >= RY) continue;
#pragma unroll
                for (int k2 = 0; k2 < 3; ++k2)
#pragma unroll
                  for (int rx = 0; rx < R; ++rx)
                    acc[sl][a][rx] =
                        fmaf(wr[k0][k1 * 3 + k2], b[SH + rx * S2 + k2], acc[sl][a][rx]);
              }
            }
          }
        }
        const int jo = t - (K0 - 1);
        const int sl = (u + 1) % K0;
        if (jo >= 0) {
          float* yp = yc + (long long)(o0s + jo) * p.O[1] * p.O[2];
#pragma unroll
          for (int a = 0; a < RY; ++a) {
            if (o1s + a < p.O[1]) {
              float* yr = yp + (long long)a * p.O[2];
              if (vec) {
                *reinterpret_cast<float4*>(yr) =
                    make_float4(acc[sl][a][0], acc[sl][a][1], acc[sl][a][2], acc[sl][a][3]);
              } else {
#pragma unroll
                for (int rx = 0; rx < R; ++rx)
                  if (o2s + rx < p.O[2]) yr[rx] = acc[sl][a][rx];
              }
            }
          }
        }
#pragma unroll
        for (int a = 0; a < RY; ++a)
#pragma unroll
          for (int rx = 0; rx < R; ++rx) acc[sl][a][rx] = bv;
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

bool direct_tiled_geometry(const DirectParams& p, int* W1, int* W2p) {
  const int s2 = p.s[2], d2 = p.d[2];
  if (p.cin_g != 1 || p.s[0] != 1 || p.d[0] != 1) return false;
  if (p.k[0] > 8 || p.k[1] > 8 || p.k[2] > kDirectMaxK2) return false;
  if (p.cout_g * p.k[0] * p.k[1] * p.k[2] > 16 * 8 * 8 * kDirectMaxK2 / 8) return false;
  const int TX = 16 * kDirectRun;
  const int w1 = (kTileY - 1) * p.s[1] + (p.k[1] - 1) * p.d[1] + 1;
  const int w2 = (TX - 1) * s2 + (p.k[2] - 1) * d2 + 1;
  // segment reads (16-byte loads from column 4 s2 tx) run past the used
  // columns; the row, a multiple of 4 words, holds them
  const int seg = (kDirectRun - 1) * s2 + (kDirectMaxK2 - 1) * d2 + 1;
  int w2p = 15 * kDirectRun * s2 + (seg + 3) / 4 * 4;
  if (w2p < w2) w2p = w2;
  w2p = (w2p + 3) / 4 * 4;
  // rows read: for y reuse up to RY + k1 - 1 past the thread's first row
  const int w1r = p.s[1] == 1 && p.d[1] == 1 ? (kTileY - 4) + 4 + p.k[1] - 1 : w1;
  const int rows = w1 > w1r ? w1 : w1r;
  if ((long long)(p.k[0] + 1) * rows * w2p > kTiledSmemFloats) return false;
  *W1 = rows;
  *W2p = w2p;
  return true;
}

// Channels-last form for 3 x 3 (y, x) filters with stride and dilation 1
// along y: a thread owns one output channel and a 4 x 4 (y, x) block at one
// (n, o0); items are ordered with the output channel fastest, so the lanes
// of a warp read and write consecutive channels.  Each input row segment
// (the 4 + 2 columns the block needs, stride C apart) feeds every output row
// that reads it.
template <int S2>
__global__ void __launch_bounds__(256, 2) direct_ndhwc_k3_kernel(const __grid_constant__ DirectParams p,
                                                              int nyb) {
  constexpr int R = kDirectRun, RY = 4;
  constexpr int NS = (R - 1) * S2 + 3;  // segment columns
  const long long items = (long long)p.N * p.O[0] * nyb * p.nrun2 * p.Cout;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < items;
       it += (long long)gridDim.x * blockDim.x) {
    long long q = it;
    const int oc = (int)(q % p.Cout);
    q /= p.Cout;
    const int r2 = (int)(q % p.nrun2);
    q /= p.nrun2;
    const int yb = (int)(q % nyb);
    q /= nyb;
    const int o0 = (int)(q % p.O[0]);
    const int n = (int)(q / p.O[0]);
    const int ic0 = (oc / p.cout_g) * p.cin_g;
    const int o2s = r2 * R, o1s = yb * RY;
    const int x2s = o2s * S2 - p.p[2], y1s = o1s - p.p[1];
    const float bv = p.bias ? __ldg(p.bias + oc) : 0.f;
    float acc[RY][R];
#pragma unroll
    for (int a = 0; a < RY; ++a)
#pragma unroll
      for (int r = 0; r < R; ++r) acc[a][r] = bv;
    const int kv = p.k[0] * 9;
    for (int ci = 0; ci < p.cin_g; ++ci) {
      const int ic = ic0 + ci;
      for (int k0 = 0; k0 < p.k[0]; ++k0) {
        const int z = o0 * p.s[0] - p.p[0] + k0 * p.d[0];
        if ((unsigned)z >= (unsigned)p.S[0]) continue;
        const float* wk = p.w + ((long long)oc * p.cin_g + ci) * kv + k0 * 9;
        float wr[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) wr[i] = __ldg(wk + i);
        const float* zp = p.x + ((long long)n * p.S[0] + z) * p.S[1] * p.S[2] * p.C + ic;
        float seg[RY + 2][NS];
#pragma unroll
        for (int r = 0; r < RY + 2; ++r) {
          const int yi = y1s + r;
          const bool rok = (unsigned)yi < (unsigned)p.S[1];
          const float* rowp = zp + (long long)yi * p.S[2] * p.C;
#pragma unroll
          for (int j = 0; j < NS; ++j) {
            const int xi = x2s + j;
            seg[r][j] = (rok && (unsigned)xi < (unsigned)p.S[2]) ? __ldg(rowp + (long long)xi * p.C)
                                                                 : 0.f;
          }
        }
#pragma unroll
        for (int k1 = 0; k1 < 3; ++k1)
#pragma unroll
          for (int k2 = 0; k2 < 3; ++k2) {
            const float wv = wr[k1 * 3 + k2];
#pragma unroll
            for (int a = 0; a < RY; ++a)
#pragma unroll
              for (int rx = 0; rx < R; ++rx)
                acc[a][rx] = fmaf(wv, seg[a + k1][rx * S2 + k2], acc[a][rx]);
          }
      }
    }
#pragma unroll
    for (int a = 0; a < RY; ++a) {
      const int yo1 = o1s + a;
      if (yo1 >= p.O[1]) break;
      float* yrow = p.y + (((long long)n * p.O[0] + o0) * p.O[1] + yo1) * p.O[2] * p.Cout + oc;
#pragma unroll
      for (int rx = 0; rx < R; ++rx)
        if (o2s + rx < p.O[2]) yrow[(long long)(o2s + rx) * p.Cout] = acc[a][rx];
    }
  }
}

// Channels-last streaming form: one input channel per group, a 3 x 3 (y, x)
// filter plane, stride and dilation 1 along axes 0 and 1, dilation 1 along x.
// A CTA of 8 warps owns a block of 32 output channels (one per lane), a
// (4 NWY) x (4 NWX) output tile (a 4 x 4 (y, x) block per warp) and a run of
// `chunk` output planes.  It walks the input planes under that run once:
// each plane's window (all rows and columns the tile reads, the channels of
// the block) is copied to shared memory with cp.async, laid out
// [row][column][32] so that a thread's window reads are conflict-free and
// sit at fixed offsets from one base; the next planes' copies are in flight
// while a plane is computed (a ring of NBUF planes).  A plane is added into
// the K0 output planes it feeds, whose accumulators rotate through K0
// register slots; an output plane is complete after its last tap, then
// stored (a warp writes 32 consecutive channels) and its slot restarted.
template <int S2>
struct StreamTile {
  static constexpr int R = kDirectRun, RY = 4;
  static constexpr int NWY = S2 == 1 ? 2 : 4, NWX = 8 / NWY;  // warps along y, x
  static constexpr int TY = RY * NWY, TX = R * NWX;           // output tile
  static constexpr int WR = TY + 2, WC = (TX - 1) * S2 + 3;   // window rows, columns
  static constexpr int PLANE = WR * WC * 32;                  // floats per window plane
  static constexpr int NBUF = S2 == 1 ? 3 : 2;                // ring depth
  static constexpr int NS = (R - 1) * S2 + 3;                 // a thread's window columns
};

template <int K0, int S2, bool V16>
__global__ void __launch_bounds__(256, 2) direct_ndhwc_stream_kernel(
    const __grid_constant__ DirectParams p, int ntx, int nty, int ncb, int chunk, int nch,
    int lg_cg) {
  using T = StreamTile<S2>;
  constexpr int R = T::R, RY = T::RY, NR = RY + 2, NS = T::NS;
  extern __shared__ __align__(16) float ring[];  // NBUF x WR x WC x 32
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wy = warp / T::NWX, wx = warp % T::NWX;
  // CTA = (x tile fastest, y tile, channel block, plane chunk, n)
  long long q = blockIdx.x;
  const int tx = (int)(q % ntx);
  q /= ntx;
  const int ty = (int)(q % nty);
  q /= nty;
  const int cb = (int)(q % ncb);
  q /= ncb;
  const int ch = (int)(q % nch);
  const int n = (int)(q / nch);
  const int icb = 32 >> lg_cg;  // input channels of the block
  const int ic0 = cb * icb;
  const int oc = cb * 32 + lane;
  const bool oc_ok = oc < p.Cout;
  const int o0s = ch * chunk;
  const int cnt = min(chunk, p.O[0] - o0s);
  const int y1w = ty * T::TY - p.p[1], x2w = tx * T::TX * S2 - p.p[2];  // window origin in x
  const long long rs = (long long)p.S[2] * p.C, ps = (long long)p.S[1] * rs;
  const float* xn = p.x + (long long)n * p.S[0] * ps;
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
  const int zb = o0s - p.p[0];  // input plane of step 0
  const int nsteps = cnt + K0 - 1;

  // copy input plane zb + t of the window to ring slot t % NBUF (zero outside x)
  auto issue = [&](int t) {
    const int z = zb + t;
    if (t < nsteps && (unsigned)z < (unsigned)p.S[0]) {
      const float* xz = xn + (long long)z * ps;
      const uint32_t dst0 = ring_s + (uint32_t)((t % T::NBUF) * T::PLANE) * 4u;
      if (V16) {
        const int per = icb >> 2;  // 16-byte pieces per position
        for (int i = threadIdx.x; i < T::WR * T::WC * per; i += 256) {
          const int pos = i / per, c4 = (i - pos * per) * 4;
          const int r = pos / T::WC, c = pos - r * T::WC;
          const int yy = y1w + r, xx = x2w + c;
          const bool ok = (unsigned)yy < (unsigned)p.S[1] && (unsigned)xx < (unsigned)p.S[2] &&
                          ic0 + c4 < p.C;
          const float* src = ok ? xz + (long long)yy * rs + (long long)xx * p.C + ic0 + c4 : p.x;
          cp16z(dst0 + (uint32_t)(pos * 32 + c4) * 4u, src, ok);
        }
      } else {
        for (int i = threadIdx.x; i < T::WR * T::WC * icb; i += 256) {
          const int pos = i / icb, c = i - pos * icb;
          const int r = pos / T::WC, cc = pos - r * T::WC;
          const int yy = y1w + r, xx = x2w + cc;
          const bool ok = (unsigned)yy < (unsigned)p.S[1] && (unsigned)xx < (unsigned)p.S[2] &&
                          ic0 + c < p.C;
          const float* src = ok ? xz + (long long)yy * rs + (long long)xx * p.C + ic0 + c : p.x;
          cp4z(dst0 + (uint32_t)(pos * 32 + c) * 4u, src, ok);
        }
      }
    }
    cp_commit_direct();
  };

  float wr[K0][9];
  const float* wk = p.w + (long long)(oc_ok ? oc : 0) * (K0 * 9);
#pragma unroll
  for (int k0 = 0; k0 < K0; ++k0)
#pragma unroll
    for (int i = 0; i < 9; ++i) wr[k0][i] = oc_ok ? __ldg(wk + k0 * 9 + i) : 0.f;
  const float bv = (oc_ok && p.bias) ? __ldg(p.bias + oc) : 0.f;
  float acc[K0][RY][R];
#pragma unroll
  for (int s = 0; s < K0; ++s)
#pragma unroll
    for (int a = 0; a < RY; ++a)
#pragma unroll
      for (int r = 0; r < R; ++r) acc[s][a][r] = bv;
  // this thread's outputs: rows o1s + a, columns o2s + rx
  const int o1s = ty * T::TY + wy * RY, o2s = tx * T::TX + wx * R;
  unsigned omask = 0;
#pragma unroll
  for (int a = 0; a < RY; ++a)
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (oc_ok && o1s + a < p.O[1] && o2s + r < p.O[2]) omask |= 1u << (a * R + r);
  const long long ors = (long long)p.O[2] * p.Cout;
  float* yw = p.y + ((long long)n * p.O[0] * p.O[1] + o1s) * ors + (long long)o2s * p.Cout + oc;
  // window base of this thread (its first row and column, its input channel)
  const int wbase = ((wy * RY) * T::WC + wx * R * S2) * 32 + (lane >> lg_cg);

#pragma unroll
  for (int t = 0; t < T::NBUF - 1; ++t) issue(t);
  for (int t0 = 0; t0 < nsteps; t0 += K0) {
#pragma unroll
    for (int u = 0; u < K0; ++u) {
      const int t = t0 + u;
      if (t < nsteps) {
        // plane t landed (this thread's copies, then everyone's); the slot
        // refilled next was last read in step t - 1, which every thread has left
        if (T::NBUF == 3) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        issue(t + T::NBUF - 1);
        const int z = zb + t;
        if ((unsigned)z < (unsigned)p.S[0]) {
          // step t: input plane zb + t feeds local output plane t - k0 by tap
          // k0, held in slot (u - k0) mod K0
          const float* wp = ring + (t % T::NBUF) * T::PLANE + wbase;
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            float seg[NS];
#pragma unroll
            for (int j = 0; j < NS; ++j) seg[j] = wp[(r * T::WC + j) * 32];
#pragma unroll
            for (int k0 = 0; k0 < K0; ++k0) {
              const int sl = (u - k0 + K0) % K0;
#pragma unroll
              for (int k1 = 0; k1 < 3; ++k1) {
                const int a = r - k1;
                if (a < 0 || a >= RY) continue;
#pragma unroll
                for (int k2 = 0; k2 < 3; ++k2)
#pragma unroll
                  for (int rx = 0; rx < R; ++rx)
                    acc[sl][a][rx] = fmaf(wr[k0][k1 * 3 + k2], seg[rx * S2 + k2], acc[sl][a][rx]);
              }
            }
          }
        }
        // local plane t - (K0 - 1) has had its last tap: store it, restart its slot
        const int jo = t - (K0 - 1);
        const int sl = (u + 1) % K0;
        if (jo >= 0) {
          float* yp = yw + (long long)(o0s + jo) * p.O[1] * ors;
#pragma unroll
          for (int a = 0; a < RY; ++a)
#pragma unroll
            for (int rx = 0; rx < R; ++rx)
              if ((omask >> (a * R + rx)) & 1u) yp[a * ors + (long long)rx * p.Cout] = acc[sl][a][rx];
        }
#pragma unroll
        for (int a = 0; a < RY; ++a)
#pragma unroll
          for (int rx = 0; rx < R; ++rx) acc[sl][a][rx] = bv;
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Output-plane chunking of a streaming form: the chunk count whose (waves of
// resident CTAs) x (input planes walked per CTA) is least; a chunk of c output
// planes walks c + k0 - 1 input planes.  At most max_chunks chunks and
// max_ctas CTAs in all.
static int stream_chunks(const DirectParams& p, long long ctas_per_chunk, long long resident,
                         long long max_ctas, int max_chunks) {
  int best = 1;
  long long best_cost = -1;
  for (int nc = 1; nc <= p.O[0] && nc <= max_chunks; ++nc) {
    const int ck = (p.O[0] + nc - 1) / nc;
    if ((p.O[0] + ck - 1) / ck != nc) continue;
    if (nc * ctas_per_chunk > max_ctas) break;
    const long long waves = (nc * ctas_per_chunk + resident - 1) / resident;
    const long long cost = waves * (ck + p.k[0] - 1);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = nc;
    }
  }
  return best;
}

// CTAs of the streaming form per output-plane chunk: (x tiles) x (y tiles) x
// (32-channel blocks) x N
static long long stream_ctas_per_chunk(const DirectParams& p) {
  const int tx = p.s[2] == 1 ? StreamTile<1>::TX : StreamTile<2>::TX;
  const int ty = p.s[2] == 1 ? StreamTile<1>::TY : StreamTile<2>::TY;
  return (long long)((p.O[2] + tx - 1) / tx) * ((p.O[1] + ty - 1) / ty) * ((p.Cout + 31) / 32) *
         p.N;
}

template <int K0, int S2, bool V16>
static cudaError_t stream_launch(const DirectParams& p, unsigned grid, int ntx, int nty, int ncb,
                                 int chunk, int nch, int lg_cg, cudaStream_t st) {
  using T = StreamTile<S2>;
  const size_t smem = (size_t)T::NBUF * T::PLANE * sizeof(float);
  direct_ndhwc_stream_kernel<K0, S2, V16><<<grid, 256, smem, st>>>(p, ntx, nty, ncb, chunk, nch,
                                                                   lg_cg);
  return cudaGetLastError();
}

template <int K0, int S2, bool V16>
static cudaError_t stream_set_smem() {
  using T = StreamTile<S2>;
  return cudaFuncSetAttribute(direct_ndhwc_stream_kernel<K0, S2, V16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)(T::NBUF * T::PLANE * sizeof(float)));
}

cudaError_t direct_set_smem() {
  cudaError_t e = cudaSuccess;
  auto take = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
  take(stream_set_smem<1, 1, true>());
  take(stream_set_smem<2, 1, true>());
  take(stream_set_smem<3, 1, true>());
  take(stream_set_smem<1, 1, false>());
  take(stream_set_smem<2, 1, false>());
  take(stream_set_smem<3, 1, false>());
  take(stream_set_smem<1, 2, true>());
  take(stream_set_smem<2, 2, true>());
  take(stream_set_smem<3, 2, true>());
  take(stream_set_smem<1, 2, false>());
  take(stream_set_smem<2, 2, false>());
  take(stream_set_smem<3, 2, false>());
  return e;
}

template <int S2, bool V16>
static cudaError_t stream_launch_k(const DirectParams& p, unsigned grid, int ntx, int nty, int ncb,
                                   int chunk, int nch, int lg_cg, cudaStream_t st) {
  if (p.k[0] == 3) return stream_launch<3, S2, V16>(p, grid, ntx, nty, ncb, chunk, nch, lg_cg, st);
  if (p.k[0] == 2) return stream_launch<2, S2, V16>(p, grid, ntx, nty, ncb, chunk, nch, lg_cg, st);
  return stream_launch<1, S2, V16>(p, grid, ntx, nty, ncb, chunk, nch, lg_cg, st);
}

template <bool NDHWC>
static cudaError_t launch_layout(const DirectParams& p, unsigned blocks, cudaStream_t st) {
  const int s2 = p.s[2], d2 = p.d[2];
  if (s2 == 1 && d2 == 1) direct_conv_kernel<NDHWC, 1, 1><<<blocks, 256, 0, st>>>(p);
  else if (s2 == 1) direct_conv_kernel<NDHWC, 1, 2><<<blocks, 256, 0, st>>>(p);
  else if (d2 == 1) direct_conv_kernel<NDHWC, 2, 1><<<blocks, 256, 0, st>>>(p);
  else direct_conv_kernel<NDHWC, 2, 2><<<blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

// NCDHW streaming form: eligibility and grid ((x, y) tiles, plane chunks,
// n x Cout)
static bool tiled_stream_eligible(const DirectParams& p) {
  return p.cin_g == 1 && p.k[0] == 3 && p.k[1] == 3 && p.k[2] == 3 && p.s[0] == 1 &&
         p.d[0] == 1 && p.s[1] == 1 && p.d[1] == 1 && p.d[2] == 1 && (p.s[2] == 1 || p.s[2] == 2);
}
static long long tiled_stream_tiles(const DirectParams& p) {
  return (long long)((p.O[2] + 16 * kDirectRun - 1) / (16 * kDirectRun)) *
         ((p.O[1] + kTileY - 1) / kTileY);
}

template <int S2, int SH, bool V16>
static cudaError_t tiled_stream_launch(const DirectParams& p, dim3 grid, int ntx, int chunk,
                                       cudaStream_t st) {
  const size_t smem = (size_t)PlaneTile<S2>::NBUF * PlaneTile<S2>::PLANE * sizeof(float);
  direct_tiled_stream_kernel<S2, SH, V16><<<grid, 128, smem, st>>>(p, ntx, chunk);
  return cudaGetLastError();
}

template <int S2>
static cudaError_t tiled_stream_launch_s(const DirectParams& p, dim3 grid, int ntx, int chunk,
                                         bool v16, cudaStream_t st) {
  if (!v16) return tiled_stream_launch<S2, 0, false>(p, grid, ntx, chunk, st);
  // smem column 0 is the 16-byte boundary at or before the window's first
  // input column x0 * s2 - p2 (x0 a multiple of 64): SH = -p2 mod 4
  switch (((-p.p[2]) % 4 + 4) % 4) {
    case 0: return tiled_stream_launch<S2, 0, true>(p, grid, ntx, chunk, st);
    case 1: return tiled_stream_launch<S2, 1, true>(p, grid, ntx, chunk, st);
    case 2: return tiled_stream_launch<S2, 2, true>(p, grid, ntx, chunk, st);
    default: return tiled_stream_launch<S2, 3, true>(p, grid, ntx, chunk, st);
  }
}

int direct_form(const DirectParams& p, bool ndhwc) {
  if (!ndhwc && tiled_stream_eligible(p) && (long long)p.N * p.Cout <= 65535 &&
      tiled_stream_tiles(p) <= 0x7fffffffLL)
    return kDirectTiledStream;
  int W1 = 0, W2p = 0;
  if (!ndhwc && direct_tiled_geometry(p, &W1, &W2p)) {
    const int TX = 16 * kDirectRun;
    const long long tiles = (long long)((p.O[2] + TX - 1) / TX) * ((p.O[1] + kTileY - 1) / kTileY);
    const long long nz = (long long)p.N * (p.Cout / p.cout_g);
    if (tiles <= 0x7fffffffLL && nz <= 65535) return kDirectTiled;
  }
  if (ndhwc && ndhwc_stream_eligible(p) && stream_ctas_per_chunk(p) <= 0x7fffffffLL)
    return kDirectNdhwcStream;
  if (ndhwc && p.k[1] == 3 && p.k[2] == 3 && p.s[1] == 1 && p.d[1] == 1 && p.d[2] == 1)
    return kDirectNdhwcK3;
  return kDirectGeneral;
}

cudaError_t direct_conv_launch(const DirectParams& p, bool ndhwc, int sm_count, cudaStream_t st) {
  const int form = direct_form(p, ndhwc);
  if (form == kDirectTiledStream) {
    const long long tiles = tiled_stream_tiles(p);
    const long long per = tiles * p.N * p.Cout;  // CTAs per plane chunk
    // 4 CTAs of 128 threads per SM (the kernel's residency)
    const int nch = stream_chunks(p, per, 4LL * sm_count, 0x7fffffffLL * 65535LL, 65535);
    const int chunk = (p.O[0] + nch - 1) / nch;
    const dim3 grid((unsigned)tiles, (unsigned)nch, (unsigned)(p.N * p.Cout));
    const int ntx = (p.O[2] + 16 * kDirectRun - 1) / (16 * kDirectRun);
    // 16-byte copies: x on 16 bytes and rows a multiple of 4 floats
    const bool v16 = (reinterpret_cast<uintptr_t>(p.x) & 15) == 0 && (p.S[2] & 3) == 0;
    return p.s[2] == 1 ? tiled_stream_launch_s<1>(p, grid, ntx, chunk, v16, st)
                       : tiled_stream_launch_s<2>(p, grid, ntx, chunk, v16, st);
  }
  if (form == kDirectTiled) {
    int W1 = 0, W2p = 0;
    direct_tiled_geometry(p, &W1, &W2p);
    const int TX = 16 * kDirectRun;
    const long long tiles = (long long)((p.O[2] + TX - 1) / TX) * ((p.O[1] + kTileY - 1) / kTileY);
    const long long nz = (long long)p.N * (p.Cout / p.cout_g);
    // output planes per CTA: enough CTAs for ~4 waves of 4 per SM, at least 4
    // planes (so at most 16 chunks per SM)
    long long want = 16LL * sm_count;
    long long chunks = std::max(1LL, std::min<long long>(p.O[0], want / std::max(1LL, tiles * nz)));
    int chunk = (int)((p.O[0] + chunks - 1) / chunks);
    if (chunk < 4) chunk = std::min(4, p.O[0]);
    chunks = (p.O[0] + chunk - 1) / chunk;
    if (chunks > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)tiles, (unsigned)chunks, (unsigned)nz);
    const int s2 = p.s[2], d2 = p.d[2];
    const bool k3 = p.k[1] == 3 && p.k[2] == 3 && p.s[1] == 1 && p.d[1] == 1;
    const size_t smem = (size_t)(p.k[0] + 1) * W1 * W2p * sizeof(float);  // <= 44 KB
    if (s2 == 1 && d2 == 1) {
      if (k3) direct_tiled_kernel<1, 1, 3><<<grid, 128, smem, st>>>(p, W1, W2p, chunk);
      else direct_tiled_kernel<1, 1, 0><<<grid, 128, smem, st>>>(p, W1, W2p, chunk);
    } else if (s2 == 1) {
      direct_tiled_kernel<1, 2, 0><<<grid, 128, smem, st>>>(p, W1, W2p, chunk);
    } else if (d2 == 1) {
      if (k3) direct_tiled_kernel<2, 1, 3><<<grid, 128, smem, st>>>(p, W1, W2p, chunk);
      else direct_tiled_kernel<2, 1, 0><<<grid, 128, smem, st>>>(p, W1, W2p, chunk);
    } else {
      direct_tiled_kernel<2, 2, 0><<<grid, 128, smem, st>>>(p, W1, W2p, chunk);
    }
    return cudaGetLastError();
  }
  if (form == kDirectNdhwcStream) {
    int lg_cg = 0;
    while ((1 << lg_cg) < p.cout_g) ++lg_cg;
    const int tw = p.s[2] == 1 ? StreamTile<1>::TX : StreamTile<2>::TX;
    const int th = p.s[2] == 1 ? StreamTile<1>::TY : StreamTile<2>::TY;
    const int ntx = (p.O[2] + tw - 1) / tw, nty = (p.O[1] + th - 1) / th;
    const int ncb = (p.Cout + 31) / 32;
    const long long per = stream_ctas_per_chunk(p);  // <= INT32_MAX (direct_form)
    const int nch = stream_chunks(p, per, 2LL * sm_count, 0x7fffffffLL, 0x7fffffff);
    const int chunk = (p.O[0] + nch - 1) / nch;
    const long long grid = per * nch;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // 16-byte copies: channel rows and the block's first channel on 16 bytes
    const int icb = 32 >> lg_cg;
    const bool v16 = (reinterpret_cast<uintptr_t>(p.x) & 15) == 0 && (p.C & 3) == 0 && (icb & 3) == 0;
    const unsigned g = (unsigned)grid;
    if (p.s[2] == 1)
      return v16 ? stream_launch_k<1, true>(p, g, ntx, nty, ncb, chunk, nch, lg_cg, st)
                 : stream_launch_k<1, false>(p, g, ntx, nty, ncb, chunk, nch, lg_cg, st);
    return v16 ? stream_launch_k<2, true>(p, g, ntx, nty, ncb, chunk, nch, lg_cg, st)
               : stream_launch_k<2, false>(p, g, ntx, nty, ncb, chunk, nch, lg_cg, st);
  }
  if (form == kDirectNdhwcK3) {
    const int nyb = (p.O[1] + 3) / 4;
    const long long items = (long long)p.N * p.O[0] * nyb * p.nrun2 * p.Cout;
    long long blocks = (items + 255) / 256;
    if (blocks > 8LL * sm_count) blocks = 8LL * sm_count;
    if (blocks < 1) blocks = 1;
    if (p.s[2] == 1) direct_ndhwc_k3_kernel<1><<<(unsigned)blocks, 256, 0, st>>>(p, nyb);
    else direct_ndhwc_k3_kernel<2><<<(unsigned)blocks, 256, 0, st>>>(p, nyb);
    return cudaGetLastError();
  }
  // persistent grid: 8 CTAs of 256 threads per SM, fewer for small problems
  long long blocks = (p.items + 255) / 256;
  if (blocks > 8LL * sm_count) blocks = 8LL * sm_count;
  if (blocks < 1) blocks = 1;
  return ndhwc ? launch_layout<true>(p, (unsigned)blocks, st)
               : launch_layout<false>(p, (unsigned)blocks, st);
}

// [N][A][B] -> [N][B][A] through 32x32 shared-memory tiles (both sides
// coalesced); grid (tilesA * tilesB, N), 32x8 threads.
__global__ void __launch_bounds__(256) transpose_kernel(const float* __restrict__ in,
                                                        float* __restrict__ out, long long A,
                                                        long long B, long long tilesB) {
  __shared__ float tile[32][33];
  const long long n = blockIdx.y;
  const long long ta = blockIdx.x / tilesB, tb = blockIdx.x % tilesB;
  const long long a0 = ta * 32, b0 = tb * 32;
  const float* src = in + n * A * B;
  float* dst = out + n * A * B;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const long long a = a0 + i, b = b0 + threadIdx.x;
    if (a < A && b < B) tile[i][threadIdx.x] = src[a * B + b];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const long long b = b0 + i, a = a0 + threadIdx.x;
    if (a < A && b < B) dst[b * A + a] = tile[threadIdx.x][i];
  }
}

cudaError_t transpose_launch(const float* in, float* out, int N, long long A, long long B,
                             cudaStream_t st) {
  const long long ta = (A + 31) / 32, tb = (B + 31) / 32;
  if (ta * tb > 0x7fffffffLL || N > 65535) return cudaErrorInvalidValue;
  transpose_kernel<<<dim3((unsigned)(ta * tb), (unsigned)N), dim3(32, 8), 0, st>>>(in, out, A, B,
                                                                                  tb);
  return cudaGetLastError();
}

}  // namespace tc3d
