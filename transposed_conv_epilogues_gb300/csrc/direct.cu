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

template <bool NDHWC>
static cudaError_t launch_layout(const DirectParams& p, unsigned blocks, cudaStream_t st) {
  const int s2 = p.s[2], d2 = p.d[2];
  if (s2 == 1 && d2 == 1) direct_conv_kernel<NDHWC, 1, 1><<<blocks, 256, 0, st>>>(p);
  else if (s2 == 1) direct_conv_kernel<NDHWC, 1, 2><<<blocks, 256, 0, st>>>(p);
  else if (d2 == 1) direct_conv_kernel<NDHWC, 2, 1><<<blocks, 256, 0, st>>>(p);
  else direct_conv_kernel<NDHWC, 2, 2><<<blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t direct_conv_launch(const DirectParams& p, bool ndhwc, int sm_count, cudaStream_t st) {
  int W1 = 0, W2p = 0;
  if (!ndhwc && direct_tiled_geometry(p, &W1, &W2p)) {
    const int TX = 16 * kDirectRun;
    const long long tiles = (long long)((p.O[2] + TX - 1) / TX) * ((p.O[1] + kTileY - 1) / kTileY);
    const long long nz = (long long)p.N * (p.Cout / p.cout_g);
    // output planes per CTA: enough CTAs for ~4 waves of 4 per SM, at least 4 planes
    long long want = 16LL * sm_count;
    long long chunks = std::max(1LL, std::min<long long>(p.O[0], want / std::max(1LL, tiles * nz)));
    int chunk = (int)((p.O[0] + chunks - 1) / chunks);
    if (chunk < 4) chunk = std::min(4, p.O[0]);
    chunks = (p.O[0] + chunk - 1) / chunk;
    if (tiles <= 0x7fffffffLL && chunks <= 65535 && nz <= 65535) {
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
  }
  if (ndhwc && p.k[1] == 3 && p.k[2] == 3 && p.s[1] == 1 && p.d[1] == 1 && p.d[2] == 1) {
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
