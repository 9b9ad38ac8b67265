// direct.cu -- direct fp32 convolution for grouped / depthwise convs with few
// channels per group, in NCDHW or NDHWC, and the layout transpose used around
// the engine for channels-last input.
//
// The sum is the direct-convolution formula of the page "Kimi-K2.6 l1_p59"
// with its group rule (output channel oc reads the input channels of group
// oc / (Cout/G)): y[n,oc,o] = bias[oc] + sum_{ci,k} w[oc,ci,k] *
// x[n, g*cin_g + ci, o*s - p + d*k], zero outside x.
#include "direct.cuh"

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
