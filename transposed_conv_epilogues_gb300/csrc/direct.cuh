// direct.cuh -- CUDA-core paths for convolutions the tensor-core engine maps
// poorly: grouped / depthwise convs with few channels per group (direct fp32
// multiply-adds), and the channels-last (NDHWC) layout (native in the direct
// kernel; a tiled transpose around the engine otherwise).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace tc3d {

// Direct kernel limits: along the contiguous output axis a thread computes
// kDirectRun consecutive outputs from one register segment of the input row,
// so stride and dilation along that axis are template parameters (1 or 2) and
// its kernel extent is at most kDirectMaxK2.
constexpr int kDirectRun = 4;
constexpr int kDirectMaxK2 = 7;

struct DirectParams {
  const float* x;     // [N, C, S0, S1, S2] or, channels-last, [N, S0, S1, S2, C]
  const float* w;     // [Cout, C/G, k0, k1, k2]
  const float* bias;  // [Cout] or nullptr
  float* y;           // [N, Cout, O0, O1, O2] or [N, O0, O1, O2, Cout]
  int N, C, S[3], Cout, k[3], s[3], p[3], d[3], cin_g, cout_g;
  int O[3];
  int nrun2;          // runs of kDirectRun outputs along axis 2: ceil(O2 / kDirectRun)
  long long items;    // N * Cout * O0 * O1 * nrun2
};

// Whether the direct kernel takes a conv: few channels per group and an
// axis-2 stride / dilation / extent it is built for.
inline bool direct_eligible(int cin_g, int cout_g, int s2, int d2, int k2) {
  return cin_g * cout_g <= 16 && (s2 == 1 || s2 == 2) && (d2 == 1 || d2 == 2) &&
         k2 <= kDirectMaxK2;
}

cudaError_t direct_conv_launch(const DirectParams& p, bool ndhwc, int sm_count, cudaStream_t st);

// Layout transposes of an [N][A][B] float array to [N][B][A] (A, B >= 1):
// NDHWC -> NCDHW with A = S0*S1*S2, B = C, and back with A = C, B = S.
cudaError_t transpose_launch(const float* in, float* out, int N, long long A, long long B,
                             cudaStream_t st);

}  // namespace tc3d
