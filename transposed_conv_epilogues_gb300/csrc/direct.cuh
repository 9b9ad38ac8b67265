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

// Shared-memory tiled form (NCDHW, one input channel per group, stride and
// dilation 1 along axis 0): a CTA of 128 threads computes a kTileY x 64
// output tile over a chunk of output planes, for every output channel of a
// group, each thread a 4 x 4 block (y, x); a ring of k0 + 1 input planes
// (W1 rows x W2p columns) must fit kTiledSmemFloats.
constexpr int kTileY = 32;
constexpr int kTiledSmemFloats = 11 * 1024;
// slab extents of the tiled form for a conv, or false when it does not apply
bool direct_tiled_geometry(const DirectParams& p, int* W1, int* W2p);

// Channels-last streaming form: one input channel per group and a channel
// multiplier (cout_g) that divides 32; k0 <= 3 with stride and dilation 1
// along axis 0; a 3 x 3 (y, x) filter plane with stride and dilation 1 along
// y and dilation 1 along x.
inline bool ndhwc_stream_eligible(const DirectParams& p) {
  return p.cin_g == 1 && (32 % p.cout_g) == 0 && p.k[0] >= 1 && p.k[0] <= 3 && p.s[0] == 1 &&
         p.d[0] == 1 &&
         p.k[1] == 3 && p.k[2] == 3 && p.s[1] == 1 && p.d[1] == 1 && p.d[2] == 1 &&
         (p.s[2] == 1 || p.s[2] == 2);
}

// The direct kernel a conv takes (the layout flag: channels-last)
enum DirectForm {
  kDirectGeneral = 0,
  kDirectTiled = 1,
  kDirectNdhwcK3 = 2,
  kDirectNdhwcStream = 3,
  kDirectTiledStream = 4
};
int direct_form(const DirectParams& p, bool ndhwc);

// Opts the streaming form's kernels into their shared-memory size (once per
// device, before the first direct_conv_launch).
cudaError_t direct_set_smem();

cudaError_t direct_conv_launch(const DirectParams& p, bool ndhwc, int sm_count, cudaStream_t st);

// Layout transposes of an [N][A][B] float array to [N][B][A] (A, B >= 1):
// NDHWC -> NCDHW with A = S0*S1*S2, B = C, and back with A = C, B = S.
cudaError_t transpose_launch(const float* in, float* out, int N, long long A, long long B,
                             cudaStream_t st);

}  // namespace tc3d
