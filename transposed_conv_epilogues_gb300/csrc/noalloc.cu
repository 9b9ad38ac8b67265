// noalloc.cu -- conv_maxpool_lse_relu for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc: code running inside an allocator or a
// memory-pool callback, plugin hosts that own every device allocation, or
// real-time paths where an allocation (and its implicit synchronisation) is
// not allowed.  They cannot provide the workspace the regular entry point
// needs for its packed weights.  This variant takes its scratch from a fixed
// array compiled into the library instead; the caller passes only inputs and
// outputs.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/tc3d.h"

// The scratch every call of the entry point below uses.  Each GPU that loads
// the library holds one copy of it until the process exits.
static __device__ __align__(256) unsigned char tc3d_noalloc_scratch[TC3D_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name only stands in for the device object, so its address must
// be looked up once per device (with that device current) and passed on.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();  // the failure is reported here, not by the next launch check
    return TC3D_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, tc3d_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return TC3D_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return TC3D_OK;
}

}  // namespace

extern "C" int tc3d_conv_maxpool_lse_relu_noalloc(const float* x, const float* w,
                                                  const float* bias, float* y, int N, int Cin,
                                                  int S0, int S1, int S2, int Cout, int k0,
                                                  int k1, int k2, const int stride[3],
                                                  const int pad[3], const int dilation[3],
                                                  const int output_padding[3], int groups,
                                                  cudaStream_t stream) {
  size_t need = 0;
  int rc = tc3d_workspace_bytes(TC3D_OP_CONV_MAXPOOL_LSE_RELU, N, Cin, S0, S1, S2, Cout, k0, k1,
                                k2, stride, pad, dilation, output_padding, groups, &need);
  if (rc) return rc;
  if (need > (size_t)TC3D_NOALLOC_SCRATCH_BYTES) return TC3D_ERR_WORKSPACE;
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  // The whole region a call uses (the packed weights) is rewritten by that
  // call before it is read, so nothing has to be cleared between calls.
  return tc3d_conv_maxpool_lse_relu(x, w, bias, y, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride,
                                    pad, dilation, output_padding, groups, scratch,
                                    (size_t)TC3D_NOALLOC_SCRATCH_BYTES, stream);
}
