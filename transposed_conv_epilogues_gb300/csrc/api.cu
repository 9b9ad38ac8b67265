// api.cu -- the C ABI (include/tc3d.h): argument checks, plans, tensor-map
// encoding and the launches of one call, all enqueued on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/tc3d.h"
#include "engine.cuh"
#include "plan.h"
#include "direct.cuh"
#include "pool.cuh"

using namespace tc3d;

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s

std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};

// The kernels bound their waits in SM clock cycles; 2.1 cycles per ns is the
// top clock, so at lower clocks a wait may last somewhat longer in time.
unsigned long long timeout_cycles(unsigned long long ns) { return ns * 21ull / 10ull; }

struct DeviceState {
  bool init = false;
  int status = TC3D_OK;
  int sm_count = 0;
  int* err = nullptr;  // device address of the error word
  bool smem_set[5] = {false, false, false, false, false};  // per kernel id
  bool gram_smem_set = false;
  bool direct_smem_set = false;
  bool lag_smem_set = false;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;


int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TC3D_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    d.init = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      d.status = TC3D_ERR_CUDA;
    } else if (major != 10 || minor != 3) {
      d.status = TC3D_ERR_DEVICE;  // the kernels are built for sm_103a only
    } else if (error_flag_address(&d.err) != cudaSuccess) {
      d.status = TC3D_ERR_CUDA;
    }
    if (!g_encode && d.status == TC3D_OK) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) == cudaSuccess &&
          q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  *out = &d;
  return d.status;
}

Problem make_problem(int op, int N, int Cin, int S0, int S1, int S2, int Cout, int k0, int k1,
                     int k2, const int stride[3], const int pad[3], const int dil[3],
                     const int out_pad[3], int groups) {
  Problem pb;
  std::memset(&pb, 0, sizeof(pb));
  pb.op = op;
  pb.N = N;
  pb.Cin = Cin;
  pb.S[0] = S0;
  pb.S[1] = S1;
  pb.S[2] = S2;
  pb.Cout = Cout;
  pb.k[0] = k0;
  pb.k[1] = k1;
  pb.k[2] = k2;
  for (int a = 0; a < 3; ++a) {
    pb.stride[a] = stride ? stride[a] : 1;
    pb.pad[a] = pad ? pad[a] : 0;
    pb.dil[a] = dil ? dil[a] : 1;
    pb.out_pad[a] = out_pad ? out_pad[a] : 0;
  }
  pb.groups = groups;
  return pb;
}

int plan_for(int op, int N, int Cin, int S0, int S1, int S2, int Cout, int k0, int k1, int k2,
             const int stride[3], const int pad[3], const int dil[3], const int out_pad[3],
             int groups, Plan* pl) {
  if (!stride || !pad || !dil) return TC3D_ERR_NULL;
  Problem pb = make_problem(op, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil, out_pad,
                            groups);
  return make_plan(pb, pl);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int set_smem(DeviceState* d, int kid) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!d->smem_set[kid]) {
    if (engine_set_smem(kid, kMaxSmem) != cudaSuccess) return TC3D_ERR_CUDA;
    d->smem_set[kid] = true;
  }
  return TC3D_OK;
}

void fill_params(const Plan& pl, EngineParams* ep) {
  std::memset(ep, 0, sizeof(*ep));
  const Problem& pb = pl.pb;
  ep->timeout_cycles = timeout_cycles(g_timeout_ns.load());
  ep->N = pb.N;
  ep->C = pb.Cin;
  ep->Cout = pb.Cout;
  ep->G = pb.groups;
  ep->cin_g = pl.cin_g;
  ep->cout_g = pl.cout_g;
  for (int a = 0; a < 3; ++a) {
    ep->S[a] = pb.S[a];
    ep->O[a] = (int)pl.O[a];
    ep->P[a] = (int)pl.P[a];
    ep->M[a] = pl.M[a];
    ep->s_in[a] = pl.s_in[a];
    ep->s_out[a] = pl.s_out[a];
    ep->u_min[a] = pl.u_min[a];
    ep->nU[a] = pl.nU[a];
    for (int t = 0; t < kMaxAxisTaps; ++t) ep->u_rel[a][t] = pl.u_rel[a][t];
    ep->nRaxis[a] = pl.nRaxis[a];
    int mask = 0;
    for (int i = 0; i < pl.nRaxis[a]; ++i) {
      ep->r_axis[a][i] = pl.r_axis[a][i];
      mask |= 1 << pl.r_axis[a][i];
    }
    ep->cls_mask[a] = mask;
    ep->Q[a] = pl.Q[a];
    ep->Pq[a] = pl.Pq[a];
    ep->T[a] = pl.T[a];
    ep->ntile[a] = pl.ntile[a];
    ep->ntile_div[a] = make_fastdiv(pl.ntile[a]);
    // the planner builds Q and Pq as powers of two
    ep->lQ[a] = 0;
    while ((1 << ep->lQ[a]) < pl.Q[a]) ++ep->lQ[a];
    ep->lPq[a] = 0;
    while ((1 << ep->lPq[a]) < pl.Pq[a]) ++ep->lPq[a];
    ep->box[a] = pl.box[a];
  }
  {
    // class tables of the one-class store path (the plan checked that the
    // offsets from a row's first output fit in an int)
    const int F = pl.s_out[0] * pl.s_out[1] * pl.s_out[2];
    const long long o12 = (long long)pl.O[1] * pl.O[2];
    ep->cls_fast = pl.cls_fast;
    for (int f = 0; f < 8 && f < F; ++f) {
      const int r2 = f % pl.s_out[2], r1 = (f / pl.s_out[2]) % pl.s_out[1],
                r0 = f / (pl.s_out[2] * pl.s_out[1]);
      const long long off = r0 * o12 + (long long)r1 * pl.O[2] + r2;
      ep->cls_off[f] = (int)std::min<long long>(off, INT32_MAX);
      ep->cls_r[f] = r0 | (r1 << 8) | (r2 << 16);
      if (pl.nR == 1 && r0 == pl.r_axis[0][0] && r1 == pl.r_axis[1][0] && r2 == pl.r_axis[2][0])
        ep->cls_star = f;
    }
  }
  ep->nUtot = pl.nU[0] * pl.nU[1] * pl.nU[2];
  ep->nR = pl.nR;
  ep->nEmpty = pl.nEmpty;
  ep->ocb = pl.ocb;
  ep->n_tile = pl.n_tile;
  ep->nb_per_group = pl.nb_per_group;
  ep->n_colblocks = pl.n_colblocks;
  ep->n_acc = pl.n_acc;
  ep->dbuf = pl.dbuf;
  ep->a_stages = pl.a_stages;
  ep->ks_stage = pl.ks_stage;
  ep->view = pl.view;
  ep->cl = pl.cl;
  ep->cl_cb = pl.cl_cb;
  ep->nslots = pl.nslots;
  ep->slot_bytes = (unsigned)pl.slot_bytes;
  ep->wide = pl.wide;
  ep->acc_cols = pl.acc_cols;
  ep->tiles = (int)pl.tiles;
  ep->cin_chunk = pl.cin_chunk;
  ep->n_chunks = pl.n_chunks;
  ep->k_chunk = pl.k_chunk;
  ep->ksteps_chunk = pl.ksteps_chunk;
  ep->raw_stages = pl.raw_stages;
  ep->raw_stage_bytes = (unsigned)pl.raw_stage_bytes;
  ep->b_resident = pl.b_resident;
  ep->b_stages = pl.b_stages;
  ep->b_stage_bytes = (unsigned)pl.b_stage_bytes;
  const SmemLayout L = smem_layout(pl);
  ep->sm_raw = (unsigned)L.raw;
  ep->sm_b = (unsigned)L.b;
  ep->sm_xs = (unsigned)L.xs;
  ep->sm_ktab = (unsigned)L.ktab;
  ep->sm_misc = (unsigned)L.misc;
  ep->sm_bar = (unsigned)L.bar;
}

// Encode the 5-D tensor map over x, or leave use_tma = 0 (plain-load producer)
// when x or its strides break TMA's 16-byte rules.
void encode_xmap(const Plan& pl, const float* x, EngineParams* ep) {
  const Problem& pb = pl.pb;
  ep->use_tma = 0;
  if (pl.cl) {
    // channels-last: x as (C, S2, S1, S0, N), box cl_cb x B2 x B1 x B0 x 1
    if (!g_encode || !aligned(x, 16) || (pb.Cin % 4) != 0) return;
    cuuint64_t dims[5] = {(cuuint64_t)pb.Cin, (cuuint64_t)pb.S[2], (cuuint64_t)pb.S[1],
                          (cuuint64_t)pb.S[0], (cuuint64_t)pb.N};
    cuuint64_t strides[4];
    strides[0] = (cuuint64_t)pb.Cin * 4;
    strides[1] = strides[0] * pb.S[2];
    strides[2] = strides[1] * pb.S[1];
    strides[3] = strides[2] * pb.S[0];
    for (int i = 0; i < 4; ++i)
      if (strides[i] >= (1ull << 40)) return;
    cuuint32_t box[5] = {(cuuint32_t)pl.cl_cb, (cuuint32_t)pl.box[2], (cuuint32_t)pl.box[1],
                         (cuuint32_t)pl.box[0], 1};
    for (int i = 0; i < 5; ++i)
      if (box[i] == 0 || box[i] > 256) return;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(&ep->xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, const_cast<float*>(x),
                          dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) ep->use_tma = 1;
    return;
  }
  if (!g_encode || !aligned(x, 16) || (pb.S[2] % 4) != 0) return;
  cuuint64_t dims[5] = {(cuuint64_t)pb.S[2], (cuuint64_t)pb.S[1], (cuuint64_t)pb.S[0],
                        (cuuint64_t)pb.Cin, (cuuint64_t)pb.N};
  cuuint64_t strides[4];
  strides[0] = (cuuint64_t)pb.S[2] * 4;
  strides[1] = strides[0] * pb.S[1];
  strides[2] = strides[1] * pb.S[0];
  strides[3] = strides[2] * pb.Cin;
  for (int i = 0; i < 4; ++i)
    if (strides[i] >= (1ull << 40)) return;
  cuuint32_t box[5] = {(cuuint32_t)pl.box[2], (cuuint32_t)pl.box[1], (cuuint32_t)pl.box[0],
                       (cuuint32_t)pl.cin_chunk, 1};
  for (int i = 0; i < 5; ++i)
    if (box[i] == 0 || box[i] > 256) return;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(&ep->xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, const_cast<float*>(x),
                        dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) ep->use_tma = 1;
}

// Tensor map of the lag kernel: x as (S2, S1, S0, C, N), box 40 x 3 x 4 x C
// x 1 (one warp's window rows of 4 consecutive planes).  False (the Gram kernel then takes the statistics) when x or its rows
// break TMA's 16-byte rules.
bool encode_lag_map(const Problem& pb, const float* x, LagParams* lp) {
  std::memset(lp, 0, sizeof(*lp));
  if (!g_encode || !aligned(x, 16) || (pb.S[2] % 4) != 0) return false;
  cuuint64_t dims[5] = {(cuuint64_t)pb.S[2], (cuuint64_t)pb.S[1], (cuuint64_t)pb.S[0],
                        (cuuint64_t)pb.Cin, (cuuint64_t)pb.N};
  cuuint64_t strides[4];
  strides[0] = (cuuint64_t)pb.S[2] * 4;
  strides[1] = strides[0] * pb.S[1];
  strides[2] = strides[1] * pb.S[0];
  strides[3] = strides[2] * pb.Cin;
  for (int i = 0; i < 4; ++i)
    if (strides[i] >= (1ull << 40)) return false;
  cuuint32_t box[5] = {(cuuint32_t)kLagBoxCols, (cuuint32_t)kLagBoxRows, (cuuint32_t)kLagChunk,
                       (cuuint32_t)pb.Cin, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return g_encode(&lp->xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, const_cast<float*>(x), dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of the pooled-conv kernel: x as (S2, S1, S0, C, N), box 36 x 9 x
// 3 x C x 1.  False (the engine then runs the pooled conv) when x or its
// rows break TMA's 16-byte rules.
bool encode_pooled_map(const Problem& pb, const float* x, PooledParams* pq) {
  std::memset(pq, 0, sizeof(*pq));
  if (!g_encode || !aligned(x, 16) || (pb.S[2] % 4) != 0) return false;
  cuuint64_t dims[5] = {(cuuint64_t)pb.S[2], (cuuint64_t)pb.S[1], (cuuint64_t)pb.S[0],
                        (cuuint64_t)pb.Cin, (cuuint64_t)pb.N};
  cuuint64_t strides[4];
  strides[0] = (cuuint64_t)pb.S[2] * 4;
  strides[1] = strides[0] * pb.S[1];
  strides[2] = strides[1] * pb.S[0];
  strides[3] = strides[2] * pb.Cin;
  for (int i = 0; i < 4; ++i)
    if (strides[i] >= (1ull << 40)) return false;
  cuuint32_t box[5] = {(cuuint32_t)kPooledBoxCols, (cuuint32_t)kPooledBoxRows, 3,
                       (cuuint32_t)pb.Cin, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return g_encode(&pq->xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, const_cast<float*>(x), dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fill_ctr: the engine's bias-fill counter, zeroed by the pack kernel (or nullptr)
int launch_pack(const Plan& pl, const float* w, float* wpack, int sm_count, cudaStream_t st,
                unsigned long long* fill_ctr = nullptr) {
  PackParams pp;
  std::memset(&pp, 0, sizeof(pp));
  pp.w = w;
  pp.zero_ctr = fill_ctr;
  pp.out = wpack;
  pp.transposed = pl.transposed;
  pp.cin_g = pl.cin_g;
  pp.cout_g = pl.cout_g;
  for (int a = 0; a < 3; ++a) {
    pp.k[a] = pl.pb.k[a];
    pp.nU[a] = pl.nU[a];
    pp.nRaxis[a] = pl.nRaxis[a];
    for (int r = 0; r < kMaxClassesAxis; ++r)
      for (int t = 0; t < kMaxAxisTaps; ++t) pp.kidx[a][r][t] = pl.kidx[a][r][t];
  }
  pp.nUtot = pl.nU[0] * pl.nU[1] * pl.nU[2];
  pp.nR = pl.nR;
  pp.ocb = pl.ocb;
  pp.n_tile = pl.n_tile;
  pp.nb_per_group = pl.nb_per_group;
  pp.n_colblocks = pl.n_colblocks;
  pp.cin_chunk = pl.cin_chunk;
  pp.n_chunks = pl.n_chunks;
  pp.k_chunk = pl.k_chunk;
  pp.ksteps_chunk = pl.ksteps_chunk;
  pp.octet_major = pl.view;
  pp.tap_major = pl.cl;
  pp.total = pl.ws_wpack_bytes / 4;
  long long blocks = (pp.total + 255) / 256;
  if (blocks > (long long)sm_count * 8) blocks = (long long)sm_count * 8;
  return pack_launch(pp, (unsigned)blocks, st) == cudaSuccess ? TC3D_OK : TC3D_ERR_CUDA;
}

// The bias fill of the outputs no engine tile writes (a transposed conv's
// tap-less classes and rows past its row grid)
FillParams make_fill(const Plan& pl, const float* bias, float* y) {
  FillParams fp;
  fp.y = y;
  fp.bias = bias;
  fp.ctr = nullptr;
  fp.NC = (int)(pl.pb.N * pl.pb.Cout);
  fp.Cout = (int)pl.pb.Cout;
  for (int a = 0; a < 3; ++a) {
    fp.O[a] = (int)pl.O[a];
    fp.zl[a] = (int)std::min<int64_t>(pl.O[a], (int64_t)pl.s_out[a] * pl.M[a]);
  }
  // the engine's rows: the (r0, r1) pair of its one class with taps; with
  // stride 2 along y it also writes the other y class's rows of its planes
  const bool ybeside = pl.s_out[1] == 2;
  fp.s0 = pl.fill_rows ? pl.s_out[0] : 0;
  fp.s1 = pl.fill_rows ? (ybeside ? 1 : pl.s_out[1]) : 0;
  fp.r0 = pl.fill_rows ? pl.r_axis[0][0] : 0;
  fp.r1 = pl.fill_rows && !ybeside ? pl.r_axis[1][0] : 0;
  return fp;
}

int launch_engine(const Plan& pl, int epi, const float* x, const float* wpack, const float* bias,
                  float* y, float2* partials, DeviceState* d, cudaStream_t st,
                  const float2* bn_affine = nullptr, unsigned long long* fill_ctr = nullptr) {
  // the store epilogue's fill warp does the bias fill; without tiles the
  // stand-alone fill kernel does it
  const bool fill = epi == EPI_STORE && pl.fill_slab;
  if (pl.tiles == 0)
    return !fill || fill_slab_launch(make_fill(pl, bias, y), st) == cudaSuccess ? TC3D_OK
                                                                               : TC3D_ERR_CUDA;
  EngineParams ep;
  fill_params(pl, &ep);
  ep.fill_on = fill ? 1 : 0;
  if (fill) {
    if (!fill_ctr) return TC3D_ERR_UNSUPPORTED;
    ep.fill = make_fill(pl, bias, y);
    ep.fill.ctr = fill_ctr;
  }
  ep.x = x;
  ep.wpack = wpack;
  ep.bias = bias;
  ep.y = y;
  ep.partials = partials;
  ep.bn_affine = bn_affine;
  ep.err = d->err;
  encode_xmap(pl, x, &ep);
  const unsigned grid = (unsigned)engine_grid(pl, d->sm_count);
  ep.part_slots = (int)bn_part_slots(pl, grid);
  const int kid = pl.view ? kEngineView : pl.cl ? kEngineCl : epi;
  int rc = set_smem(d, kid);
  if (rc) return rc;
  return engine_launch(kid, ep, grid, (size_t)pl.smem_bytes, st) == cudaSuccess ? TC3D_OK
                                                                               : TC3D_ERR_CUDA;
}

int common_checks(const float* x, const float* w, const float* y, const float* bias,
                  const void* ws, size_t ws_bytes, int64_t ws_total) {
  if (!x || !w || !y) return TC3D_ERR_NULL;
  if (!aligned(x, 4) || !aligned(w, 4) || !aligned(y, 4) || (bias && !aligned(bias, 4)))
    return TC3D_ERR_ALIGN;
  if (!ws || ws_bytes < (size_t)ws_total) return TC3D_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return TC3D_ERR_ALIGN;
  return TC3D_OK;
}

// BatchNorm arguments of the two BN-pool entry points (running_mean and
// running_var only for evaluation mode)
struct BnArgs {
  const float* gamma = nullptr;
  const float* beta = nullptr;
  const float* rmean = nullptr;
  const float* rvar = nullptr;
  float eps = 0.f;
};

// Plans of one call: the engine plan of the operation and, for the BN-pool
// ops, the algebraic path when it applies (it then replaces the engine plan's
// launches and sets the workspace size).
struct CallPlan {
  Plan pl;
  PoolPlan pp;
  bool pool_ok = false;  // the algebraic path applies
  bool pool = false;     // and is taken
  bool ndhwc = false;    // channels-last x and y (OP_CONV_NDHWC)
  bool direct = false;   // the direct CUDA-core conv kernel
  Problem upb;           // the caller's problem (the engine plan may use a merged form)
  int64_t ws_xt_off = 0, ws_yt_off = 0;  // channels-last through the engine: NCDHW copies
  int64_t ws_total = 0;
};

int plan_call(int op, int N, int Cin, int S0, int S1, int S2, int Cout, int k0, int k1, int k2,
              const int stride[3], const int pad[3], const int dil[3], const int out_pad[3],
              int groups, CallPlan* cp) {
  cp->ndhwc = op == OP_CONV_NDHWC;
  int rc;
  if (cp->ndhwc) {
    // channels-last: the engine's channels-last mode where it applies, else
    // the NCDHW plan of the transposed copies
    if (!stride || !pad || !dil) return TC3D_ERR_NULL;
    Problem pb = make_problem(OP_CONV, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil,
                              out_pad, groups);
    pb.cl = 1;
    rc = make_plan(pb, &cp->pl);
    if (rc == TC3D_OK && !cp->pl.cl) {
      pb.cl = 0;
      rc = make_plan(pb, &cp->pl);
    }
  } else {
    rc = plan_for(op, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil, out_pad, groups,
                  &cp->pl);
  }
  if (rc) return rc;
  cp->upb = make_problem(cp->ndhwc ? OP_CONV : op, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride,
                         pad, dil, out_pad, groups);
  // the direct kernel: grouped convs with few channels per group (the
  // engine's GEMM-N would be mostly padding), and any such conv in
  // channels-last layout
  const Problem& pb = cp->upb;
  if (pb.op == OP_CONV && (pb.groups > 1 || cp->ndhwc))
    cp->direct = direct_eligible(cp->pl.cin_g, cp->pl.cout_g, pb.stride[2], pb.dil[2], pb.k[2]);
  // the algebraic path: always for running statistics; for batch statistics
  // where its statistics run in lag form, or where the fused engine epilogue
  // cannot run (the patch-Gram kernel measured slower than that epilogue on
  // the 64 x 3 x 32^3 workload, and much faster than the full-output fallback)
  cp->pool_ok = is_bn_op(op) && make_pool_plan(cp->pl, &cp->pp) == TC3D_OK;
  cp->pool = cp->pool_ok && (op == OP_CONVT_BN_EVAL || !cp->pl.fused || cp->pp.lag);
  cp->ws_total = cp->pool ? cp->pp.ws_total : cp->pl.ws_total;
  if (cp->direct) {
    cp->ws_total = 256;  // nothing is staged
  } else if (cp->ndhwc && !cp->pl.cl) {
    // channels-last through the engine: x and y transposed to NCDHW copies
    // (the transpose grid: batch in y, 32 x 32 tiles in x)
    const int64_t sv = (int64_t)pb.S[0] * pb.S[1] * pb.S[2];
    const int64_t ov = cp->pl.O[0] * cp->pl.O[1] * cp->pl.O[2];
    auto tiles = [](int64_t a, int64_t b) { return ((a + 31) / 32) * ((b + 31) / 32); };
    if (pb.N > 65535 || tiles(sv, pb.Cin) > INT32_MAX || tiles(pb.Cout, ov) > INT32_MAX)
      return TC3D_ERR_UNSUPPORTED;
    const int64_t xs = (int64_t)pb.N * pb.Cin * pb.S[0] * pb.S[1] * pb.S[2] * 4;
    cp->ws_xt_off = (cp->ws_total + 255) / 256 * 256;
    cp->ws_yt_off = (cp->ws_xt_off + xs + 255) / 256 * 256;
    cp->ws_total = cp->ws_yt_off + cp->pl.y_elems * 4;
  }
  return TC3D_OK;
}

// The direct kernel's parameters for a planned call (data pointers null)
DirectParams direct_params(const CallPlan& cp) {
  const Plan& pl = cp.pl;
  const Problem& pb = cp.upb;
  DirectParams dp;
  std::memset(&dp, 0, sizeof(dp));
  dp.N = pb.N;
  dp.C = pb.Cin;
  dp.Cout = pb.Cout;
  dp.cin_g = pl.cin_g;
  dp.cout_g = pl.cout_g;
  for (int a = 0; a < 3; ++a) {
    dp.S[a] = pb.S[a];
    dp.k[a] = pb.k[a];
    dp.s[a] = pb.stride[a];
    dp.p[a] = pb.pad[a];
    dp.d[a] = pb.dil[a];
    dp.O[a] = (int)pl.O_user[a];
  }
  dp.nrun2 = (dp.O[2] + kDirectRun - 1) / kDirectRun;
  dp.items = (long long)pb.N * pb.Cout * dp.O[0] * dp.O[1] * dp.nrun2;
  return dp;
}

// The direct conv kernel (grouped convs with few channels per group; NCDHW
// or channels-last)
int run_direct(const CallPlan& cp, const float* x, const float* w, const float* bias, float* y,
               DeviceState* d, cudaStream_t st) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!d->direct_smem_set) {
      if (direct_set_smem() != cudaSuccess) return TC3D_ERR_CUDA;
      d->direct_smem_set = true;
    }
  }
  DirectParams dp = direct_params(cp);
  dp.x = x;
  dp.w = w;
  dp.bias = bias;
  dp.y = y;
  return direct_conv_launch(dp, cp.ndhwc, d->sm_count, st) == cudaSuccess ? TC3D_OK
                                                                         : TC3D_ERR_CUDA;
}

// The algebraic BN-pool path: [Gram matrices, their reduction,] finalize
// (statistics, folded weights and bias), weight pack, pooled convolution.
int run_pool(int op, const CallPlan& cp, const float* x, const float* w, const float* bias,
             const BnArgs& bn, float* y, void* ws, DeviceState* d, cudaStream_t st) {
  const Plan& pl = cp.pl;
  const PoolPlan& pp = cp.pp;
  const Problem& pb = pl.pb;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* wpack = reinterpret_cast<float*>(wsb + pp.ws_wpack_off);
  float* w2 = reinterpret_cast<float*>(wsb + pp.ws_w2_off);
  float* b2 = reinterpret_cast<float*>(wsb + pp.ws_b2_off);
  double* gsum = nullptr;
  const float* lrs = nullptr;
  LagParams lp;
  if (op == OP_CONVT_BN_POOL && pp.lag && encode_lag_map(pb, x, &lp)) {
    // batch statistics in lag form: region sums, reduced over the grid
    lp.part = reinterpret_cast<float*>(wsb + pp.ws_lpart_off);
    lp.rs = reinterpret_cast<float*>(wsb + pp.ws_lrs_off);
    lp.err = d->err;
    lp.timeout_cycles = timeout_cycles(g_timeout_ns.load());
    lp.N = pb.N;
    for (int a = 0; a < 3; ++a) {
      lp.L[a] = pb.S[a];
      lp.nseg[a] = pp.lag_nseg[a];
      lp.bulk[a] = pp.lag_bulk[a];
      for (int i = 0; i <= kLagMaxSeg; ++i) lp.seg[a][i] = pp.lag_seg[a][i];
    }
    for (int a = 0; a < 3; ++a) {
      lp.nrange[a] = pp.lag_nrange[a];
      for (int k = 0; k < 4; ++k)
        for (int e = 0; e < 2; ++e) lp.range[a][k][e] = pp.lag_range[a][k][e];
    }
    lp.nbox = pp.lag_nbox;
    lp.nb1 = pp.lag_nb1;
    lp.nb2 = pp.lag_nb2;
    for (int i = 0; i < kLagMaxSeg; ++i) lp.nc[i] = pp.lag_nc[i];
    for (int i = 0; i <= kLagMaxSeg; ++i) lp.cta0[i] = pp.lag_cta0[i];
    lp.grid = pp.lag_grid;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      if (!d->lag_smem_set) {
        if (lag_set_smem() != cudaSuccess) return TC3D_ERR_CUDA;
        d->lag_smem_set = true;
      }
    }
    if (lag_launch(lp, pb.Cin, st) != cudaSuccess) return TC3D_ERR_CUDA;
    lrs = lp.rs;
  } else if (op == OP_CONVT_BN_POOL) {
    GramParams gp;
    std::memset(&gp, 0, sizeof(gp));
    gp.x = x;
    gp.part = reinterpret_cast<float*>(wsb + pp.ws_gpart_off);
    gp.N = pb.N;
    gp.C = pb.Cin;
    gp.D = pp.D;
    gp.V = pp.D / pb.Cin;
    gp.nb = (pp.D + 7) / 8;
    gp.nblk = gp.nb * (gp.nb + 1) / 2;
    for (int a = 0; a < 3; ++a) {
      gp.L[a] = pb.S[a];
      gp.nU[a] = pp.nU[a];
      for (int i = 0; i < kMaxAxisTaps; ++i) gp.U[a][i] = pp.U[a][i];
    }
    gp.nbox = pp.nbox;
    gp.vec16 = aligned(x, 16) && pb.S[2] % 4 == 0;
    // CTAs per box in proportion to its cost, two per SM in all; each box at
    // least 8 and never more than its units
    int64_t cost[kGramMaxBoxes], all = 0;
    for (int b = 0; b < pp.nbox; ++b) {
      for (int a = 0; a < 3; ++a) {
        gp.box_lo[b][a] = pp.box_lo[b][a];
        gp.box_ext[b][a] = pp.box_hi[b][a] - pp.box_lo[b][a];
        gp.box_perm[b][a] = pp.box_perm[b][a];
      }
      gp.box_Tn[b] = pp.box_Tn[b];
      gp.box_T1[b] = pp.box_T1[b];
      gp.box_T2[b] = pp.box_T2[b];
      gp.box_W1[b] = pp.box_W1[b];
      gp.box_W2p[b] = pp.box_W2p[b];
      const int A0 = pp.box_perm[b][0], A1 = pp.box_perm[b][1], A2 = pp.box_perm[b][2];
      gp.box_nt1[b] = (gp.box_ext[b][A1] + pp.box_T1[b] - 1) / pp.box_T1[b];
      gp.box_nt2[b] = (gp.box_ext[b][A2] + pp.box_T2[b] - 1) / pp.box_T2[b];
      gp.box_units[b] = (int64_t)((pb.N + pp.box_Tn[b] - 1) / pp.box_Tn[b]) * gp.box_ext[b][A0] *
                        gp.box_nt1[b] * gp.box_nt2[b];
      // rows, plus the unit's staging: a word per staged slab float, a
      // quarter word where rows move as 16-byte copies
      const int64_t slab = (int64_t)pp.box_Tn[b] * pb.Cin * pp.nU[A0] * pp.box_W1[b] * pp.box_W2p[b];
      const int z2s = pp.box_lo[b][2] + pp.U[2][0];
      const bool v16 = gp.vec16 && A2 == 2 && z2s >= 0 && z2s % 4 == 0 &&
                       (gp.box_nt2[b] == 1 || pp.box_T2[b] % 4 == 0);
      cost[b] = pp.box_rows[b] + gp.box_units[b] * (v16 ? slab / 4 : slab);
      all += cost[b];
    }
    // all CTAs resident at once: two per SM, the per-box minimum of 8 included
    const int64_t budget =
        std::min<int64_t>(kGramMaxCtas, 2LL * d->sm_count) - 8LL * pp.nbox;
    gp.box_cta0[0] = 0;
    for (int b = 0; b < pp.nbox; ++b) {
      // at least 8 CTAs (or one per unit): thin boxes are latency-bound
      const int64_t share = std::max<int64_t>(8, budget * cost[b] / std::max<int64_t>(all, 1));
      gp.box_cta0[b + 1] =
          gp.box_cta0[b] + (int)std::max<int64_t>(1, std::min<int64_t>(gp.box_units[b], share));
    }
    gsum = reinterpret_cast<double*>(wsb + pp.ws_gsum_off);
    {
      std::lock_guard<std::mutex> lk(g_mu);
      if (!d->gram_smem_set) {
        if (gram_set_smem() != cudaSuccess) return TC3D_ERR_CUDA;
        d->gram_smem_set = true;
      }
    }
    if (gram_launch(gp, (unsigned)gp.box_cta0[pp.nbox], st) != cudaSuccess ||
        gram_reduce_launch(gp.part, gp.box_cta0, pp.nbox, pp.cls_coef, pp.ncls, gsum, st) !=
            cudaSuccess)
      return TC3D_ERR_CUDA;
  }
  PoolFinParams fp;
  std::memset(&fp, 0, sizeof(fp));
  fp.w = w;
  fp.bias = bias;
  fp.gamma = bn.gamma;
  fp.beta = bn.beta;
  fp.rmean = bn.rmean;
  fp.rvar = bn.rvar;
  fp.gcls = gsum;
  fp.lrs = lrs;
  // the pooled conv: on CUDA cores where its kernel takes the problem (few
  // channels, at most 3 taps per axis, TMA-loadable x), else through the
  // engine; the finalize writes the summed weights in the layout it reads
  PooledParams pq;
  bool pooled = false;
  {
    int Ke[3], P[3];
    for (int a = 0; a < 3; ++a) {
      Ke[a] = pp.Ke[a];
      P[a] = (int)pl.P[a];
    }
    pooled = pooled_ok(pb.Cin, pb.Cout, Ke, P, pb.N) && encode_pooled_map(pb, x, &pq);
  }
  fp.pooled_layout = pooled ? 1 : 0;
  fp.w2_stride = pooled_coutp(pb.Cout);
  fp.w2 = w2;
  fp.b2 = b2;
  // lag form with the pooled conv: the pooled conv applies the scale, so the
  // summed weights need not wait for the statistics
  fp.s2 = lrs && pooled ? b2 + pb.Cout : nullptr;
  fp.pool_ctr = pooled ? reinterpret_cast<unsigned*>(b2 + 2 * pb.Cout) : nullptr;
  fp.eps = bn.eps;
  fp.count = (double)pb.N * (double)pl.O[0] * (double)pl.O[1] * (double)pl.O[2];
  fp.inv_count = 1.0 / fp.count;
  fp.Cin = pb.Cin;
  fp.Cout = pb.Cout;
  fp.V = pp.D / pb.Cin;
  for (int a = 0; a < 3; ++a) {
    fp.k[a] = pb.k[a];
    fp.pad[a] = pb.pad[a];
    fp.dil[a] = pb.dil[a];
    fp.nU[a] = pp.nU[a];
    fp.e_min[a] = pp.e_min[a];
    fp.Ke[a] = pp.Ke[a];
    for (int r = 0; r < 2; ++r) {
      fp.ntap[a][r] = pp.ntap[a][r];
      for (int i = 0; i < kMaxAxisTaps; ++i) {
        fp.tap_k[a][r][i] = pp.tap_k[a][r][i];
        fp.tap_u[a][r][i] = pp.tap_u[a][r][i];
      }
    }
  }
  // summed taps: bit k of wkmask[a][e] iff 0 <= 2 (e_min + e) - p + d k <= 3
  for (int a = 0; a < 3; ++a)
    for (int e = 0; e < kMaxAxisTaps; ++e) {
      unsigned m = 0;
      if (e < pp.Ke[a])
        for (int k = 0; k < pb.k[a]; ++k) {
          const int j = 2 * (pp.e_min[a] + e) - pb.pad[a] + pb.dil[a] * k;
          if (j >= 0 && j <= 3) m |= 1u << k;
        }
      fp.wkmask[a][e] = m;
    }
  fp.ncls = pp.ncls;
  // the class entries: (ci, taps t0, t1, t2) in patch order of the class
  fp.ent_off[0] = 0;
  for (int c = 0; c < pp.ncls; ++c) {
    const int r0 = pp.cls_r[c][0], r1 = pp.cls_r[c][1], r2 = pp.cls_r[c][2];
    const int n0 = pp.ntap[0][r0], n1 = pp.ntap[1][r1], n2 = pp.ntap[2][r2];
    int row = fp.ent_off[c];
    for (int ci = 0; ci < pb.Cin; ++ci)
      for (int t0 = 0; t0 < n0; ++t0)
        for (int t1 = 0; t1 < n1; ++t1)
          for (int t2 = 0; t2 < n2; ++t2, ++row) {
            const int v0 = pp.tap_u[0][r0][t0], v1 = pp.tap_u[1][r1][t1], v2 = pp.tap_u[2][r2][t2];
            fp.ent_d[row] = ci * fp.V + (v0 * pp.nU[1] + v1) * pp.nU[2] + v2;
            fp.ent_w[row] = ((ci * pb.k[0] + pp.tap_k[0][r0][t0]) * pb.k[1] + pp.tap_k[1][r1][t1]) *
                                pb.k[2] +
                            pp.tap_k[2][r2][t2];
            fp.ent_cv[row] = ci | v0 << 4 | v1 << 8 | v2 << 12;
            fp.ent_box[row] = pp.lag ? (pp.lag_ridx[0][r0][v0] * pp.lag_nrange[1] +
                                        pp.lag_ridx[1][r1][v1]) *
                                               pp.lag_nrange[2] +
                                           pp.lag_ridx[2][r2][v2]
                                     : 0;
          }
    fp.ent_off[c + 1] = row;
  }
  for (int c = 0; c < 8; ++c)
    for (int a = 0; a < 3; ++a) fp.cls_r[c][a] = pp.cls_r[c][a];
  if (lrs) {
    // the lag kernel's box sums, reduced; then the finalize, a CTA per channel
    if (lag_finalize_launch(fp, lp.part, lp.grid, lp.nbox * kLagSlots, st) != cudaSuccess)
      return TC3D_ERR_CUDA;
  } else if (pool_finalize_launch(fp, st) != cudaSuccess) {
    return TC3D_ERR_CUDA;
  }
  if (pooled) {
    pq.w2 = w2;
    pq.b2 = b2;
    pq.s2 = fp.s2;
    pq.ctr = fp.pool_ctr;
    pq.y = y;
    pq.err = d->err;
    pq.timeout_cycles = timeout_cycles(g_timeout_ns.load());
    pq.N = pb.N;
    pq.Cin = pb.Cin;
    pq.Cout = pb.Cout;
    pq.coutp = pooled_coutp(pb.Cout);
    for (int a = 0; a < 3; ++a) {
      pq.P[a] = (int)pl.P[a];
      pq.pad[a] = -pp.e_min[a];
    }
    pq.nq1b = (pq.P[1] + kPooledRows - 1) / kPooledRows;
    pq.nq2b = (pq.P[2] + kPooledQ2 - 1) / kPooledQ2;
    return pooled_launch(pq, d->sm_count, st) == cudaSuccess ? TC3D_OK : TC3D_ERR_CUDA;
  }
  int rc = launch_pack(pp.cplan, w2, wpack, d->sm_count, st);
  if (rc) return rc;
  return launch_engine(pp.cplan, pp.cplan.epi, x, wpack, b2, y, nullptr, d, st);
}

int run(int op, const float* x, const float* w, const float* bias, const BnArgs& bn, float* y,
        int N, int Cin, int S0, int S1, int S2, int Cout, int k0, int k1, int k2,
        const int stride[3], const int pad[3], const int dil[3], const int out_pad[3],
        int groups, void* ws, size_t ws_bytes, cudaStream_t st) {
  CallPlan cp;
  int rc = plan_call(op, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil, out_pad, groups,
                     &cp);
  if (rc) return rc;
  const Plan& pl = cp.pl;
  const float* gamma = bn.gamma;
  const float* beta = bn.beta;
  const float eps = bn.eps;
  if (is_bn_op(op) && !(eps >= 0.0f)) return TC3D_ERR_SHAPE;
  if (op == OP_CONVT_BN_EVAL && (!bn.rmean || !bn.rvar)) return TC3D_ERR_NULL;
  rc = common_checks(x, w, y, bias, ws, ws_bytes, cp.ws_total);
  if (rc) return rc;
  if ((gamma && !aligned(gamma, 4)) || (beta && !aligned(beta, 4)) ||
      (bn.rmean && !aligned(bn.rmean, 4)) || (bn.rvar && !aligned(bn.rvar, 4)))
    return TC3D_ERR_ALIGN;
  DeviceState* d = nullptr;
  rc = device_state(&d);
  if (rc) return rc;
  if (cp.pool) return run_pool(op, cp, x, w, bias, bn, y, ws, d, st);
  if (cp.direct) return run_direct(cp, x, w, bias, y, d, st);
  if (cp.ndhwc && !cp.pl.cl) {
    // channels-last through the engine: x -> NCDHW, the conv, y -> NDHWC
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    float* xt = reinterpret_cast<float*>(wsb + cp.ws_xt_off);
    float* yt = reinterpret_cast<float*>(wsb + cp.ws_yt_off);
    const Problem& pb = pl.pb;
    const long long sv = (long long)pb.S[0] * pb.S[1] * pb.S[2];
    const long long ov = (long long)pl.O[0] * pl.O[1] * pl.O[2];
    if (transpose_launch(x, xt, pb.N, sv, pb.Cin, st) != cudaSuccess) return TC3D_ERR_CUDA;
    float* wpack = reinterpret_cast<float*>(wsb + pl.ws_wpack_off);
    rc = launch_pack(pl, w, wpack, d->sm_count, st);
    if (rc) return rc;
    rc = launch_engine(pl, pl.epi, xt, wpack, bias, yt, nullptr, d, st);
    if (rc) return rc;
    return transpose_launch(yt, y, pb.N, pb.Cout, ov, st) == cudaSuccess ? TC3D_OK
                                                                         : TC3D_ERR_CUDA;
  }
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* wpack = reinterpret_cast<float*>(wsb + pl.ws_wpack_off);
  // the bias fill (a transposed conv's tap-less outputs) runs inside the engine
  unsigned long long* ctr =
      pl.fill_slab ? reinterpret_cast<unsigned long long*>(wsb + pl.ws_ctr_off) : nullptr;
  rc = launch_pack(pl, w, wpack, d->sm_count, st, ctr);
  if (rc) return rc;
  if (!is_bn_op(op)) return launch_engine(pl, pl.epi, x, wpack, bias, y, nullptr, d, st, nullptr, ctr);

  float2* stat = reinterpret_cast<float2*>(wsb + pl.ws_stat_off);
  const long long pvol = (long long)pl.P[0] * pl.P[1] * pl.P[2];
  const unsigned blocks =
      (unsigned)std::min<long long>((pl.y_elems + 255) / 256, (long long)d->sm_count * 8);
  if (op == OP_CONVT_BN_EVAL) {
    // running statistics: the affine map is known before the convolution,
    // so the fused epilogue stores final values (bias folded into the shift)
    if (bn_eval_affine_launch(bn.rmean, bn.rvar, gamma, beta, pl.fused ? bias : nullptr, eps,
                              Cout, stat, st) != cudaSuccess)
      return TC3D_ERR_CUDA;
    if (pl.fused) return launch_engine(pl, EPI_BN_POOL, x, wpack, bias, y, nullptr, d, st, stat);
    float* full = reinterpret_cast<float*>(wsb + pl.ws_full_off);
    rc = launch_engine(pl, EPI_STORE, x, wpack, bias, full, nullptr, d, st, nullptr, ctr);
    if (rc) return rc;
    const int O[3] = {(int)pl.O[0], (int)pl.O[1], (int)pl.O[2]};
    const int P[3] = {(int)pl.P[0], (int)pl.P[1], (int)pl.P[2]};
    return bn_pool4_launch(full, y, N, Cout, O, P, stat, blocks, st) == cudaSuccess
               ? TC3D_OK
               : TC3D_ERR_CUDA;
  }
  if (pl.fused) {
    float2* part = reinterpret_cast<float2*>(wsb + pl.ws_part_off);
    rc = launch_engine(pl, EPI_BN_POOL, x, wpack, bias, y, part, d, st);
    if (rc) return rc;
    const double count = (double)N * (double)pl.O[0] * (double)pl.O[1] * (double)pl.O[2];
    const int slots = (int)bn_part_slots(pl, engine_grid(pl, d->sm_count));
    if (bn_stats_f2_launch(part, slots, bias, gamma, beta, count, eps, Cout, stat, st) !=
            cudaSuccess ||
        bn_apply_launch(y, pl.y_elems, pvol, Cout, stat, blocks, st) != cudaSuccess)
      return TC3D_ERR_CUDA;
  } else {
    float* full = reinterpret_cast<float*>(wsb + pl.ws_full_off);
    double* part2 = reinterpret_cast<double*>(wsb + pl.ws_part_off);
    rc = launch_engine(pl, EPI_STORE, x, wpack, bias, full, nullptr, d, st, nullptr, ctr);
    if (rc) return rc;
    const int O[3] = {(int)pl.O[0], (int)pl.O[1], (int)pl.O[2]};
    const int P[3] = {(int)pl.P[0], (int)pl.P[1], (int)pl.P[2]};
    if (bn_unfused_launch(full, y, part2, N, Cout, O, P, gamma, beta, eps, stat, blocks, st) !=
        cudaSuccess)
      return TC3D_ERR_CUDA;
  }
  return TC3D_OK;
}

void append(std::string& s, const char* fmt, long long v) {
  char b[96];
  snprintf(b, sizeof(b), fmt, v);
  s += b;
}

std::string describe(const Plan& pl) {
  std::string s = "{";
  append(s, "\"status\": %lld", pl.status);
  if (pl.status == TC3D_OK) {
    auto arr3 = [&](const char* name, const long long v0, long long v1, long long v2) {
      char b[160];
      snprintf(b, sizeof(b), ", \"%s\": [%lld, %lld, %lld]", name, v0, v1, v2);
      s += b;
    };
    arr3("O", pl.O[0], pl.O[1], pl.O[2]);
    arr3("P", pl.P[0], pl.P[1], pl.P[2]);
    arr3("M", pl.M[0], pl.M[1], pl.M[2]);
    arr3("s_in", pl.s_in[0], pl.s_in[1], pl.s_in[2]);
    arr3("s_out", pl.s_out[0], pl.s_out[1], pl.s_out[2]);
    arr3("u_min", pl.u_min[0], pl.u_min[1], pl.u_min[2]);
    arr3("Q", pl.Q[0], pl.Q[1], pl.Q[2]);
    arr3("Pq", pl.Pq[0], pl.Pq[1], pl.Pq[2]);
    arr3("T", pl.T[0], pl.T[1], pl.T[2]);
    arr3("box", pl.box[0], pl.box[1], pl.box[2]);
    // per-axis offsets u (absolute) and tap tables kidx[class][offset]
    s += ", \"axes\": [";
    for (int a = 0; a < 3; ++a) {
      if (a) s += ", ";
      s += "{\"u\": [";
      for (int t = 0; t < pl.nU[a]; ++t) {
        if (t) s += ", ";
        append(s, "%lld", pl.u_rel[a][t] + pl.u_min[a]);
      }
      s += "], \"classes\": [";
      for (int r = 0; r < pl.nRaxis[a]; ++r) {
        if (r) s += ", ";
        append(s, "%lld", pl.r_axis[a][r]);
      }
      s += "], \"kidx\": [";
      for (int r = 0; r < pl.nRaxis[a]; ++r) {
        if (r) s += ", ";
        s += "[";
        for (int t = 0; t < pl.nU[a]; ++t) {
          if (t) s += ", ";
          append(s, "%lld", pl.kidx[a][r][t]);
        }
        s += "]";
      }
      s += "]}";
    }
    s += "]";
    append(s, ", \"epi\": %lld", pl.epi);
    append(s, ", \"fused\": %lld", pl.fused);
    append(s, ", \"nR\": %lld", pl.nR);
    append(s, ", \"nEmpty\": %lld", pl.nEmpty);
    append(s, ", \"fill_slab\": %lld", pl.fill_slab);
    append(s, ", \"fill_rows\": %lld", pl.fill_rows);
    append(s, ", \"xslack\": %lld", pl.xslack);
    append(s, ", \"ocb\": %lld", pl.ocb);
    append(s, ", \"n_tile\": %lld", pl.n_tile);
    append(s, ", \"n_colblocks\": %lld", pl.n_colblocks);
    append(s, ", \"n_acc\": %lld", pl.n_acc);
    append(s, ", \"dbuf\": %lld", pl.dbuf);
    append(s, ", \"a_stages\": %lld", pl.a_stages);
    append(s, ", \"ks_stage\": %lld", pl.ks_stage);
    append(s, ", \"view\": %lld", pl.view);
    append(s, ", \"cl\": %lld", pl.cl);
    append(s, ", \"cl_cb\": %lld", pl.cl_cb);
    append(s, ", \"reshaped\": %lld", pl.reshaped);
    append(s, ", \"nslots\": %lld", pl.nslots);
    append(s, ", \"slot_bytes\": %lld", pl.slot_bytes);
    append(s, ", \"wide\": %lld", pl.wide);
    append(s, ", \"acc_cols\": %lld", pl.acc_cols);
    append(s, ", \"tiles\": %lld", pl.tiles);
    append(s, ", \"cin_chunk\": %lld", pl.cin_chunk);
    append(s, ", \"n_chunks\": %lld", pl.n_chunks);
    append(s, ", \"k_chunk\": %lld", pl.k_chunk);
    append(s, ", \"ksteps_chunk\": %lld", pl.ksteps_chunk);
    append(s, ", \"raw_stages\": %lld", pl.raw_stages);
    append(s, ", \"raw_stage_bytes\": %lld", pl.raw_stage_bytes);
    append(s, ", \"b_resident\": %lld", pl.b_resident);
    append(s, ", \"b_stages\": %lld", pl.b_stages);
    append(s, ", \"b_stage_bytes\": %lld", pl.b_stage_bytes);
    append(s, ", \"smem_bytes\": %lld", pl.smem_bytes);
    append(s, ", \"ws_total\": %lld", pl.ws_total);
    append(s, ", \"y_elems\": %lld", pl.y_elems);
  }
  s += "}";
  return s;
}

}  // namespace

extern "C" {

int tc3d_conv3d_fwd(const float* x, const float* w, const float* bias, float* y, int N, int Cin,
                    int S0, int S1, int S2, int Cout, int k0, int k1, int k2, const int stride[3],
                    const int pad[3], const int dilation[3], const int output_padding[3],
                    int groups, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return run(OP_CONV, x, w, bias, BnArgs(), y, N, Cin, S0, S1, S2, Cout, k0, k1, k2,
             stride, pad, dilation, output_padding, groups, workspace, workspace_bytes, stream);
}

int tc3d_conv_transpose3d_fwd(const float* x, const float* w, const float* bias, float* y, int N,
                              int Cin, int S0, int S1, int S2, int Cout, int k0, int k1, int k2,
                              const int stride[3], const int pad[3], const int dilation[3],
                              const int output_padding[3], int groups, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  return run(OP_CONVT, x, w, bias, BnArgs(), y, N, Cin, S0, S1, S2, Cout, k0, k1,
             k2, stride, pad, dilation, output_padding, groups, workspace, workspace_bytes,
             stream);
}

int tc3d_conv_maxpool_lse_relu(const float* x, const float* w, const float* bias, float* y, int N,
                               int Cin, int S0, int S1, int S2, int Cout, int k0, int k1, int k2,
                               const int stride[3], const int pad[3], const int dilation[3],
                               const int output_padding[3], int groups, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  return run(OP_CONV_POOL_LSE, x, w, bias, BnArgs(), y, N, Cin, S0, S1, S2, Cout,
             k0, k1, k2, stride, pad, dilation, output_padding, groups, workspace,
             workspace_bytes, stream);
}

int tc3d_convT_bn_avgpool(const float* x, const float* w, const float* bias, const float* gamma,
                          const float* beta, float eps, float* y, int N, int Cin, int S0, int S1,
                          int S2, int Cout, int k0, int k1, int k2, const int stride[3],
                          const int pad[3], const int dilation[3], const int output_padding[3],
                          int groups, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  BnArgs bn;
  bn.gamma = gamma;
  bn.beta = beta;
  bn.eps = eps;
  return run(OP_CONVT_BN_POOL, x, w, bias, bn, y, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride,
             pad, dilation, output_padding, groups, workspace, workspace_bytes, stream);
}

int tc3d_convT_bneval_avgpool(const float* x, const float* w, const float* bias,
                              const float* running_mean, const float* running_var,
                              const float* gamma, const float* beta, float eps, float* y, int N,
                              int Cin, int S0, int S1, int S2, int Cout, int k0, int k1, int k2,
                              const int stride[3], const int pad[3], const int dilation[3],
                              const int output_padding[3], int groups, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  BnArgs bn;
  bn.gamma = gamma;
  bn.beta = beta;
  bn.rmean = running_mean;
  bn.rvar = running_var;
  bn.eps = eps;
  return run(OP_CONVT_BN_EVAL, x, w, bias, bn, y, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride,
             pad, dilation, output_padding, groups, workspace, workspace_bytes, stream);
}

int tc3d_conv3d_fwd_ndhwc(const float* x, const float* w, const float* bias, float* y, int N,
                          int Cin, int S0, int S1, int S2, int Cout, int k0, int k1, int k2,
                          const int stride[3], const int pad[3], const int dilation[3],
                          const int output_padding[3], int groups, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  return run(OP_CONV_NDHWC, x, w, bias, BnArgs(), y, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride,
             pad, dilation, output_padding, groups, workspace, workspace_bytes, stream);
}

int tc3d_workspace_bytes(int op, int N, int Cin, int S0, int S1, int S2, int Cout, int k0, int k1,
                         int k2, const int stride[3], const int pad[3], const int dilation[3],
                         const int output_padding[3], int groups, size_t* bytes) {
  if (!bytes) return TC3D_ERR_NULL;
  CallPlan cp;
  int rc = plan_call(op, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dilation,
                     output_padding, groups, &cp);
  if (rc) return rc;
  *bytes = (size_t)cp.ws_total;
  return TC3D_OK;
}

int tc3d_out_shape(int op, int N, int Cin, int S0, int S1, int S2, int Cout, int k0, int k1,
                   int k2, const int stride[3], const int pad[3], const int dilation[3],
                   const int output_padding[3], int groups, int64_t out_dims[5]) {
  if (!out_dims) return TC3D_ERR_NULL;
  CallPlan cp;
  int rc = plan_call(op, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dilation,
                     output_padding, groups, &cp);
  if (rc) return rc;
  const Plan& pl = cp.pl;
  out_dims[0] = N;
  if (op == OP_CONV_NDHWC) {  // channels-last y: [N, O0, O1, O2, Cout]
    for (int a = 0; a < 3; ++a) out_dims[1 + a] = pl.O_user[a];
    out_dims[4] = Cout;
  } else if (op == OP_CONV || op == OP_CONVT) {
    out_dims[1] = Cout;
    for (int a = 0; a < 3; ++a) out_dims[2 + a] = pl.O_user[a];
  } else {
    out_dims[1] = op == OP_CONV_POOL_LSE ? 1 : Cout;
    for (int a = 0; a < 3; ++a) out_dims[2 + a] = pl.P[a];
  }
  return TC3D_OK;
}

int tc3d_plan_describe(int op, int N, int Cin, int S0, int S1, int S2, int Cout, int k0, int k1,
                       int k2, const int stride[3], const int pad[3], const int dilation[3],
                       const int output_padding[3], int groups, char* buf, size_t buflen) {
  CallPlan cp;
  int rc = plan_call(op, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dilation,
                     output_padding, groups, &cp);
  Plan& pl = cp.pl;
  if (rc == TC3D_ERR_NULL) pl.status = rc;
  if (buf && buflen) {
    std::string s = describe(pl);
    if (pl.status == TC3D_OK && (op == OP_CONV || op == OP_CONV_NDHWC)) {
      s.pop_back();
      append(s, ", \"direct\": %lld", cp.direct ? 1 : 0);
      append(s, ", \"direct_form\": %lld",
             cp.direct ? (long long)direct_form(direct_params(cp), cp.ndhwc) : -1LL);
      append(s, ", \"ndhwc\": %lld", cp.ndhwc ? 1 : 0);
      s += "}";
    }
    if (pl.status == TC3D_OK && is_bn_op(op)) {
      // the algebraic path: patch size, boxes, classes, the pooled conv
      s.pop_back();
      append(s, ", \"pool_path\": %lld", cp.pool ? 1 : 0);
      append(s, ", \"pool_ok\": %lld", cp.pool_ok ? 1 : 0);
      if (cp.pool_ok) {
        const PoolPlan& pp = cp.pp;
        append(s, ", \"pool_D\": %lld", pp.D);
        append(s, ", \"pool_nbox\": %lld", pp.nbox);
        append(s, ", \"pool_ncls\": %lld", pp.ncls);
        char b[160];
        snprintf(b, sizeof(b), ", \"pool_M\": [%d, %d, %d], \"pool_Ke\": [%d, %d, %d]", pp.M[0],
                 pp.M[1], pp.M[2], pp.Ke[0], pp.Ke[1], pp.Ke[2]);
        s += b;
        snprintf(b, sizeof(b), ", \"pool_e_min\": [%d, %d, %d]", pp.e_min[0], pp.e_min[1],
                 pp.e_min[2]);
        s += b;
        append(s, ", \"pool_conv_tiles\": %lld", pp.cplan.tiles);
        // tables: offsets U, per axis and class the (tap, offset index)
        // pairs, the boxes, and per class its sign on each box
        s += ", \"pool_U\": [";
        for (int a = 0; a < 3; ++a) {
          s += a ? ", [" : "[";
          for (int i = 0; i < pp.nU[a]; ++i) append(s, i ? ", %lld" : "%lld", pp.U[a][i]);
          s += "]";
        }
        s += "], \"pool_taps\": [";
        for (int a = 0; a < 3; ++a) {
          s += a ? ", [" : "[";
          for (int r = 0; r < 2; ++r) {
            s += r ? ", [" : "[";
            for (int i = 0; i < pp.ntap[a][r]; ++i) {
              snprintf(b, sizeof(b), "%s[%d, %d]", i ? ", " : "", pp.tap_k[a][r][i],
                       pp.tap_u[a][r][i]);
              s += b;
            }
            s += "]";
          }
          s += "]";
        }
        s += "], \"pool_boxes\": [";
        for (int i = 0; i < pp.nbox; ++i) {
          snprintf(b, sizeof(b), "%s[%d, %d, %d, %d, %d, %d]", i ? ", " : "", pp.box_lo[i][0],
                   pp.box_lo[i][1], pp.box_lo[i][2], pp.box_hi[i][0], pp.box_hi[i][1],
                   pp.box_hi[i][2]);
          s += b;
        }
        append(s, "], \"lag\": %lld", pp.lag);
        if (pp.lag) {
          append(s, ", \"lag_grid\": %lld", pp.lag_grid);
          append(s, ", \"lag_nb\": [%lld", pp.lag_nb1);
          append(s, ", %lld]", pp.lag_nb2);
          s += ", \"lag_seg\": [";
          for (int a = 0; a < 3; ++a) {
            s += a ? ", [" : "[";
            for (int i = 0; i <= pp.lag_nseg[a]; ++i) append(s, i ? ", %lld" : "%lld", pp.lag_seg[a][i]);
            s += "]";
          }
          append(s, "], \"lag_bulk\": [%lld", pp.lag_bulk[0]);
          append(s, ", %lld", pp.lag_bulk[1]);
          append(s, ", %lld]", pp.lag_bulk[2]);
          s += ", \"lag_nc\": [";
          for (int i = 0; i < pp.lag_nseg[0]; ++i) append(s, i ? ", %lld" : "%lld", pp.lag_nc[i]);
          s += "], \"lag_cta0\": [";
          for (int i = 0; i <= pp.lag_nseg[0]; ++i) append(s, i ? ", %lld" : "%lld", pp.lag_cta0[i]);
          // per axis, class value r and offset index: [segment lo, hi)
          s += "], \"lag_srange\": [";
          for (int a = 0; a < 3; ++a) {
            s += a ? ", [" : "[";
            for (int r = 0; r < 2; ++r) {
              s += r ? ", [" : "[";
              for (int i = 0; i < pp.nU[a]; ++i) {
                snprintf(b, sizeof(b), "%s[%d, %d]", i ? ", " : "", pp.lag_srange[a][r][i][0],
                         pp.lag_srange[a][r][i][1]);
                s += b;
              }
              s += "]";
            }
            s += "]";
          }
          s += "]";
        }
        s += ", \"pool_cls\": [";
        for (int c = 0; c < pp.ncls; ++c) {
          snprintf(b, sizeof(b), "%s[[%d, %d, %d], [", c ? ", " : "", pp.cls_r[c][0],
                   pp.cls_r[c][1], pp.cls_r[c][2]);
          s += b;
          for (int i = 0; i < pp.nbox; ++i) append(s, i ? ", %lld" : "%lld", pp.cls_coef[c][i]);
          s += "]]";
        }
        s += "]";
      }
      s += "}";
    }
    size_t n = std::min(buflen - 1, s.size());
    std::memcpy(buf, s.data(), n);
    buf[n] = 0;
  }
  return rc;
}

int tc3d_last_device_error(cudaStream_t stream) {
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return TC3D_ERR_CUDA;
  int flag = 0, zero = 0;
  if (cudaMemcpy(&flag, d->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return TC3D_ERR_CUDA;
  if (flag && cudaMemcpy(d->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return TC3D_ERR_CUDA;
  return flag ? TC3D_ERR_DEVICE_TIMEOUT : TC3D_OK;
}

void tc3d_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : kDefaultTimeoutNs); }

int tc3d_selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream) {
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  if (wait_timeout_launch(d->err, timeout_cycles(timeout_ns), stream) != cudaSuccess)
    return TC3D_ERR_CUDA;
  return tc3d_last_device_error(stream);
}

const char* tc3d_status_string(int status) {
  switch (status) {
    case TC3D_OK: return "ok";
    case TC3D_ERR_NULL: return "a required pointer is NULL";
    case TC3D_ERR_SHAPE: return "non-positive size or empty output";
    case TC3D_ERR_GROUPS: return "channels not divisible by groups";
    case TC3D_ERR_OUTPUT_PADDING: return "output_padding out of range";
    case TC3D_ERR_ALIGN: return "misaligned pointer";
    case TC3D_ERR_WORKSPACE: return "workspace missing or too small";
    case TC3D_ERR_UNSUPPORTED: return "outside the implemented limits";
    case TC3D_ERR_CUDA: return "CUDA runtime error";
    case TC3D_ERR_DEVICE_TIMEOUT: return "a device-side wait ran out of time";
    case TC3D_ERR_DEVICE: return "device is not compute capability 10.3 (sm_103a)";
    default: return "unknown status";
  }
}

}  // extern "C"
