// gdn_rmsnorm.cu -- the gated RMSNorm epilogue on the core's output o ("linear attention
// cp #1035", section "What does this PR do": the output goes through RMSNorm, the gate and
// the output projection; the test report names the module "RMSNormGated").  Per row of D
// elements (one token and V head), with r = 1 / sqrt(mean(o^2) + eps) and n = o r:
//   y  = n w silu(z)
//   dn = dy w silu(z),  do = r (dn - n mean(dn n)),  dz = dy n w silu'(z),
//   dw = sum over rows of dy n silu(z)
// A warp owns a row (4 adjacent elements per lane and 128-element chunk, one 8- or
// 16-byte access each); the row's sums are warp reductions.  Bandwidth-bound.  The
// backward runs a fixed grid of at most RN_BCTAS CTAs (4 per SM of a 152-SM GPU, all
// resident at once for D <= 128) whose warps stride over the rows two at a time (the loads of both
// rows issued together) and keep their lane's dw terms in registers; per-CTA partials
// (8 warps in a fixed order), then a column-parallel fp64 sum over the CTAs in a fixed
// order.  The CTA count depends only on the row count, so dw is deterministic.
#include <cuda_bf16.h>
#include <string.h>

#include "gdn.h"
#include "gdn_vec.cuh"

namespace gdn {
namespace {

using namespace vec;

constexpr int RN_NT = 256;      // 8 warps
constexpr int RN_FROWS = 4;     // rows per warp, forward (their loads issued together)
constexpr int RN_BROWS = 2;     // rows per warp and step, backward (loads issued together)
constexpr int RN_BCTAS = 608;   // CTAs of the backward at most
constexpr int RN_MAXD = 512;    // 4 chunks of 128 elements

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct RnArgs {
  int64_t rows;
  int D;
  float eps;
  const void* o;
  const void* z;
  const float* w;
  const void* dy;
  void* out0;   // y, or do
  void* out1;   // dz
  float* part;  // [CTAs][D] partial dw
};

// NV: 128-element chunks per row
template <int NV, typename T>
__global__ void __launch_bounds__(RN_NT) k_rmsnorm_gated_fwd(RnArgs ar) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t r0 = ((int64_t)blockIdx.x * (RN_NT / 32) + warp) * RN_FROWS;
  float o[RN_FROWS][NV][4], z[RN_FROWS][NV][4];
#pragma unroll
  for (int q = 0; q < RN_FROWS; ++q)
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int e = k * 128 + lane * 4;
      const bool ok = r0 + q < ar.rows && e < ar.D;
      const int64_t off = (r0 + q) * ar.D + e;
#pragma unroll
      for (int j = 0; j < 4; ++j) o[q][k][j] = z[q][k][j] = 0.f;
      if (ok) {
        ld4(reinterpret_cast<const T*>(ar.o) + off, o[q][k]);
        ld4(reinterpret_cast<const T*>(ar.z) + off, z[q][k]);
      }
    }
#pragma unroll
  for (int q = 0; q < RN_FROWS; ++q) {
    if (r0 + q >= ar.rows) break;
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int j = 0; j < 4; ++j) ss = fmaf(o[q][k][j], o[q][k][j], ss);
    const float r = rsqrtf(warp_sum(ss) / (float)ar.D + ar.eps);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int e = k * 128 + lane * 4;
      if (e >= ar.D) continue;
      float w[4], y[4];
      ld4(ar.w + e, w);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float zz = z[q][k][j];
        y[j] = o[q][k][j] * r * w[j] * (zz * sigm(zz));
      }
      st4(reinterpret_cast<T*>(ar.out0) + (r0 + q) * ar.D + e, y);
    }
  }
}

template <int NV, typename T>
__global__ void __launch_bounds__(RN_NT, NV == 1 ? 4 : 1) k_rmsnorm_gated_bwd(RnArgs ar) {
  __shared__ float red[RN_NT / 32][RN_MAXD];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t step = (int64_t)gridDim.x * (RN_NT / 32) * RN_BROWS;
  float dwa[NV][4], w[NV][4];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int e = k * 128 + lane * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) dwa[k][j] = w[k][j] = 0.f;
    if (e < ar.D) ld4(ar.w + e, w[k]);
  }
  for (int64_t r0 = ((int64_t)blockIdx.x * (RN_NT / 32) + warp) * RN_BROWS; r0 < ar.rows;
       r0 += step) {
    float o[RN_BROWS][NV][4], z[RN_BROWS][NV][4], g[RN_BROWS][NV][4];
#pragma unroll
    for (int q = 0; q < RN_BROWS; ++q)
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int e = k * 128 + lane * 4;
#pragma unroll
        for (int j = 0; j < 4; ++j) o[q][k][j] = z[q][k][j] = g[q][k][j] = 0.f;
        if (r0 + q < ar.rows && e < ar.D) {
          const int64_t off = (r0 + q) * ar.D + e;
          ld4(reinterpret_cast<const T*>(ar.o) + off, o[q][k]);
          ld4(reinterpret_cast<const T*>(ar.z) + off, z[q][k]);
          ld4(reinterpret_cast<const T*>(ar.dy) + off, g[q][k]);
        }
      }
#pragma unroll
    for (int q = 0; q < RN_BROWS; ++q) {
      const int64_t row = r0 + q;
      if (row >= ar.rows) break;
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) ss = fmaf(o[q][k][j], o[q][k][j], ss);
      const float r = rsqrtf(warp_sum(ss) / (float)ar.D + ar.eps);
      // n = o r (kept in o), dn = dy w silu(z) (kept in g); dz needs dy n w silu'(z)
      float dzv[NV][4], dot = 0.f;
#pragma unroll
      for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float n = o[q][k][j] * r, zz = z[q][k][j], s = sigm(zz), sl = zz * s,
                      dy = g[q][k][j];
          dwa[k][j] = fmaf(dy * n, sl, dwa[k][j]);
          dzv[k][j] = dy * n * w[k][j] * s * (1.f + zz * (1.f - s));
          o[q][k][j] = n;
          g[q][k][j] = dy * w[k][j] * sl;
          dot = fmaf(g[q][k][j], n, dot);
        }
      const float m = warp_sum(dot) / (float)ar.D;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int e = k * 128 + lane * 4;
        if (e >= ar.D) continue;
        float d[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) d[j] = r * (g[q][k][j] - o[q][k][j] * m);
        const int64_t off = row * ar.D + e;
        st4(reinterpret_cast<T*>(ar.out0) + off, d);
        st4(reinterpret_cast<T*>(ar.out1) + off, dzv[k]);
      }
    }
  }
  // this CTA's dw: its 8 warps added in order
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int e = k * 128 + lane * 4;
    if (e < ar.D)
#pragma unroll
      for (int j = 0; j < 4; ++j) red[warp][e + j] = dwa[k][j];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < ar.D; e += RN_NT) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < RN_NT / 32; ++q) s += red[q][e];
    ar.part[(int64_t)blockIdx.x * ar.D + e] = s;
  }
}

// dw[e] = sum over the n_part CTA partials, in fp64: 32 columns per CTA, warp w adds the
// partials w, w + 8, ... in order, then warp 0 adds the 8 warp sums in order.
__global__ void __launch_bounds__(256) k_rmsnorm_reduce(int64_t n_part, int D,
                                                        const float* __restrict__ part,
                                                        float* dw) {
  __shared__ double acc[8][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  double s = 0.0;
  if (e < D)
    for (int64_t p = warp; p < n_part; p += 8) s += part[p * D + e];
  acc[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && e < D) {
    double t = 0.0;
#pragma unroll
    for (int q = 0; q < 8; ++q) t += acc[q][lane];
    dw[e] = (float)t;
  }
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

gdn_status check_problem(const gdn_rmsnorm_problem* p) {
  if (!p) return GDN_ERR_INVALID_ARG;
  if (p->dtype != GDN_BF16 && p->dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
  if (p->rows < 0 || p->D < 1 || !(p->eps >= 0.f) || p->rows > ((int64_t)1 << 34))
    return GDN_ERR_INVALID_ARG;
  if (p->D % 4 != 0 || p->D > RN_MAXD) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

int64_t bwd_ctas(const gdn_rmsnorm_problem* p) {
  const int64_t per = (RN_NT / 32) * RN_BROWS;
  const int64_t n = (p->rows + per - 1) / per;
  return n < RN_BCTAS ? n : RN_BCTAS;
}

template <typename T, int NV>
cudaError_t launch_fwd(const RnArgs& ar, cudaStream_t st) {
  const int64_t per = (RN_NT / 32) * RN_FROWS;
  k_rmsnorm_gated_fwd<NV, T><<<(unsigned)((ar.rows + per - 1) / per), RN_NT, 0, st>>>(ar);
  return cudaGetLastError();
}
template <typename T, int NV>
cudaError_t launch_bwd(const RnArgs& ar, int64_t ctas, cudaStream_t st) {
  k_rmsnorm_gated_bwd<NV, T><<<(unsigned)ctas, RN_NT, 0, st>>>(ar);
  return cudaGetLastError();
}
template <typename T>
cudaError_t launch_fwd_t(const RnArgs& ar, cudaStream_t st) {
  switch ((ar.D + 127) / 128) {
    case 1: return launch_fwd<T, 1>(ar, st);
    case 2: return launch_fwd<T, 2>(ar, st);
    case 3: return launch_fwd<T, 3>(ar, st);
    default: return launch_fwd<T, 4>(ar, st);
  }
}
template <typename T>
cudaError_t launch_bwd_t(const RnArgs& ar, int64_t ctas, cudaStream_t st) {
  switch ((ar.D + 127) / 128) {
    case 1: return launch_bwd<T, 1>(ar, ctas, st);
    case 2: return launch_bwd<T, 2>(ar, ctas, st);
    case 3: return launch_bwd<T, 3>(ar, ctas, st);
    default: return launch_bwd<T, 4>(ar, ctas, st);
  }
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status gdn_rmsnorm_gated_fwd(const gdn_rmsnorm_problem* p, const void* o, const void* z,
                                 const float* w, void* y, void* stream) {
  gdn_status s = check_problem(p);
  if (s != GDN_OK) return s;
  if (!w || !aligned16(w)) return GDN_ERR_INVALID_ARG;
  if (p->rows == 0) return GDN_OK;
  if (!o || !z || !y || !aligned16(o) || !aligned16(z) || !aligned16(y))
    return GDN_ERR_INVALID_ARG;
  RnArgs ar;
  memset(&ar, 0, sizeof(ar));
  ar.rows = p->rows;
  ar.D = p->D;
  ar.eps = p->eps;
  ar.o = o;
  ar.z = z;
  ar.w = w;
  ar.out0 = y;
  cudaStream_t st = (cudaStream_t)stream;
  const cudaError_t e = p->dtype == GDN_BF16 ? launch_fwd_t<__nv_bfloat16>(ar, st)
                                             : launch_fwd_t<float>(ar, st);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_rmsnorm_gated_bwd_workspace_size(const gdn_rmsnorm_problem* p, size_t* bytes) {
  if (!bytes) return GDN_ERR_INVALID_ARG;
  gdn_status s = check_problem(p);
  if (s != GDN_OK) return s;
  *bytes = (size_t)bwd_ctas(p) * (size_t)p->D * sizeof(float);
  return GDN_OK;
}

gdn_status gdn_rmsnorm_gated_bwd(const gdn_rmsnorm_problem* p, const void* o, const void* z,
                                 const float* w, const void* dy, void* d_o, void* dz, float* dw,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  gdn_status s = check_problem(p);
  if (s != GDN_OK) return s;
  if (!w || !dw || !aligned16(w) || !aligned16(dw)) return GDN_ERR_INVALID_ARG;
  const bool empty = p->rows == 0;
  if (!empty && (!o || !z || !dy || !d_o || !dz || !aligned16(o) || !aligned16(z) ||
                 !aligned16(dy) || !aligned16(d_o) || !aligned16(dz)))
    return GDN_ERR_INVALID_ARG;
  const int64_t ctas = bwd_ctas(p);
  const size_t need = (size_t)ctas * (size_t)p->D * sizeof(float);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return GDN_ERR_WORKSPACE;
  RnArgs ar;
  memset(&ar, 0, sizeof(ar));
  ar.rows = p->rows;
  ar.D = p->D;
  ar.eps = p->eps;
  ar.o = o;
  ar.z = z;
  ar.w = w;
  ar.dy = dy;
  ar.out0 = d_o;
  ar.out1 = dz;
  ar.part = (float*)workspace;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  if (!empty)
    e = p->dtype == GDN_BF16 ? launch_bwd_t<__nv_bfloat16>(ar, ctas, st)
                             : launch_bwd_t<float>(ar, ctas, st);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  k_rmsnorm_reduce<<<(unsigned)((p->D + 31) / 32), 256, 0, st>>>(ctas, p->D,
                                                                 (const float*)workspace, dw);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // extern "C"
