// gdn_tc_qk.cu -- last step of the bf16 backward: the gradients of the raw q and
// k from the per-V-head gradients of q_hat and k_hat that the chunk-parallel
// gradient kernel (gdn_tc_grad.cu) leaves in the workspace.
#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include "gdn_internal.h"
#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

using namespace tc;

// ============================================================================
// k_qk_grad_tc: dq, dk from the per-V-head bf16 gradients of q_hat, k_hat:
// summed over the r V heads of a Q/K head, then back through the scale and the
// L2 norm (q_hat = s q / |q|: dq = s (g - u (u . g)) / |q| with u = q / |q|).
// One warp per (row, token, Q/K head); lane l holds columns 4l .. 4l+3.
// ============================================================================
struct QkArgs {
  int64_t B, T, Ts, Tp, Hqk, H, r;
  int l2norm;
  float eps, scale;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* dqp;
  const __nv_bfloat16* dkp;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
};

__device__ __forceinline__ void ld4bf(const __nv_bfloat16* p, float* x) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
  const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
  x[0] = a.x; x[1] = a.y; x[2] = c.x; x[3] = c.y;
}

__global__ void __launch_bounds__(256) k_qk_grad_tc(QkArgs ar) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rowid = (int64_t)blockIdx.x * 8 + warp;
  if (rowid >= ar.B * ar.T * ar.Hqk) return;
  const int64_t hq = rowid % ar.Hqk, t = (rowid / ar.Hqk) % ar.T, b = rowid / (ar.Hqk * ar.T);
  const int64_t xo = ((b * ar.Ts + t) * ar.Hqk + hq) * 128 + lane * 4;
  float xq[4], xk[4], gq[4] = {0.f, 0.f, 0.f, 0.f}, gk[4] = {0.f, 0.f, 0.f, 0.f};
  ld4bf(ar.q + xo, xq);
  ld4bf(ar.k + xo, xk);
  for (int64_t h = hq * ar.r; h < (hq + 1) * ar.r; ++h) {
    const int64_t po = ((b * ar.Tp + t) * ar.H + h) * 128 + lane * 4;
    float a[4], c[4];
    ld4bf(ar.dqp + po, a);
    ld4bf(ar.dkp + po, c);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      gq[e] += a[e];
      gk[e] += c[e];
    }
  }
  float sq = 0.f, sk = 0.f, pq = 0.f, pk = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    sq = fmaf(xq[e], xq[e], sq);
    sk = fmaf(xk[e], xk[e], sk);
    pq = fmaf(xq[e], gq[e], pq);
    pk = fmaf(xk[e], gk[e], pk);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sq += __shfl_xor_sync(0xffffffffu, sq, o);
    sk += __shfl_xor_sync(0xffffffffu, sk, o);
    pq += __shfl_xor_sync(0xffffffffu, pq, o);
    pk += __shfl_xor_sync(0xffffffffu, pk, o);
  }
  float rq = 1.f, rk = 1.f, prq = 0.f, prk = 0.f;
  if (ar.l2norm) {
    rq = rsqrtf(sq + ar.eps);
    rk = rsqrtf(sk + ar.eps);
    prq = pq * rq * rq;
    prk = pk * rk * rk;
  }
  float oq[4], ok[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    oq[e] = ar.scale * (gq[e] - xq[e] * prq) * rq;
    ok[e] = (gk[e] - xk[e] * prk) * rk;
  }
  uint2 vq, vk;
  vq.x = pack_bf16(oq[0], oq[1]);
  vq.y = pack_bf16(oq[2], oq[3]);
  vk.x = pack_bf16(ok[0], ok[1]);
  vk.y = pack_bf16(ok[2], ok[3]);
  *reinterpret_cast<uint2*>(ar.dq + xo) = vq;
  *reinterpret_cast<uint2*>(ar.dk + xo) = vk;
}

}  // namespace

cudaError_t launch_qk_grad_tc(const Prob& pr, const Inputs& in, const WS& ws, void* dq, void* dk,
                              cudaStream_t st) {
  const int64_t rows = pr.B * pr.T * pr.Hqk;
  if (rows == 0) return cudaSuccess;
  QkArgs ar;
  ar.B = pr.B; ar.T = pr.T; ar.Ts = pr.Ts; ar.Tp = pr.Tp; ar.Hqk = pr.Hqk; ar.H = pr.H;
  ar.r = pr.r; ar.l2norm = pr.l2norm; ar.eps = pr.eps; ar.scale = pr.scale;
  ar.q = (const __nv_bfloat16*)in.q; ar.k = (const __nv_bfloat16*)in.k;
  ar.dqp = (const __nv_bfloat16*)ws.dqp; ar.dkp = (const __nv_bfloat16*)ws.dkp;
  ar.dq = (__nv_bfloat16*)dq; ar.dk = (__nv_bfloat16*)dk;
  k_qk_grad_tc<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(ar);
  return cudaGetLastError();
}

}  // namespace gdn
