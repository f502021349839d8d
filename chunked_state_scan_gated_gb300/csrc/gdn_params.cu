// gdn_params.cu -- gradients of the gate parameters.
//
// The gates of the core are g = -exp(A_log[h]) softplus(a + dt_bias[h]) and
// beta = sigmoid(b) ("Linear Attention CP 融合算子 PR #1114 测试报告", section 4.1
// lists dg and dbeta among the core's gradients; its accuracy checks cover the
// parameter gradients, A_log and dt_bias included).  From dg, dbeta this kernel
// forms da, db and the per-head sums dA_log, ddt_bias:
//   da_t = dg_t * (-exp(A_log)) * sigmoid(a_t + dt_bias)      (softplus' = sigmoid)
//   db_t = dbeta_t * beta_t (1 - beta_t)
//   ddt_bias = sum_t da_t,  dA_log = sum_t dg_t g_t           (dg/dA_log = g)
// Padded tokens (t >= valid_len) have g, beta fixed at 0: zero da, db, no share
// of the sums.  One CTA per head sums its tokens in a fixed order (fp64), so
// the result is deterministic.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int PT = 256;

__device__ __forceinline__ float ldg_in(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ldg_in(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}

template <typename TIn>
__global__ void __launch_bounds__(PT) k_gate_param_bwd(int64_t B, int64_t T, int64_t Ts,
                                                       int64_t H, const TIn* __restrict__ a,
                                                       const TIn* __restrict__ b,
                                                       const float* __restrict__ A_log,
                                                       const float* __restrict__ dt_bias,
                                                       const int32_t* __restrict__ valid_len,
                                                       const float* __restrict__ dg,
                                                       const float* __restrict__ dbeta,
                                                       float* da, float* db, float* dA_log,
                                                       float* ddt_bias) {
  __shared__ double red[2][PT / 32];
  const int64_t h = blockIdx.x;
  const float ea = expf(A_log[h]), bias = dt_bias[h];
  double sA = 0.0, sdt = 0.0;
  for (int64_t bb = 0; bb < B; ++bb) {
    int64_t L = T;
    if (valid_len) {
      L = valid_len[bb];
      L = L < 0 ? 0 : (L > T ? T : L);
    }
    for (int64_t t = threadIdx.x; t < T; t += PT) {
      const int64_t gi = (bb * Ts + t) * H + h;
      float va = 0.f, vb = 0.f;
      if (t < L) {
        const float x = ldg_in(a, gi) + bias;
        const float sg = 1.f / (1.f + expf(-x));
        const float sp = x > 20.f ? x : log1pf(expf(x));
        const float dsp = x > 20.f ? 1.f : sg;
        const float be = 1.f / (1.f + expf(-ldg_in(b, gi)));
        const float gg = dg[gi];
        va = -gg * ea * dsp;
        vb = dbeta[gi] * be * (1.f - be);
        sdt += (double)va;
        sA += (double)gg * (double)(-ea * sp);
      }
      da[gi] = va;
      db[gi] = vb;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sA += __shfl_xor_sync(0xffffffffu, sA, o);
    sdt += __shfl_xor_sync(0xffffffffu, sdt, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red[0][warp] = sA;
    red[1][warp] = sdt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double x = 0.0, y = 0.0;
    for (int w = 0; w < PT / 32; ++w) {
      x += red[0][w];
      y += red[1][w];
    }
    dA_log[h] = (float)x;
    ddt_bias[h] = (float)y;
  }
}

}  // namespace

cudaError_t launch_gate_param_bwd(const Prob& pr, const void* a, const void* b,
                                  const float* A_log, const float* dt_bias,
                                  const int32_t* valid_len, const float* dg, const float* dbeta,
                                  float* da, float* db, float* dA_log, float* ddt_bias,
                                  cudaStream_t st) {
  if (pr.H == 0) return cudaSuccess;
  const dim3 grid((unsigned)pr.H);
  if (pr.dtype == GDN_BF16)
    k_gate_param_bwd<__nv_bfloat16><<<grid, PT, 0, st>>>(
        pr.B, pr.T, pr.Ts, pr.H, (const __nv_bfloat16*)a, (const __nv_bfloat16*)b, A_log, dt_bias,
        valid_len, dg, dbeta, da, db, dA_log, ddt_bias);
  else
    k_gate_param_bwd<float><<<grid, PT, 0, st>>>(pr.B, pr.T, pr.Ts, pr.H, (const float*)a,
                                                 (const float*)b, A_log, dt_bias, valid_len, dg,
                                                 dbeta, da, db, dA_log, ddt_bias);
  return cudaGetLastError();
}

}  // namespace gdn
