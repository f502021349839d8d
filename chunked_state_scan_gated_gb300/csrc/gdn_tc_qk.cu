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
// Sixteen lanes per (row, token, Q/K head); lane l of the group holds columns
// 8l .. 8l+7, so every access is 16 bytes and a warp covers two rows.
// ============================================================================
struct QkArgs {
  int64_t B, T, Ts, Tp, Hqk, H, r;
  int l2norm;
  float eps, scale;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* dqp;
  const __nv_bfloat16* dkp;
  const int32_t* valid_len;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
};

__device__ __forceinline__ void ld8bf(const __nv_bfloat16* p, float* x) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

constexpr int QK_ROWS = 16;  // rows per 256-thread block

__global__ void __launch_bounds__(256) k_qk_grad_tc(QkArgs ar) {
  const int sub = threadIdx.x & 15;
  const uint32_t rowid = blockIdx.x * QK_ROWS + (threadIdx.x >> 4);  // below 2^31 (host)
  if (rowid >= (uint32_t)(ar.B * ar.T * ar.Hqk)) return;  // whole 16-lane groups leave together
  const unsigned gmask = 0xffffu << (threadIdx.x & 16);
  const uint32_t q1 = rowid / (uint32_t)ar.Hqk;
  const int64_t hq = rowid - q1 * (uint32_t)ar.Hqk, t = q1 % (uint32_t)ar.T,
                b = q1 / (uint32_t)ar.T;
  const int64_t xo = ((b * ar.Ts + t) * ar.Hqk + hq) * 128 + sub * 8;
  const int64_t po0 = ((b * ar.Tp + t) * ar.H + hq * ar.r) * 128 + sub * 8;
  if (ar.valid_len) {  // padded token: zero gradient (its chunk may not have been computed)
    int64_t L = ar.valid_len[b];
    L = L < 0 ? 0 : (L > ar.T ? ar.T : L);
    if (t >= L) {
      *reinterpret_cast<uint4*>(ar.dq + xo) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(ar.dk + xo) = make_uint4(0, 0, 0, 0);
      return;
    }
  }
  float xq[8], xk[8], gq[8], gk[8];
  ld8bf(ar.q + xo, xq);
  ld8bf(ar.k + xo, xk);
  ld8bf(ar.dqp + po0, gq);
  ld8bf(ar.dkp + po0, gk);
  for (int64_t j = 1; j < ar.r; ++j) {
    float a[8], c[8];
    ld8bf(ar.dqp + po0 + j * 128, a);
    ld8bf(ar.dkp + po0 + j * 128, c);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      gq[e] += a[e];
      gk[e] += c[e];
    }
  }
  float sq = 0.f, sk = 0.f, pq = 0.f, pk = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    sq = fmaf(xq[e], xq[e], sq);
    sk = fmaf(xk[e], xk[e], sk);
    pq = fmaf(xq[e], gq[e], pq);
    pk = fmaf(xk[e], gk[e], pk);
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    sq += __shfl_xor_sync(gmask, sq, o);
    sk += __shfl_xor_sync(gmask, sk, o);
    pq += __shfl_xor_sync(gmask, pq, o);
    pk += __shfl_xor_sync(gmask, pk, o);
  }
  float rq = 1.f, rk = 1.f, prq = 0.f, prk = 0.f;
  if (ar.l2norm) {
    rq = rsqrtf(sq + ar.eps);
    rk = rsqrtf(sk + ar.eps);
    prq = pq * rq * rq;
    prk = pk * rk * rk;
  }
  float oq[8], ok[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    oq[e] = ar.scale * (gq[e] - xq[e] * prq) * rq;
    ok[e] = (gk[e] - xk[e] * prk) * rk;
  }
  uint4 vq, vk;
  vq.x = pack_bf16(oq[0], oq[1]);
  vq.y = pack_bf16(oq[2], oq[3]);
  vq.z = pack_bf16(oq[4], oq[5]);
  vq.w = pack_bf16(oq[6], oq[7]);
  vk.x = pack_bf16(ok[0], ok[1]);
  vk.y = pack_bf16(ok[2], ok[3]);
  vk.z = pack_bf16(ok[4], ok[5]);
  vk.w = pack_bf16(ok[6], ok[7]);
  *reinterpret_cast<uint4*>(ar.dq + xo) = vq;
  *reinterpret_cast<uint4*>(ar.dk + xo) = vk;
}

// ============================================================================
// k_pad_tail_zero: zero the tokens of every row from the end of its last chunk that
// holds a valid token (ceil(valid_len / 64) * 64) to T, in a token-major tensor of
// `row` bytes per token.  The tensor-core kernels skip chunks of padding only, so
// their outputs there (o; dv, dg, dbeta) are written here instead.  grid (x, B).
// ============================================================================
template <typename U>
__global__ void __launch_bounds__(256) k_pad_tail_zero(const int32_t* __restrict__ valid_len,
                                                       int64_t T, int64_t Ts, int64_t row,
                                                       uint8_t* __restrict__ dst) {
  const int64_t b = blockIdx.y;
  int64_t L = valid_len[b];
  L = L < 0 ? 0 : (L > T ? T : L);
  const int64_t start = (L + 63) / 64 * 64;
  if (start >= T) return;
  const int64_t per = row / (int64_t)sizeof(U);
  const int64_t n = (T - start) * per;
  U* base = reinterpret_cast<U*>(dst + (b * Ts + start) * row);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    base[i] = U{};
}

}  // namespace

cudaError_t launch_pad_tail_zero(const Prob& pr, const int32_t* valid_len, void* dst,
                                 int64_t row_bytes, cudaStream_t st) {
  if (!valid_len || !dst || pr.B == 0 || pr.T == 0 || row_bytes <= 0) return cudaSuccess;
  const dim3 grid(64, (unsigned)pr.B);
  uint8_t* d = (uint8_t*)dst;
  if (row_bytes % 16 == 0 && ((uintptr_t)dst & 15u) == 0)
    k_pad_tail_zero<uint4><<<grid, 256, 0, st>>>(valid_len, pr.T, pr.Ts, row_bytes, d);
  else
    k_pad_tail_zero<uint32_t><<<grid, 256, 0, st>>>(valid_len, pr.T, pr.Ts, row_bytes, d);
  return cudaGetLastError();
}

cudaError_t launch_qk_grad_tc(const Prob& pr, const Inputs& in, const WS& ws, void* dq, void* dk,
                              cudaStream_t st) {
  const int64_t rows = pr.B * pr.T * pr.Hqk;
  if (rows == 0) return cudaSuccess;
  if (rows >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;  // 32-bit row indices
  QkArgs ar;
  ar.B = pr.B; ar.T = pr.T; ar.Ts = pr.Ts; ar.Tp = pr.Tp; ar.Hqk = pr.Hqk; ar.H = pr.H;
  ar.r = pr.r; ar.l2norm = pr.l2norm; ar.eps = pr.eps; ar.scale = pr.scale;
  ar.q = (const __nv_bfloat16*)in.q; ar.k = (const __nv_bfloat16*)in.k;
  ar.dqp = (const __nv_bfloat16*)ws.dqp; ar.dkp = (const __nv_bfloat16*)ws.dkp;
  ar.valid_len = in.valid_len;
  ar.dq = (__nv_bfloat16*)dq; ar.dk = (__nv_bfloat16*)dk;
  k_qk_grad_tc<<<(unsigned)((rows + QK_ROWS - 1) / QK_ROWS), 256, 0, st>>>(ar);
  return cudaGetLastError();
}

}  // namespace gdn
