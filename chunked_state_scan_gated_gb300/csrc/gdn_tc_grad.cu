// gdn_tc_grad.cu -- chunk-parallel local gradients of the bf16 backward, in
// feature-major ("transposed") form on tcgen05.
//
// Given a chunk's start state S and the gradient dS of its end state (bf16 tile
// images from the forward and reverse chains) and the prologue's W, U, P, T
// tiles, every local gradient of the chunk follows from (notation of
// gdn_simt.cu; kt_t = e^{G_C - G_t}, X_v = T^T dV', X_w = T^T dW):
//
//   V'  = U - W S,                dV' = P^T dO + diag(kt) K dS
//   dq  = diag(gamma) dO S^T + (dP o Gamma) K,          dP = dO V'^T (lower)
//   dk  = (dP o Gamma)^T Q + diag(kt) V' dS^T + diag(beta gamma) X_w + E K + E^T K
//   dv  = diag(beta) X_v,         dW = -dV' S^T
//   dA  = -X_v V'^T (strictly lower; equal to -(X_v U^T + X_w W^T) since W S = U - V'),
//   E   = dA o beta_i Gamma,      dbeta, dG from row dots of the same pieces.
//
// Every product whose result has a 128-wide feature side is computed transposed
// (feature x token: V'^T = U^T - S^T W^T, dV'^T, S dO^T, S dV'^T, dS V'^T,
// dV'^T T, dW^T T, K^T (dP o Gamma)^T, Q^T (dP o Gamma) + K^T E^T + K^T E), so
// that it is an M = 128 MMA whose accumulator row is a feature and every thread of
// the CTA owns one feature row and 32 token columns.  Only the token x token
// products (dP, dA, K K^T) are M = 64.  Dots over the feature dimension become
// column sums over the CTA, taken with a warp transpose-reduce.  The outputs dv,
// dq_hat, dk_hat are staged token-major in shared memory and written by TMA.
#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include "gdn_internal.h"
#include "gdn_tc_common.cuh"

namespace gdn {

bool tc_make_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t Ts, int64_t heads);

namespace {

using namespace tc;

constexpr int GT = 256;
// Shared-memory map (1024-byte aligned regions).
constexpr uint32_t R_Q = 0;          // q_hat [tok][dk] (two 8 KB atoms), scale included
constexpr uint32_t R_K = 16384;      // k_hat [tok][dk]
constexpr uint32_t R_V = 32768;      // v [tok][dv]
constexpr uint32_t R_DO = 49152;     // dO [tok][dv]; after round B: dv staging [tok][dv]
constexpr uint32_t R_S = 65536;      // S image [dk rows][dv] (two [128][64] atoms); then Z scratch
constexpr uint32_t R_DS = 98304;     // dS image; after round B: dq_hat, dk_hat staging
constexpr uint32_t R_W = 131072;     // W [tok][dk]; after round A: dW^T [dk][tok]
constexpr uint32_t R_U = 147456;     // U [tok][dv]; after round A: X_v^T [dv][tok]
constexpr uint32_t R_P = 163840;     // P [i][j]; in round B's epilogue: dP o Gamma
constexpr uint32_t R_T = 172032;     // T [i][j]; in round C's epilogue: E
constexpr uint32_t R_VT = 180224;    // V'^T [dv][tok] ([128][64] atom)
constexpr uint32_t R_DVT = 196608;   // dV'^T [dv][tok]
constexpr uint32_t R_SC = 212992;    // scalars
constexpr uint32_t SC_BYTES = 8 * 64 * 4 + 4 * 4 * 64 * 4 + 128 * 4 + 64;
constexpr uint32_t GR_SMEM = R_SC + SC_BYTES + 1024;

struct Grad2Args {
  int64_t T, Ts, H, r, NC, Tp;
  int l2norm;
  float eps, scale;
  const __nv_bfloat16* a;
  const __nv_bfloat16* b;
  const float* A_log;
  const float* dt_bias;
  const int32_t* valid_len;
  float* dg;           // [B, Ts, H]
  float* dbeta;
  const uint8_t* hc;   // chunk-start states, 32 KB tile images
  const uint8_t* dhc;  // chunk-end state gradients, 32 KB tile images
  const uint8_t* wim;  // prologue tile images: W, U, P, T
  const uint8_t* uim;
  const uint8_t* pim;
  const uint8_t* tim;
  int* status;
};

// Lane l ends with the sum over the warp's 32 lanes of p[l] (31 shuffles).
template <int K>
__device__ __forceinline__ void xr_stage(float (&p)[32], int lane) {
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const bool up = (lane & K) != 0;
    const float send = up ? p[i] : p[i + K];
    const float keep = up ? p[i + K] : p[i];
    p[i] = keep + __shfl_xor_sync(0xffffffffu, send, K);
  }
}
__device__ __forceinline__ float xreduce32(float (&p)[32], int lane) {
  xr_stage<16>(p, lane);
  xr_stage<8>(p, lane);
  xr_stage<4>(p, lane);
  xr_stage<2>(p, lane);
  xr_stage<1>(p, lane);
  return p[0];
}

// Element (t, f) of a token-major [64][128] bf16 tile (two K-major atoms).
__device__ __forceinline__ uint32_t tf_off(int t, int f) {
  return (uint32_t)((f >> 6) * 8192 + t * 128 + (((((f & 63) >> 3) ^ t) & 7) << 4) + (f & 7) * 2);
}
__device__ __forceinline__ float ld_bf(const uint8_t* p) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}
__device__ __forceinline__ void st_bf(uint8_t* p, float x) {
  *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(x);
}

#define GRAD_SYNC()             \
  do {                          \
    fence_proxy_async();        \
    tc_fence_before();          \
    __syncthreads();            \
    tc_fence_after();           \
    if (*s_abort) goto done;    \
  } while (0)

__global__ void __launch_bounds__(GT, 1)
    k_grad2_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
               const __grid_constant__ CUtensorMap mdv, const __grid_constant__ CUtensorMap mdqp,
               const __grid_constant__ CUtensorMap mdkp, Grad2Args ar) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t base = smem_u32(sm);
  float* sG = (float*)(sm + R_SC);     // cumulative gate (log2 units)
  float* sGam = sG + 64;
  float* sBeta = sGam + 64;
  float* sKt = sBeta + 64;
  float* sDG = sKt + 64;               // dG terms of P and A (row and column sums)
  float* sDB = sDG + 64;               // dbeta terms of A
  float* sFin = sDB + 64;              // final dG
  float* sMisc = sFin + 64;            // [8] block partials of <S, dS>
  float* sRed = sMisc + 64;            // [4 types][4 quadrants][64 tokens] column partials
  float* sDBh = sRed + 4 * 4 * 64;     // [2 halves][64] dbeta terms of A
  uint64_t* bar_ld = (uint64_t*)(sDBh + 128);
  uint64_t* bar_mma = bar_ld + 1;
  uint32_t* s_tmem = (uint32_t*)(bar_ld + 2);
  int* s_abort = (int*)(s_tmem + 1);
  float* sZ = (float*)(sm + R_S);      // fp32 64 x 64, row stride 65, once S is consumed

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int fr = quad * 32 + lane;     // feature row (TMEM lane) of M = 128 results
  const bool own64 = lane < 16;        // owns row ri of M = 64 results
  const int ri = quad * 16 + (lane & 15);
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t hq = h / ar.r, bh = b * ar.H + h;
  const int64_t t0 = c * 64;
  int64_t L = ar.T;
  if (ar.valid_len) {
    L = ar.valid_len[b];
    if (L < 0 || L > ar.T) L = L < 0 ? 0 : ar.T;
  }
  enum { RQ = 0, RV = 1, RKW = 2, RKD = 3 };  // column-sum types

  if (tid == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
    *s_abort = 0;
  }
  if (warp == 0) tmem_alloc(s_tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  if (tid == 0) {
    const int64_t im = bh * ar.NC + c;
    mbar_arrive_expect_tx(bar_ld, 4 * 16384u + 2 * 32768u + 2 * 16384u + 2 * 8192u);
    for (int at = 0; at < 2; ++at) {
      tma_load_4d(sm + R_Q + at * 8192, &mq, at * 64, (int)hq, (int)t0, (int)b, bar_ld);
      tma_load_4d(sm + R_K + at * 8192, &mk, at * 64, (int)hq, (int)t0, (int)b, bar_ld);
      tma_load_4d(sm + R_V + at * 8192, &mv, at * 64, (int)h, (int)t0, (int)b, bar_ld);
      tma_load_4d(sm + R_DO + at * 8192, &mdo, at * 64, (int)h, (int)t0, (int)b, bar_ld);
    }
    bulk_load(sm + R_S, ar.hc + im * 32768, 32768, bar_ld);
    bulk_load(sm + R_DS, ar.dhc + im * 32768, 32768, bar_ld);
    bulk_load(sm + R_W, ar.wim + im * 16384, 16384, bar_ld);
    bulk_load(sm + R_U, ar.uim + im * 16384, 16384, bar_ld);
    bulk_load(sm + R_P, ar.pim + im * 8192, 8192, bar_ld);
    bulk_load(sm + R_T, ar.tim + im * 8192, 8192, bar_ld);
  }
  if (tid < 64) {
    const int64_t t = t0 + tid;
    float g = 0.f, be = 0.f;
    if (t < L) {
      const int64_t gi = (b * ar.Ts + t) * ar.H + h;
      const float x = __bfloat162float(ar.a[gi]) + ar.dt_bias[h];
      const float sp = x > 20.f ? x : log1pf(expf(x));
      g = -expf(ar.A_log[h]) * sp;
      be = 1.f / (1.f + expf(-__bfloat162float(ar.b[gi])));
    }
    sG[tid] = g * kLog2e;
    sBeta[tid] = be;
    sDG[tid] = 0.f;
    sDB[tid] = 0.f;
  }
  __syncthreads();
  cumsum64f(sG);
  __syncthreads();
  if (tid < 64) {
    sGam[tid] = exp2f(sG[tid]);
    sKt[tid] = dexp_(sG[63], sG[tid]);
  }
  if (!mbar_wait(bar_ld, 0, ar.status, kStatusTimeout)) *s_abort = 1;
  // q, k rows normalised in place (16 threads per row); padded dO rows zeroed
  for (int it = 0; it < 8; ++it) {
    const int rr = (tid >> 4) + 16 * it;
    const bool isk = rr >= 64;
    const int sub = tid & 15, at = sub >> 3, ch = sub & 7, r6 = rr & 63;
    const uint32_t off = (isk ? R_K : R_Q) + at * 8192 + kmaj_chunk(r6, ch);
    float x[8];
    ld_chunk(sm, off, x);
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
    ss += __shfl_xor_sync(0xffffffffu, ss, 8);
    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    float s = ar.l2norm ? rsqrtf(ss + ar.eps) : 1.f;
    if (!isk) s *= ar.scale;
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] *= s;
    st_chunk(sm, off, x);
  }
  if (t0 + 64 > L) {
    for (int idx = tid; idx < 1024; idx += GT) {
      const int i = idx >> 4, cc = idx & 15;
      if (t0 + i >= L)
        *reinterpret_cast<uint4*>(sm + R_DO + (cc >> 3) * 8192 + kmaj_chunk(i, cc & 7)) = make_uint4(0, 0, 0, 0);
    }
  }
  {
    uint32_t ph = 0;
    float dqT[32], dkT[32];  // this thread's feature row fr of dq_hat^T, dk_hat^T, tokens 32 half + e
    const uint32_t idA = idesc_bf16(128, 64, 1, 0);  // A MN-major (feature rows), B K-major
    const uint32_t idB = idesc_bf16(128, 64, 0, 1);  // A K-major, B MN-major
    const uint32_t idC = idesc_bf16(128, 64, 1, 1);  // both MN-major
    const uint32_t idD = idesc_bf16(128, 64, 0, 0);  // both K-major
    GRAD_SYNC();
    // ---- round A: S^T W^T -> [0,64), dO^T P -> [64,128), dS^T K^T -> [128,192), S dO^T -> [192,256)
    if (tid == 0) {
      for (int ks = 0; ks < 8; ++ks) {  // K = dk (S^T W^T, dS^T K^T) or dv (S dO^T)
        const uint32_t at = ks >> 2, kk = ks & 3;
        mma_bf16(tmem, sdesc(base + R_S + ks * 2048, 16384, 1024),
                 sdesc(base + R_W + at * 8192 + kk * 32, 16, 1024), idA, ks > 0);
        mma_bf16(tmem + 128, sdesc(base + R_DS + ks * 2048, 16384, 1024),
                 sdesc(base + R_K + at * 8192 + kk * 32, 16, 1024), idA, ks > 0);
        mma_bf16(tmem + 192, sdesc(base + R_S + at * 16384 + kk * 32, 16, 1024),
                 sdesc(base + R_DO + at * 8192 + kk * 32, 16, 1024), idD, ks > 0);
      }
      for (int ks = 0; ks < 4; ++ks)  // K = tokens
        mma_bf16(tmem + 64, sdesc(base + R_DO + ks * 2048, 8192, 1024),
                 sdesc(base + R_P + ks * 2048, 8192, 1024), idC, ks > 0);
      mma_commit(bar_mma);
    }
    {  // <S, dS> (same tile layout): block partials into sMisc
      float acc = 0.f;
      for (int q = tid; q < 2048; q += GT) {
        float x[8], y[8];
        ld_chunk(sm + R_S, q * 16, x);
        ld_chunk(sm + R_DS, q * 16, y);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(x[e], y[e], acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) sMisc[warp] = acc;
    }
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    {
      const int f = fr;
      float ws[32], a1[32], a2[32];
      tmem_ld32(tmem + lane_off + 32 * half, ws);
      tmem_ld32(tmem + lane_off + 64 + 32 * half, a1);
      tmem_ld32(tmem + lane_off + 128 + 32 * half, a2);
      tmem_ld32(tmem + lane_off + 192 + 32 * half, dqT);
      float pq[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int t = 32 * half + e;
        ws[e] = ld_bf(sm + R_U + tf_off(t, f)) - ws[e];   // V'^T
        a1[e] = fmaf(sKt[t], a2[e], a1[e]);                 // dV'^T
        dqT[e] *= sGam[t];                                  // (diag(gamma) dO S^T)^T
        pq[e] = ld_bf(sm + R_Q + tf_off(t, f)) * dqT[e];    // q_t . (gamma_t S dO_t)
      }
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        st_chunk(sm + R_VT, kmaj_chunk(f, 4 * half + cc), &ws[cc * 8]);
        st_chunk(sm + R_DVT, kmaj_chunk(f, 4 * half + cc), &a1[cc * 8]);
      }
      sRed[(RQ * 4 + quad) * 64 + 32 * half + lane] = xreduce32(pq, lane);
    }
    GRAD_SYNC();
    // ---- round B: S dV'^T -> [0,64) (-dW^T), dS V'^T -> [64,128), dV'^T T -> [128,192) (X_v^T),
    //      dO V'^T -> [192,256) (dP, M = 64), K K^T -> [256,320) (M = 64)
    if (tid == 0) {
      const uint32_t id64b = idesc_bf16(64, 64, 0, 1), id64d = idesc_bf16(64, 64, 0, 0);
      for (int ks = 0; ks < 8; ++ks) {  // K = dv (S, dS, dO rows) or dk (K K^T)
        const uint32_t at = ks >> 2, kk = ks & 3;
        mma_bf16(tmem, sdesc(base + R_S + at * 16384 + kk * 32, 16, 1024),
                 sdesc(base + R_DVT + ks * 2048, 8192, 1024), idB, ks > 0);
        mma_bf16(tmem + 64, sdesc(base + R_DS + at * 16384 + kk * 32, 16, 1024),
                 sdesc(base + R_VT + ks * 2048, 8192, 1024), idB, ks > 0);
        mma_bf16(tmem + 192, sdesc(base + R_DO + at * 8192 + kk * 32, 16, 1024),
                 sdesc(base + R_VT + ks * 2048, 8192, 1024), id64b, ks > 0);
        mma_bf16(tmem + 256, sdesc(base + R_K + at * 8192 + kk * 32, 16, 1024),
                 sdesc(base + R_K + at * 8192 + kk * 32, 16, 1024), id64d, ks > 0);
      }
      for (int ks = 0; ks < 4; ++ks)  // K = tokens
        mma_bf16(tmem + 128, sdesc(base + R_DVT + ks * 32, 16, 1024),
                 sdesc(base + R_T + ks * 2048, 8192, 1024), idB, ks > 0);
      mma_commit(bar_mma);
    }
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    {
      const int f = fr;
      float x[32], pk[32];
      tmem_ld32(tmem + lane_off + 32 * half, x);           // S dV'^T = -dW^T
#pragma unroll
      for (int e = 0; e < 32; ++e) x[e] = -x[e];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) st_chunk(sm + R_W, kmaj_chunk(f, 4 * half + cc), &x[cc * 8]);
      tmem_ld32(tmem + lane_off + 64 + 32 * half, x);      // (V' dS^T)^T
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int t = 32 * half + e;
        dkT[e] = sKt[t] * x[e];
        pk[e] = ld_bf(sm + R_K + tf_off(t, f)) * x[e];    // k_t . (V' dS^T)_t
      }
      sRed[(RKD * 4 + quad) * 64 + 32 * half + lane] = xreduce32(pk, lane);
      tmem_ld32(tmem + lane_off + 128 + 32 * half, x);     // X_v^T
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) st_chunk(sm + R_U, kmaj_chunk(f, 4 * half + cc), &x[cc * 8]);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int t = 32 * half + e;
        pk[e] = ld_bf(sm + R_V + tf_off(t, f)) * x[e];    // v_t . X_v,t
        st_bf(sm + R_DO + tf_off(t, f), (t0 + t < L) ? sBeta[t] * x[e] : 0.f);  // dv staging
      }
      sRed[(RV * 4 + quad) * 64 + 32 * half + lane] = xreduce32(pk, lane);
      float dp[32];
      tmem_ld32(tmem + lane_off + 192 + 32 * half, dp);    // dP (M = 64 layout)
      if (own64) {
        const int i = ri;
        float pv[32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) ld_chunk(sm + R_P, kmaj_chunk(i, half * 4 + cc), &pv[cc * 8]);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = half * 32 + cc * 8 + e;
            const float dpv = (j <= i) ? dp[cc * 8 + e] : 0.f;
            sZ[i * 65 + j] = dpv * pv[cc * 8 + e];                  // dP o P
            y[e] = (j <= i) ? dpv * dexp_(sG[i], sG[j]) : 0.f;      // dP o Gamma
          }
          st_chunk(sm + R_P, kmaj_chunk(i, half * 4 + cc), y);       // over P (this thread's)
        }
      }
    }
    GRAD_SYNC();
    if (tid == 0) {  // dv tile (tokens past T are clipped by the tensor map)
      tma_store_4d(&mdv, sm + R_DO, 0, (int)h, (int)t0, (int)b);
      tma_store_4d(&mdv, sm + R_DO + 8192, 64, (int)h, (int)t0, (int)b);
      bulk_commit();
    }
    if (tid < 64) {  // gate terms of P: sum_j Z_ij - sum_j Z_ji
      float acc = 0.f;
      for (int j = 0; j < 64; ++j) acc += sZ[tid * 65 + j] - sZ[j * 65 + tid];
      sDG[tid] += acc;
    }
    // ---- round C: dW^T T -> [0,64) (X_w^T), K^T (dP o Gamma)^T -> [64,128),
    //      X_v V'^T -> [128,192) (dA', M = 64); K K^T stays in [256,320)
    if (tid == 0) {
      const uint32_t id64c = idesc_bf16(64, 64, 1, 1);
      for (int ks = 0; ks < 4; ++ks) {  // K = tokens
        mma_bf16(tmem, sdesc(base + R_W + ks * 32, 16, 1024),
                 sdesc(base + R_T + ks * 2048, 8192, 1024), idB, ks > 0);
        mma_bf16(tmem + 64, sdesc(base + R_K + ks * 2048, 8192, 1024),
                 sdesc(base + R_P + ks * 32, 16, 1024), idA, ks > 0);
      }
      for (int ks = 0; ks < 8; ++ks)  // K = dv
        mma_bf16(tmem + 128, sdesc(base + R_U + ks * 2048, 8192, 1024),
                 sdesc(base + R_VT + ks * 2048, 8192, 1024), id64c, ks > 0);
      mma_commit(bar_mma);
    }
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    {
      const int f = fr;
      float x[32], pk[32];
      tmem_ld32(tmem + lane_off + 32 * half, x);           // X_w^T
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int t = 32 * half + e;
        const float bg = sBeta[t] * sGam[t];
        dkT[e] = fmaf(bg, x[e], dkT[e]);
        pk[e] = ld_bf(sm + R_K + tf_off(t, f)) * x[e];    // k_t . X_w,t
      }
      sRed[(RKW * 4 + quad) * 64 + 32 * half + lane] = xreduce32(pk, lane);
      tmem_ld32(tmem + lane_off + 64 + 32 * half, x);      // (dP o Gamma) K, transposed
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int t = 32 * half + e;
        st_bf(sm + R_DS + tf_off(t, f), (t0 + t < L) ? dqT[e] + x[e] : 0.f);  // dq_hat staging
      }
      float da[32], kk[32];
      tmem_ld32(tmem + lane_off + 128 + 32 * half, da);    // dA' (M = 64 layout)
      tmem_ld32(tmem + lane_off + 256 + 32 * half, kk);    // K K^T (M = 64 layout)
      if (own64) {
        const int i = ri;
        const float be = sBeta[i];
        float part = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float ex[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = half * 32 + cc * 8 + e;
            const float gmm = (j < i) ? dexp_(sG[i], sG[j]) : 0.f;
            const float dA = (j < i) ? -da[cc * 8 + e] : 0.f;
            const float kg = kk[cc * 8 + e] * gmm;
            part = fmaf(dA, kg, part);                 // dbeta: dA (k_i . k_j) Gamma
            sZ[i * 65 + j] = dA * be * kg;             // dA o A
            ex[e] = dA * be * gmm;                     // E
          }
          st_chunk(sm + R_T, kmaj_chunk(i, half * 4 + cc), ex);   // E over T
        }
        sDBh[half * 64 + i] = part;
      }
    }
    GRAD_SYNC();
    if (tid == 0) {  // dq_hat tile
      tma_store_4d(&mdqp, sm + R_DS, 0, (int)h, (int)t0, (int)b);
      tma_store_4d(&mdqp, sm + R_DS + 8192, 64, (int)h, (int)t0, (int)b);
      bulk_commit();
    }
    if (tid < 64) {
      float acc = 0.f;
      for (int j = 0; j < 64; ++j) acc += sZ[tid * 65 + j] - sZ[j * 65 + tid];
      sDG[tid] += acc;
    }
    // ---- round D: Q^T (dP o Gamma) + K^T E^T + K^T E -> [0,64)
    if (tid == 0) {
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem, sdesc(base + R_Q + ks * 2048, 8192, 1024),
                 sdesc(base + R_P + ks * 2048, 8192, 1024), idC, ks > 0);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem, sdesc(base + R_K + ks * 2048, 8192, 1024),
                 sdesc(base + R_T + ks * 32, 16, 1024), idA, 1);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem, sdesc(base + R_K + ks * 2048, 8192, 1024),
                 sdesc(base + R_T + ks * 2048, 8192, 1024), idC, 1);
      mma_commit(bar_mma);
    }
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    {
      const int f = fr;
      float x[32];
      tmem_ld32(tmem + lane_off + 32 * half, x);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int t = 32 * half + e;
        st_bf(sm + R_DS + 16384 + tf_off(t, f), (t0 + t < L) ? dkT[e] + x[e] : 0.f);  // dk_hat
      }
    }
    GRAD_SYNC();
    if (tid == 0) {
      tma_store_4d(&mdkp, sm + R_DS + 16384, 0, (int)h, (int)t0, (int)b);
      tma_store_4d(&mdkp, sm + R_DS + 16384 + 8192, 64, (int)h, (int)t0, (int)b);
      bulk_commit();
    }
    // ---- gate gradients: column sums of the four row dots, Kt terms, state term
    if (tid < 64) {
      const int t = tid;
      float rq = 0.f, rv = 0.f, rkw = 0.f, rkd = 0.f;
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        rq += sRed[(RQ * 4 + qd) * 64 + t];
        rv += sRed[(RV * 4 + qd) * 64 + t];
        rkw += sRed[(RKW * 4 + qd) * 64 + t];
        rkd += sRed[(RKD * 4 + qd) * 64 + t];
      }
      const float be = sBeta[t], gm = sGam[t];
      const float s_t = sKt[t] * rkd;                       // Kt term of dG_t
      float d = sDG[t] + rq + be * gm * rkw;
      if (t < 63) d -= s_t;
      sFin[t] = d;
      sDB[t] += rv + gm * rkw + sDBh[t] + sDBh[64 + t];
      sRed[t] = (t < 63) ? s_t : 0.f;                       // reuse: Kt terms to sum into dG_C
    }
    __syncthreads();
    if (tid == 0) {
      float tot = 0.f;
      for (int i = 0; i < 63; ++i) tot += sRed[i];
      float sd = 0.f;
      for (int w = 0; w < GT / 32; ++w) sd += sMisc[w];
      sFin[63] += tot + sGam[63] * sd;
    }
    __syncthreads();
    if (tid < 32) {  // dg_j = sum_{i >= j} dG_i (reverse cumsum, warp 0)
      float v0 = sFin[63 - tid], v1 = sFin[31 - tid];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, v0, o);
        const float y1 = __shfl_up_sync(0xffffffffu, v1, o);
        if (tid >= o) {
          v0 += y0;
          v1 += y1;
        }
      }
      v1 += __shfl_sync(0xffffffffu, v0, 31);
      __syncwarp();
      sFin[63 - tid] = v0;
      sFin[31 - tid] = v1;
    }
    __syncthreads();
    if (tid < 64) {
      const int64_t t = t0 + tid;
      if (t < ar.T) {
        const int64_t gi = (b * ar.Ts + t) * ar.H + h;
        const bool valid = t < L;
        ar.dg[gi] = valid ? sFin[tid] : 0.f;   // natural-log units (log2 only enters exponents)
        ar.dbeta[gi] = valid ? sDB[tid] : 0.f;
      }
    }
  }
done:
  if (tid == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_grad2_tc(const Prob& pr, const Inputs& in, const WS& ws, const void* hc,
                            const void* dhc, void* dv, float* dg, float* dbeta, cudaStream_t st) {
  if (pr.B == 0 || pr.NC == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv, mdo, mdv, mdqp, mdkp;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  memset(&mdo, 0, sizeof(mdo));
  memset(&mdv, 0, sizeof(mdv));
  memset(&mdqp, 0, sizeof(mdqp));
  memset(&mdkp, 0, sizeof(mdkp));
  if (!tc_make_map(&mq, in.q, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(&mk, in.k, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(&mv, in.v, pr.B, pr.T, pr.Ts, pr.H) ||
      !tc_make_map(&mdo, in.dO, pr.B, pr.T, pr.Ts, pr.H) ||
      !tc_make_map(&mdv, dv, pr.B, pr.T, pr.Ts, pr.H) ||
      !tc_make_map(&mdqp, ws.dqp, pr.B, pr.Tp, pr.Tp, pr.H) ||
      !tc_make_map(&mdkp, ws.dkp, pr.B, pr.Tp, pr.Tp, pr.H))
    return cudaErrorInvalidValue;
  Grad2Args ar;
  ar.T = pr.T; ar.Ts = pr.Ts; ar.H = pr.H; ar.r = pr.r; ar.NC = pr.NC; ar.Tp = pr.Tp;
  ar.l2norm = pr.l2norm; ar.eps = pr.eps; ar.scale = pr.scale;
  ar.a = (const __nv_bfloat16*)in.a; ar.b = (const __nv_bfloat16*)in.b;
  ar.A_log = in.A_log; ar.dt_bias = in.dt_bias; ar.valid_len = in.valid_len;
  ar.dg = dg; ar.dbeta = dbeta; ar.status = ws.status;
  ar.hc = (const uint8_t*)hc; ar.dhc = (const uint8_t*)dhc;
  ar.wim = (const uint8_t*)ws.wim; ar.uim = (const uint8_t*)ws.uim;
  ar.pim = (const uint8_t*)ws.pim; ar.tim = (const uint8_t*)ws.tim;
  cudaError_t e = cudaFuncSetAttribute(k_grad2_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)GR_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)pr.NC, (unsigned)pr.H, (unsigned)pr.B);
  k_grad2_tc<<<grid, GT, GR_SMEM, st>>>(mq, mk, mv, mdo, mdv, mdqp, mdkp, ar);
  return cudaGetLastError();
}

}  // namespace gdn
