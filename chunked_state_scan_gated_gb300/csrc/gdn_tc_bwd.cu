// gdn_tc_bwd.cu -- chunk-parallel local gradients of the bf16 backward (tcgen05).
//
// Given every chunk's start state S and the gradient dS of its end state (both
// bf16, produced by the forward and reverse state chains of gdn_tc_chain.cu),
// each chunk's gradients are independent of every other chunk's; k_grad_tc
// computes them one CTA per (chunk, V head) from the chunk's inputs, recomputing
// the chunk-local intermediates (nothing per chunk is kept by the forward).
#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include <mutex>

#include "gdn_internal.h"
#include "gdn_tc_common.cuh"

namespace gdn {

// Tensor-map encoder of gdn_tc_maps.cu for the [B, Ts, heads, 128] inputs.
bool tc_make_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t Ts, int64_t heads);

namespace {

using namespace tc;

constexpr int FT = 256;

#define PHASE_SYNC()            \
  do {                          \
    fence_proxy_async();        \
    tc_fence_before();          \
    __syncthreads();            \
    tc_fence_after();           \
    if (*s_abort) goto done;    \
  } while (0)

}  // namespace

// ============================================================================
// k_grad_tc: every local gradient of one chunk and one V head, given S (the
// state at the chunk start), dS (the gradient of the state at its end), q, k,
// v, dO and the gates; one CTA per (chunk, V head, batch row), chunk-parallel.
// With X_v = T^T dV', X_w = T^T dW (Lambda of the triangular system):
//   dq  = diag(gamma) dO S^T + (dP o Gamma) K,      dP = dO V'^T (lower)
//   dk  = (dP o Gamma)^T Q + diag(kt) V' dS^T + diag(beta gamma) X_w + E K + E^T K
//   dv  = diag(beta) X_v,  dW = -dV' S^T,
//   dA  = -(X_v U^T + X_w W^T) = -X_v V'^T (strictly lower; W S = U - V'),
//   E = dA o beta_i Gamma
//   dbeta, dG: row dots of the same pieces; dg = reverse cumsum of dG.
// All MMAs are M = 64: row r of an accumulator lives in TMEM lane
// (r % 16) + 32 (r / 16), so threads with lane < 16 of each warp own one row.
namespace {

constexpr uint32_t G_Q = 0, G_K = 16384, G_W = 32768, G_V = 49152, G_DO = 65536;  // [64][128]
constexpr uint32_t G_S = 81920, G_DS = 114688;      // [128][128], atoms of 16 KB
constexpr uint32_t G_TU = 147456;                   // U [64][128] (prologue image)
constexpr uint32_t G_P = 163840, G_TP = 172032;     // [64][64]; P later E; Y of the solve in TP
constexpr uint32_t G_VP = 180224;                   // V' [64][128]; later dP o Gamma [64][64]
constexpr uint32_t G_DV = 196608, G_DW = 212992;    // dV', dW [64][128]; earlier fp32 A, T
constexpr uint32_t G_SC = 229376;                   // scalars
constexpr uint32_t G_SMEM = G_SC + 1792 + 1024;


struct GradArgs {
  int64_t T, Ts, H, r, NC, Tp;
  int l2norm;
  float eps, scale;
  const __nv_bfloat16* a;
  const __nv_bfloat16* b;
  const float* A_log;
  const float* dt_bias;
  const int32_t* valid_len;
  __nv_bfloat16* dv;   // [B, Ts, H, 128]
  float* dg;           // [B, Ts, H]
  float* dbeta;
  __nv_bfloat16* dqp;  // [B][Tp][H][128] per-V-head gradient of q_hat (bf16)
  __nv_bfloat16* dkp;
  const uint8_t* hc;   // chunk-start states, 32 KB tile images
  const uint8_t* dhc;  // chunk-end state gradients, 32 KB tile images
  const uint8_t* wim;  // prologue tile images of the chunk: W, U, P, T
  const uint8_t* uim;
  const uint8_t* pim;
  const uint8_t* tim;
  int* status;
};

__device__ __forceinline__ uint4 pack8g(const float* x) {
  uint4 v;
  v.x = pack_bf16(x[0], x[1]);
  v.y = pack_bf16(x[2], x[3]);
  v.z = pack_bf16(x[4], x[5]);
  v.w = pack_bf16(x[6], x[7]);
  return v;
}

// 64 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  float a[32], c[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, c);
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    v[j] = a[j];
    v[32 + j] = c[j];
  }
}

__global__ void __launch_bounds__(FT, 1)
    k_grad_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
              GradArgs ar) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t base = smem_u32(sm);
  float* sG = (float*)(sm + G_SC);     // cumulative gate (log2 units)
  float* sGam = sG + 64;
  float* sBeta = sGam + 64;
  float* sKt = sBeta + 64;
  float* sDG = sKt + 64;               // dG terms computed row-wise by threads 0..63
  float* sMisc = sDG + 64;             // [8] block partials of <S, dS>
  // half-row partial sums, [2][64] each, in the T tile's slot (free after R5)
  float* sRed = (float*)(sm + G_TP);   // dG
  float* sRedB = sRed + 128;           // dbeta
  float* sRedS = sRedB + 128;          // Kt terms
  uint64_t* bar_ld = (uint64_t*)(sm + G_SC + 1536);
  uint64_t* bar_mma = bar_ld + 1;
  uint32_t* s_tmem = (uint32_t*)(bar_ld + 2);
  int* s_abort = (int*)(s_tmem + 1);
  float* sZ = (float*)(sm + G_S);      // fp32 64 x 64, row stride 65, after S is consumed

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const bool own = lane < 16;          // owns accumulator row `ri` of M = 64 results
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
    // chunk tiles of the prologue: W, U (over T_u/T_w), P, T
    const int64_t im = bh * ar.NC + c;
    mbar_arrive_expect_tx(bar_ld, 131072u + 49152u);
    bulk_load(sm + G_W, ar.wim + im * 16384, 16384, bar_ld);
    bulk_load(sm + G_TU, ar.uim + im * 16384, 16384, bar_ld);
    bulk_load(sm + G_P, ar.pim + im * 8192, 8192, bar_ld);
    bulk_load(sm + G_TP, ar.tim + im * 8192, 8192, bar_ld);
    for (int at = 0; at < 2; ++at) {
      tma_load_4d(sm + G_Q + at * 8192, &mq, at * 64, (int)hq, (int)t0, (int)b, bar_ld);
      tma_load_4d(sm + G_K + at * 8192, &mk, at * 64, (int)hq, (int)t0, (int)b, bar_ld);
      tma_load_4d(sm + G_V + at * 8192, &mv, at * 64, (int)h, (int)t0, (int)b, bar_ld);
      tma_load_4d(sm + G_DO + at * 8192, &mdo, at * 64, (int)h, (int)t0, (int)b, bar_ld);
    }
    // chunk-start state and chunk-end state gradient: 32 KB tile images of the chains
    bulk_load(sm + G_S, ar.hc + im * 32768, 32768, bar_ld);
    bulk_load(sm + G_DS, ar.dhc + im * 32768, 32768, bar_ld);
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
  }
  __syncthreads();
  cumsum64f(sG);
  __syncthreads();
  if (tid < 64) {
    sGam[tid] = exp2f(sG[tid]);
    sKt[tid] = dexp_(sG[63], sG[tid]);
  }
  if (!mbar_wait(bar_ld, 0, ar.status, kStatusTimeout)) *s_abort = 1;
  // norms (in place) and padded dO rows
  for (int it = 0; it < 8; ++it) {
    const int rr = (tid >> 4) + 16 * it;
    const bool isk = rr >= 64;
    const int sub = tid & 15, at = sub >> 3, ch = sub & 7, r6 = rr & 63;
    const uint32_t off = (isk ? G_K : G_Q) + at * 8192 + kmaj_chunk(r6, ch);
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
    for (int idx = tid; idx < 1024; idx += FT) {
      const int i = idx >> 4, cc = idx & 15;
      if (t0 + i >= L)
        *reinterpret_cast<uint4*>(sm + G_DO + (cc >> 3) * 8192 + kmaj_chunk(i, cc & 7)) = make_uint4(0, 0, 0, 0);
    }
  }
  {
  uint32_t ph = 0;
  float dGacc = 0.f, dbacc = 0.f, sKacc = 0.f;  // this thread's half-row partial sums
  float dq[64], dk[64];
  const uint32_t id64 = idesc_bf16(64, 64, 0, 0);
  const uint32_t id128kn = idesc_bf16(64, 128, 0, 1);
  const uint32_t id128kk = idesc_bf16(64, 128, 0, 0);
  const uint32_t id128mn = idesc_bf16(64, 128, 1, 1);
  PHASE_SYNC();
  // ---- RT3: W S -> [384,512), K dS -> [0,128), P^T dO -> [128,256), dO S^T -> [256,384)
  if (tid == 0) {
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t at = ks >> 2, kk = ks & 3;
      mma_bf16(tmem + 384, sdesc(base + G_W + at * 8192 + kk * 32, 16, 1024),
               sdesc(base + G_S + ks * 2048, 16384, 1024), id128kn, ks > 0);
      mma_bf16(tmem, sdesc(base + G_K + at * 8192 + kk * 32, 16, 1024),
               sdesc(base + G_DS + ks * 2048, 16384, 1024), id128kn, ks > 0);
      mma_bf16(tmem + 256, sdesc(base + G_DO + at * 8192 + kk * 32, 16, 1024),
               sdesc(base + G_S + at * 16384 + kk * 32, 16, 1024), id128kk, ks > 0);
    }
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tmem + 128, sdesc(base + G_P + ks * 2048, 8192, 1024),
               sdesc(base + G_DO + ks * 2048, 8192, 1024), id128mn, ks > 0);
    mma_commit(bar_mma);
  }
  // <S, dS> (both tiles share the TMA layout): block reduction into sMisc[0]
  {
    float acc = 0.f;
    for (int q = tid; q < 2048; q += FT) {
      float x[8], y[8];
      ld_chunk(sm + G_S, q * 16, x);
      ld_chunk(sm + G_DS, q * 16, y);
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
    float ws[64], kd[64], pd[64];
    tmem_ld64(tmem + lane_off + 384 + half * 64, ws);
    tmem_ld64(tmem + lane_off + half * 64, kd);
    tmem_ld64(tmem + lane_off + 128 + half * 64, pd);
    tmem_ld64(tmem + lane_off + 256 + half * 64, dq);
    if (own) {
      const int i = ri;
      const float kt = sKt[i], gm = sGam[i];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {       // V' = U - W S (U image over T_u, T_w)
        float u[8];
        ld_chunk(sm + G_TU + half * 8192, kmaj_chunk(i, cc), u);
#pragma unroll
        for (int e = 0; e < 8; ++e) ws[cc * 8 + e] = u[e] - ws[cc * 8 + e];
      }
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        kd[j] = fmaf(kt, kd[j], pd[j]);       // dV'
        dq[j] *= gm;                          // diag(gamma) dO S^T
      }
      float part = 0.f;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        st_chunk(sm + G_VP + half * 8192, kmaj_chunk(i, cc), &ws[cc * 8]);
        st_chunk(sm + G_DV + half * 8192, kmaj_chunk(i, cc), &kd[cc * 8]);
        float qx[8];
        ld_chunk(sm + G_Q + half * 8192, kmaj_chunk(i, cc), qx);
#pragma unroll
        for (int e = 0; e < 8; ++e) part = fmaf(qx[e], dq[cc * 8 + e], part);
      }
      dGacc += part;                          // q_i . (gamma_i S dO_i)
    }
  }
  PHASE_SYNC();
  // ---- R4: dV' S^T -> [0,128), V' dS^T -> [128,256), X_v = T^T dV' -> [256,384),
  //      dP = dO V'^T -> [384,448), K K^T -> [448,512)
  if (tid == 0) {
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t at = ks >> 2, kk = ks & 3;
      mma_bf16(tmem, sdesc(base + G_DV + at * 8192 + kk * 32, 16, 1024),
               sdesc(base + G_S + at * 16384 + kk * 32, 16, 1024), id128kk, ks > 0);
      mma_bf16(tmem + 128, sdesc(base + G_VP + at * 8192 + kk * 32, 16, 1024),
               sdesc(base + G_DS + at * 16384 + kk * 32, 16, 1024), id128kk, ks > 0);
      mma_bf16(tmem + 384, sdesc(base + G_DO + at * 8192 + kk * 32, 16, 1024),
               sdesc(base + G_VP + at * 8192 + kk * 32, 16, 1024), id64, ks > 0);
      mma_bf16(tmem + 448, sdesc(base + G_K + at * 8192 + kk * 32, 16, 1024),
               sdesc(base + G_K + at * 8192 + kk * 32, 16, 1024), id64, ks > 0);
    }
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tmem + 256, sdesc(base + G_TP + ks * 2048, 8192, 1024),
               sdesc(base + G_DV + ks * 2048, 8192, 1024), id128mn, ks > 0);
    mma_commit(bar_mma);
  }
  if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
  ph ^= 1;
  tc_fence_after();
  {
    const int i = ri;
    const int64_t t = t0 + i;
    const bool valid = t < L;
    float x[64];
    tmem_ld64(tmem + lane_off + half * 64, x);   // dV' S^T = -dW
    if (own) {
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = -x[j];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) st_chunk(sm + G_DW + half * 8192, kmaj_chunk(ri, cc), &x[cc * 8]);
    }
    tmem_ld64(tmem + lane_off + 128 + half * 64, x);  // dKt = V' dS^T
    if (own) {
      const float kt = sKt[i];
      float part = 0.f;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float kx[8];
        ld_chunk(sm + G_K + half * 8192, kmaj_chunk(i, cc), kx);
#pragma unroll
        for (int e = 0; e < 8; ++e) part = fmaf(kx[e], x[cc * 8 + e], part);
      }
      sKacc = kt * part;
#pragma unroll
      for (int j = 0; j < 64; ++j) dk[j] = kt * x[j];
    }
    tmem_ld64(tmem + lane_off + 256 + half * 64, x);    // X_v
    if (own) {
      const float be = sBeta[i];
      float part = 0.f;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float vx[8];
        ld_chunk(sm + G_V + half * 8192, kmaj_chunk(i, cc), vx);
#pragma unroll
        for (int e = 0; e < 8; ++e) part = fmaf(x[cc * 8 + e], vx[e], part);
        st_chunk(sm + G_DS + half * 8192, kmaj_chunk(i, cc), &x[cc * 8]);   // X_v over dS
      }
      dbacc += part;
      if (t < ar.T) {
        uint4* dst = reinterpret_cast<uint4*>(ar.dv + ((b * ar.Ts + t) * ar.H + h) * 128 + half * 64);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = valid ? be * x[cc * 8 + e] : 0.f;
          dst[cc] = pack8g(y);
        }
      }
    }
    float dp[32];
    tmem_ld32(tmem + lane_off + 384 + half * 32, dp);
    if (own) {
      float pv[32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) ld_chunk(sm + G_P, kmaj_chunk(i, half * 4 + cc), &pv[cc * 8]);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = half * 32 + cc * 8 + e;
          const float dpv = (j <= i) ? dp[cc * 8 + e] : 0.f;
          sZ[i * 65 + j] = dpv * pv[cc * 8 + e];                   // dP o P
          y[e] = (j <= i) ? dpv * dexp_(sG[i], sG[j]) : 0.f;       // dP o Gamma
        }
        st_chunk(sm + G_W, kmaj_chunk(i, half * 4 + cc), y);      // over W (consumed)
      }
    }
  }
  PHASE_SYNC();
  if (tid < 64) {  // gate terms of P: sum_j Z_ij - sum_j Z_ji
    float acc = 0.f;
    for (int j = 0; j < 64; ++j) acc += sZ[tid * 65 + j] - sZ[j * 65 + tid];
    sDG[tid] += acc;
  }
  // ---- R5: X_w = T^T dW -> [0,128), (dP o Gamma) K -> [128,256),
  //      dA' = X_v V'^T -> [256,320) (= X_v U^T + X_w W^T, since W S = U - V')
  if (tid == 0) {
    for (int ks = 0; ks < 4; ++ks) {
      mma_bf16(tmem, sdesc(base + G_TP + ks * 2048, 8192, 1024),
               sdesc(base + G_DW + ks * 2048, 8192, 1024), id128mn, ks > 0);
      mma_bf16(tmem + 128, sdesc(base + G_W + ks * 32, 16, 1024),
               sdesc(base + G_K + ks * 2048, 8192, 1024), id128kn, ks > 0);
    }
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t at = ks >> 2, kk = ks & 3;
      mma_bf16(tmem + 256, sdesc(base + G_DS + at * 8192 + kk * 32, 16, 1024),
               sdesc(base + G_VP + at * 8192 + kk * 32, 16, 1024), id64, ks > 0);
    }
    mma_commit(bar_mma);
  }
  if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
  ph ^= 1;
  tc_fence_after();
  {
    const int i = ri;
    const int64_t t = t0 + i;
    const bool valid = t < L;
    float x[64];
    tmem_ld64(tmem + lane_off + half * 64, x);  // X_w
    if (own) {
      const float be = sBeta[i], gm = sGam[i];
      float part = 0.f;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float kx[8];
        ld_chunk(sm + G_K + half * 8192, kmaj_chunk(i, cc), kx);
#pragma unroll
        for (int e = 0; e < 8; ++e) part = fmaf(x[cc * 8 + e], kx[e], part);
      }
      dbacc += gm * part;
      dGacc += be * gm * part;
#pragma unroll
      for (int j = 0; j < 64; ++j) dk[j] = fmaf(be * gm, x[j], dk[j]);
    }
    tmem_ld64(tmem + lane_off + 128 + half * 64, x);  // (dP o Gamma) K
    if (own && t < ar.Tp) {
      uint4* dst = reinterpret_cast<uint4*>(ar.dqp + ((b * ar.Tp + t) * ar.H + h) * 128 + half * 64);
#pragma unroll
      for (int j = 0; j < 64; j += 8) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = valid ? dq[j + e] + x[j + e] : 0.f;
        dst[j >> 3] = pack8g(y);
      }
    }
    float da[32], kk[32];
    tmem_ld32(tmem + lane_off + 256 + half * 32, da);
    tmem_ld32(tmem + lane_off + 448 + half * 32, kk);
    if (own) {
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
        st_chunk(sm + G_P, kmaj_chunk(i, half * 4 + cc), ex);   // E over P
      }
      dbacc += part;
    }
  }
  PHASE_SYNC();
  if (tid < 64) {
    float acc = 0.f;
    for (int j = 0; j < 64; ++j) acc += sZ[tid * 65 + j] - sZ[j * 65 + tid];
    sDG[tid] += acc;
  }
  // ---- R6: dk += (dP o Gamma)^T Q + E K + E^T K -> [0,128)
  if (tid == 0) {
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tmem, sdesc(base + G_W + ks * 2048, 8192, 1024),
               sdesc(base + G_Q + ks * 2048, 8192, 1024), id128mn, ks > 0);
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tmem, sdesc(base + G_P + ks * 32, 16, 1024),
               sdesc(base + G_K + ks * 2048, 8192, 1024), id128kn, 1);
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tmem, sdesc(base + G_P + ks * 2048, 8192, 1024),
               sdesc(base + G_K + ks * 2048, 8192, 1024), id128mn, 1);
    mma_commit(bar_mma);
  }
  if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
  ph ^= 1;
  tc_fence_after();
  {
    float x[64];
    tmem_ld64(tmem + lane_off + half * 64, x);
    const int i = ri;
    const int64_t t = t0 + i;
    if (own && t < ar.Tp) {
      const bool valid = t < L;
      uint4* dst = reinterpret_cast<uint4*>(ar.dkp + ((b * ar.Tp + t) * ar.H + h) * 128 + half * 64);
#pragma unroll
      for (int j = 0; j < 64; j += 8) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = valid ? dk[j + e] + x[j + e] : 0.f;
        dst[j >> 3] = pack8g(y);
      }
    }
    if (own) {
      sRed[half * 64 + i] = dGacc;
      sRedB[half * 64 + i] = dbacc;
      sRedS[half * 64 + i] = sKacc;
    }
  }
  __syncthreads();
  // ---- gate gradients: Kt terms, state term, reverse cumsum
  if (tid < 64) {
    const int i = tid;
    const float s_i = sRedS[i] + sRedS[64 + i];
    float d = sDG[i] + sRed[i] + sRed[64 + i];
    if (i < 63) d -= s_i;
    sDG[i] = d;
    sRed[i] = (i < 63) ? s_i : 0.f;   // reuse: Kt terms to sum into dG_C
  }
  __syncthreads();
  if (tid == 0) {
    float tot = 0.f;
    for (int i = 0; i < 63; ++i) tot += sRed[i];
    float sd = 0.f;
    for (int w = 0; w < FT / 32; ++w) sd += sMisc[w];
    sDG[63] += tot + sGam[63] * sd;
  }
  __syncthreads();
  if (tid < 32) {  // dg_j = sum_{i >= j} dG_i (reverse cumsum, warp 0)
    float v0 = sDG[63 - tid], v1 = sDG[31 - tid];
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
    sDG[63 - tid] = v0;
    sDG[31 - tid] = v1;
  }
  __syncthreads();
  if (tid < 64) {
    const int64_t t = t0 + tid;
    if (t < ar.T) {
      const int64_t gi = (b * ar.Ts + t) * ar.H + h;
      const bool valid = t < L;
      // dG was accumulated in natural-log units (the log2 scaling only enters exponents)
      ar.dg[gi] = valid ? sDG[tid] : 0.f;
      ar.dbeta[gi] = valid ? sRedB[tid] + sRedB[64 + tid] : 0.f;
    }
  }
  }
done:
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

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

cudaError_t launch_grad_tc(const Prob& pr, const Inputs& in, const WS& ws, const void* hc,
                           const void* dhc, void* dv, float* dg, float* dbeta, cudaStream_t st) {
  if (pr.B == 0 || pr.NC == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv, mdo;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  memset(&mdo, 0, sizeof(mdo));
  if (!tc_make_map(&mq, in.q, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(&mk, in.k, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(&mv, in.v, pr.B, pr.T, pr.Ts, pr.H) ||
      !tc_make_map(&mdo, in.dO, pr.B, pr.T, pr.Ts, pr.H))
    return cudaErrorInvalidValue;
  GradArgs ar;
  ar.T = pr.T; ar.Ts = pr.Ts; ar.H = pr.H; ar.r = pr.r; ar.NC = pr.NC; ar.Tp = pr.Tp;
  ar.l2norm = pr.l2norm; ar.eps = pr.eps; ar.scale = pr.scale;
  ar.a = (const __nv_bfloat16*)in.a; ar.b = (const __nv_bfloat16*)in.b;
  ar.A_log = in.A_log; ar.dt_bias = in.dt_bias; ar.valid_len = in.valid_len;
  ar.dv = (__nv_bfloat16*)dv; ar.dg = dg; ar.dbeta = dbeta;
  ar.dqp = (__nv_bfloat16*)ws.dqp; ar.dkp = (__nv_bfloat16*)ws.dkp; ar.status = ws.status;
  ar.hc = (const uint8_t*)hc; ar.dhc = (const uint8_t*)dhc;
  ar.wim = (const uint8_t*)ws.wim; ar.uim = (const uint8_t*)ws.uim;
  ar.pim = (const uint8_t*)ws.pim; ar.tim = (const uint8_t*)ws.tim;
  cudaError_t e = cudaFuncSetAttribute(k_grad_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)G_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)pr.NC, (unsigned)pr.H, (unsigned)pr.B);
  k_grad_tc<<<grid, FT, G_SMEM, st>>>(mq, mk, mv, mdo, ar);
  return cudaGetLastError();
}

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
