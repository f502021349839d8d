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
// the CTA owns one feature row and 16 token columns.  Only the token x token
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

constexpr int GT = 512;
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
constexpr uint32_t SC_BYTES = 7 * 64 * 4 + 4 * 4 * 64 * 4 + 4 * 64 * 4 + 8 * 64 * 4 + 64;  // + 4 barriers
constexpr uint32_t GR_SMEM = R_SC + SC_BYTES + 1024;
static_assert(GR_SMEM <= 232448, "shared memory of k_grad2_tc");

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

// 16 consecutive fp32 columns of this thread's TMEM lane (warp-wide).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Transpose-reduce of p[16] over the warp: lanes l and l ^ 16 both end with the sum
// over all 32 lanes of p[l & 15] (15 + 1 shuffles).
template <int K>
__device__ __forceinline__ void xr_stage(float (&p)[16], int lane) {
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const bool up = (lane & K) != 0;
    const float send = up ? p[i] : p[i + K];
    const float keep = up ? p[i + K] : p[i];
    p[i] = keep + __shfl_xor_sync(0xffffffffu, send, K);
  }
}
__device__ __forceinline__ float xreduce16(float (&p)[16], int lane) {
  xr_stage<8>(p, lane);
  xr_stage<4>(p, lane);
  xr_stage<2>(p, lane);
  xr_stage<1>(p, lane);
  return p[0] + __shfl_xor_sync(0xffffffffu, p[0], 16);
}

// Element (t, f) of a token-major [64][128] bf16 tile (two K-major atoms).
__device__ __forceinline__ uint32_t tf_off(int t, int f) {
  return (uint32_t)((f >> 6) * 8192 + t * 128 + (((((f & 63) >> 3) ^ t) & 7) << 4) + (f & 7) * 2);
}
// Element (i, j) of a 64 x 64 fp32 scratch matrix (XOR-swizzled rows: a warp reading a
// row or a column of it touches 32 distinct banks).
__device__ __forceinline__ int zoff(int i, int j) { return i * 64 + (j ^ (i & 31)); }
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

// 512 threads: warp w reads TMEM lane quadrant q = w & 3 and token columns
// 16 (w >> 2) .. +15.  In an M = 128 result thread (q, lane) owns feature row
// 32 q + lane; in an M = 64 result (row r in lane (r % 16) + 32 (r / 16)) lanes
// 0..15 of quadrant q own token row 16 q + lane.
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
  float* sDB = sKt + 64;               // dbeta (final)
  float* sFin = sDB + 64;              // final dG
  float* sMisc = sFin + 64;            // [16] warp partials of <S, dS>
  float* sRed = sMisc + 64;            // [4 types][4 quadrants][64 tokens] column partials
  float* sDBh = sRed + 4 * 4 * 64;     // [4 column parts][64] dbeta terms of A
  float* sPart = sDBh + 4 * 64;        // [8 parts][64] gate terms of P and A (row - column sums)
  uint64_t* bar_qk = (uint64_t*)(sPart + 8 * 64);  // q, k tiles
  uint64_t* bar_a = bar_qk + 1;                      // S, dS, W, dO, P (round A)
  uint64_t* bar_b = bar_qk + 2;                      // U, V, T
  uint64_t* bar_mma = bar_qk + 3;
  uint32_t* s_tmem = (uint32_t*)(bar_qk + 4);
  int* s_abort = (int*)(s_tmem + 1);
  float* sZb = (float*)(sm + R_S);           // dP o P (round B), once S is consumed
  float* sZc = (float*)(sm + R_S + 16384);   // dA o A (round C)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, part = warp >> 2;
  const int fr = quad * 32 + lane;     // feature row (TMEM lane) of M = 128 results
  const int cb = 16 * part;            // first token column of this thread
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
    mbar_init(bar_qk, 1);
    mbar_init(bar_a, 1);
    mbar_init(bar_b, 1);
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
    mbar_arrive_expect_tx(bar_qk, 2 * 16384u);
    for (int at = 0; at < 2; ++at) {
      tma_load_4d(sm + R_Q + at * 8192, &mq, at * 64, (int)hq, (int)t0, (int)b, bar_qk);
      tma_load_4d(sm + R_K + at * 8192, &mk, at * 64, (int)hq, (int)t0, (int)b, bar_qk);
    }
    mbar_arrive_expect_tx(bar_a, 2 * 32768u + 2 * 16384u + 8192u);
    bulk_load(sm + R_S, ar.hc + im * 32768, 32768, bar_a);
    bulk_load(sm + R_W, ar.wim + im * 16384, 16384, bar_a);
    bulk_load(sm + R_DS, ar.dhc + im * 32768, 32768, bar_a);
    for (int at = 0; at < 2; ++at)
      tma_load_4d(sm + R_DO + at * 8192, &mdo, at * 64, (int)h, (int)t0, (int)b, bar_a);
    bulk_load(sm + R_P, ar.pim + im * 8192, 8192, bar_a);
    mbar_arrive_expect_tx(bar_b, 2 * 16384u + 8192u);
    bulk_load(sm + R_U, ar.uim + im * 16384, 16384, bar_b);
    bulk_load(sm + R_T, ar.tim + im * 8192, 8192, bar_b);
    for (int at = 0; at < 2; ++at)
      tma_load_4d(sm + R_V + at * 8192, &mv, at * 64, (int)h, (int)t0, (int)b, bar_b);
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
  }
  __syncthreads();
  cumsum64f(sG);
  __syncthreads();
  if (tid < 64) {
    sGam[tid] = exp2f(sG[tid]);
    sKt[tid] = dexp_(sG[63], sG[tid]);
  }
  if (!mbar_wait(bar_qk, 0, ar.status, kStatusTimeout)) *s_abort = 1;
  // q, k rows normalised in place (16 threads per row); padded dO rows zeroed
  for (int it = 0; it < 4; ++it) {
    const int rr = (tid >> 4) + 32 * it;
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
  if (!mbar_wait(bar_a, 0, ar.status, kStatusTimeout)) *s_abort = 1;
  if (t0 + 64 > L) {
    for (int idx = tid; idx < 1024; idx += GT) {
      const int i = idx >> 4, cc = idx & 15;
      if (t0 + i >= L)
        *reinterpret_cast<uint4*>(sm + R_DO + (cc >> 3) * 8192 + kmaj_chunk(i, cc & 7)) = make_uint4(0, 0, 0, 0);
    }
  }
  {
    // Descriptors of every operand tile: the start address sits in the low 14 bits
    // (address >> 4), so a tile at byte offset `off` is the base descriptor + off / 16.
    const uint64_t d16 = sdesc(base, 16, 1024), d8192 = sdesc(base, 8192, 1024),
                   d16384 = sdesc(base, 16384, 1024);
    auto dsc16 = [&](uint32_t off) { return d16 + (off >> 4); };
    auto dsc8192 = [&](uint32_t off) { return d8192 + (off >> 4); };
    auto dsc16384 = [&](uint32_t off) { return d16384 + (off >> 4); };
    uint32_t ph = 0;
    float dqT[16], dkT[16];  // this thread's feature row fr of dq_hat^T, dk_hat^T, tokens cb + e
    const uint32_t idA = idesc_bf16(128, 64, 1, 0);  // A MN-major (feature rows), B K-major
    const uint32_t idB = idesc_bf16(128, 64, 0, 1);  // A K-major, B MN-major
    const uint32_t idC = idesc_bf16(128, 64, 1, 1);  // both MN-major
    const uint32_t idD = idesc_bf16(128, 64, 0, 0);  // both K-major
    GRAD_SYNC();
    // ---- round A: S^T W^T -> [0,64), dO^T P -> [64,128), dS^T K^T -> [128,192),
    //      S dO^T -> [192,256), K K^T -> [256,320) (M = 64; read in round C's epilogue)
    if (tid == 0) {
      const uint32_t id64d = idesc_bf16(64, 64, 0, 0);
      for (int ks = 0; ks < 8; ++ks) {  // K = dk (S^T W^T, dS^T K^T, K K^T) or dv (S dO^T)
        const uint32_t at = ks >> 2, kk = ks & 3;
        mma_bf16(tmem, dsc16384(R_S + ks * 2048),
                 dsc16(R_W + at * 8192 + kk * 32), idA, ks > 0);
        mma_bf16(tmem + 128, dsc16384(R_DS + ks * 2048),
                 dsc16(R_K + at * 8192 + kk * 32), idA, ks > 0);
        mma_bf16(tmem + 192, dsc16(R_S + at * 16384 + kk * 32),
                 dsc16(R_DO + at * 8192 + kk * 32), idD, ks > 0);
        mma_bf16(tmem + 256, dsc16(R_K + at * 8192 + kk * 32),
                 dsc16(R_K + at * 8192 + kk * 32), id64d, ks > 0);
      }
      for (int ks = 0; ks < 4; ++ks)  // K = tokens
        mma_bf16(tmem + 64, dsc8192(R_DO + ks * 2048),
                 dsc8192(R_P + ks * 2048), idC, ks > 0);
      mma_commit(bar_mma);
    }
    {  // <S, dS> (same tile layout): warp partials into sMisc
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
    if (!mbar_wait(bar_b, 0, ar.status, kStatusTimeout)) *s_abort = 1;
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    {  // V'^T and dV'^T: the operands of round B
      const int f = fr;
      float ws[16], a1[16], a2[16];
      tmem_ld16(tmem + lane_off + cb, ws);
      tmem_ld16(tmem + lane_off + 64 + cb, a1);
      tmem_ld16(tmem + lane_off + 128 + cb, a2);
      tmem_ld16(tmem + lane_off + 192 + cb, dqT);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        ws[e] = ld_bf(sm + R_U + tf_off(t, f)) - ws[e];   // V'^T
        a1[e] = fmaf(sKt[t], a2[e], a1[e]);                 // dV'^T
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        st_chunk(sm + R_VT, kmaj_chunk(f, 2 * part + cc), &ws[cc * 8]);
        st_chunk(sm + R_DVT, kmaj_chunk(f, 2 * part + cc), &a1[cc * 8]);
      }
    }
    GRAD_SYNC();
    // ---- round B: S dV'^T -> [0,64) (-dW^T), dS V'^T -> [64,128), dV'^T T -> [128,192) (X_v^T),
    //      dO V'^T -> [192,256) (dP, M = 64)
    if (tid == 0) {
      const uint32_t id64b = idesc_bf16(64, 64, 0, 1);
      for (int ks = 0; ks < 8; ++ks) {  // K = dv
        const uint32_t at = ks >> 2, kk = ks & 3;
        mma_bf16(tmem, dsc16(R_S + at * 16384 + kk * 32),
                 dsc8192(R_DVT + ks * 2048), idB, ks > 0);
        mma_bf16(tmem + 64, dsc16(R_DS + at * 16384 + kk * 32),
                 dsc8192(R_VT + ks * 2048), idB, ks > 0);
        mma_bf16(tmem + 192, dsc16(R_DO + at * 8192 + kk * 32),
                 dsc8192(R_VT + ks * 2048), id64b, ks > 0);
      }
      for (int ks = 0; ks < 4; ++ks)  // K = tokens
        mma_bf16(tmem + 128, dsc16(R_DVT + ks * 32),
                 dsc8192(R_T + ks * 2048), idB, ks > 0);
      mma_commit(bar_mma);
    }
    {  // while round B runs: (diag(gamma) dO S^T)^T and q_t . (gamma_t S dO_t)
      const int f = fr;
      float pq[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        dqT[e] *= sGam[t];
        pq[e] = ld_bf(sm + R_Q + tf_off(t, f)) * dqT[e];
      }
      const float red = xreduce16(pq, lane);
      if (lane < 16) sRed[(RQ * 4 + quad) * 64 + cb + lane] = red;
    }
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    {  // -dW^T, X_v^T and dP o Gamma: the operands of round C
      const int f = fr;
      float x[16];
      tmem_ld16(tmem + lane_off + cb, x);                  // S dV'^T = -dW^T
#pragma unroll
      for (int e = 0; e < 16; ++e) x[e] = -x[e];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) st_chunk(sm + R_W, kmaj_chunk(f, 2 * part + cc), &x[cc * 8]);
      tmem_ld16(tmem + lane_off + 128 + cb, x);            // X_v^T
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) st_chunk(sm + R_U, kmaj_chunk(f, 2 * part + cc), &x[cc * 8]);
      float dp[16];
      tmem_ld16(tmem + lane_off + 192 + cb, dp);           // dP (M = 64 layout)
      if (own64) {
        const int i = ri;
        float pv[16];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) ld_chunk(sm + R_P, kmaj_chunk(i, 2 * part + cc), &pv[cc * 8]);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = cb + cc * 8 + e;
            const float dpv = (j <= i) ? dp[cc * 8 + e] : 0.f;
            sZb[zoff(i, j)] = dpv * pv[cc * 8 + e];                 // dP o P
            y[e] = (j <= i) ? dpv * dexp_(sG[i], sG[j]) : 0.f;      // dP o Gamma
          }
          st_chunk(sm + R_P, kmaj_chunk(i, 2 * part + cc), y);       // over P (this thread's)
        }
      }
    }
    GRAD_SYNC();
    // ---- round C: dW^T T -> [320,384) (X_w^T), K^T (dP o Gamma)^T -> [384,448),
    //      X_v V'^T -> [448,512) (dA', M = 64); K K^T stays in [256,320)
    if (tid == 0) {
      const uint32_t id64c = idesc_bf16(64, 64, 1, 1);
      for (int ks = 0; ks < 4; ++ks) {  // K = tokens
        mma_bf16(tmem + 320, dsc16(R_W + ks * 32),
                 dsc8192(R_T + ks * 2048), idB, ks > 0);
        mma_bf16(tmem + 384, dsc8192(R_K + ks * 2048),
                 dsc16(R_P + ks * 32), idA, ks > 0);
      }
      for (int ks = 0; ks < 8; ++ks)  // K = dv
        mma_bf16(tmem + 448, dsc8192(R_U + ks * 2048),
                 dsc8192(R_VT + ks * 2048), id64c, ks > 0);
      mma_commit(bar_mma);
    }
    {  // while round C runs: Kt part of dk, dv, and the row dots of V' dS^T and X_v
      const int f = fr;
      float x[16], pk[16];
      tmem_ld16(tmem + lane_off + 64 + cb, x);             // (V' dS^T)^T
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        dkT[e] = sKt[t] * x[e];
        pk[e] = ld_bf(sm + R_K + tf_off(t, f)) * x[e];    // k_t . (V' dS^T)_t
      }
      float red = xreduce16(pk, lane);
      if (lane < 16) sRed[(RKD * 4 + quad) * 64 + cb + lane] = red;
      tmem_ld16(tmem + lane_off + 128 + cb, x);            // X_v^T
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        pk[e] = ld_bf(sm + R_V + tf_off(t, f)) * x[e];    // v_t . X_v,t
        st_bf(sm + R_DO + tf_off(t, f), (t0 + t < L) ? sBeta[t] * x[e] : 0.f);  // dv staging
      }
      red = xreduce16(pk, lane);
      if (lane < 16) sRed[(RV * 4 + quad) * 64 + cb + lane] = red;
    }
    {  // gate terms of P: sum_j Z_ij - sum_j Z_ji, 8 column parts of 8
      const int i = tid & 63, p8 = tid >> 6;
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = p8 * 8 + e;
        acc += sZb[zoff(i, j)] - sZb[zoff(j, i)];
      }
      sPart[p8 * 64 + i] = acc;
    }
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    {  // E (operand of round D), dA o A, dbeta terms of A
      float da[16], kk[16];
      tmem_ld16(tmem + lane_off + 448 + cb, da);           // dA' (M = 64 layout)
      tmem_ld16(tmem + lane_off + 256 + cb, kk);           // K K^T (M = 64 layout)
      if (own64) {
        const int i = ri;
        const float be = sBeta[i];
        float pt = 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float ex[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = cb + cc * 8 + e;
            const float gmm = (j < i) ? dexp_(sG[i], sG[j]) : 0.f;
            const float dA = (j < i) ? -da[cc * 8 + e] : 0.f;
            const float kg = kk[cc * 8 + e] * gmm;
            pt = fmaf(dA, kg, pt);                     // dbeta: dA (k_i . k_j) Gamma
            sZc[zoff(i, j)] = dA * be * kg;            // dA o A
            ex[e] = dA * be * gmm;                     // E
          }
          st_chunk(sm + R_T, kmaj_chunk(i, 2 * part + cc), ex);   // E over T
        }
        sDBh[part * 64 + i] = pt;
      }
    }
    GRAD_SYNC();
    // ---- round D: Q^T (dP o Gamma) + K^T E^T + K^T E -> [0,64)
    if (tid == 0) {
      tma_store_4d(&mdv, sm + R_DO, 0, (int)h, (int)t0, (int)b);  // dv tile (clipped past T)
      tma_store_4d(&mdv, sm + R_DO + 8192, 64, (int)h, (int)t0, (int)b);
      bulk_commit();
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem, dsc8192(R_Q + ks * 2048),
                 dsc8192(R_P + ks * 2048), idC, ks > 0);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem, dsc8192(R_K + ks * 2048),
                 dsc16(R_T + ks * 32), idA, 1);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem, dsc8192(R_K + ks * 2048),
                 dsc8192(R_T + ks * 2048), idC, 1);
      mma_commit(bar_mma);
    }
    {  // while round D runs: X_w part of dk, dq_hat staging, row dots of X_w
      const int f = fr;
      float x[16], pk[16];
      tmem_ld16(tmem + lane_off + 320 + cb, x);            // X_w^T
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        const float bg = sBeta[t] * sGam[t];
        dkT[e] = fmaf(bg, x[e], dkT[e]);
        pk[e] = ld_bf(sm + R_K + tf_off(t, f)) * x[e];    // k_t . X_w,t
      }
      const float red = xreduce16(pk, lane);
      if (lane < 16) sRed[(RKW * 4 + quad) * 64 + cb + lane] = red;
      tmem_ld16(tmem + lane_off + 384 + cb, x);            // (dP o Gamma) K, transposed
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        st_bf(sm + R_DS + tf_off(t, f), (t0 + t < L) ? dqT[e] + x[e] : 0.f);  // dq_hat staging
      }
    }
    {  // gate terms of A, added to this thread's slot of the P terms
      const int i = tid & 63, p8 = tid >> 6;
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = p8 * 8 + e;
        acc += sZc[zoff(i, j)] - sZc[zoff(j, i)];
      }
      sPart[p8 * 64 + i] += acc;
    }
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    {
      const int f = fr;
      float x[16];
      tmem_ld16(tmem + lane_off + cb, x);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        st_bf(sm + R_DS + 16384 + tf_off(t, f), (t0 + t < L) ? dkT[e] + x[e] : 0.f);  // dk_hat
      }
    }
    GRAD_SYNC();
    if (tid == 0) {
      tma_store_4d(&mdqp, sm + R_DS, 0, (int)h, (int)t0, (int)b);  // dq_hat tile
      tma_store_4d(&mdqp, sm + R_DS + 8192, 64, (int)h, (int)t0, (int)b);
      tma_store_4d(&mdkp, sm + R_DS + 16384, 0, (int)h, (int)t0, (int)b);
      tma_store_4d(&mdkp, sm + R_DS + 16384 + 8192, 64, (int)h, (int)t0, (int)b);
      bulk_commit();
    }
    // ---- gate gradients: column sums of the four row dots, Kt terms, state term
    if (tid < 64) {
      const int t = tid;
      float rq = 0.f, rv = 0.f, rkw = 0.f, rkd = 0.f, zp = 0.f;
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        rq += sRed[(RQ * 4 + qd) * 64 + t];
        rv += sRed[(RV * 4 + qd) * 64 + t];
        rkw += sRed[(RKW * 4 + qd) * 64 + t];
        rkd += sRed[(RKD * 4 + qd) * 64 + t];
      }
#pragma unroll
      for (int p8 = 0; p8 < 8; ++p8) zp += sPart[p8 * 64 + t];
      const float be = sBeta[t], gm = sGam[t];
      const float s_t = sKt[t] * rkd;                       // Kt term of dG_t
      float d = zp + rq + be * gm * rkw;
      if (t < 63) d -= s_t;
      sFin[t] = d;
      sDB[t] = rv + gm * rkw + sDBh[t] + sDBh[64 + t] + sDBh[128 + t] + sDBh[192 + t];
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
  if (*s_abort && tid == 0) {  // let the loads still in flight land before the CTA exits
    mbar_wait(bar_qk, 0, nullptr, 0);
    mbar_wait(bar_a, 0, nullptr, 0);
    mbar_wait(bar_b, 0, nullptr, 0);
  }
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
