// gdn_simt.cu -- fp32 CUDA-core kernels of the chunked gated delta rule.
//
// This is the exact-arithmetic path (fp32 FMAs, never TF32): it serves the fp32
// I/O mode and is the semantic anchor of the tensor-core kernels.  The chunked
// form evaluated here, per (batch row, V head) and chunk of C = 64 tokens with
// chunk-start state S (dk x dv):
//
//   G_i = sum_{j<=i} g_j, gamma_i = exp(G_i), Gamma_ij = exp(G_i - G_j) (i >= j)
//   A   = tril(diag(beta) K K^T o Gamma, -1),  T = (I + A)^-1
//   W   = T diag(beta gamma) K,  U = T diag(beta) V
//   V'  = U - W S
//   O   = diag(gamma) Q S + tril(Q K^T o Gamma) V'
//   S  <- gamma_C S + Kt^T V',  Kt_j = exp(G_C - G_j) k_j
//
// The chunk size 64 and head dim 128 are the pages' fused-backend shape
// ("Linear Attention CP 融合算子 PR #1114 测试报告", section 3.1); the affine
// segment summary [M | S] and its composition come from "linear attention cp
// #1035", section "What does this PR do" (p2p / all_gather modes).
//
// The cumulative gate G is kept in fp64: with the default gate distribution it
// reaches about -500 inside a chunk, and fp32 differences G_i - G_j would carry
// ~3e-5 absolute error into every decay factor exp(G_i - G_j).
//
// Work is split into: a chunk-parallel prologue (norms, gates, T, W, U), a
// sequential state pass per (V head, column slice, segment), a chunk-parallel
// output pass, a reverse state-gradient pass and a chunk-parallel gradient pass.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int NT = 256;      // threads per block
constexpr int CS = 32;       // state columns per scan block
constexpr int CSO = 64;      // output columns per output block
constexpr int LS = 65;       // leading dim of 64x64 tiles

template <typename TIn>
__device__ __forceinline__ float ldf(const TIn* p, int64_t i);
template <>
__device__ __forceinline__ float ldf<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}
template <typename TIn>
__device__ __forceinline__ void stf(TIn* p, int64_t i, float x);
template <>
__device__ __forceinline__ void stf<float>(float* p, int64_t i, float x) { p[i] = x; }
template <>
__device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16* p, int64_t i, float x) {
  p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Valid length of row b, clamped to [0, T]; flags the status word when clamping.
__device__ __forceinline__ int64_t row_len(const int32_t* valid_len, int64_t b, int64_t T,
                                           int* status, bool flag) {
  if (!valid_len) return T;
  int64_t L = valid_len[b];
  if (L < 0 || L > T) {
    if (flag && status && threadIdx.x == 0) atomicOr(status, kStatusClamped);
    L = L < 0 ? 0 : T;
  }
  return L;
}

// C(i,j) = alpha * sum_l A(i,l) B(l,j) (+ C(i,j) when accumulate), i < m, j < n.
// A(i,l) = A[i*sam + l*sak], B(l,j) = B[l*sbk + j*sbn], C(i,j) = C[i*scm + j*scn].
// 4x4 register micro-tiles strided over the block.  C must not alias A or B.
__device__ void blk_gemm(int m, int n, int kk, float alpha, const float* __restrict__ A,
                         int64_t sam, int64_t sak, const float* __restrict__ B, int64_t sbk,
                         int64_t sbn, bool accumulate, float* C, int64_t scm, int64_t scn) {
  const int tm = (m + 3) >> 2, tn = (n + 3) >> 2;
  for (int tile = threadIdx.x; tile < tm * tn; tile += blockDim.x) {
    const int i0 = (tile / tn) * 4, j0 = (tile % tn) * 4;
    float acc[4][4];
#pragma unroll
    for (int ii = 0; ii < 4; ++ii)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) acc[ii][jj] = 0.f;
    for (int l = 0; l < kk; ++l) {
      float av[4], bv[4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) av[ii] = (i0 + ii < m) ? A[(i0 + ii) * sam + l * sak] : 0.f;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) bv[jj] = (j0 + jj < n) ? B[l * sbk + (j0 + jj) * sbn] : 0.f;
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[ii][jj] = fmaf(av[ii], bv[jj], acc[ii][jj]);
    }
#pragma unroll
    for (int ii = 0; ii < 4; ++ii)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
        if (i0 + ii < m && j0 + jj < n) {
          float* c = C + (i0 + ii) * scm + (j0 + jj) * scn;
          *c = accumulate ? fmaf(alpha, acc[ii][jj], *c) : alpha * acc[ii][jj];
        }
  }
}

// Inclusive prefix sum of x[0..63] in place, by warp 0.
__device__ void cumsum64(double* x) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    double v0 = x[lane], v1 = x[lane + 32];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      double y0 = __shfl_up_sync(0xffffffffu, v0, o);
      double y1 = __shfl_up_sync(0xffffffffu, v1, o);
      if (lane >= o) {
        v0 += y0;
        v1 += y1;
      }
    }
    v1 += __shfl_sync(0xffffffffu, v0, 31);
    x[lane] = v0;
    x[lane + 32] = v1;
  }
}

// Reverse (suffix) sum of x[0..63] in place: x_j <- sum_{i >= j} x_i, by warp 0.
__device__ void revsum64(float* x) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float v0 = x[31 - lane + 32], v1 = x[31 - lane];  // reversed order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      float y0 = __shfl_up_sync(0xffffffffu, v0, o);
      float y1 = __shfl_up_sync(0xffffffffu, v1, o);
      if (lane >= o) {
        v0 += y0;
        v1 += y1;
      }
    }
    v1 += __shfl_sync(0xffffffffu, v0, 31);
    __syncwarp();
    x[63 - lane] = v0;
    x[31 - lane] = v1;
  }
}

// exp(Ga - Gb) from fp64 cumulative gates (the difference is taken in fp64).
__device__ __forceinline__ float dexp(double ga, double gb) { return expf((float)(ga - gb)); }

struct KArgs {
  int64_t B, T, Ts, Hqk, H, dk, dv, r, NC, Tp, CPS;
  int P, l2norm;
  float eps, scale;
};

KArgs kargs(const Prob& p) {
  KArgs a;
  a.B = p.B; a.T = p.T; a.Ts = p.Ts; a.Hqk = p.Hqk; a.H = p.H; a.dk = p.dk; a.dv = p.dv;
  a.r = p.r; a.NC = p.NC; a.Tp = p.Tp; a.CPS = p.CPS; a.P = p.P; a.l2norm = p.l2norm;
  a.eps = p.eps; a.scale = p.scale;
  return a;
}

// ------------------------------------------------------------------ prologue
// grid (NC, Hqk, B): normalise q, k of the chunk (once per Q/K head), then per V
// head of the group: gates, cumulative gate, A, T = (I + A)^-1, W and U.
template <typename TIn>
__global__ void __launch_bounds__(NT) k_prep(KArgs ka, const TIn* __restrict__ q,
                                            const TIn* __restrict__ k, const TIn* __restrict__ v,
                                            const TIn* __restrict__ a, const TIn* __restrict__ bb,
                                            const float* __restrict__ A_log,
                                            const float* __restrict__ dt_bias,
                                            const int32_t* __restrict__ valid_len, WS ws,
                                            int need_q, int need_T) {
  extern __shared__ double smd[];
  const int dk = (int)ka.dk, dv = (int)ka.dv;
  const int LK = dk + 1, LV = dv + 1;
  double* gG = smd;                     // [64] cumulative gate (fp64)
  float* sm = (float*)(smd + 64);
  float* Ks = sm;               // [64][LK]
  float* Vs = Ks + 64 * LK;     // [64][LV]
  float* As = Vs + 64 * LV;     // [64][LS]
  float* Tms = As + 64 * LS;    // [64][LS]
  float* T2 = Tms + 64 * LS;    // [64][LS]
  float* gB = T2 + 64 * LS;     // [64]
  const int64_t c = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
  const int64_t t0 = c * kChunk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t L = row_len(valid_len, b, ka.T, ws.status, hq == 0 && c == 0);

  // q and k rows: one warp per token, norm over dk
  for (int i = warp; i < kChunk; i += NT / 32) {
    const int64_t t = t0 + i;
    const bool in = t < ka.T;
    const int64_t src = ((b * ka.Ts + t) * ka.Hqk + hq) * ka.dk;
    const int64_t dst = ((b * ka.Hqk + hq) * ka.Tp + t) * ka.dk;
    for (int which = 0; which < 2; ++which) {
      if (which == 0 && !need_q) continue;
      const TIn* x = which == 0 ? q : k;
      float xv[4];
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = lane + 32 * e;
        xv[e] = (in && col < dk) ? ldf(x, src + col) : 0.f;
        ss = fmaf(xv[e], xv[e], ss);
      }
      ss = warp_sum(ss);
      float s = ka.l2norm ? rsqrtf(ss + ka.eps) : 1.f;
      if (which == 0) s *= ka.scale;
      float* outp = which == 0 ? ws.Qh : ws.Kh;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = lane + 32 * e;
        if (col < dk) {
          outp[dst + col] = xv[e] * s;
          if (which == 1) Ks[i * LK + col] = xv[e] * s;
        }
      }
    }
  }
  __syncthreads();

  for (int64_t h = hq * ka.r; h < (hq + 1) * ka.r; ++h) {
    const int64_t bh = b * ka.H + h;
    if (tid < kChunk) {
      const int64_t t = t0 + tid;
      float g = 0.f, be = 0.f;
      if (t < L) {
        const int64_t gi = (b * ka.Ts + t) * ka.H + h;
        const float x = ldf(a, gi) + dt_bias[h];
        const float sp = x > 20.f ? x : log1pf(expf(x));
        g = -expf(A_log[h]) * sp;
        be = 1.f / (1.f + expf(-ldf(bb, gi)));
      }
      gG[tid] = (double)g;
      gB[tid] = be;
    }
    __syncthreads();
    cumsum64(gG);
    __syncthreads();
    if (tid < kChunk) {
      ws.G[bh * ka.Tp + t0 + tid] = gG[tid];
      ws.Bt[bh * ka.Tp + t0 + tid] = gB[tid];
    }
    // A = tril(diag(beta) K K^T o Gamma, -1)
    blk_gemm(kChunk, kChunk, dk, 1.f, Ks, LK, 1, Ks, 1, LK, false, As, LS, 1);
    __syncthreads();
    for (int e = tid; e < kChunk * kChunk; e += NT) {
      const int i = e >> 6, j = e & 63;
      As[i * LS + j] = (i > j) ? gB[i] * As[i * LS + j] * dexp(gG[i], gG[j]) : 0.f;
    }
    __syncthreads();
    // T = (I + A)^-1 by forward substitution, one column per thread
    if (tid < kChunk) {
      const int j = tid;
      for (int i = 0; i < kChunk; ++i) {
        float x = 0.f;
        if (i == j) {
          x = 1.f;
        } else if (i > j) {
          for (int l = j; l < i; ++l) x = fmaf(-As[i * LS + l], Tms[l * LS + j], x);
        }
        Tms[i * LS + j] = x;
      }
    }
    __syncthreads();
    if (need_T && ws.Tm) {
      float* Tg = ws.Tm + (bh * ka.NC + c) * (kChunk * kChunk);
      for (int e = tid; e < kChunk * kChunk; e += NT) Tg[e] = Tms[(e >> 6) * LS + (e & 63)];
    }
    // W = T diag(beta gamma) K
    for (int e = tid; e < kChunk * kChunk; e += NT) {
      const int i = e >> 6, j = e & 63;
      T2[i * LS + j] = Tms[i * LS + j] * gB[j] * dexp(gG[j], 0.0);
    }
    __syncthreads();
    blk_gemm(kChunk, dk, kChunk, 1.f, T2, LS, 1, Ks, LK, 1, false, ws.W + (bh * ka.Tp + t0) * dk,
             dk, 1);
    __syncthreads();
    // U = T diag(beta) V (skipped when v is not given: the gradient summary never reads U)
    if (v == nullptr) continue;
    for (int e = tid; e < kChunk * dv; e += NT) {
      const int i = e / dv, col = e % dv;
      const int64_t t = t0 + i;
      Vs[i * LV + col] = t < ka.T ? ldf(v, ((b * ka.Ts + t) * ka.H + h) * ka.dv + col) : 0.f;
    }
    for (int e = tid; e < kChunk * kChunk; e += NT) {
      const int i = e >> 6, j = e & 63;
      T2[i * LS + j] = Tms[i * LS + j] * gB[j];
    }
    __syncthreads();
    blk_gemm(kChunk, dv, kChunk, 1.f, T2, LS, 1, Vs, LV, 1, false, ws.U + (bh * ka.Tp + t0) * dv,
             dv, 1);
    __syncthreads();
  }
}

// ---------------------------------------------------------------- state scan
// grid (ceil(width / CS), H, B * nseg).  mode 0: state of width dv from `init`;
// mode 1: [M | S] of width dk + dv from [I | 0].
__global__ void __launch_bounds__(NT) k_state_scan(KArgs ka, WS ws, int mode, int seg_first,
                                                  int nseg, const float* __restrict__ init,
                                                  int64_t init_seg_stride, float* Hc, float* Vn,
                                                  float* final_out, float* M_out, float* S_out,
                                                  int64_t out_seg_stride) {
  extern __shared__ double smd[];
  const int dk = (int)ka.dk, dv = (int)ka.dv;
  const int LK = dk + 1;
  const int width = mode == 1 ? dk + dv : dv;
  double* gG = smd;               // [64]
  float* sm = (float*)(smd + 64);
  float* Xs = sm;                 // [dk][CS]
  float* Ws = Xs + dk * CS;       // [64][LK]
  float* Ks = Ws + 64 * LK;       // [64][LK]
  float* Vp = Ks + 64 * LK;       // [64][CS]
  float* V2 = Vp + 64 * CS;       // [64][CS]
  float* kt = V2 + 64 * CS;       // [64]
  const int tid = threadIdx.x;
  const int c0 = blockIdx.x * CS;
  const int64_t h = blockIdx.y;
  const int64_t b = blockIdx.z / nseg;
  const int seg = seg_first + (int)(blockIdx.z % nseg);
  const int64_t hq = h / ka.r, bh = b * ka.H + h;
  const int64_t cs = (int64_t)seg * ka.CPS;
  const int64_t ce = cs + ka.CPS < ka.NC ? cs + ka.CPS : ka.NC;

  for (int e = tid; e < dk * CS; e += NT) {
    const int i = e / CS, col = c0 + e % CS;
    float x = 0.f;
    if (mode == 1) {
      x = (col < dk && col == i) ? 1.f : 0.f;
    } else if (init && col < dv) {
      x = init[seg * init_seg_stride + (bh * dk + i) * dv + col];
    }
    Xs[e] = x;
  }
  __syncthreads();

  for (int64_t c = cs; c < ce; ++c) {
    const int64_t t0 = c * kChunk;
    const float* Wg = ws.W + (bh * ka.Tp + t0) * dk;
    const float* Kg = ws.Kh + ((b * ka.Hqk + hq) * ka.Tp + t0) * dk;
    for (int e = tid; e < 64 * dk; e += NT) {
      const int i = e / dk, col = e % dk;
      Ws[i * LK + col] = Wg[e];
      Ks[i * LK + col] = Kg[e];
    }
    if (tid < 64) gG[tid] = ws.G[bh * ka.Tp + t0 + tid];
    for (int e = tid; e < 64 * CS; e += NT) {
      const int i = e / CS, col = c0 + e % CS;
      float u = 0.f;
      if (mode == 1) {
        if (col >= dk && col < width) u = ws.U[(bh * ka.Tp + t0 + i) * dv + (col - dk)];
      } else if (col < dv) {
        u = ws.U[(bh * ka.Tp + t0 + i) * dv + col];
      }
      Vp[e] = u;
    }
    if (mode == 0 && Hc) {
      float* dst = Hc + (bh * ka.NC + c) * dk * dv;
      for (int e = tid; e < dk * CS; e += NT) {
        const int i = e / CS, col = c0 + e % CS;
        if (col < dv) dst[i * dv + col] = Xs[e];
      }
    }
    __syncthreads();
    // V' = U - W X
    blk_gemm(kChunk, CS, dk, -1.f, Ws, LK, 1, Xs, CS, 1, true, Vp, CS, 1);
    if (tid < 64) kt[tid] = dexp(gG[63], gG[tid]);
    __syncthreads();
    if (mode == 0 && Vn) {
      for (int e = tid; e < 64 * CS; e += NT) {
        const int i = e / CS, col = c0 + e % CS;
        if (col < dv) Vn[(bh * ka.Tp + t0 + i) * dv + col] = Vp[e];
      }
    }
    const float gC = dexp(gG[63], 0.0);
    for (int e = tid; e < 64 * CS; e += NT) V2[e] = kt[e / CS] * Vp[e];
    for (int e = tid; e < dk * CS; e += NT) Xs[e] *= gC;
    __syncthreads();
    // X <- gamma_C X + Kt^T V'
    blk_gemm(dk, CS, kChunk, 1.f, Ks, 1, LK, V2, CS, 1, true, Xs, CS, 1);
    __syncthreads();
  }

  const bool last = seg == ka.P - 1;
  for (int e = tid; e < dk * CS; e += NT) {
    const int i = e / CS, col = c0 + e % CS;
    if (mode == 0) {
      if (final_out && last && col < dv) final_out[(bh * dk + i) * dv + col] = Xs[e];
    } else {
      if (col < dk) {
        if (M_out) M_out[seg * out_seg_stride / dv * dk + (bh * dk + i) * dk + col] = Xs[e];
      } else if (col < width) {
        if (S_out) S_out[seg * out_seg_stride + (bh * dk + i) * dv + (col - dk)] = Xs[e];
      }
    }
  }
}

// -------------------------------------------------------------------- output
// grid (NC, H * ceil(dv / CSO), B): O = diag(gamma) Q S + tril(Q K^T o Gamma) V'.
template <typename TIn>
__global__ void __launch_bounds__(NT) k_output(KArgs ka, WS ws, const int32_t* __restrict__ valid_len,
                                              TIn* __restrict__ o) {
  extern __shared__ double smd[];
  const int dk = (int)ka.dk, dv = (int)ka.dv;
  const int LK = dk + 1;
  const int nsl = (dv + CSO - 1) / CSO;
  double* gG = smd;             // [64]
  float* sm = (float*)(smd + 64);
  float* Qs = sm;               // [64][LK]
  float* Ks = Qs + 64 * LK;     // [64][LK]
  float* Ps = Ks + 64 * LK;     // [64][LS]
  float* Hs = Ps + 64 * LS;     // [dk][CSO]
  float* Vp = Hs + dk * CSO;    // [64][CSO]
  float* Os = Vp + 64 * CSO;    // [64][CSO]
  const int tid = threadIdx.x;
  const int64_t c = blockIdx.x, b = blockIdx.z;
  const int64_t h = blockIdx.y / nsl;
  const int c0 = (int)(blockIdx.y % nsl) * CSO;
  const int64_t hq = h / ka.r, bh = b * ka.H + h;
  const int64_t t0 = c * kChunk;
  const int64_t L = row_len(valid_len, b, ka.T, ws.status, false);

  const float* Qg = ws.Qh + ((b * ka.Hqk + hq) * ka.Tp + t0) * dk;
  const float* Kg = ws.Kh + ((b * ka.Hqk + hq) * ka.Tp + t0) * dk;
  for (int e = tid; e < 64 * dk; e += NT) {
    const int i = e / dk, col = e % dk;
    Qs[i * LK + col] = Qg[e];
    Ks[i * LK + col] = Kg[e];
  }
  if (tid < 64) gG[tid] = ws.G[bh * ka.Tp + t0 + tid];
  const float* Hg = ws.Hc + (bh * ka.NC + c) * dk * dv;
  for (int e = tid; e < dk * CSO; e += NT) {
    const int i = e / CSO, col = c0 + e % CSO;
    Hs[e] = col < dv ? Hg[i * dv + col] : 0.f;
  }
  for (int e = tid; e < 64 * CSO; e += NT) {
    const int i = e / CSO, col = c0 + e % CSO;
    Vp[e] = col < dv ? ws.Vn[(bh * ka.Tp + t0 + i) * dv + col] : 0.f;
  }
  __syncthreads();
  blk_gemm(kChunk, kChunk, dk, 1.f, Qs, LK, 1, Ks, 1, LK, false, Ps, LS, 1);
  blk_gemm(kChunk, CSO, dk, 1.f, Qs, LK, 1, Hs, CSO, 1, false, Os, CSO, 1);
  __syncthreads();
  for (int e = tid; e < 64 * 64; e += NT) {
    const int i = e >> 6, j = e & 63;
    Ps[i * LS + j] = i >= j ? Ps[i * LS + j] * dexp(gG[i], gG[j]) : 0.f;
  }
  for (int e = tid; e < 64 * CSO; e += NT) Os[e] *= dexp(gG[e / CSO], 0.0);
  __syncthreads();
  blk_gemm(kChunk, CSO, kChunk, 1.f, Ps, LS, 1, Vp, CSO, 1, true, Os, CSO, 1);
  __syncthreads();
  for (int e = tid; e < 64 * CSO; e += NT) {
    const int i = e / CSO, col = c0 + e % CSO;
    const int64_t t = t0 + i;
    if (t < ka.T && col < dv) stf(o, ((b * ka.Ts + t) * ka.H + h) * ka.dv + col, t < L ? Os[e] : 0.f);
  }
}

// ------------------------------------------------------ state-gradient scan
// grid (ceil(dv / CS), H, B * nseg), chunks in reverse.  dX is the gradient of
// the state at the end of the current chunk.  dV' = P^T dO + Kt dX,
// dX <- gamma_C dX + (diag(gamma) Q)^T dO - W^T dV'.
template <typename TIn>
__global__ void __launch_bounds__(NT) k_dstate_scan(KArgs ka, WS ws, const int32_t* __restrict__ valid_len,
                                                   const TIn* __restrict__ dO, int mode,
                                                   int seg_first, int nseg,
                                                   const float* __restrict__ init,
                                                   int64_t init_seg_stride, float* start_out,
                                                   float* D_out, int64_t out_seg_stride) {
  extern __shared__ double smd[];
  const int dk = (int)ka.dk, dv = (int)ka.dv;
  const int LK = dk + 1;
  double* gG = smd;              // [64]
  float* sm = (float*)(smd + 64);
  float* dXs = sm;               // [dk][CS]
  float* Qs = dXs + dk * CS;     // [64][LK]
  float* Ks = Qs + 64 * LK;      // [64][LK]
  float* Ws = Ks + 64 * LK;      // [64][LK]
  float* Ps = Ws + 64 * LK;      // [64][LS]
  float* dOs = Ps + 64 * LS;     // [64][CS]
  float* dVp = dOs + 64 * CS;    // [64][CS]
  float* kt = dVp + 64 * CS;     // [64]
  const int tid = threadIdx.x;
  const int c0 = blockIdx.x * CS;
  const int64_t h = blockIdx.y;
  const int64_t b = blockIdx.z / nseg;
  const int seg = seg_first + (int)(blockIdx.z % nseg);
  const int64_t hq = h / ka.r, bh = b * ka.H + h;
  const int64_t cs = (int64_t)seg * ka.CPS;
  const int64_t ce = cs + ka.CPS < ka.NC ? cs + ka.CPS : ka.NC;
  const int64_t L = row_len(valid_len, b, ka.T, ws.status, false);

  for (int e = tid; e < dk * CS; e += NT) {
    const int i = e / CS, col = c0 + e % CS;
    dXs[e] = (mode == 0 && init && col < dv) ? init[seg * init_seg_stride + (bh * dk + i) * dv + col]
                                             : 0.f;
  }
  __syncthreads();

  for (int64_t c = ce - 1; c >= cs; --c) {
    const int64_t t0 = c * kChunk;
    const float* Qg = ws.Qh + ((b * ka.Hqk + hq) * ka.Tp + t0) * dk;
    const float* Kg = ws.Kh + ((b * ka.Hqk + hq) * ka.Tp + t0) * dk;
    const float* Wg = ws.W + (bh * ka.Tp + t0) * dk;
    for (int e = tid; e < 64 * dk; e += NT) {
      const int i = e / dk, col = e % dk;
      Qs[i * LK + col] = Qg[e];
      Ks[i * LK + col] = Kg[e];
      Ws[i * LK + col] = Wg[e];
    }
    if (tid < 64) gG[tid] = ws.G[bh * ka.Tp + t0 + tid];
    for (int e = tid; e < 64 * CS; e += NT) {
      const int i = e / CS, col = c0 + e % CS;
      const int64_t t = t0 + i;
      dOs[e] = (t < L && col < dv) ? ldf(dO, ((b * ka.Ts + t) * ka.H + h) * ka.dv + col) : 0.f;
    }
    if (mode == 0 && ws.dHc) {
      float* dst = ws.dHc + (bh * ka.NC + c) * dk * dv;
      for (int e = tid; e < dk * CS; e += NT) {
        const int i = e / CS, col = c0 + e % CS;
        if (col < dv) dst[i * dv + col] = dXs[e];
      }
    }
    __syncthreads();
    blk_gemm(kChunk, kChunk, dk, 1.f, Qs, LK, 1, Ks, 1, LK, false, Ps, LS, 1);
    // K dX (scaled by kt below)
    blk_gemm(kChunk, CS, dk, 1.f, Ks, LK, 1, dXs, CS, 1, false, dVp, CS, 1);
    if (tid < 64) kt[tid] = dexp(gG[63], gG[tid]);
    __syncthreads();
    for (int e = tid; e < 64 * 64; e += NT) {
      const int i = e >> 6, j = e & 63;
      Ps[i * LS + j] = i >= j ? Ps[i * LS + j] * dexp(gG[i], gG[j]) : 0.f;
    }
    for (int e = tid; e < 64 * CS; e += NT) dVp[e] *= kt[e / CS];
    __syncthreads();
    // dV' += P^T dO
    blk_gemm(kChunk, CS, kChunk, 1.f, Ps, 1, LS, dOs, CS, 1, true, dVp, CS, 1);
    __syncthreads();
    if (mode == 0 && ws.dVn) {
      for (int e = tid; e < 64 * CS; e += NT) {
        const int i = e / CS, col = c0 + e % CS;
        if (col < dv) ws.dVn[(bh * ka.Tp + t0 + i) * dv + col] = dVp[e];
      }
    }
    const float gC = dexp(gG[63], 0.0);
    for (int e = tid; e < dk * CS; e += NT) dXs[e] *= gC;
    for (int e = tid; e < 64 * CS; e += NT) dOs[e] *= dexp(gG[e / CS], 0.0);
    __syncthreads();
    blk_gemm(dk, CS, kChunk, 1.f, Qs, 1, LK, dOs, CS, 1, true, dXs, CS, 1);
    __syncthreads();
    blk_gemm(dk, CS, kChunk, -1.f, Ws, 1, LK, dVp, CS, 1, true, dXs, CS, 1);
    __syncthreads();
  }

  for (int e = tid; e < dk * CS; e += NT) {
    const int i = e / CS, col = c0 + e % CS;
    if (col >= dv) continue;
    if (mode == 1) {
      if (D_out) D_out[seg * out_seg_stride + (bh * dk + i) * dv + col] = dXs[e];
    } else if (start_out && seg == 0) {
      start_out[(bh * dk + i) * dv + col] = dXs[e];
    }
  }
}

// ------------------------------------------------------------------ gradients
// grid (NC, H, B).  All local gradients of one chunk and V head, given the chunk
// start state Hc, the gradient of its end state dHc, V' and dV'.
template <typename TIn>
__global__ void __launch_bounds__(NT) k_grad(KArgs ka, WS ws, const TIn* __restrict__ v,
                                            const TIn* __restrict__ dO,
                                            const int32_t* __restrict__ valid_len,
                                            TIn* __restrict__ dv_out, float* __restrict__ dg_out,
                                            float* __restrict__ dbeta_out) {
  extern __shared__ double smd[];
  const int dk = (int)ka.dk, dv = (int)ka.dv;
  const int LK = dk + 1;
  const int LX = (dk > dv ? dk : dv) + 1;
  double* gG = smd;            // [64] cumulative gate (fp64)
  float* sm = (float*)(smd + 64);
  float* Qs = sm;              // [64][LX]  q_hat, later dKt, later dW
  float* Ks = Qs + 64 * LX;    // [64][LX]  k_hat
  float* X1 = Ks + 64 * LX;    // [64][LX]  dO, later dV'
  float* X2 = X1 + 64 * LX;    // [64][LX]  V', later V
  float* X3 = X2 + 64 * LX;    // [64][LX]  dq_hat, later dk_hat accumulator
  float* Y1 = X3 + 64 * LX;    // [64][LS]  P, later dT, dA, E
  float* Y2 = Y1 + 64 * LS;    // [64][LS]  dP o Gamma, later Tt dT, K K^T
  float* Y3 = Y2 + 64 * LS;    // [64][LS]  T
  float* gB = Y3 + 64 * LS;    // [64]
  float* gam = gB + 64;        // [64]
  float* kt = gam + 64;        // [64]
  float* dG = kt + 64;         // [64]
  float* dbe = dG + 64;        // [64]
  float* red = dbe + 64;       // [NT/32 + 1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t hq = h / ka.r, bh = b * ka.H + h;
  const int64_t t0 = c * kChunk;
  const int64_t L = row_len(valid_len, b, ka.T, ws.status, false);
  const float* Hg = ws.Hc + (bh * ka.NC + c) * dk * dv;
  const float* dHg = ws.dHc + (bh * ka.NC + c) * dk * dv;
  (void)LK;

  // 1. q_hat, k_hat, gates, T
  {
    const float* Qg = ws.Qh + ((b * ka.Hqk + hq) * ka.Tp + t0) * dk;
    const float* Kg = ws.Kh + ((b * ka.Hqk + hq) * ka.Tp + t0) * dk;
    for (int e = tid; e < 64 * dk; e += NT) {
      const int i = e / dk, col = e % dk;
      Qs[i * LX + col] = Qg[e];
      Ks[i * LX + col] = Kg[e];
    }
    const float* Tg = ws.Tm + (bh * ka.NC + c) * (kChunk * kChunk);
    for (int e = tid; e < 64 * 64; e += NT) Y3[(e >> 6) * LS + (e & 63)] = Tg[e];
    if (tid < 64) {
      const double g = ws.G[bh * ka.Tp + t0 + tid];
      gG[tid] = g;
      gB[tid] = ws.Bt[bh * ka.Tp + t0 + tid];
      gam[tid] = dexp(g, 0.0);
      dG[tid] = 0.f;
      dbe[tid] = 0.f;
    }
    // 3. dO (masked) and V'
    for (int e = tid; e < 64 * dv; e += NT) {
      const int i = e / dv, col = e % dv;
      const int64_t t = t0 + i;
      X1[i * LX + col] = t < L ? ldf(dO, ((b * ka.Ts + t) * ka.H + h) * ka.dv + col) : 0.f;
      X2[i * LX + col] = ws.Vn[(bh * ka.Tp + t0 + i) * dv + col];
    }
  }
  __syncthreads();
  if (tid < 64) kt[tid] = dexp(gG[63], gG[tid]);
  // 2. P = Q K^T (masked below); 4. dP = dO V'^T
  blk_gemm(kChunk, kChunk, dk, 1.f, Qs, LX, 1, Ks, 1, LX, false, Y1, LS, 1);
  blk_gemm(kChunk, kChunk, dv, 1.f, X1, LX, 1, X2, 1, LX, false, Y2, LS, 1);
  __syncthreads();
  for (int e = tid; e < 64 * 64; e += NT) {
    const int i = e >> 6, j = e & 63;
    const float gm = i >= j ? dexp(gG[i], gG[j]) : 0.f;
    Y1[i * LS + j] *= gm;   // P
    if (i < j) Y2[i * LS + j] = 0.f;
  }
  __syncthreads();
  // 5. gate terms of P: dG_i += sum_j dP_ij P_ij - sum_j dP_ji P_ji
  if (tid < 64) {
    const int i = tid;
    float acc = 0.f;
    for (int j = 0; j < 64; ++j) acc += Y2[i * LS + j] * Y1[i * LS + j] - Y2[j * LS + i] * Y1[j * LS + i];
    dG[i] += acc;
  }
  __syncthreads();
  for (int e = tid; e < 64 * 64; e += NT) {
    const int i = e >> 6, j = e & 63;
    if (i >= j) Y2[i * LS + j] *= dexp(gG[i], gG[j]);  // dP o Gamma
  }
  // 6. dq_hat = diag(gamma) dO Hc^T + (dP o Gamma) K
  blk_gemm(kChunk, dk, dv, 1.f, X1, LX, 1, Hg, 1, dv, false, X3, LX, 1);
  __syncthreads();
  for (int e = tid; e < 64 * dk; e += NT) X3[(e / dk) * LX + e % dk] *= gam[e / dk];
  __syncthreads();
  // state term of the gate: dG_i += q_i . (gamma_i Hc dO_i)
  for (int i = warp; i < 64; i += NT / 32) {
    float acc = 0.f;
    for (int col = lane; col < dk; col += 32) acc += Qs[i * LX + col] * X3[i * LX + col];
    acc = warp_sum(acc);
    if (lane == 0) dG[i] += acc;
  }
  __syncthreads();
  blk_gemm(kChunk, dk, kChunk, 1.f, Y2, LS, 1, Ks, LX, 1, true, X3, LX, 1);
  __syncthreads();
  for (int e = tid; e < 64 * dk; e += NT) {
    const int i = e / dk, col = e % dk;
    const int64_t t = t0 + i;
    if (t < ka.Tp) ws.dqp[((b * ka.Tp + t) * ka.H + h) * dk + col] = t < L ? X3[i * LX + col] : 0.f;
  }
  __syncthreads();
  // 7. dk_hat accumulator: (dP o Gamma)^T Q
  blk_gemm(kChunk, dk, kChunk, 1.f, Y2, 1, LS, Qs, LX, 1, false, X3, LX, 1);
  // 8. dV'
  for (int e = tid; e < 64 * dv; e += NT) {
    const int i = e / dv, col = e % dv;
    X1[i * LX + col] = ws.dVn[(bh * ka.Tp + t0 + i) * dv + col];
  }
  __syncthreads();
  // 9. dKt = V' dHc^T (into Qs)
  blk_gemm(kChunk, dk, dv, 1.f, X2, LX, 1, dHg, 1, dv, false, Qs, LX, 1);
  __syncthreads();
  {
    // s_j = Kt_j . dKt_j;  dG_j -= s_j;  dG_C += sum_j s_j + gamma_C <Hc, dHc>.
    // The j = C-1 term (weight exp(0) = 1) enters dG_C and dG_{C-1} with opposite
    // signs and cancels exactly; it is left out on both sides, otherwise its
    // rounding residue would be spread by the reverse cumsum over tokens whose
    // gate gradient is O(alpha).
    float tot = 0.f;
    for (int i = warp; i < 63; i += NT / 32) {
      float acc = 0.f;
      for (int col = lane; col < dk; col += 32) acc += Ks[i * LX + col] * Qs[i * LX + col];
      acc = warp_sum(acc) * kt[i];
      if (lane == 0) dG[i] -= acc;
      tot += acc;
    }
    float hs = 0.f;
    for (int e = tid; e < dk * dv; e += NT) hs += Hg[e] * dHg[e];
    hs = warp_sum(hs);
    if (lane == 0) red[warp] = tot + hs * gam[63];
    __syncthreads();
    if (tid == 0) {
      float s = 0.f;
      for (int w = 0; w < NT / 32; ++w) s += red[w];
      dG[63] += s;
    }
  }
  for (int e = tid; e < 64 * dk; e += NT) {
    const int i = e / dk, col = e % dk;
    X3[i * LX + col] += kt[i] * Qs[i * LX + col];
  }
  __syncthreads();
  // 10. dW = -dV' Hc^T (into Qs); 11. V (into X2)
  blk_gemm(kChunk, dk, dv, -1.f, X1, LX, 1, Hg, 1, dv, false, Qs, LX, 1);
  for (int e = tid; e < 64 * dv; e += NT) {
    const int i = e / dv, col = e % dv;
    const int64_t t = t0 + i;
    X2[i * LX + col] = t < ka.T ? ldf(v, ((b * ka.Ts + t) * ka.H + h) * ka.dv + col) : 0.f;
  }
  __syncthreads();
  // 12. dv = diag(beta) T^T dV';  dbeta_i += (T^T dV')_i . v_i
  for (int i = warp; i < 64; i += NT / 32) {
    const int64_t t = t0 + i;
    float part = 0.f;
    for (int col = lane; col < dv; col += 32) {
      float x = 0.f;
      for (int j = i; j < 64; ++j) x = fmaf(Y3[j * LS + i], X1[j * LX + col], x);
      part = fmaf(x, X2[i * LX + col], part);
      if (t < ka.T) stf(dv_out, ((b * ka.Ts + t) * ka.H + h) * ka.dv + col, t < L ? gB[i] * x : 0.f);
    }
    part = warp_sum(part);
    if (lane == 0) dbe[i] += part;
  }
  // 13. dk_hat += diag(beta gamma) T^T dW;  dbeta_i += gamma_i (T^T dW)_i . k_i;
  //     dG_i += beta_i gamma_i (T^T dW)_i . k_i
  for (int i = warp; i < 64; i += NT / 32) {
    float part = 0.f;
    for (int col = lane; col < dk; col += 32) {
      float y = 0.f;
      for (int j = i; j < 64; ++j) y = fmaf(Y3[j * LS + i], Qs[j * LX + col], y);
      part = fmaf(y, Ks[i * LX + col], part);
      X3[i * LX + col] += gB[i] * gam[i] * y;
    }
    part = warp_sum(part);
    if (lane == 0) {
      dbe[i] += gam[i] * part;
      dG[i] += gB[i] * gam[i] * part;
    }
  }
  __syncthreads();
  // 14. dT = dV' (diag(beta) V)^T + dW (diag(beta gamma) K)^T
  blk_gemm(kChunk, kChunk, dv, 1.f, X1, LX, 1, X2, 1, LX, false, Y1, LS, 1);
  blk_gemm(kChunk, kChunk, dk, 1.f, Qs, LX, 1, Ks, 1, LX, false, Y2, LS, 1);
  __syncthreads();
  for (int e = tid; e < 64 * 64; e += NT) {
    const int i = e >> 6, j = e & 63;
    Y1[i * LS + j] = gB[j] * Y1[i * LS + j] + gB[j] * gam[j] * Y2[i * LS + j];
  }
  __syncthreads();
  // 15. dA = -T^T dT T^T, strictly lower
  blk_gemm(kChunk, kChunk, kChunk, 1.f, Y3, 1, LS, Y1, LS, 1, false, Y2, LS, 1);
  __syncthreads();
  blk_gemm(kChunk, kChunk, kChunk, -1.f, Y2, LS, 1, Y3, 1, LS, false, Y1, LS, 1);
  __syncthreads();
  // 16. K K^T (into Y2)
  blk_gemm(kChunk, kChunk, dk, 1.f, Ks, LX, 1, Ks, 1, LX, false, Y2, LS, 1);
  __syncthreads();
  if (tid < 64) {
    const int i = tid;
    float db = 0.f, row = 0.f, col = 0.f;
    for (int j = 0; j < i; ++j) {
      const float kk = Y2[i * LS + j] * dexp(gG[i], gG[j]);   // (k_i.k_j) Gamma_ij
      db += Y1[i * LS + j] * kk;
      row += Y1[i * LS + j] * gB[i] * kk;                        // dA_ij A_ij
    }
    for (int j = i + 1; j < 64; ++j) {
      const float kk = Y2[j * LS + i] * dexp(gG[j], gG[i]);
      col += Y1[j * LS + i] * gB[j] * kk;                        // dA_ji A_ji
    }
    dbe[i] += db;
    dG[i] += row - col;
  }
  __syncthreads();
  for (int e = tid; e < 64 * 64; e += NT) {
    const int i = e >> 6, j = e & 63;
    Y1[i * LS + j] = i > j ? Y1[i * LS + j] * gB[i] * dexp(gG[i], gG[j]) : 0.f;  // E
  }
  __syncthreads();
  // 17. dk_hat += E K + E^T K
  blk_gemm(kChunk, dk, kChunk, 1.f, Y1, LS, 1, Ks, LX, 1, true, X3, LX, 1);
  __syncthreads();
  blk_gemm(kChunk, dk, kChunk, 1.f, Y1, 1, LS, Ks, LX, 1, true, X3, LX, 1);
  __syncthreads();
  // 18. store dk_hat, 19. dg = reverse cumsum of dG, dbeta
  for (int e = tid; e < 64 * dk; e += NT) {
    const int i = e / dk, col = e % dk;
    const int64_t t = t0 + i;
    ws.dkp[((b * ka.Tp + t) * ka.H + h) * dk + col] = t < L ? X3[i * LX + col] : 0.f;
  }
  revsum64(dG);
  __syncthreads();
  if (tid < 64) {
    const int64_t t = t0 + tid;
    if (t < ka.T) {
      const int64_t gi = (b * ka.Ts + t) * ka.H + h;
      dg_out[gi] = t < L ? dG[tid] : 0.f;
      dbeta_out[gi] = t < L ? dbe[tid] : 0.f;
    }
  }
}

// grid (ceil(B*T*Hqk / 8)), one warp per (b, t, hq): sum the per-V-head
// gradients of q_hat and k_hat over the group, then back through norm and scale.
template <typename TIn>
__global__ void __launch_bounds__(NT) k_qk_grad(KArgs ka, WS ws, const TIn* __restrict__ q,
                                               const TIn* __restrict__ k, TIn* __restrict__ dq,
                                               TIn* __restrict__ dk_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (NT / 32) + warp;
  if (row >= ka.B * ka.T * ka.Hqk) return;
  const int64_t hq = row % ka.Hqk, t = (row / ka.Hqk) % ka.T, b = row / (ka.Hqk * ka.T);
  const int dk = (int)ka.dk;
  for (int which = 0; which < 2; ++which) {
    const TIn* x = which == 0 ? q : k;
    const float* part = which == 0 ? ws.dqp : ws.dkp;
    TIn* out = which == 0 ? dq : dk_out;
    const float s = which == 0 ? ka.scale : 1.f;
    const int64_t xo = ((b * ka.Ts + t) * ka.Hqk + hq) * ka.dk;
    float xv[4], gv[4];
    float ss = 0.f, xg = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = lane + 32 * e;
      xv[e] = col < dk ? ldf(x, xo + col) : 0.f;
      float g = 0.f;
      if (col < dk)
        for (int64_t h = hq * ka.r; h < (hq + 1) * ka.r; ++h)
          g += part[((b * ka.Tp + t) * ka.H + h) * dk + col];
      gv[e] = g;
      ss = fmaf(xv[e], xv[e], ss);
      xg = fmaf(xv[e], g, xg);
    }
    ss = warp_sum(ss);
    xg = warp_sum(xg);
    float rn = 1.f, proj = 0.f;
    if (ka.l2norm) {
      rn = rsqrtf(ss + ka.eps);
      proj = xg * rn * rn;  // (u . g) / n with u = x / n
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = lane + 32 * e;
      if (col < dk) stf(out, xo + col, s * (gv[e] - xv[e] * proj) * rn);
    }
  }
}

// ---------------------------------------------------------- compose / prefix
// grid (n, ceil((dk + dv) / CS)): columns of [M | S] = M2 [M1 | S1] + [0 | S2].
__global__ void __launch_bounds__(NT) k_compose(int64_t dk, int64_t dv, const float* __restrict__ M2,
                                               const float* __restrict__ S2,
                                               const float* __restrict__ M1,
                                               const float* __restrict__ S1, float* M, float* S) {
  extern __shared__ float sm[];
  float* Bs = sm;            // [dk][CS]
  float* Cs = Bs + dk * CS;  // [dk][CS]
  const int64_t e0 = blockIdx.x;
  const int c0 = blockIdx.y * CS;
  const int width = (int)(dk + dv);
  for (int e = threadIdx.x; e < dk * CS; e += NT) {
    const int i = e / CS, col = c0 + e % CS;
    float x = 0.f;
    if (col < dk) x = M1[(e0 * dk + i) * dk + col];
    else if (col < width) x = S1[(e0 * dk + i) * dv + (col - dk)];
    Bs[e] = x;
  }
  __syncthreads();
  blk_gemm((int)dk, CS, (int)dk, 1.f, M2 + e0 * dk * dk, dk, 1, Bs, CS, 1, false, Cs, CS, 1);
  __syncthreads();
  for (int e = threadIdx.x; e < dk * CS; e += NT) {
    const int i = e / CS, col = c0 + e % CS;
    if (col < dk) M[(e0 * dk + i) * dk + col] = Cs[e];
    else if (col < width) {
      const int64_t o = (e0 * dk + i) * dv + (col - dk);
      S[o] = Cs[e] + S2[o];
    }
  }
}

// Exclusive prefix over segments, grid (n, ceil(dv / PCS)), 256 threads.
// transpose = 0: X <- M[s] X + S[s] for s = 0, 1, ...; transpose = 1: X <- M[s]^T X + S[s]
// for s = P-1, P-2, ...  Each step multiplies a dk x dk map by the block's dk x PCS
// slice of X in fp32: the map is staged in shared memory (padded rows, conflict-free
// in both orientations; two buffers, the next map prefetched into registers while
// the current one is used) and every thread accumulates a 4 x 4 register tile.
constexpr int PCS = 32;          // state columns per prefix block
constexpr int PLD = 129;         // shared-memory row stride of a map
constexpr int PMAXR = kMaxHeadDim / (NT / 32);        // map rows per warp (16)
constexpr int PMAXC = kMaxHeadDim / 32;               // map columns per lane (4)
__device__ __forceinline__ void prefix_block(int64_t n, int64_t P, int64_t dk, int64_t dv,
                                             const float* __restrict__ M,
                                             const float* __restrict__ S,
                                             const float* __restrict__ x0, float* out_seq,
                                             float* out_last, int transpose) {
  extern __shared__ float sm[];
  float* Ms0 = sm;                               // [2][dk][PLD]
  float* Xs = sm + 2 * kMaxHeadDim * PLD;        // [dk][PCS]
  const int64_t e0 = blockIdx.x;
  const int c0 = blockIdx.y * PCS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ndk = (int)dk;
  const int rg = tid >> 3, cg = tid & 7;         // rows 4 rg .. +3, columns c0 + 4 cg .. +3
  float x[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = rg * 4 + r, col = c0 + cg * 4 + c;
      x[r][c] = (x0 && i < ndk && col < dv) ? x0[(e0 * dk + i) * dv + col] : 0.f;
    }
  float pre[PMAXR][PMAXC];  // map prefetch: rows warp + 8 a, columns lane + 32 b
  auto prefetch = [&](int64_t s) {
    const float* Mg = M + (s * n + e0) * dk * dk;
#pragma unroll
    for (int a = 0; a < PMAXR; ++a)
#pragma unroll
      for (int bb = 0; bb < PMAXC; ++bb) {
        const int r = warp + 8 * a, l = lane + 32 * bb;
        pre[a][bb] = (r < ndk && l < ndk) ? Mg[(int64_t)r * ndk + l] : 0.f;
      }
  };
  const int64_t s_first = transpose ? P - 1 : 0;
  prefetch(s_first);
  for (int64_t step = 0; step < P; ++step) {
    const int64_t s = transpose ? P - 1 - step : step;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = rg * 4 + r, col = c0 + cg * 4 + c;
        if (i < ndk && col < dv) out_seq[((s * n + e0) * dk + i) * dv + col] = x[r][c];
      }
    const bool apply = transpose ? (s > 0 || out_last) : (s < P - 1 || out_last);
    if (!apply) break;
    float* Ms = Ms0 + (step & 1) * kMaxHeadDim * PLD;
#pragma unroll
    for (int a = 0; a < PMAXR; ++a)
#pragma unroll
      for (int bb = 0; bb < PMAXC; ++bb) Ms[(warp + 8 * a) * PLD + lane + 32 * bb] = pre[a][bb];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) Xs[(rg * 4 + r) * PCS + cg * 4 + c] = x[r][c];
    __syncthreads();
    const int64_t s_next = transpose ? s - 1 : s + 1;
    if (step + 1 < P) prefetch(s_next);
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = rg * 4 + r, col = c0 + cg * 4 + c;
        acc[r][c] = (i < ndk && col < dv) ? S[((s * n + e0) * dk + i) * dv + col] : 0.f;
      }
    const int sa_i = transpose ? 1 : PLD, sa_l = transpose ? PLD : 1;
    for (int l = 0; l < ndk; ++l) {
      const float4 xv = *reinterpret_cast<const float4*>(Xs + l * PCS + cg * 4);
      float av[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) av[r] = Ms[(rg * 4 + r) * sa_i + l * sa_l];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        acc[r][0] = fmaf(av[r], xv.x, acc[r][0]);
        acc[r][1] = fmaf(av[r], xv.y, acc[r][1]);
        acc[r][2] = fmaf(av[r], xv.z, acc[r][2]);
        acc[r][3] = fmaf(av[r], xv.w, acc[r][3]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) x[r][c] = acc[r][c];
    __syncthreads();  // Xs is rewritten at the next step
  }
  if (out_last) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = rg * 4 + r, col = c0 + cg * 4 + c;
        if (i < ndk && col < dv) out_last[(e0 * dk + i) * dv + col] = x[r][c];
      }
  }
}

__global__ void __launch_bounds__(NT, 1) k_prefix(int64_t n, int64_t P, int64_t dk, int64_t dv,
                                                 const float* __restrict__ M,
                                                 const float* __restrict__ S,
                                                 const float* __restrict__ x0, float* out_seq,
                                                 float* out_last, int transpose) {
  prefix_block(n, P, dk, dv, M, S, x0, out_seq, out_last, transpose);
}

// The forward prefix (blockIdx.z = 0: H_in from M, S, h0) and the reverse prefix
// (blockIdx.z = 1: dH_out from M^T, D, dHT) of the backward in one launch.
__global__ void __launch_bounds__(NT, 1) k_prefix_pair(int64_t n, int64_t P, int64_t dk,
                                                      int64_t dv, const float* __restrict__ M,
                                                      const float* __restrict__ S,
                                                      const float* __restrict__ h0, float* Hin,
                                                      const float* __restrict__ D,
                                                      const float* __restrict__ dHT,
                                                      float* dHout) {
  if (blockIdx.z == 0)
    prefix_block(n, P, dk, dv, M, S, h0, Hin, nullptr, 0);
  else
    prefix_block(n, P, dk, dv, M, D, dHT, dHout, nullptr, 1);
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

// ============================================================== launchers

cudaError_t launch_prep(const Prob& pr, const Inputs& in, const WS& ws, bool need_q, bool need_T,
                        cudaStream_t st) {
  if (pr.B == 0 || pr.NC == 0) return cudaSuccess;
  const int LK = (int)pr.dk + 1, LV = (int)pr.dv + 1;
  const size_t smem = 64 * sizeof(double) + sizeof(float) * (size_t)(64 * LK + 64 * LV + 3 * 64 * LS + 64);
  dim3 grid((unsigned)pr.NC, (unsigned)pr.Hqk, (unsigned)pr.B);
  const KArgs ka = kargs(pr);
  cudaError_t e;
  if (pr.dtype == GDN_BF16) {
    auto kern = k_prep<__nv_bfloat16>;
    if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
    kern<<<grid, NT, smem, st>>>(ka, (const __nv_bfloat16*)in.q, (const __nv_bfloat16*)in.k,
                                 (const __nv_bfloat16*)in.v, (const __nv_bfloat16*)in.a,
                                 (const __nv_bfloat16*)in.b, in.A_log, in.dt_bias, in.valid_len,
                                 ws, need_q ? 1 : 0, need_T ? 1 : 0);
  } else {
    auto kern = k_prep<float>;
    if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
    kern<<<grid, NT, smem, st>>>(ka, (const float*)in.q, (const float*)in.k, (const float*)in.v,
                                 (const float*)in.a, (const float*)in.b, in.A_log, in.dt_bias,
                                 in.valid_len, ws, need_q ? 1 : 0, need_T ? 1 : 0);
  }
  return cudaGetLastError();
}

cudaError_t launch_state_scan(const Prob& pr, const WS& ws, int mode, int seg_first, int nseg,
                              const float* init, int64_t init_seg_stride, float* Hc, float* Vn,
                              float* final_out, float* M_out, float* S_out,
                              int64_t out_seg_stride, cudaStream_t st) {
  if (pr.B == 0 || nseg <= 0) return cudaSuccess;
  const int width = mode == 1 ? (int)(pr.dk + pr.dv) : (int)pr.dv;
  const int LK = (int)pr.dk + 1;
  const size_t smem = 64 * sizeof(double) + sizeof(float) * (size_t)(pr.dk * CS + 2 * 64 * LK + 2 * 64 * CS + 64);
  dim3 grid((unsigned)((width + CS - 1) / CS), (unsigned)pr.H, (unsigned)(pr.B * nseg));
  cudaError_t e;
  if ((e = set_smem(k_state_scan, smem)) != cudaSuccess) return e;
  k_state_scan<<<grid, NT, smem, st>>>(kargs(pr), ws, mode, seg_first, nseg, init,
                                       init_seg_stride, Hc, Vn, final_out, M_out, S_out,
                                       out_seg_stride);
  return cudaGetLastError();
}

cudaError_t launch_output(const Prob& pr, const Inputs& in, const WS& ws, void* o,
                          cudaStream_t st) {
  if (pr.B == 0 || pr.NC == 0) return cudaSuccess;
  const int LK = (int)pr.dk + 1;
  const int nsl = (int)((pr.dv + CSO - 1) / CSO);
  const size_t smem =
      64 * sizeof(double) + sizeof(float) * (size_t)(2 * 64 * LK + 64 * LS + pr.dk * CSO + 2 * 64 * CSO);
  dim3 grid((unsigned)pr.NC, (unsigned)(pr.H * nsl), (unsigned)pr.B);
  cudaError_t e;
  if (pr.dtype == GDN_BF16) {
    auto kern = k_output<__nv_bfloat16>;
    if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
    kern<<<grid, NT, smem, st>>>(kargs(pr), ws, in.valid_len, (__nv_bfloat16*)o);
  } else {
    auto kern = k_output<float>;
    if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
    kern<<<grid, NT, smem, st>>>(kargs(pr), ws, in.valid_len, (float*)o);
  }
  return cudaGetLastError();
}

cudaError_t launch_dstate_scan(const Prob& pr, const Inputs& in, const WS& ws, int mode,
                               int seg_first, int nseg, const float* init,
                               int64_t init_seg_stride, float* start_out, float* D_out,
                               int64_t out_seg_stride, cudaStream_t st) {
  if (pr.B == 0 || nseg <= 0) return cudaSuccess;
  const int LK = (int)pr.dk + 1;
  const size_t smem =
      64 * sizeof(double) + sizeof(float) * (size_t)(pr.dk * CS + 3 * 64 * LK + 64 * LS + 2 * 64 * CS + 64);
  dim3 grid((unsigned)((pr.dv + CS - 1) / CS), (unsigned)pr.H, (unsigned)(pr.B * nseg));
  cudaError_t e;
  if (pr.dtype == GDN_BF16) {
    auto kern = k_dstate_scan<__nv_bfloat16>;
    if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
    kern<<<grid, NT, smem, st>>>(kargs(pr), ws, in.valid_len, (const __nv_bfloat16*)in.dO, mode,
                                 seg_first, nseg, init, init_seg_stride, start_out, D_out,
                                 out_seg_stride);
  } else {
    auto kern = k_dstate_scan<float>;
    if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
    kern<<<grid, NT, smem, st>>>(kargs(pr), ws, in.valid_len, (const float*)in.dO, mode,
                                 seg_first, nseg, init, init_seg_stride, start_out, D_out,
                                 out_seg_stride);
  }
  return cudaGetLastError();
}

cudaError_t launch_grad(const Prob& pr, const Inputs& in, const WS& ws, void* dv, float* dg,
                        float* dbeta, cudaStream_t st) {
  if (pr.B == 0 || pr.NC == 0) return cudaSuccess;
  const int LX = (int)(pr.dk > pr.dv ? pr.dk : pr.dv) + 1;
  const size_t smem = 64 * sizeof(double) +
                      sizeof(float) * (size_t)(5 * 64 * LX + 3 * 64 * LS + 5 * 64 + NT / 32 + 8);
  dim3 grid((unsigned)pr.NC, (unsigned)pr.H, (unsigned)pr.B);
  cudaError_t e;
  if (pr.dtype == GDN_BF16) {
    auto kern = k_grad<__nv_bfloat16>;
    if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
    kern<<<grid, NT, smem, st>>>(kargs(pr), ws, (const __nv_bfloat16*)in.v,
                                 (const __nv_bfloat16*)in.dO, in.valid_len, (__nv_bfloat16*)dv, dg,
                                 dbeta);
  } else {
    auto kern = k_grad<float>;
    if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
    kern<<<grid, NT, smem, st>>>(kargs(pr), ws, (const float*)in.v, (const float*)in.dO,
                                 in.valid_len, (float*)dv, dg, dbeta);
  }
  return cudaGetLastError();
}

cudaError_t launch_qk_grad(const Prob& pr, const Inputs& in, const WS& ws, void* dq, void* dk,
                           cudaStream_t st) {
  const int64_t rows = pr.B * pr.T * pr.Hqk;
  if (rows == 0) return cudaSuccess;
  dim3 grid((unsigned)((rows + NT / 32 - 1) / (NT / 32)));
  if (pr.dtype == GDN_BF16)
    k_qk_grad<__nv_bfloat16><<<grid, NT, 0, st>>>(kargs(pr), ws, (const __nv_bfloat16*)in.q,
                                                  (const __nv_bfloat16*)in.k, (__nv_bfloat16*)dq,
                                                  (__nv_bfloat16*)dk);
  else
    k_qk_grad<float><<<grid, NT, 0, st>>>(kargs(pr), ws, (const float*)in.q, (const float*)in.k,
                                          (float*)dq, (float*)dk);
  return cudaGetLastError();
}

cudaError_t launch_compose(int64_t n, int64_t dk, int64_t dv, const float* M2, const float* S2,
                           const float* M1, const float* S1, float* M, float* S,
                           cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * (size_t)(2 * dk * CS);
  dim3 grid((unsigned)n, (unsigned)((dk + dv + CS - 1) / CS));
  cudaError_t e;
  if ((e = set_smem(k_compose, smem)) != cudaSuccess) return e;
  k_compose<<<grid, NT, smem, st>>>(dk, dv, M2, S2, M1, S1, M, S);
  return cudaGetLastError();
}

cudaError_t launch_prefix(int64_t n, int64_t P, int64_t dk, int64_t dv, const float* M,
                          const float* S, const float* h0, float* Hin, float* Hout,
                          cudaStream_t st) {
  if (n == 0 || P == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * (size_t)(2 * kMaxHeadDim * PLD + kMaxHeadDim * PCS);
  dim3 grid((unsigned)n, (unsigned)((dv + PCS - 1) / PCS));
  cudaError_t e;
  if ((e = set_smem(k_prefix, smem)) != cudaSuccess) return e;
  k_prefix<<<grid, NT, smem, st>>>(n, P, dk, dv, M, S, h0, Hin, Hout, 0);
  return cudaGetLastError();
}

cudaError_t launch_prefix_bwd(int64_t n, int64_t P, int64_t dk, int64_t dv, const float* M,
                              const float* D, const float* dHT, float* dHout, float* dH0,
                              cudaStream_t st) {
  if (n == 0 || P == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * (size_t)(2 * kMaxHeadDim * PLD + kMaxHeadDim * PCS);
  dim3 grid((unsigned)n, (unsigned)((dv + PCS - 1) / PCS));
  cudaError_t e;
  if ((e = set_smem(k_prefix, smem)) != cudaSuccess) return e;
  k_prefix<<<grid, NT, smem, st>>>(n, P, dk, dv, M, D, dHT, dHout, dH0, 1);
  return cudaGetLastError();
}

cudaError_t launch_prefix_pair(int64_t n, int64_t P, int64_t dk, int64_t dv, const float* M,
                               const float* S, const float* h0, float* Hin, const float* D,
                               const float* dHT, float* dHout, cudaStream_t st) {
  if (n == 0 || P == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * (size_t)(2 * kMaxHeadDim * PLD + kMaxHeadDim * PCS);
  dim3 grid((unsigned)n, (unsigned)((dv + PCS - 1) / PCS), 2);
  cudaError_t e;
  if ((e = set_smem(k_prefix_pair, smem)) != cudaSuccess) return e;
  k_prefix_pair<<<grid, NT, smem, st>>>(n, P, dk, dv, M, S, h0, Hin, D, dHT, dHout);
  return cudaGetLastError();
}

}  // namespace gdn
