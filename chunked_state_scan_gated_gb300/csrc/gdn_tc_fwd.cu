// gdn_tc_fwd.cu -- tensor-core (tcgen05) chunk scan of the bf16 forward.
//
// One CTA runs the chunked gated delta rule over the chunks of one segment of
// one (batch row, V head), dk = dv = 128, C = 64, keeping the state S in fp32
// registers and every chunk intermediate on chip (nothing but the inputs, the
// output and the state crosses HBM).  Per chunk (notation of gdn_simt.cu):
//
//   TMA      Q, K, V tiles (128-byte swizzle) -> shared memory
//   SIMT     gates, cumulative gate G, row norms (q, k scaled in place)
//   MMA1     [Q;K] K^T                   -> P = tril(QK^T o Gamma), A
//   SIMT     T = (I + A)^-1 (blocked fp32 solve), T_u = T diag(beta),
//            T_w = T diag(beta gamma)
//   MMA2     [T_u;T_w] K, [T_u;T_w] V    -> W (rows 64..127), U (rows 0..63)
//   MMA3     [W;Q] S                     -> W S (rows 0..63), Q S (rows 64..127)
//   SIMT     V' = U - W S, V2 = diag(exp(G_C - G)) V', O0 = diag(gamma) Q S
//   MMA4     K^T V2                      -> S <- gamma_C S + K^T V2
//   MMA5     [0;P] V'                    -> O = O0 + P V'
//
// All MMAs are M = 128 (bf16 x bf16 -> fp32 accumulators in TMEM).  The same
// kernel produces segment summaries (the "p2p" map H_out = M H_in + S of
// "linear attention cp #1035"): the S part runs the scan from zero without
// output, the M part runs it on the columns of M from the identity with U = 0.
// The chunk size and head dim are the fused backend's shape of the
// "Linear Attention CP 融合算子 PR #1114 测试报告", section 3.1.
#include <cuda.h>
#include <cuda_bf16.h>
#include <mutex>

#include "gdn_internal.h"
#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int FT = 256;  // threads per CTA (8 warps; warps w and w+4 share a TMEM lane quadrant)

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr uint32_t ATOM = 24576;            // one 64-column atom of [W | Q | K], 3 x 8 KB
constexpr uint32_t OFF_W = 0, OFF_Q = 8192, OFF_K = 16384;
constexpr uint32_t OFF_V = 49152, LBO_V = 8192;      // V tile, two 8 KB atoms
constexpr uint32_t OFF_TA = 65536;                   // [T_u; T_w] 128 x 64
constexpr uint32_t OFF_PZ = 81920;                   // [0; P]    128 x 64
constexpr uint32_t OFF_S = 98304, LBO_S = 16384;     // S bf16 (MN-major, 128 x 128)
constexpr uint32_t OFF_VP = 131072, OFF_V2 = 147456, LBO_VP = 8192;  // V', V2 (64 x 128)
constexpr uint32_t OFF_A = 131072;                   // fp32 A (aliases V', V2: used earlier)
constexpr uint32_t OFF_T = OFF_A + 64 * LDA * 4;
constexpr uint32_t OFF_Y = OFF_T + 64 * LDA * 4;     // 3 x 256 fp32
constexpr uint32_t OFF_QKW1 = 172032;                // second [W | Q | K] buffer (prefetch)
constexpr uint32_t OFF_SC = OFF_QKW1 + 2 * ATOM;     // scalars, barriers
constexpr uint32_t SMEM_BYTES = OFF_SC + 2048 + 1024;

enum { MODE_APPLY = 0, MODE_SUM = 1, MODE_STATES = 2 };

struct TcArgs {
  int64_t T, Ts, H, r, NC, CPS;
  int P, l2norm;
  float eps, scale;
  const __nv_bfloat16* a;
  const __nv_bfloat16* b;
  const float* A_log;
  const float* dt_bias;
  const int32_t* valid_len;
  const float* init;
  int64_t init_seg_stride;
  __nv_bfloat16* o;
  float* final_out;
  float* M_out;
  float* S_out;
  int64_t out_seg_stride;
  __nv_bfloat16* hc;  // MODE_STATES: chunk-start states [B][H][NC][128][128]
  int* status;
  int mode, seg_first, nseg;
};

#define PHASE_SYNC()            \
  do {                          \
    fence_proxy_async();        \
    tc_fence_before();          \
    __syncthreads();            \
    tc_fence_after();           \
    if (*s_abort) goto done;    \
  } while (0)

__global__ void __launch_bounds__(FT, 1)
    k_chunk_scan_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, TcArgs ar) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t base = smem_u32(sm);
  float* sG = (float*)(sm + OFF_SC);             // [64] cumulative gate, log2 units
  float* sGam = (float*)(sm + OFF_SC + 512);     // [64]
  float* sBeta = sGam + 64;                      // [64]
  float* sKt = sBeta + 64;                       // [64]
  uint64_t* bar_qk = (uint64_t*)(sm + OFF_SC + 1536);  // [2]: Q/K tiles of buffers 0, 1
  uint64_t* bar_v = bar_qk + 2;
  uint64_t* bar_mma = bar_qk + 3;
  uint32_t* s_tmem = (uint32_t*)(bar_qk + 4);
  int* s_abort = (int*)(s_tmem + 1);
  float* sA = (float*)(sm + OFF_A);
  float* sT = (float*)(sm + OFF_T);
  float* sY = (float*)(sm + OFF_Y);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int row = quad * 32 + lane;  // accumulator row / TMEM lane of this thread
  const bool apply = ar.mode == MODE_APPLY;            // reads q, writes o
  const bool states = ar.mode == MODE_STATES;          // writes every chunk-start state
  const bool mpart = ar.mode == MODE_SUM && blockIdx.x == 1;
  const int64_t h = blockIdx.y;
  const int64_t b = blockIdx.z / ar.nseg;
  const int seg = ar.seg_first + (int)(blockIdx.z % ar.nseg);
  const int64_t hq = h / ar.r, bh = b * ar.H + h;
  const int64_t cs = (int64_t)seg * ar.CPS;
  const int64_t ce = cs + ar.CPS < ar.NC ? cs + ar.CPS : ar.NC;
  int64_t L = ar.T;
  if (ar.valid_len) {
    L = ar.valid_len[b];
    if (L < 0 || L > ar.T) {
      if (tid == 0 && ar.status) atomicOr(ar.status, kStatusClamped);
      L = L < 0 ? 0 : ar.T;
    }
  }

  if (tid == 0) {
    mbar_init(bar_qk, 1);
    mbar_init(bar_qk + 1, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
    *s_abort = 0;
  }
  if (warp == 0) tmem_alloc(s_tmem, 512);
  // zero the first 64 rows of [0; P] and, without Q, the Q tiles
  for (int e = tid; e < 512; e += FT) {
    reinterpret_cast<uint4*>(sm + OFF_PZ)[e] = make_uint4(0, 0, 0, 0);
    if (!apply) {
      for (int bufi = 0; bufi < 2; ++bufi) {
        const uint32_t qb = bufi ? OFF_QKW1 : 0u;
        reinterpret_cast<uint4*>(sm + qb + OFF_Q)[e] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(sm + qb + ATOM + OFF_Q)[e] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tX = tmem, tD3 = tmem + 256;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;

  float S[64];   // state row `row`, columns half*64 .. half*64+63
  float U[64];   // U (rows 0..63) or gamma Q S (rows 64..127)
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    const int col = half * 64 + j;
    float x = 0.f;
    if (apply || states) {
      if (ar.init) x = ar.init[seg * ar.init_seg_stride + (bh * 128 + row) * 128 + col];
    } else if (mpart) {
      x = (row == col) ? 1.f : 0.f;
    }
    S[j] = x;
  }
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) st_chunk(sm + OFF_S, mnmaj_chunk(row, half * 8 + cc, LBO_S), &S[cc * 8]);

  {
    uint32_t ph_mma = 0;
    const uint32_t id_qk = idesc_bf16(128, 64, 0, 0);
    const uint32_t id_kn = idesc_bf16(128, 128, 0, 1);
    const uint32_t id_mn = idesc_bf16(128, 128, 1, 1);
    const uint32_t qk_bytes = (apply ? 16384u : 0u) + 16384u;
    // loads of chunk c into Q/K buffer (c - cs) & 1 and the V tile
    auto issue_qk = [&](int64_t c) {
      const uint32_t qb = ((c - cs) & 1) ? OFF_QKW1 : 0u;
      uint64_t* bar = bar_qk + ((c - cs) & 1);
      mbar_arrive_expect_tx(bar, qk_bytes);
      for (int at = 0; at < 2; ++at) {
        if (apply) tma_load_4d(sm + qb + at * ATOM + OFF_Q, &mq, at * 64, (int)hq, (int)(c * 64), (int)b, bar);
        tma_load_4d(sm + qb + at * ATOM + OFF_K, &mk, at * 64, (int)hq, (int)(c * 64), (int)b, bar);
      }
    };
    auto issue_v = [&](int64_t c) {
      mbar_arrive_expect_tx(bar_v, 16384u);
      for (int at = 0; at < 2; ++at)
        tma_load_4d(sm + OFF_V + at * LBO_V, &mv, at * 64, (int)h, (int)(c * 64), (int)b, bar_v);
    };
    // gate inputs of chunk c (registers of threads 0..63)
    float a_next = 0.f, b_next = 0.f;
    auto load_gates = [&](int64_t c) {
      const int64_t t = c * 64 + tid;
      if (tid < 64 && t < L) {
        const int64_t gi = (b * ar.Ts + t) * ar.H + h;
        a_next = __bfloat162float(ar.a[gi]);
        b_next = __bfloat162float(ar.b[gi]);
      }
    };
    if (cs < ce) {
      if (tid == 0) {
        issue_qk(cs);
        if (!mpart) issue_v(cs);
      }
      load_gates(cs);
    }
    for (int64_t c = cs; c < ce; ++c) {
      const int64_t t0 = c * 64;
      const int64_t kloc = c - cs;
      const uint32_t qkw = (kloc & 1) ? OFF_QKW1 : 0u;
      // ---- prefetch chunk c+1 (its Q/K buffer was last used by chunk c-1) and gates
      fence_proxy_async();
      __syncthreads();
      if (tid == 0 && c + 1 < ce) issue_qk(c + 1);
      if (tid < 64) {
        const int64_t t = t0 + tid;
        float g = 0.f, be = 0.f;
        if (t < L) {
          const float x = a_next + ar.dt_bias[h];
          const float sp = x > 20.f ? x : log1pf(expf(x));
          g = -expf(ar.A_log[h]) * sp;
          be = 1.f / (1.f + expf(-b_next));
        }
        sG[tid] = g * kLog2e;
        sBeta[tid] = be;
      }
      if (c + 1 < ce) load_gates(c + 1);
      __syncthreads();
      cumsum64f(sG);
      __syncthreads();
      if (tid < 64) {
        sGam[tid] = exp2f(sG[tid]);
        sKt[tid] = dexp_(sG[63], sG[tid]);
      }
      if (!mbar_wait(bar_qk + (kloc & 1), (uint32_t)((kloc >> 1) & 1), ar.status, kStatusTimeout))
        *s_abort = 1;
      if (!mpart && !mbar_wait(bar_v, (uint32_t)(kloc & 1), ar.status, kStatusTimeout)) *s_abort = 1;
      if (states) {  // chunk-start state, bf16 row-major [dk][dv]
        uint4* dst = reinterpret_cast<uint4*>(ar.hc + ((bh * ar.NC + c) * 128 + row) * 128 + half * 64);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint4 pk;
          pk.x = pack_bf16(S[cc * 8 + 0], S[cc * 8 + 1]);
          pk.y = pack_bf16(S[cc * 8 + 2], S[cc * 8 + 3]);
          pk.z = pack_bf16(S[cc * 8 + 4], S[cc * 8 + 5]);
          pk.w = pack_bf16(S[cc * 8 + 6], S[cc * 8 + 7]);
          dst[cc] = pk;
        }
      }
      // ---- row norms (16 threads per row), q scaled by scale/|q|, k by 1/|k|
      for (int it = 0; it < 8; ++it) {
        const int rr = (tid >> 4) + 16 * it;
        const bool isk = rr >= 64;
        if (!isk && !apply) continue;  // uniform per warp (row pairs never straddle 64)
        const int sub = tid & 15, at = sub >> 3, ch = sub & 7, r6 = rr & 63;
        const uint32_t off = qkw + at * ATOM + (isk ? OFF_K : OFF_Q) + kmaj_chunk(r6, ch);
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
      PHASE_SYNC();
      // ---- MMA1: [Q;K] K^T
      if (tid == 0) {
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t at = ks >> 2, kk = ks & 3;
          mma_bf16(tX, sdesc(base + qkw + at * ATOM + OFF_Q + kk * 32, 16, 1024),
                   sdesc(base + qkw + at * ATOM + OFF_K + kk * 32, 16, 1024), id_qk, ks > 0);
        }
        mma_commit(bar_mma);
      }
      if (!mbar_wait(bar_mma, ph_mma, ar.status, kStatusTimeout)) *s_abort = 1;
      ph_mma ^= 1;
      tc_fence_after();
      {
        float v[32];
        tmem_ld32(tX + lane_off + half * 32, v);
        if (row < 64) {
          if (apply) {
            const int i = row;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              float p[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int j = half * 32 + cc * 8 + e;
                p[e] = (j <= i) ? v[cc * 8 + e] * dexp_(sG[i], sG[j]) : 0.f;
              }
              st_chunk(sm + OFF_PZ, kmaj_chunk(64 + i, half * 4 + cc), p);
            }
          }
        } else {
          const int i = row - 64;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = half * 32 + e;
            sA[i * LDA + j] = (j < i) ? sBeta[i] * v[e] * dexp_(sG[i], sG[j]) : 0.f;
          }
        }
      }
      PHASE_SYNC();
      // ---- T = (I + A)^-1; stage [T_u; T_w]
      solve_unit_lower64(sA, sT, sY);
      for (int q = 0; q < 4; ++q) {
        const int idx = tid + FT * q;
        const int rr = idx >> 3, cc = idx & 7, i = rr & 63;
        const bool w = rr >= 64;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = cc * 8 + e;
          x[e] = (j <= i) ? sT[i * LDA + j] * sBeta[j] * (w ? sGam[j] : 1.f) : 0.f;
        }
        st_chunk(sm + OFF_TA, kmaj_chunk(rr, cc), x);
      }
      PHASE_SYNC();
      // ---- MMA2: W = T_w K, U = T_u V
      if (tid == 0) {
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = sdesc(base + OFF_TA + ks * 32, 16, 1024);
          mma_bf16(tX, ad, sdesc(base + qkw + OFF_K + ks * 2048, ATOM, 1024), id_kn, ks > 0);
          if (!mpart) mma_bf16(tX + 128, ad, sdesc(base + OFF_V + ks * 2048, LBO_V, 1024), id_kn, ks > 0);
        }
        mma_commit(bar_mma);
      }
      if (!mbar_wait(bar_mma, ph_mma, ar.status, kStatusTimeout)) *s_abort = 1;
      ph_mma ^= 1;
      tc_fence_after();
      if (tid == 0 && !mpart && c + 1 < ce) issue_v(c + 1);  // V(c) consumed by MMA2
      if (quad >= 2) {
        const int i = row - 64;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[32];
          tmem_ld32(tX + lane_off + half * 64 + hh * 32, v);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            st_chunk(sm + qkw + half * ATOM + OFF_W, kmaj_chunk(i, hh * 4 + cc), &v[cc * 8]);
        }
      } else {
        if (!mpart) {
          float v[32];
          tmem_ld32(tX + lane_off + 128 + half * 64, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) U[j] = v[j];
          tmem_ld32(tX + lane_off + 128 + half * 64 + 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) U[32 + j] = v[j];
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) U[j] = 0.f;
        }
      }
      PHASE_SYNC();
      // ---- MMA3: [W; Q] S
      if (tid == 0) {
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t at = ks >> 2, kk = ks & 3;
          mma_bf16(tD3, sdesc(base + qkw + at * ATOM + OFF_W + kk * 32, 16, 1024),
                   sdesc(base + OFF_S + ks * 2048, LBO_S, 1024), id_kn, ks > 0);
        }
        mma_commit(bar_mma);
      }
      if (!mbar_wait(bar_mma, ph_mma, ar.status, kStatusTimeout)) *s_abort = 1;
      ph_mma ^= 1;
      tc_fence_after();
      if (quad < 2) {
        const int i = row;
        const float kt = sKt[i];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[32];
          tmem_ld32(tD3 + lane_off + half * 64 + hh * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = U[hh * 32 + e] - v[e];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int chn = half * 8 + hh * 4 + cc;
            st_chunk(sm + OFF_VP, mnmaj_chunk(i, chn, LBO_VP), &v[cc * 8]);
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = v[cc * 8 + e] * kt;
            st_chunk(sm + OFF_V2, mnmaj_chunk(i, chn, LBO_VP), x);
          }
        }
      } else if (apply) {
        const float gm = sGam[row - 64];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[32];
          tmem_ld32(tD3 + lane_off + half * 64 + hh * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) U[hh * 32 + e] = gm * v[e];
        }
      }
      PHASE_SYNC();
      // ---- MMA4: K^T V2 (state update); MMA5: [0; P] V' (output)
      if (tid == 0) {
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tX, sdesc(base + qkw + OFF_K + ks * 2048, ATOM, 1024),
                   sdesc(base + OFF_V2 + ks * 2048, LBO_VP, 1024), id_mn, ks > 0);
        if (apply)
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tD3, sdesc(base + OFF_PZ + ks * 32, 16, 1024),
                     sdesc(base + OFF_VP + ks * 2048, LBO_VP, 1024), id_kn, ks > 0);
        mma_commit(bar_mma);
      }
      if (!mbar_wait(bar_mma, ph_mma, ar.status, kStatusTimeout)) *s_abort = 1;
      ph_mma ^= 1;
      tc_fence_after();
      {
        const float gC = sGam[63];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[32];
          tmem_ld32(tX + lane_off + half * 64 + hh * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) S[hh * 32 + e] = fmaf(gC, S[hh * 32 + e], v[e]);
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          st_chunk(sm + OFF_S, mnmaj_chunk(row, half * 8 + cc, LBO_S), &S[cc * 8]);
        if (apply && quad >= 2) {
          const int i = row - 64;
          const int64_t t = t0 + i;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float v[32];
            tmem_ld32(tD3 + lane_off + half * 64 + hh * 32, v);
            if (t < ar.T) {
              uint4* dst = reinterpret_cast<uint4*>(ar.o + ((b * ar.Ts + t) * ar.H + h) * 128 + half * 64 + hh * 32);
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = t < L ? U[hh * 32 + cc * 8 + e] + v[cc * 8 + e] : 0.f;
                uint4 pk;
                pk.x = pack_bf16(x[0], x[1]);
                pk.y = pack_bf16(x[2], x[3]);
                pk.z = pack_bf16(x[4], x[5]);
                pk.w = pack_bf16(x[6], x[7]);
                dst[cc] = pk;
              }
            }
          }
        }
      }
      PHASE_SYNC();
    }
  }
  // ---- final state
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    const int col = half * 64 + j;
    const int64_t off = (bh * 128 + row) * 128 + col;
    if (apply) {
      if (ar.final_out && seg == ar.P - 1) ar.final_out[off] = S[j];
    } else if (mpart) {
      if (ar.M_out) ar.M_out[seg * ar.out_seg_stride + off] = S[j];
    } else {
      if (ar.S_out) ar.S_out[seg * ar.out_seg_stride + off] = S[j];
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

// [B, Ts, heads, 128] bf16 tensor, boxes of 64 tokens x 64 columns of one head.
bool make_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t Ts, int64_t heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {128, (cuuint64_t)heads, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {256, (cuuint64_t)(heads * 256), (cuuint64_t)(Ts * heads * 256)};
  cuuint32_t box[4] = {64, 1, 64, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_make_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t Ts, int64_t heads) {
  return make_map(m, ptr, B, T, Ts, heads);
}

// [n][128][128] bf16 matrices (chunk states, state gradients), boxes of 128 rows x 64 columns.
bool tc_make_state_map(CUtensorMap* m, const void* ptr, int64_t n) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || n <= 0) return false;
  cuuint64_t dims[4] = {128, 128, (cuuint64_t)n, 1};
  cuuint64_t strides[3] = {256, 32768, (cuuint64_t)(n * 32768)};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_path(const Prob& pr) {
  return pr.dtype == GDN_BF16 && pr.dk == 128 && pr.dv == 128 && pr.B > 0 && pr.NC > 0;
}

cudaError_t launch_chunk_scan_tc(const Prob& pr, const Inputs& in, const WS& ws, int mode,
                                 int seg_first, int nseg, const float* init,
                                 int64_t init_seg_stride, void* o, float* final_out,
                                 float* M_out, float* S_out, int64_t out_seg_stride,
                                 void* hc, cudaStream_t st) {
  if (nseg <= 0 || pr.B == 0 || pr.NC == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  const void* qptr = in.q ? in.q : in.k;  // summaries never read q
  if (!make_map(&mq, qptr, pr.B, pr.T, pr.Ts, pr.Hqk) || !make_map(&mk, in.k, pr.B, pr.T, pr.Ts, pr.Hqk))
    return cudaErrorInvalidValue;
  const void* vptr = in.v ? in.v : in.k;
  if (!make_map(&mv, vptr, pr.B, pr.T, pr.Ts, in.v ? pr.H : pr.Hqk)) return cudaErrorInvalidValue;
  TcArgs ar;
  ar.T = pr.T; ar.Ts = pr.Ts; ar.H = pr.H; ar.r = pr.r; ar.NC = pr.NC; ar.CPS = pr.CPS;
  ar.P = pr.P; ar.l2norm = pr.l2norm; ar.eps = pr.eps; ar.scale = pr.scale;
  ar.a = (const __nv_bfloat16*)in.a; ar.b = (const __nv_bfloat16*)in.b;
  ar.A_log = in.A_log; ar.dt_bias = in.dt_bias; ar.valid_len = in.valid_len;
  ar.init = init; ar.init_seg_stride = init_seg_stride;
  ar.o = (__nv_bfloat16*)o; ar.final_out = final_out;
  ar.M_out = M_out; ar.S_out = S_out; ar.out_seg_stride = out_seg_stride;
  ar.hc = (__nv_bfloat16*)hc;
  ar.status = ws.status;
  ar.mode = mode; ar.seg_first = seg_first; ar.nseg = nseg;
  cudaError_t e = cudaFuncSetAttribute(k_chunk_scan_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(mode == MODE_SUM ? 2 : 1, (unsigned)pr.H, (unsigned)(pr.B * nseg));
  k_chunk_scan_tc<<<grid, FT, SMEM_BYTES, st>>>(mq, mk, mv, ar);
  return cudaGetLastError();
}

}  // namespace gdn
