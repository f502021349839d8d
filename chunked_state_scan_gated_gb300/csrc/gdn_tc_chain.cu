// gdn_tc_chain.cu -- tensor-core (tcgen05) chunk prologue and forward state chain
// of the bf16 path (dk = dv = 128, C = 64).
//
// The chunked gated delta rule (notation of gdn_simt.cu) splits into work that
// depends only on one chunk's inputs and a short recurrence on the state:
//
//   chunk-local   G = cumsum(g), gamma = e^G, P = tril(Q K^T o Gamma),
//                 A = tril(diag(beta) K K^T o Gamma, -1), T = (I + A)^-1,
//                 W = T diag(beta gamma) K,  U = T diag(beta) V
//   recurrence    V' = U - W S,  O = diag(gamma) Q S + P V',
//                 S <- gamma_C S + K^T diag(e^{G_C - G}) V'
//
// k_prep_tc runs the chunk-local part once for every (chunk, V head) in
// parallel and leaves its results in the workspace as bf16 "tile images": the
// exact bytes of a 128-byte-swizzled K-major shared-memory tile, so that a
// consumer fetches each with one plain bulk copy and hands it to tcgen05.mma
// as is.  With the depthwise Conv1D + SiLU of "linear attention cp #1035" in front
// (gdn_fwd_conv), k_prep_tc<true> loads the Conv1D inputs instead, convolves each
// chunk's tiles in shared memory and writes the activated q, k, v once for the
// later kernels.  k_chain_tc then walks the chunks of one segment of one (batch row,
// V head) with the state in fp32 registers and only the two state products
// per chunk (W S, then K^T V2) on its critical path.  It produces segment
// summaries (the "p2p" map H_out = M H_in + S of "linear attention cp #1035":
// M from the identity with U = 0, S from zero), the token output from a given
// initial state, or every chunk-start state for the backward.
//
// Tile images (bf16): a [64][128] matrix is two 8 KB atoms (columns 0..63,
// 64..127); row r, 16-byte chunk c of an atom sits at r*128 + ((c ^ r) & 7)*16.
// A [64][64] matrix is one atom.
#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include "gdn_internal.h"
#include "gdn_tc_common.cuh"
#include "gdn_vec.cuh"

namespace gdn {

bool tc_make_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t Ts, int64_t heads);
bool tc_make_map_rows(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t Ts,
                      int64_t heads, int rows);

namespace {

using namespace tc;

constexpr uint32_t kImg = 16384;   // bytes of a [64][128] tile image
constexpr uint32_t kImgP = 8192;   // bytes of a [64][64] tile image

__device__ __forceinline__ uint32_t img_chunk(int r, int c16) {  // 16-byte chunk c16 (0..15) of row r
  return (uint32_t)((c16 >> 3) * 8192) + kmaj_chunk(r, c16 & 7);
}

__device__ __forceinline__ uint4 pack8(const float* x) {
  uint4 v;
  v.x = pack_bf16(x[0], x[1]);
  v.y = pack_bf16(x[2], x[3]);
  v.z = pack_bf16(x[4], x[5]);
  v.w = pack_bf16(x[6], x[7]);
  return v;
}

__device__ __forceinline__ int64_t clamp_len(const int32_t* valid_len, int64_t b, int64_t T,
                                             int* status, bool report) {
  if (!valid_len) return T;
  int64_t L = valid_len[b];
  if (L < 0 || L > T) {
    if (report && status) atomicOr(status, kStatusClamped);
    L = L < 0 ? 0 : T;
  }
  return L;
}

// ============================================================================
// k_prep_tc: persistent, min(B H NC, 2 SMs) CTAs of 256 threads (two per SM), each
// walking chunks.  Warp w reads TMEM lane quadrant w & 3 (tile row `row`) and handles
// column half w >> 2 of that row.
//
// The q and k row norms come from the diagonal of one product [Q;K][Q;K]^T of
// the raw tiles, so neither tile is rewritten for the norm: every later use of
// q_hat = rq q and k_hat = rk k applies the per-token factors rq = scale / |q|,
// rk = 1 / |k| (kept in the workspace) to an fp32 result or to a row of bf16 operands.
// With the Conv1D in front (k_prep_tc<true>), the tiles arrive as the Conv1D inputs
// x and are replaced in place by SiLU(conv(x)) before their first product (q, k at the
// chunk start, v before the U product), each activated row also written out as q, k, v.
// ============================================================================
constexpr int PT = 256;
constexpr uint32_t P_QK = 0;                   // atoms a at a*16384: [Q_a | K_a], raw, 8 KB each
constexpr uint32_t P_PST = P_QK + 16384;       // P image staging (Q_1: free after [Q;K][Q;K]^T)
constexpr uint32_t P_V = 32768;                // V atoms at a*8192
constexpr uint32_t P_TA = 49152;               // [T_u; T_w], 128 x 64 K-major
constexpr uint32_t P_A = 65536;                // fp32 A [64][LDA]
constexpr uint32_t P_T = P_A + 64 * LDA * 4;   // fp32 T [64][LDA]
constexpr uint32_t P_Y = P_T + 64 * LDA * 4;   // solve scratch, 8 warps x 128 floats
constexpr uint32_t P_SC = P_Y + 1024 * 4;      // gates, row factors, barriers
constexpr uint32_t P_SMEM = P_SC + 1536 + 64 + 1024;
// With the Conv1D in front: the 3 tokens before the chunk of x_q, x_k, x_v (3 x 256 bytes
// each, unswizzled), read by the convolution of the chunk's first rows.
constexpr uint32_t P_LB = (P_SC + 1536 + 64 + 127) / 128 * 128;
constexpr uint32_t P_SMEM_CONV = P_LB + 3 * 768 + 1024;

// Writes T diag(beta) (rows 0..63) and T diag(beta gamma rk) (rows 64..127) of the
// 128 x 64 K-major bf16 tile [T_u; T_w] as the solve finalises each entry of T.
struct TaEmit {
  uint8_t* tile;
  const float* cu;  // beta
  const float* cw;  // beta gamma rk
  __device__ __forceinline__ void one(int i, int j, float x) const {
    const uint32_t off = kmaj_chunk(i, j >> 3) + (j & 7) * 2;
    *reinterpret_cast<__nv_bfloat16*>(tile + off) = __float2bfloat16_rn(x * cu[j]);
    *reinterpret_cast<__nv_bfloat16*>(tile + 8192 + off) = __float2bfloat16_rn(x * cw[j]);
  }
  __device__ __forceinline__ void two(int i, int j, float x0, float x1) const {
    const uint32_t off = kmaj_chunk(i, j >> 3) + (j & 7) * 2;
    *reinterpret_cast<uint32_t*>(tile + off) = pack_bf16(x0 * cu[j], x1 * cu[j + 1]);
    *reinterpret_cast<uint32_t*>(tile + 8192 + off) = pack_bf16(x0 * cw[j], x1 * cw[j + 1]);
  }
};

struct PrepArgs {
  int64_t T, Ts, H, Hqk, r, NC;
  int l2norm;
  float eps, scale;
  const __nv_bfloat16* a;
  const __nv_bfloat16* b;
  const float* A_log;
  const float* dt_bias;
  const int32_t* valid_len;
  float* rqk;    // [B][Hqk][NC][128]: rq of the chunk's 64 tokens, then rk
  uint8_t* wim;  // [B][H][NC] images of W
  uint8_t* uim;  // [B][H][NC] images of U
  uint8_t* pim;  // [B][H][NC] images of P (64 x 64)
  uint8_t* tim;  // [B][H][NC] images of T = (I + A)^-1 (64 x 64), or null
  float* gl;     // [B][H][NC][64] cumulative gate in log2 units
  int* status;
  int64_t NW;    // B * H * NC chunks of work
  // Conv1D + SiLU in front (index 0: q, 1: k, 2: v); the tiles are loaded from x
  int convK;                       // taps, 1..4
  const float* cw[3];              // [channels][convK]
  const float* cb[3];              // [channels] or null
  const __nv_bfloat16* chalo[3];   // [B][convK - 1][channels] or null (zeros)
  __nv_bfloat16* cy[3];            // the activated q, k, v, written for the later kernels
};

// Taps and bias of channels ch .. ch + 7 of w [C][KK] (8 KK contiguous floats) and bias
// [C], as float4 loads; wv[j][i] holds the tap of x~[t - 3 + i] (zero for i < 4 - KK).
template <int KK>
__device__ __forceinline__ void conv_taps_k(const float* __restrict__ w,
                                            const float* __restrict__ bias, int64_t ch,
                                            float (&wv)[8][4], float (&bv)[8]) {
  float t[8 * KK];
  const float4* w4 = reinterpret_cast<const float4*>(w + ch * KK);  // 16-byte aligned: ch % 8 == 0
#pragma unroll
  for (int q = 0; q < 2 * KK; ++q) {
    const float4 f = __ldg(w4 + q);
    t[4 * q] = f.x; t[4 * q + 1] = f.y; t[4 * q + 2] = f.z; t[4 * q + 3] = f.w;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) wv[j][i] = (i >= 4 - KK) ? t[j * KK + i - (4 - KK)] : 0.f;
  if (bias) {
    const float4 b0 = __ldg(reinterpret_cast<const float4*>(bias + ch));
    const float4 b1 = __ldg(reinterpret_cast<const float4*>(bias + ch) + 1);
    bv[0] = b0.x; bv[1] = b0.y; bv[2] = b0.z; bv[3] = b0.w;
    bv[4] = b1.x; bv[5] = b1.y; bv[6] = b1.z; bv[7] = b1.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) bv[j] = 0.f;
  }
}
__device__ __forceinline__ void conv_taps(const float* w, const float* bias, int K, int64_t ch,
                                          float (&wv)[8][4], float (&bv)[8]) {
  switch (K) {
    case 1: conv_taps_k<1>(w, bias, ch, wv, bv); break;
    case 2: conv_taps_k<2>(w, bias, ch, wv, bv); break;
    case 3: conv_taps_k<3>(w, bias, ch, wv, bv); break;
    default: conv_taps_k<4>(w, bias, ch, wv, bv); break;
  }
}

// Two fp32 lanes at once: fma.rn.f32x2 rounds each lane as fmaf does.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}

// Causal depthwise Conv1D + SiLU of one 8-channel column (16-byte chunk `ccs` of a
// 128-byte-swizzled 64-row atom) over rows u0 .. u0 + N - 1 of the tile, in place: row u
// (token t0 + u) becomes SiLU(bias + sum of the KK taps over x~[t - KK + 1 .. t]), rounded
// to bf16, with the same operation order and rounding as the stand-alone Conv1D pass
// (channel pairs on packed fp32 operations), so both give the same bits.  back[i] holds the
// inputs of token u0 - 3 + i (bf16, 8 channels); wv, bv the column's taps and bias
// (conv_taps).  Rows past the end of the row (t0 + u >= T) become zero, as a copy of the
// activated tensor would read there; the others also go to y + u * ystride when y is set.
template <int N, int KK>
__device__ __forceinline__ void conv_column(uint8_t* atom, int ccs, int u0,
                                            const uint4 (&back)[3], const float (&wv)[8][4],
                                            const float (&bv)[8], int64_t t0, int64_t T,
                                            __nv_bfloat16* y, int64_t ystride) {
  float xw[3][8];
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const uint32_t wd[4] = {back[i].x, back[i].y, back[i].z, back[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[e]));
      xw[i][2 * e] = f.x;
      xw[i][2 * e + 1] = f.y;
    }
  }
#pragma unroll
  for (int r = 0; r < N; ++r) {
    const int u = u0 + r;
    const uint32_t off = kmaj_chunk(u, ccs);
    float xc[8];
    ld_chunk(atom, off, xc);
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      float2 acc = make_float2(bv[j], bv[j + 1]);
#pragma unroll
      for (int i = 4 - KK; i < 3; ++i)
        acc = fma2(make_float2(wv[j][i], wv[j + 1][i]), make_float2(xw[i][j], xw[i][j + 1]), acc);
      acc = fma2(make_float2(wv[j][3], wv[j + 1][3]), make_float2(xc[j], xc[j + 1]), acc);
      o[j] = acc.x * vec::sigm(acc.x);
      o[j + 1] = acc.y * vec::sigm(acc.y);
    }
    uint4 packed = make_uint4(0, 0, 0, 0);
    if (t0 + u < T) {
      packed.x = pack_bf16(o[0], o[1]);
      packed.y = pack_bf16(o[2], o[3]);
      packed.z = pack_bf16(o[4], o[5]);
      packed.w = pack_bf16(o[6], o[7]);
      if (y) *reinterpret_cast<uint4*>(y + u * ystride) = packed;
    }
    *reinterpret_cast<uint4*>(atom + off) = packed;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      xw[0][j] = xw[1][j];
      xw[1][j] = xw[2][j];
      xw[2][j] = xc[j];
    }
  }
}
template <int N>
__device__ __forceinline__ void conv_column_k(int K, uint8_t* atom, int ccs, int u0,
                                              const uint4 (&back)[3], const float (&wv)[8][4],
                                              const float (&bv)[8], int64_t t0, int64_t T,
                                              __nv_bfloat16* y, int64_t ystride) {
  switch (K) {
    case 1: conv_column<N, 1>(atom, ccs, u0, back, wv, bv, t0, T, y, ystride); break;
    case 2: conv_column<N, 2>(atom, ccs, u0, back, wv, bv, t0, T, y, ystride); break;
    case 3: conv_column<N, 3>(atom, ccs, u0, back, wv, bv, t0, T, y, ystride); break;
    default: conv_column<N, 4>(atom, ccs, u0, back, wv, bv, t0, T, y, ystride); break;
  }
}

// The inputs of token u (relative to the chunk start t0) of an 8-channel column: a row of the
// tile (u >= 0), of the halo (first chunk of a row), zero before the halo, or the copy of the
// 3 tokens before the chunk (side: rows of 256 bytes, 16-byte chunk cc).
__device__ __forceinline__ uint4 conv_back_row(const uint8_t* atom, int ccs, const uint8_t* side,
                                               int cc, int u, int64_t c,
                                               const __nv_bfloat16* halo, int K, int64_t b,
                                               int64_t C, int64_t ch) {
  if (u >= 0) return *reinterpret_cast<const uint4*>(atom + kmaj_chunk(u, ccs));
  if (c == 0) {
    const int hr = K - 1 + u;  // halo row of token u
    if (!halo || hr < 0) return make_uint4(0, 0, 0, 0);
    return *reinterpret_cast<const uint4*>(halo + (b * (K - 1) + hr) * C + ch);
  }
  return *reinterpret_cast<const uint4*>(side + (u + 3) * 256 + cc * 16);
}

// CONV: the q, k, v tiles are loaded from the Conv1D inputs x (maps mq, mk, mv), with the 3
// tokens before the chunk (maps mlq, mlk, mlv), and convolved in place before their first use.
template <bool CONV>
__global__ void __launch_bounds__(PT, 2)
    k_prep_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mlq,
              const __grid_constant__ CUtensorMap mlk, const __grid_constant__ CUtensorMap mlv,
              PrepArgs ar) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t base = smem_u32(sm);
  // operand descriptors: base descriptor + byte offset / 16 (the start address field)
  const uint64_t d16 = sdesc(base, 16, 1024), d8192 = sdesc(base, 8192, 1024),
                 d16384 = sdesc(base, 16384, 1024);
  float* sG = (float*)(sm + P_SC);
  float* sGam = sG + 64;
  float* sBeta = sGam + 64;
  float* sInv = sBeta + 64;  // [128]: rq (rows 0..63), rk (rows 64..127)
  float* sCw = sInv + 128;   // [64]: beta gamma rk, the column factors of T_w
  uint64_t* bar_qk = (uint64_t*)(sm + P_SC + 1536);
  uint64_t* bar_v = bar_qk + 1;
  uint64_t* bar_mma = bar_qk + 2;
  uint64_t* bar_w = bar_qk + 3;  // the W product (the U product completes on bar_mma)
  uint32_t* s_tmem = (uint32_t*)(bar_qk + 4);
  int* s_abort = (int*)(s_tmem + 1);
  float* sA = (float*)(sm + P_A);
  float* sT = (float*)(sm + P_T);
  float* sY = (float*)(sm + P_Y);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int row = quad * 32 + lane;  // TMEM lane of this thread
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const int tg = tid - 64;  // gate warps 2, 3: token tg
  const bool gate_warp = warp == 2 || warp == 3;

  // Persistent: CTA i takes chunks w = i, i + gridDim.x, ... (w: c = w % NC, h = (w / NC) % H,
  // b = w / (NC H); 32-bit index arithmetic, the host keeps NW below 2^31), skipping chunks of
  // padding only (every consumer skips them).  The next chunk's q, k copies go out as soon as
  // the current chunk's last product has read k, its gate inputs are read a chunk ahead, and
  // its v copy goes out before the current chunk's solve.
  struct Item {
    int64_t c, h, b;
  };
  auto item_of = [&](int64_t w) {
    const uint32_t uw = (uint32_t)w, q1 = uw / (uint32_t)ar.NC;
    return Item{(int64_t)(uw - q1 * (uint32_t)ar.NC), (int64_t)(q1 % (uint32_t)ar.H),
                (int64_t)(q1 / (uint32_t)ar.H)};
  };
  auto len_of = [&](int64_t bb, bool report) { return clamp_len(ar.valid_len, bb, ar.T, ar.status, report); };
  auto next_live = [&](int64_t w) {
    for (; w < ar.NW; w += gridDim.x) {
      if (!ar.valid_len) break;
      const Item it = item_of(w);
      if (it.c * 64 < len_of(it.b, false)) break;
    }
    return w;
  };
  auto issue_qk = [&](const Item& it) {
    mbar_arrive_expect_tx(bar_qk, CONV ? 32768u + 1536u : 32768u);
    for (int at = 0; at < 2; ++at) {
      tma_load_4d(sm + P_QK + at * 16384, &mq, at * 64, (int)(it.h / ar.r), (int)(it.c * 64),
                  (int)it.b, bar_qk);
      tma_load_4d(sm + P_QK + at * 16384 + 8192, &mk, at * 64, (int)(it.h / ar.r),
                  (int)(it.c * 64), (int)it.b, bar_qk);
    }
    if (CONV) {  // tokens t0 - 3 .. t0 - 1 (zero-filled before the row's first token)
      tma_load_4d(sm + P_LB, &mlq, 0, (int)(it.h / ar.r), (int)(it.c * 64) - 3, (int)it.b,
                  bar_qk);
      tma_load_4d(sm + P_LB + 768, &mlk, 0, (int)(it.h / ar.r), (int)(it.c * 64) - 3,
                  (int)it.b, bar_qk);
    }
  };
  auto issue_v = [&](const Item& it) {
    mbar_arrive_expect_tx(bar_v, CONV ? 16384u + 768u : 16384u);
    for (int at = 0; at < 2; ++at)
      tma_load_4d(sm + P_V + at * 8192, &mv, at * 64, (int)it.h, (int)(it.c * 64), (int)it.b,
                  bar_v);
    if (CONV)
      tma_load_4d(sm + P_LB + 1536, &mlv, 0, (int)it.h, (int)(it.c * 64) - 3, (int)it.b, bar_v);
  };
  // Gate inputs (warps 2, 3: a, b, dt_bias, A_log of token tg), kept as loaded: their first
  // use, in the chunk's gate step, is where the threads wait for them.
  __nv_bfloat16 ra = __float2bfloat16_rn(0.f), rb = ra;
  float dtb = 0.f, alog = 0.f;
  bool glive = false;
  auto gate_load = [&](const Item& it) {
    glive = gate_warp && it.c * 64 + tg < len_of(it.b, false);
    if (glive) {
      const int64_t gi = (it.b * ar.Ts + it.c * 64 + tg) * ar.H + it.h;
      ra = ar.a[gi];
      rb = ar.b[gi];
      dtb = ar.dt_bias[it.h];
      alog = ar.A_log[it.h];
    }
  };
  uint32_t pend = 0;  // tid 0: 1 = a q/k copy, 2 = a v copy in flight (drained on an abort)

  const int64_t w0 = next_live(blockIdx.x);
  if (w0 < ar.NW) gate_load(item_of(w0));
  if (tid == 0) {  // the barriers are this thread's own: the first copies go out at once
    mbar_init(bar_qk, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_w, 1);
    fence_barrier_init();
    *s_abort = 0;
    if (w0 < ar.NW) {
      issue_qk(item_of(w0));
      issue_v(item_of(w0));
      pend = 3;
    }
  }
  if (warp == 0) tmem_alloc(s_tmem, 256);
  for (int e = tid; e < 1024; e += PT)  // [T_u; T_w]: the solve writes only the lower triangle
    reinterpret_cast<uint4*>(sm + P_TA)[e] = make_uint4(0, 0, 0, 0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  for (int64_t w = w0, kk = 0; w < ar.NW; ++kk) {
  const Item cur = item_of(w);
  const int64_t wn = next_live(w + gridDim.x);
  const int64_t c = cur.c, h = cur.h, b = cur.b;
  const int64_t hq = h / ar.r, bh = b * ar.H + h;
  (void)len_of(b, tid == 0 && c == 0 && h == 0);  // (reports a clamped valid_len once)
  const uint32_t par = (uint32_t)(kk & 1);
  // ---- [Q; K] [Q; K]^T -> cols [0, 128): row norms on the diagonal, Q K^T and K K^T in cols
  //      64..127, issued as soon as q and k land; the gates are formed meanwhile
  if (CONV) {  // every thread waits for the x tiles: the Conv1D + SiLU runs in place first
    // lane: q or k (tq), 8-channel column cc; warp: tokens 8 warp .. + 7.  The taps are
    // read while the copies land.
    const int jc = tid & 31, tq = jc >> 4, cc = jc & 15, u0 = warp * 8;
    const int64_t C = ar.Hqk * 128, ch = hq * 128 + cc * 8;
    float wv[8][4], bv[8];
    conv_taps(tq ? ar.cw[1] : ar.cw[0], tq ? ar.cb[1] : ar.cb[0], ar.convK, ch, wv, bv);
    const bool landed = !*s_abort && mbar_wait(bar_qk, par, ar.status, kStatusTimeout);
    if (!landed) *s_abort = 1;
    if (tid == 0 && landed) pend &= ~1u;
    __syncthreads();
    if (*s_abort) goto done;
    {
      uint8_t* atom = sm + P_QK + (cc >> 3) * 16384 + tq * 8192;
      const __nv_bfloat16* halo = tq ? ar.chalo[1] : ar.chalo[0];
      uint4 back[3];
#pragma unroll
      for (int i = 0; i < 3; ++i)
        back[i] = conv_back_row(atom, cc & 7, sm + P_LB + tq * 768, cc, u0 - 3 + i, c, halo,
                                ar.convK, b, C, ch);
      __syncthreads();  // the rows before each thread's own are read: convolve in place
      __nv_bfloat16* y = h % ar.r ? nullptr  // one V head of the group writes q and k
                                  : (tq ? ar.cy[1] : ar.cy[0]) + (b * ar.Ts + c * 64) * C + ch;
      conv_column_k<8>(ar.convK, atom, cc & 7, u0, back, wv, bv, c * 64, ar.T, y, C);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (tid == 0) {
    if (*s_abort) {  // (the previous chunk gave up before issuing this chunk's copies)
    } else if (!CONV && !mbar_wait(bar_qk, par, ar.status, kStatusTimeout)) {
      *s_abort = 1;
    } else {
      if (!CONV) pend &= ~1u;
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 128, 0, 0);
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t at = ks >> 2, k4 = ks & 3;
        const uint64_t d = (d16 + ((P_QK + at * 16384 + k4 * 32) >> 4));
        mma_bf16(tmem, d, d, id, ks > 0);
      }
      mma_commit(bar_mma);
    }
  }
  if (gate_warp) {  // g, beta and the cumulative gate in log2 units (scan over 64 tokens)
    float g = 0.f, be = 0.f;
    if (glive) {
      const float xa = __bfloat162float(ra) + dtb;
      const float sp = xa > 20.f ? xa : log1pf(expf(xa));
      g = -expf(alog) * sp;
      be = 1.f / (1.f + expf(-__bfloat162float(rb)));
    }
    float v = g * kLog2e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (tg == 31) sY[0] = v;  // the first half's total (the solve's scratch is free until then)
    asm volatile("bar.sync 1, 64;" ::: "memory");
    if (tg >= 32) v += sY[0];
    sG[tg] = v;
    sBeta[tg] = be;
    sGam[tg] = exp2f(v);
    ar.gl[(bh * ar.NC + c) * 64 + tg] = v;
    if (wn < ar.NW) gate_load(item_of(wn));  // the next chunk's, read a chunk ahead
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*s_abort) goto done;
  if (!mbar_wait(bar_mma, 0, ar.status, kStatusTimeout)) *s_abort = 1;
  tc_fence_after();
  float v[32];  // row . k_j for j = 32*half + e (read with the diagonal block: one wait)
  if (half == 0) {  // diagonal element (row, row) sits in column group `quad`, element `lane`
    float d[32];
    tmem_ld32x2(tmem + lane_off + 32 * quad, d, tmem + lane_off + 64 + 32 * half, v);
    float nrm = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) nrm = (e == lane) ? d[e] : nrm;
    float inv = ar.l2norm ? rsqrtf(nrm + ar.eps) : 1.f;
    if (row < 64) inv *= ar.scale;
    sInv[row] = inv;
  } else {
    tmem_ld32(tmem + lane_off + 64 + 32 * half, v);
  }
  __syncthreads();
  if (h % ar.r == 0 && tid < 128) ar.rqk[((b * ar.Hqk + hq) * ar.NC + c) * 128 + tid] = sInv[tid];
  if (tid >= 128 && tid < 192) sCw[tid - 128] = sBeta[tid - 128] * sGam[tid - 128] * sInv[tid - 64];
  {
    const int i = row & 63;
    const float gi = sG[i], si = sInv[row];
    // v[e] <- row . k_j rk_j e^{G_i - G_j} (j = 32 half + e), zero above the diagonal; a
    // warp whose 32 columns all lie above its rows (half 1, rows 0..31) has nothing to do
    const bool upper = half * 32 > i;  // uniform across the warp
    if (!upper) {
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 g4 = *reinterpret_cast<const float4*>(sG + half * 32 + 4 * q4);
        const float4 r4 = *reinterpret_cast<const float4*>(sInv + 64 + half * 32 + 4 * q4);
        const float gg[4] = {g4.x, g4.y, g4.z, g4.w}, rr[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = 4 * q4 + u, j = half * 32 + e;
          v[e] = (j <= i) ? v[e] * rr[u] * exp2f(gi - gg[u]) : 0.f;
        }
      }
    }
    if (row < 64) {  // P = tril(Q K^T o Gamma) with the norm factors: bf16 image, staged
      uint8_t* dst = sm + P_PST;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) p[e] = upper ? 0.f : si * v[cc * 8 + e];
        *reinterpret_cast<uint4*>(dst + kmaj_chunk(i, half * 4 + cc)) = pack8(p);
      }
    } else if (!upper) {  // A = strictly lower part, times beta_i (the solve never reads above it)
      const float bs = sBeta[i] * si;
      float4* dst = reinterpret_cast<float4*>(sA + i * LDA + half * 32);
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        float w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = half * 32 + 4 * q4 + u;
          w[u] = (j < i) ? bs * v[4 * q4 + u] : 0.f;
        }
        dst[q4] = make_float4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  if (tid == 64) bulk_wait_read();  // the previous chunk's W image (over sT) has been read
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {  // the P image, then this chunk's v (the previous U image has been read)
    bulk_store(ar.pim + (bh * ar.NC + c) * (int64_t)kImgP, sm + P_PST, kImgP);
    bulk_commit();
    if (kk > 0) {
      bulk_wait_read_but1();
      issue_v(cur);
      pend |= 2u;
    }
  }
  // T = (I + A)^-1, with [T_u; T_w] = [T diag(beta); T diag(beta gamma rk)] (bf16, W is
  // formed from raw k) written as each entry of T is final
  solve_unit_lower64_mma(sA, sT, sY, LDA, TaEmit{sm + P_TA, sBeta, sCw});
  // [T_u; T_w] is final: the W product (it needs only that tile and k) goes out at once, so
  // that k's slot, and with it the next chunk's q/k copies, free up as early as possible
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, 128, 0, 1);
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tmem + 128, (d16 + ((P_TA + ks * 32) >> 4)),
               (d16384 + ((P_QK + 8192 + ks * 2048) >> 4)), id, ks > 0);
    mma_commit(bar_w);
  }
  if (ar.tim) {  // T for the backward, bf16 image, staged where A was (the solve is done)
    uint8_t* dst = sm + P_A;
    for (int e = tid; e < 512; e += PT) {
      const int i = e >> 3, cc = e & 7;
      float x[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int j = cc * 8 + q;
        x[q] = (j <= i) ? sT[i * LDA + j] : 0.f;
      }
      *reinterpret_cast<uint4*>(dst + kmaj_chunk(i, cc)) = pack8(x);
    }
  }
  // the Conv1D + SiLU of the v tile comes after the copy lands; its taps are read first.
  // 16-lane groups: 8-channel column cc, tokens 4 (tid / 16) .. + 3
  const int vcc = tid & 15, vu0 = (tid >> 4) * 4;
  const int64_t vC = ar.H * 128, vch = h * 128 + vcc * 8;
  float vwv[8][4], vbv[8];
  if (CONV) conv_taps(ar.cw[2], ar.cb[2], ar.convK, vch, vwv, vbv);
  if (!mbar_wait(bar_v, par, ar.status, kStatusTimeout)) *s_abort = 1;
  if (tid == 0) pend &= ~2u;
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*s_abort) goto done;
  if (CONV) {
    uint8_t* atom = sm + P_V + (vcc >> 3) * 8192;
    uint4 back[3];
#pragma unroll
    for (int i = 0; i < 3; ++i)
      back[i] = conv_back_row(atom, vcc & 7, sm + P_LB + 1536, vcc, vu0 - 3 + i, c, ar.chalo[2],
                              ar.convK, b, vC, vch);
    __syncthreads();
    conv_column_k<4>(ar.convK, atom, vcc & 7, vu0, back, vwv, vbv, c * 64, ar.T,
                     ar.cy[2] + (b * ar.Ts + c * 64) * vC + vch, vC);
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  // ---- [T_u; T_w] V -> cols [0,128) (U in rows 0..63); [T_u; T_w] K -> cols [128,256) (W in
  //      64..127, issued above)
  if (tid == 0) {
    if (ar.tim) {  // the T image (group 2)
      bulk_store(ar.tim + (bh * ar.NC + c) * (int64_t)kImgP, sm + P_A, kImgP);
      bulk_commit();
    }
    // the next chunk's q and k go where this chunk's are once the W product has read k and
    // the P image has read its staging (every group but the T image's)
    if (!mbar_wait(bar_w, par, ar.status, kStatusTimeout)) *s_abort = 1;
    if (ar.tim) bulk_wait_read_but1(); else bulk_wait_read();
    if (wn < ar.NW && !*s_abort) {
      issue_qk(item_of(wn));
      pend |= 1u;
    }
    const uint32_t id = idesc_bf16(128, 128, 0, 1);
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tmem, (d16 + ((P_TA + ks * 32) >> 4)), (d8192 + ((P_V + ks * 2048) >> 4)), id,
               ks > 0);
    mma_commit(bar_mma);
  }
  {  // U (rows 0..63: quadrants 0, 1) staged where V was once its product is done, W (rows
     // 64..127: quadrants 2, 3) over the solve's T tile (free since the T image was staged);
     // each half stores its image as soon as its 128 threads have staged it
    const bool isw = row >= 64;
    const int i = row & 63;
    if (!mbar_wait(isw ? bar_w : bar_mma, isw ? par : 1, ar.status, kStatusTimeout)) *s_abort = 1;
    tc_fence_after();
    uint8_t* dst = sm + (isw ? P_T : P_V);
    const uint32_t src = tmem + lane_off + (isw ? 128 : 0) + 64 * half;
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) {
      float v[32];
      tmem_ld32(src + q2 * 32, v);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        *reinterpret_cast<uint4*>(dst + img_chunk(i, half * 8 + q2 * 4 + cc)) = pack8(&v[cc * 8]);
    }
    fence_proxy_async();
    tc_fence_before();
    if (isw) asm volatile("bar.sync 3, 128;" ::: "memory");  // warps 2, 3, 6, 7
    else asm volatile("bar.sync 2, 128;" ::: "memory");      // warps 0, 1, 4, 5
    if (tid == 0) {
      bulk_store(ar.uim + (bh * ar.NC + c) * (int64_t)kImg, sm + P_V, kImg);
      bulk_commit();
    } else if (tid == 64) {
      bulk_store(ar.wim + (bh * ar.NC + c) * (int64_t)kImg, sm + P_T, kImg);
      bulk_commit();
    }
  }
  w = wn;
  }  // chunk loop
  if (tid == 0 || tid == 64) bulk_wait_read();  // shared memory is released when the CTA exits

done:
  if (*s_abort && tid == 0) {  // let the copies still in flight land before the CTA exits
    if (pend & 1u) {
      mbar_wait(bar_qk, 0, nullptr, 0);
      mbar_wait(bar_qk, 1, nullptr, 0);
    }
    if (pend & 2u) {
      mbar_wait(bar_v, 0, nullptr, 0);
      mbar_wait(bar_v, 1, nullptr, 0);
    }
    bulk_wait_read();  // and the stores issued so far read their staging
  }
  if (*s_abort && tid == 64) bulk_wait_read();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ============================================================================
// k_chain_tc: grid (parts, H, B * nseg), 256 threads.  Warp w reads TMEM lane
// quadrant w & 3 (state row `row`) and owns state columns (w >> 2) * 64 .. +63.
// q and k tiles are the raw inputs (TMA); their norm factors rq, rk come from
// the prologue and are applied to the rows of V2 and of the product Q S.
// ============================================================================
constexpr int CT = 256;
enum { CH_APPLY = 0, CH_SUM = 1, CH_STATES = 2 };

// Summary / states layout (one buffer; two CTAs fit on an SM).
constexpr uint32_t S_XA = 0;        // atoms a at a*16384: [W_a | K_a]
constexpr uint32_t S_U = 32768;     // U image
constexpr uint32_t S_S = 49152;     // state, bf16, MN-major (column halves 16 KB apart)
constexpr uint32_t S_V2 = 81920;    // V2^T = (diag(rk e^{G_C - G}) V')^T [dv][tok], K-major
constexpr uint32_t S_NI = 98304;    // -I (64 x 64 bf16): U^T (-I) = -U^T as an MMA term
constexpr uint32_t S_G = 106496;    // G of the chunk (64 floats), then rk (64 floats)
constexpr uint32_t S_SC = 107008;   // barriers
constexpr uint32_t S_SMEM = S_SC + 128 + 1024;

// Apply layout ([W | Q | K] double-buffered; U, P single).
constexpr uint32_t A_XA = 0;        // buffer x at x*49152; atoms a at a*24576: [W_a | Q_a | K_a]
constexpr uint32_t A_U = 98304;
constexpr uint32_t A_PZ = 114688;   // [0; P]: 64 zero rows then P, 128 x 64 K-major
constexpr uint32_t A_S = 131072;
constexpr uint32_t A_VP = 163840;   // V'
constexpr uint32_t A_V2 = 180224;
constexpr uint32_t A_G = 196608;    // buffer x at x*768: G (64 floats), rq (64), rk (64)
constexpr uint32_t A_O = 198656;    // output tile [64 tokens][128] (two K-major atoms), TMA-stored
constexpr uint32_t A_SC = 215040;
constexpr uint32_t A_SMEM = A_SC + 128 + 1024;

struct ChainArgs {
  int64_t T, Ts, H, Hqk, r, NC, CPS;
  int P;
  const float* rqk;
  const uint8_t* wim;
  const uint8_t* uim;
  const uint8_t* pim;
  const float* gl;
  const int32_t* valid_len;
  const float* init;
  int64_t init_seg_stride;
  __nv_bfloat16* o;
  float* final_out;
  float* M_out;
  float* S_out;
  int64_t out_seg_stride;
  uint8_t* hc;        // CH_STATES: chunk-start states, [B][H][NC] 32 KB bf16 tile images
  int* status;
  int seg_first, nseg;
};

#define CHAIN_SYNC()            \
  do {                          \
    fence_proxy_async();        \
    tc_fence_before();          \
    __syncthreads();            \
    tc_fence_after();           \
    if (*s_abort) goto done;    \
  } while (0)

// One CTA of the chain: `part` (summary: 0 = S, 1 = M), head h, zi = row * nseg + segment.
template <int MODE>
__device__ __forceinline__ void chain_cta(const CUtensorMap& mq, const CUtensorMap& mk,
                                          const CUtensorMap& mo, const ChainArgs& ar, int part,
                                          int64_t h, int64_t zi) {
  constexpr bool kApply = MODE == CH_APPLY;
  constexpr uint32_t XSTR = kApply ? 24576 : 16384;  // atom stride in the [W | (Q) | K] block
  constexpr uint32_t KOFF = kApply ? 16384 : 8192;   // K's offset inside an atom
  constexpr uint32_t OFF_S = kApply ? A_S : S_S;
  constexpr uint32_t OFF_U = kApply ? A_U : S_U;
  constexpr uint32_t OFF_V2 = kApply ? A_V2 : S_V2;
  constexpr uint32_t OFF_SC = kApply ? A_SC : S_SC;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t base = smem_u32(sm);
  // operand descriptors: base descriptor + byte offset / 16 (the start address field)
  const uint64_t d16 = sdesc(base, 16, 1024), d8192 = sdesc(base, 8192, 1024),
                 d16384 = sdesc(base, 16384, 1024);
  const uint64_t dxs = sdesc(base, XSTR, 1024);
  // apply: xa0, xa1, u, p, mma; otherwise: w, k, u, -, mma
  uint64_t* bars = (uint64_t*)(sm + OFF_SC);
  uint64_t* bar_u = bars + 2;
  uint64_t* bar_mma = bars + 4;
  uint32_t* s_tmem = (uint32_t*)(bars + 6);
  int* s_abort = (int*)(s_tmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int row = quad * 32 + lane;
  const bool mpart = MODE == CH_SUM && part == 1;
  const bool needU = !mpart;
  const int64_t b = zi / ar.nseg;
  const int seg = ar.seg_first + (int)(zi % ar.nseg);
  const int64_t hq = h / ar.r, bh = b * ar.H + h;
  const int64_t cs = (int64_t)seg * ar.CPS;
  const int64_t L = clamp_len(ar.valid_len, b, ar.T, ar.status, false);
  // chunks of padding only (from ceil(L / 64) on) leave the state unchanged: not walked
  const int64_t ce = min(cs + ar.CPS < ar.NC ? cs + ar.CPS : ar.NC, (L + 63) / 64);
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  uint32_t pend = 0;  // tid 0: barriers with a copy or MMA in flight (drained on an abort)

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(bars + i, 1);
    mbar_init(bar_mma, kApply ? 2 : 1);  // apply: MMA_b and MMA_c come from tid 0 and 32
    fence_barrier_init();
    *s_abort = 0;
  }
  if (warp == 0) tmem_alloc(s_tmem, 256);
  if (kApply)  // zero rows of [0; P]
    for (int e = tid; e < 512; e += CT) reinterpret_cast<uint4*>(sm + A_PZ)[e] = make_uint4(0, 0, 0, 0);
  if (!kApply && needU)  // -I, the operand that adds -U^T to the first product
    for (int e = tid; e < 512; e += CT) {
      const int r = e >> 3, cc = e & 7;
      float x[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) x[q] = (r == cc * 8 + q) ? -1.f : 0.f;
      st_chunk(sm + S_NI, kmaj_chunk(r, cc), x);
    }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tA = tmem, tB = tmem + 128;

  float S[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    const int col = half * 64 + j;
    float x = 0.f;
    if (MODE != CH_SUM) {
      if (ar.init) x = ar.init[seg * ar.init_seg_stride + (bh * 128 + row) * 128 + col];
    } else if (mpart) {
      x = (row == col) ? 1.f : 0.f;
    }
    S[j] = x;
  }
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) st_chunk(sm + OFF_S, mnmaj_chunk(row, half * 8 + cc, 16384), &S[cc * 8]);
  fence_proxy_async();  // the first MMA_a reads the initial state tile
  __syncthreads();

  {
    const uint8_t* wsrc = ar.wim + bh * ar.NC * (int64_t)kImg;
    const uint8_t* usrc = ar.uim + bh * ar.NC * (int64_t)kImg;
    const uint8_t* psrc = ar.pim + bh * ar.NC * (int64_t)kImgP;
    const float* gsrc = ar.gl + bh * ar.NC * 64;
    const float* rsrc = ar.rqk + (b * ar.Hqk + hq) * ar.NC * 128;
    // ---- load issue (tid 0 only)
    auto issue_x = [&](int64_t c, uint64_t* bar, uint32_t xa, uint32_t gbuf) {
      // apply: W, Q, K, G, rq, rk; otherwise W only
      mbar_arrive_expect_tx(bar, kApply ? 3 * kImg + 768 : kImg);
      for (int a = 0; a < 2; ++a) {
        bulk_load(sm + xa + a * XSTR, wsrc + c * kImg + a * 8192, 8192, bar);
        if (kApply) {
          tma_load_4d(sm + xa + a * XSTR + 8192, &mq, a * 64, (int)hq, (int)(c * 64), (int)b, bar);
          tma_load_4d(sm + xa + a * XSTR + KOFF, &mk, a * 64, (int)hq, (int)(c * 64), (int)b, bar);
        }
      }
      if (kApply) {
        bulk_load(sm + gbuf, gsrc + c * 64, 256, bar);
        bulk_load(sm + gbuf + 256, rsrc + c * 128, 512, bar);
      }
    };
    auto issue_k = [&](int64_t c) {  // summary / states: K, G, rk
      mbar_arrive_expect_tx(bars + 1, kImg + 512);
      for (int a = 0; a < 2; ++a)
        tma_load_4d(sm + S_XA + a * XSTR + KOFF, &mk, a * 64, (int)hq, (int)(c * 64), (int)b, bars + 1);
      bulk_load(sm + S_G, gsrc + c * 64, 256, bars + 1);
      bulk_load(sm + S_G + 256, rsrc + c * 128 + 64, 256, bars + 1);
    };
    auto issue_u = [&](int64_t c) {
      mbar_arrive_expect_tx(bar_u, kImg);
      bulk_load(sm + OFF_U, usrc + c * kImg, kImg, bar_u);
    };
    auto issue_p = [&](int64_t c) {
      mbar_arrive_expect_tx(bars + 3, kImgP);
      bulk_load(sm + A_PZ + 8192, psrc + c * kImgP, kImgP, bars + 3);
    };
    if (tid == 0 && cs < ce) {
      if (kApply) {
        issue_x(cs, bars + 0, A_XA, A_G);
        pend |= 1u;
        if (cs + 1 < ce) {
          issue_x(cs + 1, bars + 1, A_XA + 49152, A_G + 768);
          pend |= 2u;
        }
        issue_u(cs);
        issue_p(cs);
        pend |= 4u | 8u;
      } else {
        issue_x(cs, bars + 0, S_XA, 0);
        issue_k(cs);
        pend |= 1u | 2u;
        if (needU) {
          issue_u(cs);
          pend |= 4u;
        }
      }
    }
    for (int64_t c = cs; c < ce; ++c) {
      const int64_t k = c - cs;
      const int64_t t0 = c * 64;
      const uint32_t par = (uint32_t)(k & 1);
      const uint32_t bi = kApply ? (uint32_t)(k & 1) : 0u;
      const uint32_t xa = kApply ? A_XA + bi * 49152 : S_XA;
      // per-chunk vectors: G, then (apply) rq, then rk
      const float* sGc = (const float*)(sm + (kApply ? A_G + bi * 768 : S_G));
      const float* sRk = sGc + (kApply ? 128 : 64);
      const uint32_t xpar = kApply ? (uint32_t)((k >> 1) & 1) : par;
      uint64_t* bar_x = bars + (kApply ? bi : 0);
      // ---- inputs of chunk c: W (and q, k, gates for apply) before MMA_a
      if (kApply || tid == 0) {
        if (!mbar_wait(bar_x, xpar, ar.status, kStatusTimeout)) *s_abort = 1;
        if (tid == 0) pend &= kApply ? ~(1u << bi) : ~1u;
      }
      // the loop's last barrier already ordered the state tile S(c) before MMA_a; the q
      // tile is used raw (its rows' factors gamma_i rq_i are applied to Q S in TMEM)
      // pull the tiles of the next loads into L2, from warp 2 while thread 0 issues this
      // chunk's products (each prefetch takes ~100 cycles to issue; warp 2 is idle until
      // the first product's epilogue)
      if (tid == 64) {
        if (!kApply && c + 1 < ce) {
          l2_prefetch(wsrc + (c + 1) * kImg, kImg);
          if (needU) l2_prefetch(usrc + (c + 1) * kImg, kImg);
          l2_prefetch_tile(&mk, 0, (int)hq, (int)((c + 1) * 64), (int)b);
          l2_prefetch_tile(&mk, 64, (int)hq, (int)((c + 1) * 64), (int)b);
          l2_prefetch(gsrc + (c + 1) * 64, 256);
          l2_prefetch(rsrc + (c + 1) * 128 + 64, 256);
        }
        if (kApply && c + 1 < ce) {
          l2_prefetch(usrc + (c + 1) * kImg, kImg);
          l2_prefetch(psrc + (c + 1) * kImgP, kImgP);
        }
        if (kApply && c + 2 < ce) {
          l2_prefetch(wsrc + (c + 2) * kImg, kImg);
          for (int a = 0; a < 2; ++a) {
            l2_prefetch_tile(&mq, a * 64, (int)hq, (int)((c + 2) * 64), (int)b);
            l2_prefetch_tile(&mk, a * 64, (int)hq, (int)((c + 2) * 64), (int)b);
          }
          l2_prefetch(gsrc + (c + 2) * 64, 256);
          l2_prefetch(rsrc + (c + 2) * 128, 512);
        }
      }
      // chunk-start state: the bf16 S tile image, as is (states; apply when asked to keep
      // them), stored by warp 2 so that thread 0 goes straight to the products
      const bool keep_s = MODE == CH_STATES || (kApply && ar.hc != nullptr);
      if (keep_s && tid == 64) {
        bulk_store(ar.hc + (bh * ar.NC + c) * (int64_t)(2 * kImg), sm + OFF_S, 2 * kImg);
        bulk_commit();
      }
      // ---- MMA_a: apply [W; Q] S -> tA (W S in rows 0..63); otherwise, feature-major,
      //      S^T W^T + U^T (-I) = -V'^T -> tA (M = 128 rows of dv, 64 token columns)
      if (tid == 0) {
        if (kApply) {
          const uint32_t id = idesc_bf16(128, 128, 0, 1);
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t at = ks >> 2, kk = ks & 3;
            mma_bf16(tA, (d16 + ((xa + at * XSTR + kk * 32) >> 4)),
                     (d16384 + ((OFF_S + ks * 2048) >> 4)), id, ks > 0);
          }
        } else {
          const uint32_t id = idesc_bf16(128, 64, 1, 0);
          for (int ks = 0; ks < 8; ++ks)  // K = dk
            mma_bf16(tA, (d16384 + ((OFF_S + ks * 2048) >> 4)),
                     (d16 + ((xa + (ks >> 2) * XSTR + (ks & 3) * 32) >> 4)), id, ks > 0);
          if (needU) {
            if (!mbar_wait(bar_u, par, ar.status, kStatusTimeout)) *s_abort = 1;
            pend &= ~4u;
            for (int ks = 0; ks < 4; ++ks)  // K = tokens
              mma_bf16(tA, (d8192 + ((OFF_U + ks * 2048) >> 4)), (d16 + ((S_NI + ks * 32) >> 4)),
                       id, 1);
          }
        }
        mma_commit(bar_mma);
        pend |= 16u;
      } else if (kApply && tid == 32) {
        mma_commit(bar_mma);  // nothing issued in this round: arrives at once
      }
      if (!kApply) {  // k tile, gates and rk of chunk c: first needed for V2 and MMA_b
        if (!mbar_wait(bars + 1, par, ar.status, kStatusTimeout)) *s_abort = 1;
        if (tid == 0) pend &= ~2u;
      }
      const float gC = exp2f(sGc[63]);
      // token row of V' owned by this thread: M = 128 (apply: quadrants 0, 1) or M = 64
      // accumulator layout (row r in TMEM lane (r % 16) + 32 (r / 16): lanes 0..15)
      const int vi = row;  // apply: token row of V' (quadrants 0, 1 of the M = 128 result)
      const float kt = exp2f(sGc[63] - sGc[vi & 63]) * sRk[vi & 63];
      if (kApply && quad < 2) {
        if (!mbar_wait(bar_u, par, ar.status, kStatusTimeout)) *s_abort = 1;
        if (tid == 0) pend &= ~4u;
      }
      if (!mbar_wait(bar_mma, 0, ar.status, kStatusTimeout)) *s_abort = 1;
      if (tid == 0) pend &= ~16u;
      tc_fence_after();
      if (!kApply && tid == 0 && c + 1 < ce) {  // W(c) consumed
        issue_x(c + 1, bars + 0, S_XA, 0);
        pend |= 1u;
      }
      if (!kApply) {  // V2^T = -rk e^{G_C - G} tA: thread row `row` (dv), tokens 32 half + e
        float v[32];
        tmem_ld32(tA + lane_off + half * 32, v);
        const int tl = half * 32 + lane;
        const float ktr = exp2f(sGc[63] - sGc[tl]) * sRk[tl];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] *= -__shfl_sync(0xffffffffu, ktr, e);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) st_chunk(sm + S_V2, kmaj_chunk(row, half * 4 + cc), &v[cc * 8]);
      } else if (quad < 2) {  // V' = U - W S, V2 = rk e^{G_C - G} V'
        const int i = vi;
        const bool own = true;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[32];
          tmem_ld32(tA + lane_off + half * 64 + hh * 32, v);
          if (!own) continue;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int chn = half * 8 + hh * 4 + cc;
            float u[8];
            if (needU) {
              ld_chunk(sm + OFF_U, img_chunk(i, chn), u);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) u[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) u[e] -= v[cc * 8 + e];
            if (kApply) st_chunk(sm + A_VP, mnmaj_chunk(i, chn, 8192), u);
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = kt * u[e];
            st_chunk(sm + OFF_V2, mnmaj_chunk(i, chn, 8192), x);
          }
        }
      }
      if (kApply && quad >= 2) {  // Q S (rows 64..127 of tA) times gamma_i rq_i, in place,
        // while quadrants 0, 1 form V'; MMA_c then adds P V' to the scaled rows
        const int i = row - 64;
        const float f = exp2f(sGc[i]) * sGc[64 + i];
        float v0[32], v1[32];
        tmem_ld32x2(tA + lane_off + half * 64, v0, tA + lane_off + half * 64 + 32, v1);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          v0[e] *= f;
          v1[e] *= f;
        }
        tmem_st32x2(tA + lane_off + half * 64, v0, tA + lane_off + half * 64 + 32, v1);
      }
      // the S tile (states) and the previous O tile (apply) are rewritten below
      if ((kApply && tid == 0) || (keep_s && tid == 64)) bulk_wait_read();
      CHAIN_SYNC();
      // ---- MMA_b: K^T V2 -> tB; apply: MMA_c: [0; P] V' accumulated into tA rows 64..127
      if (tid == 64 && needU && c + 1 < ce) issue_u(c + 1);  // U(c) consumed; off thread 0
      if (tid == 0) {
        if (needU && c + 1 < ce) pend |= 4u;  // (issued by warp 2)
        const uint32_t id = idesc_bf16(128, 128, 1, kApply ? 1 : 0);  // B: V2 (apply) or V2^T
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tB, (dxs + ((xa + KOFF + ks * 2048) >> 4)),
                   kApply ? (d8192 + ((OFF_V2 + ks * 2048) >> 4)) : (d16 + ((S_V2 + ks * 32) >> 4)),
                   id, ks > 0);
        mma_commit(bar_mma);
        pend |= 16u;
      } else if (kApply && tid == 32) {  // MMA_c into tA, in parallel with MMA_b
        if (!mbar_wait(bars + 3, par, ar.status, kStatusTimeout)) *s_abort = 1;
        const uint32_t id2 = idesc_bf16(128, 128, 0, 1);
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tA, (d16 + ((A_PZ + ks * 32) >> 4)), (d8192 + ((A_VP + ks * 2048) >> 4)), id2,
                   1);
        mma_commit(bar_mma);
      }
      if (!mbar_wait(bar_mma, 1, ar.status, kStatusTimeout)) *s_abort = 1;
      if (tid == 0) pend &= kApply ? ~(16u | 8u) : ~16u;  // (P consumed by tid 32's products)
      tc_fence_after();
      if (c + 1 < ce) {
        if (kApply) {  // copies from warp 4; thread 0 keeps the drain record
          if (tid == 128) {
            issue_p(c + 1);  // P(c) consumed by MMA_c
            if (c + 2 < ce) issue_x(c + 2, bars + bi, xa, A_G + bi * 768);  // buffer bi free
          }
          if (tid == 0) pend |= 8u | (c + 2 < ce ? 1u << bi : 0u);
        } else if (tid == 0) {
          issue_k(c + 1);  // K(c) consumed by MMA_b; G(c), rk(c) already read
          pend |= 2u;
        }
      }
      {  // S <- gamma_C S + K^T V2
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[32];
          tmem_ld32(tB + lane_off + half * 64 + hh * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) S[hh * 32 + e] = fmaf(gC, S[hh * 32 + e], v[e]);
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          st_chunk(sm + OFF_S, mnmaj_chunk(row, half * 8 + cc, 16384), &S[cc * 8]);
      }
      if (kApply && quad >= 2) {  // O = gamma Q S + P V' (rows 64..127 of tA) -> staging tile
        const int i = row - 64;
        const int64_t t = t0 + i;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[32];
          tmem_ld32(tA + lane_off + half * 64 + hh * 32, v);
          if (t >= L) {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0.f;
          }
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            st_chunk(sm + A_O + half * 8192, kmaj_chunk(i, hh * 4 + cc), &v[cc * 8]);
        }
      }
      CHAIN_SYNC();
      if (kApply && tid == 0) {  // tokens past T are clipped by the tensor map
        tma_store_4d(&mo, sm + A_O, 0, (int)h, (int)t0, (int)b);
        tma_store_4d(&mo, sm + A_O + 8192, 64, (int)h, (int)t0, (int)b);
        bulk_commit();
      }
    }
  }
  {  // ---- final state
    float* dst = nullptr;
    if (kApply) {
      if (seg == ar.P - 1) dst = ar.final_out;
    } else if (MODE == CH_SUM) {
      dst = mpart ? ar.M_out : ar.S_out;
      if (dst) dst += seg * ar.out_seg_stride;
    }
    if (dst) {
      float4* d4 = reinterpret_cast<float4*>(dst + (bh * 128 + row) * 128 + half * 64);
#pragma unroll
      for (int j = 0; j < 16; ++j) d4[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
    }
  }
done:
  if (tid == 0 || tid == 64) bulk_wait_all();  // stores read shared memory until they complete
  if (tid == 0 && pend) {  // abort: let every copy and MMA still in flight finish first
    for (int i = 0; i < 5; ++i)
      if (pend & (1u << i)) {
        // one of the two parities is the phase in flight; the other returns at once
        mbar_wait(bars + i, 0, nullptr, 0);
        mbar_wait(bars + i, 1, nullptr, 0);
      }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ============================================================================
// k_dchain_tc: the reverse chain of the backward, grid (1, H, B * nseg), 256
// threads, chunks of one segment walked from the last to the first.  With dS
// the gradient of the state at the end of a chunk:
//
//   dV' = P^T dO + diag(rk e^{G_C - G}) K dS
//   dS <- gamma_C dS + (diag(gamma rq) Q)^T dO - W^T dV'
//
// mode 0 stores every chunk's dS (bf16) and the start gradient of segment 0;
// mode 1 starts from dS = 0 and returns the segment's gradient summary D (the
// reverse-direction state-gradient pass of "linear attention cp #1035").
// ============================================================================
constexpr uint32_t D_XA = 0;        // atoms a at a*16384: [K_a | Q_a] (q rows scaled in place)
constexpr uint32_t D_W = 32768;     // W image
constexpr uint32_t D_P = 49152;     // P image (8 KB)
constexpr uint32_t D_DO = 57344;    // dO tile [tok][dv]; later -dV'^T [dv][tok] (K-major)
constexpr uint32_t D_DS = 73728;    // dS, bf16, MN-major (halves 16 KB apart)
constexpr uint32_t D_G = 106496;    // G, rq, rk of the chunk (64 floats each)
constexpr uint32_t D_SC = 107264;   // barriers
constexpr uint32_t D_SMEM = D_SC + 128 + 1024;

struct DchainArgs {
  int64_t T, Ts, H, Hqk, r, NC, CPS;
  const float* rqk;
  const uint8_t* wim;
  const uint8_t* pim;
  const float* gl;
  const int32_t* valid_len;
  const float* init;          // mode 0: gradient at the end of each segment
  int64_t init_seg_stride;
  uint8_t* dhc;               // mode 0: chunk-end state gradients, [B][H][NC] 32 KB tile images
  float* start_out;           // mode 0: gradient at the start of segment 0
  float* D_out;               // mode 1: gradient summaries
  int64_t out_seg_stride;
  int* status;
  int mode, seg_first, nseg;
};

// One CTA of the reverse chain: head h, zi = row * nseg + segment.
__device__ __forceinline__ void dchain_cta(const CUtensorMap& mq, const CUtensorMap& mk,
                                           const CUtensorMap& mdo, const DchainArgs& ar,
                                           int64_t h, int64_t zi) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t base = smem_u32(sm);
  // operand descriptors: base descriptor + byte offset / 16 (the start address field)
  const uint64_t d16 = sdesc(base, 16, 1024), d8192 = sdesc(base, 8192, 1024),
                 d16384 = sdesc(base, 16384, 1024);
  uint64_t* bars = (uint64_t*)(sm + D_SC);  // a: K, Q, P, G/rq/rk; b: W, dO; mma; Qg^T dO
  uint64_t* bar_a = bars, *bar_b = bars + 1, *bar_mma = bars + 2, *bar_q = bars + 3;
  uint32_t* s_tmem = (uint32_t*)(bars + 4);
  int* s_abort = (int*)(s_tmem + 1);
  const float* sG = (const float*)(sm + D_G);
  const float* sRq = sG + 64;
  const float* sRk = sG + 128;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int row = quad * 32 + lane;
  const bool store = ar.mode == 0;
  const int64_t b = zi / ar.nseg;
  const int seg = ar.seg_first + (int)(zi % ar.nseg);
  const int64_t hq = h / ar.r, bh = b * ar.H + h;
  const int64_t cs = (int64_t)seg * ar.CPS;
  const int64_t L = clamp_len(ar.valid_len, b, ar.T, ar.status, false);
  // chunks of padding only pass the state gradient through unchanged: not walked
  const int64_t ce = min(cs + ar.CPS < ar.NC ? cs + ar.CPS : ar.NC, (L + 63) / 64);
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  uint32_t pend = 0;

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(bars + i, 1);
    fence_barrier_init();
    *s_abort = 0;
  }
  if (warp == 0) tmem_alloc(s_tmem, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tV = tmem, tV2 = tmem + 64, tS = tmem + 128;

  float dS[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    const int col = half * 64 + j;
    dS[j] = (store && ar.init) ? ar.init[seg * ar.init_seg_stride + (bh * 128 + row) * 128 + col] : 0.f;
  }
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) st_chunk(sm + D_DS, mnmaj_chunk(row, half * 8 + cc, 16384), &dS[cc * 8]);
  fence_proxy_async();  // the first round 1a reads the initial dS tile
  __syncthreads();

  {
    const uint8_t* wsrc = ar.wim + bh * ar.NC * (int64_t)kImg;
    const uint8_t* psrc = ar.pim + bh * ar.NC * (int64_t)kImgP;
    const float* gsrc = ar.gl + bh * ar.NC * 64;
    const float* rsrc = ar.rqk + (b * ar.Hqk + hq) * ar.NC * 128;
    auto issue_a = [&](int64_t c) {
      mbar_arrive_expect_tx(bar_a, 2 * kImg + kImgP + 768);
      for (int a = 0; a < 2; ++a) {
        tma_load_4d(sm + D_XA + a * 16384, &mk, a * 64, (int)hq, (int)(c * 64), (int)b, bar_a);
        tma_load_4d(sm + D_XA + a * 16384 + 8192, &mq, a * 64, (int)hq, (int)(c * 64), (int)b, bar_a);
      }
      bulk_load(sm + D_P, psrc + c * kImgP, kImgP, bar_a);
      bulk_load(sm + D_G, gsrc + c * 64, 256, bar_a);
      bulk_load(sm + D_G + 256, rsrc + c * 128, 512, bar_a);
    };
    auto issue_b = [&](int64_t c) {
      mbar_arrive_expect_tx(bar_b, 2 * kImg);
      bulk_load(sm + D_W, wsrc + c * kImg, kImg, bar_b);
      for (int a = 0; a < 2; ++a)
        tma_load_4d(sm + D_DO + a * 8192, &mdo, a * 64, (int)h, (int)(c * 64), (int)b, bar_b);
    };
    if (tid == 0 && cs < ce) {
      issue_a(ce - 1);
      issue_b(ce - 1);
      pend |= 3u;
    }
    for (int64_t c = ce - 1; c >= cs; --c) {
      const int64_t k = ce - 1 - c;
      const int64_t t0 = c * 64;
      const uint32_t par = (uint32_t)(k & 1);
      if (tid == 160 && c - 1 >= cs) {  // pull the tiles of chunk c-1 into L2 (warp 5)
        const int tp = (int)((c - 1) * 64);
        for (int a = 0; a < 2; ++a) {
          l2_prefetch_tile(&mk, a * 64, (int)hq, tp, (int)b);
          l2_prefetch_tile(&mq, a * 64, (int)hq, tp, (int)b);
          l2_prefetch_tile(&mdo, a * 64, (int)h, tp, (int)b);
        }
        l2_prefetch(psrc + (c - 1) * kImgP, kImgP);
        l2_prefetch(wsrc + (c - 1) * kImg, kImg);
        l2_prefetch(gsrc + (c - 1) * 64, 256);
        l2_prefetch(rsrc + (c - 1) * 128, 512);
      }
      if (!mbar_wait(bar_a, par, ar.status, kStatusTimeout)) *s_abort = 1;
      if (!mbar_wait(bar_b, par, ar.status, kStatusTimeout)) *s_abort = 1;
      if (tid == 0) pend &= ~3u;
      // k is used raw (its rows' factors rk e^{G_C - G} scale the token columns of dS^T K^T
      // in the epilogue); q rows are scaled by gamma rq while round 1a runs
      const float gC = exp2f(sG[63]);
      const int tl = half * 32 + lane;  // this lane's token column of the epilogue
      const float ktr = exp2f(sG[63] - sG[tl]) * sRk[tl];
      if (t0 + 64 > L) {  // zero dO rows past valid_len (a CTA-uniform branch)
        for (int e = tid; e < 1024; e += CT) {
          const int i = e >> 4, cc = e & 15;
          if (t0 + i >= L)
            *reinterpret_cast<uint4*>(sm + D_DO + mnmaj_chunk(i, cc, 8192)) = make_uint4(0, 0, 0, 0);
        }
        CHAIN_SYNC();
      }
      if (store && tid == 64) {  // gradient of chunk c's end state: the bf16 dS tile image, as is
        // (warp 2: thread 0 goes straight to the products)
        bulk_store(ar.dhc + (bh * ar.NC + c) * (int64_t)(2 * kImg), sm + D_DS, 2 * kImg);
        bulk_commit();
      }
      // ---- round 1a: dO^T P -> tV, dS^T K^T -> tV2 (feature-major: M = 128 rows of dv,
      //      64 token columns; the previous step's last barrier ordered dS)
      if (tid == 0) {
        const uint32_t idv = idesc_bf16(128, 64, 1, 1);
        for (int ks = 0; ks < 4; ++ks)  // K = tokens i
          mma_bf16(tV, (d8192 + ((D_DO + ks * 2048) >> 4)), (d8192 + ((D_P + ks * 2048) >> 4)),
                   idv, ks > 0);
        const uint32_t idk = idesc_bf16(128, 64, 1, 0);
        for (int ks = 0; ks < 8; ++ks)  // K = dk
          mma_bf16(tV2, (d16384 + ((D_DS + ks * 2048) >> 4)),
                   (d16 + ((D_XA + (ks >> 2) * 16384 + (ks & 3) * 32) >> 4)), idk, ks > 0);
        mma_commit(bar_mma);
        pend |= 4u;
      }
      for (int e = tid; e < 1024; e += CT) {  // Qg = diag(gamma rq) Q, in place
        const int r = e >> 4, at = (e >> 3) & 1, p = e & 7;
        scale_chunk(sm, D_XA + at * 16384 + 8192 + r * 128 + p * 16, exp2f(sG[r]) * sRq[r]);
      }
      CHAIN_SYNC();
      // ---- round 1b: Qg^T dO -> tS
      if (tid == 0) {
        const uint32_t idmm = idesc_bf16(128, 128, 1, 1);
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tS, (d16384 + ((D_XA + 8192 + ks * 2048) >> 4)),
                   (d8192 + ((D_DO + ks * 2048) >> 4)), idmm, ks > 0);
        mma_commit(bar_q);
        pend |= 8u;
      }
      if (!mbar_wait(bar_mma, 0, ar.status, kStatusTimeout)) *s_abort = 1;
      if (tid == 0) pend &= ~4u;
      tc_fence_after();
      {  // -dV'^T = -(tV + tV2 diag(rk e^{G_C - G})): thread row `row` (dv), tokens 32 half + e,
        // stored K-major over the dO tile once round 1b has read it
        // (16 columns at a time: the 64 dS registers stay live)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[16], w[16];
          tmem_ld16x2(tV + lane_off + half * 32 + hh * 16, tV2 + lane_off + half * 32 + hh * 16, v, w);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            v[e] = -fmaf(__shfl_sync(0xffffffffu, ktr, hh * 16 + e), w[e], v[e]);
          if (hh == 0) {
            if (!mbar_wait(bar_q, par, ar.status, kStatusTimeout)) *s_abort = 1;
            if (tid == 0) pend &= ~8u;
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
            st_chunk(sm + D_DO, kmaj_chunk(row, half * 4 + hh * 2 + cc), &v[cc * 8]);
        }
      }
      if (store && tid == 64) bulk_wait_read();  // the dS tile is rewritten below
      CHAIN_SYNC();
      // ---- tS += W^T (-dV')  (B from the K-major -dV'^T tile)
      if (tid == 0) {
        const uint32_t id = idesc_bf16(128, 128, 1, 0);
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tS, (d8192 + ((D_W + ks * 2048) >> 4)), (d16 + ((D_DO + ks * 32) >> 4)), id,
                   1);
        mma_commit(bar_mma);
        pend |= 4u;
        if (c - 1 >= cs) pend |= 1u;  // (issued by warp 3)
      } else if (tid == 96 && c - 1 >= cs) {  // K, Q, P of chunk c consumed by rounds 1a, 1b;
        issue_a(c - 1);                        // gates read above
      }
      if (!mbar_wait(bar_mma, 1, ar.status, kStatusTimeout)) *s_abort = 1;
      if (tid == 0) pend &= ~4u;
      tc_fence_after();
      if (c - 1 >= cs) {  // W and the dO / -dV' tile consumed: warp 4 copies, thread 0 records
        if (tid == 128) issue_b(c - 1);
        if (tid == 0) pend |= 2u;
      }
      {  // dS <- gamma_C dS + tS
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[32];
          tmem_ld32(tS + lane_off + half * 64 + hh * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) dS[hh * 32 + e] = fmaf(gC, dS[hh * 32 + e], v[e]);
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          st_chunk(sm + D_DS, mnmaj_chunk(row, half * 8 + cc, 16384), &dS[cc * 8]);
      }
      CHAIN_SYNC();
    }
  }
  {
    float* dst = nullptr;
    if (store) {
      if (seg == 0) dst = ar.start_out;
    } else if (ar.D_out) {
      dst = ar.D_out + seg * ar.out_seg_stride;
    }
    if (dst) {
      float4* d4 = reinterpret_cast<float4*>(dst + (bh * 128 + row) * 128 + half * 64);
#pragma unroll
      for (int j = 0; j < 16; ++j) d4[j] = make_float4(dS[4 * j], dS[4 * j + 1], dS[4 * j + 2], dS[4 * j + 3]);
    }
  }
done:
  if (tid == 64) bulk_wait_all();
  if (tid == 0 && pend) {
    for (int i = 0; i < 4; ++i)
      if (pend & (1u << i)) {
        mbar_wait(bars + i, 0, nullptr, 0);
        mbar_wait(bars + i, 1, nullptr, 0);
      }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

template <int MODE>
__global__ void __launch_bounds__(CT, MODE == CH_APPLY ? 1 : 2)
    k_chain_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mo, ChainArgs ar) {
  chain_cta<MODE>(mq, mk, mo, ar, (int)blockIdx.x, blockIdx.y, blockIdx.z);
}

__global__ void __launch_bounds__(CT, 2)
    k_dchain_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                const __grid_constant__ CUtensorMap mdo, DchainArgs ar) {
  dchain_cta(mq, mk, mdo, ar, blockIdx.y, blockIdx.z);
}

// A forward chain pass and an independent reverse chain pass in one launch, so that
// the CTAs of both fill the GPU together: z in [0, nf) runs the forward chain (with
// `parts` parts per segment folded into z), z in [nf, nf + nr) the reverse chain.
template <int MODE>
__global__ void __launch_bounds__(CT, 2)
    k_chain_pair_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mo, const __grid_constant__ CUtensorMap mdo,
                    ChainArgs fa, DchainArgs ra, int parts, int64_t nf) {
  const int64_t z = blockIdx.z;
  if (z < nf)
    chain_cta<MODE>(mq, mk, mo, fa, (int)(z % parts), blockIdx.y, z / parts);
  else
    dchain_cta(mq, mk, mdo, ra, blockIdx.y, z - nf);
}

template <typename K>
cudaError_t smem_attr(K kern, uint32_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_prep_tc(const Prob& pr, const Inputs& in, const WS& ws, cudaStream_t st) {
  if (pr.B == 0 || pr.NC == 0) return cudaSuccess;
  const ConvIn* cv = in.conv;  // set: the tiles come from the Conv1D inputs
  CUtensorMap mq, mk, mv, mlq, mlk, mlv;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  if (!tc_make_map(&mq, cv ? cv->x[0] : in.q, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(&mk, cv ? cv->x[1] : in.k, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(&mv, cv ? cv->x[2] : in.v, pr.B, pr.T, pr.Ts, pr.H))
    return cudaErrorInvalidValue;
  if (cv) {
    memset(&mlq, 0, sizeof(mlq));
    memset(&mlk, 0, sizeof(mlk));
    memset(&mlv, 0, sizeof(mlv));
    if (!tc_make_map_rows(&mlq, cv->x[0], pr.B, pr.T, pr.Ts, pr.Hqk, 3) ||
        !tc_make_map_rows(&mlk, cv->x[1], pr.B, pr.T, pr.Ts, pr.Hqk, 3) ||
        !tc_make_map_rows(&mlv, cv->x[2], pr.B, pr.T, pr.Ts, pr.H, 3))
      return cudaErrorInvalidValue;
  } else {
    mlq = mq;  // (not read)
    mlk = mk;
    mlv = mv;
  }
  PrepArgs ar;
  ar.T = pr.T; ar.Ts = pr.Ts; ar.H = pr.H; ar.Hqk = pr.Hqk; ar.r = pr.r; ar.NC = pr.NC;
  ar.l2norm = pr.l2norm; ar.eps = pr.eps; ar.scale = pr.scale;
  ar.a = (const __nv_bfloat16*)in.a; ar.b = (const __nv_bfloat16*)in.b;
  ar.A_log = in.A_log; ar.dt_bias = in.dt_bias; ar.valid_len = in.valid_len;
  ar.rqk = ws.rqk; ar.wim = (uint8_t*)ws.wim; ar.uim = (uint8_t*)ws.uim;
  ar.pim = (uint8_t*)ws.pim; ar.tim = (uint8_t*)ws.tim; ar.gl = ws.gl;
  ar.status = ws.status;
  ar.NW = pr.B * pr.H * pr.NC;
  ar.convK = cv ? cv->K : 0;
  for (int i = 0; i < 3; ++i) {
    ar.cw[i] = cv ? cv->w[i] : nullptr;
    ar.cb[i] = cv ? cv->bias[i] : nullptr;
    ar.chalo[i] = cv ? (const __nv_bfloat16*)cv->halo[i] : nullptr;
    ar.cy[i] = cv ? (__nv_bfloat16*)cv->y[i] : nullptr;
  }
  if (ar.NW + 1024 >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;  // 32-bit chunk indices
  const int64_t nblk = ar.NW < 2 * (int64_t)device_sms() ? ar.NW : 2 * (int64_t)device_sms();
  cudaError_t e;
  if (cv) {
    if ((e = smem_attr(k_prep_tc<true>, P_SMEM_CONV)) != cudaSuccess) return e;
    k_prep_tc<true><<<(unsigned)nblk, PT, P_SMEM_CONV, st>>>(mq, mk, mv, mlq, mlk, mlv, ar);
  } else {
    if ((e = smem_attr(k_prep_tc<false>, P_SMEM)) != cudaSuccess) return e;
    k_prep_tc<false><<<(unsigned)nblk, PT, P_SMEM, st>>>(mq, mk, mv, mlq, mlk, mlv, ar);
  }  // two CTAs per SM, persistent
  return cudaGetLastError();
}

namespace {

// Tensor maps and arguments of a forward chain pass.
bool chain_setup(const Prob& pr, const Inputs& in, const WS& ws, int seg_first, int nseg,
                 const float* init, int64_t init_seg_stride, void* o, float* final_out,
                 float* M_out, float* S_out, int64_t out_seg_stride, void* hc, CUtensorMap* mq,
                 CUtensorMap* mk, CUtensorMap* mo, ChainArgs* ar) {
  memset(mq, 0, sizeof(*mq));
  memset(mk, 0, sizeof(*mk));
  memset(mo, 0, sizeof(*mo));
  const void* qptr = in.q ? in.q : in.k;  // summaries and states never read q
  const void* optr = o ? o : in.k;        // only apply writes o
  if (!tc_make_map(mq, qptr, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(mk, in.k, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(mo, optr, pr.B, pr.T, pr.Ts, o ? pr.H : pr.Hqk))
    return false;
  ar->T = pr.T; ar->Ts = pr.Ts; ar->H = pr.H; ar->Hqk = pr.Hqk; ar->r = pr.r; ar->NC = pr.NC;
  ar->CPS = pr.CPS; ar->P = pr.P;
  ar->rqk = ws.rqk;
  ar->wim = (const uint8_t*)ws.wim; ar->uim = (const uint8_t*)ws.uim;
  ar->pim = (const uint8_t*)ws.pim; ar->gl = ws.gl;
  ar->valid_len = in.valid_len;
  ar->init = init; ar->init_seg_stride = init_seg_stride;
  ar->o = (__nv_bfloat16*)o; ar->final_out = final_out;
  ar->M_out = M_out; ar->S_out = S_out; ar->out_seg_stride = out_seg_stride;
  ar->hc = (uint8_t*)hc;
  ar->status = ws.status;
  ar->seg_first = seg_first; ar->nseg = nseg;
  return true;
}

// Tensor maps and arguments of a reverse chain pass.
bool dchain_setup(const Prob& pr, const Inputs& in, const WS& ws, int mode, int seg_first,
                  int nseg, const float* init, int64_t init_seg_stride, void* dhc,
                  float* start_out, float* D_out, int64_t out_seg_stride, CUtensorMap* mq,
                  CUtensorMap* mk, CUtensorMap* mdo, DchainArgs* ar) {
  memset(mq, 0, sizeof(*mq));
  memset(mk, 0, sizeof(*mk));
  memset(mdo, 0, sizeof(*mdo));
  if (!tc_make_map(mq, in.q, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(mk, in.k, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(mdo, in.dO, pr.B, pr.T, pr.Ts, pr.H))
    return false;
  ar->T = pr.T; ar->Ts = pr.Ts; ar->H = pr.H; ar->Hqk = pr.Hqk; ar->r = pr.r; ar->NC = pr.NC;
  ar->CPS = pr.CPS;
  ar->rqk = ws.rqk; ar->wim = (const uint8_t*)ws.wim; ar->pim = (const uint8_t*)ws.pim;
  ar->gl = ws.gl; ar->valid_len = in.valid_len;
  ar->init = init; ar->init_seg_stride = init_seg_stride;
  ar->dhc = (uint8_t*)dhc; ar->start_out = start_out; ar->D_out = D_out;
  ar->out_seg_stride = out_seg_stride; ar->status = ws.status;
  ar->mode = mode; ar->seg_first = seg_first; ar->nseg = nseg;
  return true;
}

}  // namespace

cudaError_t launch_chain_tc(const Prob& pr, const Inputs& in, const WS& ws, int mode,
                            int seg_first, int nseg, const float* init, int64_t init_seg_stride,
                            void* o, float* final_out, float* M_out, float* S_out,
                            int64_t out_seg_stride, void* hc, cudaStream_t st) {
  if (nseg <= 0 || pr.B == 0 || pr.NC == 0) return cudaSuccess;
  CUtensorMap mq, mk, mo;
  ChainArgs ar;
  if (!chain_setup(pr, in, ws, seg_first, nseg, init, init_seg_stride, o, final_out, M_out, S_out,
                   out_seg_stride, hc, &mq, &mk, &mo, &ar))
    return cudaErrorInvalidValue;
  cudaError_t e;
  dim3 grid(mode == CH_SUM ? 2 : 1, (unsigned)pr.H, (unsigned)(pr.B * nseg));
  if (mode == CH_APPLY) {
    if ((e = smem_attr(k_chain_tc<CH_APPLY>, A_SMEM)) != cudaSuccess) return e;
    k_chain_tc<CH_APPLY><<<grid, CT, A_SMEM, st>>>(mq, mk, mo, ar);
  } else if (mode == CH_SUM) {
    if ((e = smem_attr(k_chain_tc<CH_SUM>, S_SMEM)) != cudaSuccess) return e;
    k_chain_tc<CH_SUM><<<grid, CT, S_SMEM, st>>>(mq, mk, mo, ar);
  } else {
    if ((e = smem_attr(k_chain_tc<CH_STATES>, S_SMEM)) != cudaSuccess) return e;
    k_chain_tc<CH_STATES><<<grid, CT, S_SMEM, st>>>(mq, mk, mo, ar);
  }
  return cudaGetLastError();
}

cudaError_t launch_dchain_tc(const Prob& pr, const Inputs& in, const WS& ws, int mode,
                             int seg_first, int nseg, const float* init, int64_t init_seg_stride,
                             void* dhc, float* start_out, float* D_out, int64_t out_seg_stride,
                             cudaStream_t st) {
  if (nseg <= 0 || pr.B == 0 || pr.NC == 0) return cudaSuccess;
  CUtensorMap mq, mk, mdo;
  DchainArgs ar;
  if (!dchain_setup(pr, in, ws, mode, seg_first, nseg, init, init_seg_stride, dhc, start_out,
                    D_out, out_seg_stride, &mq, &mk, &mdo, &ar))
    return cudaErrorInvalidValue;
  cudaError_t e = smem_attr(k_dchain_tc, D_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(1, (unsigned)pr.H, (unsigned)(pr.B * nseg));
  k_dchain_tc<<<grid, CT, D_SMEM, st>>>(mq, mk, mdo, ar);
  return cudaGetLastError();
}

cudaError_t launch_chain_pair_tc(const Prob& pr, const Inputs& in, const WS& ws, int fmode,
                                 const ChainPass& f, int rmode, const ReversePass& r,
                                 cudaStream_t st) {
  if (f.nseg <= 0) return launch_dchain_tc(pr, in, ws, rmode, r.seg_first, r.nseg, r.init,
                                           r.init_seg_stride, r.dhc, r.start_out, r.D_out,
                                           r.out_seg_stride, st);
  if (r.nseg <= 0) return launch_chain_tc(pr, in, ws, fmode, f.seg_first, f.nseg, f.init,
                                          f.init_seg_stride, nullptr, nullptr, f.M_out, f.S_out,
                                          f.out_seg_stride, f.hc, st);
  if (pr.B == 0 || pr.NC == 0) return cudaSuccess;
  CUtensorMap mq, mk, mo, mq2, mk2, mdo;
  ChainArgs fa;
  DchainArgs ra;
  if (!chain_setup(pr, in, ws, f.seg_first, f.nseg, f.init, f.init_seg_stride, nullptr, nullptr,
                   f.M_out, f.S_out, f.out_seg_stride, f.hc, &mq, &mk, &mo, &fa) ||
      !dchain_setup(pr, in, ws, rmode, r.seg_first, r.nseg, r.init, r.init_seg_stride, r.dhc,
                    r.start_out, r.D_out, r.out_seg_stride, &mq2, &mk2, &mdo, &ra))
    return cudaErrorInvalidValue;
  const int parts = fmode == CH_SUM ? 2 : 1;
  const int64_t nf = (int64_t)parts * pr.B * f.nseg, nr = pr.B * (int64_t)r.nseg;
  const uint32_t smem = S_SMEM > D_SMEM ? S_SMEM : D_SMEM;
  dim3 grid(1, (unsigned)pr.H, (unsigned)(nf + nr));
  cudaError_t e;
  if (fmode == CH_SUM) {
    if ((e = smem_attr(k_chain_pair_tc<CH_SUM>, smem)) != cudaSuccess) return e;
    k_chain_pair_tc<CH_SUM><<<grid, CT, smem, st>>>(mq, mk, mo, mdo, fa, ra, parts, nf);
  } else {
    if ((e = smem_attr(k_chain_pair_tc<CH_STATES>, smem)) != cudaSuccess) return e;
    k_chain_pair_tc<CH_STATES><<<grid, CT, smem, st>>>(mq, mk, mo, mdo, fa, ra, parts, nf);
  }
  return cudaGetLastError();
}

}  // namespace gdn
