// gdn_conv.cu -- causal depthwise Conv1D + SiLU over time, forward and backward, with
// the left halo of a segment ("linear attention cp #1035", section "What does this PR
// do": the depthwise Conv1D that feeds the Gated DeltaNet; in "p2p" mode a rank
// receives only the left halo the Conv1D needs from its neighbour and sends back its
// gradient).  For row b, channel c, x~ = the row preceded by the K - 1 halo tokens:
//   a[t] = bias + sum_{i<K} w[i] x~[t - (K-1) + i],  y[t] = a[t] sigmoid(a[t])
//   ds[t] = dy[t] sigmoid(a) (1 + a (1 - sigmoid(a)))
//   dx~[s] = sum_i w[i] ds[s + (K-1) - i],  dw[i] = sum_{b,t} ds[t] x~[t-(K-1)+i],
//   dbias = sum_{b,t} ds[t]
//
// Bandwidth-bound: every element of x (and dy) is read once from HBM and every output
// written once.  A CTA takes 128 channels of a tile of tokens and first copies the rows it
// reads into shared memory with 16-byte cp.async copies (all of them in flight at once;
// halo rows from the halo, rows outside the row's tokens zero-filled), then computes from
// there: a thread owns 4 adjacent channels and walks a run of the tile's tokens with the
// last K - 1 inputs (and, backward, the last K - 1 ds) in registers, storing each output
// straight to global memory.  The backward's walk is unrolled over its run, with the
// bounds checks compiled out for the tiles that need none, and does its arithmetic on
// channel pairs with packed f32x2 operations; it recomputes a and ds of the K - 1 tokens
// after each run to form their dx.  dw and dbias: per-CTA partials (the
// CTA's 8 runs summed in a fixed order) in the workspace, then one pass that sums the
// partials of every tile in a fixed order (fp64).
#include <cuda_bf16.h>
#include <string.h>

#include <type_traits>

#include "gdn.h"
#include "gdn_vec.cuh"

namespace gdn {
namespace {

using namespace vec;

constexpr int CONV_NT = 256;  // threads: 32 channel quads x 8 token runs
constexpr int CONV_CH = 128;  // channels per CTA
// tokens per CTA: forward 256 (bf16) / 128 (fp32), backward half that, so that a CTA's
// staged rows take ~66 KB.  Forward: three CTAs per SM (shared memory; 62 registers at
// K = 4).  Backward: two CTAs per SM (100 registers at K = 4)
template <typename T>
struct Tile {
  static constexpr int ROWB = CONV_CH * (int)sizeof(T);  // bytes of one staged token row
  static constexpr int TOKF = 512 / (int)sizeof(T);
  static constexpr int TOKB = 256 / (int)sizeof(T);
};

// 16-byte global -> shared copy; with valid == false it writes 16 zero bytes (src unread)
__device__ __forceinline__ void cp16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}


// Two fp32 lanes at once (sm_100+ packed f32x2 arithmetic; each lane rounds as the scalar
// operation does).
__device__ __forceinline__ uint64_t f2bits(float2 a) { return *reinterpret_cast<uint64_t*>(&a); }
__device__ __forceinline__ float2 bits2f(uint64_t d) { return *reinterpret_cast<float2*>(&d); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2bits(a)), "l"(f2bits(b)), "l"(f2bits(c)));
  return bits2f(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2bits(a)), "l"(f2bits(b)));
  return bits2f(d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2bits(a)), "l"(f2bits(b)));
  return bits2f(d);
}
__device__ __forceinline__ void ld4p(const __nv_bfloat16* p, float2 (&v)[2]) {
  float x[4];
  ld4(p, x);
  v[0] = make_float2(x[0], x[1]);
  v[1] = make_float2(x[2], x[3]);
}
__device__ __forceinline__ void ld4p(const float* p, float2 (&v)[2]) {
  const float4 f = *reinterpret_cast<const float4*>(p);
  v[0] = make_float2(f.x, f.y);
  v[1] = make_float2(f.z, f.w);
}

struct ConvArgs {
  int64_t B, T, Ts, C;
  const void* x;
  const float* w;
  const float* bias;
  const void* halo;
  const void* dy;
  void* y;          // forward output, or dx
  void* dhalo;
  float* part;      // [B * tiles][C][K + 1] per-CTA partials of dw, dbias
  int64_t tiles;    // token tiles per row
};

// Copies rows s0 .. s0 + n - 1 (tokens of row b; negative: the halo) of channels c0 ..
// c0 + 127 of `src` into dst (Tile<T>::ROWB bytes per row); rows outside [-(K-1), T)
// (or negative ones without a halo) and channels past C are zero-filled.
template <int K, typename T>
__device__ __forceinline__ void stage(uint8_t* dst, const ConvArgs& ar, const void* src,
                                      const void* halo, int64_t b, int64_t s0, int n,
                                      int64_t c0) {
  constexpr int CPR = Tile<T>::ROWB / 16;  // 16-byte chunks per row
  for (int e = threadIdx.x; e < n * CPR; e += CONV_NT) {
    const int r = e / CPR, q = e % CPR;
    const int64_t s = s0 + r, c = c0 + q * (16 / (int)sizeof(T));
    const T* p = reinterpret_cast<const T*>(ar.x);  // any valid address when nothing is read
    bool ok = c < ar.C;
    if (s >= 0 && s < ar.T) {
      p = reinterpret_cast<const T*>(src) + (b * ar.Ts + s) * ar.C + c;
    } else if (s < 0 && halo) {
      p = reinterpret_cast<const T*>(halo) + (b * (K - 1) + (K - 1) + s) * ar.C + c;
    } else {
      ok = false;
    }
    cp16(dst + r * Tile<T>::ROWB + q * 16, ok ? (const void*)p : ar.x, ok);
  }
  cp_wait_all();
}

template <int K, typename T>
__global__ void __launch_bounds__(CONV_NT) k_conv_fwd(ConvArgs ar) {
  extern __shared__ __align__(16) uint8_t smx[];
  constexpr int TOK = Tile<T>::TOKF, RUN = TOK / 8;
  const int lane = threadIdx.x & 31, run = threadIdx.x >> 5;
  const int64_t c0 = (int64_t)blockIdx.y * CONV_CH, c = c0 + lane * 4;
  const int64_t b = blockIdx.z;
  const int64_t t0 = (int64_t)blockIdx.x * TOK;
  // staged row r holds token t0 - (K - 1) + r
  stage<K, T>(smx, ar, ar.x, ar.halo, b, t0 - (K - 1), TOK + K - 1, c0);
  __syncthreads();
  const int u0 = run * RUN;
  if (c >= ar.C || t0 + u0 >= ar.T) return;
  const int uend = (int)(t0 + u0 + RUN < ar.T ? u0 + RUN : ar.T - t0);
  float w[4][K], bs[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int i = 0; i < K; ++i) w[j][i] = ar.w[(c + j) * K + i];
    bs[j] = ar.bias ? ar.bias[c + j] : 0.f;
  }
  const T* xs = reinterpret_cast<const T*>(smx) + lane * 4;
  float xw[K][4];  // xw[0 .. K-2]: x~[t-K+1 .. t-1]; xw[K-1]: x[t]
#pragma unroll
  for (int i = 0; i < K - 1; ++i) ld4(xs + (u0 + i) * CONV_CH, xw[i]);
  T* y = reinterpret_cast<T*>(ar.y) + (b * ar.Ts + t0) * ar.C + c;
#pragma unroll 4
  for (int u = u0; u < uend; ++u) {
    ld4(xs + (u + K - 1) * CONV_CH, xw[K - 1]);
    float o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a = bs[j];
#pragma unroll
      for (int i = 0; i < K; ++i) a = fmaf(w[j][i], xw[i][j], a);
      o[j] = a * sigm(a);
    }
    st4(y + (int64_t)u * ar.C, o);
#pragma unroll
    for (int i = 0; i < K - 1; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) xw[i][j] = xw[i + 1][j];
  }
}

template <int K, typename T>
__global__ void __launch_bounds__(CONV_NT) k_conv_bwd(ConvArgs ar) {
  extern __shared__ __align__(16) uint8_t smx[];
  constexpr int TOK = Tile<T>::TOKB, RUN = TOK / 8;
  constexpr int XROWS = TOK + 2 * (K - 1), DROWS = TOK + K - 1;
  const int lane = threadIdx.x & 31, run = threadIdx.x >> 5;
  const int64_t c0 = (int64_t)blockIdx.y * CONV_CH, c = c0 + lane * 4;
  const int64_t b = blockIdx.z;
  const int64_t t0 = (int64_t)blockIdx.x * TOK;
  uint8_t* xsb = smx;                                 // row r: token t0 - (K - 1) + r
  uint8_t* dysb = smx + XROWS * Tile<T>::ROWB;        // row r: token t0 + r
  stage<K, T>(xsb, ar, ar.x, ar.halo, b, t0 - (K - 1), XROWS, c0);
  stage<K, T>(dysb, ar, ar.dy, nullptr, b, t0, DROWS, c0);
  __syncthreads();
  const int u0 = run * RUN;
  const bool live = c < ar.C && t0 + u0 < ar.T;
  float2 acc[2][K + 1];  // channel pairs (0, 1), (2, 3): dw taps, then dbias
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int i = 0; i <= K; ++i) acc[p][i] = make_float2(0.f, 0.f);
  if (live) {
    const int uend = (int)(t0 + u0 + RUN < ar.T ? u0 + RUN : ar.T - t0);  // own tokens
    // tokens at or past ulast have no ds (clamped before the cast: T - t0 may exceed int)
    const int64_t rest = ar.T - t0, span = TOK + 2 * (K - 1);
    const int ulast = (int)(rest < span ? rest : span);
    float2 w[2][K], bs[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
#pragma unroll
      for (int i = 0; i < K; ++i)
        w[p][i] = make_float2(ar.w[(c + 2 * p) * K + i], ar.w[(c + 2 * p + 1) * K + i]);
      bs[p] = ar.bias ? make_float2(ar.bias[c + 2 * p], ar.bias[c + 2 * p + 1])
                      : make_float2(0.f, 0.f);
    }
    const T* xs = reinterpret_cast<const T*>(xsb) + lane * 4;
    const T* dys = reinterpret_cast<const T*>(dysb) + lane * 4;
    // rings over the window: at step k (token u = u0 + k) slot (k + i) % K holds x~[u-K+1+i]
    // and ds[u-K+1+i] (i = 0 .. K-1); the loop is unrolled, so the slots are fixed registers
    float2 xw[K][2];
    float2 dsw[K][2];
#pragma unroll
    for (int i = 0; i < K - 1; ++i) {
      ld4p(xs + (u0 + i) * CONV_CH, xw[i]);
      dsw[i][0] = dsw[i][1] = make_float2(0.f, 0.f);  // ds before the run feeds no dx it emits
    }
    T* dx = reinterpret_cast<T*>(ar.y) + (b * ar.Ts + t0) * ar.C + c;
    T* dh = reinterpret_cast<T*>(ar.dhalo);
    const int e_first = t0 + u0 == 0 ? -(K - 1) : u0;  // the row's first run also emits dhalo
    // FULL: the run and the K-1 tokens after it lie inside the row, so no step needs a
    // bounds check (every tile but a row's last)
    auto walk = [&](auto full_tag) {
      constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
      for (int k = 0; k < RUN + K - 1; ++k) {
        const int u = u0 + k;
        if (!FULL && u >= uend + K - 1) break;
        if (FULL || u < ulast) {
          ld4p(xs + (u + K - 1) * CONV_CH, xw[(k + K - 1) % K]);
          float2 g[2];
          ld4p(dys + u * CONV_CH, g);
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            float2 a = bs[p];
#pragma unroll
            for (int i = 0; i < K; ++i) a = fma2(w[p][i], xw[(k + i) % K][p], a);
            const float2 s = make_float2(sigm(a.x), sigm(a.y));
            const float2 one = make_float2(1.f, 1.f);
            const float2 t = fma2(a, add2(one, make_float2(-s.x, -s.y)), one);  // 1 + a (1 - s)
            dsw[(k + K - 1) % K][p] = mul2(mul2(g[p], s), t);
          }
        } else {
          dsw[(k + K - 1) % K][0] = dsw[(k + K - 1) % K][1] = make_float2(0.f, 0.f);
        }
        if (FULL ? (k < RUN) : (u < uend)) {  // own token: dw, dbias
#pragma unroll
          for (int p = 0; p < 2; ++p) {
#pragma unroll
            for (int i = 0; i < K; ++i)
              acc[p][i] = fma2(dsw[(k + K - 1) % K][p], xw[(k + i) % K][p], acc[p][i]);
            acc[p][K] = add2(acc[p][K], dsw[(k + K - 1) % K][p]);
          }
        }
        const int e = u - (K - 1);  // dx~[e] = sum_i w[i] ds[u - i]
        const bool emit = FULL ? (k >= K - 1 || e >= e_first) : (e >= e_first && e < uend);
        if (emit) {
          float o[4];
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            float2 v = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < K; ++i) v = fma2(w[p][i], dsw[(k + K - 1 - i) % K][p], v);
            o[2 * p] = v.x;
            o[2 * p + 1] = v.y;
          }
          if (e >= 0)
            st4(dx + (int64_t)e * ar.C, o);
          else if (dh)
            st4(dh + (b * (K - 1) + (K - 1) + e) * ar.C + c, o);
        }
      }
    };
    if (t0 + u0 + RUN + 2 * (K - 1) <= ar.T && uend == u0 + RUN)
      walk(std::true_type{});
    else
      walk(std::false_type{});
  }
  // this CTA's partial sums (in the staged-x space, no longer read): its 8 runs added in
  // order by the threads of run 0
  __syncthreads();
  float* red = reinterpret_cast<float*>(smx);  // [8][CONV_CH][K + 1]
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i <= K; ++i)
      red[(run * CONV_CH + lane * 4 + j) * (K + 1) + i] = (j & 1) ? acc[j >> 1][i].y : acc[j >> 1][i].x;
  __syncthreads();
  if (run == 0 && c < ar.C) {
    float* dst = ar.part + ((b * ar.tiles + blockIdx.x) * ar.C + c) * (K + 1);
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i <= K; ++i) {
        float s = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r) s += red[(r * CONV_CH + lane * 4 + j) * (K + 1) + i];
        dst[j * (K + 1) + i] = s;
      }
  }
}

// dw[c][i] and dbias[c]: the partials of every (row, tile), in order, summed in fp64
__global__ void __launch_bounds__(256) k_conv_reduce(int64_t n_part, int64_t C, int K,
                                                     const float* __restrict__ part, float* dw,
                                                     float* dbias) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= C * (K + 1)) return;
  const int64_t c = idx / (K + 1);
  const int i = (int)(idx % (K + 1));
  double s = 0.0;
  for (int64_t p = 0; p < n_part; ++p) s += part[p * C * (K + 1) + idx];
  if (i < K)
    dw[c * K + i] = (float)s;
  else if (dbias)
    dbias[c] = (float)s;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// the problem's fields; fills the launch geometry
gdn_status check_problem(const gdn_conv_problem* p, ConvArgs* ar) {
  if (!p) return GDN_ERR_INVALID_ARG;
  if (p->dtype != GDN_BF16 && p->dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
  const int64_t Ts = p->T_stride == 0 ? p->T : p->T_stride;
  if (p->B < 0 || p->T < 0 || p->C < 1 || Ts < p->T) return GDN_ERR_INVALID_ARG;
  // grid: token tiles (x), 128-channel blocks (y <= 32768), rows (z <= 65535)
  if (p->B > 65535 || p->T > ((int64_t)1 << 34) || p->C > ((int64_t)1 << 22))
    return GDN_ERR_INVALID_ARG;
  // rows are staged in 16-byte copies: C elements must fill whole 16-byte chunks
  const int64_t esize = p->dtype == GDN_BF16 ? 2 : 4;
  if (p->K < 1 || p->K > 4 || (p->C * esize) % 16 != 0) return GDN_ERR_UNSUPPORTED;
  memset(ar, 0, sizeof(*ar));
  ar->B = p->B;
  ar->T = p->T;
  ar->Ts = Ts;
  ar->C = p->C;
  return GDN_OK;
}

int64_t tiles_of(const ConvArgs& ar, bool bf16, bool bwd) {
  const int64_t tok = bf16 ? (bwd ? Tile<__nv_bfloat16>::TOKB : Tile<__nv_bfloat16>::TOKF)
                           : (bwd ? Tile<float>::TOKB : Tile<float>::TOKF);
  return (ar.T + tok - 1) / tok;
}

// the problem and the pointers both calls take
gdn_status check(const gdn_conv_problem* p, const void* x, const float* w, const float* bias,
                 const void* halo, const void* out, ConvArgs* ar) {
  gdn_status s = check_problem(p, ar);
  if (s != GDN_OK) return s;
  const bool empty = ar->B == 0 || ar->T == 0;
  if (!w || !aligned16(w) || (bias && !aligned16(bias)) || (halo && !aligned16(halo)))
    return GDN_ERR_INVALID_ARG;
  if (!empty && (!x || !out || !aligned16(x) || !aligned16(out))) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

size_t bwd_workspace_bytes(const ConvArgs& ar, int K, bool bf16) {
  return (size_t)(ar.B * tiles_of(ar, bf16, true)) * (size_t)ar.C * (size_t)(K + 1) *
         sizeof(float);
}

// dynamic shared memory of the two kernels (the staged rows)
template <int K, typename T>
constexpr int fwd_smem() { return (Tile<T>::TOKF + K - 1) * Tile<T>::ROWB; }
template <int K, typename T>
constexpr int bwd_smem() {
  return (2 * Tile<T>::TOKB + 3 * (K - 1)) * Tile<T>::ROWB > 8 * CONV_CH * (K + 1) * 4
             ? (2 * Tile<T>::TOKB + 3 * (K - 1)) * Tile<T>::ROWB
             : 8 * CONV_CH * (K + 1) * 4;
}

template <int K, typename T>
cudaError_t launch_fwd_t(ConvArgs ar, cudaStream_t st) {
  constexpr int smem = fwd_smem<K, T>();
  cudaError_t e = cudaFuncSetAttribute(k_conv_fwd<K, T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ar.tiles = (ar.T + Tile<T>::TOKF - 1) / Tile<T>::TOKF;
  dim3 grid((unsigned)ar.tiles, (unsigned)((ar.C + CONV_CH - 1) / CONV_CH), (unsigned)ar.B);
  k_conv_fwd<K, T><<<grid, CONV_NT, smem, st>>>(ar);
  return cudaGetLastError();
}
template <int K>
cudaError_t launch_fwd_k(const ConvArgs& ar, bool bf16, cudaStream_t st) {
  return bf16 ? launch_fwd_t<K, __nv_bfloat16>(ar, st) : launch_fwd_t<K, float>(ar, st);
}

template <int K, typename T>
cudaError_t launch_bwd_t(ConvArgs ar, cudaStream_t st) {
  constexpr int smem = bwd_smem<K, T>();
  cudaError_t e = cudaFuncSetAttribute(k_conv_bwd<K, T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ar.tiles = (ar.T + Tile<T>::TOKB - 1) / Tile<T>::TOKB;
  dim3 grid((unsigned)ar.tiles, (unsigned)((ar.C + CONV_CH - 1) / CONV_CH), (unsigned)ar.B);
  k_conv_bwd<K, T><<<grid, CONV_NT, smem, st>>>(ar);
  return cudaGetLastError();
}
template <int K>
cudaError_t launch_bwd_k(const ConvArgs& ar, bool bf16, cudaStream_t st) {
  return bf16 ? launch_bwd_t<K, __nv_bfloat16>(ar, st) : launch_bwd_t<K, float>(ar, st);
}

gdn_status cuda_ok(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status gdn_conv_silu_fwd(const gdn_conv_problem* p, const void* x, const float* w,
                             const float* bias, const void* halo, void* y, void* stream) {
  ConvArgs ar;
  gdn_status s = check(p, x, w, bias, halo, y, &ar);
  if (s != GDN_OK) return s;
  if (ar.B == 0 || ar.T == 0) return GDN_OK;
  ar.x = x;
  ar.w = w;
  ar.bias = bias;
  ar.halo = p->K > 1 ? halo : nullptr;
  ar.y = y;
  const bool bf16 = p->dtype == GDN_BF16;
  cudaStream_t st = (cudaStream_t)stream;
  switch (p->K) {
    case 1: return cuda_ok(launch_fwd_k<1>(ar, bf16, st));
    case 2: return cuda_ok(launch_fwd_k<2>(ar, bf16, st));
    case 3: return cuda_ok(launch_fwd_k<3>(ar, bf16, st));
    default: return cuda_ok(launch_fwd_k<4>(ar, bf16, st));
  }
}

gdn_status gdn_conv_silu_bwd_workspace_size(const gdn_conv_problem* p, size_t* bytes) {
  if (!bytes) return GDN_ERR_INVALID_ARG;
  ConvArgs ar;
  gdn_status s = check_problem(p, &ar);
  if (s != GDN_OK) return s;
  *bytes = bwd_workspace_bytes(ar, p->K, p->dtype == GDN_BF16);
  return GDN_OK;
}

gdn_status gdn_conv_silu_bwd(const gdn_conv_problem* p, const void* x, const float* w,
                             const float* bias, const void* halo, const void* dy, void* dx,
                             float* dw, float* dbias, void* dhalo, void* workspace,
                             size_t workspace_bytes, void* stream) {
  ConvArgs ar;
  gdn_status s = check(p, x, w, bias, halo, dx, &ar);
  if (s != GDN_OK) return s;
  const bool empty = ar.B == 0 || ar.T == 0;
  if (!dw || !aligned16(dw) || (dbias && !aligned16(dbias)) || (dhalo && !aligned16(dhalo)) ||
      (!empty && (!dy || !aligned16(dy))))
    return GDN_ERR_INVALID_ARG;
  const size_t need = bwd_workspace_bytes(ar, p->K, p->dtype == GDN_BF16);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return GDN_ERR_WORKSPACE;
  const int K = p->K;
  const bool bf16 = p->dtype == GDN_BF16;
  cudaStream_t st = (cudaStream_t)stream;
  ar.x = x;
  ar.w = w;
  ar.bias = bias;
  ar.halo = K > 1 ? halo : nullptr;
  ar.dy = dy;
  ar.y = dx;
  ar.dhalo = K > 1 ? dhalo : nullptr;
  ar.part = (float*)workspace;
  cudaError_t e = cudaSuccess;
  if (K > 1 && dhalo && ar.T == 0 && ar.B > 0) {  // no tokens: the halo gets no gradient
    const size_t hb = (size_t)ar.B * (K - 1) * ar.C * (bf16 ? 2 : 4);
    if ((e = cudaMemsetAsync(dhalo, 0, hb, st)) != cudaSuccess) return GDN_ERR_CUDA;
  }
  if (!empty) {
    switch (K) {
      case 1: e = launch_bwd_k<1>(ar, bf16, st); break;
      case 2: e = launch_bwd_k<2>(ar, bf16, st); break;
      case 3: e = launch_bwd_k<3>(ar, bf16, st); break;
      default: e = launch_bwd_k<4>(ar, bf16, st); break;
    }
    if (e != cudaSuccess) return GDN_ERR_CUDA;
  }
  const int64_t n = ar.C * (K + 1);
  const int64_t n_part = ar.B * tiles_of(ar, bf16, true);
  k_conv_reduce<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(n_part, ar.C, K,
                                                             (const float*)workspace, dw, dbias);
  return cuda_ok(cudaGetLastError());
}

}  // extern "C"
