// gdn_tc_fwd.cu -- fused tensor-core forward of the bf16 path (dk = dv = 128, C = 64).
//
// The chunked gated delta rule (notation of gdn_tc_chain.cu):
//
//   chunk-local   G = cumsum(g), gamma = e^G, P = tril(Q K^T o Gamma),
//                 A = tril(diag(beta) K K^T o Gamma, -1), T = (I + A)^-1,
//                 W = T diag(beta gamma) K,  U = T diag(beta) V
//   recurrence    V' = U - W S,  O = diag(gamma) Q S + P V',
//                 S <- gamma_C S + K~^T V',  K~ = diag(e^{G_C - G}) K
//
// Two kernels, and nothing else of the chunk reaches global memory:
//
// k_tsolve (grid: chunk x Q/K head x row) forms K K^T, Q K^T and the q, k
// norms once per Q/K head, then for each of the r V heads of the group the
// gates, A, the triangular solve T = (I + A)^-1, P and the per-token factors of
// the chunk, and stores one 25.5 KB record per (chunk, V head): T_u = T
// diag(beta), T_w = T diag(beta gamma rk) and P as bf16 tile images, then G, rq,
// rk, gamma rk, gamma rq and rk e^{G_C - G} (fp32).
//
// k_fwd_tc (grid: work item x V head x row; one CTA per SM, 16 warps) walks
// the chunks of one segment of one (row, V head).  A prologue warp group
// prepares chunk n + 1 -- [T_u; 0] V -> U straight
// into the accumulator that chunk n + 1's state product will add to, [0; T_w] K
// -> W (stored negated), the scaled query rows -- while the chain warps run
// chunk n: U + [-W; Qg] S gives V' (and diag(gamma) Q S) in one M = 128 product;
// V' and V2 = diag(rk e^{G_C - G}) V' go to shared memory; then K^T V2 and
// [. ; P] V' (the state update and the intra-chunk part of O), S <- gamma_C S +
// K^T V2 in fp32 registers.  Three TMEM accumulators rotate, so that reading
// O out of one overlaps the next chunk's products into the others.
//
// Work items: APPLY (token output from an initial state, and the final state),
// SUMS (state reached from zero: the S of a segment summary H_out = M H_in + S
// of "linear attention cp #1035", "p2p") and SUMM (the segment's transition M,
// the same chain from the identity with U = 0).  One launch can mix them.
#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include "gdn_internal.h"
#include "gdn_tc_common.cuh"

namespace gdn {

bool tc_make_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t Ts, int64_t heads);

namespace {

using namespace tc;

// Per (chunk, V head) record written by k_tsolve: the T_u, T_w and P images, then six
// 64-float vectors.
constexpr uint32_t kTu = 8192;
constexpr uint32_t kTwOff = kTu;                 // T_w = T diag(beta gamma rk)
constexpr uint32_t kPoff = 2 * kTu;              // P = tril(Q K^T o Gamma) with the norm factors
constexpr uint32_t kVecOff = 3 * kTu;
constexpr uint32_t kVecBytes = 6 * 64 * 4;
constexpr uint32_t kRec = kVecOff + kVecBytes;
enum { V_G = 0, V_RQ = 64, V_RK = 128, V_CW = 192, V_QF = 256, V_KF = 320 };

// ---------------------------------------------------------------------------
// Shared by both kernels: the row a CTA works on, gates, row norms, waits.
// ---------------------------------------------------------------------------
struct RowInfo {
  int64_t b;      // batch row of the tensors
  int64_t t0;     // first token of the sequence inside that row
  int64_t len;    // tokens of the sequence (valid ones: the rest of its chunks are masked)
  int64_t nch;    // chunks walked
  int64_t cbase;  // index of the sequence's first chunk in the record store
};

__device__ __forceinline__ RowInfo row_info(int64_t row, int64_t T, int64_t NC,
                                            const int32_t* valid_len, int* status,
                                            bool report) {
  RowInfo ri;
  ri.b = row;
  ri.t0 = 0;
  ri.nch = NC;
  ri.cbase = row * NC;
  int64_t L = T;
  if (valid_len) {
    L = valid_len[row];
    if (L < 0 || L > T) {
      if (report && status) atomicOr(status, kStatusClamped);
      L = L < 0 ? 0 : T;
    }
  }
  ri.len = L;
  return ri;
}

// g in log2 units and beta of one token (zero for masked tokens).
__device__ __forceinline__ void gate_of(float a, float b, float A_log, float dt_bias, bool valid,
                                        float* gl, float* beta) {
  float g = 0.f, be = 0.f;
  if (valid) {
    const float x = a + dt_bias;
    const float sp = x > 20.f ? x : log1pf(expf(x));
    g = -expf(A_log) * sp;
    be = 1.f / (1.f + expf(-b));
  }
  *gl = g * kLog2e;
  *beta = be;
}

// Inclusive prefix sum over the 64 values v of threads 0..63 of a two-warp group
// (`lane`, `w` = 0 or 1 the warp of the group); `carry` is a shared float.
// Every thread of both warps must call it; named barrier `barid` over 64 threads.
__device__ __forceinline__ float scan64(float v, int lane, int w, float* carry, int barid) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (w == 0 && lane == 31) *carry = v;
  asm volatile("bar.sync %0, 64;" ::"r"(barid) : "memory");
  if (w == 1) v += *carry;
  return v;
}

// Sum of squares of row r of a [64][128] bf16 tile held as two K-major 128B-swizzled
// atoms `astride` bytes apart (fixed order).
__device__ __forceinline__ float row_sumsq(const uint8_t* tile, uint32_t astride, int r) {
  float s = 0.f;
#pragma unroll
  for (int a = 0; a < 2; ++a) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float x[8];
      ld_chunk(tile + a * astride, kmaj_chunk(r, c), x);
#pragma unroll
      for (int e = 0; e < 8; ++e) s = fmaf(x[e], x[e], s);
    }
  }
  return s;
}

// Hardware base-2 exponential (ex2.approx: relative error ~2^-22, far below the bf16
// operands it scales).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns, to every participant, whether any of them passed
// `pred` true: a group leaves a loop together or not at all.
__device__ __forceinline__ bool named_sync_any(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// One try_wait that lets the hardware suspend the thread (up to kSuspendNs) until the
// phase completes, instead of spinning: waiting warps leave their issue slots to the
// warps that compute.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool try_wait_suspend(uint32_t addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(addr), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return done != 0;
}

// Bounded wait that also gives up as soon as another role of the CTA has aborted.
// (Every thread that calls it polls; callers that must agree combine the results.)
__device__ __forceinline__ bool wait_ph(uint64_t* bar, uint32_t parity, int* status,
                                        volatile int* abort_flag) {
  const uint32_t addr = smem_u32(bar);
  if (try_wait_suspend(addr, parity)) return true;
  const uint64_t t0 = global_timer();
  for (;;) {
    if (try_wait_suspend(addr, parity)) return true;
    if (abort_flag && *abort_flag) return false;
    if (global_timer() - t0 > kWaitLimitNs) {
      if (abort_flag) *abort_flag = 1;
      if (status) atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// The same wait for a whole warp: lane 0 polls, every lane gets its answer.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status,
                                          volatile int* abort_flag) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_ph(bar, parity, status, abort_flag);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Four 16-column TMEM loads of this thread's lane (columns c0 .. c0 + 63), one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t c0, float (&v)[64]) {
  tmem_ld16x4(c0, c0 + 16, c0 + 32, c0 + 48, *reinterpret_cast<float(*)[16]>(&v[0]),
              *reinterpret_cast<float(*)[16]>(&v[16]), *reinterpret_cast<float(*)[16]>(&v[32]),
              *reinterpret_cast<float(*)[16]>(&v[48]));
}
// Two 16-column loads (columns c0 .. c0 + 31), one wait.
__device__ __forceinline__ void tmem_ld32w(uint32_t c0, float (&v)[32]) {
  tmem_ld16x2(c0, c0 + 16, *reinterpret_cast<float(*)[16]>(&v[0]),
              *reinterpret_cast<float(*)[16]>(&v[16]));
}

// ============================================================================
// k_tsolve: grid (NC, Hqk, rows), 256 threads.
// ============================================================================
constexpr int TS_THREADS = 256;
constexpr uint32_t TS_A = 0;                       // fp32 A [64][LDA]
constexpr uint32_t TS_T = TS_A + 64 * LDA * 4;     // fp32 T [64][LDA]
constexpr uint32_t TS_Y = TS_T + 64 * LDA * 4;     // solve scratch, 8 warps x 128 floats
constexpr uint32_t TS_K = 38912;                   // k tile: two 8 KB atoms (the 8 KB before
                                                   // atom 0 are the junk rows of the Gram)
constexpr uint32_t TS_Q = TS_K + 16384;            // q tile (norms only)
constexpr uint32_t TS_OUT = TS_Q + 16384;          // record staging: T_u, T_w, P images, vectors
constexpr uint32_t TS_VEC = TS_OUT + 26624;        // G[64], beta[64], rk[64], rq[64], cw[64], carry
constexpr uint32_t TS_BAR = TS_VEC + 1536;
constexpr uint32_t TS_SMEM = TS_BAR + 64 + 1024;
static_assert(TS_Y + 4096 <= TS_K, "solve buffers overlap the k tile");
static_assert(TS_OUT % 1024 == 0 && kRec % 16 == 0 && kRec <= 26624, "record staging");

struct TsolveArgs {
  int64_t T, H, Hqk, r, NC, NCtot;
  int l2norm, has_q;
  float eps, scale;
  const __nv_bfloat16* a;
  const __nv_bfloat16* b;
  int64_t Ts;
  const float* A_log;
  const float* dt_bias;
  const int32_t* valid_len;
  uint8_t* rec;  // [H][NCtot] records
  int* status;
};

// T diag(beta) and T diag(beta gamma rk) entries (images kTu bytes apart), written as the
// solve finalises them.
struct TuEmit {
  uint8_t* tile;
  const float* beta;
  const float* cw;  // beta gamma rk
  __device__ __forceinline__ void one(int i, int j, float x) const {
    const uint32_t off = kmaj_chunk(i, j >> 3) + (j & 7) * 2;
    *reinterpret_cast<__nv_bfloat16*>(tile + off) = __float2bfloat16_rn(x * beta[j]);
    *reinterpret_cast<__nv_bfloat16*>(tile + kTu + off) = __float2bfloat16_rn(x * cw[j]);
  }
  __device__ __forceinline__ void two(int i, int j, float x0, float x1) const {
    const uint32_t off = kmaj_chunk(i, j >> 3) + (j & 7) * 2;
    *reinterpret_cast<uint32_t*>(tile + off) = pack_bf16(x0 * beta[j], x1 * beta[j + 1]);
    *reinterpret_cast<uint32_t*>(tile + kTu + off) = pack_bf16(x0 * cw[j], x1 * cw[j + 1]);
  }
};

__global__ void __launch_bounds__(TS_THREADS, 2)
    k_tsolve(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mq,
             TsolveArgs ar) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t base = smem_u32(sm);
  float* sA = (float*)(sm + TS_A);
  float* sT = (float*)(sm + TS_T);
  float* sY = (float*)(sm + TS_Y);
  float* sG = (float*)(sm + TS_VEC);
  float* sBeta = sG + 64;
  float* sRk = sG + 128;
  float* sRq = sG + 192;
  float* sCw = sG + 256;     // beta gamma rk
  float* sCarry = sG + 320;
  float* sOutVec = (float*)(sm + TS_OUT + kVecOff);
  uint64_t* bar_k = (uint64_t*)(sm + TS_BAR);
  uint64_t* bar_g = bar_k + 1;
  uint32_t* s_tmem = (uint32_t*)(bar_k + 2);
  volatile int* s_abort = (volatile int*)(s_tmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t c = blockIdx.x, hq = blockIdx.y, row = blockIdx.z;
  const RowInfo ri = row_info(row, ar.T, ar.NC, ar.valid_len, ar.status, false);
  if (c >= ri.nch) return;
  const int64_t tc0 = ri.t0 + c * 64;  // first token of the chunk

  if (tid == 0) {
    mbar_init(bar_k, 1);
    mbar_init(bar_g, 1);
    fence_barrier_init();
    *s_abort = 0;
  }
  if (warp == 0) tmem_alloc(s_tmem, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_k, ar.has_q ? 32768u : 16384u);
    for (int at = 0; at < 2; ++at) {
      tma_load_4d(sm + TS_K + at * 8192, &mk, at * 64, (int)hq, (int)tc0, (int)ri.b, bar_k);
      if (ar.has_q)
        tma_load_4d(sm + TS_Q + at * 8192, &mq, at * 64, (int)hq, (int)tc0, (int)ri.b, bar_k);
    }
  }
  if (tid == 0 && !wait_ph(bar_k, 0, ar.status, s_abort)) *s_abort = 1;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*s_abort) goto done;
  if (tid == 0) {  // K K^T (columns 0..63) and Q K^T (64..127) in TMEM lanes 64..127; rows
                   // 0..63 of each A operand are the 8 KB before the tile (junk)
    const uint32_t id = idesc_bf16(128, 64, 0, 0);
    const uint64_t d = sdesc(base, 16, 1024);
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t at = ks >> 2, kk = ks & 3;
      const uint32_t kb = TS_K + at * 8192 + kk * 32, qb = TS_Q + at * 8192 + kk * 32;
      mma_bf16(tmem, d + ((kb - 8192) >> 4), d + (kb >> 4), id, ks > 0);
      if (ar.has_q) mma_bf16(tmem + 64, d + ((qb - 8192) >> 4), d + (kb >> 4), id, ks > 0);
    }
    mma_commit(bar_g);
  }
  if (tid < 64) {
    const float ss = row_sumsq(sm + TS_K, 8192, tid);
    sRk[tid] = ar.l2norm ? rsqrtf(ss + ar.eps) : 1.f;
  } else if (tid < 128) {
    float f = ar.scale;
    if (ar.has_q && ar.l2norm) f *= rsqrtf(row_sumsq(sm + TS_Q, 8192, tid - 64) + ar.eps);
    sRq[tid - 64] = f;
  }
  if (tid == 0 && !wait_ph(bar_g, 0, ar.status, s_abort)) *s_abort = 1;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*s_abort) goto done;
  {
    const int quad = warp & 3, half = warp >> 2;
    const bool kr = quad >= 2;             // warps holding rows of K K^T and Q K^T
    const int i = (quad & 1) * 32 + lane;  // row of K K^T / Q K^T
    float kk[32], qk[32];
    if (kr) {
      tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + half * 32, kk);
      if (ar.has_q) tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + 64 + half * 32, qk);
    }
    for (int j = 0; j < (int)ar.r; ++j) {
      const int64_t hv = hq * ar.r + j;
      if (tid < 64) {
        const int64_t t = c * 64 + tid;
        const int64_t gi = (ri.b * ar.Ts + ri.t0 + t) * ar.H + hv;
        float gl = 0.f, be = 0.f;
        const bool valid = t < ri.len;
        gate_of(valid ? __bfloat162float(ar.a[gi]) : 0.f, valid ? __bfloat162float(ar.b[gi]) : 0.f,
                ar.A_log[hv], ar.dt_bias[hv], valid, &gl, &be);
        const float G = scan64(gl, lane, warp, sCarry, 1);
        sG[tid] = G;
        sBeta[tid] = be;
      }
      if (tid == 0) bulk_wait_read();  // the previous head's store has read the staging record
      __syncthreads();
      for (int e = tid; e < 1024; e += TS_THREADS)  // entries above the diagonal stay zero
        reinterpret_cast<uint4*>(sm + TS_OUT)[e] = make_uint4(0, 0, 0, 0);
      if (tid < 64) {  // the chunk's per-token factors for the forward chain
        const float G = sG[tid], gam = exp2f(G), rk = sRk[tid], rq = sRq[tid];
        sCw[tid] = sBeta[tid] * gam * rk;
        sOutVec[V_G + tid] = G;
        sOutVec[V_RQ + tid] = rq;
        sOutVec[V_RK + tid] = rk;
        sOutVec[V_CW + tid] = gam * rk;
        sOutVec[V_QF + tid] = gam * rq;
        sOutVec[V_KF + tid] = exp2f(sG[63] - G) * rk;
      }
      if (kr) {  // A = tril(diag(beta) K K^T o Gamma, -1) and P = tril(Q K^T o Gamma)
        const float gi_ = sG[i], f = sBeta[i] * sRk[i], fq = sRq[i];
        float pv[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int jj = half * 32 + e;
          const float dj = sRk[jj] * exp2f(gi_ - sG[jj]);
          sA[i * LDA + jj] = (jj < i) ? f * kk[e] * dj : 0.f;
          pv[e] = (ar.has_q && jj <= i) ? fq * qk[e] * dj : 0.f;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) st_chunk(sm + TS_OUT + kPoff, kmaj_chunk(i, half * 4 + cc), &pv[cc * 8]);
      }
      __syncthreads();
      solve_unit_lower64_mma(sA, sT, sY, LDA, TuEmit{sm + TS_OUT, sBeta, sCw});
      fence_proxy_async();
      __syncthreads();
      if (tid == 0) {
        bulk_store(ar.rec + (hv * ar.NCtot + ri.cbase + c) * (int64_t)kRec, sm + TS_OUT, kRec);
        bulk_commit();
      }
    }
  }
done:
  if (tid == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// ============================================================================
// k_fwd_tc: grid (items, H, rows), 512 threads, one CTA per SM.
//
// Warps: 0 loads (TMA for k, q, v; bulk copies of the chunk record), 1 issues
// the chain products, 2 the prologue products, 3 idle, 4..11 run the chain
// epilogues and own the fp32 state (warp w: TMEM lane quadrant w & 3, state
// columns ((w - 4) >> 2) * 64 .. + 63), 12..15 run the prologue.
// ============================================================================
constexpr int FW_THREADS = 512;
enum { FW_APPLY = 0, FW_SUMS = 1, FW_SUMM = 2 };

// shared memory (offsets from the 1024-aligned base)
constexpr uint32_t F_KQ = 0;         // per dk half a (32 KB apart): [K0 | Q0 | Q1 | K1]
constexpr uint32_t F_KQ_A = 32768;
constexpr uint32_t F_WQ = 65536;     // per dk half a (16 KB apart): [-W_a | Qg_a], 128 x 64 K-major
constexpr uint32_t F_V = 98304;      // v tile, two 8 KB atoms (MN-major B operand)
constexpr uint32_t F_TU = 114688;    // [T_u | 0 | T_w], three 64 x 64 K-major images
constexpr uint32_t F_V2 = 139264;    // V2 = diag(rk e^{G_C - G}) V', bf16, MN-major [token][dv]
constexpr uint32_t F_P = 155648;     // P of chunk slot s at F_P + 8 KB s (the 8 KB before each
                                     // are the junk rows 0..63 of the [. ; P] operand)
constexpr uint32_t F_S = 172032;     // state, bf16, MN-major [dk][dv] (column halves 16 KB apart)
constexpr uint32_t F_VP = 204800;    // V', bf16, MN-major [token][dv] (halves 8 KB apart)
constexpr uint32_t F_VEC = 221184;   // per slot (1.5 KB): the chunk record's vectors
constexpr uint32_t F_BAR = F_VEC + 2 * kVecBytes;
constexpr uint32_t F_SMEM = F_BAR + 512 + 1024;
static_assert(F_SMEM <= 232448, "shared memory");

// k slot s and q slot s inside a dk half: [K0 | Q0 | Q1 | K1]
__device__ __forceinline__ uint32_t k_slot(int s) { return s ? 24576u : 0u; }
__device__ __forceinline__ uint32_t q_slot(int s) { return s ? 16384u : 8192u; }

// TMEM: three chain accumulators (128 columns each) and W's product.  Chunk k (counted
// from the segment's first chunk) uses accumulator k % 3 as R1 (U, then + [-W; Qg] S,
// then + [. ; P] V') and (k + 2) % 3 as R2 (K^T V2).
constexpr uint32_t TM_ZW = 384;
__device__ __forceinline__ uint32_t acc_col(int64_t k, int off) { return (uint32_t)(((k + off) % 3) * 128); }
// Number of uses (as R1 or R2) of accumulator a by chunks before chunk c: its completion
// index on that accumulator's release barrier.
__device__ __forceinline__ uint32_t acc_use(int64_t c, int a) {
  uint32_t n = (uint32_t)(2 * (c / 3));
  for (int r = 0; r < (int)(c % 3); ++r) n += (r == a || r == (a + 1) % 3) ? 1u : 0u;
  return n;
}

// barrier indices (the multi-slot barriers take consecutive entries)
enum {
  B_FK = 0,            // [2] k slot filled
  B_EK = B_FK + 2,     // [2] k slot and vector slot released: state update read (8 arrivals)
  B_FVEC = B_EK + 2,   // [2] vectors (and P) of the chunk loaded
  B_FQ = B_FVEC + 2,   // [2] q slot filled
  B_EQ = B_FQ + 2,     // [2] q slot released (scaled rows written)
  B_FV = B_EQ + 2,     // v tile loaded
  B_FTU,               // T_u and T_w loaded
  B_EV,                // v, T_u, T_w released (U and W products done)
  B_L6,                // U and W products done
  B_EZW,               // W accumulator read
  B_EP,                // [2] P slot released (P V' done)
  B_EWQ = B_EP + 2,    // [-W; Qg] released (its product done)
  B_RDY,               // [2] chunk slot ready for the chain
  B_M1 = B_RDY + 2,    // R1 += [-W; Qg] S done
  B_M2,                // K^T V2 done
  B_M3,                // [. ; P] V' done
  B_E1,                // V', V2 written (4 arrivals)
  B_E2,                // state tile written (8 arrivals)
  B_FREE,              // [3] accumulator released by its readers (8 arrivals)
  B_DR1 = B_FREE + 3,  // chain products drained (abort path)
  B_DR2,               // prologue products drained (abort path)
  B_NUM
};
static_assert(B_EWQ == B_EP + 2 && B_M1 == B_RDY + 2 && B_DR1 == B_FREE + 3 &&
                  B_NUM * 8 + 16 <= 512,
              "barrier layout");

struct FwdItem {
  int mode, seg;
};
constexpr int kMaxItems = FwdWork::kMax;

struct FwdArgs {
  int64_t T, Ts, H, Hqk, r, NC, NCtot, CPS;
  int P;
  const int32_t* valid_len;
  const uint8_t* rec;
  const float* init;        // APPLY: start state of segment s at init + s * init_stride (or null)
  int64_t init_stride;
  const float* init0;       // APPLY of segment 0: its start state (h0; may be null)
  __nv_bfloat16* o;
  float* final_out;         // APPLY of the last segment: the final state (may be null)
  float* S_out;             // SUMS: S of segment s at S_out + s * out_stride
  float* M_out;             // SUMM: M of segment s at M_out + s * out_stride
  int64_t out_stride;
  int* status;
  int nitems;
  FwdItem items[kMaxItems];
};

__global__ void __launch_bounds__(FW_THREADS, 1)
    k_fwd_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
             const __grid_constant__ CUtensorMap mv, const __grid_constant__ FwdArgs ar) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t base = smem_u32(sm);
  uint64_t* bars = (uint64_t*)(sm + F_BAR);
  uint32_t* s_tmem = (uint32_t*)(bars + B_NUM);
  volatile int* s_abort = (volatile int*)(s_tmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const FwdItem item = ar.items[blockIdx.x];
  const int mode = item.mode, seg = item.seg;
  const bool apply = mode == FW_APPLY, needU = mode != FW_SUMM;
  const int64_t h = blockIdx.y, row = blockIdx.z;
  const int64_t hq = h / ar.r;
  const RowInfo ri = row_info(row, ar.T, ar.NC, ar.valid_len, ar.status,
                              tid == 0 && h == 0 && blockIdx.x == 0);
  const int64_t cs = (int64_t)seg * ar.CPS;
  const int64_t ce = cs + ar.CPS < ri.nch ? cs + ar.CPS : ri.nch;
  const int64_t nloc = ce > cs ? ce - cs : 0;  // chunks of this work item

  if (tid == 0) {
    for (int i = 0; i < B_NUM; ++i) {
      uint32_t cnt = 1;
      if (i == B_E1) cnt = 4;
      if (i == B_E2 || i == B_EK || i == B_EK + 1 || (i >= B_FREE && i < B_FREE + 3)) cnt = 8;
      mbar_init(bars + i, cnt);
    }
    fence_barrier_init();
    *s_abort = 0;
  }
  if (warp == 0) tmem_alloc(s_tmem, 512);
  for (int e = tid; e < 512; e += FW_THREADS)  // the zero block between T_u and T_w
    reinterpret_cast<uint4*>(sm + F_TU + 8192)[e] = make_uint4(0, 0, 0, 0);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint64_t dbase = sdesc(base, 16, 1024);  // + byte offset / 16 = descriptor of a tile
  int* st = ar.status;

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    const uint8_t* recs = ar.rec + (h * ar.NCtot + ri.cbase) * (int64_t)kRec;
    uint32_t nk[2] = {0, 0}, nqf[2] = {0, 0}, nvec[2] = {0, 0}, ntu = 0, nv = 0;
    for (int64_t k = 0; k < nloc; ++k) {
      const int64_t n = cs + k;
      const int s = (int)(k & 1);
      const uint32_t j = (uint32_t)(k >> 1);
      const int64_t tc0 = ri.t0 + n * 64;
      const uint8_t* rec = recs + n * (int64_t)kRec;
      // the k slot, the vector slot and the P slot of chunk n (their last readers: the state
      // update and the P V' product of chunk n - 2)
      if (j > 0 && !warp_wait(bars + B_EK + s, (j - 1) & 1, st, s_abort)) break;
      if (apply && j > 0 && !warp_wait(bars + B_EP + s, (j - 1) & 1, st, s_abort)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bars + B_FVEC + s, kVecBytes + (apply ? 8192u : 0u));
        bulk_load(sm + F_VEC + s * kVecBytes, rec + kVecOff, kVecBytes, bars + B_FVEC + s);
        if (apply) bulk_load(sm + F_P + s * 8192, rec + kPoff, 8192, bars + B_FVEC + s);
        mbar_arrive_expect_tx(bars + B_FK + s, 16384u);
        for (int a = 0; a < 2; ++a)
          tma_load_4d(sm + F_KQ + a * F_KQ_A + k_slot(s), &mk, a * 64, (int)hq, (int)tc0,
                      (int)ri.b, bars + B_FK + s);
      }
      ++nk[s];
      ++nvec[s];
      if (apply) {
        if (j > 0 && !warp_wait(bars + B_EQ + s, (j - 1) & 1, st, s_abort)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bars + B_FQ + s, 16384u);
          for (int a = 0; a < 2; ++a)
            tma_load_4d(sm + F_KQ + a * F_KQ_A + q_slot(s), &mq, a * 64, (int)hq, (int)tc0,
                        (int)ri.b, bars + B_FQ + s);
        }
        ++nqf[s];
      }
      if (k > 0 && !warp_wait(bars + B_EV, (uint32_t)((k - 1) & 1), st, s_abort)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bars + B_FTU, 2 * kTu);
        bulk_load(sm + F_TU, rec, kTu, bars + B_FTU);
        bulk_load(sm + F_TU + 16384, rec + kTwOff, kTu, bars + B_FTU);
        if (needU) {
          mbar_arrive_expect_tx(bars + B_FV, 16384u);
          for (int a = 0; a < 2; ++a)
            tma_load_4d(sm + F_V + a * 8192, &mv, a * 64, (int)h, (int)tc0, (int)ri.b,
                        bars + B_FV);
        }
      }
      ++ntu;
      if (needU) ++nv;
      if (lane == 0 && k + 1 < nloc) {  // pull the next chunk's tiles into L2 meanwhile
        const int tn = (int)(tc0 + 64);
        l2_prefetch(rec + kRec, kRec);
        for (int a = 0; a < 2; ++a) {
          l2_prefetch_tile(&mk, a * 64, (int)hq, tn, (int)ri.b);
          if (apply) l2_prefetch_tile(&mq, a * 64, (int)hq, tn, (int)ri.b);
          if (needU) l2_prefetch_tile(&mv, a * 64, (int)h, tn, (int)ri.b);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && *s_abort) {  // let the last fill of every buffer land before exit
      for (int s = 0; s < 2; ++s) {
        if (nk[s]) mbar_wait(bars + B_FK + s, (nk[s] - 1) & 1, nullptr, 0);
        if (nvec[s]) mbar_wait(bars + B_FVEC + s, (nvec[s] - 1) & 1, nullptr, 0);
        if (nqf[s]) mbar_wait(bars + B_FQ + s, (nqf[s] - 1) & 1, nullptr, 0);
      }
      if (ntu) mbar_wait(bars + B_FTU, (ntu - 1) & 1, nullptr, 0);
      if (nv) mbar_wait(bars + B_FV, (nv - 1) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ chain products
    if (lane == 0) {
      const uint32_t id_a = idesc_bf16(128, 128, 0, 1);  // [-W; Qg] S, [. ; P] V'
      const uint32_t id_b = idesc_bf16(128, 128, 1, 1);  // K^T V2
      bool issued = false;
      for (int64_t k = 0; k < nloc; ++k) {
        const int s = (int)(k & 1);
        const uint32_t j = (uint32_t)(k >> 1), ph = (uint32_t)(k & 1);
        const int a1 = (int)(k % 3), a2 = (int)((k + 2) % 3);
        const uint32_t r1 = tmem + acc_col(k, 0), r2 = tmem + acc_col(k, 2);
        if (!wait_ph(bars + B_RDY + s, j & 1, st, s_abort)) break;  // implies U is in R1
        if (!wait_ph(bars + B_E2, ph, st, s_abort)) break;          // state tile of chunk k
        // without U (transitions) the product overwrites R1: its last use must be over
        if (!needU && k >= 2 &&
            !wait_ph(bars + B_FREE + a1, acc_use(k - 2, a1) & 1, st, s_abort))
          break;
        tc_fence_after();
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t at = ks >> 2, kk = ks & 3;
          mma_bf16(r1, dbase + ((F_WQ + at * 16384 + kk * 32) >> 4),
                   sdesc(base + F_S + ks * 2048, 16384, 1024), id_a, (needU || ks > 0) ? 1u : 0u);
        }
        mma_commit(bars + B_M1);
        mma_commit(bars + B_EWQ);
        issued = true;
        if (!wait_ph(bars + B_E1, ph, st, s_abort)) break;
        // R2 is overwritten: its last use (R1 of chunk k - 1) must be over
        if (k >= 1 && !wait_ph(bars + B_FREE + a2, acc_use(k - 1, a2) & 1, st, s_abort)) break;
        tc_fence_after();
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(r2, sdesc(base + F_KQ + k_slot(s) + ks * 2048, F_KQ_A, 1024),
                   sdesc(base + F_V2 + ks * 2048, 8192, 1024), id_b, ks > 0);
        mma_commit(bars + B_M2);
        if (apply) {
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(r1, dbase + ((F_P + s * 8192 - 8192 + ks * 32) >> 4),
                     sdesc(base + F_VP + ks * 2048, 8192, 1024), id_a, 1);
          mma_commit(bars + B_M3);
          mma_commit(bars + B_EP + s);
        }
      }
      if (*s_abort && issued) {  // every product issued so far has landed
        mma_commit(bars + B_DR1);
        mbar_wait(bars + B_DR1, 0, nullptr, 0);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ prologue products
    if (lane == 0) {
      const uint32_t id_l = idesc_bf16(128, 128, 0, 1);  // [T_u;0] V, [0;T_w] K
      bool issued = false;
      for (int64_t k = 0; k < nloc; ++k) {
        const int s = (int)(k & 1);
        const uint32_t ph = (uint32_t)(k & 1);
        const int a1 = (int)(k % 3);
        if (!wait_ph(bars + B_FTU, ph, st, s_abort)) break;
        if (!wait_ph(bars + B_FK + s, (uint32_t)((k >> 1) & 1), st, s_abort)) break;
        if (needU && !wait_ph(bars + B_FV, ph, st, s_abort)) break;
        if (k > 0 && !wait_ph(bars + B_EZW, (uint32_t)((k - 1) & 1), st, s_abort)) break;
        // U goes into chunk k's R1, whose last use (R2 of chunk k - 2) must be over
        if (needU && k >= 2 &&
            !wait_ph(bars + B_FREE + a1, acc_use(k - 2, a1) & 1, st, s_abort))
          break;
        tc_fence_after();
        if (needU)
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + acc_col(k, 0), dbase + ((F_TU + ks * 32) >> 4),
                     sdesc(base + F_V + ks * 2048, 8192, 1024), id_l, ks > 0);
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + TM_ZW, dbase + ((F_TU + 8192 + ks * 32) >> 4),
                   sdesc(base + F_KQ + k_slot(s) + ks * 2048, F_KQ_A, 1024), id_l, ks > 0);
        mma_commit(bars + B_L6);
        mma_commit(bars + B_EV);
        issued = true;
      }
      if (*s_abort && issued) {
        mma_commit(bars + B_DR2);
        mbar_wait(bars + B_DR2, 0, nullptr, 0);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ chain epilogues
    const int quad = warp & 3, half = (warp - 4) >> 2;
    const int r = quad * 32 + lane;  // state row (dk) / TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int64_t bh = ri.b * ar.H + h;
    float S[64];
    {
      const float* src = nullptr;
      if (apply) src = seg == 0 ? ar.init0 : (ar.init ? ar.init + seg * ar.init_stride : nullptr);
#pragma unroll
      for (int e = 0; e < 64; ++e) {
        const int col = half * 64 + e;
        float x = 0.f;
        if (src) x = src[(bh * 128 + r) * 128 + col];
        else if (mode == FW_SUMM) x = (r == col) ? 1.f : 0.f;
        S[e] = x;
      }
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) st_chunk(sm + F_S, mnmaj_chunk(r, half * 8 + cc, 16384), &S[cc * 8]);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + B_E2);
    }
    for (int64_t k = 0; k < nloc; ++k) {
      const int64_t n = cs + k;
      const int s = (int)(k & 1);
      const uint32_t j = (uint32_t)(k >> 1), ph = (uint32_t)(k & 1);
      const int a1 = (int)(k % 3), a2 = (int)((k + 2) % 3);
      const uint32_t r1 = tmem + acc_col(k, 0), r2 = tmem + acc_col(k, 2);
      if (!warp_wait(bars + B_RDY + s, j & 1, st, s_abort)) break;  // the gates of chunk n
      const float* vec = (const float*)(sm + F_VEC + s * kVecBytes);
      const float gC = ex2(vec[V_G + 63]);
      if (quad < 2) {  // V' (rows 0..63 of R1) and V2 for token row r, columns half * 64 ..
        if (!warp_wait(bars + B_M1, ph, st, s_abort)) break;
        tc_fence_after();
        const float kf = vec[V_KF + r];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[32];
          tmem_ld32w(r1 + lane_off + half * 64 + hh * 32, v);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int c16 = half * 8 + hh * 4 + cc;
            if (apply) st_chunk(sm + F_VP, mnmaj_chunk(r, c16, 8192), &v[cc * 8]);
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = v[cc * 8 + e] * kf;
            st_chunk(sm + F_V2, mnmaj_chunk(r, c16, 8192), x);
          }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bars + B_E1);
          mbar_arrive(bars + B_FREE + a1);  // rows 0..63 of R1 are read
        }
      }
      if (!warp_wait(bars + B_M2, ph, st, s_abort)) break;
      tc_fence_after();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v[32];
        tmem_ld32w(r2 + lane_off + half * 64 + hh * 32, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) S[hh * 32 + e] = fmaf(gC, S[hh * 32 + e], v[e]);
      }
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) st_chunk(sm + F_S, mnmaj_chunk(r, half * 8 + cc, 16384), &S[cc * 8]);
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bars + B_E2);
        mbar_arrive(bars + B_EK + s);      // k slot and the chunk's vectors are done
        mbar_arrive(bars + B_FREE + a2);   // R2 is read
      }
      if (quad >= 2) {
        if (apply) {  // O rows (TMEM lanes 64..127 of R1) -> o
          if (!warp_wait(bars + B_M3, ph, st, s_abort)) break;
          tc_fence_after();
          const int i = r - 64;
          const int64_t t = n * 64 + i;
          const bool valid = t < ri.len;
          const bool inside = ri.t0 + t < ar.T;  // the tensor's rows end at T
          __nv_bfloat16* dst = ar.o + ((ri.b * ar.Ts + ri.t0 + t) * ar.H + h) * 128 + half * 64;
          uint4 w[8];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float v[32];
            tmem_ld32w(r1 + lane_off + half * 64 + hh * 32, v);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              w[hh * 4 + cc].x = valid ? pack_bf16(v[cc * 8 + 0], v[cc * 8 + 1]) : 0u;
              w[hh * 4 + cc].y = valid ? pack_bf16(v[cc * 8 + 2], v[cc * 8 + 3]) : 0u;
              w[hh * 4 + cc].z = valid ? pack_bf16(v[cc * 8 + 4], v[cc * 8 + 5]) : 0u;
              w[hh * 4 + cc].w = valid ? pack_bf16(v[cc * 8 + 6], v[cc * 8 + 7]) : 0u;
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars + B_FREE + a1);  // rows 64..127 of R1 are read
          if (inside) {
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) *reinterpret_cast<uint4*>(dst + cc * 8) = w[cc];
          }
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(bars + B_FREE + a1);  // nothing of R1 to read here
        }
      }
    }
    if (!*s_abort) {  // the state after the segment
      float* dst = nullptr;
      if (mode == FW_APPLY) {
        if (seg == ar.P - 1) dst = ar.final_out;
      } else if (mode == FW_SUMS) {
        dst = ar.S_out ? ar.S_out + seg * ar.out_stride : nullptr;
      } else {
        dst = ar.M_out ? ar.M_out + seg * ar.out_stride : nullptr;
      }
      if (dst) {
        float4* d4 = reinterpret_cast<float4*>(dst + (bh * 128 + r) * 128 + half * 64);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          d4[e] = make_float4(S[4 * e], S[4 * e + 1], S[4 * e + 2], S[4 * e + 3]);
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ prologue
    // Every decision to leave the loop is taken together (named_sync_any), so that no
    // thread of the group is left waiting at a named barrier.
    const int pt = tid - 384;       // 0..127
    const int pw = warp - 12;       // 0..3 (also the TMEM lane quadrant)
    for (int64_t k = 0; k < nloc; ++k) {
      const int s = (int)(k & 1);
      const uint32_t j = (uint32_t)(k >> 1), ph = (uint32_t)(k & 1);
      const float* vec = (const float*)(sm + F_VEC + s * kVecBytes);
      // [-W; Qg] is free once the previous chunk's state product is done with it
      bool ok = warp_wait(bars + B_FVEC + s, j & 1, st, s_abort) &&
                (!apply || warp_wait(bars + B_FQ + s, j & 1, st, s_abort)) &&
                (k == 0 || warp_wait(bars + B_EWQ, (uint32_t)((k - 1) & 1), st, s_abort));
      if (named_sync_any(3, 128, !ok)) break;
      if (apply) {  // Qg = diag(gamma rq) Q into rows 64..127 of [-W; Qg]: row pt / 2, dk half pt % 2
        const int qi = pt >> 1, a = pt & 1;
        const uint8_t* qsrc = sm + F_KQ + q_slot(s) + a * F_KQ_A;
        const float f = vec[V_QF + qi];
        float x[8][8];
#pragma unroll
        for (int cj = 0; cj < 8; ++cj) ld_chunk(qsrc, kmaj_chunk(qi, cj), x[cj]);
#pragma unroll
        for (int cj = 0; cj < 8; ++cj) {
#pragma unroll
          for (int q = 0; q < 8; ++q) x[cj][q] *= f;
          st_chunk(sm + F_WQ + a * 16384 + 8192, kmaj_chunk(qi, cj), x[cj]);
        }
        named_sync(3, 128);
        if (pt == 0) mbar_arrive(bars + B_EQ + s);  // q slot read
      }
      ok = warp_wait(bars + B_L6, ph, st, s_abort);
      if (named_sync_any(3, 128, !ok)) break;
      tc_fence_after();
      if (pw >= 2) {  // -W (TMEM lanes 64..127 of the W product) into rows 0..63 of [-W; Qg]
        const int i = (pw & 1) * 32 + lane;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[64];
          tmem_ld64(tmem + TM_ZW + ((uint32_t)(pw * 32) << 16) + hh * 64, v);
#pragma unroll
          for (int e = 0; e < 64; ++e) v[e] = -v[e];
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) st_chunk(sm + F_WQ + hh * 16384, kmaj_chunk(i, cc), &v[cc * 8]);
        }
        fence_proxy_async();
      }
      fence_proxy_async();
      tc_fence_before();
      named_sync(3, 128);
      if (pt == 0) {
        mbar_arrive(bars + B_EZW);
        mbar_arrive(bars + B_RDY + s);
      }
    }
  }
  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <typename K>
cudaError_t smem_attr_fwd(K kernel, uint32_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

size_t fwd_record_bytes() { return kRec; }

cudaError_t launch_tsolve_tc(const Prob& pr, const Inputs& in, const WS& ws, cudaStream_t st) {
  if (pr.B == 0 || pr.NC == 0) return cudaSuccess;
  CUtensorMap mk, mq;
  memset(&mk, 0, sizeof(mk));
  memset(&mq, 0, sizeof(mq));
  if (!tc_make_map(&mk, in.k, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(&mq, in.q ? in.q : in.k, pr.B, pr.T, pr.Ts, pr.Hqk))
    return cudaErrorInvalidValue;
  TsolveArgs ar;
  ar.T = pr.T; ar.H = pr.H; ar.Hqk = pr.Hqk; ar.r = pr.r; ar.NC = pr.NC; ar.NCtot = pr.B * pr.NC;
  ar.l2norm = pr.l2norm; ar.has_q = in.q != nullptr; ar.eps = pr.eps; ar.scale = pr.scale;
  ar.a = (const __nv_bfloat16*)in.a; ar.b = (const __nv_bfloat16*)in.b; ar.Ts = pr.Ts;
  ar.A_log = in.A_log; ar.dt_bias = in.dt_bias; ar.valid_len = in.valid_len;
  ar.rec = (uint8_t*)ws.tu; ar.status = ws.status;
  cudaError_t e = smem_attr_fwd(k_tsolve, TS_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)pr.NC, (unsigned)pr.Hqk, (unsigned)pr.B);
  k_tsolve<<<grid, TS_THREADS, TS_SMEM, st>>>(mk, mq, ar);
  return cudaGetLastError();
}

cudaError_t launch_fwd_tc(const Prob& pr, const Inputs& in, const WS& ws, const FwdWork& w,
                          cudaStream_t st) {
  if (pr.B == 0 || pr.NC == 0 || w.nitems <= 0) return cudaSuccess;
  if (w.nitems > kMaxItems) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  const void* qptr = in.q ? in.q : in.k;  // summaries never read q
  const void* vptr = in.v ? in.v : in.k;  // transitions never read v
  if (!tc_make_map(&mq, qptr, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(&mk, in.k, pr.B, pr.T, pr.Ts, pr.Hqk) ||
      !tc_make_map(&mv, vptr, pr.B, pr.T, pr.Ts, in.v ? pr.H : pr.Hqk))
    return cudaErrorInvalidValue;
  FwdArgs ar;
  memset(&ar, 0, sizeof(ar));
  ar.T = pr.T; ar.Ts = pr.Ts; ar.H = pr.H; ar.Hqk = pr.Hqk; ar.r = pr.r; ar.NC = pr.NC;
  ar.NCtot = pr.B * pr.NC; ar.CPS = pr.CPS; ar.P = pr.P;
  ar.valid_len = in.valid_len;
  ar.rec = (const uint8_t*)ws.tu;
  ar.init = w.init; ar.init_stride = w.init_stride; ar.init0 = w.init0;
  ar.o = (__nv_bfloat16*)w.o; ar.final_out = w.final_out;
  ar.S_out = w.S_out; ar.M_out = w.M_out; ar.out_stride = w.out_stride;
  ar.status = ws.status;
  ar.nitems = w.nitems;
  for (int i = 0; i < w.nitems; ++i) {
    ar.items[i].mode = w.mode[i];
    ar.items[i].seg = w.seg[i];
  }
  cudaError_t e = smem_attr_fwd(k_fwd_tc, F_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)w.nitems, (unsigned)pr.H, (unsigned)pr.B);
  k_fwd_tc<<<grid, FW_THREADS, F_SMEM, st>>>(mq, mk, mv, ar);
  return cudaGetLastError();
}

}  // namespace gdn
