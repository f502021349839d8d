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
// Shared memory: thirteen 16 KB slots (the state S always in slots 4-5; P and T share
// slot 10) whose roles alternate between two layouts from one chunk to the next, so
// that every input tile of the next chunk lands in a slot the current chunk has
// already finished with (see k_grad2_tc), then the scalars.
constexpr uint32_t SLOT = 16384;
constexpr uint32_t R_SC = 13 * SLOT;  // scalars
constexpr uint32_t SC_BYTES = 2 * 4 * 64 * 4 + 3 * 64 * 4 + 4 * 4 * 64 * 4 + 3 * 4 * 64 * 4 +
                               2 * 128 * 4 + 128;
constexpr uint32_t GR_SMEM = R_SC + SC_BYTES + 1024;
static_assert(GR_SMEM <= 232448, "shared memory of k_grad2_tc");

// Byte offsets of the tiles of one chunk.  q, k: q_hat, k_hat [tok][dk] (two 8 KB atoms,
// normalised in place); v, dO: [tok][dv] (dO later the dv staging); s: S image [dk][dv]
// (two [128][64] atoms 16 KB apart); ds0, ds1: the two atoms of the dS image (later the
// dq_hat and dk_hat staging); w: W [tok][dk], later dW^T [dk][tok]; u: U [tok][dv], later
// X_v^T; p: P, later dP o Gamma; t: T, later E; vt, dvt: V'^T and dV'^T [dv][tok].
struct Lay {
  uint32_t q, k, v, dO, s, ds0, ds1, w, u, p, t, vt, dvt;
};
// Layout 0 (even chunks of a CTA) and 1 (odd chunks).  Going 0 -> 1 the next chunk's
// dO goes where dV'^T was (free once round B is done), its U where V was (after round
// B's epilogue), its dS where U and V'^T were and its W where dW^T was (after round C),
// its V where the dv staging was (after the dv store); 1 -> 0 mirrors it.
__device__ __forceinline__ Lay layout_of(int par) {
  Lay L;
  L.q = 0;
  L.k = SLOT;
  L.s = 4 * SLOT;
  L.w = 8 * SLOT;
  L.p = 10 * SLOT;
  L.t = 10 * SLOT + 8192;
  if (par == 0) {
    L.v = 2 * SLOT; L.dO = 3 * SLOT; L.ds0 = 6 * SLOT; L.ds1 = 7 * SLOT;
    L.u = 9 * SLOT; L.vt = 11 * SLOT; L.dvt = 12 * SLOT;
  } else {
    L.u = 2 * SLOT; L.v = 3 * SLOT; L.vt = 6 * SLOT; L.dvt = 7 * SLOT;
    L.ds0 = 9 * SLOT; L.ds1 = 11 * SLOT; L.dO = 12 * SLOT;
  }
  return L;
}

struct Grad2Args {
  int64_t T, Ts, H, r, NC, Tp, NW;  // NW = B * H * NC chunks of work
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
  const float* rqk;    // [B][Hqk][NC][128] q, k row factors of the prologue (rq with the scale)
  const float* gl;     // [B][H][NC][64] cumulative gates of the prologue (log2 units)
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

// Transpose-reduce of p[16] within each 16-lane half of the warp: lane l ends with the
// sum over its half of p[l & 15] (15 shuffles).
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
__device__ __forceinline__ float xreduce_half(float (&p)[16], int lane) {
  xr_stage<8>(p, lane);
  xr_stage<4>(p, lane);
  xr_stage<2>(p, lane);
  xr_stage<1>(p, lane);
  return p[0];
}
// Over the whole warp: lanes l and l ^ 16 both end with the sum of p[l & 15].
__device__ __forceinline__ float xreduce16(float (&p)[16], int lane) {
  const float x = xreduce_half(p, lane);
  return x + __shfl_xor_sync(0xffffffffu, x, 16);
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

// Persistent: grid min(NW, SMs) x 512 threads, one CTA per SM; CTA i takes chunks
// i, i + gridDim.x, ... (chunk w: c = w % NC, h = (w / NC) % H, b = w / (NC H)) and,
// while it works on one, copies the next one's tiles into the slots it has freed.
// Warp w reads TMEM lane quadrant q = w & 3 and token columns 16 (w >> 2) .. +15.  In
// an M = 128 result thread (q, lane) owns feature row 32 q + lane; in an M = 64 result
// (row r in lane (r % 16) + 32 (r / 16)) lanes 0..15 of quadrant q own token row 16 q + lane.
__global__ void __launch_bounds__(GT, 1)
    k_grad2_tc(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
               const __grid_constant__ CUtensorMap mdv, const __grid_constant__ CUtensorMap mdqp,
               const __grid_constant__ CUtensorMap mdkp, Grad2Args ar) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t base = smem_u32(sm);
  // per chunk, two buffers (chunk k uses buffer k & 1): cumulative gate G (log2 units),
  // gamma = 2^G, beta, Kt = 2^(G_C - G)
  float* sGate = (float*)(sm + R_SC);
  float* sDB = sGate + 2 * 256;        // dbeta (final)
  float* sFin = sDB + 64;              // final dG
  float* sMisc = sFin + 64;            // [16] warp partials of <S, dS>
  float* sRed = sMisc + 64;            // [4 types][4 quadrants][64 tokens] column partials
  float* sDBh = sRed + 4 * 4 * 64;     // [4 column parts][64] dbeta terms of A
  float* sZr = sDBh + 4 * 64;          // [4 column parts][64 rows] row sums of dP o P + dA o A
  float* sZc = sZr + 4 * 64;           // [4 row quadrants][64 columns] their column sums
  float* sRqk = sZc + 4 * 64;          // per layout: rq (64), rk (64) of the chunk's q, k rows
  uint64_t* bars = (uint64_t*)(sRqk + 2 * 128);  // per layout: q/k, round-A tiles, U/V/T; MMA
  uint64_t* bar_mma = bars + 6;
  uint64_t* bar_g = bars + 7;          // per layout: the chunk's cumulative gates G
  uint32_t* s_tmem = (uint32_t*)(bars + 9);
  int* s_abort = (int*)(s_tmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, part = warp >> 2;
  const int fr = quad * 32 + lane;     // feature row (TMEM lane) of M = 128 results
  const int cb = 16 * part;            // first token column of this thread
  const bool own64 = lane < 16;        // owns row ri of M = 64 results
  const int ri = quad * 16 + (lane & 15);
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const bool issuer = warp < 5 && lane == 0;  // issues one product per MMA round
  const bool mover = tid == 160;  // issues every tile copy and store (warp 5: no MMA issue)
  enum { RQ = 0, RV = 1, RKW = 2, RKD = 3 };  // column-sum types
  enum { GQK = 0, GA = 1, GB = 2 };            // load groups
  uint32_t armed = 0;  // the arming thread (the mover; warp 6 for q, k and G): bit 3 l + g,
                       // group g of layout l armed and not yet consumed; bit 6 + l, the G copy
                       // of layout l

  if (tid == 0) {
    for (int i = 0; i < 6; ++i) mbar_init(bars + i, 1);
    mbar_init(bar_g, 1);
    mbar_init(bar_g + 1, 1);
    mbar_init(bar_mma, 5);  // each round's products are issued from five warps (lane 0 of 0..4)
    fence_barrier_init();
    *s_abort = 0;
  }
  if (warp == 0) tmem_alloc(s_tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  // Descriptors of every operand tile: the start address sits in the low 14 bits
  // (address >> 4), so a tile at byte offset `off` is the base descriptor + off / 16.
  const uint64_t d16 = sdesc(base, 16, 1024), d8192 = sdesc(base, 8192, 1024),
                 d16384 = sdesc(base, 16384, 1024);
  auto dsc16 = [&](uint32_t off) { return d16 + (off >> 4); };
  auto dsc8192 = [&](uint32_t off) { return d8192 + (off >> 4); };
  auto dsc16384 = [&](uint32_t off) { return d16384 + (off >> 4); };
  const uint32_t idA = idesc_bf16(128, 64, 1, 0);  // A MN-major (feature rows), B K-major
  const uint32_t idB = idesc_bf16(128, 64, 0, 1);  // A K-major, B MN-major
  const uint32_t idC = idesc_bf16(128, 64, 1, 1);  // both MN-major
  const uint32_t idD = idesc_bf16(128, 64, 0, 0);  // both K-major
  uint32_t ph = 0;                                 // parity of bar_mma

  // ---- tile copies of chunk w into layout `lay` (tid 0)
  struct Item {
    int64_t c, h, b, hq, im, t0;
  };
  // chunk w: 32-bit index arithmetic (the host keeps NW below 2^31; 64-bit division costs
  // ~80 instructions, and every thread runs this twice per chunk)
  auto item_of = [&](int64_t w) {
    Item it;
    const uint32_t uw = (uint32_t)w, q1 = uw / (uint32_t)ar.NC, hh = q1 % (uint32_t)ar.H;
    it.c = uw - q1 * (uint32_t)ar.NC;
    it.h = hh;
    it.b = q1 / (uint32_t)ar.H;
    it.hq = hh / (uint32_t)ar.r;
    it.im = (it.b * ar.H + it.h) * ar.NC + it.c;
    it.t0 = it.c * 64;
    return it;
  };
  auto arm = [&](int l, int g, uint32_t bytes) {
    mbar_arrive_expect_tx(bars + 3 * l + g, bytes);
    armed |= 1u << (3 * l + g);
  };
  auto tile2 = [&](uint32_t dst, const CUtensorMap* m, int64_t head, const Item& it, uint64_t* bar) {
    for (int at = 0; at < 2; ++at)
      tma_load_4d(sm + dst + at * 8192, m, at * 64, (int)head, (int)it.t0, (int)it.b, bar);
  };
  auto ld_qk = [&](const Item& it, const Lay& L, int l) {  // q, k tiles and their row factors
    arm(l, GQK, 2 * 16384u + 512u);
    tile2(L.q, &mq, it.hq, it, bars + 3 * l + GQK);
    tile2(L.k, &mk, it.hq, it, bars + 3 * l + GQK);
    bulk_load(sRqk + l * 128, ar.rqk + ((it.b * (ar.H / ar.r) + it.hq) * ar.NC + it.c) * 128, 512,
              bars + 3 * l + GQK);
  };
  auto ld_s = [&](const Item& it, const Lay& L, int l) {
    bulk_load(sm + L.s, ar.hc + it.im * 32768, 32768, bars + 3 * l + GA);
  };
  auto ld_ds = [&](const Item& it, const Lay& L, int l) {
    bulk_load(sm + L.ds0, ar.dhc + it.im * 32768, 16384, bars + 3 * l + GA);
    bulk_load(sm + L.ds1, ar.dhc + it.im * 32768 + 16384, 16384, bars + 3 * l + GA);
  };
  auto ld_w = [&](const Item& it, const Lay& L, int l) {
    bulk_load(sm + L.w, ar.wim + it.im * 16384, 16384, bars + 3 * l + GA);
  };
  auto ld_do = [&](const Item& it, const Lay& L, int l) { tile2(L.dO, &mdo, it.h, it, bars + 3 * l + GA); };
  auto ld_p = [&](const Item& it, const Lay& L, int l) {
    bulk_load(sm + L.p, ar.pim + it.im * 8192, 8192, bars + 3 * l + GA);
  };
  auto ld_u = [&](const Item& it, const Lay& L, int l) {
    bulk_load(sm + L.u, ar.uim + it.im * 16384, 16384, bars + 3 * l + GB);
  };
  auto ld_t = [&](const Item& it, const Lay& L, int l) {
    bulk_load(sm + L.t, ar.tim + it.im * 8192, 8192, bars + 3 * l + GB);
  };
  auto ld_v = [&](const Item& it, const Lay& L, int l) { tile2(L.v, &mv, it.h, it, bars + 3 * l + GB); };
  constexpr uint32_t kBytesA = 32768u + 32768u + 16384u + 16384u + 8192u;  // S, dS, W, dO, P
  constexpr uint32_t kBytesB = 16384u + 8192u + 16384u;                    // U, T, V

  // Gates of a chunk in buffer dst (G, gamma, beta, Kt at 0, 64, 128, 192): G, the cumulative
  // gate in log2 units, is the prologue's (copied in by warp 6, on bar_g); warps 14 and 15
  // (token = tid - 448: no MMA issue, no copies) form gamma = 2^G, beta = sigmoid(b) and
  // Kt = 2^(G_C - G) from it.
  // Their b input is read early into a register so that its latency stays off the chunk's
  // critical path.
  struct GateIn {
    float xb;
    bool live;
  };
  auto gate_in = [&](const Item& it) {
    const int t = tid - 448;
    int64_t Lg = ar.T;
    if (ar.valid_len) {
      Lg = ar.valid_len[it.b];
      if (Lg < 0 || Lg > ar.T) Lg = Lg < 0 ? 0 : ar.T;
    }
    GateIn gi{0.f, it.t0 + t < Lg};
    if (gi.live) gi.xb = __bfloat162float(ar.b[(it.b * ar.Ts + it.t0 + t) * ar.H + it.h]);
    return gi;
  };
  auto ld_g = [&](const Item& it, int l) {  // mover: the chunk's G into buffer l
    armed |= 1u << (6 + l);
    mbar_arrive_expect_tx(bar_g + l, 256);
    bulk_load(sGate + l * 256, ar.gl + it.im * 64, 256, bar_g + l);
  };
  auto gates = [&](const GateIn& gi, float* dst) {
    const int t = tid - 448;
    const float G = dst[t];
    dst[64 + t] = exp2f(G);
    dst[128 + t] = gi.live ? 1.f / (1.f + expf(-gi.xb)) : 0.f;
    dst[192 + t] = dexp_(dst[63], G);
  };

  // The CTA's chunks, skipping those of padding only (from ceil(valid_len / 64) on: the
  // chains and the prologue skip them too; their outputs are zeroed by a separate pass).
  auto next_live = [&](int64_t w) {
    for (; w < ar.NW; w += gridDim.x) {
      if (!ar.valid_len) break;
      const uint32_t uw = (uint32_t)w, q1 = uw / (uint32_t)ar.NC;
      int64_t Lb = ar.valid_len[q1 / (uint32_t)ar.H];
      Lb = Lb < 0 ? 0 : (Lb > ar.T ? ar.T : Lb);
      if ((int64_t)(uw - q1 * (uint32_t)ar.NC) * 64 < Lb) break;
    }
    return w;
  };
  const int64_t w0 = next_live(blockIdx.x);
  GateIn gnext{0.f, false};  // warps 14, 15: b of the next chunk's gates
  if (warp >= 14 && w0 < ar.NW) {
    const Item it0 = item_of(w0);
    const GateIn g0 = gate_in(it0);
    if (!mbar_wait(bar_g, 0, ar.status, kStatusTimeout)) *s_abort = 1;
    gates(g0, sGate);
  }
  if (tid == 192 && w0 < ar.NW) ld_g(item_of(w0), 0);  // (warp 6 arms every G copy)
  if (mover && w0 < ar.NW) {  // every tile of the first chunk
    const Item it = item_of(w0);
    const Lay L = layout_of(0);
    ld_qk(it, L, 0);
    arm(0, GA, kBytesA);
    ld_s(it, L, 0);
    ld_w(it, L, 0);
    ld_ds(it, L, 0);
    ld_do(it, L, 0);
    ld_p(it, L, 0);
    arm(0, GB, kBytesB);
    ld_u(it, L, 0);
    ld_t(it, L, 0);
    ld_v(it, L, 0);
  }

  for (int64_t w = w0, wn = 0, k = 0; w < ar.NW; w = wn, ++k) {
    const int lc = (int)(k & 1), ln = lc ^ 1;
    const uint32_t bpar = (uint32_t)((k >> 1) & 1);  // phase parity of this layout's barriers
    const Lay L = layout_of(lc);
    const Lay N = layout_of(ln);
    const Item it = item_of(w);
    wn = next_live(w + gridDim.x);
    const bool more = wn < ar.NW;
    const Item nx = item_of(more ? wn : w);
    const int64_t h = it.h, b = it.b, t0 = it.t0;
    int64_t L_len = ar.T;
    if (ar.valid_len) {
      L_len = ar.valid_len[b];
      if (L_len < 0 || L_len > ar.T) L_len = L_len < 0 ? 0 : ar.T;
    }
    const uint32_t dsl = L.ds1 - L.ds0;  // atom stride of the dS image
    const uint64_t dds = sdesc(base, dsl, 1024);
    auto dscDS = [&](uint32_t off) { return dds + (off >> 4); };

    float* sG = sGate + lc * 256;  // this chunk's gates (written during the previous chunk)
    float* sGam = sG + 64;
    float* sBeta = sG + 128;
    float* sKt = sG + 192;
    __syncthreads();  // the previous chunk's scalars have been consumed, these gates written
    if (tid == 192) {  // this chunk's G has landed (warps 14, 15 waited for it); the next G
      if (mbar_wait(bar_g + lc, bpar, ar.status, kStatusTimeout)) armed &= ~(1u << (6 + lc));
      if (more) ld_g(nx, ln);  // into the other buffer, free since the previous chunk ended
    }
    if (mover && k > 0) {  // tiles of this chunk that waited for the previous stores
      bulk_wait_read();  // the previous chunk's dv, dq, dk stores have read their slots
      if (lc == 1)
        ld_v(it, L, lc);  // where the dv staging was
      else
        ld_u(it, L, lc);  // where the dq staging was
    }
    if (!mbar_wait(bars + 3 * lc + GQK, bpar, ar.status, kStatusTimeout)) *s_abort = 1;
    // q, k rows scaled in place by the prologue's row factors (rq = scale / |q| or the scale
    // alone, rk = 1 / |k| or 1; rows 0..63 of the factors are q's, 64..127 k's), 16 threads
    // per row; padded dO rows zeroed
    {
      const float* sR = sRqk + lc * 128;
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        const int rr = (tid >> 4) + 32 * i4;  // q rows, then k rows
        const int sub = tid & 15, at = sub >> 3, ch = sub & 7, r6 = rr & 63;
        const uint32_t off = (rr >= 64 ? L.k : L.q) + at * 8192 + kmaj_chunk(r6, ch);
        const float f = sR[rr];
        float x[8];
        ld_chunk(sm, off, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= f;  // (fp32 product, one rounding)
        st_chunk(sm, off, x);
      }
    }
    if (!mbar_wait(bars + 3 * lc + GA, bpar, ar.status, kStatusTimeout)) *s_abort = 1;
    armed &= ~((1u << (3 * lc + GQK)) | (1u << (3 * lc + GA)));
    if (t0 + 64 > L_len) {
      for (int idx = tid; idx < 1024; idx += GT) {
        const int i = idx >> 4, cc = idx & 15;
        if (t0 + i >= L_len)
          *reinterpret_cast<uint4*>(sm + L.dO + (cc >> 3) * 8192 + kmaj_chunk(i, cc & 7)) = make_uint4(0, 0, 0, 0);
      }
    }
    float dqT[16], dkT[16];  // this thread's feature row fr of dq_hat^T, dk_hat^T, tokens cb + e
    GRAD_SYNC();
    // ---- round A: S^T W^T -> [0,64), dO^T P -> [64,128), dS^T K^T -> [128,192),
    //      S dO^T -> [192,256), K K^T -> [256,320) (M = 64; read in round C's epilogue)
    // (one thread per product, five warps: a single thread issues tcgen05.mma at a far lower
    // rate than the tensor core retires these small shapes)
    if (issuer) {
      if (warp == 0) {
        for (int ks = 0; ks < 8; ++ks)  // K = dk
          mma_bf16(tmem, dsc16384(L.s + ks * 2048), dsc16(L.w + (ks >> 2) * 8192 + (ks & 3) * 32),
                   idA, ks > 0);
      } else if (warp == 1) {
        for (int ks = 0; ks < 8; ++ks)  // K = dk
          mma_bf16(tmem + 128, dscDS(L.ds0 + ks * 2048),
                   dsc16(L.k + (ks >> 2) * 8192 + (ks & 3) * 32), idA, ks > 0);
      } else if (warp == 2) {
        for (int ks = 0; ks < 8; ++ks)  // K = dv
          mma_bf16(tmem + 192, dsc16(L.s + (ks >> 2) * 16384 + (ks & 3) * 32),
                   dsc16(L.dO + (ks >> 2) * 8192 + (ks & 3) * 32), idD, ks > 0);
      } else if (warp == 3) {
        const uint32_t id64d = idesc_bf16(64, 64, 0, 0);
        for (int ks = 0; ks < 8; ++ks) {  // K = dk
          const uint64_t d = dsc16(L.k + (ks >> 2) * 8192 + (ks & 3) * 32);
          mma_bf16(tmem + 256, d, d, id64d, ks > 0);
        }
      } else {
        for (int ks = 0; ks < 4; ++ks)  // K = tokens
          mma_bf16(tmem + 64, dsc8192(L.dO + ks * 2048), dsc8192(L.p + ks * 2048), idC, ks > 0);
      }
      mma_commit(bar_mma);
    }
    {  // <S, dS> (same tile layout): warp partials into sMisc, from warps 6.. only (the
       // round's issuers wait on the tensor core's queue and warp 5 issues the copies; their
       // partials are zero)
      float acc = 0.f;
      for (int q = tid - 192; q >= 0 && q < 2048; q += GT - 192) {
        float x[8], y[8];
        ld_chunk(sm + L.s, q * 16, x);
        ld_chunk(sm + ((q < 1024) ? L.ds0 : L.ds1) + (q & 1023) * 16, 0, y);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(x[e], y[e], acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) sMisc[warp] = acc;
    }
    if (!mbar_wait(bars + 3 * lc + GB, bpar, ar.status, kStatusTimeout)) *s_abort = 1;
    armed &= ~(1u << (3 * lc + GB));
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    {  // V'^T and dV'^T: the operands of round B
      const int f = fr;
      float ws[16], a1[16], a2[16];
      tmem_ld16x4(tmem + lane_off + cb, tmem + lane_off + 64 + cb, tmem + lane_off + 128 + cb,
                  tmem + lane_off + 192 + cb, ws, a1, a2, dqT);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        ws[e] = ld_bf(sm + L.u + tf_off(t, f)) - ws[e];   // V'^T
        a1[e] = fmaf(sKt[t], a2[e], a1[e]);                // dV'^T
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        st_chunk(sm + L.vt, kmaj_chunk(f, 2 * part + cc), &ws[cc * 8]);
        st_chunk(sm + L.dvt, kmaj_chunk(f, 2 * part + cc), &a1[cc * 8]);
      }
    }
    if (mover) bulk_wait_read();  // the previous chunk's dq/dk/dv stores have read their slots
    GRAD_SYNC();
    // ---- round B: S dV'^T -> [0,64) (-dW^T), dS V'^T -> [64,128), dV'^T T -> [128,192) (X_v^T),
    //      dO V'^T -> [192,256) (dP, M = 64)
    if (issuer) {
      if (warp == 0) {
        for (int ks = 0; ks < 8; ++ks)  // K = dv
          mma_bf16(tmem, dsc16(L.s + (ks >> 2) * 16384 + (ks & 3) * 32),
                   dsc8192(L.dvt + ks * 2048), idB, ks > 0);
      } else if (warp == 1) {
        for (int ks = 0; ks < 8; ++ks)  // K = dv
          mma_bf16(tmem + 64, dsc16(((ks >> 2) ? L.ds1 : L.ds0) + (ks & 3) * 32),
                   dsc8192(L.vt + ks * 2048), idB, ks > 0);
      } else if (warp == 2) {
        const uint32_t id64b = idesc_bf16(64, 64, 0, 1);
        for (int ks = 0; ks < 8; ++ks)  // K = dv
          mma_bf16(tmem + 192, dsc16(L.dO + (ks >> 2) * 8192 + (ks & 3) * 32),
                   dsc8192(L.vt + ks * 2048), id64b, ks > 0);
      } else if (warp == 3) {
        for (int ks = 0; ks < 4; ++ks)  // K = tokens
          mma_bf16(tmem + 128, dsc16(L.dvt + ks * 32), dsc8192(L.t + ks * 2048), idB, ks > 0);
      }
      mma_commit(bar_mma);
    }
    if (more && warp >= 14) gnext = gate_in(nx);  // lands before the tail
    {  // while round B runs: (diag(gamma) dO S^T)^T and q_t . (gamma_t S dO_t)
      const int f = fr;
      float pq[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        dqT[e] *= sGam[t];
        pq[e] = ld_bf(sm + L.q + tf_off(t, f)) * dqT[e];
      }
      const float red = xreduce16(pq, lane);
      if (lane < 16) sRed[(RQ * 4 + quad) * 64 + cb + lane] = red;
    }
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    if (mover && more) {  // S and dV'^T are consumed: the next chunk's S (and dO)
      arm(ln, GA, kBytesA);
      ld_s(nx, N, ln);
      if (lc == 0) ld_do(nx, N, ln);
    }
    {  // -dW^T, X_v^T and dP o Gamma: the operands of round C
      const int f = fr;
      // S dV'^T = -dW^T, X_v^T and dP (M = 64 layout)
      float x[16], xv[16], dp[16], z[16];
      tmem_ld16x3(tmem + lane_off + cb, tmem + lane_off + 128 + cb, tmem + lane_off + 192 + cb, x,
                  xv, dp);
#pragma unroll
      for (int e = 0; e < 16; ++e) x[e] = -x[e];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) st_chunk(sm + L.w, kmaj_chunk(f, 2 * part + cc), &x[cc * 8]);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) st_chunk(sm + L.u, kmaj_chunk(f, 2 * part + cc), &xv[cc * 8]);
      const int i = ri;
      float pv[16];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) ld_chunk(sm + L.p, kmaj_chunk(i, 2 * part + cc), &pv[cc * 8]);
      float zr = 0.f;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = cb + cc * 8 + e;
          const float dpv = (own64 && j <= i) ? dp[cc * 8 + e] : 0.f;
          z[cc * 8 + e] = dpv * pv[cc * 8 + e];                  // dP o P
          zr += z[cc * 8 + e];
          y[e] = (j <= i) ? dpv * dexp_(sG[i], sG[j]) : 0.f;    // dP o Gamma
        }
        if (own64) st_chunk(sm + L.p, kmaj_chunk(i, 2 * part + cc), y);  // over P (this thread's)
      }
      const float zc = xreduce_half(z, lane);  // column cb + lane of dP o P over this quadrant's rows
      if (own64) {
        sZr[part * 64 + i] = zr;
        sZc[quad * 64 + cb + lane] = zc;
      }
    }
    GRAD_SYNC();
    // ---- round C: dW^T T -> [320,384) (X_w^T), K^T (dP o Gamma)^T -> [384,448),
    //      X_v V'^T -> [448,512) (dA', M = 64); K K^T stays in [256,320)
    if (issuer) {
      if (warp == 0) {
        for (int ks = 0; ks < 4; ++ks)  // K = tokens
          mma_bf16(tmem + 320, dsc16(L.w + ks * 32), dsc8192(L.t + ks * 2048), idB, ks > 0);
      } else if (warp == 1) {
        for (int ks = 0; ks < 4; ++ks)  // K = tokens
          mma_bf16(tmem + 384, dsc8192(L.k + ks * 2048), dsc16(L.p + ks * 32), idA, ks > 0);
      } else if (warp == 2) {
        const uint32_t id64c = idesc_bf16(64, 64, 1, 1);
        for (int ks = 0; ks < 8; ++ks)  // K = dv
          mma_bf16(tmem + 448, dsc8192(L.u + ks * 2048), dsc8192(L.vt + ks * 2048), id64c, ks > 0);
      }
      mma_commit(bar_mma);  // warps 3, 4 have nothing to issue: their commits arrive at once
    }
    {  // while round C runs: Kt part of dk, dv, and the row dots of V' dS^T and X_v
      const int f = fr;
      float x[16], xv[16], pk[16];
      tmem_ld16x2(tmem + lane_off + 64 + cb, tmem + lane_off + 128 + cb, x, xv);  // (V' dS^T)^T, X_v^T
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        dkT[e] = sKt[t] * x[e];
        pk[e] = ld_bf(sm + L.k + tf_off(t, f)) * x[e];    // k_t . (V' dS^T)_t
      }
      float red = xreduce16(pk, lane);
      if (lane < 16) sRed[(RKD * 4 + quad) * 64 + cb + lane] = red;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        pk[e] = ld_bf(sm + L.v + tf_off(t, f)) * xv[e];   // v_t . X_v,t
        st_bf(sm + L.dO + tf_off(t, f), (t0 + t < L_len) ? sBeta[t] * xv[e] : 0.f);  // dv staging
      }
      red = xreduce16(pk, lane);
      if (lane < 16) sRed[(RV * 4 + quad) * 64 + cb + lane] = red;
    }
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    if (mover && more) {  // dW^T, X_v^T and V'^T (and dV'^T) are consumed: next W and dS
      ld_w(nx, N, ln);
      ld_ds(nx, N, ln);
      if (lc == 1) {
        arm(ln, GB, kBytesB);
        ld_v(nx, N, ln);
      }
    }
    {  // E (operand of round D), dA o A, dbeta terms of A
      float da[16], kk[16], z[16];
      tmem_ld16x2(tmem + lane_off + 448 + cb, tmem + lane_off + 256 + cb, da, kk);  // dA', K K^T (M = 64)
      const int i = ri;
      const float be = sBeta[i];
      float pt = 0.f, zr = 0.f;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float ex[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = cb + cc * 8 + e;
          const bool lo = own64 && j < i;
          const float gmm = lo ? dexp_(sG[i], sG[j]) : 0.f;
          const float dA = lo ? -da[cc * 8 + e] : 0.f;
          const float kg = kk[cc * 8 + e] * gmm;
          pt = fmaf(dA, kg, pt);                       // dbeta: dA (k_i . k_j) Gamma
          z[cc * 8 + e] = dA * be * kg;                // dA o A
          zr += z[cc * 8 + e];
          ex[e] = dA * be * gmm;                       // E
        }
        if (own64) st_chunk(sm + L.t, kmaj_chunk(i, 2 * part + cc), ex);   // E over T
      }
      const float zc = xreduce_half(z, lane);
      if (own64) {
        sDBh[part * 64 + i] = pt;
        sZr[part * 64 + i] += zr;
        sZc[quad * 64 + cb + lane] += zc;
      }
    }
    GRAD_SYNC();
    // ---- round D: Q^T (dP o Gamma) -> [0,64), K^T E^T -> [64,128), K^T E -> [128,192)
    //      (three products from three warps, summed in the epilogue)
    if (mover) {
      tma_store_4d(&mdv, sm + L.dO, 0, (int)h, (int)t0, (int)b);  // dv tile (clipped past T)
      tma_store_4d(&mdv, sm + L.dO + 8192, 64, (int)h, (int)t0, (int)b);
      bulk_commit();
    }
    if (issuer) {
      if (warp == 0) {
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem, dsc8192(L.q + ks * 2048), dsc8192(L.p + ks * 2048), idC, ks > 0);
      } else if (warp == 1) {
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + 64, dsc8192(L.k + ks * 2048), dsc16(L.t + ks * 32), idA, ks > 0);
      } else if (warp == 2) {
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + 128, dsc8192(L.k + ks * 2048), dsc8192(L.t + ks * 2048), idC, ks > 0);
      }
      mma_commit(bar_mma);
    }
    if (mover) {
      if (more && lc == 0) {  // V (read before the last barrier) is consumed: the next U
        arm(ln, GB, kBytesB);
        ld_u(nx, N, ln);
      }
      if (more && lc == 1) ld_do(nx, N, ln);  // ... and, the other way round, the next dO
    }
    {  // while round D runs: X_w part of dk, dq_hat staging, row dots of X_w
      const int f = fr;
      float x[16], xd[16], pk[16];
      tmem_ld16x2(tmem + lane_off + 320 + cb, tmem + lane_off + 384 + cb, x, xd);  // X_w^T, ((dP o Gamma) K)^T
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        const float bg = sBeta[t] * sGam[t];
        dkT[e] = fmaf(bg, x[e], dkT[e]);
        pk[e] = ld_bf(sm + L.k + tf_off(t, f)) * x[e];    // k_t . X_w,t
      }
      const float red = xreduce16(pk, lane);
      if (lane < 16) sRed[(RKW * 4 + quad) * 64 + cb + lane] = red;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        st_bf(sm + L.ds0 + tf_off(t, f), (t0 + t < L_len) ? dqT[e] + xd[e] : 0.f);  // dq_hat staging
      }
    }
    if (!mbar_wait(bar_mma, ph, ar.status, kStatusTimeout)) *s_abort = 1;
    ph ^= 1;
    tc_fence_after();
    if (mover && more) {  // P (dP o Gamma) and T (E) are consumed
      ld_p(nx, N, ln);
      ld_t(nx, N, ln);
    }
    {
      const int f = fr;
      float x[16], y[16], z3[16];
      tmem_ld16x3(tmem + lane_off + cb, tmem + lane_off + 64 + cb, tmem + lane_off + 128 + cb, x, y,
                  z3);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = cb + e;
        st_bf(sm + L.ds1 + tf_off(t, f), (t0 + t < L_len) ? dkT[e] + x[e] + y[e] + z3[e] : 0.f);  // dk_hat
      }
    }
    GRAD_SYNC();
    if (mover) {
      tma_store_4d(&mdqp, sm + L.ds0, 0, (int)h, (int)t0, (int)b);  // dq_hat tile
      tma_store_4d(&mdqp, sm + L.ds0 + 8192, 64, (int)h, (int)t0, (int)b);
      tma_store_4d(&mdkp, sm + L.ds1, 0, (int)h, (int)t0, (int)b);
      tma_store_4d(&mdkp, sm + L.ds1 + 8192, 64, (int)h, (int)t0, (int)b);
      bulk_commit();
    } else if (tid == 192 && more) {  // q and k are consumed (round D and the dots above): the
      ld_qk(nx, N, ln);                // next ones from warp 6, which arms and drains them
    }
    // ---- gate gradients: column sums of the four row dots, Kt terms, state term; the
    //      next chunk's gates meanwhile (warps 14, 15)
    if (tid < 64) {
      const int t = tid;
      float rq = 0.f, rv = 0.f, rkw = 0.f, rkd = 0.f, zp = 0.f;
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        rq += sRed[(RQ * 4 + qd) * 64 + t];
        rv += sRed[(RV * 4 + qd) * 64 + t];
        rkw += sRed[(RKW * 4 + qd) * 64 + t];
        rkd += sRed[(RKD * 4 + qd) * 64 + t];
        zp += sZr[qd * 64 + t] - sZc[qd * 64 + t];  // row sums minus column sums of Z
      }
      const float be = sBeta[t], gm = sGam[t];
      const float s_t = sKt[t] * rkd;                       // Kt term of dG_t
      float d = zp + rq + be * gm * rkw;
      if (t < 63) d -= s_t;
      sFin[t] = d;
      sDB[t] = rv + gm * rkw + sDBh[t] + sDBh[64 + t] + sDBh[128 + t] + sDBh[192 + t];
      sRed[t] = (t < 63) ? s_t : 0.f;                       // reuse: Kt terms to sum into dG_C
    } else if (more && warp >= 14) {
      if (!mbar_wait(bar_g + ln, (uint32_t)(((k + 1) >> 1) & 1), ar.status, kStatusTimeout))
        *s_abort = 1;
      gates(gnext, sGate + ln * 256);
    }
    __syncthreads();
    if (tid < 32) {  // dG_C gets the Kt terms and the state term; then dg_j = sum_{i >= j} dG_i
      float tot = sRed[tid] + sRed[32 + tid], sd = tid < GT / 32 ? sMisc[tid] : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        sd += __shfl_xor_sync(0xffffffffu, sd, o);
      }
      float v0 = sFin[63 - tid], v1 = sFin[31 - tid];
      if (tid == 0) v0 += tot + sGam[63] * sd;
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
      sFin[63 - tid] = v0;
      sFin[31 - tid] = v1;
    }
    __syncthreads();
    if (tid < 64) {
      const int64_t t = t0 + tid;
      if (t < ar.T) {
        const int64_t gi = (b * ar.Ts + t) * ar.H + h;
        const bool valid = t < L_len;
        ar.dg[gi] = valid ? sFin[tid] : 0.f;   // natural-log units (log2 only enters exponents)
        ar.dbeta[gi] = valid ? sDB[tid] : 0.f;
      }
    }
  }
done:
  if (mover) bulk_wait_all();
  if (armed) {  // abort: let every copy still in flight land before the CTA exits
    for (int i = 0; i < 8; ++i)
      if (armed & (1u << i)) {
        // one of the two parities is the phase in flight; the other returns at once
        uint64_t* bar = i < 6 ? bars + i : bar_g + (i - 6);
        mbar_wait(bar, 0, nullptr, 0);
        mbar_wait(bar, 1, nullptr, 0);
      }
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
  ar.NW = pr.B * pr.H * pr.NC;
  if (ar.NW + 1024 >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;  // 32-bit chunk indices
  ar.l2norm = pr.l2norm; ar.eps = pr.eps; ar.scale = pr.scale;
  ar.a = (const __nv_bfloat16*)in.a; ar.b = (const __nv_bfloat16*)in.b;
  ar.A_log = in.A_log; ar.dt_bias = in.dt_bias; ar.valid_len = in.valid_len;
  ar.dg = dg; ar.dbeta = dbeta; ar.status = ws.status;
  ar.hc = (const uint8_t*)hc; ar.dhc = (const uint8_t*)dhc;
  ar.wim = (const uint8_t*)ws.wim; ar.uim = (const uint8_t*)ws.uim;
  ar.pim = (const uint8_t*)ws.pim; ar.tim = (const uint8_t*)ws.tim;
  ar.rqk = ws.rqk; ar.gl = ws.gl;
  cudaError_t e = cudaFuncSetAttribute(k_grad2_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)GR_SMEM);
  if (e != cudaSuccess) return e;
  const int64_t nblk = ar.NW < device_sms() ? ar.NW : device_sms();  // one CTA per SM
  k_grad2_tc<<<(unsigned)nblk, GT, GR_SMEM, st>>>(mq, mk, mv, mdo, mdv, mdqp, mdkp, ar);
  return cudaGetLastError();
}

}  // namespace gdn
