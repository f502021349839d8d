// gdn_api.cu -- the extern "C" entry points declared in include/gdn.h:
// validation, workspace layout and the order of kernel launches.
//
// Segments follow the p2p / all_gather algebra of "linear attention cp #1035",
// run on one GPU.  bf16 path (tensor cores): chunk prologue (norm factors,
// gates, W, U, P tiles) -> summaries [M|S] of segments 0..P-2 -> exclusive
// prefix H_in -> forward chain of every segment from its H_in (token output).
// Backward: prologue -> summaries + prefix -> forward chain storing every
// chunk-start state -> gradient summaries D of segments 1..P-1 -> reverse
// prefix dH_out -> reverse chain storing every chunk-end state gradient ->
// chunk-parallel local gradients -> Q/K head sum and norm chain.
// fp32 path (CUDA cores): the same algebra with the kernels of gdn_simt.cu.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "gdn_internal.h"

// Scratch of gdn_fwd_noalloc: one fixed array per device, reserved when the
// library's device code is loaded and held until the process exits.  Host code
// must never use this name as an address (on the host it is only a stand-in);
// the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_gdn_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

namespace gdn {
namespace {

constexpr int64_t kTargetBlocks = 304;  // scan blocks to aim for (two per SM of a 152-SM part)
constexpr int kScanCols = 32;           // state columns per scan block

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Pointer must be non-null and 16-byte aligned unless the tensor is empty.
bool ok_ptr(const void* p, int64_t numel) {
  if (numel == 0) return p == nullptr || aligned16(p);
  return p != nullptr && aligned16(p);
}
bool ok_opt(const void* p) { return p == nullptr || aligned16(p); }

}  // namespace

// SM count of the current device (152 on GB300 when no device can be queried), cached
// per device.
int device_sms() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices] = {};
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;
  }
  if (dev >= 0 && dev < kMaxDevices && (n = cache[dev].load(std::memory_order_relaxed)) > 0)
    return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

namespace {

// Segment count of the tensor-core path: the P that minimises a model of the chain
// launches of a training step (gdn_fwd_ctx + gdn_bwd_ctx).  Every chain pass runs
// ceil(CTAs / slots) waves of ceil(NC / P) chunk steps (slots = SMs, or 2 x SMs for the
// passes that fit two CTAs on an SM) plus a fixed cost per wave; the step times (us,
// GB300, T = 32K) are those of the forward summaries (3.3), the apply chain (3.3), the
// gradient summaries (4.9) and the states + state-gradient pair (4.4), and each prefix
// step costs ~7.7 us.  The model reproduces the measured best P at T = 8K, 32K, 64K.
int auto_segments_tc(int64_t BH, int64_t NC, int sms) {
  double best = 1e300;
  int best_p = 1;
  for (int64_t P = 1; P <= 64 && P <= NC; ++P) {
    const int64_t cps = (NC + P - 1) / P, pe = (NC + cps - 1) / cps;
    auto waves = [](int64_t n, int64_t slots) { return (double)((n + slots - 1) / slots); };
    const double w_sum = waves(2 * BH * pe, 2 * sms), w_app = waves(BH * pe, sms);
    const double w_gs = pe > 1 ? waves(BH * (pe - 1), 2 * sms) : 0.0;
    const double w_st = waves(2 * BH * pe, 2 * sms);
    const double t = cps * (w_sum * 3.34 + w_app * 3.25 + w_gs * 4.9 + w_st * 4.44) +
                     15.0 * (w_sum + w_app + w_gs + w_st) + 2 * (pe - 1) * 7.7;
    if (t < best - 1e-9) {
      best = t;
      best_p = (int)pe;
    }
  }
  return best_p;
}

int auto_segments(int64_t B, int64_t H, int64_t dv, int64_t NC, bool tensor_core) {
  if (NC <= 1) return 1;
  if (tensor_core) return auto_segments_tc(B * H, NC, device_sms());
  const int64_t per_seg = B * H * ((dv + kScanCols - 1) / kScanCols);
  int64_t want = (kTargetBlocks + per_seg - 1) / (per_seg > 0 ? per_seg : 1);
  int64_t P = 1;
  while (P < want) P <<= 1;
  if (P > NC) P = NC;
  if (P > 64) P = 64;
  return (int)P;
}

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

gdn_status resolve_op(const gdn_problem* p, int op, Prob* out) {
  if (!p || !out) return GDN_ERR_INVALID_ARG;
  if (p->dtype != GDN_FP32 && p->dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (p->B < 0 || p->T < 0 || p->Hqk < 1 || p->H < 1 || p->dk < 1 || p->dv < 1)
    return GDN_ERR_INVALID_ARG;
  if (p->H % p->Hqk != 0) return GDN_ERR_INVALID_ARG;
  if (p->T_stride != 0 && p->T_stride < p->T) return GDN_ERR_INVALID_ARG;
  if (!(p->l2_eps >= 0.f)) return GDN_ERR_INVALID_ARG;
  if (p->segments < 0) return GDN_ERR_INVALID_ARG;
  if (p->B > (int64_t)1 << 30 || p->T > (int64_t)1 << 34 || p->H > 4096)
    return GDN_ERR_INVALID_ARG;
  if (p->chunk != kChunk) return GDN_ERR_UNSUPPORTED;
  if (p->dk % 16 != 0 || p->dv % 16 != 0 || p->dk > kMaxHeadDim || p->dv > kMaxHeadDim)
    return GDN_ERR_UNSUPPORTED;
  if (p->dtype == GDN_BF16 && (p->dk != 128 || p->dv != 128)) return GDN_ERR_UNSUPPORTED;
  Prob r;
  r.dtype = p->dtype;
  r.B = p->B;
  r.T = p->T;
  r.Ts = p->T_stride == 0 ? p->T : p->T_stride;
  r.Hqk = p->Hqk;
  r.H = p->H;
  r.dk = p->dk;
  r.dv = p->dv;
  r.r = p->H / p->Hqk;
  r.l2norm = p->l2norm_qk ? 1 : 0;
  r.eps = p->l2_eps;
  r.scale = p->scale > 0.f ? p->scale : 1.0f / sqrtf((float)p->dk);
  r.NC = (p->T + kChunk - 1) / kChunk;
  r.Tp = r.NC * kChunk;
  const int64_t maxP = r.NC > 1 ? r.NC : 1;
  if (p->segments > maxP) return GDN_ERR_INVALID_ARG;
  const bool tcp = r.dtype == GDN_BF16 && r.dk == 128 && r.dv == 128 && r.B > 0 && r.NC > 0;
  int P = p->segments > 0 ? p->segments : auto_segments(r.B, r.H, r.dv, r.NC, tcp);
  if (op == GDN_OP_SUMMARY || op == GDN_OP_SUMMARY_BWD) P = 1;
  r.CPS = r.NC > 0 ? (r.NC + P - 1) / P : 0;
  r.P = r.CPS > 0 ? (int)((r.NC + r.CPS - 1) / r.CPS) : 1;
  *out = r;
  return GDN_OK;
}

gdn_status resolve(const gdn_problem* p, Prob* out) { return resolve_op(p, GDN_OP_FWD, out); }

size_t workspace_layout(const Prob& pr, int op, void* base, WS* ws) {
  WS w;
  memset(&w, 0, sizeof(w));
  size_t off = 0;
  char* b = (char*)base;
  auto take = [&](size_t nfloat) -> float* {
    float* ptr = base ? (float*)(b + off) : nullptr;
    off = align_up(off + nfloat * sizeof(float));
    return ptr;
  };
  const size_t B = pr.B, H = pr.H, Hqk = pr.Hqk, dk = pr.dk, dv = pr.dv, Tp = pr.Tp,
               NC = pr.NC, P = pr.P;
  // With a forward context on the tensor-core path the prologue's outputs live in the
  // context (written by gdn_fwd_ctx, read by gdn_bwd_ctx), not in the workspace.
  const bool in_ctx = (op == GDN_OP_FWD_CTX || op == GDN_OP_BWD_CTX) && tc_path(pr);
  if (op == GDN_OP_FWD_CTX) op = GDN_OP_FWD;
  if (op == GDN_OP_BWD_CTX) op = GDN_OP_BWD;
  const bool bwd = op == GDN_OP_BWD;
  const bool fwd = op == GDN_OP_FWD;
  w.status = (int*)take(64);
  if (in_ctx) {
    if (fwd && P > 1) w.Sseg = take(P * B * H * dk * dv);
    if (bwd) {  // the chunk-start states come from the context too
      if (P > 1) {
        w.Dseg = take(P * B * H * dk * dv);
        w.dHout = take(P * B * H * dk * dv);
      }
      w.dhc16 = take(B * H * NC * dk * dv / 2);
      w.dqp = take(B * Tp * H * dk / 2);  // bf16
      w.dkp = take(B * Tp * H * dk / 2);
    }
    if (ws) *ws = w;
    return off;
  }
  auto take_prep = [&]() {  // norm factors, gates and tile images of the tensor-core prologue
    w.rqk = take(B * Hqk * NC * 128);
    w.wim = take(B * H * NC * 4096);
    w.uim = take(B * H * NC * 4096);
    w.pim = take(B * H * NC * 2048);
    w.gl = take(B * H * NC * 64);
    if (bwd) w.tim = take(B * H * NC * 2048);
  };
  if (tc_path(pr) && bwd) {
    take_prep();
    if (P > 1) {
      w.Mseg = take(P * B * H * dk * dk);
      w.Sseg = take(P * B * H * dk * dv);
      w.Hin = take(P * B * H * dk * dv);
      w.Dseg = take(P * B * H * dk * dv);
      w.dHout = take(P * B * H * dk * dv);
    }
    w.hc16 = take(B * H * NC * dk * dv / 2);
    w.dhc16 = take(B * H * NC * dk * dv / 2);
    w.dqp = take(B * Tp * H * dk / 2);  // bf16
    w.dkp = take(B * Tp * H * dk / 2);
    if (ws) *ws = w;
    return off;
  }
  if (tc_path(pr) && (fwd || op == GDN_OP_SUMMARY)) {
    take_prep();
    if (fwd && P > 1) {
      w.Mseg = take(P * B * H * dk * dk);
      w.Sseg = take(P * B * H * dk * dv);
      w.Hin = take(P * B * H * dk * dv);
    }
    if (ws) *ws = w;
    return off;
  }
  w.Qh = take(B * Hqk * Tp * dk);
  w.Kh = take(B * Hqk * Tp * dk);
  w.G = (double*)take(2 * B * H * Tp);
  w.Bt = take(B * H * Tp);
  w.W = take(B * H * Tp * dk);
  w.U = take(B * H * Tp * dv);
  if (bwd) w.Tm = take(B * H * NC * 64 * 64);
  if (fwd || bwd) {
    w.Hc = take(B * H * NC * dk * dv);
    w.Vn = take(B * H * Tp * dv);
    if (P > 1) {
      w.Mseg = take(P * B * H * dk * dk);
      w.Sseg = take(P * B * H * dk * dv);
      w.Hin = take(P * B * H * dk * dv);
    }
  }
  if (bwd) {
    w.dHc = take(B * H * NC * dk * dv);
    w.dVn = take(B * H * Tp * dv);
    if (P > 1) {
      w.Dseg = take(P * B * H * dk * dv);
      w.dHout = take(P * B * H * dk * dv);
    }
    w.dqp = take(B * Tp * H * dk);
    w.dkp = take(B * Tp * H * dk);
  }
  if (ws) *ws = w;
  return off;
}

namespace {

gdn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

// Launch filter of one call: run every kernel (only < 0), only the kernel with
// launch index `only`, or none (dry run that counts launches and names one).
struct Sched {
  int only = -1;
  bool dry = false;
  int want = -1;
  int idx = 0;
  const char* name = nullptr;
  bool go(const char* nm) {
    const int i = idx++;
    if (dry) {
      if (i == want) name = nm;
      return false;
    }
    return only < 0 || only == i;
  }
};

#define GDN_TRY(expr)                              \
  do {                                             \
    cudaError_t e_ = (expr);                       \
    if (e_ != cudaSuccess) return GDN_ERR_CUDA;    \
  } while (0)

#define GDN_RUN(sched, name, expr)                 \
  do {                                             \
    if ((sched).go(name)) GDN_TRY(expr);           \
  } while (0)

gdn_status prepare(const gdn_problem* p, int op, void* workspace, size_t workspace_bytes,
                   cudaStream_t st, Prob* pr, WS* ws) {
  gdn_status s = resolve_op(p, op, pr);
  if (s != GDN_OK) return s;
  const size_t need = workspace_layout(*pr, op, nullptr, nullptr);
  if (workspace == nullptr || workspace_bytes < need) return GDN_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return GDN_ERR_INVALID_ARG;
  workspace_layout(*pr, op, workspace, ws);
  if (cudaMemsetAsync(ws->status, 0, sizeof(int), st) != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}

bool inputs_ok(const Prob& pr, const Inputs& in, bool need_q, bool need_v) {
  const int64_t nqk = pr.B * pr.T * pr.Hqk * pr.dk;
  const int64_t nv = pr.B * pr.T * pr.H * pr.dv;
  const int64_t ng = pr.B * pr.T * pr.H;
  if (need_q && !ok_ptr(in.q, nqk)) return false;
  if (!ok_ptr(in.k, nqk)) return false;
  if (need_v && !ok_ptr(in.v, nv)) return false;
  if (!ok_ptr(in.a, ng) || !ok_ptr(in.b, ng)) return false;
  if (!ok_ptr(in.A_log, pr.H) || !ok_ptr(in.dt_bias, pr.H)) return false;
  if (!ok_opt(in.valid_len)) return false;
  return true;
}

// Forward context (gdn_fwd_ctx / gdn_bwd_ctx): the transitions M of every segment and
// the start states H_in of every segment, fp32, [P][B][H][dk][dk] then [P][B][H][dk][dv];
// on the tensor-core path then the chunk prologue's outputs (norm factors, gates and the
// W, U, P, T tile images) and the bf16 image of every chunk-start state (written by the
// forward's output chain), which the backward reads instead of recomputing them.
struct Ctx {
  float* M;
  float* Hin;
  WS pro;  // rqk, wim, uim, pim, tim, gl, hc16 (tensor-core path), else all null
};
size_t ctx_layout(const Prob& pr, void* base, Ctx* c) {
  Ctx x;
  memset(&x, 0, sizeof(x));
  char* b = (char*)base;
  size_t off = 0;
  auto take = [&](size_t nfloat) -> float* {
    float* ptr = base ? (float*)(b + off) : nullptr;
    off = align_up(off + nfloat * sizeof(float));
    return ptr;
  };
  const size_t B = pr.B, H = pr.H, Hqk = pr.Hqk, NC = pr.NC, P = pr.P;
  x.M = take(P * B * H * pr.dk * pr.dk);
  x.Hin = take(P * B * H * pr.dk * pr.dv);
  if (tc_path(pr)) {
    x.pro.rqk = take(B * Hqk * NC * 128);
    x.pro.wim = take(B * H * NC * 4096);
    x.pro.uim = take(B * H * NC * 4096);
    x.pro.pim = take(B * H * NC * 2048);
    x.pro.tim = take(B * H * NC * 2048);
    x.pro.gl = take(B * H * NC * 64);
    x.pro.hc16 = take(B * H * NC * pr.dk * pr.dv / 2);
  }
  if (c) *c = x;
  return off;
}
size_t ctx_bytes(const Prob& pr) { return ctx_layout(pr, nullptr, nullptr); }
Ctx ctx_of(const Prob& pr, void* base) {
  Ctx c;
  ctx_layout(pr, base, &c);
  return c;
}
// The prologue outputs of a context call: the workspace pointers redirected into the context.
void use_ctx_prologue(const Prob& pr, const Ctx& cx, WS* ws) {
  if (!tc_path(pr)) return;
  ws->rqk = cx.pro.rqk;
  ws->wim = cx.pro.wim;
  ws->uim = cx.pro.uim;
  ws->pim = cx.pro.pim;
  ws->tim = cx.pro.tim;
  ws->gl = cx.pro.gl;
  ws->hc16 = cx.pro.hc16;
}
// H_in of the only segment: h0, or zero
cudaError_t ctx_single(const Prob& pr, const float* h0, float* Hin, cudaStream_t st) {
  const size_t n = (size_t)pr.B * pr.H * pr.dk * pr.dv * sizeof(float);
  if (n == 0) return cudaSuccess;
  return h0 ? cudaMemcpyAsync(Hin, h0, n, cudaMemcpyDeviceToDevice, st)
            : cudaMemsetAsync(Hin, 0, n, st);
}

cudaError_t pad_zero_grads(const Prob& pr, const int32_t* valid_len, void* dv, float* dg,
                           float* dbeta, cudaStream_t st) {
  cudaError_t e = launch_pad_tail_zero(pr, valid_len, dv, pr.H * pr.dv * 2, st);
  if (e == cudaSuccess) e = launch_pad_tail_zero(pr, valid_len, dg, pr.H * 4, st);
  if (e == cudaSuccess) e = launch_pad_tail_zero(pr, valid_len, dbeta, pr.H * 4, st);
  return e;
}

gdn_status run_forward(const Prob& pr, const Inputs& in, const float* h0, void* o, float* hT,
                       const WS& ws, cudaStream_t st, Sched& sc, const Ctx* cx = nullptr) {
  const float* init = h0;
  int64_t init_stride = 0;
  const int64_t sstride = pr.B * pr.H * pr.dk * pr.dv;
  if (tc_path(pr)) {
    GDN_RUN(sc, "prep_tc", launch_prep_tc(pr, in, ws, st));
    if (cx) {  // summaries of every segment; the transitions and start states are kept
      if (pr.P > 1) {
        GDN_RUN(sc, "summary_chain_tc",
                launch_chain_tc(pr, in, ws, 1, 0, pr.P, nullptr, 0, nullptr, nullptr, cx->M,
                                ws.Sseg, sstride, nullptr, st));
        GDN_RUN(sc, "prefix",
                launch_prefix(pr.B * pr.H, pr.P, pr.dk, pr.dv, cx->M, ws.Sseg, h0, cx->Hin,
                              nullptr, st));
      } else {
        GDN_RUN(sc, "ctx_init", ctx_single(pr, h0, cx->Hin, st));
      }
      init = cx->Hin;
      init_stride = sstride;
    } else if (pr.P > 1) {
      GDN_RUN(sc, "summary_chain_tc",
              launch_chain_tc(pr, in, ws, 1, 0, pr.P - 1, nullptr, 0, nullptr, nullptr, ws.Mseg,
                              ws.Sseg, sstride, nullptr, st));
      GDN_RUN(sc, "prefix",
              launch_prefix(pr.B * pr.H, pr.P, pr.dk, pr.dv, ws.Mseg, ws.Sseg, h0, ws.Hin,
                            nullptr, st));
      init = ws.Hin;
      init_stride = sstride;
    }
    GDN_RUN(sc, "apply_chain_tc",
            launch_chain_tc(pr, in, ws, 0, 0, pr.P, init, init_stride, o, hT, nullptr, nullptr,
                            0, cx ? ws.hc16 : nullptr, st));  // context: keep chunk-start states
    if (in.valid_len)  // chunks of padding only were skipped: their outputs are zero
      GDN_RUN(sc, "pad_zero", launch_pad_tail_zero(pr, in.valid_len, o, pr.H * pr.dv * 2, st));
    return GDN_OK;
  }
  GDN_RUN(sc, "prep", launch_prep(pr, in, ws, true, false, st));
  if (cx) {
    if (pr.P > 1) {
      GDN_RUN(sc, "summary_scan",
              launch_state_scan(pr, ws, 1, 0, pr.P, nullptr, 0, nullptr, nullptr, nullptr, cx->M,
                                ws.Sseg, sstride, st));
      GDN_RUN(sc, "prefix",
              launch_prefix(pr.B * pr.H, pr.P, pr.dk, pr.dv, cx->M, ws.Sseg, h0, cx->Hin,
                            nullptr, st));
    } else {
      GDN_RUN(sc, "ctx_init", ctx_single(pr, h0, cx->Hin, st));
    }
    init = cx->Hin;
    init_stride = sstride;
  } else if (pr.P > 1) {
    GDN_RUN(sc, "summary_scan",
            launch_state_scan(pr, ws, 1, 0, pr.P - 1, nullptr, 0, nullptr, nullptr, nullptr,
                              ws.Mseg, ws.Sseg, sstride, st));
    GDN_RUN(sc, "prefix",
            launch_prefix(pr.B * pr.H, pr.P, pr.dk, pr.dv, ws.Mseg, ws.Sseg, h0, ws.Hin, nullptr,
                          st));
    init = ws.Hin;
    init_stride = sstride;
  }
  GDN_RUN(sc, "state_scan",
          launch_state_scan(pr, ws, 0, 0, pr.P, init, init_stride, ws.Hc, ws.Vn, hT, nullptr,
                            nullptr, 0, st));
  GDN_RUN(sc, "output", launch_output(pr, in, ws, o, st));
  return GDN_OK;
}

gdn_status run_backward(const Prob& pr, const Inputs& in, const float* h0, const float* dHT,
                        void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dH0,
                        const WS& ws, cudaStream_t st, Sched& sc, const Ctx* cx = nullptr) {
  const int64_t sstride = pr.B * pr.H * pr.dk * pr.dv;
  if (tc_path(pr)) {
    const float* init = h0;
    int64_t init_stride = 0;
    if (!cx) GDN_RUN(sc, "prep_tc", launch_prep_tc(pr, in, ws, st));  // else kept by the forward
    const float* dinit = dHT;
    int64_t dinit_stride = 0;
    if (cx) {  // segment start states from the forward: only the reverse summaries and prefix
      init = cx->Hin;
      init_stride = sstride;
      if (pr.P > 1) {
        GDN_RUN(sc, "grad_summary_tc",
                launch_dchain_tc(pr, in, ws, 1, 1, pr.P - 1, nullptr, 0, nullptr, nullptr,
                                 ws.Dseg, sstride, st));
        GDN_RUN(sc, "prefix_bwd",
                launch_prefix_bwd(pr.B * pr.H, pr.P, pr.dk, pr.dv, cx->M, ws.Dseg, dHT,
                                  ws.dHout, nullptr, st));
        dinit = ws.dHout;
        dinit_stride = sstride;
      }
    } else if (pr.P > 1) {
      // forward summaries of every segment (M feeds both prefixes) with the gradient
      // summaries of segments 1..P-1, then both prefixes in one launch
      const ChainPass f{0, pr.P, nullptr, 0, ws.Mseg, ws.Sseg, sstride, nullptr};
      const ReversePass r{1, pr.P - 1, nullptr, 0, nullptr, nullptr, ws.Dseg, sstride};
      GDN_RUN(sc, "summary_pair_tc", launch_chain_pair_tc(pr, in, ws, 1, f, 1, r, st));
      GDN_RUN(sc, "prefix_pair",
              launch_prefix_pair(pr.B * pr.H, pr.P, pr.dk, pr.dv, ws.Mseg, ws.Sseg, h0, ws.Hin,
                                 ws.Dseg, dHT, ws.dHout, st));
      init = ws.Hin;
      init_stride = sstride;
      dinit = ws.dHout;
      dinit_stride = sstride;
    }
    if (cx && tc_path(pr)) {  // chunk-start states kept by the forward: the reverse chain alone
      GDN_RUN(sc, "dstates_chain_tc",
              launch_dchain_tc(pr, in, ws, 0, 0, pr.P, dinit, dinit_stride, ws.dhc16, dH0,
                               nullptr, 0, st));
    } else {  // every chunk-start state with every chunk-end state gradient
      const ChainPass f{0, pr.P, init, init_stride, nullptr, nullptr, 0, ws.hc16};
      const ReversePass r{0, pr.P, dinit, dinit_stride, ws.dhc16, dH0, nullptr, 0};
      GDN_RUN(sc, "states_pair_tc", launch_chain_pair_tc(pr, in, ws, 2, f, 0, r, st));
    }
    GDN_RUN(sc, "grad_tc", launch_grad2_tc(pr, in, ws, ws.hc16, ws.dhc16, dv, dg, dbeta, st));
    GDN_RUN(sc, "qk_grad_tc", launch_qk_grad_tc(pr, in, ws, dq, dk, st));  // masks padding
    if (in.valid_len)  // chunks of padding only were skipped: their gradients are zero
      GDN_RUN(sc, "pad_zero", pad_zero_grads(pr, in.valid_len, dv, dg, dbeta, st));
    return GDN_OK;
  }
  GDN_RUN(sc, "prep", launch_prep(pr, in, ws, true, true, st));
  const float* init = h0;
  int64_t init_stride = 0;
  if (cx) {
    init = cx->Hin;
    init_stride = sstride;
  } else if (pr.P > 1) {
    GDN_RUN(sc, "summary_scan",
            launch_state_scan(pr, ws, 1, 0, pr.P, nullptr, 0, nullptr, nullptr, nullptr, ws.Mseg,
                              ws.Sseg, sstride, st));
    GDN_RUN(sc, "prefix",
            launch_prefix(pr.B * pr.H, pr.P, pr.dk, pr.dv, ws.Mseg, ws.Sseg, h0, ws.Hin, nullptr,
                          st));
    init = ws.Hin;
    init_stride = sstride;
  }
  GDN_RUN(sc, "state_scan",
          launch_state_scan(pr, ws, 0, 0, pr.P, init, init_stride, ws.Hc, ws.Vn, nullptr, nullptr,
                            nullptr, 0, st));
  const float* dinit = dHT;
  int64_t dinit_stride = 0;
  if (pr.P > 1) {
    GDN_RUN(sc, "grad_summary_scan",
            launch_dstate_scan(pr, in, ws, 1, 1, pr.P - 1, nullptr, 0, nullptr, ws.Dseg, sstride,
                               st));
    GDN_RUN(sc, "prefix_bwd",
            launch_prefix_bwd(pr.B * pr.H, pr.P, pr.dk, pr.dv, cx ? cx->M : ws.Mseg, ws.Dseg,
                              dHT, ws.dHout, nullptr, st));
    dinit = ws.dHout;
    dinit_stride = sstride;
  }
  GDN_RUN(sc, "dstate_scan",
          launch_dstate_scan(pr, in, ws, 0, 0, pr.P, dinit, dinit_stride, dH0, nullptr, 0, st));
  GDN_RUN(sc, "grad", launch_grad(pr, in, ws, dv, dg, dbeta, st));
  GDN_RUN(sc, "qk_grad", launch_qk_grad(pr, in, ws, dq, dk, st));
  return GDN_OK;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_DEVICE_TIMEOUT: return "GDN_ERR_DEVICE_TIMEOUT";
  }
  return "GDN_ERR_UNKNOWN";
}

int32_t gdn_abi_version(void) { return GDN_ABI_VERSION; }

void gdn_problem_init(gdn_problem* p) {
  if (!p) return;
  memset(p, 0, sizeof(*p));
  p->dtype = GDN_BF16;
  p->chunk = kChunk;
  p->l2norm_qk = 1;
  p->l2_eps = 1e-6f;
  p->scale = 0.f;
  p->segments = 0;
}

gdn_status gdn_query_support(const gdn_problem* p) {
  Prob pr;
  return resolve_op(p, GDN_OP_FWD, &pr);
}

gdn_status gdn_resolved_segments(const gdn_problem* p, int32_t op, int32_t* segments) {
  if (!segments || op < GDN_OP_FWD || op > GDN_OP_BWD_CTX) return GDN_ERR_INVALID_ARG;
  if (op == GDN_OP_FWD_CTX) op = GDN_OP_FWD;
  if (op == GDN_OP_BWD_CTX) op = GDN_OP_BWD;
  Prob pr;
  gdn_status s = resolve_op(p, op, &pr);
  if (s != GDN_OK) return s;
  *segments = pr.P;
  return GDN_OK;
}

gdn_status gdn_workspace_size(const gdn_problem* p, int32_t op, size_t* bytes) {
  if (!bytes || op < GDN_OP_FWD || op > GDN_OP_BWD_CTX) return GDN_ERR_INVALID_ARG;
  Prob pr;
  gdn_status s = resolve_op(p, op, &pr);
  if (s != GDN_OK) return s;
  *bytes = workspace_layout(pr, op, nullptr, nullptr);
  return GDN_OK;
}

static gdn_status fwd_impl(const gdn_problem* p, const void* q, const void* k, const void* v,
                           const void* a, const void* b, const float* A_log,
                           const float* dt_bias, const float* h0, const int32_t* valid_len,
                           void* o, float* hT, void* workspace, size_t workspace_bytes,
                           void* stream, Sched& sc, void* ctx = nullptr,
                           size_t ctx_size = 0, bool with_ctx = false,
                           const gdn_conv_qkv* conv = nullptr) {
  Prob pr;
  gdn_status s = resolve_op(p, GDN_OP_FWD, &pr);
  if (s != GDN_OK) return s;
  Inputs in{q, k, v, a, b, A_log, dt_bias, valid_len, nullptr};
  if (!inputs_ok(pr, in, true, true)) return GDN_ERR_INVALID_ARG;
  if (!ok_ptr(o, pr.B * pr.T * pr.H * pr.dv) || !ok_opt(h0) || !ok_opt(hT))
    return GDN_ERR_INVALID_ARG;
  ConvIn cv;  // the Conv1D in front (q, k, v are its outputs y)
  if (conv) {
    const int64_t C[3] = {pr.Hqk * pr.dk, pr.Hqk * pr.dk, pr.H * pr.dv};
    const int64_t es = pr.dtype == GDN_BF16 ? 2 : 4;
    for (int i = 0; i < 3; ++i) {
      const int64_t n = pr.B * pr.T * C[i], span = pr.B * pr.Ts * C[i] * es;
      if (!ok_ptr(conv->x[i], n) || !ok_ptr(conv->w[i], C[i]) || !ok_opt(conv->bias[i]) ||
          !ok_opt(conv->halo[i]))
        return GDN_ERR_INVALID_ARG;
      const uintptr_t x0 = (uintptr_t)conv->x[i], y0 = (uintptr_t)conv->y[i];
      if (n > 0 && x0 < y0 + (uintptr_t)span && y0 < x0 + (uintptr_t)span)
        return GDN_ERR_INVALID_ARG;  // y overlaps its x
      cv.x[i] = conv->x[i];
      cv.w[i] = conv->w[i];
      cv.bias[i] = conv->bias[i];
      cv.halo[i] = conv->K > 1 ? conv->halo[i] : nullptr;
      cv.y[i] = conv->y[i];
    }
    if (conv->K < 1 || conv->K > 4) return GDN_ERR_UNSUPPORTED;
    cv.K = conv->K;
  }
  Ctx cx;
  if (with_ctx) {
    if (ctx == nullptr || !aligned16(ctx) || ctx_size < ctx_bytes(pr)) return GDN_ERR_INVALID_ARG;
    cx = ctx_of(pr, ctx);
  }
  WS ws;
  cudaStream_t st = (cudaStream_t)stream;
  if ((s = prepare(p, with_ctx ? GDN_OP_FWD_CTX : GDN_OP_FWD, workspace, workspace_bytes, st,
                   &pr, &ws)) != GDN_OK)
    return s;
  if (with_ctx) use_ctx_prologue(pr, cx, &ws);
  if (conv && tc_path(pr)) {
    in.conv = &cv;  // the chunk prologue convolves x itself and writes y
  } else if (conv) {  // other paths: the stand-alone Conv1D, then the forward
    for (int i = 0; i < 3; ++i) {
      gdn_conv_problem cp;
      cp.dtype = pr.dtype;
      cp.K = cv.K;
      cp.B = pr.B;
      cp.T = pr.T;
      cp.C = i < 2 ? pr.Hqk * pr.dk : pr.H * pr.dv;
      cp.T_stride = pr.Ts;
      if ((s = gdn_conv_silu_fwd(&cp, cv.x[i], cv.w[i], cv.bias[i], cv.halo[i], cv.y[i],
                                 stream)) != GDN_OK)
        return s;
    }
  }
  s = run_forward(pr, in, h0, o, hT, ws, st, sc, with_ctx ? &cx : nullptr);
  if (s == GDN_OK && conv && valid_len) {  // y of the chunks of padding only: zero
    const int64_t es = pr.dtype == GDN_BF16 ? 2 : 4;
    for (int i = 0; i < 3 && s == GDN_OK; ++i)
      s = cuda_status(launch_pad_tail_zero(pr, valid_len, cv.y[i],
                                           (i < 2 ? pr.Hqk * pr.dk : pr.H * pr.dv) * es, st));
  }
  return s;
}

static gdn_status bwd_impl(const gdn_problem* p, const void* q, const void* k, const void* v,
                           const void* a, const void* b, const float* A_log,
                           const float* dt_bias, const float* h0, const int32_t* valid_len,
                           const void* dO, const float* dHT, void* dq, void* dk, void* dv,
                           float* dg, float* dbeta, float* dH0, void* workspace,
                           size_t workspace_bytes, void* stream, Sched& sc,
                           const void* ctx = nullptr, size_t ctx_size = 0,
                           bool with_ctx = false) {
  Prob pr;
  gdn_status s = resolve_op(p, GDN_OP_BWD, &pr);
  if (s != GDN_OK) return s;
  Inputs in{q, k, v, a, b, A_log, dt_bias, valid_len, dO};
  if (!inputs_ok(pr, in, true, true)) return GDN_ERR_INVALID_ARG;
  const int64_t nqk = pr.B * pr.T * pr.Hqk * pr.dk, nv = pr.B * pr.T * pr.H * pr.dv,
                ng = pr.B * pr.T * pr.H;
  if (!ok_ptr(dO, nv) || !ok_opt(dHT) || !ok_opt(h0) || !ok_opt(dH0)) return GDN_ERR_INVALID_ARG;
  if (!ok_ptr(dq, nqk) || !ok_ptr(dk, nqk) || !ok_ptr(dv, nv) || !ok_ptr(dg, ng) ||
      !ok_ptr(dbeta, ng))
    return GDN_ERR_INVALID_ARG;
  Ctx cx;
  if (with_ctx) {
    if (ctx == nullptr || !aligned16(ctx) || ctx_size < ctx_bytes(pr)) return GDN_ERR_INVALID_ARG;
    cx = ctx_of(pr, const_cast<void*>(ctx));
  }
  WS ws;
  cudaStream_t st = (cudaStream_t)stream;
  if ((s = prepare(p, with_ctx ? GDN_OP_BWD_CTX : GDN_OP_BWD, workspace, workspace_bytes, st,
                   &pr, &ws)) != GDN_OK)
    return s;
  if (with_ctx) use_ctx_prologue(pr, cx, &ws);
  return run_backward(pr, in, h0, dHT, dq, dk, dv, dg, dbeta, dH0, ws, st, sc,
                      with_ctx ? &cx : nullptr);
}

gdn_status gdn_fwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                   const void* a, const void* b, const float* A_log, const float* dt_bias,
                   const float* h0, const int32_t* valid_len, void* o, float* hT,
                   void* workspace, size_t workspace_bytes, void* stream) {
  Sched sc;
  return fwd_impl(p, q, k, v, a, b, A_log, dt_bias, h0, valid_len, o, hT, workspace,
                  workspace_bytes, stream, sc);
}

gdn_status gdn_fwd_kernel(const gdn_problem* p, int32_t index, const void* q, const void* k,
                          const void* v, const void* a, const void* b, const float* A_log,
                          const float* dt_bias, const float* h0, const int32_t* valid_len,
                          void* o, float* hT, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (index < 0) return GDN_ERR_INVALID_ARG;
  Sched sc;
  sc.only = index;
  return fwd_impl(p, q, k, v, a, b, A_log, dt_bias, h0, valid_len, o, hT, workspace,
                  workspace_bytes, stream, sc);
}

gdn_status gdn_bwd_kernel(const gdn_problem* p, int32_t index, const void* q, const void* k,
                          const void* v, const void* a, const void* b, const float* A_log,
                          const float* dt_bias, const float* h0, const int32_t* valid_len,
                          const void* dO, const float* dHT, void* dq, void* dk, void* dv,
                          float* dg, float* dbeta, float* dH0, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (index < 0) return GDN_ERR_INVALID_ARG;
  Sched sc;
  sc.only = index;
  return bwd_impl(p, q, k, v, a, b, A_log, dt_bias, h0, valid_len, dO, dHT, dq, dk, dv, dg,
                  dbeta, dH0, workspace, workspace_bytes, stream, sc);
}

gdn_status gdn_ctx_size(const gdn_problem* p, size_t* bytes) {
  if (!bytes) return GDN_ERR_INVALID_ARG;
  Prob pr;
  gdn_status s = resolve_op(p, GDN_OP_FWD, &pr);
  if (s != GDN_OK) return s;
  *bytes = ctx_bytes(pr);
  return GDN_OK;
}

gdn_status gdn_fwd_ctx(const gdn_problem* p, const void* q, const void* k, const void* v,
                       const void* a, const void* b, const float* A_log, const float* dt_bias,
                       const float* h0, const int32_t* valid_len, void* o, float* hT, void* ctx,
                       size_t ctx_bytes_, void* workspace, size_t workspace_bytes,
                       void* stream) {
  Sched sc;
  return fwd_impl(p, q, k, v, a, b, A_log, dt_bias, h0, valid_len, o, hT, workspace,
                  workspace_bytes, stream, sc, ctx, ctx_bytes_, true);
}

gdn_status gdn_bwd_ctx(const gdn_problem* p, const void* q, const void* k, const void* v,
                       const void* a, const void* b, const float* A_log, const float* dt_bias,
                       const void* ctx, size_t ctx_bytes_, const int32_t* valid_len,
                       const void* dO, const float* dHT, void* dq, void* dk, void* dv, float* dg,
                       float* dbeta, float* dH0, void* workspace, size_t workspace_bytes,
                       void* stream) {
  Sched sc;
  return bwd_impl(p, q, k, v, a, b, A_log, dt_bias, nullptr, valid_len, dO, dHT, dq, dk, dv, dg,
                  dbeta, dH0, workspace, workspace_bytes, stream, sc, ctx, ctx_bytes_, true);
}

gdn_status gdn_fwd_conv(const gdn_problem* p, const gdn_conv_qkv* conv, const void* a,
                        const void* b, const float* A_log, const float* dt_bias, const float* h0,
                        const int32_t* valid_len, void* o, float* hT, void* ctx, size_t ctx_bytes_,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (!conv) return GDN_ERR_INVALID_ARG;
  Sched sc;
  return fwd_impl(p, conv->y[0], conv->y[1], conv->y[2], a, b, A_log, dt_bias, h0, valid_len, o,
                  hT, workspace, workspace_bytes, stream, sc, ctx, ctx_bytes_, ctx != nullptr,
                  conv);
}

gdn_status gdn_fwd_ctx_kernel(const gdn_problem* p, int32_t index, const void* q, const void* k,
                              const void* v, const void* a, const void* b, const float* A_log,
                              const float* dt_bias, const float* h0, const int32_t* valid_len,
                              void* o, float* hT, void* ctx, size_t ctx_bytes_, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (index < 0) return GDN_ERR_INVALID_ARG;
  Sched sc;
  sc.only = index;
  return fwd_impl(p, q, k, v, a, b, A_log, dt_bias, h0, valid_len, o, hT, workspace,
                  workspace_bytes, stream, sc, ctx, ctx_bytes_, true);
}

gdn_status gdn_bwd_ctx_kernel(const gdn_problem* p, int32_t index, const void* q, const void* k,
                              const void* v, const void* a, const void* b, const float* A_log,
                              const float* dt_bias, const void* ctx, size_t ctx_bytes_,
                              const int32_t* valid_len, const void* dO, const float* dHT,
                              void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dH0,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (index < 0) return GDN_ERR_INVALID_ARG;
  Sched sc;
  sc.only = index;
  return bwd_impl(p, q, k, v, a, b, A_log, dt_bias, nullptr, valid_len, dO, dHT, dq, dk, dv, dg,
                  dbeta, dH0, workspace, workspace_bytes, stream, sc, ctx, ctx_bytes_, true);
}

gdn_status gdn_kernel_info(const gdn_problem* p, int32_t op, int32_t index, int32_t* count,
                           const char** name) {
  if (op != GDN_OP_FWD && op != GDN_OP_BWD && op != GDN_OP_FWD_CTX && op != GDN_OP_BWD_CTX)
    return GDN_ERR_INVALID_ARG;
  const bool fwd = op == GDN_OP_FWD || op == GDN_OP_FWD_CTX;
  const bool with_ctx = op == GDN_OP_FWD_CTX || op == GDN_OP_BWD_CTX;
  Prob pr;
  gdn_status s = resolve_op(p, fwd ? GDN_OP_FWD : GDN_OP_BWD, &pr);
  if (s != GDN_OK) return s;
  Sched sc;
  sc.dry = true;
  sc.want = index;
  WS ws;
  memset(&ws, 0, sizeof(ws));
  Inputs in{};
  Ctx cx;
  memset(&cx, 0, sizeof(cx));
  if (fwd)
    run_forward(pr, in, nullptr, nullptr, nullptr, ws, nullptr, sc, with_ctx ? &cx : nullptr);
  else
    run_backward(pr, in, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                 ws, nullptr, sc, with_ctx ? &cx : nullptr);
  if (count) *count = sc.idx;
  if (name) *name = sc.name;
  return (index >= 0 && index >= sc.idx) ? GDN_ERR_INVALID_ARG : GDN_OK;
}

gdn_status gdn_apply_state(const gdn_problem* p, const void* q, const void* k, const void* v,
                           const void* a, const void* b, const float* A_log,
                           const float* dt_bias, const float* Hin, const int32_t* valid_len,
                           void* o, float* hT, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (Hin == nullptr) return GDN_ERR_INVALID_ARG;
  return gdn_fwd(p, q, k, v, a, b, A_log, dt_bias, Hin, valid_len, o, hT, workspace,
                 workspace_bytes, stream);
}

gdn_status gdn_bwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                   const void* a, const void* b, const float* A_log, const float* dt_bias,
                   const float* h0, const int32_t* valid_len, const void* dO, const float* dHT,
                   void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dH0,
                   void* workspace, size_t workspace_bytes, void* stream) {
  Sched sc;
  return bwd_impl(p, q, k, v, a, b, A_log, dt_bias, h0, valid_len, dO, dHT, dq, dk, dv, dg,
                  dbeta, dH0, workspace, workspace_bytes, stream, sc);
}

gdn_status gdn_apply_state_bwd(const gdn_problem* p, const void* q, const void* k,
                               const void* v, const void* a, const void* b, const float* A_log,
                               const float* dt_bias, const float* Hin,
                               const int32_t* valid_len, const void* dO, const float* dHout,
                               void* dq, void* dk, void* dv, float* dg, float* dbeta,
                               float* dHin, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (Hin == nullptr) return GDN_ERR_INVALID_ARG;
  return gdn_bwd(p, q, k, v, a, b, A_log, dt_bias, Hin, valid_len, dO, dHout, dq, dk, dv, dg,
                 dbeta, dHin, workspace, workspace_bytes, stream);
}

gdn_status gdn_gate_param_bwd(const gdn_problem* p, const void* a, const void* b,
                              const float* A_log, const float* dt_bias, const int32_t* valid_len,
                              const float* dg, const float* dbeta, float* da, float* db,
                              float* dA_log, float* ddt_bias, void* stream) {
  Prob pr;
  gdn_status s = resolve_op(p, GDN_OP_BWD, &pr);
  if (s != GDN_OK) return s;
  const int64_t ng = pr.B * pr.T * pr.H;
  if (!ok_ptr(a, ng) || !ok_ptr(b, ng) || !ok_ptr(dg, ng) || !ok_ptr(dbeta, ng) ||
      !ok_ptr(da, ng) || !ok_ptr(db, ng) || !ok_ptr(A_log, pr.H) || !ok_ptr(dt_bias, pr.H) ||
      !ok_ptr(dA_log, pr.H) || !ok_ptr(ddt_bias, pr.H) || !ok_opt(valid_len))
    return GDN_ERR_INVALID_ARG;
  return cuda_status(launch_gate_param_bwd(pr, a, b, A_log, dt_bias, valid_len, dg, dbeta, da, db,
                                           dA_log, ddt_bias, (cudaStream_t)stream));
}

gdn_status gdn_summary(const gdn_problem* p, const void* k, const void* v, const void* a,
                       const void* b, const float* A_log, const float* dt_bias,
                       const int32_t* valid_len, float* M, float* S, void* workspace,
                       size_t workspace_bytes, void* stream) {
  Prob pr;
  gdn_status s = resolve_op(p, GDN_OP_SUMMARY, &pr);
  if (s != GDN_OK) return s;
  Inputs in{nullptr, k, v, a, b, A_log, dt_bias, valid_len, nullptr};
  if (!inputs_ok(pr, in, false, true)) return GDN_ERR_INVALID_ARG;
  if (!ok_ptr(M, pr.B * pr.H * pr.dk * pr.dk) || !ok_ptr(S, pr.B * pr.H * pr.dk * pr.dv))
    return GDN_ERR_INVALID_ARG;
  WS ws;
  cudaStream_t st = (cudaStream_t)stream;
  if ((s = prepare(p, GDN_OP_SUMMARY, workspace, workspace_bytes, st, &pr, &ws)) != GDN_OK)
    return s;
  if (tc_path(pr)) {
    in.q = k;  // the prologue reads a q tile; a summary never uses it
    GDN_TRY(launch_prep_tc(pr, in, ws, st));
    GDN_TRY(launch_chain_tc(pr, in, ws, 1, 0, 1, nullptr, 0, nullptr, nullptr, M, S, 0, nullptr,
                            st));
    return GDN_OK;
  }
  GDN_TRY(launch_prep(pr, in, ws, false, false, st));
  GDN_TRY(launch_state_scan(pr, ws, 1, 0, 1, nullptr, 0, nullptr, nullptr, nullptr, M, S, 0, st));
  return GDN_OK;
}

gdn_status gdn_summary_bwd(const gdn_problem* p, const void* q, const void* k, const void* a,
                           const void* b, const float* A_log, const float* dt_bias,
                           const int32_t* valid_len, const void* dO, float* D,
                           void* workspace, size_t workspace_bytes, void* stream) {
  Prob pr;
  gdn_status s = resolve_op(p, GDN_OP_SUMMARY_BWD, &pr);
  if (s != GDN_OK) return s;
  // The gradient summary does not depend on v: the prologue skips U when v is null.
  Inputs in{q, k, nullptr, a, b, A_log, dt_bias, valid_len, dO};
  if (!inputs_ok(pr, in, true, false)) return GDN_ERR_INVALID_ARG;
  if (!ok_ptr(dO, pr.B * pr.T * pr.H * pr.dv) || !ok_ptr(D, pr.B * pr.H * pr.dk * pr.dv))
    return GDN_ERR_INVALID_ARG;
  WS ws;
  cudaStream_t st = (cudaStream_t)stream;
  if ((s = prepare(p, GDN_OP_SUMMARY_BWD, workspace, workspace_bytes, st, &pr, &ws)) != GDN_OK)
    return s;
  GDN_TRY(launch_prep(pr, in, ws, true, false, st));
  GDN_TRY(launch_dstate_scan(pr, in, ws, 1, 0, 1, nullptr, 0, nullptr, D, 0, st));
  return GDN_OK;
}

gdn_status gdn_compose(int64_t n, int64_t dk, int64_t dv, const float* M2, const float* S2,
                       const float* M1, const float* S1, float* M, float* S, void* stream) {
  if (n < 0 || dk < 1 || dv < 1) return GDN_ERR_INVALID_ARG;
  if (dk > kMaxHeadDim || dv > kMaxHeadDim) return GDN_ERR_UNSUPPORTED;
  const int64_t nm = n * dk * dk, ns = n * dv * dk;
  if (!ok_ptr(M2, nm) || !ok_ptr(M1, nm) || !ok_ptr(M, nm) || !ok_ptr(S2, ns) ||
      !ok_ptr(S1, ns) || !ok_ptr(S, ns))
    return GDN_ERR_INVALID_ARG;
  return cuda_status(launch_compose(n, dk, dv, M2, S2, M1, S1, M, S, (cudaStream_t)stream));
}

gdn_status gdn_prefix_compose(int64_t n, int64_t P, int64_t dk, int64_t dv, const float* M,
                              const float* S, const float* h0, float* Hin, float* Hout,
                              void* stream) {
  if (n < 0 || P < 1 || dk < 1 || dv < 1) return GDN_ERR_INVALID_ARG;
  if (dk > kMaxHeadDim || dv > kMaxHeadDim) return GDN_ERR_UNSUPPORTED;
  const int64_t nm = P * n * dk * dk, ns = P * n * dk * dv;
  if (!ok_ptr(M, nm) || !ok_ptr(S, ns) || !ok_ptr(Hin, ns) || !ok_opt(h0) || !ok_opt(Hout))
    return GDN_ERR_INVALID_ARG;
  return cuda_status(launch_prefix(n, P, dk, dv, M, S, h0, Hin, Hout, (cudaStream_t)stream));
}

gdn_status gdn_prefix_compose_bwd(int64_t n, int64_t P, int64_t dk, int64_t dv, const float* M,
                                  const float* D, const float* dHT, float* dHout, float* dH0,
                                  void* stream) {
  if (n < 0 || P < 1 || dk < 1 || dv < 1) return GDN_ERR_INVALID_ARG;
  if (dk > kMaxHeadDim || dv > kMaxHeadDim) return GDN_ERR_UNSUPPORTED;
  const int64_t nm = P * n * dk * dk, ns = P * n * dk * dv;
  if (!ok_ptr(M, nm) || !ok_ptr(D, ns) || !ok_ptr(dHout, ns) || !ok_opt(dHT) || !ok_opt(dH0))
    return GDN_ERR_INVALID_ARG;
  return cuda_status(
      launch_prefix_bwd(n, P, dk, dv, M, D, dHT, dHout, dH0, (cudaStream_t)stream));
}

// Device address of g_gdn_noalloc_scratch on the current device, looked up once
// per device (with that device current) and cached.
static gdn_status noalloc_scratch(void** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_gdn_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return GDN_ERR_CUDA;
    addr[dev] = ptr;
  }
  *out = addr[dev];
  return GDN_OK;
}

gdn_status gdn_fwd_noalloc(const gdn_problem* p, const void* q, const void* k, const void* v,
                           const void* a, const void* b, const float* A_log,
                           const float* dt_bias, const float* h0, const int32_t* valid_len,
                           void* o, float* hT, void* stream) {
  Prob pr;
  gdn_status s = resolve_op(p, GDN_OP_FWD, &pr);
  if (s != GDN_OK) return s;
  if (workspace_layout(pr, GDN_OP_FWD, nullptr, nullptr) > (size_t)GDN_NOALLOC_SCRATCH_BYTES)
    return GDN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if ((s = noalloc_scratch(&scratch)) != GDN_OK) return s;
  Sched sc;
  return fwd_impl(p, q, k, v, a, b, A_log, dt_bias, h0, valid_len, o, hT, scratch,
                  (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream, sc);
}

gdn_status gdn_noalloc_check_device_status(void* stream) {
  void* scratch = nullptr;
  gdn_status s = noalloc_scratch(&scratch);
  if (s != GDN_OK) return s;
  return gdn_check_device_status(scratch, stream);
}

gdn_status gdn_check_device_status(void* workspace, void* stream) {
  if (workspace == nullptr || ((uintptr_t)workspace & 255u) != 0) return GDN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return GDN_ERR_CUDA;
  if (word & kStatusTimeout) return GDN_ERR_DEVICE_TIMEOUT;
  if (word & kStatusClamped) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

}  // extern "C"
