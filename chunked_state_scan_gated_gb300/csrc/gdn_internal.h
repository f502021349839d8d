// gdn_internal.h -- shared declarations of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kChunk = 64;          // tokens per chunk
constexpr int kMaxHeadDim = 128;    // largest dk / dv
constexpr int kStatusClamped = 1;   // device status bit: a valid_len was outside [0, T]
constexpr int kStatusTimeout = 2;   // device status bit: a bounded wait ran out

// A validated problem with every derived size.
struct Prob {
  int dtype;
  int64_t B, T, Ts, Hqk, H, dk, dv, r;
  int l2norm;
  float eps, scale;
  int64_t NC;   // chunks per row, ceil(T / 64)
  int64_t Tp;   // NC * 64
  int P;        // segments
  int64_t CPS;  // chunks per segment (last one may be shorter)
};

// Workspace regions (device pointers into the caller's buffer); null when unused.
struct WS {
  int* status;  // device status word
  float* Qh;    // [B][Hqk][Tp][dk]  normalised, scaled q
  float* Kh;    // [B][Hqk][Tp][dk]  normalised k
  double* G;    // [B][H][Tp]        cumulative gate inside each chunk (fp64, see gdn_simt.cu)
  float* Bt;    // [B][H][Tp]        beta
  float* W;     // [B][H][Tp][dk]    T diag(beta*gamma) K
  float* U;     // [B][H][Tp][dv]    T diag(beta) V
  float* Tm;    // [B][H][NC][64][64] (I + A)^-1
  float* Hc;    // [B][H][NC][dk][dv] state at each chunk start
  float* Vn;    // [B][H][Tp][dv]    V' = U - W S
  float* Mseg;  // [P][B][H][dk][dk]
  float* Sseg;  // [P][B][H][dk][dv]
  float* Hin;   // [P][B][H][dk][dv]
  float* dHc;   // [B][H][NC][dk][dv] gradient of each chunk's end state
  float* dVn;   // [B][H][Tp][dv]    gradient of V'
  float* Dseg;  // [P][B][H][dk][dv]
  float* dHout; // [P][B][H][dk][dv]
  float* dqp;   // [B][Tp][H][dk]    per-V-head gradient of q_hat (bf16 on the tensor-core path)
  float* dkp;   // [B][Tp][H][dk]    per-V-head gradient of k_hat
  float* rqk;   // [B][Hqk][NC][128] per-token norm factors rq = scale/|q|, then rk = 1/|k|
  void* wim;    // [B][H][NC]   16 KB bf16 tile images of W (tensor-core path)
  void* uim;    // [B][H][NC]   16 KB tile images of U
  void* pim;    // [B][H][NC]   8 KB tile images of P = tril(Q K^T o Gamma)
  void* tim;    // [B][H][NC]   8 KB tile images of T = (I + A)^-1 (backward)
  float* gl;    // [B][H][NC][64] cumulative gate inside each chunk, log2 units
  void* hc16;   // [B][H][NC][dk][dv] bf16 chunk-start states (tensor-core backward)
  void* dhc16;  // [B][H][NC][dk][dv] bf16 chunk-end state gradients (tensor-core backward)
};

// Raw inputs of a call (device pointers; type of q..dO is Prob::dtype).
// Causal depthwise Conv1D + SiLU in front of the core (index 0: q, 1: k, 2: v): the
// tensor-core prologue loads x[i] (layout of q, k, v), convolves it in shared memory and
// writes y[i] = SiLU(conv(x[i])), which every later kernel reads as q, k, v.
struct ConvIn {
  int K;                 // taps, 1..4
  const void* x[3];      // pre-conv activations
  const float* w[3];     // [channels][K]
  const float* bias[3];  // [channels] or null
  const void* halo[3];   // [B][K-1][channels] or null (zeros)
  void* y[3];            // activated q, k, v (the Inputs' q, k, v point here)
};

struct Inputs {
  const void *q, *k, *v, *a, *b;
  const float *A_log, *dt_bias;
  const int32_t* valid_len;
  const void* dO;
  const ConvIn* conv = nullptr;  // set: the prologue runs the Conv1D + SiLU (forward only)
};

gdn_status resolve(const gdn_problem* p, Prob* out);
size_t workspace_layout(const Prob& pr, int op, void* base, WS* ws);

// ---- SIMT (fp32 CUDA-core) kernels; each returns the launch's cudaError_t ----
cudaError_t launch_prep(const Prob& pr, const Inputs& in, const WS& ws, bool need_q,
                        bool need_T, cudaStream_t st);
// mode 0: forward states (writes Hc/Vn when non-null, final state of the last
// segment to `final_out`); mode 1: summary of [M|S] (writes M/S per segment).
cudaError_t launch_state_scan(const Prob& pr, const WS& ws, int mode, int seg_first, int nseg,
                              const float* init, int64_t init_seg_stride, float* Hc, float* Vn,
                              float* final_out, float* M_out, float* S_out,
                              int64_t out_seg_stride, cudaStream_t st);
cudaError_t launch_output(const Prob& pr, const Inputs& in, const WS& ws, void* o,
                          cudaStream_t st);
// mode 0: store dHc/dVn, start gradient of segment 0 to `start_out`;
// mode 1: gradient summary from zero, start gradient of every segment to D_out[seg].
cudaError_t launch_dstate_scan(const Prob& pr, const Inputs& in, const WS& ws, int mode,
                               int seg_first, int nseg, const float* init,
                               int64_t init_seg_stride, float* start_out, float* D_out,
                               int64_t out_seg_stride, cudaStream_t st);
cudaError_t launch_grad(const Prob& pr, const Inputs& in, const WS& ws, void* dv, float* dg,
                        float* dbeta, cudaStream_t st);
cudaError_t launch_qk_grad(const Prob& pr, const Inputs& in, const WS& ws, void* dq, void* dk,
                           cudaStream_t st);
cudaError_t launch_compose(int64_t n, int64_t dk, int64_t dv, const float* M2, const float* S2,
                           const float* M1, const float* S1, float* M, float* S,
                           cudaStream_t st);
// Hin[s] for s < P; applies map s only when s < P-1 or Hout != null.
cudaError_t launch_prefix(int64_t n, int64_t P, int64_t dk, int64_t dv, const float* M,
                          const float* S, const float* h0, float* Hin, float* Hout,
                          cudaStream_t st);
// Both prefixes of the backward in one launch: Hin (forward, no Hout) and dHout (reverse, no dH0).
cudaError_t launch_prefix_pair(int64_t n, int64_t P, int64_t dk, int64_t dv, const float* M,
                               const float* S, const float* h0, float* Hin, const float* D,
                               const float* dHT, float* dHout, cudaStream_t st);
// dHout[s] for s >= 0 in reverse; applies M[s]^T . + D[s] only when s > 0 or dH0 != null.
cudaError_t launch_prefix_bwd(int64_t n, int64_t P, int64_t dk, int64_t dv, const float* M,
                              const float* D, const float* dHT, float* dHout, float* dH0,
                              cudaStream_t st);

// gate-parameter gradients from dg, dbeta (both dtypes; one CTA per head, fixed-order sums)
cudaError_t launch_gate_param_bwd(const Prob& pr, const void* a, const void* b,
                                  const float* A_log, const float* dt_bias,
                                  const int32_t* valid_len, const float* dg, const float* dbeta,
                                  float* da, float* db, float* dA_log, float* ddt_bias,
                                  cudaStream_t st);

// number of SMs of the current device (cached per device)
int device_sms();

// ---- tensor-core (tcgen05) kernels, bf16 with dk = dv = 128 ----
bool tc_path(const Prob& pr);
// chunk-parallel prologue: norm factors, gates and the W, U, P (and T) tile images
cudaError_t launch_prep_tc(const Prob& pr, const Inputs& in, const WS& ws, cudaStream_t st);
// state chain over the prologue's tiles.  mode 0 (apply): o and the final state of
// the last segment from `init`; mode 1 (summary): M_out, S_out of segments
// seg_first..; mode 2 (states): every chunk-start state into `hc` (bf16).
cudaError_t launch_chain_tc(const Prob& pr, const Inputs& in, const WS& ws, int mode,
                            int seg_first, int nseg, const float* init, int64_t init_seg_stride,
                            void* o, float* final_out, float* M_out, float* S_out,
                            int64_t out_seg_stride, void* hc, cudaStream_t st);

// reverse chain over the prologue's tiles: mode 0 stores every chunk-end state
// gradient (bf16) and the start gradient of segment 0; mode 1 writes gradient
// summaries D of segments seg_first..
cudaError_t launch_dchain_tc(const Prob& pr, const Inputs& in, const WS& ws, int mode,
                             int seg_first, int nseg, const float* init, int64_t init_seg_stride,
                             void* dhc, float* start_out, float* D_out, int64_t out_seg_stride,
                             cudaStream_t st);

// A forward chain pass (summary or states) and an independent reverse chain pass in one
// launch (the CTAs of both share the GPU); either pass may be empty (nseg <= 0).
struct ChainPass {
  int seg_first, nseg;
  const float* init;
  int64_t init_seg_stride;
  float* M_out;
  float* S_out;
  int64_t out_seg_stride;
  void* hc;
};
struct ReversePass {
  int seg_first, nseg;
  const float* init;
  int64_t init_seg_stride;
  void* dhc;
  float* start_out;
  float* D_out;
  int64_t out_seg_stride;
};
cudaError_t launch_chain_pair_tc(const Prob& pr, const Inputs& in, const WS& ws, int fmode,
                                 const ChainPass& f, int rmode, const ReversePass& r,
                                 cudaStream_t st);
// dq, dk (bf16) from the per-V-head bf16 gradients of q_hat, k_hat in ws.dqp / ws.dkp
// Zeroes tokens [ceil(valid_len[b] / 64) * 64, T) of every row b of a token-major tensor
// of row_bytes per token (row stride Ts tokens); nothing without valid_len.
cudaError_t launch_pad_tail_zero(const Prob& pr, const int32_t* valid_len, void* dst,
                                 int64_t row_bytes, cudaStream_t st);
cudaError_t launch_qk_grad_tc(const Prob& pr, const Inputs& in, const WS& ws, void* dq, void* dk,
                              cudaStream_t st);
// chunk-parallel local gradients from chunk-start states and chunk-end state gradients
// (feature-major tcgen05 products); dq_hat / dk_hat partials into ws.dqp / ws.dkp (bf16)
cudaError_t launch_grad2_tc(const Prob& pr, const Inputs& in, const WS& ws, const void* hc,
                            const void* dhc, void* dv, float* dg, float* dbeta, cudaStream_t st);

}  // namespace gdn
