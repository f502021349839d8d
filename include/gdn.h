/*
 * gdn.h -- C ABI of the GB300 Gated DeltaNet (GDN) core library.
 *
 * The operator is the gated delta rule of Qwen3.5's linear-attention layers,
 * per batch row b and value head h, with state S in R^{dk x dv}:
 *
 *   q_hat = scale * q / sqrt(|q|^2 + eps),  k_hat = k / sqrt(|k|^2 + eps)
 *   g_t   = -exp(A_log[h]) * softplus(a_t + dt_bias[h]),  alpha_t = exp(g_t)
 *   beta_t = sigmoid(b_t)
 *   S_t   = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *   o_t   = S_t^T q_t
 *
 * evaluated in chunks of 64 tokens.  Interface and conventions follow the pages:
 *  - "Linear Attention CP 融合算子 PR #1114 测试报告", section 4.1: the core takes
 *    q, k, v, g, beta and an initial state, returns the token output and the
 *    final state, and its backward returns dq, dk, dv, dg, dbeta, dH0; the 16
 *    Q/K heads are copied by grouping onto the 32 V heads (V head h reads Q/K
 *    head h / (H/Hqk)).
 *  - same report, section 3.1: fail fast, with no silent fallback, when the
 *    fast path cannot take a shape (head_dim != 128 or chunk_size != 64).
 *  - same report, section 5.2: trailing padding (B=2, valid_length=7777) gives
 *    zero output for padded tokens and leaves the state unchanged.
 *  - "linear attention cp #1035", section "What does this PR do": each rank
 *    summarises its segment as the affine map H_out = M @ H_in + S ("p2p"),
 *    the summaries of earlier ranks are merged into the initial state
 *    ("all_gather"), and the state gradient travels back the reverse way.
 *    Here the segments live on one GPU.
 *
 * Conventions for every call
 *  - Layout is token-major and contiguous: q, k [B, T_stride, Hqk, dk];
 *    v, o, dO, dv [B, T_stride, H, dv]; a, b, dg, dbeta [B, T_stride, H];
 *    only tokens [0, T) of each row are read or written.  States h0, hT, dHT,
 *    dH0, S, D, H_in [B, H, dk, dv] and M [B, H, dk, dk] are fp32 row-major.
 *    A_log and dt_bias are fp32 [H].  valid_len is int32 [B] or NULL.
 *  - Every pointer except the host `gdn_problem*` and `bytes*` arguments is a
 *    DEVICE pointer, 16-byte aligned, on the current device.  The caller owns all
 *    memory, including the workspace.  The library never allocates, frees or
 *    synchronises (gdn_check_device_status is the one synchronous call); every
 *    launch is ordered on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream).  Outputs must not alias inputs.  The library keeps no global state.
 *  - Host-side validation runs before any launch and returns a status; nothing
 *    is launched unless it returns GDN_OK.  Errors raised by CUDA while
 *    launching come back as GDN_ERR_CUDA.  Faults found by a kernel (a
 *    valid_len outside [0, T], an exhausted bounded wait) are recorded in the
 *    workspace's status word, read by gdn_check_device_status.
 *  - Results are deterministic run to run for a fixed problem and segment count.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 1

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad shape, H % Hqk != 0, ... */
  GDN_ERR_UNSUPPORTED = 2,    /* valid problem the library does not take (chunk != 64, ...) */
  GDN_ERR_WORKSPACE = 3,      /* workspace missing or smaller than gdn_workspace_size */
  GDN_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
  GDN_ERR_DEVICE_TIMEOUT = 5  /* a kernel gave up a bounded wait (device status word) */
} gdn_status;

typedef enum gdn_dtype {
  GDN_FP32 = 0,  /* fp32 I/O, fp32 arithmetic on CUDA cores; any dk, dv in {16..128}/16 */
  GDN_BF16 = 1   /* bf16 I/O, fp32 accumulation; dk = dv = 128 */
} gdn_dtype;

typedef enum gdn_op {
  GDN_OP_FWD = 0,         /* gdn_fwd, gdn_apply_state */
  GDN_OP_BWD = 1,         /* gdn_bwd, gdn_apply_state_bwd */
  GDN_OP_SUMMARY = 2,     /* gdn_summary */
  GDN_OP_SUMMARY_BWD = 3, /* gdn_summary_bwd */
  GDN_OP_FWD_CTX = 4,     /* gdn_fwd_ctx (a GDN_OP_FWD-sized workspace also suffices) */
  GDN_OP_BWD_CTX = 5      /* gdn_bwd_ctx (a GDN_OP_BWD-sized workspace also suffices) */
} gdn_op;

/* Problem description.  Fill with gdn_problem_init, then set the sizes. */
typedef struct gdn_problem {
  int32_t dtype;     /* gdn_dtype of q, k, v, a, b, o, dO, dq, dk, dv */
  int32_t chunk;     /* chunk length; must be 64 */
  int64_t B;         /* batch rows, >= 0 */
  int64_t T;         /* tokens per row handled by this call, >= 0 */
  int64_t T_stride;  /* tokens between consecutive rows in memory; 0 means T (must be >= T) */
  int64_t Hqk;       /* query/key heads, >= 1 */
  int64_t H;         /* value heads, a multiple of Hqk */
  int64_t dk;        /* key/query head dim */
  int64_t dv;        /* value head dim */
  int32_t l2norm_qk; /* 1: L2-normalise q and k inside (default); 0: use them as given */
  float l2_eps;      /* eps inside the norm, x / sqrt(|x|^2 + eps); default 1e-6 */
  float scale;       /* scale applied to q after the norm; <= 0 means 1/sqrt(dk) */
  int32_t segments;  /* sequence segments the call splits T into (time parallelism);
                        0 = automatic, else 1..ceil(T/64).  Results agree across
                        segment counts to rounding. */
} gdn_problem;

/* Human-readable name of a status. Never NULL. */
const char* gdn_status_string(gdn_status status);

/* GDN_ABI_VERSION of the loaded library. */
int32_t gdn_abi_version(void);

/* Defaults: dtype BF16, chunk 64, l2norm on, eps 1e-6, scale 1/sqrt(dk), segments auto,
   all sizes 0.  Does nothing if p is NULL. */
void gdn_problem_init(gdn_problem* p);

/*
 * Capability check ("is the problem supported?") without side effects:
 * GDN_OK, GDN_ERR_INVALID_ARG (malformed: negative sizes, H % Hqk != 0,
 * T_stride < T, eps < 0, segments out of range) or GDN_ERR_UNSUPPORTED
 * (well formed but not taken: chunk != 64, dk or dv not a multiple of 16 in
 * [16, 128], bf16 with dk or dv != 128).  Mirrors the fail-fast capability check
 * of the test report, section 3.1.
 */
gdn_status gdn_query_support(const gdn_problem* p);

/* Number of sequence segments (*segments) a call of `op` on problem p splits T into:
   p->segments when set, else the automatic choice for the current device (on the
   tensor-core path, the count that minimises a model of the chain passes' time).
   Summary calls always use 1. */
gdn_status gdn_resolved_segments(const gdn_problem* p, int32_t op, int32_t* segments);

/* Workspace bytes needed by `op` for problem p on the current device (writes *bytes).
   Always at least 256 (the device status word lives there). */
gdn_status gdn_workspace_size(const gdn_problem* p, int32_t op, size_t* bytes);

/*
 * Forward.  o = token outputs [B,T,H,dv] in p->dtype (zero for t >= valid_len[b]);
 * hT (nullable) = state after the last valid token [B,H,dk,dv] fp32.
 * h0 (nullable: zero initial state) [B,H,dk,dv] fp32.
 * Internally the sequence may be split into segments whose summaries are
 * composed on the device (the pages' p2p/all_gather algebra on one GPU).
 */
gdn_status gdn_fwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                   const void* a, const void* b, const float* A_log, const float* dt_bias,
                   const float* h0, const int32_t* valid_len, void* o, float* hT,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward of L = sum_t <dO_t, o_t> + <dHT, hT> w.r.t. the forward inputs.
 * Takes the forward inputs again and recomputes the chunk intermediates (no
 * saved context).  dO [B,T,H,dv] p->dtype (values at padded tokens are ignored);
 * dHT nullable (zero).  Writes dq, dk [B,T,Hqk,dk] and dv [B,T,H,dv] in
 * p->dtype (w.r.t. the raw q, k before the norm and scale, summed over the V
 * heads sharing a Q/K head); dg, dbeta [B,T,H] fp32 (w.r.t. g_t and beta_t);
 * dH0 [B,H,dk,dv] fp32 (nullable).  Padded tokens get zero gradients.
 */
gdn_status gdn_bwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                   const void* a, const void* b, const float* A_log, const float* dt_bias,
                   const float* h0, const int32_t* valid_len, const void* dO, const float* dHT,
                   void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dH0,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward context for a training step (no counterpart on the pages).  The forward
 * splits T into P segments (P = gdn_resolved_segments(p, GDN_OP_FWD)) and computes
 * every segment's transition M_s [dk,dk] (H_out = M_s H_in + S_s) and start state
 * H_in,s [dk,dv]; gdn_bwd recomputes both.  gdn_fwd_ctx is gdn_fwd that also keeps
 * them in `ctx`: M [P][B][H][dk][dk] then H_in [P][B][H][dk][dv], fp32, in a
 * caller-owned, 16-byte aligned device buffer of at least gdn_ctx_size bytes.  On
 * the bf16 tensor-core path (dk = dv = 128) the context also keeps the outputs of
 * the chunk prologue (per-token norm factors, cumulative gates, and bf16 tile images
 * of W = T diag(beta gamma) K, U = T diag(beta) V, P = tril(Q K^T o Gamma) and
 * T = (I + A)^-1 for every chunk and V head) and the bf16 image of every chunk-start
 * state S (written by the forward's output chain): ~41.2 KB per token at H = 32,
 * d = 128 (1.32 GiB at T = 32K, P = 9), against 36 MiB without them; the workspaces of
 * GDN_OP_FWD_CTX and GDN_OP_BWD_CTX shrink by the same images.  gdn_bwd_ctx is
 * gdn_bwd with h0 replaced by that context: it reads H_in (which already holds h0 as
 * H_in,0), M, the prologue outputs and the chunk-start states instead of recomputing
 * the forward summaries, their prefix, the prologue and the forward state chain.  The context is only valid for the same problem
 * (same resolved P), inputs and h0; the library cannot check that.  Invalid pointer
 * or size: GDN_ERR_INVALID_ARG.  gdn_fwd_ctx_kernel / gdn_bwd_ctx_kernel and the ops
 * GDN_OP_FWD_CTX / GDN_OP_BWD_CTX of gdn_kernel_info are the profiling aids below
 * for these two calls.
 */
gdn_status gdn_ctx_size(const gdn_problem* p, size_t* bytes);
gdn_status gdn_fwd_ctx(const gdn_problem* p, const void* q, const void* k, const void* v,
                       const void* a, const void* b, const float* A_log, const float* dt_bias,
                       const float* h0, const int32_t* valid_len, void* o, float* hT, void* ctx,
                       size_t ctx_bytes, void* workspace, size_t workspace_bytes, void* stream);
gdn_status gdn_bwd_ctx(const gdn_problem* p, const void* q, const void* k, const void* v,
                       const void* a, const void* b, const float* A_log, const float* dt_bias,
                       const void* ctx, size_t ctx_bytes, const int32_t* valid_len,
                       const void* dO, const float* dHT, void* dq, void* dk, void* dv, float* dg,
                       float* dbeta, float* dH0, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * Gradients of the gate parameters from the core's dg, dbeta [B,T,H] fp32 (as
 * returned by gdn_bwd).  The gates are g = -exp(A_log[h]) softplus(a + dt_bias[h])
 * and beta = sigmoid(b) (the test report, section 4.1, checks every parameter
 * gradient).  Writes da, db [B,T,H] fp32 (w.r.t. the a, b given to gdn_fwd;
 * zero for padded tokens) and dA_log, ddt_bias [H] fp32 (sums over all rows and
 * valid tokens, in a fixed order: deterministic).  a, b in p->dtype.  No
 * workspace; one launch.
 */
gdn_status gdn_gate_param_bwd(const gdn_problem* p, const void* a, const void* b,
                              const float* A_log, const float* dt_bias, const int32_t* valid_len,
                              const float* dg, const float* dbeta, float* da, float* db,
                              float* dA_log, float* ddt_bias, void* stream);

/*
 * Segment summary (PR #1035, "p2p": H_out = M @ H_in + S for the local
 * segment).  The segment is tokens [0, T) of the given rows (pass pointers to
 * the segment's first token and T_stride = the full row length).
 * M [B,H,dk,dk] = A_T ... A_1 with A_t = alpha_t (I - beta_t k_t k_t^T);
 * S [B,H,dk,dv] = state reached from zero.
 */
gdn_status gdn_summary(const gdn_problem* p, const void* k, const void* v, const void* a,
                       const void* b, const float* A_log, const float* dt_bias,
                       const int32_t* valid_len, float* M, float* S, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Gradient summary of a segment: D = d(sum_t <dO_t, o_t>)/dH_in [B,H,dk,dv].
 * Together with M it is the segment's backward affine map dH_in = M^T dH_out + D
 * (the reverse-direction state-gradient pass of PR #1035).  Independent of v and
 * of H_in.
 */
gdn_status gdn_summary_bwd(const gdn_problem* p, const void* q, const void* k, const void* a,
                           const void* b, const float* A_log, const float* dt_bias,
                           const int32_t* valid_len, const void* dO, float* D,
                           void* workspace, size_t workspace_bytes, void* stream);

/* (M, S) = (M2 M1, M2 S1 + S2) for n independent maps: M* [n,dk,dk], S* [n,dk,dv]. */
gdn_status gdn_compose(int64_t n, int64_t dk, int64_t dv, const float* M2, const float* S2,
                       const float* M1, const float* S1, float* M, float* S, void* stream);

/*
 * Exclusive prefix over P segments (PR #1035, "all_gather": merge the summaries
 * of earlier ranks into the initial state): M [P,n,dk,dk], S [P,n,dk,dv],
 * h0 [n,dk,dv] nullable (zero).  H_in[0] = h0, H_in[i] = M[i-1] H_in[i-1] + S[i-1]
 * into Hin [P,n,dk,dv]; Hout (nullable) [n,dk,dv] = M[P-1] H_in[P-1] + S[P-1].
 */
gdn_status gdn_prefix_compose(int64_t n, int64_t P, int64_t dk, int64_t dv, const float* M,
                              const float* S, const float* h0, float* Hin, float* Hout,
                              void* stream);

/*
 * Reverse exclusive prefix of state gradients: dHT [n,dk,dv] nullable (zero).
 * dH_out[P-1] = dHT, dH_out[i] = M[i+1]^T dH_out[i+1] + D[i+1] into dHout
 * [P,n,dk,dv]; dH0 (nullable) [n,dk,dv] = M[0]^T dH_out[0] + D[0].
 */
gdn_status gdn_prefix_compose_bwd(int64_t n, int64_t P, int64_t dk, int64_t dv, const float* M,
                                  const float* D, const float* dHT, float* dHout, float* dH0,
                                  void* stream);

/*
 * State apply (PR #1035, "p2p": once the initial state arrives, compute the
 * segment's token output): the forward of a segment from Hin [B,H,dk,dv]
 * (required).  Same as gdn_fwd with h0 = Hin; hT nullable.
 */
gdn_status gdn_apply_state(const gdn_problem* p, const void* q, const void* k, const void* v,
                           const void* a, const void* b, const float* A_log,
                           const float* dt_bias, const float* Hin, const int32_t* valid_len,
                           void* o, float* hT, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Backward of a segment started from Hin, given the gradient dHout of its end
 * state (nullable: zero): gdn_bwd with h0 = Hin, dHT = dHout; dHin (nullable)
 * receives the gradient of its initial state.
 */
gdn_status gdn_apply_state_bwd(const gdn_problem* p, const void* q, const void* k,
                               const void* v, const void* a, const void* b, const float* A_log,
                               const float* dt_bias, const float* Hin,
                               const int32_t* valid_len, const void* dO, const float* dHout,
                               void* dq, void* dk, void* dv, float* dg, float* dbeta,
                               float* dHin, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * Profiling aid (no counterpart on the pages): gdn_fwd and gdn_bwd are a short
 * sequence of kernel launches.  gdn_kernel_info gives, for `op` (GDN_OP_FWD or
 * GDN_OP_BWD) and problem p, the number of launches (*count, nullable) and the
 * name of launch `index` (*name, nullable; a static string); GDN_OP_FWD_CTX and
 * GDN_OP_BWD_CTX list the launches of gdn_fwd_ctx and gdn_bwd_ctx.  gdn_fwd_kernel /
 * gdn_bwd_kernel take the arguments of gdn_fwd / gdn_bwd plus `index` and
 * launch only that kernel, so that a caller can time it alone with CUDA events.
 * They read the intermediates that the earlier kernels of the full call left in
 * the workspace: call the full gdn_fwd / gdn_bwd with the same arguments and
 * workspace first.  Results of the full call are unchanged by re-running a
 * kernel (every launch rewrites what it writes).
 */
gdn_status gdn_kernel_info(const gdn_problem* p, int32_t op, int32_t index, int32_t* count,
                           const char** name);
gdn_status gdn_fwd_kernel(const gdn_problem* p, int32_t index, const void* q, const void* k,
                          const void* v, const void* a, const void* b, const float* A_log,
                          const float* dt_bias, const float* h0, const int32_t* valid_len,
                          void* o, float* hT, void* workspace, size_t workspace_bytes,
                          void* stream);
gdn_status gdn_bwd_kernel(const gdn_problem* p, int32_t index, const void* q, const void* k,
                          const void* v, const void* a, const void* b, const float* A_log,
                          const float* dt_bias, const float* h0, const int32_t* valid_len,
                          const void* dO, const float* dHT, void* dq, void* dk, void* dv,
                          float* dg, float* dbeta, float* dH0, void* workspace,
                          size_t workspace_bytes, void* stream);
gdn_status gdn_fwd_ctx_kernel(const gdn_problem* p, int32_t index, const void* q, const void* k,
                              const void* v, const void* a, const void* b, const float* A_log,
                              const float* dt_bias, const float* h0, const int32_t* valid_len,
                              void* o, float* hT, void* ctx, size_t ctx_bytes, void* workspace,
                              size_t workspace_bytes, void* stream);
gdn_status gdn_bwd_ctx_kernel(const gdn_problem* p, int32_t index, const void* q, const void* k,
                              const void* v, const void* a, const void* b, const float* A_log,
                              const float* dt_bias, const void* ctx, size_t ctx_bytes,
                              const int32_t* valid_len, const void* dO, const float* dHT,
                              void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dH0,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward without a caller-provided workspace (no counterpart on the pages).
 * For callers that cannot allocate device memory or hand the library a buffer:
 * code running while a stream is being captured into a CUDA graph (where a
 * cudaMalloc would break the capture), operator plugins of inference runtimes
 * that give an operator no workspace hook, or hosts whose allocator must not be
 * entered from this call.  Same arguments and results as gdn_fwd, minus the
 * workspace.  Scratch is one static device array of GDN_NOALLOC_SCRATCH_BYTES
 * (64 MiB) that every GPU which loads the library reserves until the process
 * exits; problems whose gdn_workspace_size(p, GDN_OP_FWD) exceeds it are
 * rejected with GDN_ERR_UNSUPPORTED before any launch.  Nothing is allocated:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls on a device share the array, which
 * keeps the last call's contents; each call clears the part that must start at
 * zero (its status word) and overwrites the rest before reading it.  Calls that
 * can run at the same time on one GPU (on different streams, or issued from
 * host threads without an order between them) race on the array: the caller
 * must order them.  Faults that its kernels find (a valid_len outside [0, T], an
 * exhausted bounded wait) are recorded in the status word at the start of the
 * array and read with gdn_noalloc_check_device_status.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (64u << 20)
gdn_status gdn_fwd_noalloc(const gdn_problem* p, const void* q, const void* k, const void* v,
                           const void* a, const void* b, const float* A_log,
                           const float* dt_bias, const float* h0, const int32_t* valid_len,
                           void* o, float* hT, void* stream);

/*
 * gdn_check_device_status for gdn_fwd_noalloc (no counterpart on the pages):
 * synchronises `stream`, reads the status word of this device's static scratch
 * array, clears it and returns what gdn_check_device_status would.  The first
 * call on a device looks up the array's address, as gdn_fwd_noalloc does.
 */
gdn_status gdn_noalloc_check_device_status(void* stream);

/*
 * Synchronises `stream`, reads the device status word of `workspace` (written by
 * earlier calls that used it), clears it and returns GDN_OK,
 * GDN_ERR_INVALID_ARG (a kernel clamped a valid_len outside [0, T]),
 * GDN_ERR_DEVICE_TIMEOUT (a bounded wait ran out) or GDN_ERR_CUDA.
 */
gdn_status gdn_check_device_status(void* workspace, void* stream);

/*
 * Causal depthwise Conv1D + SiLU over time: the step that feeds q, k, v to the core
 * ("linear attention cp #1035", section "What does this PR do": the depthwise Conv1D
 * runs before the Gated DeltaNet, and in its "p2p" mode each rank exchanges only the
 * left halo that the Conv1D needs with its neighbour).  For row b and channel c, with
 * x~ the row preceded by the K - 1 halo tokens (zeros when halo is null):
 *   a[t] = bias[c] + sum_{i<K} w[c][i] x~[t - (K-1) + i],   y[t] = a[t] sigmoid(a[t]).
 * Backward: dx and dhalo (the gradient of the halo tokens, for the rank that sent
 * them), dw = sum_{b,t} ds x~, dbias = sum_{b,t} ds with ds = dy * silu'(a).
 * Layouts (channel innermost): x, y, dy, dx [B][T_stride][C], the first T tokens of
 * each row used; halo, dhalo [B][K-1][C]; w, dw [C][K] and bias, dbias [C] fp32.
 * x, y, dy, dx, halo, dhalo are in p->dtype (GDN_BF16 or GDN_FP32); fp32 arithmetic;
 * dw and dbias are summed in a fixed order (deterministic).  bias, halo (both calls)
 * and dbias, dhalo (backward) may be null.  The caller owns every buffer; the calls
 * are stream-ordered and never synchronise.  Errors: null required pointer, a pointer
 * not 16-byte aligned, B or T < 0, C < 1, T_stride < T: GDN_ERR_INVALID_ARG; C times the
 * element size not a multiple of 16 bytes (C % 8 for bf16, C % 4 for fp32) or K outside
 * 1..4: GDN_ERR_UNSUPPORTED; workspace smaller than gdn_conv_silu_bwd_workspace_size:
 * GDN_ERR_WORKSPACE.
 */
typedef struct {
  int32_t dtype;    /* GDN_BF16 or GDN_FP32 */
  int32_t K;        /* taps, 1..4 */
  int64_t B, T, C;  /* rows, tokens, channels */
  int64_t T_stride; /* tokens between the rows of x, y, dy, dx; 0 means T */
} gdn_conv_problem;

gdn_status gdn_conv_silu_fwd(const gdn_conv_problem* p, const void* x, const float* w,
                             const float* bias, const void* halo, void* y, void* stream);
gdn_status gdn_conv_silu_bwd_workspace_size(const gdn_conv_problem* p, size_t* bytes);
gdn_status gdn_conv_silu_bwd(const gdn_conv_problem* p, const void* x, const float* w,
                             const float* bias, const void* halo, const void* dy, void* dx,
                             float* dw, float* dbias, void* dhalo, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * The Conv1D + SiLU fused into the core's forward ("linear attention cp #1035", section
 * "What does this PR do": the depthwise Conv1D feeds q, k and v of the Gated DeltaNet; the
 * test report "Linear Attention CP 融合算子 PR #1114 测试报告" lists the fused Conv1D as not
 * yet done there).  Result: for i = q, k, v, y[i] = gdn_conv_silu_fwd of x[i] (channels
 * Hqk*dk, Hqk*dk, H*dv; taps K; same B, T, T_stride as p; the same bits), followed by
 * gdn_fwd (ctx NULL) or gdn_fwd_ctx (ctx set) with q, k, v = y[0], y[1], y[2].  On the bf16
 * tensor-core path (dk = dv = 128) the chunk prologue reads x itself: each chunk's x tiles
 * and the K - 1 tokens before them are convolved in shared memory and y is written once
 * from there, so q, k and v are never read back for the prologue; the other paths run the
 * stand-alone Conv1D, then the forward.  y holds every token of every chunk that has a valid
 * token; with valid_len, the tokens of chunks of padding only are zero.  The backward of a
 * training step is gdn_bwd_ctx on q, k, v = y, then gdn_conv_silu_bwd on each of x_q, x_k,
 * x_v with dy = dq, dk, dv.
 * Layouts: x[i], y[i] as q, k, v (p->dtype); w[i] [channels][K] fp32; bias[i] [channels]
 * fp32 or NULL; halo[i] [B][K-1][channels] in p->dtype or NULL (zeros before token 0).
 * Workspace: gdn_workspace_size of GDN_OP_FWD (ctx NULL) or GDN_OP_FWD_CTX.  Errors: those
 * of gdn_fwd / gdn_fwd_ctx; a null or misaligned x, w or y, a misaligned bias or halo, or a
 * y that overlaps its x: GDN_ERR_INVALID_ARG; K outside 1..4: GDN_ERR_UNSUPPORTED.
 */
typedef struct gdn_conv_qkv {
  int32_t K;             /* taps, 1..4 */
  const void* x[3];      /* x_q, x_k, x_v: pre-activation inputs, layouts of q, k, v */
  const float* w[3];     /* taps [channels][K] */
  const float* bias[3];  /* [channels] or NULL */
  const void* halo[3];   /* [B][K-1][channels] or NULL */
  void* y[3];            /* written: q, k, v = SiLU(conv(x)) */
} gdn_conv_qkv;

gdn_status gdn_fwd_conv(const gdn_problem* p, const gdn_conv_qkv* conv, const void* a,
                        const void* b, const float* A_log, const float* dt_bias, const float* h0,
                        const int32_t* valid_len, void* o, float* hT, void* ctx, size_t ctx_bytes,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Packed variable-length rows (several sequences in one row, each with its own state):
 * the test report's variable-length training samples ("Linear Attention CP 融合算子
 * PR #1114 测试报告", section 5.2, there as trailing padding of each batch row)
 * generalised to any number of samples per row.  Sequence i is the tokens
 * cu[i] .. cu[i+1]-1 of the row; it runs the gated delta rule from h0[i] (zero when h0
 * is NULL) and ends in h_T[i]; nothing flows across a boundary.  Gradients are those of
 * sum_t <dO_t, o_t> + sum_i <dHT[i], h_T[i]>.
 *  - p: B = 1, T = the row's token count (T_stride 0 or T); the other fields as gdn_fwd.
 *  - cu_seqlens: DEVICE int32 [n_seqs + 1]; cu_seqlens_host: the same offsets in HOST
 *    memory (0 = cu[0] <= cu[1] <= ... <= cu[n_seqs] = T), read during the call to size
 *    the launches; the two must agree.  A device copy that does not (an offset outside
 *    [0, T] or a length above the host copy's longest) is recorded in the status word
 *    and its sequence skipped; read it with gdn_varlen_check_device_status.
 *  - q, k [1,T,Hqk,dk], v, o, dO, dv [1,T,H,dv], a, b, dg, dbeta [1,T,H] as in gdn_fwd /
 *    gdn_bwd; h0, hT, dHT, dH0 [n_seqs,H,dk,dv] fp32 (nullable as in gdn_fwd / gdn_bwd).
 *  - Work: the sequences are copied into a padded batch [n_seqs, Lmax] (Lmax = the
 *    longest sequence) inside the workspace, run by the batched path with valid_len = the
 *    lengths, and the outputs copied back; on the bf16 path the chunks of the padded
 *    tails are skipped (their outputs zeroed), on the fp32 path they cost masked work.
 *  - Workspace: gdn_varlen_workspace_size (op GDN_OP_FWD or GDN_OP_BWD), 256-byte aligned.
 * Errors: as gdn_fwd / gdn_bwd; offsets that are not non-decreasing from 0 to T, B != 1
 * or n_seqs < 0: GDN_ERR_INVALID_ARG; more than 65535 sequences, or a longest sequence
 * whose widest token row (H dv or Hqk dk elements) spans 2^31 bytes or more:
 * GDN_ERR_UNSUPPORTED.  n_seqs = 0 (T = 0) does nothing.
 */
gdn_status gdn_varlen_workspace_size(const gdn_problem* p, const int32_t* cu_seqlens_host,
                                     int32_t n_seqs, int32_t op, size_t* bytes);
gdn_status gdn_fwd_varlen(const gdn_problem* p, const int32_t* cu_seqlens,
                          const int32_t* cu_seqlens_host, int32_t n_seqs, const void* q,
                          const void* k, const void* v, const void* a, const void* b,
                          const float* A_log, const float* dt_bias, const float* h0, void* o,
                          float* hT, void* workspace, size_t workspace_bytes, void* stream);
gdn_status gdn_bwd_varlen(const gdn_problem* p, const int32_t* cu_seqlens,
                          const int32_t* cu_seqlens_host, int32_t n_seqs, const void* q,
                          const void* k, const void* v, const void* a, const void* b,
                          const float* A_log, const float* dt_bias, const float* h0,
                          const void* dO, const float* dHT, void* dq, void* dk, void* dv,
                          float* dg, float* dbeta, float* dH0, void* workspace,
                          size_t workspace_bytes, void* stream);
/* Synchronises `stream`, then reads and clears the status words of a varlen call's
   workspace (its own and the batched call's): GDN_ERR_DEVICE_TIMEOUT, GDN_ERR_INVALID_ARG
   (device offsets disagreed with the host copy, or a clamped length) or GDN_OK. */
gdn_status gdn_varlen_check_device_status(void* workspace, const gdn_problem* p,
                                          const int32_t* cu_seqlens_host, int32_t n_seqs,
                                          int32_t op, void* stream);

/*
 * Gated RMSNorm on the core's output: the step after the core ("linear attention cp
 * #1035", section "What does this PR do": the output goes through RMSNorm, the gate and
 * the output projection; the test report names the module "RMSNormGated").  For every
 * row of D elements (one token and V head of o [B,T,H,dv]: rows = B*T*H, D = dv), with
 * r = 1 / sqrt(mean(o^2) + eps):   y = o r w silu(z).
 * Backward: do = r (dn - (o r) mean(dn o r)) with dn = dy w silu(z); dz = dy o r w silu'(z);
 * dw = sum over rows of dy o r silu(z) (fixed-order sum: deterministic).
 * Layouts: o, z, y, dy, do, dz [rows][D] contiguous in p->dtype (GDN_BF16 or GDN_FP32);
 * w, dw [D] fp32.  fp32 arithmetic.  The caller owns every buffer; stream-ordered, no
 * synchronisation.  Errors: null or not 16-byte aligned pointer, rows < 0, D < 1,
 * eps < 0: GDN_ERR_INVALID_ARG; D not a multiple of 4 or above 512: GDN_ERR_UNSUPPORTED;
 * workspace smaller than gdn_rmsnorm_gated_bwd_workspace_size: GDN_ERR_WORKSPACE.
 */
typedef struct {
  int32_t dtype;  /* GDN_BF16 or GDN_FP32 */
  int32_t D;      /* elements per row, a multiple of 4, at most 512 */
  int64_t rows;
  float eps;      /* 1e-6 in the layers the pages test */
} gdn_rmsnorm_problem;

gdn_status gdn_rmsnorm_gated_fwd(const gdn_rmsnorm_problem* p, const void* o, const void* z,
                                 const float* w, void* y, void* stream);
gdn_status gdn_rmsnorm_gated_bwd_workspace_size(const gdn_rmsnorm_problem* p, size_t* bytes);
gdn_status gdn_rmsnorm_gated_bwd(const gdn_rmsnorm_problem* p, const void* o, const void* z,
                                 const float* w, const void* dy, void* d_o, void* dz, float* dw,
                                 void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
