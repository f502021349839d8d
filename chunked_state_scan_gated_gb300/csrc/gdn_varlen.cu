// gdn_varlen.cu -- packed variable-length rows: several sequences in one row, each run
// from its own initial state with nothing flowing across a boundary.  The test report of
// "Linear Attention CP 融合算子 PR #1114" (section 5.2) covers variable-length training
// samples through trailing padding of each batch row (B = 2, valid_length = 7777); a
// packed row generalises it to any number of samples per row.
//
// The call lays the N packed sequences out as the rows of a padded batch [N, Lmax]
// (each sequence at the start of its own row, zeros after its length), runs the batched
// path with valid_len = the lengths (the masked path of the same report: padded tokens
// leave the state unchanged and get zero output and gradients), and copies the valid
// tokens of each output back into the packed row.  h0, h_T, dH_T and dH0 of sequence i
// are row i of the batch, so they need no copy.  The copies are bandwidth-bound 16-byte
// moves; the tensor-core path skips the chunks of a row's padded tail (only their
// outputs are zeroed).
#include <string.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of one varlen call: lengths, padded copies of the inputs and outputs, then
// the batched call's own workspace.
struct VLayout {
  size_t vlen = 0;           // int32 [N]: valid_len of the padded batch
  size_t status = 0;         // int32: bit kStatusClamped when cu_seqlens (device) was bad
  size_t in[6] = {};         // q, k, v, a, b, dO (padded, I/O dtype)
  size_t out[5] = {};        // fwd: o; bwd: dq, dk, dv, dg, dbeta (padded)
  size_t inner = 0;          // the batched call's workspace
  size_t inner_bytes = 0;
  size_t total = 0;
};

struct Shape {
  gdn_problem inner;  // the padded batch problem
  int64_t N, Lmax, T;
  size_t esz;
};

gdn_status shape_of(const gdn_problem* p, const int32_t* cu_host, int32_t n_seqs, Shape* s) {
  if (!p || n_seqs < 0 || (n_seqs > 0 && !cu_host)) return GDN_ERR_INVALID_ARG;
  if (p->B != 1 || (p->T_stride != 0 && p->T_stride != p->T)) return GDN_ERR_INVALID_ARG;
  gdn_status st = gdn_query_support(p);
  if (st != GDN_OK) return st;
  if (n_seqs == 0) {
    if (p->T != 0) return GDN_ERR_INVALID_ARG;
  } else {
    if (cu_host[0] != 0 || cu_host[n_seqs] != p->T) return GDN_ERR_INVALID_ARG;
  }
  int64_t Lmax = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    const int64_t L = (int64_t)cu_host[i + 1] - cu_host[i];
    if (L < 0) return GDN_ERR_INVALID_ARG;
    if (L > Lmax) Lmax = L;
  }
  // the copies index a sequence's bytes in 32 bits and take one grid row per sequence
  const int64_t esz = p->dtype == GDN_BF16 ? 2 : 4;
  const int64_t widest = (p->H * p->dv > p->Hqk * p->dk ? p->H * p->dv : p->Hqk * p->dk) * esz;
  if (n_seqs > 65535 || Lmax * widest >= ((int64_t)1 << 31)) return GDN_ERR_UNSUPPORTED;
  s->inner = *p;
  s->inner.B = n_seqs;
  s->inner.T = Lmax;
  s->inner.T_stride = 0;
  s->N = n_seqs;
  s->Lmax = Lmax;
  s->T = p->T;
  s->esz = p->dtype == GDN_BF16 ? 2 : 4;
  if (s->inner.segments > 0) {  // a forced segment count must fit the padded rows
    const int64_t nc = (Lmax + 63) / 64;
    if (s->inner.segments > (nc > 1 ? nc : 1)) s->inner.segments = (int32_t)(nc > 1 ? nc : 1);
  }
  return gdn_query_support(&s->inner);
}

gdn_status layout(const Shape& s, int op, VLayout* L) {
  VLayout l;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  const size_t tok = (size_t)s.N * (size_t)s.Lmax;
  const gdn_problem& q = s.inner;
  l.vlen = take((size_t)s.N * 4 + 4);
  l.status = take(4);
  const size_t qk = tok * q.Hqk * q.dk * s.esz, vv = tok * q.H * q.dv * s.esz,
               gg = tok * q.H * s.esz, g32 = tok * q.H * 4;
  l.in[0] = take(qk);
  l.in[1] = take(qk);
  l.in[2] = take(vv);
  l.in[3] = take(gg);
  l.in[4] = take(gg);
  if (op == GDN_OP_BWD) {
    l.in[5] = take(vv);
    l.out[0] = take(qk);
    l.out[1] = take(qk);
    l.out[2] = take(vv);
    l.out[3] = take(g32);
    l.out[4] = take(g32);
  } else {
    l.out[0] = take(vv);
  }
  size_t ib = 0;
  if (s.N > 0) {
    gdn_status st = gdn_workspace_size(&q, op, &ib);
    if (st != GDN_OK) return st;
  }
  l.inner = take(ib);
  l.inner_bytes = ib;
  l.total = off;
  *L = l;
  return GDN_OK;
}

// valid_len[n] = cu[n+1] - cu[n], checked against [0, Lmax] and the row (device copy of
// the offsets; a mismatch with the host copy is recorded and the row treated as empty)
__global__ void k_varlen_lengths(const int32_t* __restrict__ cu, int64_t N, int64_t Lmax,
                                 int64_t T, int32_t* vlen, int* status) {
  const int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const int64_t s = cu[n], e = cu[n + 1];
  int64_t L = e - s;
  if (s < 0 || e > T || L < 0 || L > Lmax) {
    atomicOr(status, kStatusClamped);
    L = 0;
  }
  vlen[n] = (int32_t)L;
}

// Moves `unit`-byte pieces of token rows of `row` bytes between the packed row and the
// padded batch.  Pack = false: padded[n][t] = packed[cu[n] + t] for t < len[n], zero after
// (gather).  Pack = true: packed[cu[n] + t] = padded[n][t] for t < len[n] (scatter).
// grid (x, N): blockIdx.y is the sequence; the x blocks stride over its Lmax * per pieces
// (below 2^31: checked on the host) with 32-bit index arithmetic.
template <typename U, bool Pack>
__global__ void __launch_bounds__(256) k_varlen_move(const int32_t* __restrict__ cu,
                                                     const int32_t* __restrict__ vlen, int64_t N,
                                                     int64_t Lmax, int64_t row,
                                                     const uint8_t* __restrict__ src,
                                                     uint8_t* __restrict__ dst) {
  const uint32_t per = (uint32_t)(row / (int64_t)sizeof(U));  // pieces per token row
  const int64_t n = blockIdx.y;
  const uint32_t span = (uint32_t)Lmax * per;
  const uint32_t lim = (uint32_t)vlen[n] * per;  // pieces of the valid tokens (vlen <= Lmax)
  const int64_t row0 = n * (int64_t)span;  // first piece of the sequence in the padded batch
  const int64_t pk0 = (int64_t)cu[n] * per;  // ... and in the packed row (read when valid)
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < span; i += gridDim.x * blockDim.x) {
    const bool valid = i < lim;
    if (Pack) {
      if (valid) reinterpret_cast<U*>(dst)[pk0 + i] = reinterpret_cast<const U*>(src)[row0 + i];
    } else {
      U v{};
      if (valid) v = reinterpret_cast<const U*>(src)[pk0 + i];
      reinterpret_cast<U*>(dst)[row0 + i] = v;
    }
  }
}

template <bool Pack>
cudaError_t move(const int32_t* cu, const int32_t* vlen, const Shape& s, int64_t row,
                 const void* src, void* dst, cudaStream_t st) {
  const int64_t bytes = s.N * s.Lmax * row;
  if (bytes == 0) return cudaSuccess;
  if (s.Lmax * row >= ((int64_t)1 << 31) || s.N > 65535) return cudaErrorInvalidValue;
  const int64_t per_seq_blocks = (1216 + s.N - 1) / s.N;  // ~1216 CTAs in all
  auto grid = [&](int64_t pieces) {  // pieces of the whole batch
    const int64_t per_seq = (pieces / s.N + 255) / 256;
    return dim3((unsigned)(per_seq < per_seq_blocks ? (per_seq > 0 ? per_seq : 1) : per_seq_blocks),
                (unsigned)s.N);
  };
  const uint8_t* a = (const uint8_t*)src;
  uint8_t* b = (uint8_t*)dst;
  if (row % 16 == 0) {
    k_varlen_move<uint4, Pack><<<grid(bytes / 16), 256, 0, st>>>(cu, vlen, s.N, s.Lmax, row, a, b);
  } else if (row % 8 == 0) {
    k_varlen_move<uint2, Pack><<<grid(bytes / 8), 256, 0, st>>>(cu, vlen, s.N, s.Lmax, row, a, b);
  } else if (row % 4 == 0) {
    k_varlen_move<uint32_t, Pack><<<grid(bytes / 4), 256, 0, st>>>(cu, vlen, s.N, s.Lmax, row,
                                                                   a, b);
  } else {
    k_varlen_move<uint16_t, Pack><<<grid(bytes / 2), 256, 0, st>>>(cu, vlen, s.N, s.Lmax, row,
                                                                   a, b);
  }
  return cudaGetLastError();
}

#define VL_TRY(expr)                           \
  do {                                         \
    cudaError_t e_ = (expr);                   \
    if (e_ != cudaSuccess) return GDN_ERR_CUDA; \
  } while (0)

// Common front: shapes, workspace checks, lengths.
gdn_status begin(const gdn_problem* p, const int32_t* cu_seqlens, const int32_t* cu_host,
                 int32_t n_seqs, int op, void* ws, size_t ws_bytes, cudaStream_t st, Shape* s,
                 VLayout* L) {
  gdn_status r = shape_of(p, cu_host, n_seqs, s);
  if (r != GDN_OK) return r;
  if ((r = layout(*s, op, L)) != GDN_OK) return r;
  if (!ws || ws_bytes < L->total) return GDN_ERR_WORKSPACE;
  if (((uintptr_t)ws & 255u) != 0) return GDN_ERR_INVALID_ARG;
  if (n_seqs > 0 && (!cu_seqlens || ((uintptr_t)cu_seqlens & 3u) != 0)) return GDN_ERR_INVALID_ARG;
  uint8_t* w = (uint8_t*)ws;
  VL_TRY(cudaMemsetAsync(w + L->status, 0, sizeof(int), st));
  if (s->N > 0)
    k_varlen_lengths<<<(unsigned)((s->N + 255) / 256), 256, 0, st>>>(
        cu_seqlens, s->N, s->Lmax, s->T, (int32_t*)(w + L->vlen), (int*)(w + L->status));
  VL_TRY(cudaGetLastError());
  return GDN_OK;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status gdn_varlen_workspace_size(const gdn_problem* p, const int32_t* cu_seqlens_host,
                                     int32_t n_seqs, int32_t op, size_t* bytes) {
  if (!bytes || (op != GDN_OP_FWD && op != GDN_OP_BWD)) return GDN_ERR_INVALID_ARG;
  Shape s;
  gdn_status r = shape_of(p, cu_seqlens_host, n_seqs, &s);
  if (r != GDN_OK) return r;
  VLayout L;
  if ((r = layout(s, op, &L)) != GDN_OK) return r;
  *bytes = L.total;
  return GDN_OK;
}

gdn_status gdn_fwd_varlen(const gdn_problem* p, const int32_t* cu_seqlens,
                          const int32_t* cu_seqlens_host, int32_t n_seqs, const void* q,
                          const void* k, const void* v, const void* a, const void* b,
                          const float* A_log, const float* dt_bias, const float* h0, void* o,
                          float* hT, void* workspace, size_t workspace_bytes, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  Shape s;
  VLayout L;
  if (!p) return GDN_ERR_INVALID_ARG;
  const int64_t T = p->T;
  const void* ins[5] = {q, k, v, a, b};
  for (const void* x : ins)
    if ((T > 0 && !x) || (x && !aligned16(x))) return GDN_ERR_INVALID_ARG;
  if ((T > 0 && !o) || (o && !aligned16(o))) return GDN_ERR_INVALID_ARG;
  gdn_status r = begin(p, cu_seqlens, cu_seqlens_host, n_seqs, GDN_OP_FWD, workspace,
                       workspace_bytes, st, &s, &L);
  if (r != GDN_OK) return r;
  if (s.N == 0) return GDN_OK;
  uint8_t* w = (uint8_t*)workspace;
  const int32_t* vlen = (const int32_t*)(w + L.vlen);
  const gdn_problem& ip = s.inner;
  const int64_t rows[5] = {ip.Hqk * ip.dk * (int64_t)s.esz, ip.Hqk * ip.dk * (int64_t)s.esz,
                           ip.H * ip.dv * (int64_t)s.esz, ip.H * (int64_t)s.esz,
                           ip.H * (int64_t)s.esz};
  for (int i = 0; i < 5; ++i)
    VL_TRY(move<false>(cu_seqlens, vlen, s, rows[i], ins[i], w + L.in[i], st));
  r = gdn_fwd(&ip, w + L.in[0], w + L.in[1], w + L.in[2], w + L.in[3], w + L.in[4], A_log,
              dt_bias, h0, vlen, w + L.out[0], hT, w + L.inner, L.inner_bytes, stream);
  if (r != GDN_OK) return r;
  VL_TRY(move<true>(cu_seqlens, vlen, s, rows[2], w + L.out[0], o, st));
  return GDN_OK;
}

gdn_status gdn_bwd_varlen(const gdn_problem* p, const int32_t* cu_seqlens,
                          const int32_t* cu_seqlens_host, int32_t n_seqs, const void* q,
                          const void* k, const void* v, const void* a, const void* b,
                          const float* A_log, const float* dt_bias, const float* h0,
                          const void* dO, const float* dHT, void* dq, void* dk, void* dv,
                          float* dg, float* dbeta, float* dH0, void* workspace,
                          size_t workspace_bytes, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  Shape s;
  VLayout L;
  if (!p) return GDN_ERR_INVALID_ARG;
  const int64_t T = p->T;
  const void* ins[6] = {q, k, v, a, b, dO};
  void* outs[5] = {dq, dk, dv, dg, dbeta};
  for (const void* x : ins)
    if ((T > 0 && !x) || (x && !aligned16(x))) return GDN_ERR_INVALID_ARG;
  for (const void* x : outs)
    if ((T > 0 && !x) || (x && !aligned16(x))) return GDN_ERR_INVALID_ARG;
  gdn_status r = begin(p, cu_seqlens, cu_seqlens_host, n_seqs, GDN_OP_BWD, workspace,
                       workspace_bytes, st, &s, &L);
  if (r != GDN_OK) return r;
  if (s.N == 0) return GDN_OK;
  uint8_t* w = (uint8_t*)workspace;
  const int32_t* vlen = (const int32_t*)(w + L.vlen);
  const gdn_problem& ip = s.inner;
  const int64_t e = (int64_t)s.esz;
  const int64_t rin[6] = {ip.Hqk * ip.dk * e, ip.Hqk * ip.dk * e, ip.H * ip.dv * e, ip.H * e,
                          ip.H * e, ip.H * ip.dv * e};
  for (int i = 0; i < 6; ++i)
    VL_TRY(move<false>(cu_seqlens, vlen, s, rin[i], ins[i], w + L.in[i], st));
  r = gdn_bwd(&ip, w + L.in[0], w + L.in[1], w + L.in[2], w + L.in[3], w + L.in[4], A_log,
              dt_bias, h0, vlen, w + L.in[5], dHT, w + L.out[0], w + L.out[1], w + L.out[2],
              (float*)(w + L.out[3]), (float*)(w + L.out[4]), dH0, w + L.inner, L.inner_bytes,
              stream);
  if (r != GDN_OK) return r;
  const int64_t rout[5] = {ip.Hqk * ip.dk * e, ip.Hqk * ip.dk * e, ip.H * ip.dv * e, ip.H * 4,
                           ip.H * 4};
  for (int i = 0; i < 5; ++i)
    VL_TRY(move<true>(cu_seqlens, vlen, s, rout[i], w + L.out[i], outs[i], st));
  return GDN_OK;
}

gdn_status gdn_varlen_check_device_status(void* workspace, const gdn_problem* p,
                                          const int32_t* cu_seqlens_host, int32_t n_seqs,
                                          int32_t op, void* stream) {
  if (!workspace || (op != GDN_OP_FWD && op != GDN_OP_BWD)) return GDN_ERR_INVALID_ARG;
  Shape s;
  gdn_status r = shape_of(p, cu_seqlens_host, n_seqs, &s);
  if (r != GDN_OK) return r;
  VLayout L;
  if ((r = layout(s, op, &L)) != GDN_OK) return r;
  uint8_t* w = (uint8_t*)workspace;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
  int own = 0;
  if (cudaMemcpy(&own, w + L.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaMemset(w + L.status, 0, sizeof(int)) != cudaSuccess) return GDN_ERR_CUDA;
  r = s.N > 0 ? gdn_check_device_status(w + L.inner, stream) : GDN_OK;
  if (r == GDN_ERR_DEVICE_TIMEOUT) return r;
  if (own & kStatusClamped) return GDN_ERR_INVALID_ARG;
  return r;
}

}  // extern "C"
