// gdn_tc_common.cuh -- sm_103a building blocks for the tensor-core kernels:
// mbarriers with bounded waits, TMA tile loads, shared-memory matrix
// descriptors (128-byte swizzle), tcgen05.mma (bf16 -> fp32 in TMEM), TMEM
// allocation and loads, and the swizzled addressing used to stage operands
// from registers.
//
// Operand layouts (bf16, 128-byte swizzle, tile base 1024-byte aligned):
//  K-major tile (rows x 64 elements along K): element (r, k) at
//    r*128 + (((k>>3) ^ (r&7)) << 4) + (k&7)*2; 8-row groups 1024 B apart (SBO);
//    a K step of 16 elements advances the descriptor start by 32 B.
//  MN-major tile (K rows, N contiguous): element (k, n) at
//    (n>>6)*LBO + (k>>3)*1024 + (k&7)*128 + ((((n&63)>>3) ^ (k&7)) << 4) + (n&7)*2;
//    a K step of 16 rows advances the start by 2048 B.
//  M = 128 accumulators: row m lives in TMEM lane m, column n in column n.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace tc {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded waits give up after 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Wait for the phase with parity `parity` of `bar` to complete, for at most
// kWaitLimitNs; returns false (and sets `timeout_bit` in *status) on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          int timeout_bit) {
  const uint32_t addr = smem_u32(bar);
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if (it == 0) t0 = global_timer();
    else if (global_timer() - t0 > kWaitLimitNs) {
      if (status) atomicOr(status, timeout_bit);
      return false;
    }
  }
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 4-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// Plain (untiled) bulk copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"((uint64_t)src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Hints that pull global data into L2 ahead of a later load (no completion to wait on).
__device__ __forceinline__ void l2_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"((uint64_t)src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void l2_prefetch_tile(const CUtensorMap* map, int c0, int c1, int c2,
                                                 int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   (uint64_t)map),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// Bulk copy of `bytes` from shared to global memory (same alignment rules), in
// this thread's bulk group; bulk_commit() closes the group, bulk_wait_read()
// waits until every committed group has finished reading shared memory.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   (uint64_t)dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
// 4-D tiled TMA store of one box from shared memory (boxes outside the tensor are clipped).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int c0, int c1,
                                             int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          (uint64_t)map),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// ... every committed group but the most recent one
__device__ __forceinline__ void bulk_wait_read_but1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, M x N, A/B K-major (0) or MN-major (1).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole-warp TMEM allocation; the base address is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols));
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-wide).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// Two 32-column loads of this thread's TMEM lane issued together, one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, float (&va)[32], uint32_t tb,
                                            float (&vb)[32]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    va[j] = __uint_as_float(r[j]);
    vb[j] = __uint_as_float(r[32 + j]);
  }
}

// Two 32-column stores to this thread's TMEM lane (warp-wide), then one wait: the stores
// are complete in TMEM when it returns (an MMA issued after a tcgen05 fence and a thread
// barrier sees them).
__device__ __forceinline__ void tmem_st32x2(uint32_t ta, const float (&va)[32], uint32_t tb,
                                            const float (&vb)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};\n"
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%1], {%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65};\n"
      "tcgen05.wait::st.sync.aligned;"
      :: "r"(ta), "r"(tb),
      "r"(__float_as_uint(va[0])), "r"(__float_as_uint(va[1])), "r"(__float_as_uint(va[2])), "r"(__float_as_uint(va[3])), "r"(__float_as_uint(va[4])), "r"(__float_as_uint(va[5])), "r"(__float_as_uint(va[6])), "r"(__float_as_uint(va[7])), "r"(__float_as_uint(va[8])), "r"(__float_as_uint(va[9])), "r"(__float_as_uint(va[10])), "r"(__float_as_uint(va[11])), "r"(__float_as_uint(va[12])), "r"(__float_as_uint(va[13])), "r"(__float_as_uint(va[14])), "r"(__float_as_uint(va[15])), "r"(__float_as_uint(va[16])), "r"(__float_as_uint(va[17])), "r"(__float_as_uint(va[18])), "r"(__float_as_uint(va[19])), "r"(__float_as_uint(va[20])), "r"(__float_as_uint(va[21])), "r"(__float_as_uint(va[22])), "r"(__float_as_uint(va[23])), "r"(__float_as_uint(va[24])), "r"(__float_as_uint(va[25])), "r"(__float_as_uint(va[26])), "r"(__float_as_uint(va[27])), "r"(__float_as_uint(va[28])), "r"(__float_as_uint(va[29])), "r"(__float_as_uint(va[30])), "r"(__float_as_uint(va[31])),
      "r"(__float_as_uint(vb[0])), "r"(__float_as_uint(vb[1])), "r"(__float_as_uint(vb[2])), "r"(__float_as_uint(vb[3])), "r"(__float_as_uint(vb[4])), "r"(__float_as_uint(vb[5])), "r"(__float_as_uint(vb[6])), "r"(__float_as_uint(vb[7])), "r"(__float_as_uint(vb[8])), "r"(__float_as_uint(vb[9])), "r"(__float_as_uint(vb[10])), "r"(__float_as_uint(vb[11])), "r"(__float_as_uint(vb[12])), "r"(__float_as_uint(vb[13])), "r"(__float_as_uint(vb[14])), "r"(__float_as_uint(vb[15])), "r"(__float_as_uint(vb[16])), "r"(__float_as_uint(vb[17])), "r"(__float_as_uint(vb[18])), "r"(__float_as_uint(vb[19])), "r"(__float_as_uint(vb[20])), "r"(__float_as_uint(vb[21])), "r"(__float_as_uint(vb[22])), "r"(__float_as_uint(vb[23])), "r"(__float_as_uint(vb[24])), "r"(__float_as_uint(vb[25])), "r"(__float_as_uint(vb[26])), "r"(__float_as_uint(vb[27])), "r"(__float_as_uint(vb[28])), "r"(__float_as_uint(vb[29])), "r"(__float_as_uint(vb[30])), "r"(__float_as_uint(vb[31]))
      : "memory");
}

// Several loads of this thread's TMEM lane issued back to back, then one wait: the
// loads overlap instead of each paying the full round trip.  (One asm statement, so that
// no use of a loaded register can be scheduled before the wait.)
__device__ __forceinline__ void tmem_ld16x2(uint32_t a0, uint32_t a1,
    float (&v0)[16], float (&v1)[16]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,"
      "%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,"
      "%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(a0), "r"(a1)
      : "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v0[j] = __uint_as_float(r[0 + j]);
#pragma unroll
  for (int j = 0; j < 16; ++j) v1[j] = __uint_as_float(r[16 + j]);
}
__device__ __forceinline__ void tmem_ld16x3(uint32_t a0, uint32_t a1, uint32_t a2,
    float (&v0)[16], float (&v1)[16], float (&v2)[16]) {
  uint32_t r[48];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,"
      "%8,%9,%10,%11,%12,%13,%14,%15}, [%48];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,"
      "%24,%25,%26,%27,%28,%29,%30,%31}, [%49];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,"
      "%40,%41,%42,%43,%44,%45,%46,%47}, [%50];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]),
        "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
        "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
      : "r"(a0), "r"(a1), "r"(a2)
      : "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v0[j] = __uint_as_float(r[0 + j]);
#pragma unroll
  for (int j = 0; j < 16; ++j) v1[j] = __uint_as_float(r[16 + j]);
#pragma unroll
  for (int j = 0; j < 16; ++j) v2[j] = __uint_as_float(r[32 + j]);
}
__device__ __forceinline__ void tmem_ld16x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
    float (&v0)[16], float (&v1)[16], float (&v2)[16], float (&v3)[16]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,"
      "%8,%9,%10,%11,%12,%13,%14,%15}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,"
      "%24,%25,%26,%27,%28,%29,%30,%31}, [%65];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,"
      "%40,%41,%42,%43,%44,%45,%46,%47}, [%66];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%48,%49,%50,%51,%52,%53,%54,%55,"
      "%56,%57,%58,%59,%60,%61,%62,%63}, [%67];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]),
        "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
        "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]),
        "=r"(r[63])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3)
      : "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v0[j] = __uint_as_float(r[0 + j]);
#pragma unroll
  for (int j = 0; j < 16; ++j) v1[j] = __uint_as_float(r[16 + j]);
#pragma unroll
  for (int j = 0; j < 16; ++j) v2[j] = __uint_as_float(r[32 + j]);
#pragma unroll
  for (int j = 0; j < 16; ++j) v3[j] = __uint_as_float(r[48 + j]);
}

// Byte offsets inside 128-byte-swizzled tiles (see the header comment).
__device__ __forceinline__ uint32_t kmaj_chunk(int r, int c) {  // 16-byte chunk c of row r
  return (uint32_t)(r * 128 + (((c ^ r) & 7) << 4));
}
__device__ __forceinline__ uint32_t mnmaj_chunk(int k, int c, uint32_t lbo) {  // n = 8c .. 8c+7
  return (uint32_t)((c >> 3) * lbo + (k >> 3) * 1024 + (k & 7) * 128 + ((((c & 7) ^ k) & 7) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Store 8 floats as bf16 into a 16-byte chunk.
__device__ __forceinline__ void st_chunk(uint8_t* base, uint32_t off, const float* x) {
  uint4 v;
  v.x = pack_bf16(x[0], x[1]);
  v.y = pack_bf16(x[2], x[3]);
  v.z = pack_bf16(x[4], x[5]);
  v.w = pack_bf16(x[6], x[7]);
  *reinterpret_cast<uint4*>(base + off) = v;
}

// Load a 16-byte chunk of 8 bf16 as floats.
__device__ __forceinline__ void ld_chunk(const uint8_t* base, uint32_t off, float* x) {
  const uint4 v = *reinterpret_cast<const uint4*>(base + off);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    const float2 f = __bfloat1622float2(b);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// Multiply a 16-byte chunk of 8 bf16 in place by f (rounded to bf16), two at a time.
__device__ __forceinline__ void scale_chunk(uint8_t* base, uint32_t off, float f) {
  uint4 v = *reinterpret_cast<const uint4*>(base + off);
  const __nv_bfloat162 f2 = __float2bfloat162_rn(f);
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    b = __hmul2(b, f2);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(base + off) = v;
}

// Leading dim of the fp32 64 x 64 tiles of the solve: 68 = 4 (mod 32) makes the tf32 A-fragment
// loads (rows g, columns t) conflict-free and the B-fragment loads (rows t, columns g) 2-way;
// rows stay 16-byte aligned for vector stores.
constexpr int LDA = 68;

// Cumulative gates are kept in fp32 and in log2 units (G * log2 e), so every
// decay factor is one exp2f of a difference; fp32 is ample at bf16 tolerance
// (the fp64 pipe of this part is far too slow for 8K differences per chunk).
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float dexp_(float ga, float gb) { return exp2f(ga - gb); }

// Inclusive prefix sum of x[0..63] in place, by warp 0.
__device__ __forceinline__ void cumsum64f(float* x) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float v0 = x[lane], v1 = x[lane + 32];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y0 = __shfl_up_sync(0xffffffffu, v0, o);
      const float y1 = __shfl_up_sync(0xffffffffu, v1, o);
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

// One warp-level tensor-core step D = A B + D on a 16 x 8 tile, tf32 operands
// (fp32 rounded to nearest), fp32 accumulation.  Fragment ownership (g = lane / 4,
// t = lane % 4): a0 (g, t), a1 (g+8, t), a2 (g, t+4), a3 (g+8, t+4);
// b0 (t, g), b1 (t+4, g); c0 (g, 2t), c1 (g, 2t+1), c2 (g+8, 2t), c3 (g+8, 2t+1).
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32_16x8x8(float (&c)[4], const float (&a)[4],
                                                const float (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(to_tf32(a[0])), "r"(to_tf32(a[1])), "r"(to_tf32(a[2])), "r"(to_tf32(a[3])),
        "r"(to_tf32(b[0])), "r"(to_tf32(b[1])));
}

// Receiver of the entries of T as the solve finalises them (nothing by default).
struct NoEmit {
  __device__ __forceinline__ void one(int, int, float) const {}
  __device__ __forceinline__ void two(int, int, float, float) const {}
};

// T = (I + A)^-1 for strictly lower A (64 x 64, fp32, leading dim lda).  The
// 16 x 16 diagonal blocks come from forward substitution on CUDA cores (four lanes per
// column of T, every thread of the CTA); the blocks below them, block diagonal by block
// diagonal, from T_ij = -T_ii (sum_{j <= m < i} A_im T_mj) with warp-level tf32 MMAs (one
// warp per 16 x 8 half block).  Y needs 8 warps x 128 floats.  Needs blockDim.x == 256.
// Every entry on or below the diagonal is also handed to emit.one(i, j, t) or, for
// the column pair j, j + 1 (j even), emit.two(i, j, t_j, t_j+1) once it is final.
template <typename Emit = NoEmit>
__device__ __forceinline__ void solve_unit_lower64_mma(const float* A, float* T, float* Y,
                                                       const int lda, const Emit& emit = Emit()) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    // column j of diagonal block b0 / 16, by columns of A: once x_l is final it is removed
    // from every later row.  Lane q of the column's four owns rows q, q + 4, q + 8, q + 12
    // and hands x_l to the other three when it owns row l, so each lane does a quarter of
    // the updates and the dependent chain is 15 shuffle + FMA steps.
    const int col = tid >> 2, q = tid & 3;
    const int b0 = (col >> 4) * 16, j = col & 15;
    float x[4];
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) x[sl] = (q + 4 * sl == j) ? 1.f : 0.f;
#pragma unroll
    for (int l = 0; l < 15; ++l) {
      const float xl = __shfl_sync(0xffffffffu, x[l >> 2], l & 3, 4);
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
        const int r = q + 4 * sl;
        const float y = fmaf(-A[(b0 + r) * lda + b0 + l], xl, x[sl]);
        x[sl] = r > l ? y : x[sl];
      }
    }
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
      const int r = q + 4 * sl;
      T[(b0 + r) * lda + b0 + j] = x[sl];  // zero above the diagonal (x = 0 for r < j)
      if (r >= j) emit.one(b0 + r, b0 + j, x[sl]);
    }
  }
  __syncthreads();
  const int g = lane >> 2, t = lane & 3;
  float* Yw = Y + warp * 128;  // [16][8] scratch of this warp
  for (int d = 1; d <= 3; ++d) {
    if (warp < 2 * (4 - d)) {
      const int bj = warp >> 1, bi = bj + d, r0 = bi * 16, n0 = bj * 16 + (warp & 1) * 8;
      // Y = A[bi, bj..bi) T[bj..bi, bj], the 8-wide K steps alternating between two
      // accumulators so that two MMA chains are in flight
      float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
      for (int m = bj * 16; m < bi * 16; m += 16) {
#pragma unroll
        for (int h8 = 0; h8 < 16; h8 += 8) {
          const int mm = m + h8;
          const float a[4] = {A[(r0 + g) * lda + mm + t], A[(r0 + g + 8) * lda + mm + t],
                              A[(r0 + g) * lda + mm + t + 4], A[(r0 + g + 8) * lda + mm + t + 4]};
          const float b[2] = {T[(mm + t) * lda + n0 + g], T[(mm + t + 4) * lda + n0 + g]};
          if (h8 == 0) mma_tf32_16x8x8(c, a, b);
          else mma_tf32_16x8x8(c2, a, b);
        }
      }
      Yw[g * 8 + 2 * t] = c[0] + c2[0];
      Yw[g * 8 + 2 * t + 1] = c[1] + c2[1];
      Yw[(g + 8) * 8 + 2 * t] = c[2] + c2[2];
      Yw[(g + 8) * 8 + 2 * t + 1] = c[3] + c2[3];
      __syncwarp();
      float e[4] = {0.f, 0.f, 0.f, 0.f}, e2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 16; k += 8) {  // T_ij = -T_ii Y (two independent products, summed)
        const float a[4] = {T[(r0 + g) * lda + r0 + k + t], T[(r0 + g + 8) * lda + r0 + k + t],
                            T[(r0 + g) * lda + r0 + k + t + 4],
                            T[(r0 + g + 8) * lda + r0 + k + t + 4]};
        const float b[2] = {Yw[(k + t) * 8 + g], Yw[(k + t + 4) * 8 + g]};
        if (k == 0) mma_tf32_16x8x8(e, a, b);
        else mma_tf32_16x8x8(e2, a, b);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) e[q] += e2[q];
      T[(r0 + g) * lda + n0 + 2 * t] = -e[0];
      T[(r0 + g) * lda + n0 + 2 * t + 1] = -e[1];
      T[(r0 + g + 8) * lda + n0 + 2 * t] = -e[2];
      T[(r0 + g + 8) * lda + n0 + 2 * t + 1] = -e[3];
      emit.two(r0 + g, n0 + 2 * t, -e[0], -e[1]);
      emit.two(r0 + g + 8, n0 + 2 * t, -e[2], -e[3]);
    }
    __syncthreads();
  }
}

}  // namespace tc
}  // namespace gdn
