// Device helpers for the sm_103a kernels: mbarrier pipeline with bounded
// waits, TMA tensor loads, ldmatrix / mma.sync fragments, cp.async gathers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/vg.h"

namespace vg {

// A pipeline wait gives up after this many nanoseconds of %globaltimer and
// reports VG_DEVERR_TIMEOUT instead of spinning forever.  A shorter bound
// set with vg_set_wait_limit_ns only reports earlier: the wait then goes on
// up to this bound, so that no copy or tensor-core operation it waits for is
// abandoned while in flight.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void flag_error(int32_t* flag, int code) {
  if (flag) atomicOr(flag, code);
}

// Atomic add with acquire-release semantics at GPU scope: the caller's
// earlier writes (and, after a CTA barrier, its CTA's) are visible to a
// thread that observes the new value, and writes observed through the old
// value are visible to the caller afterwards.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity (no suspension).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Waits whose completion is acquired at cluster scope: for a phase that
// another CTA of the cluster completes with a release at cluster scope.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity.  Past report_ns the wait ORs
// VG_DEVERR_TIMEOUT into *flag and keeps waiting; it returns false (also
// flagged) only when kWaitLimitNs has passed as well.  Under a bound shorter
// than the default it polls with the non-blocking test and reads the timer
// after every poll (a try_wait may itself sleep past a short bound).
// CLUSTER: acquire at cluster scope (see mbar_try_wait_cluster).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_checked(uint64_t* bar, uint32_t parity,
                                                  uint64_t report_ns, int32_t* flag) {
  const bool short_bound = report_ns < kWaitLimitNs;
  auto poll = [&]() {
    if (CLUSTER)
      return short_bound ? mbar_test_wait_cluster(bar, parity) : mbar_try_wait_cluster(bar, parity);
    return short_bound ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (poll()) return true;
  const uint64_t t0 = global_timer_ns();
  const int polls = short_bound ? 1 : 32;
  bool reported = false;
  while (true) {
#pragma unroll 1
    for (int i = 0; i < polls; ++i)
      if (poll()) return true;
    const uint64_t dt = global_timer_ns() - t0;
    if (!reported && (dt > report_ns || dt > kWaitLimitNs)) {
      flag_error(flag, VG_DEVERR_TIMEOUT);
      reported = true;
    }
    if (dt > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ------------------------------------------------------ thread-block clusters
// shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// 16-byte store into (possibly another CTA's) shared memory that completes 16
// bytes of transaction count on the mbarrier of the destination CTA; both
// addresses are shared::cluster addresses in that CTA.
__device__ __forceinline__ void st_async_v4(uint32_t raddr, uint4 v, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(raddr),
      "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
      : "memory");
}
// Arrive once on the mbarrier at shared::cluster address `rbar` (possibly in
// another CTA), releasing this thread's prior memory accesses at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t rbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar)
               : "memory");
}
// Split cluster barrier (every thread of every CTA arrives, then waits).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// bar.sync on a named barrier (id != 0) over `threads` threads (multiple of 32)
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------- TMA
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled tensor load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 1-D bulk copy global -> shared (size and both addresses multiples of 16 B),
// completion counted on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Order this thread's earlier generic-proxy accesses before its later
// async-proxy (TMA / bulk copy) accesses, in every state space.
__device__ __forceinline__ void fence_proxy_async_all() {
  asm volatile("fence.proxy.async;" ::: "memory");
}

// ------------------------------------------------------------ tensor cores
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile stored as
// [chunk / 8][rows][128 B] with the 128-byte swizzle (chunk ^= row & 7) that
// TMA applies with CU_TENSOR_MAP_SWIZZLE_128B.  `rows` = rows per 128-B column.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk, int rows) {
  return static_cast<uint32_t>((chunk >> 3) * rows * 128 + row * 128 +
                               (((chunk & 7) ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------- cp.async
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// 16-byte copy that reads src_bytes (0 or 16) bytes and zero-fills the rest.
__device__ __forceinline__ void cp_async_16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// cp_async_wait with a run-time count (0 .. 7; more waits as for 7).
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    default: cp_async_wait<7>(); break;
  }
}

// ------------------------------------------------- tcgen05 (5th-gen tensor cores)
// Shared-memory matrix descriptor for tcgen05.mma: start address, leading and
// stride byte offsets (all >> 4), descriptor version 1, swizzle mode
// (2 = 128-byte swizzle).  K-major 128B-swizzled operands: rows of 128 bytes,
// 8-row groups SBO = 1024 bytes apart, the K step inside a row advances the
// start address by 32 bytes (16 bf16).  MN-major 128B-swizzled operands: LBO
// = distance between 64-element blocks along M/N, SBO = distance between
// 8-row groups along K.
__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16: bf16 A and B, fp32 D,
// shape M x N, operand majors (0 = K-major, 1 = MN-major).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem desc] * B[smem desc]; issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Tensor memory allocation (one full warp); the base address lands in *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns (one TMEM lane per thread), with
// the completion wait in the same asm statement so that no register is read
// before the load has landed.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 lanes x 16 consecutive 32-bit columns, load and wait in one statement.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
// A with tensor-memory operand: D[tmem] (+)= A[tmem] * B[smem desc].  A is M
// lanes (rows) x K elements, two bf16 per 32-bit column (element 2c in the
// low half of column c); a K step of 16 is 8 columns.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// 32 lanes x 8 / 32 consecutive 32-bit columns from registers.
__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
               : "memory");
}
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- softmax
constexpr float kLog2e = 1.4426950408889634f;

// 2^x with the PTX ex2.approx instruction (2^-inf = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp2 with a -inf-safe reference: when the running max is still -inf, use 0
__device__ __forceinline__ float safe_ref(float m) { return m == -INFINITY ? 0.f : m; }

// ------------------------------------------------------------ split merge
// Log-sum-exp merge of S partial rows, run by one CTA of kMergeThreads:
//   out[d] = sum_s 2^(m_s - M) O_s[d] / sum_s 2^(m_s - M) l_s,  M = max_s m_s,
// with O_s the unnormalised partial (relative to its own m_s, base 2).
// o_base[s * o_stride + d] and ml_base[s * ml_stride + {0, 1}] = (m_s, l_s);
// the merged row goes to dst[0 .. HD) as bf16.
// Thread t owns float4 column t % (HD / 4) for splits t / (HD / 4) + k * G;
// every split's loads are issued before any is used (one round trip for
// S <= G * kMergePer).  Warp 0 forms the batch maximum, weights and
// normaliser from the (m, l) pairs with shuffles and publishes them behind
// one barrier; the G split groups are then reduced in shared memory behind
// one more.
constexpr int kMergeThreads = 128;
constexpr int kMergePer = 8;

constexpr int kMergeSmemFloats = 8 + 128 + 4 * kMergeThreads;

template <int HD>
__device__ __forceinline__ void merge_splits(const float* o_base, size_t o_stride,
                                             const float* ml_base, size_t ml_stride, int S,
                                             __nv_bfloat16* dst, float* smem_f,
                                             float* lse = nullptr) {
  constexpr int COLS = HD / 4;
  constexpr int G = kMergeThreads / COLS;
  constexpr int NB = G * kMergePer;   // splits per batch (<= 128)
  constexpr int LP = NB / 32;         // (m, l) pairs per lane of warp 0
  const int t = threadIdx.x, lane = t & 31, col = t % COLS, grp = t / COLS;
  float* red = smem_f;                                         // [8]: m_new, corr, l of the batch
  float* w_s = smem_f + 8;                                     // [NB] weights of a batch
  float4* part = reinterpret_cast<float4*>(smem_f + 8 + 128);  // [G][COLS]
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float mx_all = -INFINITY, lt_all = 0.f;
  for (int s0 = 0; s0 < S; s0 += NB) {
    float4 v[kMergePer];
#pragma unroll
    for (int k = 0; k < kMergePer; ++k) {
      const int s = s0 + grp + k * G;
      v[k] = s < S ? __ldcg(reinterpret_cast<const float4*>(o_base + (size_t)s * o_stride) + col)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // warp 0 forms the batch maximum, the weights and the normaliser from all
    // the batch's (m, l) pairs (shuffles), then one barrier publishes them
    if (t < 32) {
      float mw[LP], lw[LP];
#pragma unroll
      for (int i = 0; i < LP; ++i) {
        const int s = s0 + lane + 32 * i;
        mw[i] = s < S ? __ldcg(ml_base + (size_t)s * ml_stride) : -INFINITY;
        lw[i] = s < S ? __ldcg(ml_base + (size_t)s * ml_stride + 1) : 0.f;
      }
      float mb = mw[0];
#pragma unroll
      for (int i = 1; i < LP; ++i) mb = fmaxf(mb, mw[i]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
      const float m_new = fmaxf(mx_all, mb);
      const float ref = safe_ref(m_new);
      float lb = 0.f;
#pragma unroll
      for (int i = 0; i < LP; ++i) {
        const float w = ex2(mw[i] - ref);  // 0 past S (m = -inf)
        w_s[lane + 32 * i] = w;
        lb += w * lw[i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lb += __shfl_xor_sync(0xffffffffu, lb, o);
      if (lane == 0) {
        red[0] = m_new;
        red[1] = ex2(mx_all - ref);
        red[2] = lb;
      }
    }
    __syncthreads();
    const float corr = red[1];
    lt_all = lt_all * corr + red[2];
    mx_all = red[0];
    acc.x *= corr;
    acc.y *= corr;
    acc.z *= corr;
    acc.w *= corr;
#pragma unroll
    for (int k = 0; k < kMergePer; ++k) {
      const float w = w_s[grp + k * G];
      acc.x += w * v[k].x;
      acc.y += w * v[k].y;
      acc.z += w * v[k].z;
      acc.w += w * v[k].w;
    }
    if (s0 + NB < S) __syncthreads();  // w_s and red are rewritten by the next batch
  }
  part[grp * COLS + col] = acc;
  __syncthreads();
  if (grp == 0) {
    float4 o = part[col];
#pragma unroll
    for (int k = 1; k < G; ++k) {
      const float4 q = part[k * COLS + col];
      o.x += q.x;
      o.y += q.y;
      o.z += q.z;
      o.w += q.w;
    }
    const float inv = lt_all > 0.f ? 1.f / lt_all : 0.f;
    *reinterpret_cast<__nv_bfloat162*>(dst + col * 4) = __floats2bfloat162_rn(o.x * inv, o.y * inv);
    *reinterpret_cast<__nv_bfloat162*>(dst + col * 4 + 2) =
        __floats2bfloat162_rn(o.z * inv, o.w * inv);
    // natural-log sum of the row's exponentials: (m + log2 l) ln 2
    if (lse && col == 0) *lse = (mx_all + __log2f(lt_all)) * 0.6931471805599453f;
  }
}

}  // namespace vg
