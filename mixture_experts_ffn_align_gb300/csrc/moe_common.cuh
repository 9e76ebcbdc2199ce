// Device-side helpers shared by the kernels: the device error word, bounded
// mbarrier waits, TMA (cp.async.bulk.tensor) loads and tcgen05 (TMEM / UMMA)
// wrappers written as inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Bits of the device error word (read and cleared by moe_sync_status).
enum : int {
  kDevErrTimeout = 1,   // a bounded wait gave up
  kDevErrBadIndex = 2,  // an expert id >= E was seen
};

// The error word lives in the library's device memory; kernels receive its
// address as a parameter.
__device__ __forceinline__ void set_dev_error(int* err, int bits) {
  if (err != nullptr) atomicOr(err, bits);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Same test with acquire at cluster scope: pairs with a release by the other
// CTA of a cluster (a remote mbarrier arrive after a remote shared store).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase with `parity` of the barrier has completed.  Gives up
// when *abort becomes non-zero (another role failed) or after limit_ns of
// wall time; on a timeout it records kDevErrTimeout in *err and raises
// *abort.  Returns true if the phase completed.  CLUSTER
// selects the cluster-scope acquire.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort, uint64_t limit_ns,
                                                  int* err) {
  auto test = [&]() {
    return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (test()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (test()) return true;
    if ((it & 63) == 0) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        set_dev_error(err, kDevErrTimeout);
        if (abort != nullptr) *abort = 1;
        return false;
      }
    }
  }
}

// --------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-byte asynchronous copy global -> shared (no registers held while in
// flight); completes by commit group.
__device__ __forceinline__ void cp_async_4(uint32_t dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's most recent commit groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Raises the transaction count of the barrier's current phase by `bytes`
// without arriving (the arrival comes later from the same or another thread).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Bulk (non-tensor) copy global -> shared of `bytes` (a multiple of 16, both
// addresses 16-byte aligned), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Asks for `bytes` (a multiple of 16, 16-byte aligned) of global memory to be
// brought into L2; no completion to wait for.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Asks for a 2-D box of a tensor to be brought into L2 (no shared memory,
// no completion to wait for); used ahead of the loads of a streamed operand.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t c0,
                                                   int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

// 2-D tiled bulk tensor load global -> shared, completion counted in bytes on
// `bar`.  c0 is the innermost (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 0: evict_normal, 1: evict_last, 2: evict_first.
__device__ __forceinline__ uint64_t l2_policy(int mode) {
  return mode == 1 ? l2_policy_evict_last() : (mode == 2 ? l2_policy_evict_first()
                                                         : l2_policy_evict_normal());
}
// L2 hints of the GEMM operand loads: activations (A) and weights (B).  A
// block is re-read for every n-tile of its expert, a weight tile only by the
// expert's m-blocks running at the same time; evict_last on A and no hint on
// B measured best on the Mixtral-shaped and DeepSeek-class layers.
#ifndef MOE_GEMM_L2_A
#define MOE_GEMM_L2_A 1
#endif
#ifndef MOE_GEMM_L2_B
#define MOE_GEMM_L2_B 0
#endif

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t holder_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   holder_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
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
// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both K-major, one CTA.  kind::f16 covers
// bf16 inputs with fp32 accumulation.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same for 8-bit float inputs (e4m3 x e4m3 here), fp32 accumulation.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Block-scaled MMA (kind::mxf8f6f4, one E8M0 scale per 32 elements along K
// for each row of A and each column of B, read from tensor memory).
__device__ __forceinline__ void umma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem,
                                              uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with block scales, both operands
// K-major: bits 4-5 B scale-factor byte, 7-9 A format, 10-12 B format, 17-22
// N >> 3, 23 scale format (1 = E8M0), 24-28 M >> 4, 29-30 A scale-factor byte.
__host__ __device__ constexpr uint32_t make_idesc_block_scaled(uint32_t a_fmt, uint32_t b_fmt,
                                                                int M, int N, uint32_t sf_id) {
  return (sf_id << 4) | (a_fmt << 7) | (b_fmt << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(M >> 4) << 24) | (sf_id << 29);
}
constexpr uint32_t kFmtE2M1 = 5;  // kind::mxf8f6f4 operand format code for e2m1

// Write four consecutive 32-bit columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, uint32_t a, uint32_t b,
                                                  uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Instruction descriptor (kind::f16 / kind::f8f6f4, dense, both operands
// K-major, fp32 accumulator): bits 4-5 D format (1 = f32), 7-9 A format,
// 10-12 B format, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t a_fmt, uint32_t b_fmt, int M, int N) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kFmtBF16 = 1;  // kind::f16 operand format code for bf16
constexpr uint32_t kFmtE4M3 = 0;  // kind::f8f6f4 operand format code for e4m3

// Shared-memory matrix descriptor for a K-major tile written by TMA with
// 128-byte swizzling: rows of 128 bytes, 8-row swizzle atoms of 1024 bytes
// (stride byte offset), tile base 1024-byte aligned.  Bits 0-13 start >> 4,
// 16-29 leading byte offset >> 4 (unused for this layout), 32-45 stride byte
// offset >> 4, 46-48 fixed 0b001, 61-63 swizzle mode (2 = 128B).
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Descriptor of a 32-row x 16-byte shared-memory block stored row after row
// (no swizzle: four 8-row core matrices of 128 contiguous bytes, 128 bytes
// apart), the source shape of tmem_cp_32x128b_x4.
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;     // leading offset: the block is one core matrix wide
  d |= (uint64_t)(128u >> 4) << 32;    // between 8-row core matrices
  d |= (uint64_t)1 << 46;
  return d;
}
// Asynchronous copy of 32 rows x 128 bits of shared memory into tensor
// memory lanes 0-31 x 4 columns, repeated in all four 32-lane quadrants.
// Issued by the MMA thread, it is ordered before that thread's later MMAs.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tcgen05.cp, tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 lanes x 32 consecutive fp32 columns from tensor memory, one row per
// thread (thread i <-> lane base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 16 consecutive fp32 columns, one row per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------ CTA pairs (cluster of 2)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of both CTAs: arrive (release) and wait (acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Store to a shared variable that may live in the peer CTA.
__device__ __forceinline__ void st_shared_cluster(uint32_t cluster_addr, int v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// 16-byte store to shared memory that may live in the peer CTA.
__device__ __forceinline__ void st_shared_cluster_v4(uint32_t cluster_addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
// Orders this thread's earlier generic-proxy writes (to any state space,
// including a peer CTA's shared memory) before later async-proxy accesses.
__device__ __forceinline__ void fence_proxy_async_all() {
  asm volatile("fence.proxy.async;" ::: "memory");
}
// Arrive on an mbarrier that may live in the peer CTA.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
// Arrive on an mbarrier that may live in the peer CTA, with no memory
// ordering: for signals that carry no data through memory (a tensor-memory
// buffer read to registers, its tcgen05.ld completed).  The release form
// above costs a cluster-scope memory barrier per arrive.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
// 2-D tensor load into this CTA's shared memory whose completion is counted
// on an mbarrier of the CTA pair (here: the leader's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t cluster_bar, int32_t c0, int32_t c1,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(cluster_bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t holder_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   holder_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Arrive once on the barrier at this shared offset in every CTA of `mask`
// when the pair's tcgen05 operations issued so far by this thread complete.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
// D (M=256 over the pair: rows 0-127 in the leader's TMEM, 128-255 in the
// peer's) (+)= A (128 rows from each CTA's smem) * B^T (N/2 columns from each).
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same for 8-bit float operands (kind::f8f6f4, e4m3 x e4m3 here) on the pair.
__device__ __forceinline__ void umma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Copy of 32 rows x 128 bits of shared memory into tensor memory (as
// tmem_cp_32x128b_x4), issued by the pair's leader: each CTA's shared memory
// at this offset goes to its own tensor memory.
__device__ __forceinline__ void tmem_cp_pair_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// Block-scaled MMA on the pair (M=256 over the two CTAs): each CTA's half
// reads its rows' A scales and the full B scale operand from its own tensor
// memory at sfa_tmem / sfb_tmem.
__device__ __forceinline__ void umma_mxf8f6f4_pair(uint32_t d_tmem, uint64_t a_desc,
                                                   uint64_t b_desc, uint32_t idesc,
                                                   uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                   uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Warpgroup register reallocation: every thread of a 128-thread warpgroup
// executes the same one; increases wait until decreases elsewhere in the CTA
// have released enough of the registers the CTA was launched with.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// -------------------------------------------------------------- numerics
__device__ __forceinline__ float bf16_round(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}
// SiLU(g) = g / (1 + exp(-g)) with the fast exponential and division
// intrinsics: a few fp32 ulps of error, far below the bf16 rounding of z
// (and 4 % of the fused GEMM1's time cheaper than expf + IEEE division under
// the power cap).  g -> -inf gives -0, g -> +inf gives g.
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Optional epilogue work of the grouped GEMMs, in the order of the pages'
// GEMM post-processing (page "fused_moe.py 分析", fused_moe_kernel "后处理":
// dequant -> bias -> router weight -> cast to the output type), plus the
// gated activation recipe of the fused GEMM1 (page "Blackwell 上的 DeepGEMM
// FusedMoE（vLLM）", §2.6.4: gemm1_alpha / gemm1_beta / gemm1_clamp_limit).
struct Epilogue {
  const __nv_bfloat16* bias;   // [E, n_bias] bf16 added in fp32, or null
  int n_bias;                  // bias columns per expert (2I for GEMM1, H for GEMM2)
  const int32_t* sorted_ids;   // row -> routed item, with item_weights for the
  const float* item_weights;   //   router weight of the row (null: none)
  int R;                       // routed items; rows holding ids >= R are padding
  int recipe;                  // 0: SiLU(g) * u; 1: the alpha / beta / limit recipe
  float alpha, beta, limit;    // z = (clamp(u, -limit, limit) + beta) * g' * sigmoid(alpha g'),
                               // g' = min(g, limit); limit <= 0: no clamping
};

// Router weight of output row `row` (1 without one; 0 for a padding row).
__device__ __forceinline__ float epi_row_weight(const Epilogue& ep, size_t row) {
  if (ep.item_weights == nullptr) return 1.0f;
  const int sid = ep.sorted_ids[row];
  return sid < ep.R ? ep.item_weights[sid] : 0.0f;
}
// Bias of expert e at column col (0 without a bias).
__device__ __forceinline__ float epi_bias(const Epilogue& ep, int e, int col) {
  return ep.bias == nullptr ? 0.0f
                            : __bfloat162float(ep.bias[(size_t)e * ep.n_bias + col]);
}
// The gated activation of one (gate, up) pair.
__device__ __forceinline__ float act_glu(const Epilogue& ep, float g, float u) {
  if (ep.recipe == 0) return silu_fast(g) * u;
  if (ep.limit > 0.0f) {
    g = fminf(g, ep.limit);
    u = fminf(fmaxf(u, -ep.limit), ep.limit);
  }
  return __fdividef(g, 1.0f + __expf(-ep.alpha * g)) * (u + ep.beta);
}

// Two bf16 values as one 32-bit word, the first in the low half (memory order).
__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// 64 bytes of one output row.  Where dst is 32-byte aligned (every row of a
// tile is, when the row pitch is a multiple of 32 bytes) it goes out as two
// 256-bit stores, each filling a whole L2 sector; 16-byte stores fill half a
// sector each and take twice the load/store-queue entries, which throttled
// the epilogue warps at the end of every tile.  Otherwise four 16-byte stores.
__device__ __forceinline__ void st_row64(void* dst, const uint32_t (&w)[16]) {
  if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
    uint32_t* d = static_cast<uint32_t*>(dst);
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(d),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                 "r"(w[7])
                 : "memory");
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(d + 8),
                 "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]),
                 "r"(w[14]), "r"(w[15])
                 : "memory");
  } else {
    uint4* d = static_cast<uint4*>(dst);
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
}

// Fused GEMM1 epilogue for 32 columns of one row: the gate and up sums
// (plus bias), each rounded to bf16 as a stored H1 would be, through the gated
// activation, as 32 bf16 values at dst (16-byte aligned).
__device__ __forceinline__ void epi_glu_store32(const Epilogue& ep, int e, int gcol0, int ucol0,
                                                const uint32_t (&g)[32], const uint32_t (&u)[32],
                                                __nv_bfloat16* dst) {
  uint32_t w[16];
  const bool bias = ep.bias != nullptr;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    __nv_bfloat16 z[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float gs = __uint_as_float(g[2 * j + h]), us = __uint_as_float(u[2 * j + h]);
      if (bias) {
        gs += epi_bias(ep, e, gcol0 + 2 * j + h);
        us += epi_bias(ep, e, ucol0 + 2 * j + h);
      }
      z[h] = __float2bfloat16_rn(act_glu(ep, bf16_round(gs), bf16_round(us)));
    }
    w[j] = bf16x2_bits(z[0], z[1]);
  }
  st_row64(dst, w);
}
// Plain epilogue values of 32 columns of one row: bf16((acc + bias) * w),
// packed two per word in memory order.
__device__ __forceinline__ void epi_pack32(const Epilogue& ep, int e, int col0, float w,
                                           const uint32_t (&r)[32], uint32_t (&pk)[16]) {
  const bool bias = ep.bias != nullptr;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float v0 = __uint_as_float(r[2 * j]), v1 = __uint_as_float(r[2 * j + 1]);
    if (bias) {
      v0 += epi_bias(ep, e, col0 + 2 * j);
      v1 += epi_bias(ep, e, col0 + 2 * j + 1);
    }
    pk[j] = bf16x2_bits(__float2bfloat16_rn(v0 * w), __float2bfloat16_rn(v1 * w));
  }
}
// Plain epilogue for 32 columns of one row: bf16((acc + bias) * w) at dst.
__device__ __forceinline__ void epi_store32(const Epilogue& ep, int e, int col0, float w,
                                            const uint32_t (&r)[32], __nv_bfloat16* dst) {
  uint32_t pk[16];
  epi_pack32(ep, e, col0, w, r, pk);
  st_row64(dst, pk);
}

// fp32 -> e4m3fn, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint8_t f32_to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// Dynamic 1x128 scale: max(amax, 1e-10) / 448 in fp32 (IEEE division); with
// ue8m0, rounded up to a power of two.
__device__ __forceinline__ float act_scale(float amax, bool ue8m0) {
  float s = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
  if (ue8m0) {
    uint32_t b = __float_as_uint(s);
    if (b & 0x7FFFFFu) b = (b & 0xFF800000u) + 0x800000u;
    s = __uint_as_float(b);
  }
  return s;
}

}  // namespace moe
