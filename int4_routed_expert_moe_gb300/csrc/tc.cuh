// Blackwell tensor-core building blocks in inline PTX: mbarriers, TMA tensor
// loads, tensor-memory allocation and loads, tcgen05.mma with shared-memory
// operand descriptors. Used by the grouped (prefill) and shared FFN kernels.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void bar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// try_wait without a suspend-time hint (a short, hardware-defined window).
__device__ __forceinline__ bool bar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Non-blocking test of a phase.
__device__ __forceinline__ bool bar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t v;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(v));
  return v;
}
// Bounded wait (about one second of global time at most); false when it gave
// up. A phase that has already completed is taken at the first test.
constexpr uint64_t kWaitNs = 1000000000ull;
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity) {
  if (bar_test(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (bar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}

// ---- TMA tensor loads (tile mode), completion counted on an mbarrier ------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
        "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Generic-proxy shared-memory writes made visible to the async proxy (the
// tensor cores read operands through it).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tensor memory ---------------------------------------------------------
// Whole warp: allocates ncols columns (power of two >= 32); the TMEM address
// is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 lanes x 16 consecutive 32-bit columns: thread t of the warp receives
// lane (taddr.lane + t), columns taddr.col .. +15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 16 consecutive 32-bit columns from registers: thread t writes
// lane (taddr.lane + t).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- tcgen05.mma, kind::f16 -------------------------------------------------
// Shared-memory operand descriptor of a K-major tile in the 128-byte swizzle
// layout: rows of 64 FP16 (128 bytes) at a 128-byte pitch, 16-byte chunk c of
// row r stored at chunk position c ^ (r % 8), groups of 8 rows 1024 bytes
// apart (stride byte offset). The tile base is 1024-byte aligned; the k-th
// 16-element slice starts 32*k bytes further (the swizzle is applied to the
// address, so the start simply advances).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);       // start address
  d |= (uint64_t)(16u >> 4) << 16;                // leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;              // stride byte offset: 8 rows
  d |= (uint64_t)1 << 46;                         // descriptor version
  d |= (uint64_t)2 << 61;                         // 128-byte swizzle
  return d;
}
// Instruction descriptor: D FP32, A and B FP16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// Same with the A operand in tensor memory: row m of A in lane m, two FP16
// elements per 32-bit column in K order (a 16-element K slice = 8 columns).
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// One lane of a converged warp: true in exactly one active lane. An issuing
// loop run by the whole warp, with the tcgen05 operations under this
// predicate, keeps its warp-uniform operands uniform; the same loop run by a
// lone lane issues at about half the rate once other warps load its
// scheduler (measured on GB300: 4 MMAs + commit of N = 64 in 294 cycles
// against 576).
__device__ __forceinline__ bool elect_one() {
  uint32_t pr;
  asm volatile(
      "{\n .reg .pred P;\n elect.sync _|P, 0xffffffff;\n selp.u32 %0, 1, 0, P;\n}\n"
      : "=r"(pr));
  return pr != 0;
}
// Bounded wait by every lane of a converged warp, with one verdict for all.
__device__ __forceinline__ bool bar_wait_warp(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, bar_wait(bar, parity));
}
// The mbarrier receives one arrival when every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile.
__host__ __device__ constexpr uint32_t sw128_offset(int r, int c) {
  return (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4);
}

// ---- pipeline scaffolding of the tile kernels -------------------------------
// Roles: warp 0 issues TMA loads, warp 1 owns tensor memory and issues the
// MMAs, the remaining warps expand operands (when any) and run the epilogue.
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_addr(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// Control block after the stage area: per stage, "loads landed" (tma_full),
// "operand expanded" (a_full) and "MMAs done with the stage" (empty); the
// final accumulator barrier, the TMEM address and a block-local abort flag.
struct Ctrl {
  uint64_t* tma_full;
  uint64_t* a_full;
  uint64_t* empty;
  uint64_t* acc_full;
  uint32_t* tmem_slot;
  int* abort;
};
__device__ __forceinline__ Ctrl ctrl_at(uint8_t* p, int stages) {
  Ctrl c;
  c.tma_full = reinterpret_cast<uint64_t*>(p);
  c.a_full = c.tma_full + stages;
  c.empty = c.a_full + stages;
  c.acc_full = c.empty + stages;
  c.tmem_slot = reinterpret_cast<uint32_t*>(c.acc_full + 1);
  c.abort = reinterpret_cast<int*>(c.tmem_slot + 1);
  return c;
}

// A bounded wait expired: report it (bit 2 of the error word) and make the
// other roles of the block stop at their next check.
__device__ __forceinline__ void set_abort(const Ctrl& c, int32_t* flags) {
  atomicOr(flags, 4);
  *reinterpret_cast<volatile int*>(c.abort) = 1;
}
__device__ __forceinline__ bool aborted(const Ctrl& c) { return *reinterpret_cast<volatile int*>(c.abort) != 0; }

// Barrier initialisation and TMEM allocation; returns the TMEM base address.
__device__ __forceinline__ uint32_t gemm_setup(const Ctrl& c, int stages, uint32_t tmem_cols, int a_full_count) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      bar_init(&c.tma_full[s], 1);
      bar_init(&c.a_full[s], a_full_count);
      bar_init(&c.empty[s], 1);
    }
    bar_init(c.acc_full, 1);
    *c.abort = 0;
    bar_init_fence();
  }
  if ((threadIdx.x >> 5) == 1) tmem_alloc(c.tmem_slot, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return *c.tmem_slot;
}

__device__ __forceinline__ void gemm_teardown(uint32_t tmem, uint32_t tmem_cols) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// Producer tail after an abort: wait (bounded) for the loads still in flight.
__device__ __forceinline__ void drain_loads(const Ctrl& c, int stages, int issued) {
  for (int kt = issued > stages ? issued - stages : 0; kt < issued; ++kt)
    bar_wait(&c.tma_full[kt % stages], (kt / stages) & 1);
}

}  // namespace tc

// Host: tensor-map encoding through the driver entry point (no link-time
// dependency on the driver library). Returns MOE_OK or an error status.
int encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle);

}  // namespace moe
