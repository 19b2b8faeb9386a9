// Device-side helpers shared by the library's kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

// Programmatic dependent launch: wait for the preceding kernel's memory, and
// let the next kernel in the stream start its independent prologue.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 16-byte read-once load of weight codes: not kept in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ half2 u32_as_h2(uint32_t v) {
  return *reinterpret_cast<half2*>(&v);
}

// Eight 4-bit codes of one 32-bit word (code i in bits 4i..4i+3) as four
// FP16 pairs: q[0] = (c0, c4), q[1] = (c1, c5), q[2] = (c2, c6), q[3] = (c3, c7).
// A code c becomes the FP16 value 1024 + c (or 1024 + 16 c for the odd
// nibbles) by OR-ing it into the bit pattern of 1024; subtracting 1024 (or
// scaling by 1/16 and subtracting 64) gives c exactly.
__device__ __forceinline__ void codes_to_h2(uint32_t w, half2 (&q)[4]) {
  const uint32_t kMagic = 0x64006400u;  // (1024.0, 1024.0) in FP16
  const uint32_t t0 = (w & 0x000F000Fu) | kMagic;
  const uint32_t t1 = (w & 0x00F000F0u) | kMagic;
  const uint32_t w8 = w >> 8;
  const uint32_t t2 = (w8 & 0x000F000Fu) | kMagic;
  const uint32_t t3 = (w8 & 0x00F000F0u) | kMagic;
  const half2 k1024 = __float2half2_rn(1024.0f);
  const half2 k16th = __float2half2_rn(0.0625f);
  const half2 km64 = __float2half2_rn(-64.0f);
  q[0] = __hsub2(u32_as_h2(t0), k1024);
  q[1] = __hfma2(u32_as_h2(t1), k16th, km64);
  q[2] = __hsub2(u32_as_h2(t2), k1024);
  q[3] = __hfma2(u32_as_h2(t3), k16th, km64);
}

// Dot product of the 16 codes of two words with 16 FP16 activations stored
// as pairs xp[0..7] (pair order of codes_to_h2, word by word). Each FP16
// lane sums 8 products; the pair is then widened to FP32.
__device__ __forceinline__ float dot16_codes(uint32_t w0, uint32_t w1, const half2* xp) {
  half2 q[4];
  codes_to_h2(w0, q);
  half2 acc = __hmul2(q[0], xp[0]);
  acc = __hfma2(q[1], xp[1], acc);
  acc = __hfma2(q[2], xp[2], acc);
  acc = __hfma2(q[3], xp[3], acc);
  codes_to_h2(w1, q);
  acc = __hfma2(q[0], xp[4], acc);
  acc = __hfma2(q[1], xp[5], acc);
  acc = __hfma2(q[2], xp[6], acc);
  acc = __hfma2(q[3], xp[7], acc);
  return __low2float(acc) + __high2float(acc);
}

// Dot of 32 codes (16 bytes) with 32 activations in pair order.
__device__ __forceinline__ float dot32_codes(const uint4& w, const half2* xp) {
  return dot16_codes(w.x, w.y, xp) + dot16_codes(w.z, w.w, xp + 8);
}

// Stores eight activations a[0..7] in the pair order dot8_codes reads.
__device__ __forceinline__ void store_perm8(__half* dst, const __half* a) {
  half2* d = reinterpret_cast<half2*>(dst);
  d[0] = __halves2half2(a[0], a[4]);
  d[1] = __halves2half2(a[1], a[5]);
  d[2] = __halves2half2(a[2], a[6]);
  d[3] = __halves2half2(a[3], a[7]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + expf(-v)); }

}  // namespace moe
