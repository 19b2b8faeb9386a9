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

// Dot product of the eight 4-bit codes of one 32-bit word (code i in bits
// 4i..4i+3) with eight FP16 activations stored as the pairs
// xp[0] = (x0, x4), xp[1] = (x1, x5), xp[2] = (x2, x6), xp[3] = (x3, x7).
// A code q becomes the FP16 value 1024 + q (or 1024 + 16 q for the odd
// nibbles) by OR-ing it into the exponent pattern of 1024; subtracting 1024
// (or scaling by 1/16 and subtracting 64) gives q exactly. The four products
// of each pair lane are summed in FP16 and the pair is widened to FP32.
__device__ __forceinline__ float dot8_codes(uint32_t w, const half2* xp) {
  const uint32_t kMagic = 0x64006400u;  // (1024.0, 1024.0) in FP16
  const uint32_t t0 = (w & 0x000F000Fu) | kMagic;
  const uint32_t t1 = (w & 0x00F000F0u) | kMagic;
  const uint32_t w8 = w >> 8;
  const uint32_t t2 = (w8 & 0x000F000Fu) | kMagic;
  const uint32_t t3 = (w8 & 0x00F000F0u) | kMagic;
  const half2 k1024 = __float2half2_rn(1024.0f);
  const half2 k16th = __float2half2_rn(0.0625f);
  const half2 km64 = __float2half2_rn(-64.0f);
  const half2 q0 = __hsub2(u32_as_h2(t0), k1024);
  const half2 q1 = __hfma2(u32_as_h2(t1), k16th, km64);
  const half2 q2 = __hsub2(u32_as_h2(t2), k1024);
  const half2 q3 = __hfma2(u32_as_h2(t3), k16th, km64);
  half2 acc = __hmul2(q0, xp[0]);
  acc = __hfma2(q1, xp[1], acc);
  acc = __hfma2(q2, xp[2], acc);
  acc = __hfma2(q3, xp[3], acc);
  const float2 f = __half22float2(acc);
  return f.x + f.y;
}

// Dot of 32 codes (16 bytes) with 32 activations pre-permuted in groups of 8.
__device__ __forceinline__ float dot32_codes(const uint4& w, const half2* xp) {
  return (dot8_codes(w.x, xp) + dot8_codes(w.y, xp + 4)) +
         (dot8_codes(w.z, xp + 8) + dot8_codes(w.w, xp + 12));
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
