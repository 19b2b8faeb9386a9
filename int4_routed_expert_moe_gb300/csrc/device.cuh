// Device-side helpers shared by the library's kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
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

// Scaled-activation dot products. A 4-bit code c masked into the low bits of
// an FP16 pattern is the FP16 subnormal c * 2^-24 exactly (and the odd nibble,
// masked in place, 16c * 2^-24), so no bias has to be removed. The
// activations of a 32-element chunk are pre-scaled by an exact power of two
// 2^s (odd-nibble pairs by 2^(s-4)) chosen so that max|x| * 2^s < 2^15; every
// product c * x * 2^(s-24) is then an FP16 normal well inside range. The
// caller multiplies the FP32 result by 2^(24-s).
//   xp[0] = (x0, x4) 2^s, xp[1] = (x1, x5) 2^(s-4),
//   xp[2] = (x2, x6) 2^s, xp[3] = (x3, x7) 2^(s-4)   (per 8-element word)
__device__ __forceinline__ half2 dot8_scaled(uint32_t w, const half2* xp, half2 acc) {
  const uint32_t w8 = w >> 8;
  acc = __hfma2(u32_as_h2(w & 0x000F000Fu), xp[0], acc);
  acc = __hfma2(u32_as_h2(w & 0x00F000F0u), xp[1], acc);
  acc = __hfma2(u32_as_h2(w8 & 0x000F000Fu), xp[2], acc);
  acc = __hfma2(u32_as_h2(w8 & 0x00F000F0u), xp[3], acc);
  return acc;
}

// 16 codes (two words); each FP16 lane sums 8 products -- the two words'
// 4-product chains side by side, then added -- and is widened to FP32.
__device__ __forceinline__ float dot16_scaled(uint32_t w0, uint32_t w1, const half2* xp) {
  const half2 zero = __float2half2_rn(0.0f);
  const half2 acc = __hadd2(dot8_scaled(w0, xp, zero), dot8_scaled(w1, xp + 4, zero));
  return __low2float(acc) + __high2float(acc);
}

// Exponent s for a chunk whose largest magnitude is amax: amax * 2^s < 2^15,
// read from amax's exponent bits (amax = m 2^e with m in [0.5, 1); every
// magnitude that comes from FP16 data is 0 or an FP32 normal). Clamped to
// [-100, 100] so that 2^s, 2^(s-4) and 2^(24-s) stay FP32 normals (an
// infinite amax gives -100).
__device__ __forceinline__ int chunk_shift(float amax) {
  if (!(amax > 0.0f)) return 0;
  const int e = ((__float_as_int(amax) >> 23) & 0xff) - 126;
  return max(-100, min(100, 15 - e));
}

// 2^e as an FP32 value built from its exponent bits (|e| <= 126).
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// Eight activations a[0..7] as the four scaled pairs dot8_scaled reads; the
// power-of-two products are exact in FP32, then rounded once to FP16.
__device__ __forceinline__ void scaled_perm8(const float* a, int s, half2* out) {
  const float m0 = pow2f(s), m1 = pow2f(s - 4);
  out[0] = __floats2half2_rn(a[0] * m0, a[4] * m0);
  out[1] = __floats2half2_rn(a[1] * m1, a[5] * m1);
  out[2] = __floats2half2_rn(a[2] * m0, a[6] * m0);
  out[3] = __floats2half2_rn(a[3] * m1, a[7] * m1);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + expf(-v)); }
// Fast-intrinsic SiLU for the tensor-core epilogues (the result is rounded to
// FP16 next; relative error ~1e-6). Limits: v -> -inf gives 0, v -> +inf v.
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// ---- routing: top-k of one token in one warp (shared by moe_route and the
// streamed decode kernel) ------------------------------------------------------
// "Horizon RunMap -- Prévia Técnica", "02 / A solução": the router picks the
// experts of each token: top-k by (logit desc, index asc). a ranks before b
// in (value desc, index asc); -0 == +0 by IEEE compare.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Order-preserving key of a finite or infinite FP32 value (larger value,
// larger key; -0 and +0 share the key of +0, as they compare equal).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of one token in one warp: lane l holds experts l + 32 j (j < NJ,
// NJ >= E/32) in registers, pads (e >= E) are never picked. Each lane keeps
// its best CD not yet picked in a small sorted cache (rank order: logit
// desc, index asc); round r takes the best cache head of the warp -- the
// largest key by one warp reduction, the smallest index among equal keys by
// another -- and the owning lane pops it, refilling its cache from its
// registers when it runs dry. Lane r < k returns pick r (value, expert).
// This is moe_route's selection (top-k by (logit desc, index asc)).
template <int NJ>
__device__ __forceinline__ void warp_topk(const float (&v)[NJ], int E, int k, int lane, float& my_v, int& my_i) {
  const unsigned full = 0xffffffffu;
  int mine_n = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j) mine_n += lane + 32 * j < E;
  constexpr int CD = NJ < 2 ? NJ : 2;
  float cv[CD];
  int ci[CD];
  // The lane's best CD elements that rank after (lv, li).
  auto fill = [&](float lv, int li) {
#pragma unroll
    for (int c = 0; c < CD; ++c) {
      cv[c] = -INFINITY;
      ci[c] = INT_MAX;
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      if (e < E && ranks_before(lv, li, v[j], e)) {
        bool b[CD];
#pragma unroll
        for (int c = 0; c < CD; ++c) b[c] = ranks_before(v[j], e, cv[c], ci[c]);
#pragma unroll
        for (int c = CD - 1; c >= 1; --c) {
          if (b[c - 1]) {
            cv[c] = cv[c - 1];
            ci[c] = ci[c - 1];
          } else if (b[c]) {
            cv[c] = v[j];
            ci[c] = e;
          }
        }
        if (b[0]) {
          cv[0] = v[j];
          ci[0] = e;
        }
      }
    }
  };
  fill(INFINITY, -1);
  int taken = 0;
  my_v = 0.0f;
  my_i = -1;
#pragma unroll 1
  for (int r = 0; r < k; ++r) {
    const bool has = ci[0] != INT_MAX;
    const uint32_t key = has ? order_key(cv[0]) : 0u;  // every real key is above 0
    const uint32_t kmax = __reduce_max_sync(full, key);
    const uint32_t win = __reduce_min_sync(full, (has && key == kmax) ? (uint32_t)ci[0] : 0xffffffffu);
    const float wv = __shfl_sync(full, cv[0], (int)(win & 31));
    if (lane == r) {
      my_v = wv;
      my_i = (int)win;
    }
    if (has && (uint32_t)ci[0] == win) {
      const float pv = cv[0];
      ++taken;
#pragma unroll
      for (int c = 0; c + 1 < CD; ++c) {
        cv[c] = cv[c + 1];
        ci[c] = ci[c + 1];
      }
      cv[CD - 1] = -INFINITY;
      ci[CD - 1] = INT_MAX;
      if (ci[0] == INT_MAX && taken < mine_n) fill(pv, (int)win);
    }
  }
}

}  // namespace moe
