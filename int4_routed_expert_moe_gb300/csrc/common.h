// Shared host-side helpers of the library (no device code here).
#pragma once

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstddef>
#include <cstdint>
#include <cstdio>

#include "../../include/moe.h"

namespace moe {

// Records a thread-local failure detail and returns `status`.
int fail(int status, const char* fmt, ...);
// Clears the thread-local detail (called on entry of each ABI function).
void clear_error();

inline bool valid_shape(const moe_expert_shape* s) {
  if (!s) return false;
  const int H = s->hidden, I = s->inter, g = s->group;
  if (H <= 0 || I <= 0 || g <= 0) return false;
  if (H % 64 || I % 64 || g % 32) return false;
  if (H % g || I % g) return false;
  if (H > 8192 || I > 8192) return false;
  return true;
}

struct BlockLayout {
  size_t q_gate, q_up, q_down, s_gate, z_gate, s_up, z_up, s_down, z_down, total;
};

inline BlockLayout block_layout(int H, int I, int g) {
  BlockLayout b;
  const size_t qgu = (size_t)I * H / 2, qd = (size_t)H * I / 2;
  const size_t sgu = (size_t)I * (H / g) * 2, sd = (size_t)H * (I / g) * 2;
  b.q_gate = 0;
  b.q_up = b.q_gate + qgu;
  b.q_down = b.q_up + qgu;
  b.s_gate = b.q_down + qd;
  b.z_gate = b.s_gate + sgu;
  b.s_up = b.z_gate + sgu;
  b.z_up = b.s_up + sgu;
  b.s_down = b.z_up + sgu;
  b.z_down = b.s_down + sd;
  b.total = b.z_down + sd;
  return b;
}

#define MOE_CUDA_TRY(expr)                                                    \
  do {                                                                        \
    cudaError_t e_ = (expr);                                                  \
    if (e_ != cudaSuccess)                                                    \
      return ::moe::fail(MOE_ERR_CUDA, "%s: %s (%s:%d)", #expr,              \
                         cudaGetErrorString(e_), __FILE__, __LINE__);         \
  } while (0)

// Returns MOE_ERR_CUDA if an earlier asynchronous error is pending.
inline int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(MOE_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
  return MOE_OK;
}

}  // namespace moe
