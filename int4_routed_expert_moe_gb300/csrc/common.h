// Shared host-side helpers of the library (no device code here).
#pragma once

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstddef>
#include <cstdint>
#include <cstdio>

#include <nvtx3/nvToolsExt.h>

#include "moe.h"

namespace moe {

// NVTX range over one ABI call (host side; a no-op unless a profiler is
// attached), so timelines and `ncu --nvtx` filters see the library's calls.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

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

// Expert block layout: gate/up rows [q_gate | q_up | per-group quads
// (s_gate, z_gate, s_up, z_up)] then down rows [q_down | per-group pairs
// (s_down, z_down)], row strides rounded up to 16 bytes.
struct BlockLayout {
  size_t total, d_offset;
  uint32_t gu_row, d_row;
  uint32_t gu_q_gate, gu_q_up, gu_sz;
  uint32_t d_q, d_sz;
};

inline BlockLayout block_layout(int H, int I, int g) {
  BlockLayout b;
  b.gu_q_gate = 0;
  b.gu_q_up = (uint32_t)H / 2;
  b.gu_sz = (uint32_t)H;
  b.gu_row = (b.gu_sz + (uint32_t)(H / g) * 8u + 15u) & ~15u;
  b.d_q = 0;
  b.d_sz = (uint32_t)I / 2;
  b.d_row = (b.d_sz + (uint32_t)(I / g) * 4u + 15u) & ~15u;
  b.d_offset = (size_t)I * b.gu_row;
  b.total = b.d_offset + (size_t)H * b.d_row;
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
