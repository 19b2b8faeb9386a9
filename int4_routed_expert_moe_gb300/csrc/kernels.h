// Internal interface between the ABI dispatch and the kernel launchers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "common.h"

namespace moe {

// Byte offsets of the segments inside one expert block (see include/moe.h).
struct BlockOffsets {
  unsigned long long q_gate, q_up, q_down, s_gate, z_gate, s_up, z_up, s_down, z_down;
};

inline BlockOffsets offsets_of(const BlockLayout& b) {
  BlockOffsets o;
  o.q_gate = b.q_gate; o.q_up = b.q_up; o.q_down = b.q_down;
  o.s_gate = b.s_gate; o.z_gate = b.z_gate; o.s_up = b.s_up; o.z_up = b.z_up;
  o.s_down = b.s_down; o.z_down = b.z_down;
  return o;
}

// The workspace starts with a 256-byte header; its first int32 is the sticky
// error word.
constexpr size_t kWorkspaceHeader = 256;

struct ForwardArgs {
  int H, I, g, T, k, E, n_slots;
  const __half* x;
  const int32_t* ids;
  const float* weights;
  const uint8_t* pool;
  size_t block_bytes;
  BlockOffsets off;
  const int32_t* slot_of;
  const __half* y_shared;
  __half* y;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
};

size_t gemv_workspace_bytes(int H, int I, int T, int k);
int gemv_forward(const ForwardArgs& a);

// Token sort of the (token, choice) pairs by expert (see moe_token_sort).
int launch_token_sort(const int32_t* ids, int P, int k, int E, int32_t* offsets,
                      int32_t* pair_tok, int32_t* pair_j, cudaStream_t st);

// Fused one-kernel decode path (persistent, one block per SM).
size_t fused_workspace_bytes(int H, int I, int T, int k);
int fused_forward(const ForwardArgs& a);

size_t grouped_workspace_bytes(int H, int I, int T, int k, int E);
int grouped_forward(const ForwardArgs& a);

// Slot-table updates of one residency step, passed to the publish kernel by
// value (so no host buffer has to outlive the launch).
constexpr int kMaxSlotUpdates = 128;
struct SlotUpdates {
  int n;
  int32_t expert[kMaxSlotUpdates];
  int32_t slot[kMaxSlotUpdates];
};
// Enqueues one kernel writing slot_of[expert[i]] = slot[i] for i < n.
int publish_slot_updates(int32_t* dev_slot_of_layer, const SlotUpdates& u, cudaStream_t st);

}  // namespace moe
