// Internal interface between the ABI dispatch and the kernel launchers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "common.h"

namespace moe {

// Expert block geometry passed to kernels (see include/moe.h).
struct BlockOffsets {
  unsigned long long d_offset;  // start of the down section
  unsigned gu_row, d_row;       // row strides
  unsigned gu_q_gate, gu_q_up, gu_sz;  // in a gate/up row (sz: quads s_g, z_g, s_u, z_u)
  unsigned d_q, d_sz;                  // in a down row (sz: pairs s_d, z_d)
};

inline BlockOffsets offsets_of(const BlockLayout& b) {
  BlockOffsets o;
  o.d_offset = b.d_offset;
  o.gu_row = b.gu_row; o.d_row = b.d_row;
  o.gu_q_gate = b.gu_q_gate; o.gu_q_up = b.gu_q_up; o.gu_sz = b.gu_sz;
  o.d_q = b.d_q; o.d_sz = b.d_sz;
  return o;
}

// The workspace starts with a 256-byte header; its first int32 is the sticky
// error word, the second the streamed decode kernel's exit counter (blocks
// counted out). Then come that kernel's counters, [P] int32 (256-byte
// rounded): one per unit (distinct expert) for one routed token, the grid
// barrier's counter in the first word for several tokens. The last block out
// zeroes them, and every path keeps its scratch after them, so they stay zero
// between calls of any path.
constexpr size_t kWorkspaceHeader = 256;
inline size_t ws_scratch_offset(int P) { return kWorkspaceHeader + (((size_t)P * 4 + 255) / 256) * 256; }

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
  // Two-kernel GEMV only: device alias of the layer's page-locked host source
  // [E][block]; experts without a slot are read from it in place. NULL: none.
  const uint8_t* host = nullptr;
};

size_t gemv_workspace_bytes(int H, int I, int T, int k);
int gemv_forward(const ForwardArgs& a);

// Optional outputs of the token sort for the grouped path: the tile list of
// resident experts with pairs (tiles of up to tile_n sorted pairs) and the
// unusable-id bits of the error word (0: no slot, 1: id outside [-1, E)).
struct SortTiles {
  const int32_t* slot_of;
  int n_slots;
  int tile_n;
  int4* tiles;  // NULL: no tile list
  int32_t* n_tiles;
  int32_t* flags;
};
// Token sort of the (token, choice) pairs by expert (see moe_token_sort).
int launch_token_sort(const int32_t* ids, int P, int k, int E, int32_t* offsets,
                      int32_t* pair_tok, int32_t* pair_j, cudaStream_t st, const SortTiles* tiles);

// The current device's index and SM count (the count cached per device).
// MOE_OK, or an error status for a failed query or an index >= kMaxDevices.
constexpr int kMaxDevices = 64;
int current_device_sms(int* dev, int* sms);

// Fused one-kernel decode path (persistent, one block per SM).
size_t fused_workspace_bytes(int H, int I, int T, int k);
int fused_forward(const ForwardArgs& a);
// Same, with routing done inside the kernels from logits [T][E]; routed ids
// and weights are written to ids_out / wts_out when non-NULL.
int fused_forward_routed(const ForwardArgs& a, const float* logits, int renorm, int32_t* ids_out,
                         float* wts_out);

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
