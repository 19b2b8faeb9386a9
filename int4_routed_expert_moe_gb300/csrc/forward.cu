// ABI entry points of the routed expert FFN: argument checks and dispatch
// between the decode dequant-GEMV kernels and the grouped tensor-core path.
#include <algorithm>

#include "common.h"
#include "device.cuh"
#include "kernels.h"

namespace moe {
namespace {

// Batches the streamed decode kernel takes under MOE_PATH_AUTO: up to 16
// tokens and 256 (token, choice) pairs; larger batches take the grouped path.
constexpr int kAutoGemvMaxTokens = 16;
constexpr int kAutoGemvMaxPairs = 256;

int pick_path(int path, int T, int k) {
  if (path == MOE_PATH_AUTO)
    return (T <= kAutoGemvMaxTokens && T * k <= kAutoGemvMaxPairs) ? MOE_PATH_GEMV : MOE_PATH_GROUPED;
  return path;
}

size_t gemv_ws(int H, int I, int T, int k) {
  return std::max(fused_workspace_bytes(H, I, T, k), gemv_workspace_bytes(H, I, T, k));
}

__global__ void publish_kernel(int32_t* slot_of, SlotUpdates u) {
  const int i = threadIdx.x;
  if (i < u.n) slot_of[u.expert[i]] = u.slot[i];
}

}  // namespace

int publish_slot_updates(int32_t* dev_slot_of_layer, const SlotUpdates& u, cudaStream_t st) {
  if (u.n <= 0) return MOE_OK;
  publish_kernel<<<1, kMaxSlotUpdates, 0, st>>>(dev_slot_of_layer, u);
  return check_launch("publish_slot_updates");
}

}  // namespace moe

extern "C" {

size_t moe_forward_workspace_bytes(const moe_expert_shape* s, int T, int k, int E, int path) {
  if (!moe::valid_shape(s) || T < 0 || k < 1 || E < 1) return 0;
  const int p = moe::pick_path(path, T, k);
  if (p == MOE_PATH_GEMV || p == MOE_PATH_GEMV_UNFUSED) return moe::gemv_ws(s->hidden, s->inter, T, k);
  if (p == MOE_PATH_GROUPED) return moe::grouped_workspace_bytes(s->hidden, s->inter, T, k, E);
  return 0;
}

}  // extern "C"

namespace {

// Argument checks and the ForwardArgs shared by the expert-forward entries.
// Returns MOE_OK with *a filled, 1 for an empty batch, or an error code.
int expert_args(const char* who, const moe_expert_shape* s, const void* x, int T, const int32_t* ids,
                const float* weights, int k, int E, const void* pool, const int32_t* slot_of, int n_slots,
                const void* y_shared, void* y, void* workspace, int path, void* stream, moe::ForwardArgs* a) {
  if (!moe::valid_shape(s)) return moe::fail(MOE_ERR_SHAPE, "%s: invalid expert shape", who);
  if (T < 0 || k < 1 || k > 32 || E < 1 || E > 4096 || n_slots < 1)
    return moe::fail(MOE_ERR_ARG, "%s: bad T/k/E/n_slots (%d/%d/%d/%d)", who, T, k, E, n_slots);
  if (path != MOE_PATH_AUTO && path != MOE_PATH_GEMV && path != MOE_PATH_GROUPED &&
      path != MOE_PATH_GEMV_UNFUSED)
    return moe::fail(MOE_ERR_ARG, "%s: unknown path %d", who, path);
  if (T == 0) return 1;
  if (!x || !ids || !weights || !pool || !slot_of || !y || !workspace)
    return moe::fail(MOE_ERR_ARG, "%s: NULL pointer", who);
  if (reinterpret_cast<uintptr_t>(workspace) % 256 || reinterpret_cast<uintptr_t>(pool) % 256 ||
      reinterpret_cast<uintptr_t>(x) % 16)
    return moe::fail(MOE_ERR_ARG, "%s: workspace/pool must be 256-byte and x 16-byte aligned", who);
  const moe::BlockLayout bl = moe::block_layout(s->hidden, s->inter, s->group);
  a->H = s->hidden; a->I = s->inter; a->g = s->group; a->T = T; a->k = k; a->E = E; a->n_slots = n_slots;
  a->x = static_cast<const __half*>(x);
  a->ids = ids; a->weights = weights;
  a->pool = static_cast<const uint8_t*>(pool);
  a->block_bytes = bl.total;
  a->off = moe::offsets_of(bl);
  a->slot_of = slot_of;
  a->y_shared = static_cast<const __half*>(y_shared);
  a->y = static_cast<__half*>(y);
  a->ws = workspace;
  a->stream = static_cast<cudaStream_t>(stream);
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_expert_forward(const moe_expert_shape* s, const void* x, int T,
                       const int32_t* ids, const float* weights, int k, int E,
                       const void* pool, const int32_t* slot_of, int n_slots,
                       const void* y_shared, void* y, void* workspace,
                       size_t workspace_bytes, int path, void* stream) {
  moe::NvtxRange nvtx_range("moe_expert_forward");
  moe::clear_error();
  moe::ForwardArgs a;
  const int rc = expert_args("moe_expert_forward", s, x, T, ids, weights, k, E, pool, slot_of, n_slots, y_shared,
                             y, workspace, path, stream, &a);
  if (rc != MOE_OK) return rc == 1 ? MOE_OK : rc;
  const int p = moe::pick_path(path, T, k);
  const size_t need = moe_forward_workspace_bytes(s, T, k, E, p);
  if (workspace_bytes < need)
    return moe::fail(MOE_ERR_CAPACITY, "moe_expert_forward: workspace %zu < %zu bytes", workspace_bytes, need);
  a.ws_bytes = workspace_bytes;
  if (p == MOE_PATH_GEMV) {
    const int frc = moe::fused_forward(a);
    if (frc != MOE_ERR_UNSUPPORTED) return frc;
    moe::clear_error();  // shapes beyond the fused kernel's shared memory
    return moe::gemv_forward(a);
  }
  if (p == MOE_PATH_GEMV_UNFUSED) return moe::gemv_forward(a);
  return moe::grouped_forward(a);
}

int moe_expert_forward_zero_copy(const moe_expert_shape* s, const void* x, int T,
                                 const int32_t* ids, const float* weights, int k, int E,
                                 const void* pool, const int32_t* slot_of, int n_slots,
                                 const void* host_src, const void* y_shared, void* y,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  moe::NvtxRange nvtx_range("moe_expert_forward_zero_copy");
  moe::clear_error();
  moe::ForwardArgs a;
  const int rc = expert_args("moe_expert_forward_zero_copy", s, x, T, ids, weights, k, E, pool, slot_of, n_slots,
                             y_shared, y, workspace, MOE_PATH_GEMV_UNFUSED, stream, &a);
  if (rc != MOE_OK) return rc == 1 ? MOE_OK : rc;
  if (!host_src) return moe::fail(MOE_ERR_ARG, "moe_expert_forward_zero_copy: NULL host_src");
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, host_src) != cudaSuccess || pa.type != cudaMemoryTypeHost ||
      !pa.devicePointer) {
    cudaGetLastError();
    return moe::fail(MOE_ERR_ARG, "moe_expert_forward_zero_copy: host_src must be page-locked, mapped host memory");
  }
  // Device alias of host_src itself (an interior pointer keeps its offset).
  const uint8_t* dev_src = static_cast<const uint8_t*>(pa.devicePointer);
  if (pa.hostPointer) dev_src += static_cast<const uint8_t*>(host_src) - static_cast<const uint8_t*>(pa.hostPointer);
  if (reinterpret_cast<uintptr_t>(dev_src) % 16)
    return moe::fail(MOE_ERR_ARG, "moe_expert_forward_zero_copy: host_src must be 16-byte aligned");
  const size_t need = moe_forward_workspace_bytes(s, T, k, E, MOE_PATH_GEMV_UNFUSED);
  if (workspace_bytes < need)
    return moe::fail(MOE_ERR_CAPACITY, "moe_expert_forward_zero_copy: workspace %zu < %zu bytes", workspace_bytes,
                     need);
  a.ws_bytes = workspace_bytes;
  a.host = dev_src;
  return moe::gemv_forward(a);
}

int moe_layer_forward(const moe_expert_shape* s, const void* x, const float* logits, int T, int E,
                      int k, int renorm, int32_t* ids, float* weights, const void* pool,
                      const int32_t* slot_of, int n_slots, const void* y_shared, void* y,
                      void* workspace, size_t workspace_bytes, int path, void* stream) {
  moe::NvtxRange nvtx_range("moe_layer_forward");
  moe::clear_error();
  if (!moe::valid_shape(s)) return moe::fail(MOE_ERR_SHAPE, "moe_layer_forward: invalid expert shape");
  if (T < 0 || E < 1 || E > 4096 || k < 1 || k > 32 || k > E || n_slots < 1)
    return moe::fail(MOE_ERR_ARG, "moe_layer_forward: bad T/E/k/n_slots (%d/%d/%d/%d)", T, E, k, n_slots);
  if (path != MOE_PATH_AUTO && path != MOE_PATH_GEMV && path != MOE_PATH_GROUPED &&
      path != MOE_PATH_GEMV_UNFUSED)
    return moe::fail(MOE_ERR_ARG, "moe_layer_forward: unknown path %d", path);
  if (T == 0) return MOE_OK;
  if (!x || !logits || !ids || !weights || !pool || !slot_of || !y || !workspace)
    return moe::fail(MOE_ERR_ARG, "moe_layer_forward: NULL pointer");
  const int p = moe::pick_path(path, T, k);
  if (p == MOE_PATH_GEMV) {
    if (reinterpret_cast<uintptr_t>(workspace) % 256 || reinterpret_cast<uintptr_t>(pool) % 256 ||
        reinterpret_cast<uintptr_t>(x) % 16)
      return moe::fail(MOE_ERR_ARG, "moe_layer_forward: workspace/pool must be 256-byte and x 16-byte aligned");
    const size_t need = moe_forward_workspace_bytes(s, T, k, E, p);
    if (workspace_bytes < need)
      return moe::fail(MOE_ERR_CAPACITY, "moe_layer_forward: workspace %zu < %zu bytes", workspace_bytes, need);
    const moe::BlockLayout bl = moe::block_layout(s->hidden, s->inter, s->group);
    moe::ForwardArgs a;
    a.H = s->hidden; a.I = s->inter; a.g = s->group; a.T = T; a.k = k; a.E = E; a.n_slots = n_slots;
    a.x = static_cast<const __half*>(x);
    a.ids = ids; a.weights = weights;
    a.pool = static_cast<const uint8_t*>(pool);
    a.block_bytes = bl.total;
    a.off = moe::offsets_of(bl);
    a.slot_of = slot_of;
    a.y_shared = static_cast<const __half*>(y_shared);
    a.y = static_cast<__half*>(y);
    a.ws = workspace; a.ws_bytes = workspace_bytes;
    a.stream = static_cast<cudaStream_t>(stream);
    const int rc = moe::fused_forward_routed(a, logits, renorm, ids, weights);
    if (rc != MOE_ERR_UNSUPPORTED) return rc;
    moe::clear_error();
  }
  int rc = moe_route(logits, T, E, k, renorm, ids, weights, nullptr, stream);
  if (rc != MOE_OK) return rc;
  return moe_expert_forward(s, x, T, ids, weights, k, E, pool, slot_of, n_slots, y_shared, y,
                            workspace, workspace_bytes, path, stream);
}

int moe_workspace_clear_flags(void* workspace, void* stream) {
  moe::clear_error();
  if (!workspace) return moe::fail(MOE_ERR_ARG, "NULL workspace");
  MOE_CUDA_TRY(cudaMemsetAsync(workspace, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_workspace_flags(const void* workspace, int32_t* flags_out, void* stream) {
  moe::clear_error();
  if (!workspace || !flags_out) return moe::fail(MOE_ERR_ARG, "NULL pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_CUDA_TRY(cudaMemcpyAsync(flags_out, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  MOE_CUDA_TRY(cudaStreamSynchronize(st));
  return MOE_OK;
}

}  // extern "C"
