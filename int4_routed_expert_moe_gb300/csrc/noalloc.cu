// A routed-layer entry point for callers that cannot allocate device memory.
//
// moe_layer_forward needs a caller-provided workspace. Some callers cannot
// provide one: plugins and serving runtimes whose host framework owns every
// device allocation and forbids extra ones, and deployments with a fixed,
// pre-planned memory budget. moe_layer_forward_noalloc serves them from a
// fixed scratch array compiled into the library.
#include <mutex>

#include "common.h"
#include "kernels.h"

namespace moe {
namespace {

// Scratch of the streamed decode path (error word + h of every pair), held
// by every GPU that loads this library until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device. The first call
// on a device looks it up (cudaGetSymbolAddress); later calls reuse it.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(MOE_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_layer_forward_noalloc(const moe_expert_shape* s, const void* x,
                                         const float* logits, int T, int E, int k, int renorm,
                                         int32_t* ids, float* weights, const void* pool,
                                         const int32_t* slot_of, int n_slots,
                                         const void* y_shared, void* y, void* stream) {
  moe::NvtxRange nvtx_range("moe_layer_forward_noalloc");
  moe::clear_error();
  if (!moe::valid_shape(s)) return moe::fail(MOE_ERR_SHAPE, "moe_layer_forward_noalloc: invalid expert shape");
  if (T < 0 || E < 1 || E > 4096 || k < 1 || k > 32 || k > E || n_slots < 1)
    return moe::fail(MOE_ERR_ARG, "moe_layer_forward_noalloc: bad T/E/k/n_slots (%d/%d/%d/%d)", T, E, k, n_slots);
  if (T == 0) return MOE_OK;
  if (!x || !logits || !ids || !weights || !pool || !slot_of || !y)
    return moe::fail(MOE_ERR_ARG, "moe_layer_forward_noalloc: NULL pointer");
  if (reinterpret_cast<uintptr_t>(pool) % 256 || reinterpret_cast<uintptr_t>(x) % 16)
    return moe::fail(MOE_ERR_ARG, "moe_layer_forward_noalloc: pool must be 256-byte and x 16-byte aligned");
  const size_t need = moe::fused_workspace_bytes(s->hidden, s->inter, T, k);
  if (need > moe::kNoAllocScratchBytes)
    return moe::fail(MOE_ERR_CAPACITY,
                     "moe_layer_forward_noalloc: needs %zu bytes of scratch, the fixed array holds %zu "
                     "(T*k*inter*2 + header must stay within it)",
                     need, moe::kNoAllocScratchBytes);
  void* ws = nullptr;
  int rc = moe::scratch_address(&ws);
  if (rc != MOE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The header (error word, the kernel's counters) must start at zero for
  // this call, whatever an earlier call left in it.
  cudaError_t e = cudaMemsetAsync(ws, 0, moe::ws_scratch_offset(T * k), st);
  if (e != cudaSuccess) return moe::fail(MOE_ERR_CUDA, "clearing the scratch header: %s", cudaGetErrorString(e));
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
  a.ws = ws;
  a.ws_bytes = moe::kNoAllocScratchBytes;
  a.stream = st;
  rc = moe::fused_forward_routed(a, logits, renorm, ids, weights);
  if (rc == MOE_ERR_UNSUPPORTED)
    return moe::fail(MOE_ERR_UNSUPPORTED,
                     "moe_layer_forward_noalloc: request outside the streamed decode kernel (H <= 4096, "
                     "I <= 2048, T <= 16, T*k <= 256, E <= 1024, shared-memory fit)");
  return rc;
}

extern "C" int moe_layer_forward_noalloc_flags(int32_t* flags_out, void* stream) {
  moe::clear_error();
  if (!flags_out) return moe::fail(MOE_ERR_ARG, "moe_layer_forward_noalloc_flags: NULL flags_out");
  void* ws = nullptr;
  int rc = moe::scratch_address(&ws);
  if (rc != MOE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(flags_out, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess)
    return moe::fail(MOE_ERR_CUDA, "moe_layer_forward_noalloc_flags: %s", cudaGetErrorString(e));
  return MOE_OK;
}
