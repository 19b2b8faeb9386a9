// Router: top-k experts per token with softmax weights.
// "Horizon RunMap -- Prévia Técnica", "02 / A solução": the router chooses the
// experts of each token; it stays outside the INT4 compression.
#include <cfloat>
#include <climits>

#include "common.h"
#include "device.cuh"

namespace moe {
namespace {

// One warp per token. Lane l holds elements l, l+32, ... (PER_LANE of them);
// warp_topk picks the k best in order (per-lane cache of its best elements,
// warp reductions for the best of the round).
template <int PER_LANE>
__global__ void __launch_bounds__(128) route_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renorm,
    int32_t* __restrict__ ids, float* __restrict__ weights,
    int32_t* __restrict__ bad_tokens) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;

  float v[PER_LANE];
  bool bad = false;
  int n_neg_inf = 0;
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    const int e = lane + 32 * i;
    float x = -INFINITY;
    if (e < E) {
      x = row[e];
      if (isnan(x) || x == INFINITY) bad = true;
      if (x == -INFINITY) ++n_neg_inf;
    }
    v[i] = x;
  }
  // Pad elements (e >= E) are never picked and add 0 to the softmax sum.
  const unsigned full = 0xffffffffu;
  bad = __any_sync(full, bad);
  int total_ninf = n_neg_inf;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total_ninf += __shfl_xor_sync(full, total_ninf, o);
  if (total_ninf == E) bad = true;
  if (bad) {
    if (lane < k) {
      ids[(size_t)t * k + lane] = -1;
      weights[(size_t)t * k + lane] = 0.0f;
    }
    if (lane == 0 && bad_tokens) atomicAdd(bad_tokens, 1);
    return;
  }

  float my_v = 0.0f;
  int my_i = -1;
  warp_topk<PER_LANE>(v, E, k, lane, my_v, my_i);  // lane r < k: pick r

  // Softmax over all E in FP32, shifted by the top logit.
  const float m = __shfl_sync(full, my_v, 0);
  float s_all = 0.0f;
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) s_all += expf(v[i] - m);  // pads give 0
  s_all = warp_sum(s_all);
  const float mine = (lane < k) ? expf(my_v - m) : 0.0f;
  const float s_sel = warp_sum(mine);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_i;
    weights[(size_t)t * k + lane] = mine / (renorm ? s_sel : s_all);
  }
}

template <int PL>
cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm,
                         int32_t* ids, float* w, int32_t* bad, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((T + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_kernel<PL>, logits, T, E, k, renorm, ids, w, bad);
}

}  // namespace
}  // namespace moe

extern "C" int moe_route(const float* logits, int T, int E, int k, int renorm,
                         int32_t* ids, float* weights, int32_t* bad_tokens,
                         void* stream) {
  moe::NvtxRange nvtx_range("moe_route");
  moe::clear_error();
  if (T < 0 || E < 1 || E > 4096 || k < 1 || k > 32 || k > E)
    return moe::fail(MOE_ERR_ARG, "moe_route: need T >= 0, 1 <= k <= min(E, 32), E <= 4096 (T=%d E=%d k=%d)", T, E, k);
  if (T == 0) return MOE_OK;
  if (!logits || !ids || !weights) return moe::fail(MOE_ERR_ARG, "moe_route: NULL pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (E <= 64) e = moe::launch_route<2>(logits, T, E, k, renorm, ids, weights, bad_tokens, st);
  else if (E <= 256) e = moe::launch_route<8>(logits, T, E, k, renorm, ids, weights, bad_tokens, st);
  else if (E <= 1024) e = moe::launch_route<32>(logits, T, E, k, renorm, ids, weights, bad_tokens, st);
  else e = moe::launch_route<128>(logits, T, E, k, renorm, ids, weights, bad_tokens, st);
  if (e != cudaSuccess) return moe::fail(MOE_ERR_CUDA, "moe_route launch: %s", cudaGetErrorString(e));
  return MOE_OK;
}
