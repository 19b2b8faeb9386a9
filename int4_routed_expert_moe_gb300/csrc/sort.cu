// Token sort for the grouped executor: (token, choice) pairs grouped by
// expert, stable in the pair index p = t*k + j.
// "Horizon RunMap -- Prévia Técnica", "04 / Resultados": compact experts
// computed in groups.
//
// One block of 32 warps. Warp w owns the contiguous pair segment
// [w*seg, (w+1)*seg). Pass 1 counts, per warp and expert, the pairs of the
// segment (warp match instead of atomics). Pass 2 turns the counts into
// per-warp starting positions (prefix over warps, then a block-wide exclusive
// scan over experts, a thread per expert). Pass 3 re-walks each segment in
// order and scatters; ranks inside a 32-pair chunk come from the match mask,
// so the order is stable.
#include "common.h"
#include "device.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kSortWarps = 32;

__global__ void __launch_bounds__(kSortWarps * 32) token_sort_kernel(
    const int32_t* __restrict__ ids, int P, int k, int E, int32_t* __restrict__ offsets,
    int32_t* __restrict__ pair_tok, int32_t* __restrict__ pair_j, const SortTiles tl) {
  extern __shared__ __align__(16) int32_t sm[];
  int32_t* cnt = sm;                          // [kSortWarps][E]
  int32_t* total = sm + kSortWarps * E;       // [E + 1]
  int32_t* slot = total + E + 1;              // [E] copy of slot_of (tile list / id check only)
  int32_t* wsc = slot + E;                    // [2][kSortWarps] warp sums of the expert scans
  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < kSortWarps * E; i += blockDim.x) cnt[i] = 0;
  if (tl.tiles)
    for (int e = tid; e < E; e += blockDim.x) slot[e] = tl.slot_of[e];
  __syncthreads();
  const int seg = (P + kSortWarps - 1) / kSortWarps;
  const int p0 = warp * seg, p1 = min(P, p0 + seg);
  const unsigned lt_mask = (1u << lane) - 1u;
  // Pass 1: per-warp histogram (rounds unrolled, so that their id loads are
  // in flight together).
#pragma unroll 4
  for (int base = p0; base < p1; base += 32) {
    const int p = base + lane;
    int e = -1;
    if (p < p1) {
      e = ids[p];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned active = __ballot_sync(0xffffffffu, p < p1);
    const unsigned peers = __match_any_sync(0xffffffffu, e) & active;
    if (p < p1 && e >= 0 && (peers & lt_mask) == 0) cnt[warp * E + e] += __popc(peers);
    if (tl.tiles) {  // report unusable ids (error-word bits 0 and 1)
      int bad_id = 0, no_slot = 0;
      if (p < p1) {
        const int raw = ids[p];
        if (raw != -1 && (raw < 0 || raw >= E)) bad_id = 1;
        else if (raw >= 0) {
          const int sl = slot[raw];
          no_slot = sl < 0 || sl >= tl.n_slots;
        }
      }
      const int any_bad = __any_sync(0xffffffffu, bad_id), any_noslot = __any_sync(0xffffffffu, no_slot);
      if (lane == 0 && (any_bad || any_noslot)) atomicOr(tl.flags, (any_bad ? 2 : 0) | (any_noslot ? 1 : 0));
    }
    __syncwarp();
  }
  __syncthreads();
  // Pass 2 (thread e = expert e, E <= blockDim): the exclusive prefix of the
  // expert's counts over the warps (in place), then block-wide exclusive
  // scans over experts of the totals (the experts' first sorted positions)
  // and of the tile counts (tile list: every resident expert with pairs,
  // tiles of up to tile_n consecutive sorted pairs: slot, first position,
  // pairs, expert).
  {
    int tot = 0, tc = 0, sl = -1;
    if (tid < E) {
      for (int w = 0; w < kSortWarps; ++w) {
        const int c = cnt[w * E + tid];
        cnt[w * E + tid] = tot;
        tot += c;
      }
      if (tl.tiles) {
        sl = slot[tid];
        if (tot > 0 && sl >= 0 && sl < tl.n_slots) tc = (tot + tl.tile_n - 1) / tl.tile_n;
      }
    }
    int it = tot, ic = tc;  // inclusive within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, it, o), b = __shfl_up_sync(0xffffffffu, ic, o);
      if (lane >= o) {
        it += a;
        ic += b;
      }
    }
    if (lane == 31) {
      wsc[warp] = it;
      wsc[kSortWarps + warp] = ic;
    }
    __syncthreads();
    if (warp == 0) {  // exclusive prefix of the warp sums
      const int a = wsc[lane], b = wsc[kSortWarps + lane];
      int ia = a, ib = b;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int na = __shfl_up_sync(0xffffffffu, ia, o), nb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) {
          ia += na;
          ib += nb;
        }
      }
      wsc[lane] = ia - a;
      wsc[kSortWarps + lane] = ib - b;
    }
    __syncthreads();
    const int first = wsc[warp] + it - tot, tfirst = wsc[kSortWarps + warp] + ic - tc;
    if (tid < E) total[tid] = first;
    if (tid == E - 1) {
      total[E] = first + tot;
      if (tl.tiles) *tl.n_tiles = tfirst + tc;
    }
    for (int i = 0; i < tc; ++i)
      tl.tiles[tfirst + i] = make_int4(sl, first + i * tl.tile_n, min(tl.tile_n, tot - i * tl.tile_n), tid);
  }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) offsets[e] = total[e];
  // Pass 3: stable scatter.
#pragma unroll 4
  for (int base = p0; base < p1; base += 32) {
    const int p = base + lane;
    int e = -1;
    if (p < p1) {
      e = ids[p];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned active = __ballot_sync(0xffffffffu, p < p1);
    const unsigned peers = __match_any_sync(0xffffffffu, e) & active;
    int pos = 0;
    if (p < p1 && e >= 0) pos = total[e] + cnt[warp * E + e] + __popc(peers & lt_mask);
    __syncwarp();
    if (p < p1 && e >= 0) {
      pair_tok[pos] = p / k;
      pair_j[pos] = p - (p / k) * k;
      if ((peers & lt_mask) == 0) cnt[warp * E + e] += __popc(peers);
    }
    __syncwarp();
  }
}

}  // namespace

int launch_token_sort(const int32_t* ids, int P, int k, int E, int32_t* offsets,
                      int32_t* pair_tok, int32_t* pair_j, cudaStream_t st, const SortTiles* tiles) {
  const size_t smem = (size_t)(kSortWarps * E + 2 * E + 1 + 2 * kSortWarps) * sizeof(int32_t);
  cudaError_t e = cudaFuncSetAttribute(token_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "token_sort smem attr: %s", cudaGetErrorString(e));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kSortWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  SortTiles tl = {};
  if (tiles) tl = *tiles;
  e = cudaLaunchKernelEx(&cfg, token_sort_kernel, ids, P, k, E, offsets, pair_tok, pair_j, tl);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "token_sort launch: %s", cudaGetErrorString(e));
  return MOE_OK;
}

}  // namespace moe

extern "C" int moe_token_sort(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                              int32_t* pair_tok, int32_t* pair_j, void* stream) {
  moe::NvtxRange nvtx_range("moe_token_sort");
  moe::clear_error();
  if (T < 0 || k < 1 || E < 1 || E > 1024 || (long long)T * k > 65536)
    return moe::fail(MOE_ERR_ARG, "moe_token_sort: need E <= 1024, T*k <= 65536 (T=%d k=%d E=%d)", T, k, E);
  if (!offsets || (T > 0 && (!ids || !pair_tok || !pair_j)))
    return moe::fail(MOE_ERR_ARG, "moe_token_sort: NULL pointer");
  return moe::launch_token_sort(ids, T * k, k, E, offsets, pair_tok, pair_j,
                                static_cast<cudaStream_t>(stream), nullptr);
}
