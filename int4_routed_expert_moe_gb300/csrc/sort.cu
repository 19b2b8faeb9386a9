// Token sort for the grouped executor: (token, choice) pairs grouped by
// expert, stable in the pair index p = t*k + j.
// "Horizon RunMap -- Prévia Técnica", "04 / Resultados": compact experts
// computed in groups.
//
// One block of 32 warps (the whole sort is a few thousand pairs: one SM,
// bound by its instruction issue). Warp w owns the contiguous pair segment
// [w*seg, (w+1)*seg). Pass 1 counts, per warp and expert, the pairs of the
// segment (shared-memory atomics; the order does not matter there). Pass 2
// turns the counts into per-warp starting positions (prefix over warps, then
// a block-wide exclusive scan over experts, a thread per expert). Pass 3
// re-walks each segment in order and scatters: the lanes of a 32-pair chunk
// that hold the same expert are found by one ballot per bit of the expert id
// (a warp multisplit), and a lane's rank is the number of them below it, so
// the order is stable. The ids of the first kCachedRounds chunks of a segment
// stay in registers between the passes.
#include <mutex>

#include "common.h"
#include "device.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kSortWarps = 32;
constexpr int kCachedRounds = 8;  // P <= 32 * 32 * 8 = 8192 pairs: ids read once
// Up to this many pairs the scatter of pass 3 goes to shared memory first and
// leaves in coalesced rows: from one SM, P scattered 4-byte stores to each of
// two arrays cost about a microsecond per thousand pairs.
constexpr int kStagedPairs = 8192;

// Lanes of the warp whose key equals this lane's (keys in [0, 2^nbits);
// nbits <= 11 since E <= 1024): one ballot per key bit, keeping the lanes
// that agree on every bit.
__device__ __forceinline__ unsigned same_key_lanes(unsigned key, int nbits) {
  unsigned m = 0xffffffffu;
#pragma unroll
  for (int b = 0; b < 11; ++b) {
    if (b >= nbits) break;
    const bool bit = (key >> b) & 1u;
    const unsigned on = __ballot_sync(0xffffffffu, bit);
    m &= bit ? on : ~on;
  }
  return m;
}

__global__ void __launch_bounds__(kSortWarps * 32) token_sort_kernel(
    const int32_t* __restrict__ ids, int P, int k, int E, int32_t* __restrict__ offsets,
    int32_t* __restrict__ pair_tok, int32_t* __restrict__ pair_j, const SortTiles tl) {
  extern __shared__ __align__(16) int32_t sm[];
  int32_t* cnt = sm;                          // [kSortWarps][E]
  int32_t* total = sm + kSortWarps * E;       // [E + 1]
  int32_t* slot = total + E + 1;              // [E] copy of slot_of (tile list / id check only)
  int32_t* wsc = slot + E;                    // [2][kSortWarps] warp sums of the expert scans
  const bool staged = P <= kStagedPairs;
  int32_t* st_tok = wsc + 2 * kSortWarps;     // [P] sorted pair_tok (staged scatter only)
  int32_t* st_j = st_tok + (staged ? P : 0);  // [P] sorted pair_j
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
  const int nbits = 32 - __clz(E);  // keys e + 1 in [0, E]
  // Pass 1: per-warp histogram. The first kCachedRounds chunks' ids are
  // loaded together and kept for pass 3.
  int raw_c[kCachedRounds];
#pragma unroll
  for (int r = 0; r < kCachedRounds; ++r) {
    const int p = p0 + 32 * r + lane;
    raw_c[r] = p < p1 ? ids[p] : -1;
  }
  int bad_id = 0, no_slot = 0;
#pragma unroll
  for (int r = 0; r < kCachedRounds; ++r) {
    const int p = p0 + 32 * r + lane;
    if (p0 + 32 * r >= p1) break;
    const int raw = raw_c[r];
    if (p < p1 && raw >= 0 && raw < E) atomicAdd(&cnt[warp * E + raw], 1);
    if (tl.tiles && p < p1) {  // unusable ids (error-word bits 0 and 1)
      if (raw != -1 && (raw < 0 || raw >= E)) bad_id = 1;
      else if (raw >= 0) no_slot |= slot[raw] < 0 || slot[raw] >= tl.n_slots;
    }
  }
  for (int base = p0 + 32 * kCachedRounds; base < p1; base += 32) {
    const int p = base + lane;
    const int raw = p < p1 ? ids[p] : -1;
    if (p < p1 && raw >= 0 && raw < E) atomicAdd(&cnt[warp * E + raw], 1);
    if (tl.tiles && p < p1) {
      if (raw != -1 && (raw < 0 || raw >= E)) bad_id = 1;
      else if (raw >= 0) no_slot |= slot[raw] < 0 || slot[raw] >= tl.n_slots;
    }
  }
  if (tl.tiles) {
    const int any_bad = __any_sync(0xffffffffu, bad_id), any_noslot = __any_sync(0xffffffffu, no_slot);
    if (lane == 0 && (any_bad || any_noslot)) atomicOr(tl.flags, (any_bad ? 2 : 0) | (any_noslot ? 1 : 0));
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
  // Pass 3: stable scatter. floor(p / k) = (p * ceil(2^32 / k)) >> 32
  // exactly for p, k <= 2^16: the excess over p / k is below p / 2^32 <= 2^-16,
  // and the fractional part of p / k is at most 1 - 1 / k.
  const unsigned long long kmagic = (0x100000000ull + (unsigned)k - 1u) / (unsigned)k;
  auto scatter = [&](int p, int raw) {
    const int e = (p < p1 && raw >= 0 && raw < E) ? raw : -1;
    const unsigned peers = same_key_lanes((unsigned)(e + 1), nbits);
    int pos = 0;
    if (e >= 0) pos = total[e] + cnt[warp * E + e] + __popc(peers & lt_mask);
    __syncwarp();
    if (e >= 0) {
      const int t = (int)(((unsigned long long)p * kmagic) >> 32);  // p / k
      int32_t* dt = staged ? st_tok : pair_tok;
      int32_t* dj = staged ? st_j : pair_j;
      dt[pos] = t;
      dj[pos] = p - t * k;
      if ((peers & lt_mask) == 0) cnt[warp * E + e] += __popc(peers);
    }
    __syncwarp();
  };
#pragma unroll
  for (int r = 0; r < kCachedRounds; ++r) {
    if (p0 + 32 * r >= p1) break;
    scatter(p0 + 32 * r + lane, raw_c[r]);
  }
  for (int base = p0 + 32 * kCachedRounds; base < p1; base += 32) {
    const int p = base + lane;
    scatter(p, p < p1 ? ids[p] : -1);
  }
  if (staged) {  // the valid pairs fill sorted positions [0, total[E])
    __syncthreads();
    const int n = total[E];
    for (int i = tid; i < n; i += blockDim.x) {
      pair_tok[i] = st_tok[i];
      pair_j[i] = st_j[i];
    }
  }
}

}  // namespace

int launch_token_sort(const int32_t* ids, int P, int k, int E, int32_t* offsets,
                      int32_t* pair_tok, int32_t* pair_j, cudaStream_t st, const SortTiles* tiles) {
  const size_t smem =
      (size_t)(kSortWarps * E + 2 * E + 1 + 2 * kSortWarps + (P <= kStagedPairs ? 2 * P : 0)) * sizeof(int32_t);
  int dev = 0, n_sm = 0;
  int rc = current_device_sms(&dev, &n_sm);
  if (rc != MOE_OK) return rc;
  cudaError_t e;
  {
    // Per device, the largest dynamic shared memory granted so far.
    static std::mutex mu;
    static int granted[kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (granted[dev] < (int)smem) {
      e = cudaFuncSetAttribute(token_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "token_sort smem attr: %s", cudaGetErrorString(e));
      granted[dev] = (int)smem;
    }
  }
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
