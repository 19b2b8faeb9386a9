// Decode path: two streaming kernels per routed layer, chained with
// programmatic dependent launch.
//
// "Horizon RunMap -- Prévia Técnica", "03 / Arquitetura" and
// "08 / Comportamento do modelo": the expert kernel reads compact INT4 codes
// and FP16 scales, converts them inside the kernel (no expanded expert is
// kept) and works with FP16 activations and FP32 accumulation.
//
// Both kernels run one block per SM (G blocks). Block c owns gate/up rows
// n in [c*I/G, (c+1)*I/G) of every (token, choice) pair p and output rows
// m in [c*H/G, (c+1)*H/G) of y. In each kernel a producer warp streams the
// block's slice of expert ids[p]'s block into a ring of shared-memory stages
// with bulk async copies (cp.async.bulk, completion counted on mbarriers);
// for one decode token the ring holds every pair, so the whole slice is
// requested at once and HBM sees one deep stream.
//   * Routing (optional, moe_layer_forward): each block ranks the router
//     logits itself -- expert e is chosen at position r when exactly r
//     experts precede it in (logit desc, index asc) order -- and computes the
//     softmax weights with fixed-order reductions, so every block of both
//     kernels derives identical ids and weights without waiting for another.
//   * decode_gateup_kernel: h[p][n] = silu(W_g x_t)[n] * (W_u x_t)[n],
//     rounded to FP16 (the explicit rounding point) into the workspace.
//   * decode_down_kernel: launched while the first kernel runs; before
//     waiting on it (griddepcontrol.wait) it already requests its down-row
//     slices (the ids are final), so the down weights stream concurrently
//     with the gate/up weights. After the wait it reads h and computes
//     y[t][m] = sum_j w[t][j] * (W_d h[t*k+j])[m] (+ y_shared), combining the
//     k pairs of a token in j order (deterministic).
// The kernel boundary is the only synchronisation: nothing spins on flags
// written by other blocks. mbarrier waits are bounded; on expiry bit 2 of the
// workspace error word is set.
#include <algorithm>

#include "common.h"
#include "device.cuh"
#include "kernels.h"

namespace moe {
namespace {

// Warp counts: registers are granted to a block in units of four warps, so
// 16 + 12 warps of the two kernels fit one SM together (64K registers).
constexpr int kWarps = 8;                   // compute warps of the down kernel
constexpr int kThreads = (kWarps + 1) * 32;   // + one producer warp
constexpr int kGateWarps = 15;              // compute warps of the gate/up kernel
constexpr int kGateThreads = (kGateWarps + 1) * 32;
constexpr int kSub0 = 8;                    // gate/up ring: warps 0..7 take even pairs, 8..14 odd pairs
constexpr int kPairsPerIter = 2;
// Stage ownership when the ring wraps: a stage must always be drained by the
// same warp (down) or sub-group (gate/up) so that no consumer waits on a
// phase two fills ahead (an mbarrier parity test cannot tell those apart).
// With an even stage count, stage q % S of pair q is drained by sub-group
// q & 1 (gate/up) and by warp (q % S) % kWarps (down), each in increasing q.
// When every pair has its own stage (P <= S, one decode token), each stage
// is filled once and never released, and the gate/up warps share pairs.
constexpr int kMaxStages = 8;
constexpr unsigned kMbarTries = 50000;     // bounded mbarrier waits (~1 s)

// ---- PTX wrappers: mbarrier, bulk copies, acquire/release -----------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or about 20 us pass, instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(20000u) : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase; returns false on expiry (~1 s at most).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (unsigned i = 0; i < kMbarTries; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// ---- shared-memory stages -------------------------------------------------
__host__ __device__ inline uint32_t align16(uint32_t v) { return (v + 15u) & ~15u; }

// One stage = the block's rows of one pair's expert (rmax rows at most).
struct Stage {
  uint32_t bytes;
};
__host__ __device__ inline Stage stage_of(int rmax, uint32_t row_bytes) {
  Stage st;
  st.bytes = align16((uint32_t)rmax * row_bytes);
  return st;
}

// 32 FP16 values (64 bytes, read through L2) as the scaled pairs of
// dot16_scaled; returns their sum, and 2^(24-s) in back.
__device__ __forceinline__ float load_scaled_chunk(const __half* src, half2 (&xp)[16], float& back) {
  float v[32];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(src + 8 * q) : "memory");
    const __half* e = reinterpret_cast<const __half*>(&r);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[8 * q + i] = __half2float(e[i]);
  }
  float sum = 0.0f, amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    sum += v[i];
    amax = fmaxf(amax, fabsf(v[i]));
  }
  const int sh = chunk_shift(amax);
#pragma unroll
  for (int q = 0; q < 4; ++q) scaled_perm8(v + 8 * q, sh, xp + 4 * q);
  back = pow2f(24 - sh);
  return sum;
}

struct DecodeParams {
  const __half* x;
  const float* logits;  // [T][E] when the kernels route themselves, else NULL
  int renorm;
  const int32_t* ids;   // [T][k] given ids (logits == NULL)
  const float* wts;     // [T][k] given weights (logits == NULL)
  int32_t* ids_out;     // routed ids / weights written by block 0 (nullable)
  float* wts_out;
  const uint8_t* pool;
  unsigned long long block_bytes;
  BlockOffsets off;
  const int32_t* slot_of;
  const __half* y_shared;
  __half* y;
  int32_t* flags;  // workspace error word
  __half* hbuf;    // workspace: h [P][I]
  int H, I, g, T, k, E, n_slots, P, G, stages;
  Stage st;
  uint32_t part_off, route_off, bar_off, blk_off;  // shared-memory carve-up after the stages
};

// Per-block routing state in shared memory.
struct RouteSmem {
  int32_t* ids;    // [P]
  float* w;        // [P]
  float* exsel;    // [P]   exp(logit - max) of each chosen expert
  float* sall;     // [T]   softmax denominator per token
  float* red;      // [ceil(E/32)] sums of exp over 32-expert slices
  int32_t* bad;    // [4]:  any NaN/+inf, count of -inf, max key
  float* lg;       // [E]   logits of the token being routed
  int32_t* rank;   // [E]
  int32_t* slot;   // [E]   copy of slot_of (when slot_tab)
};

// Experts up to this count get a shared-memory copy of slot_of.
constexpr int kSlotTableMax = 1024;

__host__ __device__ inline size_t route_smem_bytes(int P, int T, int E, bool routing) {
  return (size_t)P * 12 + (size_t)T * 4 + (size_t)(4 + (E + 31) / 32) * 4 + (routing ? (size_t)E * 8 : 0) +
         (E <= kSlotTableMax ? (size_t)E * 4 : 0);
}

__device__ __forceinline__ RouteSmem route_smem(const DecodeParams& a, uint8_t* sm) {
  RouteSmem r;
  uint8_t* b = sm + a.route_off;
  r.ids = reinterpret_cast<int32_t*>(b);
  r.w = reinterpret_cast<float*>(r.ids + a.P);
  r.exsel = r.w + a.P;
  r.sall = r.exsel + a.P;
  r.red = r.sall + a.T;
  r.bad = reinterpret_cast<int32_t*>(r.red + (a.E + 31) / 32);
  r.lg = reinterpret_cast<float*>(r.bad + 4);
  r.rank = reinterpret_cast<int32_t*>(r.lg + (a.logits ? a.E : 0));
  r.slot = r.rank + (a.logits ? a.E : 0);
  return r;
}

// Order-preserving int key of a float that is not NaN (for atomicMax).
__device__ __forceinline__ int32_t float_key(float v) {
  const int32_t b = __float_as_int(v);
  return b >= 0 ? b : b ^ 0x7fffffff;
}
__device__ __forceinline__ float key_float(int32_t k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

__device__ __forceinline__ const uint8_t* resolve_slot(const DecodeParams& a, int e, int s) {
  if (e < 0 || e >= a.E || s < 0 || s >= a.n_slots) return nullptr;
  return a.pool + (size_t)s * a.block_bytes;
}

// Expert block of expert e, with unusable-id reporting by the writer block.
__device__ __forceinline__ const uint8_t* resolve_report(const DecodeParams& a, const RouteSmem& r, int e,
                                                         bool table, bool writer) {
  const int s = (e < 0 || e >= a.E) ? -1 : (table ? r.slot[e] : a.slot_of[e]);
  const uint8_t* b = resolve_slot(a, e, s);
  if (writer && !b) {
    if (e != -1 && (e < 0 || e >= a.E)) atomicOr(a.flags, 2);
    else if (e >= 0) atomicOr(a.flags, 1);
  }
  return b;
}

// "Horizon RunMap -- Prévia Técnica", "02 / A solução": the router picks the
// experts of each token. Same definition as moe_route: top-k by (logit desc,
// index asc), softmax over all E, optionally renormalised over the k; a
// token with NaN/+inf logits or all -inf gets ids -1 and weights 0.
// Per token: (A) logits to shared memory; (B) rank counts split over threads
// (thread (e, part) counts the experts of one slice of j that precede e;
// integer sums, so the order is free) and the maximum logit; (C) the chosen
// experts, their blocks and exp(logit - max), and the sum of exp over each
// slice of 32 experts (one warp, fixed tree); the slice sums are then added
// in slice order, so the denominator does not depend on the block size.
// Three block barriers per token. The weights are formed afterwards by warp
// 0 (finish_weights).
__device__ void route_block(const DecodeParams& a, const RouteSmem& r, const uint8_t** blk_of, bool table,
                            bool writer) {
  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31;
  const int nslices = (a.E + 31) / 32;
  const int parts = max(1, nt / a.E);
  const int span = (a.E + parts - 1) / parts;
  for (int t = 0; t < a.T; ++t) {
    // (A)
    if (tid == 0) {
      r.bad[0] = r.bad[1] = 0;
      r.bad[2] = float_key(-INFINITY);
    }
    for (int e = tid; e < a.E; e += nt) {
      r.lg[e] = a.logits[(size_t)t * a.E + e];
      r.rank[e] = 0;
      if (t == 0 && table) r.slot[e] = a.slot_of[e];
    }
    __syncthreads();
    // (B)
    for (int i = tid; i < a.E * parts; i += nt) {
      const int e = i % a.E, part = i / a.E;
      const float v = r.lg[e];
      if (i < a.E) {  // part 0 (whole warps while E is a multiple of 32): one atomic per warp
        const unsigned mask = __activemask();
        const int is_bad = isnan(v) || v == INFINITY;
        const int32_t kmax = __reduce_max_sync(mask, is_bad ? float_key(-INFINITY) : float_key(v));
        const int any_bad = __any_sync(mask, is_bad);
        const int ninf = __popc(__ballot_sync(mask, v == -INFINITY));
        if ((threadIdx.x & 31) == __ffs(mask) - 1) {
          if (any_bad) atomicOr(&r.bad[0], 1);
          atomicMax(&r.bad[2], kmax);
          if (ninf) atomicAdd(&r.bad[1], ninf);
        }
      }
      int cnt = 0;
      const int j1 = min(a.E, (part + 1) * span);
      for (int j = part * span; j < j1; ++j) {
        const float u = r.lg[j];
        cnt += (u > v) || (u == v && j < e);
      }
      if (cnt) atomicAdd(&r.rank[e], cnt);
    }
    __syncthreads();
    // (C)
    const bool token_bad = r.bad[0] != 0 || r.bad[1] == a.E;
    const float m = key_float(r.bad[2]);
    for (int base = warp * 32; base < a.E; base += nt) {  // warp-uniform: one slice
      const int e = base + lane;
      float ex = 0.0f;
      if (e < a.E) {
        ex = token_bad ? 0.0f : expf(r.lg[e] - m);
        const int rk = r.rank[e];
        if (rk < a.k) {
          const int q = t * a.k + rk;
          const int id = token_bad ? -1 : e;
          r.ids[q] = id;
          r.exsel[q] = ex;
          blk_of[q] = resolve_report(a, r, id, table, writer);
          if (writer && a.ids_out) a.ids_out[q] = id;
        }
      }
      ex = warp_sum(ex);
      if (lane == 0) r.red[base / 32] = ex;
    }
    __syncthreads();
    if (tid == 0) {
      float s_all = 0.0f;
      for (int i = 0; i < nslices; ++i) s_all += r.red[i];
      r.sall[t] = s_all;
    }
  }
}

// Warp 0 after route_block: w[q] = exp(l - max) / (sum over all E, or over
// the k chosen, in choice order); 0 for a token without a routing.
__device__ __forceinline__ void finish_weights(const DecodeParams& a, const RouteSmem& r, bool writer) {
  __syncwarp();
  for (int q = threadIdx.x; q < a.P; q += 32) {
    const int t = q / a.k;
    float wq = 0.0f;
    if (r.ids[q] >= 0) {
      float den = r.sall[t];
      if (a.renorm) {
        den = 0.0f;
        for (int j = 0; j < a.k; ++j) den += r.exsel[t * a.k + j];
      }
      wq = r.exsel[q] / den;
    }
    r.w[q] = wq;
    if (writer && a.wts_out) a.wts_out[q] = wq;
  }
  __syncwarp();
}

// Shared prologue: barriers, routing (or the given ids), the expert block of
// every pair (resolved once), unusable-id reporting and routed outputs. On
// return blk_of and ids are visible to the whole block; w is complete in
// warp 0 (which forms it when the block routes itself) and becomes visible
// to the other warps at their next barrier with warp 0.
// empty_count: arrivals that free a stage (odd stages: odd_count).
__device__ __forceinline__ void init_bars(const DecodeParams& a, uint64_t* full, uint64_t* empty,
                                          int empty_count, int odd_count) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], (s & 1) ? odd_count : empty_count);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
}

// Barriers (init_bars, by the caller, before any other thread uses them),
// routing or the given ids, the expert block of every pair; ends with a
// block barrier.
__device__ __forceinline__ void prologue(const DecodeParams& a, uint8_t* sm, const uint8_t** blk_of,
                                         bool writer) {
  const RouteSmem r = route_smem(a, sm);
  const bool table = a.E <= kSlotTableMax;
  if (a.logits) {
    route_block(a, r, blk_of, table, writer);
    if (threadIdx.x < 32) finish_weights(a, r, writer);
  } else {
    for (int p = threadIdx.x; p < a.P; p += blockDim.x) {
      r.ids[p] = a.ids[p];
      r.w[p] = a.wts[p];
    }
    if (table)
      for (int e = threadIdx.x; e < a.E; e += blockDim.x) r.slot[e] = a.slot_of[e];
    __syncthreads();
    for (int p = threadIdx.x; p < a.P; p += blockDim.x) {
      blk_of[p] = resolve_report(a, r, r.ids[p], table, writer);
      if (writer) {
        if (a.ids_out) a.ids_out[p] = r.ids[p];
        if (a.wts_out) a.wts_out[p] = r.w[p];
      }
    }
    __syncthreads();
  }
}

// Producer loop of one kernel: for each pair, wait for the stage to be free,
// then request the block's rows [r0, r1) of the expert's section starting at
// `section` (row stride row_bytes) -- one contiguous bulk copy.
__device__ __forceinline__ void produce(const DecodeParams& a, uint8_t* sm, uint64_t* full,
                                        uint64_t* empty, const uint8_t* const* blk_of, int r0,
                                        int r1, unsigned long long section, uint32_t row_bytes) {
  const uint32_t bytes = (uint32_t)(r1 - r0) * row_bytes;
  for (int p = 0; p < a.P; ++p) {
    const int s = p % a.stages;
    if (p >= a.stages && !mbar_wait(&empty[s], ((p / a.stages) - 1) & 1)) atomicOr(a.flags, 4);
    const uint8_t* blk = blk_of[p];
    if (!blk || bytes == 0) {
      mbar_arrive_expect_tx(&full[s], 0);
      continue;
    }
    mbar_arrive_expect_tx(&full[s], bytes);
    bulk_g2s(sm + (size_t)s * a.st.bytes, blk + section + (size_t)r0 * row_bytes, bytes, &full[s]);
  }
}

// The activations of the current token in shared memory as the scaled pairs
// of dot16_scaled, 64 bytes per 32-element chunk; piece i (16 bytes) of chunk
// cc sits at slot (i + cc/2) % 4 so that the 8 lanes of a quarter-warp, which
// read chunks cc..cc+7, hit 8 different bank groups. Per chunk: xsum = sum of
// the (unscaled) FP16 values, xback = 2^(24-s).
__device__ __forceinline__ int xslot(int cc, int i) { return cc * 4 + ((i + (cc >> 1)) & 3); }

__device__ __forceinline__ void stage_x(const __half* __restrict__ src, int H, uint4* xs4, float* xsum,
                                        float* xback, int tid, int nthreads) {
  for (int cc = tid; cc < H / 32; cc += nthreads) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 raw = *reinterpret_cast<const uint4*>(src + 32 * cc + 8 * i);
      const __half* e = reinterpret_cast<const __half*>(&raw);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[8 * i + j] = __half2float(e[j]);
    }
    float sum = 0.0f, amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      sum += v[j];
      amax = fmaxf(amax, fabsf(v[j]));
    }
    const int sh = chunk_shift(amax);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 o;
      scaled_perm8(v + 8 * i, sh, reinterpret_cast<half2*>(&o));
      xs4[xslot(cc, i)] = o;
    }
    xsum[cc] = sum;
    xback[cc] = pow2f(24 - sh);
  }
}

// Gate and up sums of one row for one lane (before the warp sum):
// s * (sum_c q_c x_c - z * sum_c x_c) over the lane's chunks cc = lane + 32 it.
// gq / xo: the lane's group index and activation slots per chunk, computed
// once per kernel.
template <int NC>
__device__ __forceinline__ void gate_up_row(const uint8_t* row, const BlockOffsets& off, int nch,
                                            int lane, const int* gq, const int* xo, const uint4* xs4,
                                            const float* xsum, const float* xback, float& ag, float& au) {
  const uint2* sz = reinterpret_cast<const uint2*>(row + off.gu_sz);  // quads per group
#pragma unroll
  for (int it = 0; it < NC; ++it) {
    const int cc = lane + 32 * it;
    if (cc < nch) {
      const uint4 wg = *reinterpret_cast<const uint4*>(row + off.gu_q_gate + 16 * cc);
      const uint4 wu = *reinterpret_cast<const uint4*>(row + off.gu_q_up + 16 * cc);
      const uint2 q = sz[gq[it]];
      uint4 xv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = xs4[xo[4 * it + i]];
      const half2* xa = reinterpret_cast<const half2*>(&xv[0]);  // pieces 0, 1 are contiguous
      const half2* xb = reinterpret_cast<const half2*>(&xv[2]);
      const float back = xback[cc];
      const float dg = (dot16_scaled(wg.x, wg.y, xa) + dot16_scaled(wg.z, wg.w, xb)) * back;
      const float du = (dot16_scaled(wu.x, wu.y, xa) + dot16_scaled(wu.z, wu.w, xb)) * back;
      const float2 sgz = __half22float2(u32_as_h2(q.x));  // (s_gate, z_gate)
      const float2 suz = __half22float2(u32_as_h2(q.y));  // (s_up, z_up)
      const float xsm = xsum[cc];
      ag += sgz.x * (dg - sgz.y * xsm);
      au += suz.x * (du - suz.y * xsm);
    }
  }
}

// Two rows (same row index of two pairs of one token) at once.
template <int NC>
__device__ __forceinline__ void gate_up_row2(const uint8_t* ra, const uint8_t* rb, const BlockOffsets& off,
                                             int nch, int lane, const int* gq, const int* xo, const uint4* xs4,
                                             const float* xsum, const float* xback, float& aga, float& aua,
                                             float& agb, float& aub) {
  const uint2* sza = reinterpret_cast<const uint2*>(ra + off.gu_sz);
  const uint2* szb = reinterpret_cast<const uint2*>(rb + off.gu_sz);
#pragma unroll
  for (int it = 0; it < NC; ++it) {
    const int cc = lane + 32 * it;
    if (cc < nch) {
      const uint4 wga = *reinterpret_cast<const uint4*>(ra + off.gu_q_gate + 16 * cc);
      const uint4 wua = *reinterpret_cast<const uint4*>(ra + off.gu_q_up + 16 * cc);
      const uint4 wgb = *reinterpret_cast<const uint4*>(rb + off.gu_q_gate + 16 * cc);
      const uint4 wub = *reinterpret_cast<const uint4*>(rb + off.gu_q_up + 16 * cc);
      const uint2 qa = sza[gq[it]];
      const uint2 qb = szb[gq[it]];
      uint4 xv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = xs4[xo[4 * it + i]];
      const half2* xa = reinterpret_cast<const half2*>(&xv[0]);
      const half2* xb = reinterpret_cast<const half2*>(&xv[2]);
      const float back = xback[cc];
      const float xsm = xsum[cc];
      const float dga = (dot16_scaled(wga.x, wga.y, xa) + dot16_scaled(wga.z, wga.w, xb)) * back;
      const float dua = (dot16_scaled(wua.x, wua.y, xa) + dot16_scaled(wua.z, wua.w, xb)) * back;
      const float dgb = (dot16_scaled(wgb.x, wgb.y, xa) + dot16_scaled(wgb.z, wgb.w, xb)) * back;
      const float dub = (dot16_scaled(wub.x, wub.y, xa) + dot16_scaled(wub.z, wub.w, xb)) * back;
      const float2 sga = __half22float2(u32_as_h2(qa.x)), sua = __half22float2(u32_as_h2(qa.y));
      const float2 sgb = __half22float2(u32_as_h2(qb.x)), sub = __half22float2(u32_as_h2(qb.y));
      aga += sga.x * (dga - sga.y * xsm);
      aua += sua.x * (dua - sua.y * xsm);
      agb += sgb.x * (dgb - sgb.y * xsm);
      aub += sub.x * (dub - sub.y * xsm);
    }
  }
}

// ---- kernel 1: gate/up dequant-GEMV + SwiGLU -------------------------------
// Stage: the block's gate/up rows [R][gu_row] (codes, scales and zeros of
// both projections per row). With a stage per pair (P <= S), the work units
// of a token are (couple, row): row r of pairs 2c and 2c + 1, computed
// together by one warp (shared activation loads, two independent chains);
// warp w takes units w, w + 15, ... Otherwise each iteration covers
// kPairsPerIter pairs of one token: warp w takes row w % 8 (+8, ...) of pair
// p + w / 8, and the sub-group releases the stage.
template <int NC>
__global__ void __launch_bounds__(kGateThreads, 2) decode_gateup_kernel(const DecodeParams a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int n0 = (int)(((long long)c * a.I) / a.G), n1 = (int)(((long long)(c + 1) * a.I) / a.G);
  const int rows = n1 - n0;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + a.bar_off);
  uint64_t* empty = full + kMaxStages;
  const uint8_t** blk_of = reinterpret_cast<const uint8_t**>(sm + a.blk_off);
  uint4* xs4 = reinterpret_cast<uint4*>(sm + a.part_off);                    // [H/32][4]
  float* xsum = reinterpret_cast<float*>(sm + a.part_off + (size_t)a.H * 2);  // [H/32]
  float* xback = xsum + a.H / 32;                                             // [H/32]
  // Independent of earlier kernels: before the wait. Every warp of the
  // sub-group that drains a stage arrives on its empty barrier.
  init_bars(a, full, empty, kSub0, kGateWarps - kSub0);
  griddep_wait();                // logits / ids and x come from earlier kernels
  prologue(a, sm, blk_of, c == 0);
  griddep_launch_dependents();  // the down kernel may start its prefetch
  if (warp == kGateWarps) {
    if (lane == 0) produce(a, sm, full, empty, blk_of, n0, n1, 0ull, a.off.gu_row);
    return;
  }
  const int nch = a.H / 32;
  int gq[NC], xo[4 * NC];
#pragma unroll
  for (int it = 0; it < NC; ++it) {
    const int cc = lane + 32 * it;
    gq[it] = (32 * cc) / a.g;
#pragma unroll
    for (int i = 0; i < 4; ++i) xo[4 * it + i] = xslot(cc, i);
  }
  if (a.P <= a.stages) {
    int cur_t = -1;
    for (int p0 = 0; p0 < a.P; p0 += a.k) {
      const int t = p0 / a.k;
      if (t != cur_t) {
        asm volatile("bar.sync 1, %0;" ::"n"(kGateWarps * 32) : "memory");  // previous x no longer read
        stage_x(a.x + (size_t)t * a.H, a.H, xs4, xsum, xback, threadIdx.x, kGateWarps * 32);
        asm volatile("bar.sync 1, %0;" ::"n"(kGateWarps * 32) : "memory");
        cur_t = t;
      }
      const int couples = (a.k + 1) / 2;
      for (int u = warp; u < couples * rows; u += kGateWarps) {
        const int cpl = u / rows, r = u - cpl * rows;
        const int qa = p0 + 2 * cpl, qb = qa + 1;
        const bool two = 2 * cpl + 1 < a.k;
        const int sa = qa % a.stages, sb = qb % a.stages;
        if (!mbar_wait(&full[sa], (qa / a.stages) & 1) && lane == 0) atomicOr(a.flags, 4);
        if (two && !mbar_wait(&full[sb], (qb / a.stages) & 1) && lane == 0) atomicOr(a.flags, 4);
        const uint8_t* ba = blk_of[qa];
        const uint8_t* bb = two ? blk_of[qb] : nullptr;
        const uint8_t* ra = sm + (size_t)sa * a.st.bytes + (size_t)r * a.off.gu_row;
        const uint8_t* rb = sm + (size_t)sb * a.st.bytes + (size_t)r * a.off.gu_row;
        float aga = 0.0f, aua = 0.0f, agb = 0.0f, aub = 0.0f;
        if (ba && bb) {
          gate_up_row2<NC>(ra, rb, a.off, nch, lane, gq, xo, xs4, xsum, xback, aga, aua, agb, aub);
        } else {
          if (ba) gate_up_row<NC>(ra, a.off, nch, lane, gq, xo, xs4, xsum, xback, aga, aua);
          if (bb) gate_up_row<NC>(rb, a.off, nch, lane, gq, xo, xs4, xsum, xback, agb, aub);
        }
        // Warp sums of the four values by a reduce-scatter butterfly (7
        // shuffles instead of 20): after the exchanges at distance 16 and 8,
        // lanes with bit 4 clear hold pair a's sums and set pair b's; bit 3
        // clear the gate sum, set the up sum; the last three levels finish
        // each sum within its group of eight lanes.
        const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1;
        const float k0 = b4 ? agb : aga, k1 = b4 ? aub : aua;
        const float w0 = k0 + __shfl_xor_sync(0xffffffffu, b4 ? aga : agb, 16);
        const float w1 = k1 + __shfl_xor_sync(0xffffffffu, b4 ? aua : aub, 16);
        float v = (b3 ? w1 : w0) + __shfl_xor_sync(0xffffffffu, b3 ? w0 : w1, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        const float up = __shfl_xor_sync(0xffffffffu, v, 8);  // lanes 0 and 16: the up sum
        if (lane == 0) a.hbuf[(size_t)qa * a.I + n0 + r] = __float2half_rn(ba ? silu_f(v) * up : 0.0f);
        if (lane == 16 && two) a.hbuf[(size_t)qb * a.I + n0 + r] = __float2half_rn(bb ? silu_f(v) * up : 0.0f);
      }
    }
    return;
  }
  const int sub = warp < kSub0 ? 0 : 1;                  // pair offset in the iteration
  const int wr = warp - sub * kSub0;                     // row lane within the sub-group
  const int nsub = sub ? kGateWarps - kSub0 : kSub0;     // warps of the sub-group
  int cur_t = -1;
  for (int p = 0; p < a.P;) {
    const int t = p / a.k;
    int np = 1;  // pairs of token t in this iteration
    while (np < kPairsPerIter && p + np < a.P && (p + np) / a.k == t) ++np;
    if (t != cur_t) {
      asm volatile("bar.sync 1, %0;" ::"n"(kGateWarps * 32) : "memory");  // previous x no longer read
      stage_x(a.x + (size_t)t * a.H, a.H, xs4, xsum, xback, threadIdx.x, kGateWarps * 32);
      asm volatile("bar.sync 1, %0;" ::"n"(kGateWarps * 32) : "memory");
      cur_t = t;
    }
    const int q = (p & 1) == sub ? p : p + 1;  // this sub-group's pair, if any
    if (q < p + np) {
      const int s = q % a.stages;
      if (!mbar_wait(&full[s], (q / a.stages) & 1) && lane == 0) atomicOr(a.flags, 4);
      const uint8_t* blk = blk_of[q];
      const uint8_t* stg = sm + (size_t)s * a.st.bytes;
      for (int r = wr; r < rows; r += nsub) {
        float ag = 0.0f, au = 0.0f;
        if (blk) gate_up_row<NC>(stg + (size_t)r * a.off.gu_row, a.off, nch, lane, gq, xo, xs4, xsum, xback, ag, au);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          ag += __shfl_xor_sync(0xffffffffu, ag, o);
          au += __shfl_xor_sync(0xffffffffu, au, o);
        }
        if (lane == 0) a.hbuf[(size_t)q * a.I + n0 + r] = __float2half_rn(blk ? silu_f(ag) * au : 0.0f);
      }
      // This warp has finished reading the stage (no sub-group barrier: the
      // stage is free once every warp of the sub-group has arrived).
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    p += np;
  }
}

// ---- kernel 2: down dequant-GEMV + top-k weighted combine -------------------
// Stage: the block's down rows [R][d_row] (codes, then scale/zero pairs).
// Warp w computes the block's rows for pairs w, w+8, ...
template <int kMaxHChunks>
__global__ void __launch_bounds__(kThreads, 3) decode_down_kernel(const DecodeParams a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int m0 = (int)(((long long)c * a.H) / a.G), m1 = (int)(((long long)(c + 1) * a.H) / a.G);
  const int rows = m1 - m0;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + a.bar_off);
  uint64_t* empty = full + kMaxStages;
  const uint8_t** blk_of = reinterpret_cast<const uint8_t**>(sm + a.blk_off);
  float* part = reinterpret_cast<float*>(sm + a.part_off);  // [P][rows]
  // Inputs the prefetch needs (logits or ids, slot_of, the pool) are final:
  // the gate/up kernel passed its own griddepcontrol.wait before signalling.
  init_bars(a, full, empty, 1, 1);
  prologue(a, sm, blk_of, false);
  const RouteSmem rt = route_smem(a, sm);
  if (warp == kWarps) {
    if (lane == 0) produce(a, sm, full, empty, blk_of, m0, m1, a.off.d_offset, a.off.d_row);
    griddep_launch_dependents();
    return;
  }
  griddep_wait();  // h of every pair is complete and visible
  griddep_launch_dependents();
  const int nch = a.I / 32;
  int gix[kMaxHChunks];
#pragma unroll
  for (int it = 0; it < kMaxHChunks; ++it) gix[it] = (32 * (lane + 32 * it)) / a.g;
  for (int q = 0; q < a.P; ++q) {
    const int s = q % a.stages;
    if (s % kWarps != warp) continue;
    const uint8_t* blk = blk_of[q];
    if (!mbar_wait(&full[s], (q / a.stages) & 1) && lane == 0) atomicOr(a.flags, 4);
    if (blk && rows > 0) {
      half2 hr[kMaxHChunks][16];
      float hsum[kMaxHChunks], hback[kMaxHChunks];
#pragma unroll
      for (int it = 0; it < kMaxHChunks; ++it) {
        const int cc = lane + 32 * it;
        if (cc < nch) hsum[it] = load_scaled_chunk(a.hbuf + (size_t)q * a.I + 32 * cc, hr[it], hback[it]);
      }
      const uint8_t* stg = sm + (size_t)s * a.st.bytes;
      for (int r0 = 0; r0 < rows; r0 += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          v[u] = 0.0f;
          const int r = r0 + u;
          if (r < rows) {
            const uint8_t* row = stg + (size_t)r * a.off.d_row;
            const uint32_t* sz = reinterpret_cast<const uint32_t*>(row + a.off.d_sz);  // pairs per group
#pragma unroll
            for (int it = 0; it < kMaxHChunks; ++it) {
              const int cc = lane + 32 * it;
              if (cc < nch) {
                const uint4 w = *reinterpret_cast<const uint4*>(row + a.off.d_q + 16 * cc);
                const float2 s2 = __half22float2(u32_as_h2(sz[gix[it]]));  // (s, z)
                const float d = (dot16_scaled(w.x, w.y, hr[it]) + dot16_scaled(w.z, w.w, hr[it] + 8)) * hback[it];
                v[u] += s2.x * (d - s2.y * hsum[it]);
              }
            }
          }
        }
        // Warp sums of the 8 rows by a reduce-scatter butterfly (9 shuffles
        // instead of 40): each exchange keeps half of the remaining rows, so
        // after distances 16, 8 and 4 a lane holds one row (bits 4, 3, 2 of
        // the lane pick it) and distances 2 and 1 finish its sum.
        const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
        float w4[4], w2[2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float keep = b4 ? v[4 + i] : v[i], send = b4 ? v[i] : v[4 + i];
          w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float keep = b3 ? w4[2 + i] : w4[i], send = b3 ? w4[i] : w4[2 + i];
          w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        float w1 = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
        w1 += __shfl_xor_sync(0xffffffffu, w1, 2);
        w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
        const int u = 4 * b4 + 2 * b3 + b2;  // the row whose total this lane holds
        if ((lane & 3) == 0 && r0 + u < rows) part[q * rows + r0 + u] = w1;
      }
    } else if (lane == 0) {
      for (int r = 0; r < rows; ++r) part[q * rows + r] = 0.0f;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");  // compute warps only
  // y[t][m0 + r] = sum_j w[t][j] * part[t*k + j][r] (+ y_shared), in j order.
  for (int i = threadIdx.x; i < a.T * rows; i += kWarps * 32) {
    const int t = i / rows, r = i - t * rows;
    float v = 0.0f;
    for (int j = 0; j < a.k; ++j) {
      const int q = t * a.k + j;
      v += rt.w[q] * part[q * rows + r];
    }
    if (a.y_shared) v += __half2float(a.y_shared[(size_t)t * a.H + m0 + r]);
    a.y[(size_t)t * a.H + m0 + r] = __float2half_rn(v);
  }
}

int g_num_sms = 0;

template <typename K>
cudaError_t launch(K kern, const DecodeParams& a, size_t smem, int threads, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // Ask for the full shared-memory carveout so that a block of the other
  // decode kernel fits on the same SM (the down kernel prefetches while the
  // gate/up kernel runs).
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.G);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// Carve-up: stages | part | route | barriers | block table. Returns total bytes.
size_t carve(DecodeParams& a, size_t part, size_t budget) {
  const size_t route = route_smem_bytes(a.P, a.T, a.E, a.logits != nullptr);
  const size_t tail = ((part + 15) & ~(size_t)15) + ((route + 15) & ~(size_t)15) + 2 * kMaxStages * 8 +
                      (size_t)a.P * 8 + 64;
  if (tail + 2 * (size_t)a.st.bytes > budget) return 0;
  a.stages = (int)std::min<size_t>(kMaxStages, (budget - tail) / a.st.bytes) & ~1;  // even
  size_t o = (size_t)a.stages * a.st.bytes;
  a.part_off = (uint32_t)o;
  o = (o + part + 15) & ~(size_t)15;
  a.route_off = (uint32_t)o;
  o = (o + route + 15) & ~(size_t)15;
  a.bar_off = (uint32_t)o;
  o += 2 * kMaxStages * 8;
  a.blk_off = (uint32_t)o;
  o += (size_t)a.P * 8;
  return o;
}

}  // namespace

size_t fused_workspace_bytes(int H, int I, int T, int k) {
  (void)H;
  return ws_scratch_offset(T * k) + (size_t)T * k * I * 2;
}

// Shared-memory budgets keep one block of each kernel resident on an SM at
// the same time (the down kernel prefetches while the gate/up kernel runs).
constexpr size_t kGateupBudget = 140 * 1024;
constexpr size_t kDownBudget = 80 * 1024;

int fused_forward_routed(const ForwardArgs& fa, const float* logits, int renorm, int32_t* ids_out,
                         float* wts_out) {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  }
  const int xc = (fa.H + 1023) / 1024, hc = (fa.I + 1023) / 1024;
  if (xc > 4 || hc > 2) return fail(MOE_ERR_UNSUPPORTED, "streamed decode: H <= 4096 and I <= 2048 only");
  DecodeParams a;
  a.H = fa.H; a.I = fa.I; a.g = fa.g; a.T = fa.T; a.k = fa.k; a.E = fa.E; a.n_slots = fa.n_slots;
  a.P = fa.T * fa.k;
  a.G = g_num_sms;
  a.x = fa.x; a.ids = fa.ids; a.wts = fa.weights; a.pool = fa.pool; a.block_bytes = fa.block_bytes;
  a.logits = logits; a.renorm = renorm; a.ids_out = ids_out; a.wts_out = wts_out;
  a.off = fa.off; a.slot_of = fa.slot_of; a.y_shared = fa.y_shared; a.y = fa.y;
  uint8_t* ws = static_cast<uint8_t*>(fa.ws);
  a.flags = reinterpret_cast<int32_t*>(ws);
  a.hbuf = reinterpret_cast<__half*>(ws + ws_scratch_offset(a.P));
  const int rgu = (a.I + a.G - 1) / a.G, rdn = (a.H + a.G - 1) / a.G;

  DecodeParams ag = a;
  ag.st = stage_of(rgu, a.off.gu_row);
  const size_t smem_g = carve(ag, (size_t)a.H * 2 + (size_t)(a.H / 32) * 8, kGateupBudget);
  DecodeParams ad = a;
  ad.st = stage_of(rdn, a.off.d_row);
  const size_t smem_d = carve(ad, (size_t)a.P * rdn * 4, kDownBudget);
  if (!smem_g || !smem_d) return fail(MOE_ERR_UNSUPPORTED, "streamed decode: shapes exceed shared memory");
  cudaError_t e;
  if (xc <= 2) e = launch(decode_gateup_kernel<2>, ag, smem_g, kGateThreads, fa.stream);
  else e = launch(decode_gateup_kernel<4>, ag, smem_g, kGateThreads, fa.stream);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "decode gate/up launch: %s", cudaGetErrorString(e));
  if (hc <= 1) e = launch(decode_down_kernel<1>, ad, smem_d, kThreads, fa.stream);
  else e = launch(decode_down_kernel<2>, ad, smem_d, kThreads, fa.stream);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "decode down launch: %s", cudaGetErrorString(e));
  return MOE_OK;
}

int fused_forward(const ForwardArgs& fa) { return fused_forward_routed(fa, nullptr, 0, nullptr, nullptr); }

}  // namespace moe
