// Decode path: one streaming kernel per routed layer.
//
// "Horizon RunMap -- Prévia Técnica", "03 / Arquitetura" and
// "08 / Comportamento do modelo": the expert kernel reads compact INT4 codes
// and FP16 scales, converts them inside the kernel (no expanded expert is
// kept) and works with FP16 activations and FP32 accumulation.
//
// One block per SM (G blocks). Block c owns gate/up rows n in
// [c*I/G, (c+1)*I/G) and output rows m in [c*H/G, (c+1)*H/G) of every expert
// the step uses; a "unit" is one distinct expert of the call, read once
// however many tokens chose it. Per call:
//   1. Routing (moe_layer_forward) inside every block with moe_route's
//      selection (top-k by (logit desc, index asc)) and softmax arithmetic,
//      so all blocks hold identical ids and weights; the activations are
//      staged in shared memory meanwhile.
//   2. A producer lane streams the block's rows of every unit into shared-
//      memory stages with bulk async copies (cp.async.bulk, completion
//      counted on mbarriers).
//   3. Compute warps form h = silu(W_g x) * (W_u x) for their rows of every
//      pair of a unit and round it to FP16 (the explicit rounding point)
//      into the workspace.
//   4. Once every block's h rows of a unit are out, the down rows of the
//      unit form the block's output rows of W_d h per pair.
//   5. y[t][m] = sum_j w[t][j] * (W_d h[t*k+j])[m] (+ y_shared), the k pairs
//      of a token combined in j order (deterministic).
// One routed token (the decode step proper): the whole block routes the
// token, every pick has its own stages, each unit is released on its own
// global counter and an exchange warp copies each unit's complete h into
// shared memory as soon as every block has released it. Several tokens: one
// ring of stages filled in order (every unit's gate/up rows, then the down
// rows of groups of units), work items dealt round-robin to the compute
// warps, and one grid barrier between the gate/up and the down items.
// The last block to finish resets the counters, so the workspace is reusable
// by the next call on the same stream. All waits are bounded; on expiry bit 2
// of the workspace error word is set and the block stops waiting.
#include <algorithm>
#include <climits>
#include <mutex>

#include "common.h"
#include "device.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kWarps = 16;                    // compute warps
constexpr int kThreads = (kWarps + 2) * 32;   // + producer warp + exchange warp
constexpr int kProducer = kWarps;
constexpr int kExchange = kWarps + 1;
constexpr int kMaxT = 16;                     // tokens per call
constexpr int kMaxP = 256;                    // (token, choice) pairs per call
constexpr int kMaxE = 1024;                   // experts (in-block tables)
static_assert(kMaxE <= 2 * kThreads, "the batched unit scan takes two experts per thread");
constexpr int kMaxRing = 32;                  // stages per ring
constexpr int kMaxFastK = 16;                 // one routed token: picks that each get their own stages
constexpr int kDownRows = 8;                  // rows per down work item
constexpr unsigned long long kWaitNs = 1000000000ull;  // bound of one mbarrier wait: ~1 s of global time
constexpr unsigned kIdleTries = 16000000;     // ~1 s of idle producer loop iterations
constexpr unsigned kSpinTries = 2000000;      // ~1 s of counter polls (one L2 round trip each)
constexpr int kCntBase = 64;                  // workspace word of unit counter 0

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
// try_wait without a suspend-time hint: the thread waits at most a short,
// hardware-defined window for the phase (a 20 us hint measured 0.7 % slower
// at the OLMoE decode shape: the hand-offs of one layer are short waits).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long v;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(v));
  return v;
}
// Bounded wait for a phase (about kWaitNs), no abort check: copies landing
// before a block exits.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  #pragma unroll 1
  while (global_ns() - t0 < kWaitNs)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// Non-blocking test of a phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__host__ __device__ inline uint32_t align16(uint32_t v) { return (v + 15u) & ~15u; }

// 32 FP16 values (64 bytes, read through L2, or from shared memory when
// SMEM) as the scaled pairs of dot16_scaled; returns their sum, and
// 2^(24-s) in back.
template <bool SMEM>
__device__ __forceinline__ float load_scaled_chunk(const __half* src, half2 (&xp)[16], float& back) {
  float v[32];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 r;
    if constexpr (SMEM) {
      r = *reinterpret_cast<const uint4*>(src + 8 * q);
    } else {
      asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(src + 8 * q) : "memory");
    }
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

struct StreamParams {
  const __half* x;
  const float* logits;  // [T][E] when the kernel routes itself, else NULL
  int renorm;
  const int32_t* ids;   // [T][k] given ids (logits == NULL)
  const float* wts;     // [T][k] given weights (logits == NULL)
  int32_t* ids_out;     // routing written by block 0 (nullable)
  float* wts_out;
  const uint8_t* pool;
  unsigned long long block_bytes;
  BlockOffsets off;
  const int32_t* slot_of;
  const __half* y_shared;
  __half* y;
  int32_t* ws;          // workspace words: [0] error, [1] done, [kCntBase + u] unit counters
  __half* hbuf;         // workspace: h [P][I]
  int H, I, g, T, k, E, n_slots, P, G;
  int Sg, Sd;           // one token: stages of the gate/up and down rings; batched: Sg stages, Sd = 0
  uint32_t sg, sd;      // one token: bytes of a stage of each ring; batched: stage bytes, one unit's down rows
  int dpack;            // batched: units whose down rows share a stage
  int rgu, rdn;         // largest row counts of a block
  int fast1;            // one token routed in the block, every unit with its own stages
  // shared-memory carve-up (byte offsets)
  uint32_t o_ring_d, o_x, o_part, o_hst, o_hsm, o_small, o_bar, smem;
};

// Small per-block tables (in shared memory at o_small).
struct Tables {
  const uint8_t** blk;  // [P] expert block of each unit
  int32_t* ids;         // [P]
  float* w;             // [P]
  int32_t* punit;       // [P] unit of each pair, -1 if it contributes nothing
  int32_t* uexp;        // [P] expert of each unit
  int32_t* uoff;        // [P+1] first sorted pair of each unit
  int32_t* upairs;      // [P] pairs sorted by unit
  int32_t* udone;       // [P] one token: gate/up items finished per unit (this block)
  int32_t* fdone;       // [2P] batched: items finished per ring fill
  int32_t* ecnt;        // [E] pairs per expert, then first sorted position
  int32_t* eunit;       // [E] unit of each expert
  int32_t* eslot;       // [E] copy of slot_of
  int32_t* misc;        // [0] units, [1] abort, [5] one token: bit u set when unit u's h copy was issued
};

__host__ __device__ inline size_t tables_bytes(int P, int E) {
  return (size_t)P * 8 + ((size_t)P * 9 + 1 + (size_t)E * 3 + 8) * 4;
}

__device__ __forceinline__ Tables tables_of(const StreamParams& a, uint8_t* sm) {
  Tables t;
  uint8_t* b = sm + a.o_small;
  t.blk = reinterpret_cast<const uint8_t**>(b);
  t.ids = reinterpret_cast<int32_t*>(b + (size_t)a.P * 8);
  t.w = reinterpret_cast<float*>(t.ids + a.P);
  t.punit = reinterpret_cast<int32_t*>(t.w + a.P);
  t.uexp = t.punit + a.P;
  t.uoff = t.uexp + a.P;
  t.upairs = t.uoff + a.P + 1;
  t.udone = t.upairs + a.P;
  t.fdone = t.udone + a.P;
  t.ecnt = t.fdone + 2 * a.P;
  t.eunit = t.ecnt + a.E;
  t.eslot = t.eunit + a.E;
  t.misc = t.eslot + a.E;
  return t;
}

// Bounded wait on an mbarrier phase; gives up at once when the block has
// already aborted. Returns false (and marks the abort) on expiry.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int32_t* abort_flag,
                                           int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  #pragma unroll 1
  do {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  } while (global_ns() - t0 < kWaitNs);
  *abort_flag = 1;
  atomicOr(err, 4);
  return false;
}


// The activations of a token in shared memory as the scaled pairs of
// dot16_scaled, 64 bytes per 32-element chunk; piece i (16 bytes) of chunk
// cc sits at slot (i + cc/2) % 4 so that the 8 lanes of a quarter-warp, which
// read chunks cc..cc+7, hit 8 different bank groups. Per chunk: xsum = sum of
// the (unscaled) FP16 values, xback = 2^(24-s).
__device__ __forceinline__ int xslot(int cc, int i) { return cc * 4 + ((i + (cc >> 1)) & 3); }

__device__ __forceinline__ void stage_x_chunk(const __half* __restrict__ src, uint4* xs4, float* xsum,
                                              float* xback, int cc) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 raw = __ldcg(reinterpret_cast<const uint4*>(src + 32 * cc + 8 * i));
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

// Gate and up sums of up to kGateRows rows (same pair) for one lane, before
// the warp sum: s * (sum_c q_c x_c - z * sum_c x_c) over the lane's chunks
// cc = lane + 32 it. The activation chunk is loaded once for all rows; the
// rows' dot products are independent chains. acc = (g0, u0, g1, u1, ...).
constexpr int kGateRows = 4;  // rows per gate/up work item (at most)
constexpr int kFastRows = 4;  // one routed token: rows per gate/up work item
template <int NC>
__device__ __forceinline__ void gate_up_rows(const uint8_t* row0, int nrows, const BlockOffsets& off, int nch,
                                             int lane, const int* gq, const uint4* xs4, const float* xsum,
                                             const float* xback, float (&acc)[2 * kGateRows]) {
#pragma unroll
  for (int it = 0; it < NC; ++it) {
    const int cc = lane + 32 * it;
    if (cc < nch) {
      uint4 xv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = xs4[xslot(cc, i)];
      const half2* xa = reinterpret_cast<const half2*>(&xv[0]);  // pieces 0, 1 are contiguous
      const half2* xb = reinterpret_cast<const half2*>(&xv[2]);
      const float back = xback[cc], xsm = xsum[cc];
#pragma unroll
      for (int rr = 0; rr < kGateRows; ++rr) {
        if (rr < nrows) {
          const uint8_t* r = row0 + (size_t)rr * off.gu_row;
          const uint4 wg = *reinterpret_cast<const uint4*>(r + off.gu_q_gate + 16 * cc);
          const uint4 wu = *reinterpret_cast<const uint4*>(r + off.gu_q_up + 16 * cc);
          const uint2 q = reinterpret_cast<const uint2*>(r + off.gu_sz)[gq[it]];
          const float dg = (dot16_scaled(wg.x, wg.y, xa) + dot16_scaled(wg.z, wg.w, xb)) * back;
          const float du = (dot16_scaled(wu.x, wu.y, xa) + dot16_scaled(wu.z, wu.w, xb)) * back;
          const float2 sgz = __half22float2(u32_as_h2(q.x)), suz = __half22float2(u32_as_h2(q.y));
          acc[2 * rr] += sgz.x * (dg - sgz.y * xsm);
          acc[2 * rr + 1] += suz.x * (du - suz.y * xsm);
        }
      }
    }
  }
}

// Warp sums of the 8 values (gate, up of 4 rows) by a reduce-scatter
// butterfly (9 shuffles): after distances 16, 8 and 4 a lane holds value
// 4*b4 + 2*b3 + b2 (lane bits), distances 2 and 1 finish it; lanes with b2
// clear hold a gate sum and take the row's up sum from the lane 4 above.
// Lanes with (lane & 7) == 0 return silu(gate) * up of row 2*b4 + b3.
__device__ __forceinline__ float swiglu_lanes(const float (&acc)[2 * kGateRows], int lane) {
  const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
  float w4[4], w2[2];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float keep = b4 ? acc[4 + q] : acc[q], send = b4 ? acc[q] : acc[4 + q];
    w4[q] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float keep = b3 ? w4[2 + q] : w4[q], send = b3 ? w4[q] : w4[2 + q];
    w2[q] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float v = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  const float up = __shfl_xor_sync(0xffffffffu, v, 4);
  return silu_f(v) * up;
}

__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Named barriers, non-aligned forms: arrivals are counted per thread, so a
// warp may reach them diverged (the .aligned bar.sync / bar.arrive would
// require a converged warp); callers reconverge first all the same.
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("barrier.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barriers (0 is __syncthreads).
constexpr int kBarCompute = 1;  // before the combine: compute warps (and, batched, the producer) wait
constexpr int kBarTables = 2;   // producer arrives with the routing tables, compute warps wait
constexpr int kBarGate = 3;     // batched: the compute warps around the grid barrier
constexpr int kBarPolled = 4;   // exchange warp arrives after its last counter poll, producer waits (64)

// A token's logits in registers (lane l: experts l + 32 j, pads -inf);
// returns false for a token without a routing (NaN/+inf logits, or every
// logit -inf).
template <int NJ>
__device__ __forceinline__ bool load_token_logits(const float* lg, int E, int lane, bool smem, float (&v)[NJ]) {
  bool bad = false;
  int ninf = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? (smem ? lg[e] : __ldcg(lg + e)) : -INFINITY;
    if (e < E) {
      bad |= isnan(v[j]) || v[j] == INFINITY;
      ninf += v[j] == -INFINITY;
    }
  }
  bad = __any_sync(0xffffffffu, bad);
  ninf = __reduce_add_sync(0xffffffffu, ninf);
  return !bad && ninf != E;
}

// The softmax weight of lane r's pick (lane < k), with moe_route's
// arithmetic: sum over all E of exp(logit - max) per lane in j order (pads
// give 0), a butterfly, then the pick's share of all E (or of the k picks).
template <int NJ>
__device__ __forceinline__ float pick_weight(const float (&v)[NJ], int k, int renorm, int lane, float my_v) {
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  float s_all = 0.0f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) s_all += expf(v[j] - m);
  s_all = warp_sum(s_all);
  const float mine = lane < k ? expf(my_v - m) : 0.0f;
  const float s_sel = warp_sum(mine);
  return mine / (renorm ? s_sel : s_all);
}

// Batched routing: warp t routes token t from its logits in shared memory
// (ids -1 and weights 0 for a token without a routing).
template <int NJ>
__device__ void route_token_warp(const StreamParams& a, const Tables& tb, const float* lg, int t) {
  const int lane = threadIdx.x & 31, k = a.k;
  float v[NJ];
  if (!load_token_logits<NJ>(lg, a.E, lane, true, v)) {
    if (lane < k) {
      tb.ids[t * k + lane] = -1;
      tb.w[t * k + lane] = 0.0f;
    }
    return;
  }
  float my_v;
  int my_i;
  warp_topk<NJ>(v, a.E, k, lane, my_v, my_i);
  const float wq = pick_weight<NJ>(v, k, a.renorm, lane, my_v);
  if (lane < k) {
    tb.ids[t * k + lane] = my_i;
    tb.w[t * k + lane] = wq;
  }
}

__device__ void route_tokens_warps(const StreamParams& a, const Tables& tb, const float* lgT) {
  const int warp = threadIdx.x >> 5, nj = (a.E + 31) / 32;
  #pragma unroll 1
  for (int t = warp; t < a.T; t += kThreads / 32) {
    const float* lg = lgT + (size_t)t * a.E;
    if (nj <= 2) route_token_warp<2>(a, tb, lg, t);
    else if (nj <= 4) route_token_warp<4>(a, tb, lg, t);
    else if (nj <= 8) route_token_warp<8>(a, tb, lg, t);
    else if (nj <= 16) route_token_warp<16>(a, tb, lg, t);
    else route_token_warp<32>(a, tb, lg, t);
  }
}

// "Horizon RunMap -- Prévia Técnica", "02 / A solução": the router picks the
// experts of the token (moe_route's definition). One routed token: the
// producer warp routes it on its own (warp_topk) while the other warps
// stage the activations. Lane j < k then resolves pick j's expert block, the
// warp writes the tables the compute warps read (units are the picks in
// choice order; every unit has its own stage in both rings) and releases
// them; lane 0 issues the gate/up copies, lanes the down copies; the
// softmax weights follow (pick_weight) and are released to the combine.
template <int NJ>
__device__ void producer_one_token(const StreamParams& a, const Tables& tb, const float* lgs, uint64_t* full_g,
                                   uint64_t* full_d, uint8_t* ring_g, uint8_t* ring_d, int n0, int rg_rows,
                                   int m0, int rd_rows, bool writer) {
  const int lane = threadIdx.x & 31;
  const int E = a.E, k = a.k;
  const uint32_t gbytes = (uint32_t)rg_rows * a.off.gu_row, dbytes = (uint32_t)rd_rows * a.off.d_row;
  float v[NJ];  // from shared memory (lgs lies in the ring: read before any copy is issued)
  const bool ok = load_token_logits<NJ>(lgs, E, lane, true, v);
  float my_v = 0.0f;
  int my_i = -1;
  if (ok) warp_topk<NJ>(v, E, k, lane, my_v, my_i);
  const uint8_t* blk = nullptr;
  int id = -1;
  if (lane < k) {
    if (ok) {
      id = my_i;
      const int sl = tb.eslot[id];
      blk = (sl >= 0 && sl < a.n_slots) ? a.pool + (size_t)sl * a.block_bytes : nullptr;
      if (!blk && writer) atomicOr(a.ws, 1);
    }
    tb.blk[lane] = blk;
    tb.ids[lane] = id;
    tb.punit[lane] = blk ? lane : -1;
    tb.uoff[lane] = lane;
    tb.upairs[lane] = lane;
    tb.udone[lane] = 0;
    if (writer && a.ids_out) a.ids_out[lane] = id;
  }
  if (lane == 0) {
    tb.misc[0] = ok ? k : 0;
    tb.uoff[k] = k;
  }
  __syncwarp();
  bar_arrive(kBarTables, kThreads);  // releases the tables to the compute warps
  // One lane issues the gate/up copies in choice order, so the stages
  // complete in the order the compute warps drain them (copies issued side by
  // side complete together).
  if (lane == 0) {
#pragma unroll 1
    for (int j = 0; j < k && gbytes; ++j) {
      const uint8_t* b = tb.blk[j];
      if (!b) continue;
      mbar_arrive_expect_tx(&full_g[j], gbytes);
      bulk_g2s(ring_g + (size_t)j * a.sg, b + (size_t)n0 * a.off.gu_row, gbytes, &full_g[j]);
    }
  }
  __syncwarp();
  // The down rows are needed only after the exchange: lane j issues pick j's.
  if (blk && dbytes) {
    mbar_arrive_expect_tx(&full_d[lane], dbytes);
    bulk_g2s(ring_d + (size_t)lane * a.sd, blk + a.off.d_offset + (size_t)m0 * a.off.d_row, dbytes, &full_d[lane]);
  }
  const float wq = ok ? pick_weight<NJ>(v, k, a.renorm, lane, my_v) : 0.0f;
  if (lane < k) {
    tb.w[lane] = wq;
    if (writer && a.wts_out) a.wts_out[lane] = wq;
  }
  __syncwarp();
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// prefetch_one_token (exchange warp, one decode token): lane u watches unit
// u (the k <= 32 units are polled together, one load per round); once every
// block has released it (acquire), the lane copies the unit's complete h into
// shared memory with a bulk copy, after a proxy fence (the h rows were written
// by ordinary stores of other SMs); the copy completes on hfull[u]. Bit u of
// tb.misc[5] is set when unit u's copy was issued.
__device__ void prefetch_one_token(const StreamParams& a, const Tables& tb, __half* hsm, uint64_t* hfull, int U,
                                   int cnt_target, volatile int32_t* abort_flag) {
  const int lane = threadIdx.x & 31;
  int32_t* cnt = a.ws + kCntBase;
  bool pending = lane < U && tb.blk[lane] != nullptr;
  unsigned tries = 0;
#pragma unroll 1
  while (pending) {
    if (ld_acquire_gpu(&cnt[lane]) >= cnt_target) {
      fence_proxy_async_global();
      mbar_arrive_expect_tx(&hfull[lane], (uint32_t)a.I * 2);
      bulk_g2s(hsm + (size_t)lane * a.I, a.hbuf + (size_t)lane * a.I, (uint32_t)a.I * 2, &hfull[lane]);
      atomicOr(&tb.misc[5], 1 << lane);
      pending = false;
    } else if (*abort_flag) {
      pending = false;
    } else if (++tries > kSpinTries) {
      *abort_flag = 1;
      atomicOr(a.ws, 4);
      pending = false;
    }
  }
}

// Down rows [r0, r0 + nrows) (nrows <= kDownRows) of one pair, from the
// stage row `stg` (row r0): part_row[q] = (W_d h)[m0 + r0 + q], the block's
// output rows. h (the pair's FP16 intermediate, I values) is read from shared
// memory (SMEM) or through L2, as the scaled pairs of dot16_scaled.
template <int NCH, bool SMEM>
__device__ __forceinline__ void down_rows(const uint8_t* stg, int nrows, const BlockOffsets& off, const __half* h,
                                          int nchh, int lane, const int* gd, float* part_row) {
  half2 hr[NCH][16];
  float hsum[NCH], hback[NCH];
#pragma unroll
  for (int it = 0; it < NCH; ++it) {
    const int cc = lane + 32 * it;
    if (cc < nchh) hsum[it] = load_scaled_chunk<SMEM>(h + 32 * cc, hr[it], hback[it]);
  }
  float v[kDownRows];
#pragma unroll
  for (int q = 0; q < kDownRows; ++q) {
    v[q] = 0.0f;
    if (q < nrows) {
      const uint8_t* row = stg + (size_t)q * off.d_row;
      const uint32_t* sz = reinterpret_cast<const uint32_t*>(row + off.d_sz);  // pairs per group
#pragma unroll
      for (int it = 0; it < NCH; ++it) {
        const int cc = lane + 32 * it;
        if (cc < nchh) {
          const uint4 w = *reinterpret_cast<const uint4*>(row + off.d_q + 16 * cc);
          const float2 s2 = __half22float2(u32_as_h2(sz[gd[it]]));  // (s, z)
          const float d = (dot16_scaled(w.x, w.y, hr[it]) + dot16_scaled(w.z, w.w, hr[it] + 8)) * hback[it];
          v[q] += s2.x * (d - s2.y * hsum[it]);
        }
      }
    }
  }
  // Warp sums of the 8 rows by a reduce-scatter butterfly (9 shuffles): each
  // exchange keeps half of the remaining rows, so after distances 16, 8 and 4
  // a lane holds one row (lane bits 4, 3, 2 pick it) and distances 2 and 1
  // finish its sum.
  const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
  float w4[4], w2[2];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float keep = b4 ? v[4 + q] : v[q], send = b4 ? v[q] : v[4 + q];
    w4[q] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float keep = b3 ? w4[2 + q] : w4[q], send = b3 ? w4[q] : w4[2 + q];
    w2[q] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float w1 = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
  w1 += __shfl_xor_sync(0xffffffffu, w1, 2);
  w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
  const int q = 4 * b4 + 2 * b3 + b2;  // the row whose total this lane holds
  if ((lane & 3) == 0 && q < nrows) part_row[q] = w1;
}

// 16 FP16 values of h (two 16-byte words read through L2: h was written by
// other SMs).
__device__ __forceinline__ void load_piece(const __half* src, uint4 (&r)[2]) {
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0].x), "=r"(r[0].y), "=r"(r[0].z), "=r"(r[0].w) : "l"(src) : "memory");
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[1].x), "=r"(r[1].y), "=r"(r[1].z), "=r"(r[1].w) : "l"(src + 8) : "memory");
}

// The 16 values of load_piece as the scaled pairs of dot16_scaled (one
// power-of-two scale for the piece); returns their sum, and 2^(24-s) in back.
__device__ __forceinline__ float scale_piece(const uint4 (&r)[2], half2 (&xp)[8], float& back) {
  float v[16];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const __half* e = reinterpret_cast<const __half*>(&r[q]);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[8 * q + i] = __half2float(e[i]);
  }
  float sum = 0.0f, amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    sum += v[i];
    amax = fmaxf(amax, fabsf(v[i]));
  }
  const int sh = chunk_shift(amax);
  scaled_perm8(v, sh, xp);
  scaled_perm8(v + 8, sh, xp + 4);
  back = pow2f(24 - sh);
  return sum;
}

// Batched path: the block's down rows [0, nrows) of one pair, from the
// stage's rows (stg, row 0): part_row[q] = (W_d h)[m0 + q]. Lane l holds h
// pieces pc = l + 32 it (16 values each) as scaled pairs; rows go 8 at a
// time, each row's sum over the pieces finished by the reduce-scatter
// butterfly of down_rows.
template <int NP>
__device__ __forceinline__ void down_pair_rows(const uint8_t* stg, int nrows, const BlockOffsets& off, int npc,
                                               int lane, const int* gp, const half2 (&hr)[NP][8],
                                               const float* hsum, const float* hback, float* part_row) {
  const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
  #pragma unroll 1
  for (int q0 = 0; q0 < nrows; q0 += kDownRows) {
    float v[kDownRows];
#pragma unroll
    for (int q = 0; q < kDownRows; ++q) {
      v[q] = 0.0f;
      if (q0 + q < nrows) {
        const uint8_t* row = stg + (size_t)(q0 + q) * off.d_row;
        const uint32_t* sz = reinterpret_cast<const uint32_t*>(row + off.d_sz);  // (s, z) per group
#pragma unroll
        for (int it = 0; it < NP; ++it) {
          const int pc = lane + 32 * it;
          if (pc < npc) {
            const uint2 w = *reinterpret_cast<const uint2*>(row + off.d_q + 8 * pc);
            const float2 s2 = __half22float2(u32_as_h2(sz[gp[it]]));
            const float d = dot16_scaled(w.x, w.y, hr[it]) * hback[it];
            v[q] += s2.x * (d - s2.y * hsum[it]);
          }
        }
      }
    }
    float w4[4], w2[2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float keep = b4 ? v[4 + q] : v[q], send = b4 ? v[q] : v[4 + q];
      w4[q] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float keep = b3 ? w4[2 + q] : w4[q], send = b3 ? w4[q] : w4[2 + q];
      w2[q] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float w1 = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
    w1 += __shfl_xor_sync(0xffffffffu, w1, 2);
    w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
    const int q = q0 + 4 * b4 + 2 * b3 + b2;
    if ((lane & 3) == 0 && q < nrows) part_row[q] = w1;
  }
}

// Batched path: wait (bounded) until the producer has issued fill `lap` of
// stage s, so that the stage's mbarrier is at that fill's phase.
__device__ __forceinline__ bool wait_fill(const int32_t* fillno, int s, int lap, volatile int32_t* abort_flag,
                                          int32_t* err) {
  unsigned tries = 0;
  #pragma unroll 1
  while (*(const volatile int32_t*)&fillno[s] <= lap) {
    if (*abort_flag) return false;
    if (++tries > kIdleTries) {
      *abort_flag = 1;
      atomicOr(err, 4);
      return false;
    }
  }
  return true;
}

template <int NCX, int NCH, bool FAST>
__global__ void __launch_bounds__(kThreads, 1) decode_stream_kernel(const StreamParams a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int c = blockIdx.x;
  const int n0 = (int)(((long long)c * a.I) / a.G), n1 = (int)(((long long)(c + 1) * a.I) / a.G);
  const int m0 = (int)(((long long)c * a.H) / a.G), m1 = (int)(((long long)(c + 1) * a.H) / a.G);
  const int rg_rows = n1 - n0, rd_rows = m1 - m0;
  constexpr int kRows = FAST ? kFastRows : kGateRows;
  const int ng = (rg_rows + kRows - 1) / kRows;            // gate/up items per unit
  const int nd = (rd_rows + kDownRows - 1) / kDownRows;   // down items per unit
  uint8_t* ring_g = sm;
  uint8_t* ring_d = sm + a.o_ring_d;
  const int nchx = a.H / 32;
  uint4* xs4 = reinterpret_cast<uint4*>(sm + a.o_x);                                // [T][H/32][4]
  float* xsum = reinterpret_cast<float*>(sm + a.o_x + (size_t)a.T * a.H * 2);       // [T][H/32]
  float* xback = xsum + (size_t)a.T * nchx;                                          // [T][H/32]
  float* part = reinterpret_cast<float*>(sm + a.o_part);                            // [P][rdn]
  __half* hst = reinterpret_cast<__half*>(sm + a.o_hst);                            // [P][rgu]
  __half* hsm = reinterpret_cast<__half*>(sm + a.o_hsm);                            // one token: [U][I]
  uint64_t* full_g = reinterpret_cast<uint64_t*>(sm + a.o_bar);
  uint64_t* empty_g = full_g + kMaxRing;
  uint64_t* full_d = empty_g + kMaxRing;
  uint64_t* empty_d = full_d + kMaxRing;
  uint64_t* hfull = empty_d + kMaxRing;  // one token: h of unit u landed in hsm
  // Batched path: fills issued per stage (the producer raises it after each
  // fill), so a consumer of fill n waits on the right phase from any warp.
  int32_t* fillno = reinterpret_cast<int32_t*>(hfull + kMaxRing);
  const Tables tb = tables_of(a, sm);
  volatile int32_t* abort_flag = tb.misc + 1;
  const bool writer = c == 0;
  int32_t* cnt = a.ws + kCntBase;
  const int cnt_target = min(a.I, a.G);  // blocks that own gate/up rows

  if (tid == 0) {
    #pragma unroll 1
    for (int s = 0; s < a.Sg; ++s) {
      mbar_init(&full_g[s], 1);
      mbar_init(&empty_g[s], (FAST && ng > 0) ? ng : 1);  // batched: the fill's last item arrives
    }
    #pragma unroll 1
    for (int s = 0; s < a.Sd; ++s) {
      mbar_init(&full_d[s], 1);
      mbar_init(&empty_d[s], nd > 0 ? nd : 1);
      mbar_init(&hfull[s], 1);
    }
    for (int s = 0; s < kMaxRing; ++s) fillno[s] = 0;
    tb.misc[1] = 0;
    tb.misc[5] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  griddep_wait();  // x, logits / ids and slot_of come from earlier work

  if constexpr (FAST) {
    // ---- one token: the producer warp routes and streams ------------------
    // The token's logits (into the ring, before any copy) and the slot table
    // go to shared memory first, one load per thread.
    float* lgs = reinterpret_cast<float*>(ring_g);
    #pragma unroll 2
    for (int e = tid; e < a.E; e += kThreads) {
      lgs[e] = __ldcg(a.logits + e);
      tb.eslot[e] = __ldcg(a.slot_of + e);
    }
    __syncthreads();
    if (warp == kProducer) {
      const int nj = (a.E + 31) / 32;
      if (nj <= 2) producer_one_token<2>(a, tb, lgs, full_g, full_d, ring_g, ring_d, n0, rg_rows, m0, rd_rows, writer);
      else if (nj <= 8) producer_one_token<8>(a, tb, lgs, full_g, full_d, ring_g, ring_d, n0, rg_rows, m0, rd_rows, writer);
      else if (nj <= 16) producer_one_token<16>(a, tb, lgs, full_g, full_d, ring_g, ring_d, n0, rg_rows, m0, rd_rows, writer);
      else producer_one_token<32>(a, tb, lgs, full_g, full_d, ring_g, ring_d, n0, rg_rows, m0, rd_rows, writer);
      bar_arrive(kBarCompute, kThreads);  // weights ready for the combine
    } else {
      // The other warps stage the activations, then wait for the tables.
      const int i0 = warp < kProducer ? tid : tid - 32;
      #pragma unroll 1
      for (int cc = i0; cc < nchx; cc += kThreads - 32) stage_x_chunk(a.x, xs4, xsum, xback, cc);
      __syncwarp();
      bar_sync(kBarTables, kThreads);
    }
    griddep_launch_dependents();
  } else {
    // ---- batched: logits (or the given ids), slot table, activations -------
    float* lgT = reinterpret_cast<float*>(sm);  // [T][E], routing scratch in the ring (no copy issued yet)
    if (a.logits) {
      const int n = a.T * a.E;
      if ((reinterpret_cast<uintptr_t>(a.logits) & 15) == 0 && (n & 3) == 0) {
        const float4* src = reinterpret_cast<const float4*>(a.logits);
        float4* dst = reinterpret_cast<float4*>(lgT);
        #pragma unroll 4
        for (int i = tid; i < n / 4; i += kThreads) dst[i] = __ldcg(src + i);
      } else {
        #pragma unroll 4
        for (int i = tid; i < n; i += kThreads) lgT[i] = __ldcg(a.logits + i);
      }
    }
    #pragma unroll 1
    for (int e = tid; e < a.E; e += kThreads) {
      tb.ecnt[e] = 0;
      tb.eslot[e] = __ldcg(a.slot_of + e);
    }
    #pragma unroll 1
    for (int q = tid; q < 2 * a.P; q += kThreads) tb.fdone[q] = 0;
    #pragma unroll 2
    for (int i = tid; i < a.T * nchx; i += kThreads) {
      const int t = i / nchx, cc = i - t * nchx;
      stage_x_chunk(a.x + (size_t)t * a.H, xs4 + (size_t)t * nchx * 4, xsum + (size_t)t * nchx,
                    xback + (size_t)t * nchx, cc);
    }
    __syncthreads();
    if (a.logits) {
      route_tokens_warps(a, tb, lgT);
    } else {
      #pragma unroll 1
      for (int p = tid; p < a.P; p += kThreads) {
        tb.ids[p] = __ldcg(a.ids + p);
        tb.w[p] = __ldcg(a.wts + p);
      }
    }
    __syncthreads();
    // Usable pairs, counted per expert; block 0 writes the routing out.
    #pragma unroll 1
    for (int p = tid; p < a.P; p += kThreads) {
      const int e = tb.ids[p];
      if (writer) {
        if (a.ids_out) a.ids_out[p] = e;
        if (a.wts_out) a.wts_out[p] = tb.w[p];
      }
      int u = -1;
      if (e >= 0 && e < a.E) {
        const int s = tb.eslot[e];
        if (s >= 0 && s < a.n_slots) {
          atomicAdd(&tb.ecnt[e], 1);
          u = 0;
        } else if (writer) {
          atomicOr(a.ws, 1);
        }
      } else if (e != -1 && writer) {
        atomicOr(a.ws, 2);
      }
      tb.punit[p] = u;
    }
    __syncthreads();
    // Units: experts with pairs, in ascending id, by a block-wide exclusive
    // scan (thread i takes experts 2i and 2i + 1; E <= 2 * kThreads).
    {
      int32_t* wsum = reinterpret_cast<int32_t*>(sm);  // [2][warps], in the routing scratch (read already)
      constexpr int kW = kThreads / 32;
      const int e0 = 2 * tid;
      const int c0 = e0 < a.E ? tb.ecnt[e0] : 0, c1 = e0 + 1 < a.E ? tb.ecnt[e0 + 1] : 0;
      const int nu = (c0 > 0) + (c1 > 0), np = c0 + c1;
      int su = nu, sp = np;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int vu = __shfl_up_sync(0xffffffffu, su, o), vp = __shfl_up_sync(0xffffffffu, sp, o);
        if (lane >= o) {
          su += vu;
          sp += vp;
        }
      }
      if (lane == 31) {
        wsum[warp] = su;
        wsum[kW + warp] = sp;
      }
      __syncthreads();
      #pragma unroll 1
      for (int w = 0; w < warp; ++w) {
        su += wsum[w];
        sp += wsum[kW + w];
      }
      int u = su - nu, pos = sp - np;
      #pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = e0 + h, n = h ? c1 : c0;
        if (e >= a.E) break;
        tb.eunit[e] = n > 0 ? u : -1;
        if (n > 0) {
          tb.uexp[u] = e;
          tb.uoff[u] = pos;
          tb.blk[u] = a.pool + (size_t)tb.eslot[e] * a.block_bytes;
          tb.ecnt[e] = pos;  // placement cursor
          ++u;
          pos += n;
        }
      }
      if (tid == kThreads - 1) {
        tb.misc[0] = su;
        tb.uoff[su] = sp;
      }
    }
    __syncthreads();
    // Pairs under their unit. Atomic cursors: the order of a unit's pairs
    // changes no result (every pair has its own h and its own down rows).
    #pragma unroll 1
    for (int p = tid; p < a.P; p += kThreads) {
      if (tb.punit[p] < 0) continue;
      const int e = tb.ids[p];
      tb.upairs[atomicAdd(&tb.ecnt[e], 1)] = p | ((p / a.k) << 16);  // pair, and its token above bit 16
      tb.punit[p] = tb.eunit[e];
    }
    __syncthreads();
    griddep_launch_dependents();

    // ---- producer: one ring, fills in order --------------------------------
    // Fill q < Ug is unit q's gate/up rows; fill Ug + j holds the down rows
    // of units j*dpack .. j*dpack + dpack - 1 (their slices side by side).
    // Fill q goes to stage q % S once the stage's previous fill is consumed;
    // the down fills need nothing but a free stage, so they stream while the
    // last gate/up rows are computed and while the blocks meet.
    if (warp == kProducer) {
      const int U = tb.misc[0];
      const int Ug = ng > 0 ? U : 0, Q = Ug + (nd > 0 ? (U + a.dpack - 1) / a.dpack : 0);
      const uint32_t gbytes = (uint32_t)rg_rows * a.off.gu_row, dbytes = (uint32_t)rd_rows * a.off.d_row;
      const int B = min(32, a.Sg);  // fills in one window: distinct stages
      int q = 0;
      // Each round the lanes look at fills q .. q+B-1; the leading run of
      // fills whose stages are free is issued at once, lane i issuing fill
      // q+i (a bulk copy takes a thread a few hundred ns to issue; lanes
      // issue side by side). If fill q's stage is still busy, wait for it.
      #pragma unroll 1
      while (q < Q) {
        const int qq = q + lane, s = qq % a.Sg, lap = qq / a.Sg;
        const bool ready = lane < B && qq < Q && (lap == 0 || mbar_test(&empty_g[s], (lap - 1) & 1));
        const unsigned m = __ballot_sync(0xffffffffu, ready);
        const int n = m == 0xffffffffu ? 32 : __ffs(~m) - 1;
        if (n == 0) {
          const int s0 = q % a.Sg, lap0 = q / a.Sg;
          if (!__all_sync(0xffffffffu, wait_phase(&empty_g[s0], (lap0 - 1) & 1, abort_flag, a.ws))) break;
          continue;
        }
        if (lane < n) {
          uint8_t* dst = ring_g + (size_t)s * a.sg;
          if (qq < Ug) {
            mbar_arrive_expect_tx(&full_g[s], gbytes);
            bulk_g2s(dst, tb.blk[qq] + (size_t)n0 * a.off.gu_row, gbytes, &full_g[s]);
          } else {
            const int u0 = (qq - Ug) * a.dpack, u1 = min(U, u0 + a.dpack);
            mbar_arrive_expect_tx(&full_g[s], (uint32_t)(u1 - u0) * dbytes);
            #pragma unroll 1
            for (int u = u0; u < u1; ++u)
              bulk_g2s(dst + (size_t)(u - u0) * a.sd, tb.blk[u] + a.off.d_offset + (size_t)m0 * a.off.d_row, dbytes,
                       &full_g[s]);
          }
          *(volatile int32_t*)&fillno[s] = lap + 1;
        }
        __syncwarp();
        q += n;
      }
      // Before the block may exit, every copy it issued has landed (bounded):
      // no fill follows the last one of each stage, so its parity is final.
      #pragma unroll 1
      for (int s = lane; s < a.Sg && s < q; s += 32) {
        const int last = s + a.Sg * ((q - 1 - s) / a.Sg);
        mbar_wait_bounded(&full_g[s], (last / a.Sg) & 1);
      }
      __syncwarp();
    }
  }
  const int U = tb.misc[0];

  if (warp == kExchange) {
    // One token: the exchange warp polls the other blocks and copies each
    // unit's complete h into shared memory (the batched path meets the
    // other blocks once, in the compute warps).
    __syncwarp();
    bar_arrive(kBarCompute, kThreads);
    if constexpr (FAST) {
      prefetch_one_token(a, tb, hsm, hfull, U, cnt_target, abort_flag);
      __syncwarp();
      bar_arrive(kBarPolled, 64);
    }
    return;
  }
  if (warp == kProducer) {
    __syncwarp();
    if constexpr (FAST) bar_sync(kBarPolled, 64);  // the exchange warp's last poll is done
    else bar_sync(kBarCompute, kThreads);          // the compute warps passed the grid barrier
    // Count the block out; the last block out resets the counters for the
    // next call (every block has passed all of its waits on them).
    if (lane == 0) {
      if (FAST && *abort_flag) {  // copies of an aborted block land before it exits
        #pragma unroll 1
        for (int u = 0; u < U; ++u) {
          if (!tb.blk[u]) continue;
          if (ng > 0) mbar_wait_bounded(&full_g[u], 0);
          if (nd > 0) mbar_wait_bounded(&full_d[u], 0);
          if ((tb.misc[5] >> u) & 1) mbar_wait_bounded(&hfull[u], 0);
        }
      }
      if (atom_add_acq_rel_gpu(&a.ws[1], 1) == a.G - 1) {
        if constexpr (FAST) {
          #pragma unroll 1
          for (int u = 0; u < U; ++u) a.ws[kCntBase + u] = 0;
        } else {
          a.ws[kCntBase] = 0;
        }
        a.ws[1] = 0;
      }
    }
    return;
  }

  if constexpr (FAST) {
    // ---- compute warps ---------------------------------------------------------
    // One token: every unit has its own stages (filled once). Item (u, r)
    // belongs to warp (u * n + r) % kWarps; gate/up items first, then down.
    int gq[NCX];
  #pragma unroll
    for (int it = 0; it < NCX; ++it) gq[it] = (32 * (lane + 32 * it)) / a.g;
    #pragma unroll 1
    for (int u = 0, s = 0, fill = 0; u < U && ng > 0; ++u, s = (s + 1 == a.Sg) ? 0 : s + 1, fill += s == 0) {
      if (!tb.blk[u]) continue;
      #pragma unroll 1
      for (int r = (warp - s * ng) & (kWarps - 1); r < ng; r += kWarps) {
        const bool ok = __all_sync(0xffffffffu, wait_phase(&full_g[s], fill & 1, abort_flag, a.ws));
        const int ra = r * kFastRows;
        const int nrows = min(kFastRows, rg_rows - ra);
        const uint8_t* rowa = ring_g + (size_t)s * a.sg + (size_t)ra * a.off.gu_row;
        #pragma unroll 1
        for (int i = tb.uoff[u]; i < tb.uoff[u + 1] && ok; ++i) {
          const int p = tb.upairs[i] & 0xffff, t = tb.upairs[i] >> 16;
          float acc[2 * kGateRows];
  #pragma unroll
          for (int q = 0; q < 2 * kGateRows; ++q) acc[q] = 0.0f;
          gate_up_rows<NCX>(rowa, nrows, a.off, nchx, lane, gq, xs4 + (size_t)t * nchx * 4, xsum + (size_t)t * nchx,
                            xback + (size_t)t * nchx, acc);
          const float hv = swiglu_lanes(acc, lane);
          const int rr = 2 * ((lane >> 4) & 1) + ((lane >> 3) & 1);  // the lane's row (lanes 0, 8, 16, 24)
          if ((lane & 7) == 0 && rr < nrows) hst[(size_t)p * a.rgu + ra + rr] = __float2half_rn(hv);
        }
        // The warp that completes the unit in this block publishes the block's
        // h rows of every pair of the unit and releases the unit (one release
        // per unit and block).
        __syncwarp();
        int last = 0;
        if (lane == 0 && ok) {
          mbar_arrive(&empty_g[s]);
          __threadfence_block();
          last = atomicAdd(&tb.udone[u], 1) == ng - 1;
        }
        if (last && lane == 0) {
          // Lane 0 stores the block's h rows of every pair of the unit itself,
          // so the release orders exactly its own stores before the count.
          __threadfence_block();  // the other warps' staged h (counted above)
          #pragma unroll 1
          for (int i = tb.uoff[u]; i < tb.uoff[u + 1]; ++i) {
            const int p = tb.upairs[i] & 0xffff;
            #pragma unroll 1
            for (int q = 0; q < rg_rows; ++q) a.hbuf[(size_t)p * a.I + n0 + q] = hst[(size_t)p * a.rgu + q];
          }
          red_release_gpu_add(&cnt[u], 1);
        }
        __syncwarp();
      }
    }
    int gd[NCH];
  #pragma unroll
    for (int it = 0; it < NCH; ++it) gd[it] = (32 * (lane + 32 * it)) / a.g;
    const int nchh = a.I / 32;
    #pragma unroll 1
    for (int u = 0, s = 0, fill = 0; u < U && nd > 0; ++u, s = (s + 1 == a.Sd) ? 0 : s + 1, fill += s == 0) {
      if (!tb.blk[u]) continue;
      #pragma unroll 1
      for (int r = (warp - s * nd) & (kWarps - 1); r < nd; r += kWarps) {
        // h of unit u complete in every block: the exchange warp copied it
        // into shared memory.
        bool ok = __all_sync(0xffffffffu, wait_phase(&hfull[s], 0, abort_flag, a.ws));
        const bool landed = __all_sync(0xffffffffu, wait_phase(&full_d[s], fill & 1, abort_flag, a.ws));
        ok = ok && landed;
        const int r0 = r * kDownRows;
        const uint8_t* stg = ring_d + (size_t)s * a.sd + (size_t)r0 * a.off.d_row;
        #pragma unroll 1
        for (int i = tb.uoff[u]; i < tb.uoff[u + 1] && ok; ++i) {
          const int p = tb.upairs[i] & 0xffff;
          const int nr = min(kDownRows, rd_rows - r0);
          down_rows<NCH, true>(stg, nr, a.off, hsm + (size_t)u * a.I, nchh, lane, gd, part + (size_t)p * a.rdn + r0);
        }
        __syncwarp();
        if (lane == 0 && landed) mbar_arrive(&empty_d[s]);
      }
    }
  } else {
    // Batched: the work items are dealt round-robin to the compute warps
    // (item j to warp j % kWarps), gate/up items first. A consumer of fill q
    // first waits until the producer has issued it (the stage's fill
    // number), so the stage's mbarrier is at that very phase; the warp that
    // finishes the last item of a fill frees its stage.
    const unsigned full = 0xffffffffu;
    const int Ug = ng > 0 ? U : 0;
    int gq[NCX];
#pragma unroll
    for (int it = 0; it < NCX; ++it) gq[it] = (32 * (lane + 32 * it)) / a.g;
    bool ok = true;
    // ---- gate/up: item j is (pair j / ng, row group j % ng) of the sorted
    // pairs (unit u's pairs sit at uoff[u] ..)
    const int NG = tb.uoff[U] * ng;
    int u = 0;
    #pragma unroll 1
    for (int j = warp; j < NG; j += kWarps) {
      const int c = j / ng, r = j - c * ng;
      while (tb.uoff[u + 1] <= c) ++u;
      const int s = u % a.Sg, lap = u / a.Sg;
      ok = __all_sync(full, wait_fill(fillno, s, lap, abort_flag, a.ws) &&
                                wait_phase(&full_g[s], lap & 1, abort_flag, a.ws));
      if (!ok) break;
      const int pr = tb.upairs[c], p = pr & 0xffff, t = pr >> 16;
      const int ra = r * kGateRows;
      const int nrows = min(kGateRows, rg_rows - ra);
      float acc[2 * kGateRows];
#pragma unroll
      for (int q = 0; q < 2 * kGateRows; ++q) acc[q] = 0.0f;
      gate_up_rows<NCX>(ring_g + (size_t)s * a.sg + (size_t)ra * a.off.gu_row, nrows, a.off, nchx, lane, gq,
                        xs4 + (size_t)t * nchx * 4, xsum + (size_t)t * nchx, xback + (size_t)t * nchx, acc);
      const float hv = swiglu_lanes(acc, lane);
      const int rr = 2 * ((lane >> 4) & 1) + ((lane >> 3) & 1);  // the lane's row (lanes 0, 8, 16, 24)
      if ((lane & 7) == 0 && rr < nrows) a.hbuf[(size_t)p * a.I + n0 + ra + rr] = __float2half_rn(hv);
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        if (atomicAdd(&tb.fdone[u], 1) == (tb.uoff[u + 1] - tb.uoff[u]) * ng - 1) mbar_arrive(&empty_g[s]);
      }
    }
    __syncwarp();
    // ---- every block's h rows are out (grid barrier, bounded) --------------
    // Thread 0 releases the block's stores (ordered before it by the block
    // barrier; the release is cumulative) and waits (acquire) until all G
    // blocks have; the second barrier passes that on.
    bar_sync(kBarGate, kWarps * 32);
    if (tid == 0) {
      int32_t* gbar = a.ws + kCntBase;
      red_release_gpu_add(gbar, 1);
      unsigned tries = 0;
      #pragma unroll 1
      while (ld_acquire_gpu(gbar) < a.G) {
        if (*abort_flag) break;
        if (++tries > kSpinTries) {
          *abort_flag = 1;
          atomicOr(a.ws, 4);
          break;
        }
      }
    }
    __syncwarp();
    bar_sync(kBarGate, kWarps * 32);
    // ---- down: item j is the pair at sorted position j (all of the
    // block's rows); the next item's h is loaded while this one computes.
    constexpr int NP = 2 * NCH;  // 16-value pieces of h per lane
    const int npc = a.I / 16;
    int gp[NP];
#pragma unroll
    for (int it = 0; it < NP; ++it) gp[it] = (16 * (lane + 32 * it)) / a.g;
    const int ND = nd > 0 ? tb.uoff[U] : 0;
    uint4 nxt[NP][2];
    auto fetch = [&](int jj) {
      const __half* h = a.hbuf + (size_t)(tb.upairs[jj] & 0xffff) * a.I;
#pragma unroll
      for (int it = 0; it < NP; ++it)
        if (lane + 32 * it < npc) load_piece(h + 16 * (lane + 32 * it), nxt[it]);
    };
    if (warp < ND && ok) fetch(warp);
    u = 0;
    #pragma unroll 1
    for (int j = warp; j < ND && ok; j += kWarps) {
      half2 hr[NP][8];
      float hsum[NP], hback[NP];
#pragma unroll
      for (int it = 0; it < NP; ++it)
        if (lane + 32 * it < npc) hsum[it] = scale_piece(nxt[it], hr[it], hback[it]);
      if (j + kWarps < ND) fetch(j + kWarps);
      while (tb.uoff[u + 1] <= j) ++u;
      const int pk = u / a.dpack, q = Ug + pk, s = q % a.Sg, lap = q / a.Sg;
      ok = __all_sync(full, wait_fill(fillno, s, lap, abort_flag, a.ws) &&
                                wait_phase(&full_g[s], lap & 1, abort_flag, a.ws));
      if (!ok) break;
      const int p = tb.upairs[j] & 0xffff;
      down_pair_rows<NP>(ring_g + (size_t)s * a.sg + (size_t)(u - pk * a.dpack) * a.sd, rd_rows, a.off, npc, lane,
                         gp, hr, hsum, hback, part + (size_t)p * a.rdn);
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        const int ua = pk * a.dpack, ub = min(U, ua + a.dpack);
        if (atomicAdd(&tb.fdone[q], 1) == tb.uoff[ub] - tb.uoff[ua] - 1) mbar_arrive(&empty_g[s]);
      }
    }
  }
  __syncwarp();
  bar_sync(kBarCompute, kThreads);
  // y[t][m0 + r] = sum_j w[t][j] * part[t*k + j][r] (+ y_shared), in j order.
  #pragma unroll 1
  for (int i = tid; i < a.T * rd_rows; i += kWarps * 32) {
    const int t = i / rd_rows, r = i - t * rd_rows;
    float v = 0.0f;
    #pragma unroll 1
    for (int j = 0; j < a.k; ++j) {
      const int p = t * a.k + j;
      if (tb.punit[p] >= 0) v += tb.w[p] * part[(size_t)p * a.rdn + r];
    }
    if (a.y_shared) v += __half2float(a.y_shared[(size_t)t * a.H + m0 + r]);
    a.y[(size_t)t * a.H + m0 + r] = __float2half_rn(v);
  }
}

// ---- host side ----------------------------------------------------------------
std::mutex g_dev_mutex;
int g_num_sms[kMaxDevices] = {0};
// Per device: the largest dynamic shared memory already granted to each kernel
// instantiation (cudaFuncSetAttribute is called only when a launch needs more).
int g_smem_set[kMaxDevices][3][2][2] = {};

int device_sms(int* dev_out, int* sms_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_num_sms[dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    g_num_sms[dev] = n;
  }
  *dev_out = dev;
  *sms_out = g_num_sms[dev];
  return MOE_OK;
}

template <int NCX, int NCH, bool FAST>
cudaError_t launch_stream(int dev, const StreamParams& a, cudaStream_t st) {
  auto kern = decode_stream_kernel<NCX, NCH, FAST>;
  const int xi = NCX == 1 ? 0 : (NCX == 2 ? 1 : 2), hi = NCH - 1;
  {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_smem_set[dev][xi][hi][FAST] < (int)a.smem) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)a.smem);
      if (e != cudaSuccess) return e;
      g_smem_set[dev][xi][hi][FAST] = (int)a.smem;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = a.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int NCX, int NCH>
cudaError_t launch_stream2(int dev, const StreamParams& a, cudaStream_t st) {
  return a.fast1 ? launch_stream<NCX, NCH, true>(dev, a, st) : launch_stream<NCX, NCH, false>(dev, a, st);
}

constexpr size_t kSmemBudget = 227 * 1024;

// Shared-memory carve-up: ring(s) (also the routing scratch) | x | part |
// h staging | h copies | tables | barriers. Returns false when the shape
// does not fit.
bool carve(StreamParams& a) {
  const size_t xbytes = (size_t)a.T * a.H * 2 + (size_t)a.T * (a.H / 32) * 8;
  const size_t partb = (size_t)a.P * a.rdn * 4;
  const size_t tabb = tables_bytes(a.P, a.E);
  const size_t barb = 6 * kMaxRing * 8;
  const uint32_t sgu = align16((uint32_t)a.rgu * a.off.gu_row), sdn = align16((uint32_t)a.rdn * a.off.d_row);
  auto r16 = [](size_t v) { return (v + 15) & ~(size_t)15; };
  auto place = [&](size_t ringb, size_t hstb, size_t hsmb) {
    size_t o = r16(ringb);
    a.o_x = (uint32_t)o;
    o += r16(xbytes);
    a.o_part = (uint32_t)o;
    o += r16(partb);
    a.o_hst = (uint32_t)o;
    o += r16(hstb);
    a.o_hsm = (uint32_t)o;
    o += r16(hsmb);
    a.o_small = (uint32_t)o;
    o += r16(tabb);
    a.o_bar = (uint32_t)o;
    o += barb;
    a.smem = (uint32_t)o;
    return o <= kSmemBudget;
  };
  // One routed token: each of the k picks gets its own stage in both rings
  // (filled once), h is staged per block and each pick's complete h is
  // copied into shared memory for the down rows.
  a.fast1 = 0;
  a.dpack = 1;
  if (a.T == 1 && a.logits != nullptr && a.k <= kMaxFastK) {
    const size_t ringb = std::max((size_t)a.k * (sgu + sdn), (size_t)a.E * 4);  // also the token's logits
    if (place(ringb, (size_t)a.P * a.rgu * 2, (size_t)a.k * a.I * 2)) {
      a.fast1 = 1;
      a.Sg = a.Sd = a.k;
      a.sg = sgu;
      a.sd = sdn;
      a.o_ring_d = (uint32_t)((size_t)a.k * sgu);
      return true;
    }
  }
  // Batched: one ring of S stages; a stage holds one unit's gate/up rows or
  // the down rows of dpack units.
  const size_t fixed = r16(xbytes) + r16(partb) + r16(tabb) + barb;
  const int dpack = std::max<int>(1, (int)(sgu / sdn));
  const uint32_t sst = align16(std::max<uint32_t>(sgu, (uint32_t)dpack * sdn));
  if (fixed + sst > kSmemBudget) return false;
  const int S = (int)std::min<size_t>(kMaxRing, (kSmemBudget - fixed) / sst);
  const size_t ringb = std::max((size_t)S * sst, a.logits ? (size_t)a.T * a.E * 4 : 0);  // routing scratch
  if (!place(ringb, 0, 0)) return false;
  a.Sg = S;
  a.Sd = 0;
  a.sg = sst;
  a.sd = sdn;
  a.dpack = dpack;
  a.o_ring_d = 0;
  return true;
}

}  // namespace

int current_device_sms(int* dev, int* sms) { return device_sms(dev, sms); }

size_t fused_workspace_bytes(int H, int I, int T, int k) {
  (void)H;
  return ws_scratch_offset(T * k) + (size_t)T * k * I * 2;
}

int fused_forward_routed(const ForwardArgs& fa, const float* logits, int renorm, int32_t* ids_out,
                         float* wts_out) {
  int dev = 0, sms = 0;
  int rc = device_sms(&dev, &sms);
  if (rc != MOE_OK) return rc;
  const int xc = (fa.H + 1023) / 1024, hc = (fa.I + 1023) / 1024;
  if (xc > 4 || hc > 2) return fail(MOE_ERR_UNSUPPORTED, "streamed decode: H <= 4096 and I <= 2048 only");
  if (fa.T > kMaxT || fa.T * fa.k > kMaxP || fa.E > kMaxE)
    return fail(MOE_ERR_UNSUPPORTED, "streamed decode: T <= %d, T*k <= %d and E <= %d only", kMaxT, kMaxP, kMaxE);
  StreamParams a;
  a.H = fa.H; a.I = fa.I; a.g = fa.g; a.T = fa.T; a.k = fa.k; a.E = fa.E; a.n_slots = fa.n_slots;
  a.P = fa.T * fa.k;
  a.G = sms;
  a.x = fa.x; a.ids = fa.ids; a.wts = fa.weights; a.pool = fa.pool; a.block_bytes = fa.block_bytes;
  a.logits = logits; a.renorm = renorm; a.ids_out = ids_out; a.wts_out = wts_out;
  a.off = fa.off; a.slot_of = fa.slot_of; a.y_shared = fa.y_shared; a.y = fa.y;
  uint8_t* ws = static_cast<uint8_t*>(fa.ws);
  a.ws = reinterpret_cast<int32_t*>(ws);
  a.hbuf = reinterpret_cast<__half*>(ws + ws_scratch_offset(a.P));
  a.rgu = (a.I + a.G - 1) / a.G;
  a.rdn = (a.H + a.G - 1) / a.G;
  if (!carve(a)) return fail(MOE_ERR_UNSUPPORTED, "streamed decode: shapes exceed shared memory");
  cudaError_t e;
  cudaStream_t st = fa.stream;
  if (xc == 1) e = hc == 1 ? launch_stream2<1, 1>(dev, a, st) : launch_stream2<1, 2>(dev, a, st);
  else if (xc == 2) e = hc == 1 ? launch_stream2<2, 1>(dev, a, st) : launch_stream2<2, 2>(dev, a, st);
  else e = hc == 1 ? launch_stream2<4, 1>(dev, a, st) : launch_stream2<4, 2>(dev, a, st);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "decode stream launch: %s", cudaGetErrorString(e));
  return MOE_OK;
}

int fused_forward(const ForwardArgs& fa) { return fused_forward_routed(fa, nullptr, 0, nullptr, nullptr); }

}  // namespace moe
