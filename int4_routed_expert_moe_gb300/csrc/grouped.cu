// Grouped (token-sorted) tensor-core path of the routed expert FFN, for
// prefill and large batches.
//
// "Horizon RunMap -- Prévia Técnica", "03 / Arquitetura" and "04 /
// Resultados": the compact INT4 experts are computed in groups of the tokens
// routed to them; the weights stay INT4 + FP16 scale/zero in memory and are
// expanded only on chip, activations are FP16 and accumulation FP32.
//
// Steps (one stream, five launches):
//   1-2. token sort: pairs p = t*k + j grouped by expert (stable), and in
//      the same kernel the tile list (for every resident expert with pairs,
//      tiles of up to 128 consecutive sorted pairs) and the unusable-id flags;
//   3. gather: X_sorted[pos] = x[token of pos], K order permuted inside each
//      8-element chunk (see dq_word);
//   4. gate/up GEMM per (tile, 128 rows of I): TMA brings the INT4 codes and
//      the scale/zero quads of W_gate and W_up plus the X tile; eight warps
//      expand the codes to FP16 in the 128-byte-swizzled K-major layout; one
//      thread issues tcgen05.mma (M = 128 rows, N = pairs, K = 16) into two
//      TMEM accumulators; the epilogue reads them back, forms
//      h = silu(gate) * up, rounds it to FP16 and stores h_sorted;
//   5. down GEMM per (tile, 128 rows of H) on h_sorted, the FP32 result of
//      pair (t, j) stored as pair_out[t*k + j];
//   6. combine: y[t] = sum_j w[t][j] * pair_out[t*k + j] in j order
//      (+ y_shared), rounded to FP16.
// Weights are the M operand (swap-AB), so each expert's codes are read once
// per tile of up to 128 pairs.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.h"
#include "device.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

int encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  const CUresult r = g_encode(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MOE_OK;
}

namespace {

constexpr int BM = 128;  // weight rows per tile (MMA M)
constexpr int BK = 64;   // K elements per pipeline step (one 128-byte swizzle row)
constexpr int BN = 128;  // sorted pairs per tile at most (MMA N)
// Warp roles: 0 codes TMA, 1 TMEM + MMA issue (accumulator 0), 2 activation
// TMA, 3 MMA issue (accumulator 1), 4..19 expand codes to FP16 and run the
// epilogue. At the small N of one expert's pairs an issuing thread needs
// about as long per MMA as the tensor pipe (~54 cycles against 32 at N = 64),
// so two issuing warps with an accumulator each keep the pipe fed; each runs
// its loop converged with one elected lane issuing (a lone issuing lane
// loses half its rate to the expand warps on its scheduler). The expansion
// is a chain of short dependent steps per warp; sixteen expand warps (four
// per SM sub-partition) keep the issue slots busy.
constexpr int kDqWarps = 16;
// The down kernel has four more warps (20..23) for its epilogue: its items are
// short (K = I), so it keeps two accumulators and the next item's MMAs run
// while these warps write the previous item's rows.
constexpr int kEpiWarps = 4;
template <int NPROJ>
constexpr int kThreadsOf = (4 + kDqWarps + (NPROJ == 1 ? kEpiWarps : 0)) * 32;
constexpr uint32_t kCodeBytes = BM * 32;      // codes of 128 rows x 64 elements
constexpr uint32_t kSzBytes = BM * 32;        // 32 bytes of scale/zero entries per row
constexpr uint32_t kXBytes = BN * BK * 2;     // activation tile, up to 128 pairs

// Ring geometry per kernel (NPROJ = 2: gate and up; 1: down). Two rings:
// codes and scale/zero entries in shared memory (freed as soon as the expand
// warps hold them in registers), and per step an activation tile in shared
// memory plus the expanded FP16 weights in tensor memory (freed together, by
// one commit per issuing warp, when the MMAs reading them complete). Keeping
// the expanded operand out of shared memory leaves its bandwidth to the TMA
// writes and the activation reads of the MMAs.
template <int NPROJ>
struct Geo {
  static constexpr int SC = NPROJ == 2 ? 12 : 16;  // code stages: 144 / 128 KB in flight per SM
  static constexpr int SA = 4;
  static constexpr int SX = SA;
  static constexpr uint32_t kC = NPROJ * kCodeBytes + kSzBytes;
  static constexpr uint32_t offX = 0, offC = SX * kXBytes, offCtrl = offC + SC * kC;
  static constexpr size_t smem = (size_t)offCtrl + 1024 + 1024;
  static constexpr uint32_t kSzEntry = NPROJ == 2 ? 8 : 4;  // bytes of one group's scale/zero entry
  static constexpr int kGAlign = NPROJ == 2 ? 2 : 4;         // entries per 16 bytes
  // Tensor memory: two accumulators in columns [0, 2*BN) (gate and up; or
  // the even and odd K slices of the down projection), then SA stages of the
  // expanded operand, 32 columns (64 FP16 of K) per projection.
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t colA(int sa, int p) { return 2 * BN + (uint32_t)(sa * NPROJ + p) * 32u; }
  static_assert(2 * BN + SA * NPROJ * 32 <= (int)kTmemCols, "tensor memory budget");
  static_assert(kC % 1024 == 0, "ring slots keep 1024-byte alignment");
  // Each ring slot must always be drained by the same expand warps (step kt
  // is taken by the warps with kt % 4 == j), so no waiter can see a phase two
  // fills ahead.
  static_assert(SC % 4 == 0 && SA % 4 == 0, "slot ownership of the interleaved expand warps");
};

// Position of element e (0..7) of an 8-element chunk in the K order used by
// the tensor-core operands: elements (0, 4, 1, 5, 2, 6, 3, 7) in that order.
__host__ __device__ constexpr int kperm_pos(int e) { return (e & 3) * 2 + (e >> 2); }

// The expanded operand holds 16 (q - z) s; the epilogue divides by 16 (exact).
constexpr float kInvAScale = 0.0625f;

// Constants of one (row, group) for dq_word, from its FP16 (s, z).
struct DqConst {
  half2 zl, zh, sl, sh, cl, ch;
};
__device__ __forceinline__ DqConst dq_const(uint32_t sz) {
  const float s = __half2float(__ushort_as_half((unsigned short)(sz & 0xFFFFu)));
  const float z = __half2float(__ushort_as_half((unsigned short)(sz >> 16)));
  const float zi = rintf(z);
  const float zl = fminf(fmaxf(zi, -1000.0f), 1000.0f);  // 1024 + zl exact in FP16
  const float zh = fabsf(zi) <= 63.0f ? zi : 0.0f;       // 1024 + 16 zh exact in FP16
  DqConst d;
  d.zl = __float2half2_rn(1024.0f + zl);
  d.zh = __float2half2_rn(1024.0f + 16.0f * zh);
  d.sl = __float2half2_rn(16.0f * s);
  d.sh = __float2half2_rn(s);
  d.cl = __float2half2_rn(16.0f * (zl - z) * s);
  d.ch = __float2half2_rn(16.0f * (zh - z) * s);
  return d;
}

__device__ __forceinline__ uint32_t h2_bits(half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Eight codes of one word (element i in bits 4i..4i+3) to eight FP16 values
// 16 (q - z) s in operand K order. Low nibbles OR-ed into 1024 give 1024 + q,
// and minus (1024 + zl) the exact q - zl; high nibbles masked in place give
// 1024 + 16 q, and minus (1024 + 16 zh) the exact 16 (q - zh). One fused
// multiply-add each (by 16 s or s) adds the rest of the zero point, 16 (zl -
// z) s or 16 (zh - z) s -- zero for an integer zero point -- and rounds once.
__device__ __forceinline__ uint4 dq_word(uint32_t w, const DqConst& d) {
  const uint32_t ml = 0x000F000Fu, mh = 0x00F000F0u, mg = 0x64006400u;
  const uint32_t w8 = w >> 8;
  uint4 o;
  o.x = h2_bits(__hfma2(__hsub2(u32_as_h2((w & ml) | mg), d.zl), d.sl, d.cl));   // elements 0, 4
  o.y = h2_bits(__hfma2(__hsub2(u32_as_h2((w & mh) | mg), d.zh), d.sh, d.ch));   // 1, 5
  o.z = h2_bits(__hfma2(__hsub2(u32_as_h2((w8 & ml) | mg), d.zl), d.sl, d.cl));  // 2, 6
  o.w = h2_bits(__hfma2(__hsub2(u32_as_h2((w8 & mh) | mg), d.zh), d.sh, d.ch));  // 3, 7
  return o;
}

struct GemmParams {
  const int4* tiles;  // (slot, first sorted position, pairs, expert)
  const int32_t* n_tiles;
  int rows;           // output rows of the weight matrix (I for gate/up, H for down)
  int K;              // reduction length (H for gate/up, I for down)
  int g;
  uint32_t g_magic;     // ceil(2^32 / g)
  uint32_t q0, q1, sz;  // byte offsets in a weight row: codes (gate or down, up), scale/zero entries
  __half* h_sorted;     // gate/up output [P][I]
  float* pair_out;      // down output [T*k][H]
  const int32_t* pair_tok;
  const int32_t* pair_j;
  int k;
  int32_t* flags;
};

struct Bars {
  uint64_t *c_full, *c_empty, *x_full, *a_full, *a_empty, *acc_full, *acc_empty, *handoff;
  uint32_t* tmem_slot;
  int* abort;
};
template <int NPROJ>
__device__ __forceinline__ Bars bars_at(uint8_t* p) {
  using G = Geo<NPROJ>;
  Bars b;
  uint64_t* q = reinterpret_cast<uint64_t*>(p);
  b.c_full = q; q += G::SC;
  b.c_empty = q; q += G::SC;
  b.x_full = q; q += G::SX;
  b.a_full = q; q += G::SA;
  b.a_empty = q; q += G::SA;
  b.acc_full = q; q += 2;
  b.acc_empty = q; q += 2;
  b.handoff = q; q += 2;
  b.tmem_slot = reinterpret_cast<uint32_t*>(q);
  b.abort = reinterpret_cast<int*>(b.tmem_slot + 1);
  return b;
}
// A bounded wait expired: report it (bit 2) and stop the block's other roles.
__device__ __forceinline__ void abort_block(const Bars& b, int32_t* flags) {
  atomicOr(flags, 4);
  *reinterpret_cast<volatile int*>(b.abort) = 1;
}
__device__ __forceinline__ bool is_aborted(const Bars& b) { return *reinterpret_cast<volatile int*>(b.abort) != 0; }
// Producer tail after an abort: wait (bounded) for its loads still in flight.
__device__ __forceinline__ void drain(uint64_t* full, int stages, int issued) {
  for (int kt = issued > stages ? issued - stages : 0; kt < issued; ++kt)
    tc::bar_wait(&full[kt % stages], (kt / stages) & 1);
}

// Work item: 128 weight rows (row block rb) x up to 128 sorted pairs of one
// expert (tile). The grid is persistent: block c takes items c, c + G, ...;
// the step counter of every ring runs on across items, so the TMA warps
// prefetch the next item's codes and activations while the current item's
// epilogue runs, and the accumulators are reused once the epilogue has read
// them (acc_empty).
//   NPROJ = 2: gate and up accumulators, epilogue h = silu(gate) * up (FP16).
//   NPROJ = 1: down accumulators (even and odd K slices), epilogue
//              pair_out[t*k + j] (FP32).
struct Item {
  int slot, pos0, n, nmma, row0;
};
__device__ __forceinline__ Item item_of(const GemmParams& a, int w, int rblocks) {
  const int4 td = a.tiles[w / rblocks];
  Item it;
  it.slot = td.x;
  it.pos0 = td.y;
  it.n = td.z;
  it.nmma = (td.z + 15) & ~15;
  it.row0 = (w % rblocks) * BM;
  return it;
}

template <int NPROJ>
__global__ void __launch_bounds__(kThreadsOf<NPROJ>, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_b,
                        const GemmParams a) {
  using G = Geo<NPROJ>;
  const int rblocks = (a.rows + BM - 1) / BM;
  const int n_items = *a.n_tiles * rblocks;
  if ((int)blockIdx.x >= n_items) return;
  const int KT = a.K / BK;
  constexpr uint32_t kTmemCols = G::kTmemCols;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = tc::align1024(smraw);
  const Bars b = bars_at<NPROJ>(sm + G::offCtrl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::tma_prefetch_desc(&map_w);
    tc::tma_prefetch_desc(&map_b);
    for (int s = 0; s < G::SC; ++s) {
      tc::bar_init(&b.c_full[s], 1);
      tc::bar_init(&b.c_empty[s], 4);  // one expand warp per lane quarter takes each step
    }
    for (int s = 0; s < G::SA; ++s) {
      tc::bar_init(&b.x_full[s], 1);
      tc::bar_init(&b.a_full[s], 4);
      tc::bar_init(&b.a_empty[s], NPROJ == 2 ? 2 : 1);  // one commit per issuing warp that reads the step
    }
    if (NPROJ == 2) {  // one accumulator pair; the expand warps run the epilogue
      tc::bar_init(&b.acc_full[0], 2);
      tc::bar_init(&b.acc_empty[0], kDqWarps);
    } else {  // two accumulators, items alternating; the epilogue warps free them
      for (int p = 0; p < 2; ++p) {
        tc::bar_init(&b.acc_full[p], 1);
        tc::bar_init(&b.acc_empty[p], kEpiWarps);
        tc::bar_init(&b.handoff[p], 1);
      }
    }
    *b.abort = 0;
    tc::bar_init_fence();
  }
  if (warp == 1) tc::tmem_alloc(b.tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *b.tmem_slot;

  if (warp == 0 || warp == 2) {
    // TMA producers, each a whole warp running its loop (waits, addresses)
    // with one elected lane issuing the copies: a lone lane's loop loses
    // issue slots to the expand warps on its scheduler. Warp 0: codes and
    // scale/zero entries of each item's rows; warp 2: the activation tile of
    // each step (64 sorted pairs per load).
    const bool codes = warp == 0;
    uint64_t* full = codes ? b.c_full : b.x_full;
    uint64_t* empty = codes ? b.c_empty : b.a_empty;
    const int S = codes ? G::SC : G::SX;
    int issued = 0;
    for (int w = blockIdx.x, li = 0; w < n_items && !__any_sync(0xffffffffu, is_aborted(b)); w += gridDim.x, ++li) {
      const Item it = item_of(a, w, rblocks);
      const uint32_t xbytes = (it.n > 64 ? 2u : 1u) * 64u * BK * 2u;
      bool ok = true;
      for (int kt = 0; kt < KT; ++kt) {
        const int g = li * KT + kt, s = g % S;
        if (g >= S && !tc::bar_wait_warp(&empty[s], ((g / S) - 1) & 1)) {
          ok = false;
          break;
        }
        const int k0 = kt * BK;
        if (tc::elect_one()) {
          if (codes) {
            uint8_t* st = sm + G::offC + (size_t)s * G::kC;
            const int gb = (int)__umulhi((uint32_t)k0, a.g_magic) / G::kGAlign * G::kGAlign;  // floor(k0 / g), aligned
            tc::bar_expect_tx(&full[s], G::kC);
            tc::tma_load_3d(st, &map_w, (int)a.q0 + k0 / 2, it.row0, it.slot, &full[s]);
            if (NPROJ == 2) tc::tma_load_3d(st + kCodeBytes, &map_w, (int)a.q1 + k0 / 2, it.row0, it.slot, &full[s]);
            tc::tma_load_3d(st + NPROJ * kCodeBytes, &map_w, (int)(a.sz + G::kSzEntry * gb), it.row0, it.slot,
                            &full[s]);
          } else {
            uint8_t* st = sm + G::offX + (size_t)s * kXBytes;
            tc::bar_expect_tx(&full[s], xbytes);
            tc::tma_load_2d(st, &map_b, k0, it.pos0, &full[s]);
            if (it.n > 64) tc::tma_load_2d(st + 64 * BK * 2, &map_b, k0, it.pos0 + 64, &full[s]);
          }
        }
        __syncwarp();
        issued = g + 1;
      }
      if (!ok) {
        if (lane == 0) abort_block(b, a.flags);
        break;
      }
    }
    if (lane == 0 && is_aborted(b)) drain(full, S, issued);
  } else if (warp == 1 || warp == 3) {
    // Issuing warp p owns accumulator p. Gate/up: the gate (p = 0) or up
    // (p = 1) projection of every item. Down: the items li with li % 2 == p,
    // all four K slices of each step, so one item's MMAs run while the
    // epilogue warps read the other accumulator; a warp starts its item once
    // the other has issued the item before (handoff), so its waits on the
    // step barriers, which complete once per step, are never a phase ahead.
    // The whole warp runs the loop (waits, descriptors) and one elected lane
    // issues: descriptors from values fixed before the loop plus one add, one
    // wait per step (a_full also stands for the activation tile, see the
    // expand warps), the abort flag read once per item.
    const int p = warp == 1 ? 0 : 1;
    const uint32_t d_tmem = tmem + (uint32_t)(p * BN);
    const uint64_t xdesc0 = tc::sw128_desc(tc::smem_addr(sm + G::offX));
    constexpr uint32_t kXDescStep = kXBytes >> 4;  // descriptor address units per activation stage
    const uint32_t a_tmem0 = tmem + G::colA(0, NPROJ == 2 ? p : 0);
    constexpr uint32_t kAColStep = G::colA(1, 0) - G::colA(0, 0);
    for (int w = blockIdx.x, li = 0; w < n_items && !__any_sync(0xffffffffu, is_aborted(b)); w += gridDim.x, ++li) {
      if (NPROJ == 1 && (li & 1) != p) continue;
      const Item it = item_of(a, w, rblocks);
      const uint32_t idesc = tc::idesc_f16(BM, it.nmma);
      // The epilogue has read this accumulator's previous item.
      const int use = NPROJ == 2 ? li : (li >> 1);  // this accumulator's use count
      uint64_t* acc_full = &b.acc_full[NPROJ == 2 ? 0 : p];
      uint64_t* acc_empty = &b.acc_empty[NPROJ == 2 ? 0 : p];
      if (NPROJ == 1 && li > 0 && !tc::bar_wait_warp(&b.handoff[p ^ 1], ((li - 1) >> 1) & 1)) {
        if (lane == 0) abort_block(b, a.flags);
        break;
      }
      if (use > 0 && !tc::bar_wait_warp(acc_empty, (use - 1) & 1)) {
        if (lane == 0) abort_block(b, a.flags);
        break;
      }
      tc::tc_fence_after();
      bool ok = true;
      for (int kt = 0; kt < KT; ++kt) {
        const int g = li * KT + kt, sa = g % G::SA;
        if (!tc::bar_wait_warp(&b.a_full[sa], (g / G::SA) & 1)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint64_t xd = xdesc0 + (uint64_t)(sa * kXDescStep);  // 128-byte-swizzled tile, 1024-aligned
        const uint32_t at = a_tmem0 + (uint32_t)sa * kAColStep;
        if (tc::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_f16_ta(d_tmem, at + kk * 8, xd + 2 * kk, idesc, kt > 0 || kk > 0);
          tc::mma_commit(&b.a_empty[sa]);
        }
        __syncwarp();
      }
      if (!ok) {
        if (lane == 0) abort_block(b, a.flags);
        break;
      }
      if (tc::elect_one()) {
        tc::mma_commit(acc_full);
        if (NPROJ == 1) tc::bar_arrive(&b.handoff[p]);  // this item's MMAs are all issued
      }
      __syncwarp();
    }
  } else if (warp < 4 + kDqWarps) {
    // Expand: warp w owns the TMEM lanes of its quarter (rows 32 (w % 4) ..
    // +31) and every fourth step (global step g = j (mod 4), j = (w - 4) / 4),
    // so four steps are expanded at once; lane t owns row 32 (w % 4) + t, all
    // 64 codes of the step (at most two scale/zero groups: one per 32).
    const int q4 = warp & 3, j4 = (warp - 4) >> 2;
    const int r = 32 * q4 + lane;
    const uint32_t tlane = tmem + ((uint32_t)(32 * q4) << 16);
    // Gate/up epilogue of item e_li: TMEM lanes of this warp's quarter, the
    // 16-column chunks j4, j4 + 4, ... of the live columns; then release the
    // accumulators. Each warp runs it after expanding its first step of the
    // next item, so the next item's first four steps are ready when the
    // accumulators are.
    auto epilogue = [&](const Item& e, int e_li) -> bool {
      const bool got = tc::bar_wait(&b.acc_full[0], e_li & 1);
      if (!got) abort_block(b, a.flags);
      tc::tc_fence_after();
      const int row = e.row0 + r;
      const bool live = got && !is_aborted(b) && row < a.rows;
      for (int c0 = 16 * j4; c0 < e.nmma; c0 += 64) {
        float gv[16], uv[16];
        tc::tmem_ld16(tlane + (uint32_t)c0, gv);
        tc::tmem_ld16(tlane + (uint32_t)(BN + c0), uv);
        tc::tmem_ld_wait();
        if (live) {
          const int prow = (row & ~7) | kperm_pos(row & 7);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < e.n)
              a.h_sorted[(size_t)(e.pos0 + c0 + j) * a.rows + prow] =
                  __float2half_rn(silu_fast(gv[j] * kInvAScale) * (uv[j] * kInvAScale));
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::bar_arrive(&b.acc_empty[0]);
      return got;
    };
    bool ok = true;
    Item prev{};
    int prev_li = -1;  // item whose epilogue this warp still owes (gate/up)
    for (int w = blockIdx.x, li = 0; w < n_items && ok; w += gridDim.x, ++li) {
      const Item it = item_of(a, w, rblocks);
      const int g0 = li * KT;
      for (int g = g0 + ((j4 - g0) % 4 + 4) % 4; g < g0 + KT; g += 4) {
        const int kt = g - g0;
        const int sc = g % G::SC, sa = g % G::SA;
        if (is_aborted(b) || !tc::bar_wait(&b.c_full[sc], (g / G::SC) & 1)) {
          abort_block(b, a.flags);
          ok = false;
          break;
        }
        const uint8_t* cs = sm + G::offC + (size_t)sc * G::kC;
        const uint32_t k0 = (uint32_t)kt * BK;
        // floor(k / g) by multiply-high with the rounded-up reciprocal (exact
        // for k, g <= 8192).
        const int gi0 = (int)__umulhi(k0, a.g_magic), gi1 = (int)__umulhi(k0 + 32u, a.g_magic);
        const int gb = gi0 / G::kGAlign * G::kGAlign;
        uint4 cw[NPROJ][2];
        DqConst d0[NPROJ], d1[NPROJ];
#pragma unroll
        for (int p = 0; p < NPROJ; ++p) {
          const uint4* src = reinterpret_cast<const uint4*>(cs + p * kCodeBytes + r * 32);
          cw[p][0] = src[0];
          cw[p][1] = src[1];
          const uint8_t* e = cs + NPROJ * kCodeBytes + r * 32 + 4 * p;
          d0[p] = dq_const(*reinterpret_cast<const uint32_t*>(e + (gi0 - gb) * G::kSzEntry));
          d1[p] = gi1 == gi0 ? d0[p] : dq_const(*reinterpret_cast<const uint32_t*>(e + (gi1 - gb) * G::kSzEntry));
        }
        __syncwarp();
        if (lane == 0) tc::bar_arrive(&b.c_empty[sc]);
        if (g >= G::SA && !tc::bar_wait(&b.a_empty[sa], ((g / G::SA) - 1) & 1)) {
          abort_block(b, a.flags);
          ok = false;
          break;
        }
        tc::tc_fence_after();
#pragma unroll
        for (int p = 0; p < NPROJ; ++p) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const DqConst& d = h ? d1[p] : d0[p];
            const uint4 c = cw[p][h];
            const uint4 o0 = dq_word(c.x, d), o1 = dq_word(c.y, d), o2 = dq_word(c.z, d), o3 = dq_word(c.w, d);
            const uint32_t v[16] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w,
                                    o2.x, o2.y, o2.z, o2.w, o3.x, o3.y, o3.z, o3.w};
            tc::tmem_st16(tlane + G::colA(sa, p) + 16u * h, v);
          }
        }
        tc::tmem_st_wait();
        tc::tc_fence_before();
        // Lane 0 of the step's quarter-0 warp also waits for the step's
        // activation tile before its arrival, so a complete a_full phase means
        // both operands are in place (the issuers wait on a_full alone).
        bool xin = true;
        if (q4 == 0 && lane == 0) xin = tc::bar_wait(&b.x_full[sa], (g / G::SX) & 1);
        if (!__shfl_sync(0xffffffffu, xin, 0)) {
          abort_block(b, a.flags);
          ok = false;
          break;
        }
        __syncwarp();
        if (lane == 0) tc::bar_arrive(&b.a_full[sa]);
        if (NPROJ == 2 && prev_li >= 0) {
          ok = epilogue(prev, prev_li);
          prev_li = -1;
          if (!ok) break;
        }
      }
      if (!ok) break;
      if (NPROJ == 1) continue;  // the epilogue warps take the down items
      if (prev_li >= 0 && !(ok = epilogue(prev, prev_li))) break;  // this warp had no step in item li
      prev = it;
      prev_li = li;
    }
    if (NPROJ == 2 && ok && prev_li >= 0) epilogue(prev, prev_li);
  } else if (NPROJ == 1) {
    // Down epilogue (warps 20..23): warp q owns the TMEM lanes of quarter q.
    // Per item: the output pair index of each column (lane l holds columns
    // l, l + 32, l + 64, l + 96), read before the accumulator is ready; then
    // the FP32 rows of the item's pairs, and the accumulator released.
    const int q4 = warp & 3;
    const uint32_t tlane = tmem + ((uint32_t)(32 * q4) << 16);
    for (int w = blockIdx.x, li = 0; w < n_items; w += gridDim.x, ++li) {
      const Item it = item_of(a, w, rblocks);
      static_assert(BN == 128, "four 32-column groups per accumulator");
      int qcol[BN / 32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        const int col = lane + 32 * c;
        qcol[c] = 0;
        if (col < it.n) qcol[c] = a.pair_tok[it.pos0 + col] * a.k + a.pair_j[it.pos0 + col];
      }
      const int pb = li & 1;
      const bool got = tc::bar_wait_warp(&b.acc_full[pb], (li >> 1) & 1);
      if (!got && lane == 0) abort_block(b, a.flags);
      tc::tc_fence_after();
      const int row = it.row0 + 32 * q4 + lane;
      const bool live = got && !is_aborted(b) && row < a.rows;
      for (int c0 = 0; c0 < it.nmma; c0 += 16) {
        float dv[16];
        tc::tmem_ld16(tlane + (uint32_t)(pb * BN + c0), dv);
        tc::tmem_ld_wait();
        const int qsrc = (c0 >> 5) == 0 ? qcol[0] : (c0 >> 5) == 1 ? qcol[1] : (c0 >> 5) == 2 ? qcol[2] : qcol[3];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int q = __shfl_sync(0xffffffffu, qsrc, (c0 & 31) + j);
          if (live && c0 + j < it.n) a.pair_out[(size_t)q * a.rows + row] = dv[j] * kInvAScale;
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::bar_arrive(&b.acc_empty[pb]);
      if (!got) break;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- small kernels -------------------------------------------------------------
// X_sorted[pos] = x[pair_tok[pos]], each 8-element chunk in operand K order.
// A warp per sorted row (rows pos < offsets[E] hold valid pairs): the row's
// token is read once and the row's 16-byte chunks are loaded side by side.
constexpr int kGatherWarps = 8;
__global__ void __launch_bounds__(kGatherWarps * 32)
    grouped_gather_kernel(const __half* __restrict__ x, int H, const int32_t* __restrict__ offsets, int E,
                          const int32_t* __restrict__ pair_tok, __half* __restrict__ xs) {
  const int pv = offsets[E];
  const int cpr = H / 8;
  const int lane = threadIdx.x & 31;
  for (int pos = blockIdx.x * kGatherWarps + (threadIdx.x >> 5); pos < pv; pos += gridDim.x * kGatherWarps) {
    const int t = pair_tok[pos];
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)pos * H);
#pragma unroll 4
    for (int ch = lane; ch < cpr; ch += 32) {
      const uint4 v = src[ch];
      const unsigned short* e = reinterpret_cast<const unsigned short*>(&v);
      uint4 o;
      o.x = (uint32_t)e[0] | ((uint32_t)e[4] << 16);
      o.y = (uint32_t)e[1] | ((uint32_t)e[5] << 16);
      o.z = (uint32_t)e[2] | ((uint32_t)e[6] << 16);
      o.w = (uint32_t)e[3] | ((uint32_t)e[7] << 16);
      dst[ch] = o;
    }
  }
}

// y[t][m] = sum_j w[t][j] * pair_out[t*k + j][m] (+ y_shared), j in order;
// pairs whose expert is not usable contribute nothing. A warp per (token,
// 256-column segment): lanes j < k resolve choice j's usability and weight
// once, then every lane loads its 8 columns of all the token's usable pair
// rows (up to 8 rows in flight) before adding them in j order.
constexpr int kCombineWarps = 8;
__global__ void __launch_bounds__(kCombineWarps * 32, 2)
    grouped_combine_kernel(const float* __restrict__ pair_out, const int32_t* __restrict__ ids,
                           const float* __restrict__ w, const int32_t* __restrict__ slot_of, int n_slots, int E,
                           int T, int k, int H, const __half* __restrict__ y_shared, __half* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int segs = (H + 255) / 256;
  const long long units = (long long)T * segs;
  for (long long u = (long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5); u < units;
       u += (long long)gridDim.x * kCombineWarps) {
    const int t = (int)(u / segs), m0 = (int)(u - (long long)t * segs) * 256 + 8 * lane;
    const bool mv = m0 < H;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int j0 = 0; j0 < k; j0 += 32) {
      // choice j0 + lane: usable, and its weight
      bool use = false;
      float wl = 0.0f;
      if (j0 + lane < k) {
        const int q = t * k + j0 + lane;
        const int e = ids[q];
        if (e >= 0 && e < E) {
          const int s = slot_of[e];
          use = s >= 0 && s < n_slots;
        }
        wl = w[q];
      }
      const unsigned um = __ballot_sync(0xffffffffu, use);
      const int nj = min(32, k - j0);
      for (int jb = 0; jb < nj; jb += 8) {
        float4 v[8][2];
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          const int j = jb + d;
          if (j < nj && ((um >> j) & 1u) && mv) {
            const float4* src = reinterpret_cast<const float4*>(pair_out + (size_t)(t * k + j0 + j) * H + m0);
            v[d][0] = src[0];
            v[d][1] = src[1];
          }
        }
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          const int j = jb + d;
          const float wj = __shfl_sync(0xffffffffu, wl, j & 31);
          if (j < nj && ((um >> j) & 1u) && mv) {
            acc[0] += wj * v[d][0].x; acc[1] += wj * v[d][0].y; acc[2] += wj * v[d][0].z; acc[3] += wj * v[d][0].w;
            acc[4] += wj * v[d][1].x; acc[5] += wj * v[d][1].y; acc[6] += wj * v[d][1].z; acc[7] += wj * v[d][1].w;
          }
        }
      }
    }
    if (mv) {
      if (y_shared) {
        const uint4 ys = *reinterpret_cast<const uint4*>(y_shared + (size_t)t * H + m0);
        const __half* e = reinterpret_cast<const __half*>(&ys);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += __half2float(e[c]);
      }
      uint4 o;
      __half* oh = reinterpret_cast<__half*>(&o);
#pragma unroll
      for (int c = 0; c < 8; ++c) oh[c] = __float2half_rn(acc[c]);
      *reinterpret_cast<uint4*>(y + (size_t)t * H + m0) = o;
    }
  }
}

// Workspace carve-up of the grouped path.
struct GroupedWs {
  size_t offsets, pair_tok, pair_j, n_tiles, tiles, xs, hs, pair_out, total;
  int max_tiles;
};
inline size_t up(size_t v, size_t a) { return (v + a - 1) / a * a; }
GroupedWs grouped_ws(int H, int I, int T, int k, int E) {
  const size_t P = (size_t)T * k;
  GroupedWs w;
  w.max_tiles = (int)(P / BN) + std::min<int>(E, (int)P) + 1;
  size_t o = ws_scratch_offset((int)P);
  w.offsets = o;  o = up(o + (size_t)(E + 1) * 4, 256);
  w.pair_tok = o; o = up(o + P * 4, 256);
  w.pair_j = o;   o = up(o + P * 4, 256);
  w.n_tiles = o;  o = up(o + 4, 256);
  w.tiles = o;    o = up(o + (size_t)w.max_tiles * 16, 1024);
  w.xs = o;       o = up(o + P * H * 2, 1024);
  w.hs = o;       o = up(o + P * I * 2, 1024);
  w.pair_out = o; o = up(o + P * H * 4, 256);
  w.total = o;
  return w;
}

// Per device: the GEMM kernels' shared-memory attribute has been set.
std::mutex g_attr_mutex;
bool g_attr_set[kMaxDevices] = {};

}  // namespace

size_t grouped_workspace_bytes(int H, int I, int T, int k, int E) { return grouped_ws(H, I, T, k, E).total; }

int grouped_forward(const ForwardArgs& a) {
  const int P = a.T * a.k;
  if (a.E > 1024 || P > 65536)
    return fail(MOE_ERR_UNSUPPORTED, "grouped path: needs E <= 1024 and T*k <= 65536 (E=%d, T*k=%d)", a.E, P);
  if (reinterpret_cast<uintptr_t>(a.y) % 16 || reinterpret_cast<uintptr_t>(a.y_shared) % 16)
    return fail(MOE_ERR_ARG, "grouped path: y and y_shared must be 16-byte aligned");
  const GroupedWs w = grouped_ws(a.H, a.I, a.T, a.k, a.E);
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  int32_t* flags = reinterpret_cast<int32_t*>(ws);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + w.offsets);
  int32_t* pair_tok = reinterpret_cast<int32_t*>(ws + w.pair_tok);
  int32_t* pair_j = reinterpret_cast<int32_t*>(ws + w.pair_j);
  int32_t* n_tiles = reinterpret_cast<int32_t*>(ws + w.n_tiles);
  int4* tiles = reinterpret_cast<int4*>(ws + w.tiles);
  __half* xs = reinterpret_cast<__half*>(ws + w.xs);
  __half* hs = reinterpret_cast<__half*>(ws + w.hs);
  float* pair_out = reinterpret_cast<float*>(ws + w.pair_out);
  cudaStream_t st = a.stream;

  SortTiles stl;
  stl.slot_of = a.slot_of;
  stl.n_slots = a.n_slots;
  stl.tile_n = BN;
  stl.tiles = tiles;
  stl.n_tiles = n_tiles;
  stl.flags = flags;
  int rc = launch_token_sort(a.ids, P, a.k, a.E, offsets, pair_tok, pair_j, st, &stl);
  if (rc != MOE_OK) return rc;
  grouped_gather_kernel<<<8 * 152, kGatherWarps * 32, 0, st>>>(a.x, a.H, offsets, a.E, pair_tok, xs);
  if ((rc = check_launch("grouped gather")) != MOE_OK) return rc;

  // Tensor maps: expert sections of the pool (bytes; rows; slots) and the
  // sorted FP16 operands (elements; sorted pairs), 128-byte swizzle.
  CUtensorMap m_gu, m_dn, m_x, m_h;
  {
    const uint64_t dims[3] = {a.off.gu_row, (uint64_t)a.I, (uint64_t)a.n_slots};
    const uint64_t str[2] = {a.off.gu_row, a.block_bytes};
    const uint32_t box[3] = {32, BM, 1};
    if ((rc = encode_tensor_map(&m_gu, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.pool, dims, str, box,
                                CU_TENSOR_MAP_SWIZZLE_NONE)) != MOE_OK)
      return rc;
  }
  {
    const uint64_t dims[3] = {a.off.d_row, (uint64_t)a.H, (uint64_t)a.n_slots};
    const uint64_t str[2] = {a.off.d_row, a.block_bytes};
    const uint32_t box[3] = {32, BM, 1};
    if ((rc = encode_tensor_map(&m_dn, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.pool + a.off.d_offset, dims, str, box,
                                CU_TENSOR_MAP_SWIZZLE_NONE)) != MOE_OK)
      return rc;
  }
  {
    const uint64_t dims[2] = {(uint64_t)a.H, (uint64_t)P};
    const uint64_t str[1] = {(uint64_t)a.H * 2};
    const uint32_t box[2] = {BK, 64};
    if ((rc = encode_tensor_map(&m_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xs, dims, str, box,
                                CU_TENSOR_MAP_SWIZZLE_128B)) != MOE_OK)
      return rc;
  }
  {
    const uint64_t dims[2] = {(uint64_t)a.I, (uint64_t)P};
    const uint64_t str[1] = {(uint64_t)a.I * 2};
    const uint32_t box[2] = {BK, 64};
    if ((rc = encode_tensor_map(&m_h, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hs, dims, str, box,
                                CU_TENSOR_MAP_SWIZZLE_128B)) != MOE_OK)
      return rc;
  }
  int dev = 0, n_sm = 0;
  if ((rc = current_device_sms(&dev, &n_sm)) != MOE_OK) return rc;
  {
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    if (!g_attr_set[dev]) {
      MOE_CUDA_TRY(cudaFuncSetAttribute(grouped_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Geo<2>::smem));
      MOE_CUDA_TRY(cudaFuncSetAttribute(grouped_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Geo<1>::smem));
      g_attr_set[dev] = true;
    }
  }
  GemmParams gp = {};
  gp.tiles = tiles;
  gp.n_tiles = n_tiles;
  gp.g = a.g;
  gp.g_magic = (uint32_t)((0x100000000ull + (uint64_t)a.g - 1) / (uint64_t)a.g);
  gp.pair_tok = pair_tok;
  gp.pair_j = pair_j;
  gp.k = a.k;
  gp.flags = flags;
  GemmParams gu = gp;
  gu.rows = a.I;
  gu.K = a.H;
  gu.q0 = a.off.gu_q_gate;
  gu.q1 = a.off.gu_q_up;
  gu.sz = a.off.gu_sz;
  gu.h_sorted = hs;
  const int gu_items = ((a.I + BM - 1) / BM) * w.max_tiles, dn_items = ((a.H + BM - 1) / BM) * w.max_tiles;
  grouped_gemm_kernel<2><<<std::min(n_sm, gu_items), kThreadsOf<2>, Geo<2>::smem, st>>>(m_gu, m_x, gu);
  if ((rc = check_launch("grouped gate/up GEMM")) != MOE_OK) return rc;
  GemmParams dn = gp;
  dn.rows = a.H;
  dn.K = a.I;
  dn.q0 = a.off.d_q;
  dn.sz = a.off.d_sz;
  dn.pair_out = pair_out;
  grouped_gemm_kernel<1><<<std::min(n_sm, dn_items), kThreadsOf<1>, Geo<1>::smem, st>>>(m_dn, m_h, dn);
  if ((rc = check_launch("grouped down GEMM")) != MOE_OK) return rc;
  grouped_combine_kernel<<<8 * 152, kCombineWarps * 32, 0, st>>>(pair_out, a.ids, a.weights, a.slot_of, a.n_slots, a.E, a.T,
                                                  a.k, a.H, a.y_shared, a.y);
  return check_launch("grouped combine");
}

}  // namespace moe
