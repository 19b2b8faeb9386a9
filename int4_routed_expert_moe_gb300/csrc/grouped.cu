// Grouped (token-sorted) tensor-core path of the routed expert FFN, for
// prefill and large batches.
//
// "Horizon RunMap -- Prévia Técnica", "03 / Arquitetura" and "04 /
// Resultados": the compact INT4 experts are computed in groups of the tokens
// routed to them; the weights stay INT4 + FP16 scale/zero in memory and are
// expanded only on chip, activations are FP16 and accumulation FP32.
//
// Steps (one stream, six launches):
//   1. token sort: pairs p = t*k + j grouped by expert (stable);
//   2. tile list: for every resident expert with pairs, tiles of up to 128
//      consecutive sorted pairs; unusable ids are reported in the flags;
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
constexpr int BK = 64;   // K elements per pipeline stage (one 128-byte swizzle row)
constexpr int BN = 128;  // sorted pairs per tile at most (MMA N)
constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2..9 expand + epilogue
constexpr int kDqWarps = 8;

// Stage layouts (offsets inside a stage; every stage starts 1024-aligned).
constexpr uint32_t kTileBytes = BM * BK * 2;  // one FP16 operand tile, 16 KB
constexpr uint32_t kCodeBytes = BM * 32;      // codes of 128 rows x 64 elements
constexpr uint32_t kSzBytes = BM * 32;        // 32 bytes of scale/zero per row
// gate/up: A_gate | A_up | B | codes_gate | codes_up | quads
constexpr uint32_t kGuAg = 0, kGuAu = kTileBytes, kGuB = 2 * kTileBytes, kGuCg = 3 * kTileBytes,
                   kGuCu = kGuCg + kCodeBytes, kGuQ = kGuCu + kCodeBytes, kGuStage = kGuQ + kSzBytes;
// down: A | B | codes | pairs
constexpr uint32_t kDnA = 0, kDnB = kTileBytes, kDnC = 2 * kTileBytes, kDnQ = kDnC + kCodeBytes,
                   kDnStage = kDnQ + kSzBytes;
constexpr int kGuStages = 3, kDnStages = 4;
constexpr uint32_t kCtrlBytes = 1024;
constexpr size_t kGuSmem = (size_t)kGuStages * kGuStage + kCtrlBytes + 1024;
constexpr size_t kDnSmem = (size_t)kDnStages * kDnStage + kCtrlBytes + 1024;
static_assert(kGuStage % 1024 == 0 && kDnStage % 1024 == 0, "stages must keep 1024-byte alignment");

// Position of element e (0..7) of an 8-element chunk in the K order used by
// the tensor-core operands: elements (0, 4, 1, 5, 2, 6, 3, 7) in that order.
__host__ __device__ constexpr int kperm_pos(int e) { return (e & 3) * 2 + (e >> 2); }

// Expands one 32-bit word of codes (elements 8w .. 8w+7, element i in bits
// 4i..4i+3) into eight FP16 weights (q - z) * s in the operand K order.
// zz = 1024 + round(z) and t = 1024 + q are exact, so t - zz = q - round(z)
// exactly; the fused multiply-add adds (round(z) - z) * s (zero for an
// integer zero point) and rounds once.
__device__ __forceinline__ uint4 dq_word(uint32_t w, half2 zz, half2 s2, half2 c2) {
  const uint32_t m = 0x000F000Fu, mg = 0x64006400u;
  const uint32_t t0 = (w & m) | mg, t1 = ((w >> 4) & m) | mg, t2 = ((w >> 8) & m) | mg,
                 t3 = ((w >> 12) & m) | mg;
  uint4 o;
  half2 h;
  h = __hfma2(__hsub2(u32_as_h2(t0), zz), s2, c2);
  o.x = *reinterpret_cast<uint32_t*>(&h);
  h = __hfma2(__hsub2(u32_as_h2(t1), zz), s2, c2);
  o.y = *reinterpret_cast<uint32_t*>(&h);
  h = __hfma2(__hsub2(u32_as_h2(t2), zz), s2, c2);
  o.z = *reinterpret_cast<uint32_t*>(&h);
  h = __hfma2(__hsub2(u32_as_h2(t3), zz), s2, c2);
  o.w = *reinterpret_cast<uint32_t*>(&h);
  return o;
}

struct DqConst {
  half2 zz, s2, c2;
};
__device__ __forceinline__ DqConst dq_const(uint32_t sz) {  // sz: (s, z) FP16 bits
  const float s = __half2float(__ushort_as_half((unsigned short)(sz & 0xFFFFu)));
  const float z = __half2float(__ushort_as_half((unsigned short)(sz >> 16)));
  const float zi = rintf(z);
  DqConst d;
  d.zz = __float2half2_rn(1024.0f + zi);
  d.s2 = __float2half2_rn(s);
  d.c2 = __float2half2_rn((zi - z) * s);
  return d;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = tc::smem_addr(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

struct Ctrl {  // at the end of the stage area
  uint64_t* tma_full;
  uint64_t* a_full;
  uint64_t* empty;
  uint64_t* acc_full;
  uint32_t* tmem_slot;
  int* abort;
};
__device__ __forceinline__ Ctrl ctrl_at(uint8_t* p, int stages) {
  Ctrl c;
  c.tma_full = reinterpret_cast<uint64_t*>(p);
  c.a_full = c.tma_full + stages;
  c.empty = c.a_full + stages;
  c.acc_full = c.empty + stages;
  c.tmem_slot = reinterpret_cast<uint32_t*>(c.acc_full + 1);
  c.abort = reinterpret_cast<int*>(c.tmem_slot + 1);
  return c;
}

__device__ __forceinline__ void set_abort(const Ctrl& c, int32_t* flags) {
  atomicOr(flags, 4);
  *reinterpret_cast<volatile int*>(c.abort) = 1;
}
__device__ __forceinline__ bool aborted(const Ctrl& c) { return *reinterpret_cast<volatile int*>(c.abort) != 0; }

struct GemmParams {
  const int4* tiles;  // (slot, first sorted position, pairs, expert)
  const int32_t* n_tiles;
  int rows;           // output rows of the weight matrix (I for gate/up, H for down)
  int K;              // reduction length (H for gate/up, I for down)
  int g;
  uint32_t q0, q1, sz;  // byte offsets in a weight row: codes (gate, up) or codes (down), scale/zero
  __half* h_sorted;     // gate/up output [P][I]
  float* pair_out;      // down output [T*k][H]
  const int32_t* pair_tok;
  const int32_t* pair_j;
  int k;
  int32_t* flags;
};

// Common set-up: barriers, TMEM allocation. Returns the TMEM base address.
__device__ __forceinline__ uint32_t gemm_setup(const Ctrl& c, int stages, uint32_t tmem_cols) {
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      tc::bar_init(&c.tma_full[s], 1);
      tc::bar_init(&c.a_full[s], kDqWarps);
      tc::bar_init(&c.empty[s], 1);
    }
    tc::bar_init(c.acc_full, 1);
    *c.abort = 0;
    tc::bar_init_fence();
  }
  if (warp == 1) tc::tmem_alloc(c.tmem_slot, tmem_cols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  return *c.tmem_slot;
}

__device__ __forceinline__ void gemm_teardown(uint32_t tmem, uint32_t tmem_cols) {
  tc::tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, tmem_cols);
  }
}

// Producer tail after an abort: wait (bounded) for the loads still in flight.
__device__ __forceinline__ void drain_loads(const Ctrl& c, int stages, int issued) {
  for (int kt = max(0, issued - stages); kt < issued; ++kt) tc::bar_wait(&c.tma_full[kt % stages], (kt / stages) & 1);
}

// ---- gate/up GEMM + SwiGLU --------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gateup_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                          const GemmParams a) {
  const int tile = blockIdx.y;
  if (tile >= *a.n_tiles) return;
  const int4 td = a.tiles[tile];
  const int slot = td.x, pos0 = td.y, n = td.z;
  const int row0 = blockIdx.x * BM;
  const int nmma = (n + 15) & ~15;
  const int KT = a.K / BK;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  const Ctrl c = ctrl_at(sm + (size_t)kGuStages * kGuStage, kGuStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::tma_prefetch_desc(&map_w);
    tc::tma_prefetch_desc(&map_x);
  }
  const uint32_t tmem = gemm_setup(c, kGuStages, 2 * BN);

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % kGuStages;
        if (kt >= kGuStages && !tc::bar_wait(&c.empty[s], ((kt / kGuStages) - 1) & 1)) {
          set_abort(c, a.flags);
          break;
        }
        if (aborted(c)) break;
        uint8_t* st = sm + (size_t)s * kGuStage;
        const int k0 = kt * BK;
        const int gb = (k0 / a.g) & ~1;  // first of the four quads loaded
        tc::bar_expect_tx(&c.tma_full[s], 3 * kCodeBytes + kTileBytes);
        tc::tma_load_3d(st + kGuCg, &map_w, (int)a.q0 + k0 / 2, row0, slot, &c.tma_full[s]);
        tc::tma_load_3d(st + kGuCu, &map_w, (int)a.q1 + k0 / 2, row0, slot, &c.tma_full[s]);
        tc::tma_load_3d(st + kGuQ, &map_w, (int)a.sz + 8 * gb, row0, slot, &c.tma_full[s]);
        tc::tma_load_2d(st + kGuB, &map_x, k0, pos0, &c.tma_full[s]);
        issued = kt + 1;
      }
      if (aborted(c)) drain_loads(c, kGuStages, issued);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(BM, nmma);
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % kGuStages;
        if (!tc::bar_wait(&c.a_full[s], (kt / kGuStages) & 1)) {
          set_abort(c, a.flags);
          break;
        }
        if (aborted(c)) break;
        tc::tc_fence_after();
        const uint32_t base = tc::smem_addr(sm + (size_t)s * kGuStage);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t bdesc = tc::sw128_desc(base + kGuB + kk * 32);
          const bool acc = kt > 0 || kk > 0;
          tc::mma_f16(tmem, tc::sw128_desc(base + kGuAg + kk * 32), bdesc, idesc, acc);
          tc::mma_f16(tmem + BN, tc::sw128_desc(base + kGuAu + kk * 32), bdesc, idesc, acc);
        }
        tc::mma_commit(&c.empty[s]);
      }
      tc::mma_commit(c.acc_full);
    }
  } else {
    const int dt = threadIdx.x - 64;  // 0..255
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % kGuStages;
      if (aborted(c)) break;
      if (!tc::bar_wait(&c.tma_full[s], (kt / kGuStages) & 1)) {
        set_abort(c, a.flags);
        break;
      }
      uint8_t* st = sm + (size_t)s * kGuStage;
      const int k0 = kt * BK;
      const int gi0 = k0 / a.g, gb = gi0 & ~1, kb = (gi0 + 1) * a.g;
#pragma unroll
      for (int pj = 0; pj < 2; ++pj) {  // projection: 0 gate, 1 up
        const int u = dt;
        const int r = u >> 1, half = u & 1;
        const uint4 cw = *reinterpret_cast<const uint4*>(st + (pj ? kGuCu : kGuCg) + r * 32 + half * 16);
        const uint8_t* qrow = st + kGuQ + r * 32;
        uint8_t* A = st + (pj ? kGuAu : kGuAg);
        const uint32_t wv[4] = {cw.x, cw.y, cw.z, cw.w};
        int gcur = -1;
        DqConst d;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = half * 4 + j;
          const int gi = (k0 + 8 * ch < kb) ? gi0 : gi0 + 1;
          if (gi != gcur) {
            d = dq_const(*reinterpret_cast<const uint32_t*>(qrow + (gi - gb) * 8 + pj * 4));
            gcur = gi;
          }
          *reinterpret_cast<uint4*>(A + tc::sw128_offset(r, ch)) = dq_word(wv[j], d.zz, d.s2, d.c2);
        }
      }
      tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) tc::bar_arrive(&c.a_full[s]);
    }
    // Epilogue: TMEM lanes of this warp's quarter, half of the columns.
    const bool ok = tc::bar_wait(c.acc_full, 0);
    if (!ok) set_abort(c, a.flags);
    tc::tc_fence_after();
    const int q4 = warp & 3, chalf = (warp - 2) >> 2;
    const int row = row0 + 32 * q4 + lane;
    const int prow = (row & ~7) | kperm_pos(row & 7);
    const bool live = ok && !aborted(c) && row < a.rows;
    for (int c0 = chalf * (BN / 2); c0 < chalf * (BN / 2) + BN / 2 && c0 < nmma; c0 += 16) {
      float gv[16], uv[16];
      tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)c0, gv);
      tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)(BN + c0), uv);
      tc::tmem_ld_wait();
      if (live) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < n)
            a.h_sorted[(size_t)(pos0 + c0 + j) * a.rows + prow] = __float2half_rn(silu_f(gv[j]) * uv[j]);
      }
    }
  }
  gemm_teardown(tmem, 2 * BN);
}

// ---- down GEMM ----------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
    grouped_down_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_h,
                        const GemmParams a) {
  const int tile = blockIdx.y;
  if (tile >= *a.n_tiles) return;
  const int4 td = a.tiles[tile];
  const int slot = td.x, pos0 = td.y, n = td.z;
  const int row0 = blockIdx.x * BM;
  const int nmma = (n + 15) & ~15;
  const int KT = a.K / BK;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  const Ctrl c = ctrl_at(sm + (size_t)kDnStages * kDnStage, kDnStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::tma_prefetch_desc(&map_w);
    tc::tma_prefetch_desc(&map_h);
  }
  const uint32_t tmem = gemm_setup(c, kDnStages, BN);

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % kDnStages;
        if (kt >= kDnStages && !tc::bar_wait(&c.empty[s], ((kt / kDnStages) - 1) & 1)) {
          set_abort(c, a.flags);
          break;
        }
        if (aborted(c)) break;
        uint8_t* st = sm + (size_t)s * kDnStage;
        const int k0 = kt * BK;
        const int gb = (k0 / a.g) & ~3;  // first of the eight pairs loaded
        tc::bar_expect_tx(&c.tma_full[s], 2 * kCodeBytes + kTileBytes);
        tc::tma_load_3d(st + kDnC, &map_w, (int)a.q0 + k0 / 2, row0, slot, &c.tma_full[s]);
        tc::tma_load_3d(st + kDnQ, &map_w, (int)a.sz + 4 * gb, row0, slot, &c.tma_full[s]);
        tc::tma_load_2d(st + kDnB, &map_h, k0, pos0, &c.tma_full[s]);
        issued = kt + 1;
      }
      if (aborted(c)) drain_loads(c, kDnStages, issued);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(BM, nmma);
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % kDnStages;
        if (!tc::bar_wait(&c.a_full[s], (kt / kDnStages) & 1)) {
          set_abort(c, a.flags);
          break;
        }
        if (aborted(c)) break;
        tc::tc_fence_after();
        const uint32_t base = tc::smem_addr(sm + (size_t)s * kDnStage);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc::mma_f16(tmem, tc::sw128_desc(base + kDnA + kk * 32), tc::sw128_desc(base + kDnB + kk * 32), idesc,
                      kt > 0 || kk > 0);
        tc::mma_commit(&c.empty[s]);
      }
      tc::mma_commit(c.acc_full);
    }
  } else {
    const int dt = threadIdx.x - 64;
    const int r = dt >> 1, half = dt & 1;
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % kDnStages;
      if (aborted(c)) break;
      if (!tc::bar_wait(&c.tma_full[s], (kt / kDnStages) & 1)) {
        set_abort(c, a.flags);
        break;
      }
      uint8_t* st = sm + (size_t)s * kDnStage;
      const int k0 = kt * BK;
      const int gi0 = k0 / a.g, gb = gi0 & ~3, kb = (gi0 + 1) * a.g;
      const uint4 cw = *reinterpret_cast<const uint4*>(st + kDnC + r * 32 + half * 16);
      const uint8_t* prow = st + kDnQ + r * 32;
      uint8_t* A = st + kDnA;
      const uint32_t wv[4] = {cw.x, cw.y, cw.z, cw.w};
      int gcur = -1;
      DqConst d;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ch = half * 4 + j;
        const int gi = (k0 + 8 * ch < kb) ? gi0 : gi0 + 1;
        if (gi != gcur) {
          d = dq_const(*reinterpret_cast<const uint32_t*>(prow + (gi - gb) * 4));
          gcur = gi;
        }
        *reinterpret_cast<uint4*>(A + tc::sw128_offset(r, ch)) = dq_word(wv[j], d.zz, d.s2, d.c2);
      }
      tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) tc::bar_arrive(&c.a_full[s]);
    }
    const bool ok = tc::bar_wait(c.acc_full, 0);
    if (!ok) set_abort(c, a.flags);
    tc::tc_fence_after();
    const int q4 = warp & 3, chalf = (warp - 2) >> 2;
    const int row = row0 + 32 * q4 + lane;
    const bool live = ok && !aborted(c) && row < a.rows;
    for (int c0 = chalf * (BN / 2); c0 < chalf * (BN / 2) + BN / 2 && c0 < nmma; c0 += 16) {
      float dv[16];
      tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)c0, dv);
      tc::tmem_ld_wait();
      if (live) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (c0 + j < n) {
            const int pos = pos0 + c0 + j;
            const size_t q = (size_t)a.pair_tok[pos] * a.k + a.pair_j[pos];
            a.pair_out[q * a.rows + row] = dv[j];
          }
        }
      }
    }
  }
  gemm_teardown(tmem, BN);
}

// ---- small kernels -------------------------------------------------------------
// Tile list (one block) and unusable-id reporting.
__global__ void grouped_tiles_kernel(const int32_t* __restrict__ ids, int P, int E,
                                     const int32_t* __restrict__ offsets, const int32_t* __restrict__ slot_of,
                                     int n_slots, int4* __restrict__ tiles, int32_t* __restrict__ n_tiles,
                                     int32_t* __restrict__ flags) {
  const int tid = threadIdx.x;
  for (int p = tid; p < P; p += blockDim.x) {
    const int e = ids[p];
    if (e != -1 && (e < 0 || e >= E)) {
      atomicOr(flags, 2);
    } else if (e >= 0) {
      const int s = slot_of[e];
      if (s < 0 || s >= n_slots) atomicOr(flags, 1);
    }
  }
  if (tid < 32) {
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + tid;
      int cnt = 0, s = -1, o0 = 0, ne = 0;
      if (e < E) {
        o0 = offsets[e];
        ne = offsets[e + 1] - o0;
        s = slot_of[e];
        if (ne > 0 && s >= 0 && s < n_slots) cnt = (ne + BN - 1) / BN;
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += v;
      }
      for (int i = 0; i < cnt; ++i)
        tiles[carry + incl - cnt + i] = make_int4(s, o0 + i * BN, min(BN, ne - i * BN), e);
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (tid == 0) *n_tiles = carry;
  }
}

// X_sorted[pos] = x[pair_tok[pos]], each 8-element chunk in operand K order.
__global__ void grouped_gather_kernel(const __half* __restrict__ x, int H, const int32_t* __restrict__ offsets,
                                      int E, const int32_t* __restrict__ pair_tok, __half* __restrict__ xs) {
  const int pv = offsets[E];
  const int cpr = H / 8;
  const long long total = (long long)pv * cpr;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int pos = (int)(i / cpr), ch = (int)(i - (long long)pos * cpr);
    const int t = pair_tok[pos];
    const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)t * H + 8 * ch);
    const unsigned short* e = reinterpret_cast<const unsigned short*>(&v);
    uint4 o;
    o.x = (uint32_t)e[0] | ((uint32_t)e[4] << 16);
    o.y = (uint32_t)e[1] | ((uint32_t)e[5] << 16);
    o.z = (uint32_t)e[2] | ((uint32_t)e[6] << 16);
    o.w = (uint32_t)e[3] | ((uint32_t)e[7] << 16);
    *reinterpret_cast<uint4*>(xs + (size_t)pos * H + 8 * ch) = o;
  }
}

// y[t][m] = sum_j w[t][j] * pair_out[t*k + j][m] (+ y_shared), j in order;
// pairs whose expert is not usable contribute nothing.
__global__ void grouped_combine_kernel(const float* __restrict__ pair_out, const int32_t* __restrict__ ids,
                                       const float* __restrict__ w, const int32_t* __restrict__ slot_of,
                                       int n_slots, int E, int T, int k, int H, const __half* __restrict__ y_shared,
                                       __half* __restrict__ y) {
  const int cpr = H / 8;
  const long long total = (long long)T * cpr;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / cpr), m0 = 8 * (int)(i - (long long)t * cpr);
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int j = 0; j < k; ++j) {
      const int q = t * k + j;
      const int e = ids[q];
      if (e < 0 || e >= E) continue;
      const int s = slot_of[e];
      if (s < 0 || s >= n_slots) continue;
      const float wj = w[q];
      const float4* src = reinterpret_cast<const float4*>(pair_out + (size_t)q * H + m0);
      const float4 v0 = src[0], v1 = src[1];
      acc[0] += wj * v0.x; acc[1] += wj * v0.y; acc[2] += wj * v0.z; acc[3] += wj * v0.w;
      acc[4] += wj * v1.x; acc[5] += wj * v1.y; acc[6] += wj * v1.z; acc[7] += wj * v1.w;
    }
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

bool g_attr_done = false;

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

  int rc = launch_token_sort(a.ids, P, a.k, a.E, offsets, pair_tok, pair_j, st);
  if (rc != MOE_OK) return rc;
  grouped_tiles_kernel<<<1, 1024, 0, st>>>(a.ids, P, a.E, offsets, a.slot_of, a.n_slots, tiles, n_tiles, flags);
  if ((rc = check_launch("grouped tiles")) != MOE_OK) return rc;
  grouped_gather_kernel<<<4 * 152, 256, 0, st>>>(a.x, a.H, offsets, a.E, pair_tok, xs);
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
    const uint32_t box[2] = {BK, BN};
    if ((rc = encode_tensor_map(&m_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xs, dims, str, box,
                                CU_TENSOR_MAP_SWIZZLE_128B)) != MOE_OK)
      return rc;
  }
  {
    const uint64_t dims[2] = {(uint64_t)a.I, (uint64_t)P};
    const uint64_t str[1] = {(uint64_t)a.I * 2};
    const uint32_t box[2] = {BK, BN};
    if ((rc = encode_tensor_map(&m_h, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hs, dims, str, box,
                                CU_TENSOR_MAP_SWIZZLE_128B)) != MOE_OK)
      return rc;
  }
  if (!g_attr_done) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(grouped_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGuSmem));
    MOE_CUDA_TRY(cudaFuncSetAttribute(grouped_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDnSmem));
    g_attr_done = true;
  }
  GemmParams gp = {};
  gp.tiles = tiles;
  gp.n_tiles = n_tiles;
  gp.g = a.g;
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
  grouped_gateup_kernel<<<dim3((a.I + BM - 1) / BM, w.max_tiles), kThreads, kGuSmem, st>>>(m_gu, m_x, gu);
  if ((rc = check_launch("grouped gate/up GEMM")) != MOE_OK) return rc;
  GemmParams dn = gp;
  dn.rows = a.H;
  dn.K = a.I;
  dn.q0 = a.off.d_q;
  dn.sz = a.off.d_sz;
  dn.pair_out = pair_out;
  grouped_down_kernel<<<dim3((a.H + BM - 1) / BM, w.max_tiles), kThreads, kDnSmem, st>>>(m_dn, m_h, dn);
  if ((rc = check_launch("grouped down GEMM")) != MOE_OK) return rc;
  grouped_combine_kernel<<<4 * 152, 256, 0, st>>>(pair_out, a.ids, a.weights, a.slot_of, a.n_slots, a.E, a.T,
                                                  a.k, a.H, a.y_shared, a.y);
  return check_launch("grouped combine");
}

}  // namespace moe
